// a1 online quantizer and a2 repack / unrepack kernels + their C ABI.
//
// Quantization rule (FastLLM page, section 3.1: groups of 128 weights along K,
// one scale and one zero point per group), evaluated in double precision so
// that every code decision is taken in one fixed precision:
//   s = (max - min)/15, s16 = fp16(s), z = clamp(round(-min/s16), 0, 15),
//   q = clamp(round(w/s16) + z, 0, 15), round = half away from zero.
// Groups of 256 (same page, section 4.2: --group-size 128 by default, 256
// allowed) are quantized by the same rule; in the interleaved layout, whose
// super-blocks always span 128 columns, both super-blocks of a group carry
// its scale and zero point, so every matmul kernel reads them unchanged.
// Groups of 64 (section 5.4: 64 for more precision): the super-blocks carry
// the scale and zero point of the even group (columns 0..63 of the 128) and
// a side array after them, one 320-byte entry per super-block in the same
// order, carries those of the odd group (128 fp16 scales, 128 zero points).
#include "fl_common.cuh"

using namespace fl;

namespace {

__device__ __forceinline__ double round_half_away(double v) {
  double t = trunc(v);
  if (fabs(v - t) >= 0.5) t += copysign(1.0, v);
  return t;
}

__device__ __forceinline__ int clamp15(double v) { return v < 0.0 ? 0 : (v > 15.0 ? 15 : static_cast<int>(v)); }

// One warp per (row n, pair of groups 2gp, 2gp+1): the pair shares a zero
// byte.  GRP/32 consecutive weights per lane.
template <int GRP>
__global__ void k_quantize(const float* __restrict__ w, int N, int K, int G, uint8_t* __restrict__ q,
                           uint16_t* __restrict__ sc, uint8_t* __restrict__ zr, int32_t* __restrict__ status) {
  constexpr int V = GRP / 32;   // 2, 4 or 8
  static_assert(V == 2 || V == 4 || V == 8, "groups of 64, 128 or 256");
  const int lane = threadIdx.x & 31;
  const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int GP = (G + 1) / 2;
  if (warp >= static_cast<long long>(N) * GP) return;
  const int n = static_cast<int>(warp / GP);
  const int gp = static_cast<int>(warp % GP);
  uint32_t zbyte = 0;
  for (int h = 0; h < 2; ++h) {
    const int g = 2 * gp + h;
    if (g >= G) break;
    float vv[V];
    const float* src = w + static_cast<size_t>(n) * K + static_cast<size_t>(g) * GRP + V * lane;
    if (V == 2) {
      const float2 v2 = *reinterpret_cast<const float2*>(src);
      vv[0] = v2.x, vv[V - 1] = v2.y;
    } else {
#pragma unroll
      for (int c = 0; c < V / 4; ++c) {
        const float4 v4 = *reinterpret_cast<const float4*>(src + 4 * c);
        vv[4 * c] = v4.x, vv[4 * c + 1] = v4.y, vv[4 * c + 2] = v4.z, vv[4 * c + 3] = v4.w;
      }
    }
    float mn = vv[0], mx = vv[0];
    int bad = 0;
#pragma unroll
    for (int j = 0; j < V; ++j) {
      mn = fminf(mn, vv[j]);
      mx = fmaxf(mx, vv[j]);
      bad |= isnan(vv[j]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      bad |= __shfl_xor_sync(0xffffffffu, bad, o);
    }
    double dmn = mn, dmx = mx;
    bool zero = false;
    if (dmn == dmx) {
      if (dmn == 0.0) zero = true;
      dmn = fmin(dmn, 0.0);
      dmx = fmax(dmx, 0.0);
    }
    uint16_t sbits = 0;
    double s16 = 0.0;
    if (!zero) {
      const __half hs = __double2half((dmx - dmn) / 15.0);
      sbits = __half_as_ushort(hs);
      s16 = static_cast<double>(__half2float(hs));
      if (bad || isinf(s16) || isnan(s16)) {
        if (lane == 0) set_status(status, FL_ERR_RANGE, n);
        zero = true;
        sbits = 0;
      } else if (s16 == 0.0) {
        zero = true;
      }
    }
    int z = 0;
    uint32_t packed = 0;
    if (!zero) {
      z = clamp15(round_half_away(-dmn / s16));
#pragma unroll
      for (int j = 0; j < V; ++j) {
        const int qq = clamp15(round_half_away(static_cast<double>(vv[j]) / s16) + z);
        packed |= static_cast<uint32_t>(qq) << (4 * j);
      }
    }
    uint8_t* qd = q + static_cast<size_t>(n) * (K / 2) + static_cast<size_t>(g) * (GRP / 2) + (V / 2) * lane;
    if (V == 2)
      *qd = static_cast<uint8_t>(packed);
    else if (V == 4)
      *reinterpret_cast<uint16_t*>(qd) = static_cast<uint16_t>(packed);
    else
      *reinterpret_cast<uint32_t*>(qd) = packed;
    if (lane == 0) sc[static_cast<size_t>(n) * G + g] = sbits;
    zbyte |= static_cast<uint32_t>(z) << (4 * h);
  }
  if (lane == 0) zr[static_cast<size_t>(n) * GP + gp] = static_cast<uint8_t>(zbyte);
}

// Output nibble e holds canonical nibble 2*(e%4) + e/4 (even columns in the
// low half-word, odd columns in the high half-word).
__device__ __forceinline__ uint32_t canon_to_tiled_word(uint32_t cw) {
  uint32_t o = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) o |= ((cw >> (4 * (2 * (e & 3) + (e >> 2)))) & 15u) << (4 * e);
  return o;
}

__device__ __forceinline__ uint32_t tiled_to_canon_word(uint32_t tw) {
  uint32_t o = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) o |= ((tw >> (4 * e)) & 15u) << (4 * (2 * (e & 3) + (e >> 2)));
  return o;
}

// Canonical group whose scale and zero point super-block (column block) g
// carries: g >> 1 for groups of 256, g for 128, 2g for 64 (the side array:
// 2g + 1).
__device__ __forceinline__ int carried_group(int g, int group, bool side) {
  return group == 256 ? (g >> 1) : group == 128 ? g : 2 * g + (side ? 1 : 0);
}

// One block per super-block (T, g), g over the K/128 column blocks, whose
// canonical arrays have Gs = K / group entries per row.
__global__ void k_repack(const uint8_t* __restrict__ q, const uint16_t* __restrict__ sc,
                         const uint8_t* __restrict__ zr, int N, int K, int G, int group,
                         uint8_t* __restrict__ out) {
  const int sbi = blockIdx.x;
  const int T = sbi / G, g = sbi % G;
  const int Gs = K / group, gs = carried_group(g, group, false);
  const int ZB = (Gs + 1) / 2;
  uint8_t* dst = out + static_cast<size_t>(sbi) * kSbBytes;
  for (int wi = threadIdx.x; wi < kSbNib / 4; wi += blockDim.x) {
    const int r = wi >> 4, pw = wi & 15;
    const int n = T * kRowTile + r;
    uint32_t o = 0;
    if (n < N) {
      // word pw of the row is word pw%4 of chunk (pw/4 - (r/2)%4) % 4, i.e. slot p
      const int p = 4 * (((pw >> 2) - (r >> 1)) & 3) + (pw & 3);
      const int wl = 4 * (p & 3) + (p >> 2);
      const uint32_t cw =
          *reinterpret_cast<const uint32_t*>(q + static_cast<size_t>(n) * (K / 2) + g * (kGroup / 2) + 4 * wl);
      o = canon_to_tiled_word(cw);
    }
    reinterpret_cast<uint32_t*>(dst)[wi] = o;
  }
  const int t = threadIdx.x;
  if (t < kRowTile) {
    const int n = T * kRowTile + t;
    reinterpret_cast<uint16_t*>(dst + kSbNib)[t] = n < N ? sc[static_cast<size_t>(n) * Gs + gs] : 0;
  }
  if (t < kRowTile / 2) {
    uint32_t b = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int n = T * kRowTile + 2 * t + h;
      if (n < N) b |= ((zr[static_cast<size_t>(n) * ZB + gs / 2] >> (4 * (gs & 1))) & 15u) << (4 * h);
    }
    dst[kSbNib + kSbScale + t] = static_cast<uint8_t>(b);
  }
}

// Groups of 64: side entry of super-block sbi (320 bytes at side + 320 sbi):
// the odd group's 128 scales, then its 128 zero points.
__global__ void k_repack_side(const uint16_t* __restrict__ sc, const uint8_t* __restrict__ zr, int N, int K, int G,
                              uint8_t* __restrict__ side) {
  const int sbi = blockIdx.x;
  const int T = sbi / G, g = sbi % G;
  const int Gs = K / 64, gs = 2 * g + 1;
  const int ZB = (Gs + 1) / 2;
  uint8_t* dst = side + static_cast<size_t>(sbi) * kSbSide;
  const int t = threadIdx.x;
  if (t < kRowTile) {
    const int n = T * kRowTile + t;
    reinterpret_cast<uint16_t*>(dst)[t] = n < N ? sc[static_cast<size_t>(n) * Gs + gs] : 0;
  }
  if (t < kRowTile / 2) {
    uint32_t b = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int n = T * kRowTile + 2 * t + h;
      if (n < N) b |= ((zr[static_cast<size_t>(n) * ZB + gs / 2] >> (4 * (gs & 1))) & 15u) << (4 * h);
    }
    dst[kSbScale + t] = static_cast<uint8_t>(b);
  }
}

// One block per (T, pair of groups 2gp, 2gp+1): a canonical zero byte spans
// two groups.  Codes come from every super-block of the two groups, the
// scale and zero point of group gs from its first super-block gs << gshift.
__global__ void k_unrepack(const uint8_t* __restrict__ in, int N, int K, int G, int gshift,
                           uint8_t* __restrict__ q, uint16_t* __restrict__ sc, uint8_t* __restrict__ zr) {
  const int Gs = G >> gshift;
  const int ZB = (Gs + 1) / 2;
  // groups of 256 (gshift 1) and 128 (0); groups of 64: k_unrepack64
  const int T = blockIdx.x / ZB, gp = blockIdx.x % ZB;
  for (int h = 0; h < 2; ++h) {
    const int gs = 2 * gp + h;
    if (gs >= Gs) break;
    for (int sub = 0; sub < (1 << gshift); ++sub) {
      const int g = (gs << gshift) + sub;
      const uint8_t* src = in + (static_cast<size_t>(T) * G + g) * kSbBytes;
      for (int wi = threadIdx.x; wi < kSbNib / 4; wi += blockDim.x) {
        const int r = wi >> 4, pw = wi & 15;
        const int n = T * kRowTile + r;
        if (n >= N) continue;
        const int p = 4 * (((pw >> 2) - (r >> 1)) & 3) + (pw & 3);
        const int wl = 4 * (p & 3) + (p >> 2);
        *reinterpret_cast<uint32_t*>(q + static_cast<size_t>(n) * (K / 2) + g * (kGroup / 2) + 4 * wl) =
            tiled_to_canon_word(reinterpret_cast<const uint32_t*>(src)[wi]);
      }
    }
    const uint8_t* src = in + (static_cast<size_t>(T) * G + (gs << gshift)) * kSbBytes;
    const int t = threadIdx.x;
    if (t < kRowTile) {
      const int n = T * kRowTile + t;
      if (n < N) sc[static_cast<size_t>(n) * Gs + gs] = reinterpret_cast<const uint16_t*>(src + kSbNib)[t];
    }
  }
  const int t = threadIdx.x;
  if (t < kRowTile) {
    const int n = T * kRowTile + t;
    if (n < N) {
      uint32_t b = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int gs = 2 * gp + h;
        if (gs >= Gs) break;
        const uint8_t* src = in + (static_cast<size_t>(T) * G + (gs << gshift)) * kSbBytes;
        b |= ((src[kSbNib + kSbScale + t / 2] >> (4 * (t & 1))) & 15u) << (4 * h);
      }
      zr[static_cast<size_t>(n) * ZB + gp] = static_cast<uint8_t>(b);
    }
  }
}

// Groups of 64, inverse of k_repack + k_repack_side: one block per (T,
// column block g); groups 2g (the super-block) and 2g+1 (its side entry)
// share one canonical zero byte.
__global__ void k_unrepack64(const uint8_t* __restrict__ in, const uint8_t* __restrict__ side, int N, int K, int G,
                             uint8_t* __restrict__ q, uint16_t* __restrict__ sc, uint8_t* __restrict__ zr) {
  const int T = blockIdx.x / G, g = blockIdx.x % G;
  const int Gs = K / 64, ZB = (Gs + 1) / 2;
  const uint8_t* src = in + (static_cast<size_t>(T) * G + g) * kSbBytes;
  const uint8_t* sd = side + (static_cast<size_t>(T) * G + g) * kSbSide;
  for (int wi = threadIdx.x; wi < kSbNib / 4; wi += blockDim.x) {
    const int r = wi >> 4, pw = wi & 15;
    const int n = T * kRowTile + r;
    if (n >= N) continue;
    const int p = 4 * (((pw >> 2) - (r >> 1)) & 3) + (pw & 3);
    const int wl = 4 * (p & 3) + (p >> 2);
    *reinterpret_cast<uint32_t*>(q + static_cast<size_t>(n) * (K / 2) + g * (kGroup / 2) + 4 * wl) =
        tiled_to_canon_word(reinterpret_cast<const uint32_t*>(src)[wi]);
  }
  const int t = threadIdx.x;
  if (t < kRowTile) {
    const int n = T * kRowTile + t;
    if (n < N) {
      sc[static_cast<size_t>(n) * Gs + 2 * g] = reinterpret_cast<const uint16_t*>(src + kSbNib)[t];
      sc[static_cast<size_t>(n) * Gs + 2 * g + 1] = reinterpret_cast<const uint16_t*>(sd)[t];
      const uint32_t z0 = (src[kSbNib + kSbScale + t / 2] >> (4 * (t & 1))) & 15u;
      const uint32_t z1 = (sd[kSbScale + t / 2] >> (4 * (t & 1))) & 15u;
      zr[static_cast<size_t>(n) * ZB + g] = static_cast<uint8_t>(z0 | (z1 << 4));
    }
  }
}

// Group sizes of the layout: 64, 128 (gshift 0) and 256 (gshift 1).
bool group_ok(int group) { return group == kGroup / 2 || group == kGroup || group == 2 * kGroup; }
int group_shift(int group) { return group == 2 * kGroup ? 1 : 0; }
bool shape_ok(int N, int K, int group) {
  return N >= 1 && K >= kGroup && K % group == 0 && K % kGroup == 0 && group_ok(group);
}

size_t tiled_bytes(int N, int K, int group) {
  const size_t T = (static_cast<size_t>(N) + kRowTile - 1) / kRowTile;
  return T * static_cast<size_t>(K / kGroup) * (kSbBytes + (group == kGroup / 2 ? kSbSide : 0));
}

}  // namespace

extern "C" int fl_int4g_repacked_bytes(int N, int K, int group, size_t* out) {
  if (!out) return FL_ERR_ARG;
  if (!group_ok(group)) return FL_ERR_UNSUPPORTED;
  if (!shape_ok(N, K, group)) return FL_ERR_ARG;
  *out = tiled_bytes(N, K, group);
  return FL_OK;
}

extern "C" int fl_int4g_quantize(const float* w, int N, int K, int group, uint8_t* q, uint16_t* scales,
                                 uint8_t* zeros, void* status, fl_stream_t stream) {
  if (!group_ok(group)) return FL_ERR_UNSUPPORTED;
  if (!shape_ok(N, K, group) || !w || !q || !scales || !zeros || !status) return FL_ERR_ARG;
  if (!flh::aligned16(w) || !flh::aligned16(q) || !flh::aligned16(scales) || !flh::aligned16(zeros) ||
      !flh::aligned16(status))
    return FL_ERR_ARG;
  const int G = K / group;
  const long long warps = static_cast<long long>(N) * ((G + 1) / 2);
  const int threads = 256;
  const long long blocks = (warps * 32 + threads - 1) / threads;
  if (blocks > 0x7fffffffLL) return FL_ERR_UNSUPPORTED;
  if (group == kGroup / 2)
    k_quantize<64><<<static_cast<unsigned>(blocks), threads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        w, N, K, G, q, scales, zeros, static_cast<int32_t*>(status));
  else if (group == kGroup)
    k_quantize<128><<<static_cast<unsigned>(blocks), threads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        w, N, K, G, q, scales, zeros, static_cast<int32_t*>(status));
  else
    k_quantize<256><<<static_cast<unsigned>(blocks), threads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        w, N, K, G, q, scales, zeros, static_cast<int32_t*>(status));
  return cudaGetLastError() == cudaSuccess ? FL_OK : FL_ERR_CUDA;
}

extern "C" int fl_int4g_repack(const uint8_t* q, const uint16_t* scales, const uint8_t* zeros, int N, int K,
                               int group, void* w_out, size_t w_out_bytes, fl_stream_t stream) {
  if (!group_ok(group)) return FL_ERR_UNSUPPORTED;
  if (!shape_ok(N, K, group) || !q || !scales || !zeros || !w_out) return FL_ERR_ARG;
  if (!flh::aligned16(q) || !flh::aligned16(scales) || !flh::aligned16(zeros) || !flh::aligned16(w_out))
    return FL_ERR_ARG;
  if (w_out_bytes < tiled_bytes(N, K, group)) return FL_ERR_ARG;
  const int G = K / kGroup;
  const long long blocks = static_cast<long long>((N + kRowTile - 1) / kRowTile) * G;
  if (blocks > 0x7fffffffLL) return FL_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  k_repack<<<static_cast<unsigned>(blocks), 256, 0, s>>>(q, scales, zeros, N, K, G, group,
                                                         static_cast<uint8_t*>(w_out));
  if (group == kGroup / 2)
    k_repack_side<<<static_cast<unsigned>(blocks), 128, 0, s>>>(
        scales, zeros, N, K, G, static_cast<uint8_t*>(w_out) + static_cast<size_t>(blocks) * kSbBytes);
  return cudaGetLastError() == cudaSuccess ? FL_OK : FL_ERR_CUDA;
}

extern "C" int fl_int4g_unrepack(const void* w, size_t w_bytes, int N, int K, int group, uint8_t* q,
                                 uint16_t* scales, uint8_t* zeros, fl_stream_t stream) {
  if (!group_ok(group)) return FL_ERR_UNSUPPORTED;
  if (!shape_ok(N, K, group) || !q || !scales || !zeros || !w) return FL_ERR_ARG;
  if (!flh::aligned16(q) || !flh::aligned16(scales) || !flh::aligned16(zeros) || !flh::aligned16(w))
    return FL_ERR_ARG;
  if (w_bytes < tiled_bytes(N, K, group)) return FL_ERR_ARG;
  const int G = K / kGroup;
  const int Gs = K / group;
  if (group == kGroup / 2) {
    const long long nsb = static_cast<long long>((N + kRowTile - 1) / kRowTile) * G;
    if (nsb > 0x7fffffffLL) return FL_ERR_UNSUPPORTED;
    const uint8_t* in = static_cast<const uint8_t*>(w);
    k_unrepack64<<<static_cast<unsigned>(nsb), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        in, in + static_cast<size_t>(nsb) * kSbBytes, N, K, G, q, scales, zeros);
    return cudaGetLastError() == cudaSuccess ? FL_OK : FL_ERR_CUDA;
  }
  const long long blocks = static_cast<long long>((N + kRowTile - 1) / kRowTile) * ((Gs + 1) / 2);
  if (blocks > 0x7fffffffLL) return FL_ERR_UNSUPPORTED;
  k_unrepack<<<static_cast<unsigned>(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint8_t*>(w), N, K, G, group_shift(group), q, scales, zeros);
  return cudaGetLastError() == cudaSuccess ? FL_OK : FL_ERR_CUDA;
}
