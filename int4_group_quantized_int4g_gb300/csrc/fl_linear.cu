// a3: int4g decode linear, y = x . deq(W)^T for M <= 32 tokens.
//
// The weights (the interleaved layout, one 8512-byte super-block per 128 rows
// x one group) stream from HBM once.  FastLLM page, section 3.1: decode is
// memory-bound, so the 4-bit codes are read once and dequantized on the fly
// inside the matmul.  GB300 design:
//  * work = the T*G super-blocks in layout order, split into P contiguous
//    ranges, one per CTA (P = number of SMs), so every SM streams the same
//    number of bytes whatever N and K are (split over K inside a row tile);
//  * one producer warp moves super-blocks and the matching 256-byte slices of
//    every token row of x into a ring of shared-memory stages with 1-D bulk
//    copies completing on mbarriers;
//  * 8 consumer warps each own 16 rows: 16 bytes of codes per lane and row
//    become 8 exact (q - z) bf16 pairs with one LOP3 + one bf16x2 subtract per
//    pair, feeding mma.sync m16n8k16 as the A operand (the K order inside a
//    group is permuted consistently for A and B, which leaves the dot product
//    unchanged); the per-group fp16 scale is applied to the fp32 group sum;
//  * a row tile split across CTAs is reduced by the last CTA to finish it
//    (atomic ticket, no waiting), summing the partials in CTA order so the
//    result is deterministic.
#include "fl_common.cuh"

using namespace fl;

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kXRowStride = 320;  // 256 B of x per row + 64 B pad: conflict-free B-fragment loads
constexpr int kMaxTokens = 32;

struct RowsParams {
  const uint8_t* w;
  const __nv_bfloat16* x;
  __nv_bfloat16* y;
  float* part;       // [P * maxseg][128][Mp] fp32 partial sums
  int32_t* cnt;      // [T][8] tickets (zero between calls)
  int32_t* status;   // 16-byte status block
  long long U;       // units = T * G
  int M, K, N, T, G, P;
  int maxseg;
  int stages;
  uint32_t stage_bytes;
};

__host__ __device__ __forceinline__ long long unit_begin(long long c, long long U, int P) { return c * U / P; }
__host__ __device__ __forceinline__ int cta_of_unit(long long u, long long U, int P) {
  return static_cast<int>(((u + 1) * P - 1) / U);
}

template <int NT>
__device__ __forceinline__ void flush_tile(const RowsParams& p, long long T, int c, long long u0, long long u1,
                                           int warp, int lane, float (&tot)[NT][4]) {
  constexpr int Mp = 8 * NT;
  const int gid = lane >> 2, tig = lane & 3;
  const long long tu0 = T * p.G, tu1 = (T + 1) * p.G;
  const int rbase = static_cast<int>(T) * kRowTile + warp * 16;
  if (tu0 >= u0 && tu1 <= u1) {
    // this CTA computed the whole row tile: write bf16 directly
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int n = rbase + gid + (e >> 1) * 8;
        const int m = nt * 8 + 2 * tig + (e & 1);
        if (n < p.N && m < p.M) p.y[static_cast<size_t>(m) * p.N + n] = __float2bfloat16_rn(tot[nt][e]);
      }
    }
    return;
  }
  const int seg = static_cast<int>(T - u0 / p.G);
  float* pp = p.part + ((static_cast<size_t>(c) * p.maxseg + seg) * kRowTile + warp * 16) * Mp;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    *reinterpret_cast<float2*>(pp + gid * Mp + nt * 8 + 2 * tig) = make_float2(tot[nt][0], tot[nt][1]);
    *reinterpret_cast<float2*>(pp + (gid + 8) * Mp + nt * 8 + 2 * tig) = make_float2(tot[nt][2], tot[nt][3]);
  }
  __threadfence();
  __syncwarp();
  const int cf = cta_of_unit(tu0, p.U, p.P), cl = cta_of_unit(tu1 - 1, p.U, p.P);
  int last = 0;
  if (lane == 0) last = atomicAdd(&p.cnt[T * kConsumerWarps + warp], 1) == cl - cf;
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  __threadfence();
  for (int e = lane; e < 16 * Mp; e += 32) {
    const int row = e / Mp, m = e % Mp;
    float sum = 0.f;
    for (int cc = cf; cc <= cl; ++cc) {
      const int sg = static_cast<int>(T - unit_begin(cc, p.U, p.P) / p.G);
      sum += __ldcg(p.part + ((static_cast<size_t>(cc) * p.maxseg + sg) * kRowTile + warp * 16 + row) * Mp + m);
    }
    const int n = rbase + row;
    if (n < p.N && m < p.M) p.y[static_cast<size_t>(m) * p.N + n] = __float2bfloat16_rn(sum);
  }
  if (lane == 0) p.cnt[T * kConsumerWarps + warp] = 0;
}

template <int NT>
__global__ void __launch_bounds__(kThreads, 1) k_linear_rows(const RowsParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(p.stages) * p.stage_bytes);
  uint64_t* empty = full + p.stages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const long long u0 = unit_begin(c, p.U, p.P), u1 = unit_begin(c + 1, p.U, p.P);

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ---------------- producer warp
    const uint64_t pol = policy_evict_first();
    const uint32_t tx = kSbBytes + static_cast<uint32_t>(p.M) * 256u;
    long long i = 0;
    for (long long u = u0; u < u1; ++u, ++i) {
      const int s = static_cast<int>(i % p.stages);
      if (i >= p.stages) {
        const uint32_t par = static_cast<uint32_t>((i / p.stages) - 1) & 1u;
        if (!mbar_wait(&empty[s], par)) {
          if (lane == 0) set_status(p.status, FL_ERR_TIMEOUT, 1);
          // let the copies already issued land before the CTA retires
          for (long long j = (i > p.stages ? i - p.stages : 0); j < i; ++j)
            mbar_wait(&full[j % p.stages], static_cast<uint32_t>(j / p.stages) & 1u);
          return;
        }
      }
      uint8_t* st = smem + static_cast<size_t>(s) * p.stage_bytes;
      const int g = static_cast<int>(u % p.G);
      if (lane == 0) mbar_arrive_expect_tx(&full[s], tx);
      __syncwarp();
      if (lane == 0) bulk_g2s_hint(st, p.w + static_cast<size_t>(u) * kSbBytes, kSbBytes, &full[s], pol);
      for (int m = lane; m < p.M; m += 32)
        bulk_g2s(st + kSbBytes + m * kXRowStride, p.x + static_cast<size_t>(m) * p.K + g * kGroup, 256u,
                 &full[s]);
    }
    return;
  }

  // ---------------- consumer warps: rows warp*16 .. warp*16+15 of each tile
  const int gid = lane >> 2, tig = lane & 3;
  const int r0 = warp * 16 + gid;
  float tot[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) tot[nt][e] = 0.f;
  long long curT = -1;
  long long i = 0;
  for (long long u = u0; u < u1; ++u, ++i) {
    const long long T = u / p.G;
    if (T != curT) {
      if (curT >= 0) {
        flush_tile<NT>(p, curT, c, u0, u1, warp, lane, tot);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) tot[nt][e] = 0.f;
      }
      curT = T;
    }
    const int s = static_cast<int>(i % p.stages);
    if (!mbar_wait(&full[s], static_cast<uint32_t>(i / p.stages) & 1u)) {
      if (lane == 0) set_status(p.status, FL_ERR_TIMEOUT, 2);
      return;
    }
    const uint8_t* sb = smem + static_cast<size_t>(s) * p.stage_bytes;
    const uint8_t* sx = sb + kSbBytes;

    const __half* sc = reinterpret_cast<const __half*>(sb + kSbNib);
    const float s0 = __half2float(sc[r0]);
    const float s1 = __half2float(sc[r0 + 8]);
    const uint32_t zb0 = sb[kSbNib + kSbScale + (r0 >> 1)];
    const uint32_t zb1 = sb[kSbNib + kSbScale + (r0 >> 1) + 4];
    const uint32_t sh = (r0 & 1) * 4;
    const uint32_t zz0 = bf16_bias_pair((zb0 >> sh) & 15u);
    const uint32_t zz1 = bf16_bias_pair((zb1 >> sh) & 15u);
    const uint4 wa = *reinterpret_cast<const uint4*>(sb + r0 * 64 + tig * 16);
    const uint4 wb = *reinterpret_cast<const uint4*>(sb + (r0 + 8) * 64 + tig * 16);

    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;

#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t qa = (&wa.x)[j], qb = (&wb.x)[j];
      uint32_t a[4], b[4];
#pragma unroll
      for (int pi = 0; pi < 4; ++pi) {
        a[pi] = bf16x2_sub(nib_pair_bf16(qa, pi), zz0);
        b[pi] = bf16x2_sub(nib_pair_bf16(qb, pi), zz1);
      }
      uint4 xv[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int m = nt * 8 + gid;
        xv[nt] = m < p.M ? *reinterpret_cast<const uint4*>(sx + m * kXRowStride + (4 * j + tig) * 16)
                         : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          mma_bf16_16816(acc[nt], a[2 * h], b[2 * h], a[2 * h + 1], b[2 * h + 1], (&xv[nt].x)[2 * h],
                         (&xv[nt].x)[2 * h + 1]);
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      tot[nt][0] = fmaf(s0, acc[nt][0], tot[nt][0]);
      tot[nt][1] = fmaf(s0, acc[nt][1], tot[nt][1]);
      tot[nt][2] = fmaf(s1, acc[nt][2], tot[nt][2]);
      tot[nt][3] = fmaf(s1, acc[nt][3], tot[nt][3]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  if (curT >= 0) flush_tile<NT>(p, curT, c, u0, u1, warp, lane, tot);
}

// ------------------------------------------------------------------ plan
struct RowsPlan {
  int T, G, P, NT, maxseg, stages;
  long long U;
  uint32_t stage_bytes;
  size_t smem, cnt_off, part_off, ws_bytes;
};

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool make_rows_plan(int M, int N, int K, int sms, RowsPlan* pl) {
  if (M < 1 || M > kMaxTokens || N < 1 || K < kGroup || K % kGroup || sms < 1) return false;
  pl->T = (N + kRowTile - 1) / kRowTile;
  pl->G = K / kGroup;
  pl->U = static_cast<long long>(pl->T) * pl->G;
  pl->P = static_cast<int>(pl->U < sms ? pl->U : sms);
  pl->NT = (M + 7) / 8;
  int maxseg = 1;
  for (int c = 0; c < pl->P; ++c) {
    const long long a = unit_begin(c, pl->U, pl->P), b = unit_begin(c + 1, pl->U, pl->P);
    const int segs = static_cast<int>((b - 1) / pl->G - a / pl->G + 1);
    if (segs > maxseg) maxseg = segs;
  }
  pl->maxseg = maxseg;
  pl->stage_bytes = static_cast<uint32_t>(align_up(kSbBytes + static_cast<size_t>(M) * kXRowStride, 128));
  int stages = static_cast<int>((200u * 1024u) / pl->stage_bytes);
  pl->stages = stages > 12 ? 12 : stages;
  pl->smem = static_cast<size_t>(pl->stages) * pl->stage_bytes + 2 * pl->stages * sizeof(uint64_t);
  pl->cnt_off = kStatusBytes;
  pl->part_off = align_up(pl->cnt_off + static_cast<size_t>(pl->T) * kConsumerWarps * 4, 256);
  pl->ws_bytes = pl->part_off + static_cast<size_t>(pl->P) * pl->maxseg * kRowTile * (8 * pl->NT) * 4;
  return true;
}

template <int NT>
int launch_rows(const RowsPlan& pl, const RowsParams& prm, cudaStream_t s) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    if (cudaFuncSetAttribute(k_linear_rows<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) !=
        cudaSuccess)
      return FL_ERR_CUDA;
    attr_done[dev] = true;
  }
  k_linear_rows<NT><<<pl.P, kThreads, pl.smem, s>>>(prm);
  return cudaGetLastError() == cudaSuccess ? FL_OK : FL_ERR_CUDA;
}

}  // namespace

// Shared with the MoE and prefill launchers.
int fl_linear_rows_workspace(int M, int N, int K, size_t* out) {
  RowsPlan pl;
  if (!make_rows_plan(M, N, K, flh::sm_count(), &pl)) return FL_ERR_ARG;
  *out = pl.ws_bytes;
  return FL_OK;
}

int fl_linear_rows(const void* x, int M, int K, const void* w, int N, void* y, void* ws, size_t ws_bytes,
                   cudaStream_t stream) {
  RowsPlan pl;
  if (!make_rows_plan(M, N, K, flh::sm_count(), &pl)) return FL_ERR_ARG;
  if (ws_bytes < pl.ws_bytes) return FL_ERR_WORKSPACE;
  RowsParams prm;
  prm.w = static_cast<const uint8_t*>(w);
  prm.x = static_cast<const __nv_bfloat16*>(x);
  prm.y = static_cast<__nv_bfloat16*>(y);
  prm.status = static_cast<int32_t*>(ws);
  prm.cnt = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + pl.cnt_off);
  prm.part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + pl.part_off);
  prm.U = pl.U;
  prm.M = M;
  prm.K = K;
  prm.N = N;
  prm.T = pl.T;
  prm.G = pl.G;
  prm.P = pl.P;
  prm.maxseg = pl.maxseg;
  prm.stages = pl.stages;
  prm.stage_bytes = pl.stage_bytes;
  switch (pl.NT) {
    case 1: return launch_rows<1>(pl, prm, stream);
    case 2: return launch_rows<2>(pl, prm, stream);
    case 3: return launch_rows<3>(pl, prm, stream);
    default: return launch_rows<4>(pl, prm, stream);
  }
}

static bool linear_args_ok(const void* x, int M, int K, const void* w, int N, const void* y, const void* ws) {
  if (!x || !w || !y || !ws) return false;
  if (M < 1 || N < 1 || K < kGroup || K % kGroup) return false;
  return flh::aligned16(x) && flh::aligned16(w) && flh::aligned16(y) && flh::aligned16(ws);
}

extern "C" int fl_int4g_linear_workspace(int M, int N, int K, size_t* out) {
  if (!out || M < 1 || N < 1 || K < kGroup || K % kGroup) return FL_ERR_ARG;
  // M > 32 runs 32-token chunks of the decode kernel on one workspace
  return fl_linear_rows_workspace(M < kMaxTokens ? M : kMaxTokens, N, K, out);
}

extern "C" int fl_int4g_linear(const void* x, int M, int K, const void* w, int N, void* y, void* ws,
                               size_t ws_bytes, fl_stream_t stream) {
  if (!linear_args_ok(x, M, K, w, N, y, ws)) return FL_ERR_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  for (int m0 = 0; m0 < M; m0 += kMaxTokens) {
    const int mm = M - m0 < kMaxTokens ? M - m0 : kMaxTokens;
    const int rc = fl_linear_rows(static_cast<const __nv_bfloat16*>(x) + static_cast<size_t>(m0) * K, mm, K, w, N,
                                  static_cast<__nv_bfloat16*>(y) + static_cast<size_t>(m0) * N, ws, ws_bytes, s);
    if (rc != FL_OK) return rc;
  }
  return FL_OK;
}
