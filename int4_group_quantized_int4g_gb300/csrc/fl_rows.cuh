// Consumer-side building block shared by the decode linear and the grouped
// MoE kernels: one 128-row x 128-column int4g super-block (interleaved layout)
// times up to 8*NT token rows of x staged in shared memory, on mma.sync.
#pragma once

#include "fl_common.cuh"

namespace fl {

constexpr int kXRowStride = 320;  // 256 B of x per staged row + 64 B pad: conflict-free B-fragment loads

// One super-block through the tensor cores, for one consumer warp: acc[nt]
// (rows r0 and r0+8 of the tile, the lane's two tokens of token tile nt) =
// sum over the group of x * (q - z)   (FOLD: of x * (128 + q));
// s0/s1 receive the rows' fp16 scales, z0/z1 their zero points.
//
// The 16 bytes a lane reads per row hold logical columns 8*(4j+tig)+0..7
// (j = word), each word giving 4 bf16 pairs (128+q) by one LOP3.  MMA step
// (j, h) uses pairs 2h, 2h+1 of word j as A and x[m][8*(4j+tig)+4h .. +3]
// as B, which is the same permutation of K on both operands.
//
// FOLD: the (128+q) codes go to the MMA as they are; the caller removes
// (128+z) * sum_k x[m,k] per row and token, instead of a bf16 subtract per
// pair on the ALU.  One accumulator chain per super-block: the callers keep
// two super-blocks in flight per warp, which covers the MMA latency, and a
// second chain would cost a merge and its own zeroing per super-block.
// ZROW: lanes whose token m >= M read their B fragment from `xzero` (256
// zero bytes in shared memory) instead of zero-filling registers per step.
// xstride: bytes between the x rows of consecutive tokens in `sx` (a
// multiple of 16, and an odd multiple of 64 for conflict-free loads).
template <int NT, bool FOLD, bool ZROW = false>
__device__ __forceinline__ void unit_dot(const uint8_t* sb, const uint8_t* sx, int M, int r0, int gid, int tig,
                                         float (&acc)[NT][4], float& s0, float& s1, uint32_t& z0, uint32_t& z1,
                                         int ntiles = NT, const uint8_t* xzero = nullptr, int xstride = kXRowStride) {
  // chunk tig of rows r0 and r0+8 (both rotated by (r0/2)%4 in the layout)
  const int pos = ((tig + (r0 >> 1)) & 3) * 16;
  const uint4 wa = *reinterpret_cast<const uint4*>(sb + r0 * 64 + pos);
  const uint4 wb = *reinterpret_cast<const uint4*>(sb + (r0 + 8) * 64 + pos);
  const __half* sc = reinterpret_cast<const __half*>(sb + kSbNib);
  s0 = __half2float(sc[r0]);
  s1 = __half2float(sc[r0 + 8]);
  const uint32_t zsh = (r0 & 1) * 4;
  z0 = (sb[kSbNib + kSbScale + (r0 >> 1)] >> zsh) & 15u;
  z1 = (sb[kSbNib + kSbScale + (r0 >> 1) + 4] >> zsh) & 15u;
  const uint32_t zz0 = bf16_bias_pair(z0), zz1 = bf16_bias_pair(z1);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
  const uint8_t* xrow[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int m = nt * 8 + gid;
    xrow[nt] = (!ZROW || m < M) ? sx + m * xstride : xzero;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t qa = (&wa.x)[j], qb = (&wb.x)[j];
    uint32_t a[4], b[4];
#pragma unroll
    for (int pi = 0; pi < 4; ++pi) {
      a[pi] = nib_pair_bf16(qa, pi);
      b[pi] = nib_pair_bf16(qb, pi);
      if (!FOLD) {
        a[pi] = bf16x2_sub(a[pi], zz0);
        b[pi] = bf16x2_sub(b[pi], zz1);
      }
    }
    uint4 xv[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int m = nt * 8 + gid;
      xv[nt] = (ZROW || m < M) ? *reinterpret_cast<const uint4*>(xrow[nt] + (4 * j + tig) * 16)
                               : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      if (nt == 0 || nt < ntiles) {   // token tiles past the last token are all zero: skipped
        mma_bf16_16816(acc[nt], a[0], b[0], a[1], b[1], xv[nt].x, xv[nt].y);
        mma_bf16_16816(acc[nt], a[2], b[2], a[3], b[3], xv[nt].z, xv[nt].w);
      }
    }
  }
}

// Groups of 64: the same product with one accumulator chain per 64-column
// group.  Words j = 0, 1 of a lane's chunk hold logical columns 0..63 of the
// super-block (its even group, whose scale and zero point are in the
// super-block), words 2, 3 columns 64..127 (the odd group: `side`, the
// super-block's 320-byte side entry, 128 scales then 128 zero points).
// acc[0] / s.[0] / z.[0]: even group; acc[1] / s.[1] / z.[1]: odd group.
template <int NT, bool FOLD, bool ZROW = false>
__device__ __forceinline__ void unit_dot64(const uint8_t* sb, const uint8_t* side, const uint8_t* sx, int M, int r0,
                                           int gid, int tig, float (&acc)[2][NT][4], float (&s0)[2], float (&s1)[2],
                                           uint32_t (&z0)[2], uint32_t (&z1)[2], int ntiles = NT,
                                           const uint8_t* xzero = nullptr, int xstride = kXRowStride) {
  const int pos = ((tig + (r0 >> 1)) & 3) * 16;
  const uint4 wa = *reinterpret_cast<const uint4*>(sb + r0 * 64 + pos);
  const uint4 wb = *reinterpret_cast<const uint4*>(sb + (r0 + 8) * 64 + pos);
  const __half* sc = reinterpret_cast<const __half*>(sb + kSbNib);
  const __half* sd = reinterpret_cast<const __half*>(side);
  s0[0] = __half2float(sc[r0]);
  s1[0] = __half2float(sc[r0 + 8]);
  s0[1] = __half2float(sd[r0]);
  s1[1] = __half2float(sd[r0 + 8]);
  const uint32_t zsh = (r0 & 1) * 4;
  z0[0] = (sb[kSbNib + kSbScale + (r0 >> 1)] >> zsh) & 15u;
  z1[0] = (sb[kSbNib + kSbScale + (r0 >> 1) + 4] >> zsh) & 15u;
  z0[1] = (side[kSbScale + (r0 >> 1)] >> zsh) & 15u;
  z1[1] = (side[kSbScale + (r0 >> 1) + 4] >> zsh) & 15u;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[hh][nt][e] = 0.f;
  const uint8_t* xrow[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int m = nt * 8 + gid;
    xrow[nt] = (!ZROW || m < M) ? sx + m * xstride : xzero;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int hh = j >> 1;
    const uint32_t qa = (&wa.x)[j], qb = (&wb.x)[j];
    const uint32_t zz0 = bf16_bias_pair(hh ? z0[1] : z0[0]), zz1 = bf16_bias_pair(hh ? z1[1] : z1[0]);
    uint32_t a[4], b[4];
#pragma unroll
    for (int pi = 0; pi < 4; ++pi) {
      a[pi] = nib_pair_bf16(qa, pi);
      b[pi] = nib_pair_bf16(qb, pi);
      if (!FOLD) {
        a[pi] = bf16x2_sub(a[pi], zz0);
        b[pi] = bf16x2_sub(b[pi], zz1);
      }
    }
    uint4 xv[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int m = nt * 8 + gid;
      xv[nt] = (ZROW || m < M) ? *reinterpret_cast<const uint4*>(xrow[nt] + (4 * j + tig) * 16)
                               : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      if (nt == 0 || nt < ntiles) {
        mma_bf16_16816(acc[hh][nt], a[0], b[0], a[1], b[1], xv[nt].x, xv[nt].y);
        mma_bf16_16816(acc[hh][nt], a[2], b[2], a[3], b[3], xv[nt].z, xv[nt].w);
      }
    }
  }
}

}  // namespace fl
