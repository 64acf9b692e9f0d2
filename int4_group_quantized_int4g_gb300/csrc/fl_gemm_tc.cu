// a4: int4g prefill GEMM on the 5th-generation tensor cores (tcgen05).
//
// y[m, n] = sum_k x[m, k] * w'[n, k] for M tokens, the dense contraction of the
// int4g linear (FastLLM page, section 3.1: 4-bit codes dequantized inside the
// matmul; fastllm README section 2: --dtype int4g applies to every linear).
//
// Work unit = (tile, group): a tile is 128 weight rows n x BN tokens m of y^T,
// a group the 128 k of one super-block.  The grid is persistent (one CTA per
// SM); CTA c owns the contiguous units [c*U/P, (c+1)*U/P) in tile-major order
// (stream-K), so every SM gets the same number of MMAs whatever the tile count.
// A tile whose groups are spread over several CTAs is finished by the last of
// them to take its ticket, the fp32 partials summed in CTA order
// (deterministic).  Roles inside a CTA (tcgen05.mma kind::f16, bf16 in, fp32
// accumulate in tensor memory):
//   warp 0        x producer: per group, two TMA boxes of BN tokens x 64 k
//                 (128-byte swizzle) into a ring of half-group stages
//   warp 2        weight producer: the super-block (8512 B) by a 1-D bulk copy
//                 into its own ring, so the dequantization runs ahead of x
//   warp 1        allocates tensor memory; lane 0 issues 8 MMAs per group
//                 (K = 16 each) with A read from tensor memory
//   warps 4..11   dequantize the super-block into an A ring in tensor memory:
//                 each weight becomes the correctly rounded bf16 of s16*(q-z)
//   warps 12..19  epilogue: tcgen05.ld of the accumulator, bf16 store of y (or
//                 an fp32 partial and a ticket), then hand the accumulator
//                 back so the next tile's MMAs overlap the stores.
// The dequantized value bf16(s16*(q-z)) is computed exactly: s16 = s_hi +
// s_lo with s_hi = bf16(s16) and s_lo exact in bf16 (<= 3 bits), t =
// s_lo*(q-z) is exact, and fma(s_hi, q-z, t) rounds once.
#include <cuda.h>
#include <type_traits>
#include <cudaTypedefs.h>

#include "fl_common.cuh"

using namespace fl;

namespace {

constexpr int kPfThreads = 20 * 32;
constexpr int kPfDeq0 = 4;    // warps 4..11 dequantize
constexpr int kPfEpi0 = 12;   // warps 12..19 epilogue

template <int BN>
struct PfCfg {
  static constexpr int kBBox = BN * 64 * 2;                  // one x box: BN tokens x 64 k bf16
  static constexpr int kBStages = BN == 256 ? 5 : 8;         // half-group x stages
  static constexpr int kSStages = BN == 256 ? 4 : 8;         // super-block stages
  static constexpr int kARing = 4;                           // dequantized A tiles (64 TMEM columns each)
  static constexpr int kStgBytes = BN / 2 * kRowTile * 2;    // y staging: BN/2 tokens x 128 rows bf16
  static constexpr int kStgOff = kBStages * kBBox;           // 1 KB aligned
  static constexpr int kSOff = kStgOff + kStgBytes;
  static constexpr int kBarOff = kSOff + kSStages * kSbBytes;
  static constexpr int kNumBars = 2 * kBStages + 2 * kSStages + 2 * kARing + 2;
  static constexpr int kSmem = kBarOff + kNumBars * 8 + 16 + 1024 /*align slack*/;
  static constexpr uint32_t kTmemCols = 512;                 // accumulator [0, BN), A ring [BN, BN + 256)
  static_assert(BN + 64 * kARing <= 512, "tensor memory");
  static_assert(kSmem <= 232448, "shared memory");
};

struct PfParams {
  const uint8_t* w;    // interleaved weights, first row tile of this launch
  const uint8_t* side; // groups of 64: side entries of the same super-blocks (else null)
  __nv_bfloat16* y;    // y + n0 (first row of this launch)
  float* part;         // 2P partial slots of 128 x BN floats, [column][row]
  int32_t* cnt;        // ticket counters [tile][8]
  int32_t* status;
  int M, N, ldy, G, mtiles, U, P;
  int tma_y;           // y written by TMA stores through a staging tile (row stride a multiple of 16 B)
};

// ------------------------------------------------------------ tcgen05 helpers
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 32 consecutive fp32 columns of the calling warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Issue a load of 16 consecutive fp32 columns (no wait).
__device__ __forceinline__ void tmem_ld16_issue(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// Wait for this thread's outstanding tensor-memory loads; the registers of
// `r` are tied to the wait so that no use of them is scheduled before it.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}
// Read NC chunks of 16 columns starting at taddr, keeping the next chunk's
// load in flight while the current one is consumed; `release` runs as soon as
// the last load has completed (the accumulator may then be overwritten).
// 4-byte asynchronous copy global -> shared (generic proxy), and the wait for
// all of this thread's copies.
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

template <int NC, typename Rel, typename Use>
__device__ __forceinline__ void pf_drain(uint32_t taddr, Rel&& release, Use&& use) {
  static_assert(NC % 2 == 0, "chunks come in pairs");
  uint32_t ra[16], rb[16];
  tmem_ld16_issue(taddr, ra);
  tmem_ld_wait(ra);
#pragma unroll
  for (int k = 0; k < NC; k += 2) {
    tmem_ld16_issue(taddr + 16 * (k + 1), rb);
    {
      float v[16];
#pragma unroll
      for (int t = 0; t < 16; ++t) v[t] = __uint_as_float(ra[t]);
      use(k, v);
    }
    tmem_ld_wait(rb);
    if (k + 2 < NC)
      tmem_ld16_issue(taddr + 16 * (k + 2), ra);
    else
      release();
    {
      float v[16];
#pragma unroll
      for (int t = 0; t < 16; ++t) v[t] = __uint_as_float(rb[t]);
      use(k + 1, v);
    }
    if (k + 2 < NC) tmem_ld_wait(ra);
  }
}

// 32 consecutive 32-bit columns of the calling warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// MMA with the A operand in tensor memory (M = 128 rows = lanes, K packed two
// 16-bit elements per 32-bit column), B in shared memory.
__device__ __forceinline__ void umma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One thread of the (converged) warp, chosen by elect.sync.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "elect.sync _|P, 0xffffffff;\n\t"
      "selp.b32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// TMA 2-D tile load global -> shared, completion counted on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// TMA 2-D tile store shared -> global (bulk group); rows/columns outside the
// tensor are not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map), "r"(c0),
               "r"(c1), "r"(smem_u32(src))
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 B apart (SBO), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1u) << 16;                  // LBO (unused for swizzled K-major)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;          // SBO
  d |= static_cast<uint64_t>(1u) << 46;                  // version
  d |= static_cast<uint64_t>(2u) << 61;                  // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major.
template <int BN>
__device__ __forceinline__ uint32_t idesc_bf16() {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
         (static_cast<uint32_t>(128 >> 4) << 24);
}

// The same with N chosen at run time (a multiple of 16, 16..256).
__device__ __forceinline__ uint32_t idesc_bf16_n(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(128 >> 4) << 24);
}

// CTA c of P owns units [unit_begin(c), unit_begin(c + 1)) of U; cta_of_unit
// inverts it.
__host__ __device__ __forceinline__ int td_unit_begin(int c, int U, int P) {
  return static_cast<int>(static_cast<long long>(c) * U / P);
}
__host__ __device__ __forceinline__ int td_cta_of_unit(int u, int U, int P) {
  return static_cast<int>((static_cast<long long>(u + 1) * P - 1) / U);
}

// bf16x2 helpers with a single rounding
__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b) {
  __nv_bfloat162 r = __hmul2(*reinterpret_cast<__nv_bfloat162*>(&a), *reinterpret_cast<__nv_bfloat162*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t bfma2(uint32_t a, uint32_t b, uint32_t c) {
  __nv_bfloat162 r = __hfma2(*reinterpret_cast<__nv_bfloat162*>(&a), *reinterpret_cast<__nv_bfloat162*>(&b),
                             *reinterpret_cast<__nv_bfloat162*>(&c));
  return *reinterpret_cast<uint32_t*>(&r);
}

// 16 columns (tokens m0..m0+15) of one accumulator row n per lane -> bf16 y.
// With an even row stride, lanes 2i and 2i+1 (rows n, n+1) swap halves so
// that each lane writes one aligned pair of adjacent rows.
__device__ __forceinline__ void pf_store_cols(const PfParams& p, int n, int m0, const float (&v)[16], int lane) {
  if ((p.ldy & 1) == 0) {
    const bool odd = lane & 1;
    const int ne = n & ~1;
#pragma unroll
    for (int t = 0; t < 16; t += 2) {
      const float send = odd ? v[t] : v[t + 1];
      const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
      const int m = m0 + t + (odd ? 1 : 0);
      const float lo = odd ? recv : v[t];
      const float hi = odd ? v[t + 1] : recv;
      if (m < p.M && ne < p.N) {
        __nv_bfloat16* dst = p.y + static_cast<size_t>(m) * p.ldy + ne;
        const __nv_bfloat162 pr = __floats2bfloat162_rn(lo, hi);
        if (ne + 1 < p.N)
          *reinterpret_cast<__nv_bfloat162*>(dst) = pr;
        else
          *dst = pr.x;
      }
    }
  } else if (n < p.N) {
#pragma unroll
    for (int t = 0; t < 16; ++t)
      if (m0 + t < p.M) p.y[static_cast<size_t>(m0 + t) * p.ldy + n] = __float2bfloat16_rn(v[t]);
  }
}

// Order in which a CTA takes its units [u0, u1): the head tile it shares
// with CTA c-1, its whole tiles, then the tail tile it shares with CTA c+1.
// CTA c+1 takes that tile first (as its head), so the last arriver of a
// split tile meets it as its own last tile: with its MMAs over and its x
// stages idle, it sums the tile in place and stores y through the staging
// tile, instead of a ticketed sum from L2 in the middle of its work (which
// held up the next tile's epilogue: M=512 K=4096 N=11008 took 50.8 us this
// way against 41.3 us).  Three contiguous segments of units.
struct PfSeq {
  int ha, hb, ta, tb;   // head [ha, hb), whole tiles [hb, ta), tail [ta, tb)
  __device__ static PfSeq make(int u0, int u1, int G) {
    PfSeq q;
    q.ha = u0;
    q.hb = u0 % G ? min(u1, (u0 / G + 1) * G) : u0;
    q.tb = u1;
    q.ta = u1 % G ? max(u1 / G * G, q.hb) : u1;
    return q;
  }
  __device__ int nh() const { return hb - ha; }
  __device__ int nw() const { return ta - hb; }
  __device__ int at(int i) const {
    if (i < nh()) return ha + i;
    if (i < nh() + nw()) return hb + (i - nh());
    return ta + (i - nh() - nw());
  }
  __device__ int seg_end(int i, int n) const { return i < nh() ? nh() : i < nh() + nw() ? nh() + nw() : n; }
};

template <int BN>
__global__ void __launch_bounds__(kPfThreads, 1) k_gemm_tc(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap ymap,
                                                    const PfParams p) {
  using C = PfCfg<BN>;
  constexpr int RA = C::kARing, NBS = C::kBStages, NSS = C::kSStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bfull = reinterpret_cast<uint64_t*>(smem + C::kBarOff);   // x stage landed
  uint64_t* bempty = bfull + NBS;                                     // MMAs reading the x stage done
  uint64_t* sfull = bempty + NBS;                                     // super-block landed
  uint64_t* sempty = sfull + NSS;                                     // super-block read by the 8 dequant warps
  uint64_t* afull = sempty + NSS;                                     // A slot written (8 dequant warps)
  uint64_t* aempty = afull + RA;                                      // MMAs reading the A slot done
  uint64_t* dfull = aempty + RA;                                      // accumulator of a tile final
  uint64_t* dempty = dfull + 1;                                       // accumulator read out (8 epilogue warps)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(dempty + 1);
  int* epi_abort = reinterpret_cast<int*>(tmem_slot + 1);
  int* done_flag = epi_abort + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const int u0 = td_unit_begin(c, p.U, p.P), nu = td_unit_begin(c + 1, p.U, p.P) - u0;
  const PfSeq sq = PfSeq::make(u0, u0 + nu, p.G);

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBS; ++i) {
      mbar_init(&bfull[i], 1);
      mbar_init(&bempty[i], 1);
    }
    for (int i = 0; i < NSS; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&sempty[i], 8);
    }
    for (int i = 0; i < RA; ++i) {
      mbar_init(&afull[i], 8);
      mbar_init(&aempty[i], 1);
    }
    mbar_init(dfull, 1);
    mbar_init(dempty, 8);
    *epi_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  cta_sync();
  tc_fence_after();
  const uint32_t tmem_d = *tmem_slot;          // accumulator: columns [0, BN)
  const uint32_t tmem_a = tmem_d + BN;         // A ring: columns [BN, BN + 64 * RA)
  pdl_launch_dependents();

  if (warp == 0) {
    // ---------------- x producer
    if (lane == 0) {
      pdl_wait();
      int j = 0;
      bool ok = true;
      for (int i = 0; i < nu && ok; ++i) {
        const int u = sq.at(i), T = u / p.G, g = u - T * p.G, mt = T % p.mtiles;
        for (int h = 0; h < 2; ++h, ++j) {
          const int b = j % NBS;
          if (j >= NBS && !mbar_wait(&bempty[b], static_cast<uint32_t>(j / NBS - 1) & 1u)) {
            set_status(p.status, FL_ERR_TIMEOUT, 31);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bfull[b], C::kBBox);
          tma_load_2d(smem + b * C::kBBox, &xmap, g * kGroup + 64 * h, mt * BN, &bfull[b]);
        }
      }
      if (!ok)   // let the copies in flight land before the CTA can exit
        for (int jj = j > NBS ? j - NBS : 0; jj < j; ++jj) mbar_wait(&bfull[jj % NBS], static_cast<uint32_t>(jj / NBS) & 1u);
    }
  } else if (warp == 2) {
    // ---------------- weight producer
    if (lane == 0) {
      pdl_wait();
      const uint64_t pol = policy_evict_first();
      int i = 0;
      bool ok = true;
      for (; i < nu; ++i) {
        const int u = sq.at(i), T = u / p.G, g = u - T * p.G, nt = T / p.mtiles;
        const int sI = i % NSS;
        if (i >= NSS && !mbar_wait(&sempty[sI], static_cast<uint32_t>(i / NSS - 1) & 1u)) {
          set_status(p.status, FL_ERR_TIMEOUT, 32);
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&sfull[sI], kSbBytes);
        bulk_g2s_hint(smem + C::kSOff + sI * kSbBytes, p.w + (static_cast<size_t>(nt) * p.G + g) * kSbBytes, kSbBytes,
                      &sfull[sI], pol);
      }
      if (!ok)
        for (int ii = i > NSS ? i - NSS : 0; ii < i; ++ii) mbar_wait(&sfull[ii % NSS], static_cast<uint32_t>(ii / NSS) & 1u);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: A from tensor memory, B (x) from shared memory.
    // The tensor pipe queues only a few MMAs, so the per-unit work of this
    // thread is kept small: counters instead of divisions, and one barrier
    // probe per unit (afull also certifies the unit's x stages: the dequant
    // warps wait for them before arriving).
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16<BN>();
      int jt = 0, a = 0, b = 0;
      uint32_t aph = 0;
      bool ok = true;
      for (int seg = 0; seg < 3 && ok; ++seg) {
        const int ub = seg == 0 ? sq.ha : seg == 1 ? sq.hb : sq.ta;
        const int ue = seg == 0 ? sq.hb : seg == 1 ? sq.ta : sq.tb;
        int g = ub % p.G;
        for (int u = ub; u < ue; ++u) {
          const bool first = g == 0 || u == ub, last = g == p.G - 1 || u == ue - 1;
          if ((first && jt > 0 && !mbar_wait(dempty, static_cast<uint32_t>(jt - 1) & 1u)) || !mbar_wait(&afull[a], aph)) {
            set_status(p.status, FL_ERR_TIMEOUT, 33);
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t b0 = smem_u32(smem + b * C::kBBox);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16_ta(tmem_d, tmem_a + a * 64 + h * 32 + kk * 8, sw128_desc(b0 + kk * 32), idesc,
                           (!first || h != 0 || kk != 0) ? 1u : 0u);
            umma_commit(&bempty[b]);
            if (++b == NBS) b = 0;
          }
          umma_commit(&aempty[a]);
          if (++a == RA) a = 0, aph ^= 1u;
          if (last) {
            umma_commit(dfull);
            ++jt;
          }
          if (++g == p.G) g = 0;
        }
      }
    }
  } else if (warp >= kPfDeq0 && warp < kPfEpi0) {
    // ---------------- dequant: thread = (weight row r = TMEM lane, K half h)
    const int q = warp & 3, h = (warp - kPfDeq0) >> 2;
    const int r = q * 32 + lane;
    const uint32_t trow = static_cast<uint32_t>(q * 32) << 16;
    for (int i = 0; i < nu; ++i) {
      const int sI = i % NSS, a = i % RA;
      // groups of 64: the upper K half takes the odd group's scale and zero
      // point from the side entry (read before the wait, to overlap it)
      const bool odd = p.side != nullptr && h == 1;
      float sf = 0.f;
      uint32_t z = 0;
      if (odd) {
        const int u = sq.at(i), T = u / p.G, g = u - T * p.G, nt = T / p.mtiles;
        const uint8_t* sd = p.side + (static_cast<size_t>(nt) * p.G + g) * kSbSide;
        sf = __half2float(__ldg(reinterpret_cast<const __half*>(sd) + r));
        z = (__ldg(sd + kSbScale + (r >> 1)) >> ((r & 1) * 4)) & 15u;
      }
      if (!mbar_wait(&sfull[sI], static_cast<uint32_t>(i / NSS) & 1u)) {
        set_status(p.status, FL_ERR_TIMEOUT, 35);
        break;
      }
      const uint8_t* sb = smem + C::kSOff + sI * kSbBytes;
      if (!odd) {
        sf = __half2float(reinterpret_cast<const __half*>(sb + kSbNib)[r]);
        z = (sb[kSbNib + kSbScale + (r >> 1)] >> ((r & 1) * 4)) & 15u;
      }
      uint4 cv[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) cv[t] = *reinterpret_cast<const uint4*>(sb + r * 64 + ((t + (r >> 1)) & 3) * 16);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sempty[sI]);
      const __nv_bfloat16 shi = __float2bfloat16_rn(sf);
      const __nv_bfloat16 slo = __float2bfloat16_rn(sf - __bfloat162float(shi));   // exact remainder
      const uint32_t hi2 = static_cast<uint32_t>(__bfloat16_as_ushort(shi)) * 0x00010001u;
      const uint32_t lo2 = static_cast<uint32_t>(__bfloat16_as_ushort(slo)) * 0x00010001u;
      const uint32_t zz = bf16_bias_pair(z);
      uint32_t o[32];
      auto unpack = [&](auto H) {
        constexpr int hh = decltype(H)::value;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int wl = 8 * hh + t;
          const uint32_t word = (&cv[wl & 3].x)[wl >> 2];
#pragma unroll
          for (int pi = 0; pi < 4; ++pi) {
            const uint32_t qz = bf16x2_sub(nib_pair_bf16(word, pi), zz);
            o[4 * t + pi] = bfma2(hi2, qz, bmul2(lo2, qz));
          }
        }
      };
      if (h == 0)
        unpack(std::integral_constant<int, 0>());
      else
        unpack(std::integral_constant<int, 1>());
      if (i >= RA && !mbar_wait(&aempty[a], static_cast<uint32_t>(i / RA - 1) & 1u)) {
        set_status(p.status, FL_ERR_TIMEOUT, 36);
        break;
      }
      tc_fence_after();
      tmem_st32(tmem_a + trow + a * 64 + h * 32, o);
      tmem_wait_st();
      // the unit's two x stages must have landed before afull is signalled
      if (!mbar_wait(&bfull[(2 * i) % NBS], static_cast<uint32_t>((2 * i) / NBS) & 1u) ||
          !mbar_wait(&bfull[(2 * i + 1) % NBS], static_cast<uint32_t>((2 * i + 1) / NBS) & 1u)) {
        set_status(p.status, FL_ERR_TIMEOUT, 34);
        break;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&afull[a]);
    }
  } else if (warp >= kPfEpi0) {
    // ---------------- epilogue: rows q*32+lane, one half of the tile's tokens
    const int e = warp - kPfEpi0, q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t tcol = tmem_d + (static_cast<uint32_t>(q * 32) << 16) + (e >> 2) * (BN / 2);
    const int col0 = (e >> 2) * (BN / 2);
    auto release_d = [&]() {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dempty);
    };
    int jt = 0;
    for (int i = 0; i < nu; ++jt) {
      const int u = sq.at(i), T = u / p.G, g = u - T * p.G;
      const int len = min(p.G - g, sq.seg_end(i, nu) - i);
      const bool whole = g == 0 && len == p.G, head = T == u0 / p.G;
      i += len;
      const bool last_of_cta = i == nu;
      // all epilogue warps take the same exit decision (they share named barriers)
      if (!mbar_wait(dfull, static_cast<uint32_t>(jt) & 1u)) *epi_abort = 1;
      named_bar(1, 256);
      if (*reinterpret_cast<volatile int*>(epi_abort)) {
        set_status(p.status, FL_ERR_TIMEOUT, 37);
        break;
      }
      tc_fence_after();
      const int nt = T / p.mtiles, mt = T % p.mtiles;
      const int n = nt * kRowTile + r, m0 = mt * BN + col0;
      if (whole && p.tma_y) {
        // two rounds of BN/2 tokens through the staging tile: TMEM -> bf16 in
        // shared memory -> one TMA store of 128 rows x BN/2 tokens
        __nv_bfloat16* stg = reinterpret_cast<__nv_bfloat16*>(smem + C::kStgOff);
#pragma unroll 1
        for (int rho = 0; rho < 2; ++rho) {
          const int lt0 = (e >> 2) * (BN / 4);
          pf_drain<BN / 64>(
              tmem_d + (static_cast<uint32_t>(q * 32) << 16) + rho * (BN / 2) + lt0,
              [&]() {
                if (rho == 1) release_d();
              },
              [&](int k, const float (&v)[16]) {
                __nv_bfloat16* dst = stg + static_cast<size_t>(lt0 + 16 * k) * kRowTile + r;
#pragma unroll
                for (int t = 0; t < 16; ++t) dst[t * kRowTile] = __float2bfloat16_rn(v[t]);
              });
          fence_proxy_async();
          named_bar(1, 256);
          if (e == 0 && lane == 0) {
            tma_store_2d(&ymap, stg, nt * kRowTile, mt * BN + rho * (BN / 2));
            bulk_commit();
            bulk_wait_read0();   // the staging tile has been read
          }
          named_bar(1, 256);
        }
        continue;
      }
      if (whole) {
        pf_drain<BN / 32>(tcol, release_d, [&](int k, const float (&v)[16]) { pf_store_cols(p, n, m0 + 16 * k, v, lane); });
        continue;
      }
      // partial tile: contributors cf..cl, summed in CTA order by the last one
      const int cf = td_cta_of_unit(T * p.G, p.U, p.P), cl = td_cta_of_unit((T + 1) * p.G - 1, p.U, p.P);
      int32_t* cnt = p.cnt + T * 8 + e;
      auto slot_of = [&](int cc) {
        return p.part + static_cast<size_t>(2 * cc + (td_unit_begin(cc, p.U, p.P) / p.G == T ? 0 : 1)) * kRowTile * BN;
      };
      int done = 0;
      if (last_of_cta) {
        // The accumulator is not needed afterwards: combine in place if all
        // other sharers are in, one decision for the 8 epilogue warps (every
        // warp's counter full), shared through the named barrier, which also
        // orders every thread's reads after the acquiring loads.
        if (e == 0) {   // lanes 0..7 acquire one warp's counter each, in parallel
          const bool in = lane >= 8 || ld_acquire_gpu(p.cnt + T * 8 + lane) == cl - cf;
          const bool all = __all_sync(0xffffffffu, in);
          if (lane == 0) *done_flag = all ? 1 : 0;
        }
        named_bar(1, 256);
        done = *reinterpret_cast<volatile int*>(done_flag);
      }
      if (done && p.tma_y && cl - cf == 1) {
        // The CTA's MMAs are over, so its x stages hold nothing: each thread
        // copies its elements of the other sharer's partial into them (all
        // copies in flight at once), then the tile goes out like a whole one:
        // accumulator + partial in CTA order, bf16 through the staging tile,
        // one TMA store per half.
        constexpr int kWarpFloats = (BN / 2) * 32;   // a warp's rows x columns of one slot
        static_assert(8 * kWarpFloats * 4 <= NBS * C::kBBox, "partial staging");
        float* stage = reinterpret_cast<float*>(smem);
        const int co = cf == c ? cl : cf;
        const bool other_first = co < c;
        {
          fence_proxy_async();   // the stages were last written by TMA
          const float* src = slot_of(co) + static_cast<size_t>(col0) * kRowTile + r;
          float* dst = stage + static_cast<size_t>(e) * kWarpFloats + lane;
#pragma unroll 8
          for (int j = 0; j < BN / 2; ++j) cp_async4(dst + j * 32, src + j * kRowTile);
          cp_async_wait_all();
        }
        named_bar(1, 256);   // every warp's part of the partial is in
        __nv_bfloat16* stg = reinterpret_cast<__nv_bfloat16*>(smem + C::kStgOff);
#pragma unroll 1
        for (int rho = 0; rho < 2; ++rho) {
          const int lt0 = (e >> 2) * (BN / 4);
          const float* sp = stage + static_cast<size_t>(q + 4 * rho) * kWarpFloats + lane;
          pf_drain<BN / 64>(
              tmem_d + (static_cast<uint32_t>(q * 32) << 16) + rho * (BN / 2) + lt0,
              [&]() {
                if (rho == 1) release_d();
              },
              [&](int k, const float (&v)[16]) {
                __nv_bfloat16* dst = stg + static_cast<size_t>(lt0 + 16 * k) * kRowTile + r;
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                  const float o = sp[(lt0 + 16 * k + t) * 32];
                  const float sum = other_first ? (0.f + o) + v[t] : (0.f + v[t]) + o;   // CTA order
                  dst[t * kRowTile] = __float2bfloat16_rn(sum);
                }
              });
          fence_proxy_async();
          named_bar(1, 256);
          if (e == 0 && lane == 0) {
            tma_store_2d(&ymap, stg, nt * kRowTile, mt * BN + rho * (BN / 2));
            bulk_commit();
            bulk_wait_read0();   // the staging tile has been read
          }
          named_bar(1, 256);
        }
        __syncwarp();
        if (lane == 0) *cnt = 0;
        continue;
      }
      if (done) {
        pf_drain<BN / 32>(tcol, release_d, [&](int k, const float (&v)[16]) {
          float acc[16];
#pragma unroll
          for (int t = 0; t < 16; ++t) acc[t] = 0.f;
          for (int cc = cf; cc <= cl; ++cc) {   // CTA order: deterministic
            if (cc == c) {
#pragma unroll
              for (int t = 0; t < 16; ++t) acc[t] += v[t];
            } else {
              const float* src = slot_of(cc) + static_cast<size_t>(col0 + 16 * k) * kRowTile + r;
#pragma unroll
              for (int t = 0; t < 16; ++t) acc[t] += __ldcg(src + t * kRowTile);
            }
          }
          pf_store_cols(p, n, m0 + 16 * k, acc, lane);
        });
        __syncwarp();
        if (lane == 0) *cnt = 0;
        continue;
      }
      float* slot = p.part + static_cast<size_t>(2 * c + (head ? 0 : 1)) * kRowTile * BN;
      pf_drain<BN / 32>(tcol, release_d, [&](int k, const float (&v)[16]) {
        float* dst = slot + static_cast<size_t>(col0 + 16 * k) * kRowTile + r;
#pragma unroll
        for (int t = 0; t < 16; ++t) __stcg(dst + t * kRowTile, v[t]);
      });
      int lastw = 0;
      if (lane == 0) {
        fence_acq_rel_gpu();
        lastw = atomicAdd(cnt, 1) == cl - cf;
        if (lastw) fence_acq_rel_gpu();
      }
      lastw = __shfl_sync(0xffffffffu, lastw, 0);
      if (!lastw) continue;
      __syncwarp();
#pragma unroll 1
      for (int k = 0; k < BN / 32; ++k) {
        float acc[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) acc[t] = 0.f;
        for (int cc = cf; cc <= cl; ++cc) {   // CTA order: deterministic
          const float* src = slot_of(cc) + static_cast<size_t>(col0 + 16 * k) * kRowTile + r;
#pragma unroll
          for (int t = 0; t < 16; ++t) acc[t] += __ldcg(src + t * kRowTile);
        }
        pf_store_cols(p, n, m0 + 16 * k, acc, lane);
      }
      __syncwarp();
      if (lane == 0) *cnt = 0;
    }
    if (e == 0 && lane == 0) bulk_wait0();   // y stores complete before the CTA exits
  }
  tc_fence_before();
  cta_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_d, C::kTmemCols);
  }
}

// ------------------------------------------------------------------ host
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// Prefill workspace: status block, ticket counters at kTicketOff, 2P
// partial slots of 128 x BN floats at kScratchOff.
int pf_bn(int M) { return M > 128 ? 256 : 128; }

size_t pf_workspace(int M) {
  const size_t P = static_cast<size_t>(flh::sm_count());
  return kScratchOff + 2 * P * kRowTile * pf_bn(M) * 4;
}

template <int BN>
int launch_tc(const void* x, int M, int K, const void* w, int N, void* y, void* ws, cudaStream_t s,
              const uint8_t* side) {
  using C = PfCfg<BN>;
  auto enc = encode_fn();
  if (!enc) return FL_ERR_CUDA;
  CUtensorMap map;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(BN)};
  const cuuint32_t estr[2] = {1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return FL_ERR_CUDA;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    if (cudaFuncSetAttribute(k_gemm_tc<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) != cudaSuccess)
      return FL_ERR_CUDA;
    attr_done[dev] = true;
  }
  // y through TMA stores when its row stride is a multiple of 16 bytes
  const int tma_y = N % 8 == 0 ? 1 : 0;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  const int G = K / kGroup, mtiles = (M + BN - 1) / BN, ntiles = (N + kRowTile - 1) / kRowTile;
  const int sms = flh::sm_count();
  // the ticket counters cover kTicketTiles tiles: larger problems run as
  // several launches over row-tile ranges, serialized on the stream
  const int nt_chunk = kTicketTiles / mtiles;
  if (nt_chunk < 1) return FL_ERR_UNSUPPORTED;
  for (int nt0 = 0; nt0 < ntiles; nt0 += nt_chunk) {
    const int nts = ntiles - nt0 < nt_chunk ? ntiles - nt0 : nt_chunk;
    PfParams p;
    p.w = static_cast<const uint8_t*>(w) + static_cast<size_t>(nt0) * G * kSbBytes;
    p.side = side ? side + static_cast<size_t>(nt0) * G * kSbSide : nullptr;
    p.y = static_cast<__nv_bfloat16*>(y) + static_cast<size_t>(nt0) * kRowTile;
    p.part = reinterpret_cast<float*>(wsb + kScratchOff);
    p.cnt = reinterpret_cast<int32_t*>(wsb + kTicketOff);
    p.status = reinterpret_cast<int32_t*>(wsb);
    p.M = M;
    p.N = N - nt0 * kRowTile < nts * kRowTile ? N - nt0 * kRowTile : nts * kRowTile;
    p.ldy = N;
    p.G = G;
    p.mtiles = mtiles;
    const long long U = static_cast<long long>(nts) * mtiles * G;
    if (U > 0x7fffffffLL / (sms + 1)) return FL_ERR_UNSUPPORTED;
    p.U = static_cast<int>(U);
    p.P = p.U < sms ? p.U : sms;
    // Few tiles: every tile split into s equal parts (s = SMs / tiles >= 2),
    // so that no tile has more than s sharers, and with s = 2 each tile's
    // last arriver meets exactly one partial (the in-place combine).  Some SMs
    // idle; contiguous ranges over all SMs would give most tiles a third
    // sharer that ends late too (M=512, K=11008: 58.8 against 50.6 us).
    {
      const int tiles = nts * mtiles, sp = sms / tiles;
      if (sp >= 2) p.P = tiles * (sp < G ? sp : G);
    }
    p.tma_y = tma_y;
    CUtensorMap ymap;
    memset(&ymap, 0, sizeof(ymap));
    if (tma_y) {
      const cuuint64_t ydims[2] = {static_cast<cuuint64_t>(p.N), static_cast<cuuint64_t>(M)};
      const cuuint64_t ystrides[1] = {static_cast<cuuint64_t>(N) * 2};
      const cuuint32_t ybox[2] = {static_cast<cuuint32_t>(kRowTile), static_cast<cuuint32_t>(BN / 2)};
      if (enc(&ymap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.y, ydims, ystrides, ybox, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return FL_ERR_CUDA;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.P));
    cfg.blockDim = dim3(kPfThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = nt0 == 0 ? 1 : 0;   // chunks after the first reuse the counters: no overlap
    if (cudaLaunchKernelEx(&cfg, k_gemm_tc<BN>, map, ymap, p) != cudaSuccess) return FL_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? FL_OK : FL_ERR_CUDA;
}

// ======================================================================
// Decode (8 < M <= 32) on tcgen05: the stream of super-blocks of the decode
// linear, split over K across the SMs like the mma.sync kernel (CTA c owns
// units [c*U/P, (c+1)*U/P) in layout order, a row tile split across CTAs is
// finished by the last CTA to take its ticket, partials summed in CTA order),
// but the dot products run on tcgen05.  One CTA per SM (a kernel that
// allocates tensor memory gets one CTA per SM), so the work runs in three
// independent chains: super-block i goes to MMA issuer i % 3 and dequant group
// i % 3.
//   warp 0        super-block producer (1-D bulk copies)
//   warp 1        x producer: the x tile (NB token rows x 128 k, rows past M
//                 read as zero) by TMA
//   warps 2..4    MMA issuers: 8 MMAs per super-block (M = 128 rows, N = NB
//                 tokens, K = 16), each issuer into its own accumulator per
//                 row tile (two tile buffers)
//   warps 5..16   dequant, three groups of four warps (one per tensor-memory
//                 quadrant): the correctly rounded bf16(s16 * (q - z)) into
//                 the group's A slot, so the accumulators hold scaled sums
//   warps 17..20  epilogue, once per row tile: the issuers' accumulators added
//                 in issuer order, then y written or the split tile handed off
// The dequant is bound by the ALU (five instructions per pair of weights, three
// of them on the bf16 pipe); one issuing thread reaches only about one
// tcgen05.mma per 65 cycles.  Both are why the work runs in three chains.
struct TdParams {
  const uint8_t* w;
  __nv_bfloat16* y;
  float* part;
  int32_t* cnt;
  int32_t* status;
  int U, M, K, N, T, G, P;
};

template <int NB>
struct TdCfg {
  static constexpr int kXBytes = NB * 256;                        // NB rows x 128 k bf16 (two swizzled halves)
  static constexpr int kChains = 3;                               // super-block i goes to issuer and dequant group i % 3
  // ring sizes are multiples of kChains: every slot, and so every barrier,
  // then has exactly one waiter chain (a parity wait is only sound when its
  // waiter cannot be two phases behind)
  static constexpr int kSbRing = 12;                              // super-blocks in flight per CTA
  static constexpr int kARing = 3;                                // dequantized A tiles (tensor memory)
  static constexpr int kXRing = 6;                                // x tiles (one per super-block's group)
  static constexpr int kSmem = kXRing * kXBytes + kSbRing * kSbBytes + 1024 /*align slack*/ + 1024 /*barriers*/;
  static_assert(kSbRing % kChains == 0 && kARing % kChains == 0 && kXRing % kChains == 0, "one chain per slot");
  static_assert((2 * kSbRing + 2 * kXRing + 2 * kARing + 4 * kChains) * 8 + 8 <= 1024, "barrier area");
  static_assert(kSmem <= 232448, "shared memory");
  static constexpr uint32_t kDCol = kARing * 64;                  // accumulators [issuer][tile buffer] of NB columns
  static_assert(kDCol + 2 * kChains * NB + 32 - NB <= 512, "tensor memory");
  static constexpr uint32_t kTmemCols = 512;
};

constexpr int kTdThreads = 21 * 32;
constexpr int kTdIss0 = 2, kTdDeq0 = 5, kTdEpi0 = 17;


// Final sums of row tile T for this epilogue thread's row: write them or hand
// them off (returns true when a ticket is owed).
template <int NB>
__device__ __forceinline__ bool td_store(const TdParams& p, int T, int c, int u0, int u1, int r, const float* tot) {
  const int n = T * kRowTile + r;
  if (T * p.G >= u0 && (T + 1) * p.G <= u1) {
    if (n < p.N) {
#pragma unroll
      for (int m = 0; m < NB; ++m)
        if (m < p.M) p.y[static_cast<size_t>(m) * p.N + n] = __float2bfloat16_rn(tot[m]);
    }
    return false;
  }
  // slot layout [token m][row r]: a warp's 32 rows are one 128-byte line per token
  float* pp = p.part + static_cast<size_t>(c + T) * kRowTile * NB + r;
#pragma unroll
  for (int m = 0; m < NB; ++m) __stcg(pp + m * kRowTile, tot[m]);
  return true;
}

template <int NB>
__device__ __forceinline__ void td_ticket(const TdParams& p, int T, int q, int lane) {
  __syncwarp();
  const int cf = td_cta_of_unit(T * p.G, p.U, p.P), cl = td_cta_of_unit((T + 1) * p.G - 1, p.U, p.P);
  int last = 0;
  // release of this warp's partials, acquire of the others' for the last arriver
  if (lane == 0) last = atom_add_acq_rel_gpu(&p.cnt[T * 8 + q], 1) == cl - cf;
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  __syncwarp();
  const int r = q * 32 + lane;
  const int n = T * kRowTile + r;
  // in halves of the tokens (registers); CTA order (deterministic); two
  // sharers' loads in flight at a time
  constexpr int H = NB / 2;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    float acc[H];
#pragma unroll
    for (int m = 0; m < H; ++m) acc[m] = 0.f;
    for (int cc = cf; cc <= cl; cc += 2) {
      const bool two = cc + 1 <= cl;
      const float* pp = p.part + static_cast<size_t>(cc + T) * kRowTile * NB + r + hh * H * kRowTile;
      float v[2][H];
#pragma unroll
      for (int m = 0; m < H; ++m) v[0][m] = __ldcg(pp + m * kRowTile);
      if (two) {
#pragma unroll
        for (int m = 0; m < H; ++m) v[1][m] = __ldcg(pp + kRowTile * NB + m * kRowTile);
      }
#pragma unroll
      for (int m = 0; m < H; ++m) acc[m] += v[0][m];
      if (two) {
#pragma unroll
        for (int m = 0; m < H; ++m) acc[m] += v[1][m];
      }
    }
    if (n < p.N) {
#pragma unroll
      for (int m = 0; m < H; ++m)
        if (hh * H + m < p.M) p.y[static_cast<size_t>(hh * H + m) * p.N + n] = __float2bfloat16_rn(acc[m]);
    }
  }
  __syncwarp();
  if (lane == 0) p.cnt[T * 8 + q] = 0;
}

template <int NB>
__global__ void __launch_bounds__(kTdThreads, 1) k_linear_tcdec(const __grid_constant__ CUtensorMap xmap, const TdParams p) {
  using C = TdCfg<NB>;
  constexpr int RS = C::kSbRing, RA = C::kARing, RX = C::kXRing, NC = C::kChains;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* xbuf = smem;                                    // [RX][NB*256] (1 KB aligned)
  uint8_t* sbuf = xbuf + RX * C::kXBytes;                  // [RS][8512]
  uint64_t* sb_full = reinterpret_cast<uint64_t*>(sbuf + RS * kSbBytes);
  uint64_t* sb_empty = sb_full + RS;   // the super-block's dequant group (4 warps)
  uint64_t* x_full = sb_empty + RS;    // [RX] x tile landed
  uint64_t* x_empty = x_full + RX;     // [RX] MMAs reading the x tile done
  uint64_t* a_full = x_empty + RX;     // A tile dequantized (4 warps)
  uint64_t* a_empty = a_full + RA;     // MMAs on the A slot done
  uint64_t* dfull = a_empty + RA;      // [issuer][tile buffer]: the issuer's last MMA of the tile done
  uint64_t* dempty = dfull + 2 * NC;   // [issuer][tile buffer]: the epilogue has read that accumulator
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(dempty + 2 * NC);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const int u0 = td_unit_begin(c, p.U, p.P), u1 = td_unit_begin(c + 1, p.U, p.P);
  const int nu = u1 - u0;
  // local end of the CTA's first row-tile segment
  const int seg0_end = min(nu, (u0 / p.G + 1) * p.G - u0);

  if (threadIdx.x == 0) {
    for (int j = 0; j < RS; ++j) {
      mbar_init(&sb_full[j], 1);
      mbar_init(&sb_empty[j], 4);
    }
    for (int xs = 0; xs < RX; ++xs) {
      mbar_init(&x_full[xs], 1);
      mbar_init(&x_empty[xs], 1);
    }
    for (int a = 0; a < RA; ++a) {
      mbar_init(&a_full[a], 4);
      mbar_init(&a_empty[a], 1);
    }
    for (int b = 0; b < 2 * NC; ++b) {
      mbar_init(&dfull[b], 1);
      mbar_init(&dempty[b], 4);
    }
    fence_mbar_init();
  }
  if (warp == kTdIss0) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  cta_sync();
  tc_fence_after();
  const uint32_t tmem_d = *tmem_slot;
  pdl_launch_dependents();

  if (warp == 0) {
    // ---------------- super-block producer (weights only: they do not depend on the previous kernel)
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      for (int i = 0; i < nu; ++i) {
        const int j = i % RS;
        if (i >= RS && !mbar_wait(&sb_empty[j], ((i / RS) - 1) & 1u)) {
          set_status(p.status, FL_ERR_TIMEOUT, 31);
          for (int jj = 0; jj < RS; ++jj) {
            const int nf = i / RS + (jj < i % RS ? 1 : 0);
            if (nf > 0) mbar_wait(&sb_full[jj], static_cast<uint32_t>(nf - 1) & 1u);
          }
          break;
        }
        mbar_arrive_expect_tx(&sb_full[j], kSbBytes);
        bulk_g2s_hint(sbuf + j * kSbBytes, p.w + static_cast<size_t>(u0 + i) * kSbBytes, kSbBytes, &sb_full[j], pol);
      }
    }
  } else if (warp == 1) {
    // ---------------- x producer: the tile of x for each super-block's group
    if (lane == 0) {
      pdl_wait();
      for (int i = 0; i < nu; ++i) {
        const int xs = i % RX;
        if (i >= RX && !mbar_wait(&x_empty[xs], static_cast<uint32_t>(i / RX - 1) & 1u)) {
          set_status(p.status, FL_ERR_TIMEOUT, 35);
          for (int jj = i > RX ? i - RX : 0; jj < i; ++jj) mbar_wait(&x_full[jj % RX], static_cast<uint32_t>(jj / RX) & 1u);
          break;
        }
        const int g = (u0 + i) % p.G;
        mbar_arrive_expect_tx(&x_full[xs], C::kXBytes);
        tma_load_2d(xbuf + xs * C::kXBytes, &xmap, g * kGroup, 0, &x_full[xs]);
        tma_load_2d(xbuf + xs * C::kXBytes + NB * 128, &xmap, g * kGroup + 64, 0, &x_full[xs]);
      }
    }
  } else if (warp < kTdDeq0) {
    // ---------------- MMA issuers: issuer e takes super-blocks e, e + 3, ...,
    // each into its own accumulator per row tile (two tile buffers, so that
    // the epilogue of one tile overlaps the next tile's MMAs).  One thread
    // issues tcgen05.mma at only about one per 65 cycles, and at N = NB the
    // tensor pipe is far from full, so three issuers triple the rate.  The
    // whole warp runs the loop (its addresses and descriptors are warp
    // uniform); one elected thread issues.
    const int e = warp - kTdIss0;
    const uint32_t idesc = idesc_bf16<NB>();
    int sa = 0, se = seg0_end, tl = 0;   // current row-tile segment [sa, se) and its ordinal
    uint32_t uses = 0;                   // bit tb: parity of this issuer's uses of tile buffer tb so far
    for (int i = e; i < nu; i += NC) {
      while (i >= se) {
        sa = se;
        se = min(nu, se + p.G);
        ++tl;
      }
      const int tb = tl & 1;
      const bool first = i - NC < sa, last = i + NC >= se;
      const int a = i % RA, xs = i % RX;
      // before the first MMA of a tile: the epilogue has read this issuer's
      // previous tile in the same buffer (if any)
      bool ok = true;
      if (first) {
        if (uses & (4u << tb)) ok = mbar_wait(&dempty[e * 2 + tb], ((uses >> tb) & 1u) ^ 1u);
        uses = (uses ^ (1u << tb)) | (4u << tb);
      }
      ok = ok && mbar_wait(&a_full[a], static_cast<uint32_t>(i / RA) & 1u) &&
           mbar_wait(&x_full[xs], static_cast<uint32_t>(i / RX) & 1u);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) set_status(p.status, FL_ERR_TIMEOUT, 32);
        break;
      }
      tc_fence_after();
      const uint32_t x0 = smem_u32(xbuf + xs * C::kXBytes);
      const uint32_t dcol = tmem_d + C::kDCol + (e * 2 + tb) * NB;
      if (elect_one()) {
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16_ta(dcol, tmem_d + a * 64 + h * 32 + kk * 8, sw128_desc(x0 + h * NB * 128 + kk * 32), idesc,
                         (!first || (h | kk) != 0) ? 1u : 0u);
        umma_commit(&x_empty[xs]);
        umma_commit(&a_empty[a]);
        if (last) umma_commit(&dfull[e * 2 + tb]);
      }
      __syncwarp();
    }
  } else if (warp < kTdEpi0) {
    // ---------------- dequant: group grp takes super-blocks grp, grp + 3, ...;
    // thread = row r (lane of the warp's quadrant), both K halves -> the
    // correctly rounded bf16(s16 * (q - z)) into the A slot, column c holding
    // k = 2c, 2c+1.  s16 = s_hi + s_lo (both bf16, the split exact);
    // s_lo * (q - z) is exact and fma(s_hi, q - z, s_lo * (q - z)) rounds once.
    const int q = warp & 3, grp = (warp - kTdDeq0) >> 2;
    const int r = q * 32 + lane;
    const uint32_t trow = static_cast<uint32_t>(q * 32) << 16;
    for (int i = grp; i < nu; i += NC) {
      const int j = i % RS, a = i % RA;
      if (!mbar_wait(&sb_full[j], (i / RS) & 1u)) {
        set_status(p.status, FL_ERR_TIMEOUT, 33);
        break;
      }
      const uint8_t* sb = sbuf + j * kSbBytes;
      const float sf = __half2float(reinterpret_cast<const __half*>(sb + kSbNib)[r]);
      const uint32_t z = (sb[kSbNib + kSbScale + (r >> 1)] >> ((r & 1) * 4)) & 15u;
      uint4 cv[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) cv[t] = *reinterpret_cast<const uint4*>(sb + r * 64 + ((t + (r >> 1)) & 3) * 16);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sb_empty[j]);
      const __nv_bfloat16 shi = __float2bfloat16_rn(sf);
      const __nv_bfloat16 slo = __float2bfloat16_rn(sf - __bfloat162float(shi));   // exact remainder
      const uint32_t hi2 = static_cast<uint32_t>(__bfloat16_as_ushort(shi)) * 0x00010001u;
      const uint32_t lo2 = static_cast<uint32_t>(__bfloat16_as_ushort(slo)) * 0x00010001u;
      const uint32_t zz = bf16_bias_pair(z);
      uint32_t o[32];
      // logical 8-column chunks wl = 8h .. 8h+7 live in 16-byte chunk wl % 4, word wl / 4
      auto unpack = [&](auto H) {
        constexpr int hh = decltype(H)::value;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int wl = 8 * hh + t;
          const uint32_t word = (&cv[wl & 3].x)[wl >> 2];
#pragma unroll
          for (int pi = 0; pi < 4; ++pi) {
            const uint32_t qz = bf16x2_sub(nib_pair_bf16(word, pi), zz);
            o[4 * t + pi] = bfma2(hi2, qz, bmul2(lo2, qz));
          }
        }
      };
      unpack(std::integral_constant<int, 0>());
      if (i >= RA && !mbar_wait(&a_empty[a], ((i / RA) - 1) & 1u)) {
        set_status(p.status, FL_ERR_TIMEOUT, 36);
        break;
      }
      tc_fence_after();
      tmem_st32(tmem_d + trow + a * 64, o);
      tmem_wait_st();   // o is rewritten with the second half
      unpack(std::integral_constant<int, 1>());
      tmem_st32(tmem_d + trow + a * 64 + 32, o);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_full[a]);
    }
  } else {
    // ---------------- epilogue: once per row tile, the sum of the issuers'
    // accumulators (in issuer order) for row r and every token.  A split tile
    // other than the CTA's last is handed off at once, overlapping the rest of
    // the stream; the last one at the end.
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t tq = tmem_d + (static_cast<uint32_t>(q * 32) << 16) + C::kDCol;
    pdl_wait();   // y and the workspace: only once the previous kernel is done
    int T = u0 / p.G, sa = 0, se = seg0_end, owed = -1;
    uint32_t dph = 0;   // bit b: parity of the next completion of accumulator barrier b
    bool ok = true;
    for (int tl = 0; sa < nu; ++tl) {
      const int tb = tl & 1, len = se - sa;
      float tot[NB];
#pragma unroll
      for (int m = 0; m < NB; ++m) tot[m] = 0.f;
      for (int e = 0; e < NC; ++e) {
        // issuer e has super-blocks in [sa, se) iff some i there has i % 3 == e
        const int off = ((e - sa) % NC + NC) % NC;
        if (off >= len) continue;
        const int b = e * 2 + tb;
        if (!mbar_wait(&dfull[b], (dph >> b) & 1u)) {
          set_status(p.status, FL_ERR_TIMEOUT, 34);
          ok = false;
          break;
        }
        dph ^= 1u << b;
        tc_fence_after();
#pragma unroll
        for (int hh = 0; hh < NB / 16; ++hh) {
          uint32_t v[16];
          tmem_ld16_issue(tq + b * NB + hh * 16, v);
          tmem_ld_wait(v);
#pragma unroll
          for (int m = 0; m < 16; ++m) tot[hh * 16 + m] += __uint_as_float(v[m]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&dempty[b]);
      }
      if (!ok) break;
      if (td_store<NB>(p, T, c, u0, u1, r, tot)) {
        if (se < nu)
          td_ticket<NB>(p, T, q, lane);
        else
          owed = T;
      }
      sa = se;
      se = min(nu, se + p.G);
      ++T;
    }
    if (ok && owed >= 0) td_ticket<NB>(p, owed, q, lane);
  }
  tc_fence_before();
  cta_sync();
  if (warp == kTdIss0) {
    tc_fence_after();
    tmem_dealloc(tmem_d, C::kTmemCols);
  }
}

template <int NB>
int launch_tcdec(const void* x, int M, int K, const void* w, int N, void* y, void* ws, size_t cnt_off,
                 size_t part_off, cudaStream_t s) {
  using C = TdCfg<NB>;
  auto enc = encode_fn();
  if (!enc) return FL_ERR_CUDA;
  CUtensorMap map;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(NB)};
  const cuuint32_t estr[2] = {1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return FL_ERR_CUDA;
  TdParams p;
  p.w = static_cast<const uint8_t*>(w);
  p.y = static_cast<__nv_bfloat16*>(y);
  p.status = static_cast<int32_t*>(ws);
  p.cnt = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + cnt_off);
  p.part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + part_off);
  p.M = M;
  p.K = K;
  p.N = N;
  p.T = (N + kRowTile - 1) / kRowTile;
  p.G = K / kGroup;
  p.U = p.T * p.G;
  const int sms = flh::sm_count();
  p.P = p.U < sms ? p.U : sms;
  // Few row tiles: P = T * s with s = SMs / T, so that the contiguous ranges
  // are s equal parts of each tile (K=4096, N=4096, M=32: 10.8 against 9.0
  // us); the partial slots (P + T of them) stay within the workspace.
  if (p.T * 2 <= sms) {
    const int sp = sms / p.T;
    p.P = p.T * (sp < p.G ? sp : p.G);
  }
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    if (cudaFuncSetAttribute(k_linear_tcdec<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) != cudaSuccess)
      return FL_ERR_CUDA;
    attr_done[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.P));
  cfg.blockDim = dim3(kTdThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, k_linear_tcdec<NB>, map, p) != cudaSuccess) return FL_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? FL_OK : FL_ERR_CUDA;
}

// ======================================================================
// Grouped expert GEMM of the MoE layer on tcgen05 (token segments of up to
// 128 positions of one expert, in expert order).  A tile is (segment s, 128
// output rows nt); tiles are split over the CTAs as whole tiles (no split-K),
// so every output element is one sum written once.  Unit i of a CTA (one
// super-block of a tile) goes to MMA issuer i % 2 and dequant group i % 2,
// each issuer accumulating into its own accumulator; the epilogue adds the
// two in issuer order.  Roles: x producer (the segment's rows rounded up to
// 32, 64 or 128 by TMA, one box per K half, so that short segments move and
// multiply only their own rows), weight producer (the segment's expert), two
// MMA issuers, two dequant groups of four warps, eight epilogue warps.
// Output: fp32 rows of the segment's positions, times wpos[pos] when given
// (the down projection), else as they are (gate/up).
struct MgParams {
  const uint8_t* w;          // routed experts back to back (when wtab is null)
  const uint8_t* const* wtab;  // device table of E expert pointers, or null
  const uint8_t* w_shared;   // shared expert (expert index E) or null
  size_t wbytes;             // bytes of one expert's interleaved matrix
  size_t side_off;           // groups of 64: offset of an expert's side array from its base (0: none)
  const int32_t* seg_e;
  const int32_t* seg_pos;
  const int32_t* seg_n;
  const int32_t* nseg;       // device: number of segments (written by the permute kernel)
  const float* wpos;         // per-position scale or null
  float* out;                // [positions][ldo]
  int ldo, G, TT, E, P;
  int32_t* status;
};

constexpr int kMgThreads = 20 * 32;

struct MgCfg {
  static constexpr int BN = 128;
  static constexpr int kRows = 32;              // the smallest x box (positions)
  static_assert((kRows << 2) == BN, "box heights 32, 64, 128");
  static constexpr int kBBox = BN * 64 * 2;     // 16 KB: one K half of a unit's x tile (BN positions x 64 k)
  static constexpr int kXStage = 2 * kBBox;     // a unit's x tile (its segment's rows), one barrier
  static constexpr int kBStages = 4;
  static constexpr int kSStages = 8;
  static constexpr int kARing = 4;
  static constexpr int kSOff = kBStages * kXStage;
  static constexpr int kBarOff = kSOff + kSStages * kSbBytes;
  static constexpr int kNumBars = 2 * kBStages + 2 * kSStages + 2 * kARing + 4;
  static constexpr int kSmem = kBarOff + kNumBars * 8 + 16 + 1024;
  static constexpr uint32_t kTmemCols = 512;   // accumulators 2 x BN, A ring 4 x 64
  static_assert(2 * BN + 64 * kARing <= 512, "tensor memory");
  static_assert(kSmem <= 232448, "shared memory");
  // unit i goes to MMA issuer and dequant group i % 2: every ring size is
  // even, so that each barrier has one waiter chain
  static_assert(kARing % 2 == 0 && kSStages % 2 == 0 && kBStages % 2 == 0, "one chain per slot");
};

// x tiles: the segment's positions rounded up to 32, 64 or 128 rows, one TMA
// box per K half from the tensor map of that box height (xm[0..2])
struct MgMaps {
  CUtensorMap xm[3];
};

__device__ __forceinline__ int mg_rows_kind(int n) { return n <= 32 ? 0 : n <= 64 ? 1 : 2; }

__global__ void __launch_bounds__(kMgThreads, 1) k_moe_gemm(const __grid_constant__ MgMaps maps, const MgParams p) {
  using C = MgCfg;
  constexpr int BN = C::BN, RA = C::kARing, NBS = C::kBStages, NSS = C::kSStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bfull = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* bempty = bfull + NBS;
  uint64_t* sfull = bempty + NBS;
  uint64_t* sempty = sfull + NSS;
  uint64_t* afull = sempty + NSS;
  uint64_t* aempty = afull + RA;
  uint64_t* dfull = aempty + RA;   // [issuer]: the issuer's last MMA of the tile done
  uint64_t* dempty = dfull + 2;    // [issuer]: the epilogue has read that accumulator
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(dempty + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBS; ++i) {
      mbar_init(&bfull[i], 1);
      mbar_init(&bempty[i], 1);
    }
    for (int i = 0; i < NSS; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&sempty[i], 4);
    }
    for (int i = 0; i < RA; ++i) {
      mbar_init(&afull[i], 4);
      mbar_init(&aempty[i], 1);
    }
    for (int e = 0; e < 2; ++e) {
      mbar_init(&dfull[e], 1);
      mbar_init(&dempty[e], 8);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  cta_sync();
  tc_fence_after();
  const uint32_t tmem_d = *tmem_slot;
  const uint32_t tmem_a = tmem_d + 2 * BN;
  pdl_launch_dependents();
  // the segment plan, the weights' selection and x come from earlier kernels
  pdl_wait();
  const int ntiles = *p.nseg * p.TT;
  const int t0 = static_cast<int>(static_cast<long long>(c) * ntiles / p.P);
  const int t1 = static_cast<int>(static_cast<long long>(c + 1) * ntiles / p.P);
  const int nu = (t1 - t0) * p.G;   // units of this CTA, tile-major

  if (warp == 0) {
    // ---------------- x producer
    if (lane == 0) {
      int j = 0;
      bool ok = true;
      for (int t = t0; t < t1 && ok; ++t) {
        const int sg = t / p.TT, pos0 = p.seg_pos[sg];
        // the segment's rows rounded up to 32, 64 or 128 (the MMA's N)
        const int kind = mg_rows_kind(p.seg_n[sg]);
        const CUtensorMap* xmap = &maps.xm[kind];
        const uint32_t bytes = static_cast<uint32_t>(2 * (C::kRows << kind) * 128);
        for (int g = 0; g < p.G; ++g, ++j) {
          const int b = j % NBS;
          if (j >= NBS && !mbar_wait(&bempty[b], static_cast<uint32_t>(j / NBS - 1) & 1u)) {
            set_status(p.status, FL_ERR_TIMEOUT, 41);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bfull[b], bytes);
          tma_load_2d(smem + b * C::kXStage, xmap, g * kGroup, pos0, &bfull[b]);
          tma_load_2d(smem + b * C::kXStage + C::kBBox, xmap, g * kGroup + 64, pos0, &bfull[b]);
        }
      }
      if (!ok)
        for (int jj = j > NBS ? j - NBS : 0; jj < j; ++jj) mbar_wait(&bfull[jj % NBS], static_cast<uint32_t>(jj / NBS) & 1u);
    }
  } else if (warp == 2) {
    // ---------------- weight producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int i = 0;
      bool ok = true;
      for (int t = t0; t < t1 && ok; ++t) {
        const int sg = t / p.TT, nt = t - sg * p.TT, e = p.seg_e[sg];
        // a bad table entry (recorded) skips the copies: the stages complete
        // without data and the tile's result is garbage
        const uint8_t* base = e == p.E ? p.w_shared : expert_base(p.w, p.wtab, p.wbytes, e, p.status);
        for (int g = 0; g < p.G; ++g, ++i) {
          const int sI = i % NSS;
          if (i >= NSS && !mbar_wait(&sempty[sI], static_cast<uint32_t>(i / NSS - 1) & 1u)) {
            set_status(p.status, FL_ERR_TIMEOUT, 42);
            ok = false;
            break;
          }
          if (!base) {
            mbar_arrive(&sfull[sI]);
            continue;
          }
          mbar_arrive_expect_tx(&sfull[sI], kSbBytes);
          bulk_g2s_hint(smem + C::kSOff + sI * kSbBytes, base + (static_cast<size_t>(nt) * p.G + g) * kSbBytes,
                        kSbBytes, &sfull[sI], pol);
        }
      }
      if (!ok)
        for (int ii = i > NSS ? i - NSS : 0; ii < i; ++ii) mbar_wait(&sfull[ii % NSS], static_cast<uint32_t>(ii / NSS) & 1u);
    }
  } else if (warp == 1 || warp == 3) {
    // ---------------- MMA issuers: issuer e takes units e, e + 2, ... into its
    // own accumulator.  The whole warp runs the loop; one elected thread
    // issues.
    const int e = warp == 1 ? 0 : 1;
    const uint32_t dcol = tmem_d + e * BN;
    int g = e, t = t0;               // group of unit i within its tile, and the tile
    while (g >= p.G) g -= p.G, ++t;
    uint32_t uses = 0;               // bit 0: parity of the tiles this issuer took part in; bit 1: any
    for (int i = e; i < nu; i += 2) {
      const int a = i % RA;
      const bool first = g < 2, last = g + 2 >= p.G;
      bool ok = true;
      if (first) {
        // the epilogue has read this accumulator's previous tile
        if (uses & 2u) ok = mbar_wait(&dempty[e], (uses & 1u) ^ 1u);
        uses = (uses ^ 1u) | 2u;
      }
      const int b = i % NBS;
      // N: the segment's positions rounded up to whole boxes (rows past the
      // segment are computed and not stored)
      const uint32_t idesc = idesc_bf16_n(C::kRows << mg_rows_kind(p.seg_n[t / p.TT]));
      ok = ok && mbar_wait(&afull[a], static_cast<uint32_t>(i / RA) & 1u) &&
           mbar_wait(&bfull[b], static_cast<uint32_t>(i / NBS) & 1u);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) set_status(p.status, FL_ERR_TIMEOUT, 43);
        break;
      }
      tc_fence_after();
      if (elect_one()) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t b0 = smem_u32(smem + b * C::kXStage + h * C::kBBox);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16_ta(dcol, tmem_a + a * 64 + h * 32 + kk * 8, sw128_desc(b0 + kk * 32), idesc,
                         (!first || h != 0 || kk != 0) ? 1u : 0u);
        }
        umma_commit(&bempty[b]);
        umma_commit(&aempty[a]);
        if (last) umma_commit(&dfull[e]);
      }
      __syncwarp();
      g += 2;
      while (g >= p.G) g -= p.G, ++t;
    }
  } else if (warp >= kPfDeq0 && warp < kPfEpi0) {
    // ---------------- dequant: group grp takes units grp, grp + 2, ...;
    // thread = row r, both K halves -> exact bf16(s16 * (q - z)) into the A
    // ring (s16 = s_hi + s_lo, both bf16, the split exact; s_lo * (q - z) is
    // exact and fma(s_hi, q - z, s_lo * (q - z)) rounds once)
    const int q = warp & 3, grp = (warp - kPfDeq0) >> 2;
    const int r = q * 32 + lane;
    const uint32_t trow = static_cast<uint32_t>(q * 32) << 16;
    for (int i = grp; i < nu; i += 2) {
      const int sI = i % NSS, a = i % RA;
      // groups of 64: the upper K half takes the odd group's scale and zero
      // point from the expert's side entry (read before the wait)
      float sf1 = 0.f;
      uint32_t z1 = 0;
      bool side_ok = false;
      if (p.side_off != 0) {
        const int t = t0 + i / p.G, g = i - (i / p.G) * p.G;
        const int sg = t / p.TT, nt = t - sg * p.TT, e = p.seg_e[sg];
        const uint8_t* base = e == p.E ? p.w_shared : expert_base(p.w, p.wtab, p.wbytes, e, p.status);
        if (base) {
          const uint8_t* sd = base + p.side_off + (static_cast<size_t>(nt) * p.G + g) * kSbSide;
          sf1 = __half2float(__ldg(reinterpret_cast<const __half*>(sd) + r));
          z1 = (__ldg(sd + kSbScale + (r >> 1)) >> ((r & 1) * 4)) & 15u;
          side_ok = true;
        }
      }
      if (!mbar_wait(&sfull[sI], static_cast<uint32_t>(i / NSS) & 1u)) {
        set_status(p.status, FL_ERR_TIMEOUT, 44);
        break;
      }
      const uint8_t* sb = smem + C::kSOff + sI * kSbBytes;
      const float sf0 = __half2float(reinterpret_cast<const __half*>(sb + kSbNib)[r]);
      const uint32_t z0 = (sb[kSbNib + kSbScale + (r >> 1)] >> ((r & 1) * 4)) & 15u;
      if (!side_ok) {
        sf1 = sf0;
        z1 = z0;
      }
      uint4 cv[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) cv[t] = *reinterpret_cast<const uint4*>(sb + r * 64 + ((t + (r >> 1)) & 3) * 16);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sempty[sI]);
      uint32_t o[32];
      // half hh of the row with scale sf and zero point z
      auto unpack = [&](auto H, float sf, uint32_t z) {
        constexpr int hh = decltype(H)::value;
        const __nv_bfloat16 shi = __float2bfloat16_rn(sf);
        const __nv_bfloat16 slo = __float2bfloat16_rn(sf - __bfloat162float(shi));
        const uint32_t hi2 = static_cast<uint32_t>(__bfloat16_as_ushort(shi)) * 0x00010001u;
        const uint32_t lo2 = static_cast<uint32_t>(__bfloat16_as_ushort(slo)) * 0x00010001u;
        const uint32_t zz = bf16_bias_pair(z);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int wl = 8 * hh + t;
          const uint32_t word = (&cv[wl & 3].x)[wl >> 2];
#pragma unroll
          for (int pi = 0; pi < 4; ++pi) {
            const uint32_t qz = bf16x2_sub(nib_pair_bf16(word, pi), zz);
            o[4 * t + pi] = bfma2(hi2, qz, bmul2(lo2, qz));
          }
        }
      };
      unpack(std::integral_constant<int, 0>(), sf0, z0);
      if (i >= RA && !mbar_wait(&aempty[a], static_cast<uint32_t>(i / RA - 1) & 1u)) {
        set_status(p.status, FL_ERR_TIMEOUT, 45);
        break;
      }
      tc_fence_after();
      tmem_st32(tmem_a + trow + a * 64, o);
      tmem_wait_st();   // o is rewritten with the second half
      unpack(std::integral_constant<int, 1>(), sf1, z1);
      tmem_st32(tmem_a + trow + a * 64 + 32, o);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&afull[a]);
    }
  } else if (warp >= kPfEpi0) {
    // ---------------- epilogue: rows q*32+lane of the tile, one half of its
    // 128 positions; the two issuers' accumulators added in issuer order
    const int ew = warp - kPfEpi0, q = warp & 3;
    const int r = q * 32 + lane;
    const int col0 = (ew >> 2) * (BN / 2);
    const uint32_t tcol = tmem_d + (static_cast<uint32_t>(q * 32) << 16) + col0;
    uint32_t dph = 0;   // bit e: parity of the next completion of dfull[e]
    int jt = 0;
    for (int t = t0; t < t1; ++t, ++jt) {
      // issuer e took part in the tile unless it has a single unit of the other parity
      const bool has0 = p.G >= 2 || ((jt * p.G) & 1) == 0;
      const bool has1 = p.G >= 2 || ((jt * p.G) & 1) == 1;
      if ((has0 && !mbar_wait(&dfull[0], dph & 1u)) || (has1 && !mbar_wait(&dfull[1], (dph >> 1) & 1u))) {
        set_status(p.status, FL_ERR_TIMEOUT, 47);
        break;
      }
      dph ^= (has0 ? 1u : 0u) | (has1 ? 2u : 0u);
      tc_fence_after();
      const int sg = t / p.TT, nt = t - sg * p.TT;
      const int pos0 = p.seg_pos[sg], n = p.seg_n[sg];
      const int col = nt * kRowTile + r;
#pragma unroll
      for (int k = 0; k < BN / 32; ++k) {
        uint32_t ra[16], rb[16];
        const bool live = col0 + 16 * k < n;   // columns past the segment were not computed for this tile
        if (live && has0) tmem_ld16_issue(tcol + 16 * k, ra);
        if (live && has1) tmem_ld16_issue(tcol + BN + 16 * k, rb);
        if (live && has0) tmem_ld_wait(ra);
        if (live && has1) tmem_ld_wait(rb);
        if (k == BN / 32 - 1) {
          // every read of both accumulators is done: the next tile's MMAs may start
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (has0) mbar_arrive(&dempty[0]);
            if (has1) mbar_arrive(&dempty[1]);
          }
        }
#pragma unroll
        for (int tt = 0; tt < 16; ++tt) {
          const float v = has0 ? (has1 ? __uint_as_float(ra[tt]) + __uint_as_float(rb[tt]) : __uint_as_float(ra[tt]))
                               : __uint_as_float(rb[tt]);
          const int m = col0 + 16 * k + tt;
          if (m < n) {
            const int pos = pos0 + m;
            const float sc = p.wpos ? p.wpos[pos] : 1.f;
            p.out[static_cast<size_t>(pos) * p.ldo + col] = sc * v;
          }
        }
      }
    }
  }
  tc_fence_before();
  cta_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_d, C::kTmemCols);
  }
}

}  // namespace

// Prefill path of fl_int4g_linear (M > 32): persistent stream-K tcgen05 GEMM.
size_t fl_linear_tc_workspace(int M) { return pf_workspace(M); }

// side: groups of 64, the side array of w (null for groups of 128 / 256).
int fl_linear_tc(const void* x, int M, int K, const void* w, int N, void* y, void* ws, cudaStream_t s,
                 const void* side) {
  const uint8_t* sd = static_cast<const uint8_t*>(side);
  if (pf_bn(M) == 256) return launch_tc<256>(x, M, K, w, N, y, ws, s, sd);
  return launch_tc<128>(x, M, K, w, N, y, ws, s, sd);
}

// Decode path of fl_int4g_linear on tcgen05 (M <= 32); the workspace layout is
// the decode kernel's: status, counters at cnt_off, partial slots at part_off
// ((P + T) slots of 128 rows x NB floats).
int fl_linear_tcdec(const void* x, int M, int K, const void* w, int N, void* y, void* ws, size_t cnt_off,
                    size_t part_off, cudaStream_t s) {
  if (M <= 16) return launch_tcdec<16>(x, M, K, w, N, y, ws, cnt_off, part_off, s);
  return launch_tcdec<32>(x, M, K, w, N, y, ws, cnt_off, part_off, s);
}

// Grouped expert GEMM of the MoE layer (see k_moe_gemm).  x: [npos, K] bf16
// rows in position order; out: [npos, ldo] fp32.  nseg, seg_* and wpos are
// device arrays written by earlier kernels on the same stream.
int fl_moe_gemm(const void* x, int npos, int K, const void* w, const void* const* wtab, const void* w_shared,
                size_t wbytes, size_t side_off, int E, int Nout, const int32_t* seg_e, const int32_t* seg_pos,
                const int32_t* seg_n, const int32_t* nseg, const float* wpos, float* out, int32_t* status,
                cudaStream_t s) {
  auto enc = encode_fn();
  if (!enc) return FL_ERR_CUDA;
  MgMaps maps;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(npos)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t estr[2] = {1, 1};
  for (int kind = 0; kind < 3; ++kind) {
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(MgCfg::kRows << kind)};
    if (enc(&maps.xm[kind], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return FL_ERR_CUDA;
  }
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    if (cudaFuncSetAttribute(k_moe_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, MgCfg::kSmem) != cudaSuccess)
      return FL_ERR_CUDA;
    attr_done[dev] = true;
  }
  MgParams p;
  p.w = static_cast<const uint8_t*>(w);
  p.wtab = reinterpret_cast<const uint8_t* const*>(wtab);
  p.w_shared = static_cast<const uint8_t*>(w_shared);
  p.wbytes = wbytes;
  p.side_off = side_off;
  p.seg_e = seg_e;
  p.seg_pos = seg_pos;
  p.seg_n = seg_n;
  p.nseg = nseg;
  p.wpos = wpos;
  p.out = out;
  p.ldo = Nout;
  p.G = K / kGroup;
  p.TT = Nout / kRowTile;
  p.E = E;
  p.P = flh::sm_count();
  p.status = status;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.P));
  cfg.blockDim = dim3(kMgThreads);
  cfg.dynamicSmemBytes = MgCfg::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, k_moe_gemm, maps, p) != cudaSuccess) return FL_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? FL_OK : FL_ERR_CUDA;
}
