// f3: fused int4g decode MLP block for M <= 8 tokens, in one launch:
//   y = D . (silu(G x) * (U x)),  G, U: [I, H], D: [H, I], int4g (interleaved).
//
// FastLLM page, section 3.1: in decode the 4-bit weights are read once and
// dequantized inside the matmul, so the layer is bound by the weight stream;
// the fastllm README, section 2 (--dtype int4g), applies int4g to every
// linear of the model, the MLP's three included.  One launch per linear
// leaves the weight stream idle between launches (the dependency release and
// the next kernel's first activations).  Here one persistent, cooperative
// grid streams all three matrices:
//  * phase A: units (tile pair a, group g) = the gate and up super-blocks of
//    rows 128a..128a+127, group g.  Split over K across the CTAs (stream-K:
//    equal contiguous unit ranges); a tile pair whose groups several CTAs
//    share is finished by the last of them to take its ticket (partials
//    summed in CTA order: deterministic).  The finisher applies SwiGLU,
//    stores h as bf16 and, per warp, the fp32 sums of its 16 stored h values
//    per token (for phase B's zero-point fold).
//  * hand-off: each CTA, once its phase-A work (tickets included) is done,
//    adds one to a grid counter (release); phase B's activations are read
//    only after the counter reaches the grid size (acquire, a bounded wait).
//    The producer keeps streaming down-projection super-blocks into its
//    ring meanwhile, so HBM stays busy across the hand-off.
//  * phase B: the down projection over h, two super-blocks per stage, with
//    the same stream-K split and ticket hand-off.
// The consumer arithmetic is the decode kernel's (mma.sync on bf16 pairs
// 128 + q unpacked by LOP3, zero point folded out with per-group token sums,
// fp16 scale applied to each fp32 group sum).  The grid counter is reset by
// the last CTA to exit, the tickets by each tile's finisher, so a successful
// call leaves the workspace's counters zero.
#include <algorithm>
#include <mutex>

#include "fl_common.cuh"
#include "fl_rows.cuh"

using namespace fl;

namespace {

constexpr int kCW = 8;                        // consumer warps, 16 rows each
constexpr int kThreads = (kCW + 1) * 32;
constexpr int kMp = 8;                        // one token tile of 8
constexpr int kMaxTok = 8;

struct MlpParams {
  const uint8_t* wg;         // gate, interleaved [I, H]
  const uint8_t* wu;         // up,   interleaved [I, H]
  const uint8_t* wd;         // down, interleaved [H, I]
  const __nv_bfloat16* x;    // [M, H]
  __nv_bfloat16* h;          // [M, I] (workspace)
  __nv_bfloat16* y;          // [M, H]
  float* hsum;               // [I/128][kCW][kMp]: per warp, sum of its 16 h values per token
  float* partA;              // [PA + TA] slots of [128 rows][kMp tokens][gate, up]
  float* partB;              // [PB + TB] slots of [128 rows][kMp tokens]
  int32_t* cntA;             // [TA][kCW] tickets
  int32_t* cntB;             // [TB][kCW]
  int32_t* bar;              // [0] CTAs done with phase A, [1] CTAs finished
  int32_t* status;
  int M, H, I;
  int TA, GA, UA, PA;        // phase A: I/128 tile pairs, H/128 groups, units, working CTAs
  int TB, GB, UB, PB;        // phase B: H/128 tiles, I/128 groups
  int P;                     // grid size
  int stages;
  uint32_t stage_bytes, bar_off, xsum_off, zrow_off;
  unsigned long long wait_ns;   // bound of the hand-off wait
};

__device__ __forceinline__ int ubegin(int c, int U, int P) {
  return static_cast<int>(static_cast<long long>(c) * U / P);
}
__device__ __forceinline__ int cta_of(int u, int U, int P) {
  return static_cast<int>((static_cast<long long>(u + 1) * P - 1) / U);
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// atomicAdd with release semantics at GPU scope (orders this thread's prior
// writes, and those it has observed, before the add); returns the old value.
__device__ __forceinline__ int atom_add_release_gpu(int32_t* p, int v) {
  int old;
  asm volatile("atom.add.release.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// h of tile pair a for the warp's 16 rows: SwiGLU of the gate and up sums,
// stored as bf16, and the warp's per-token sums of the stored values.
__device__ __forceinline__ void emit_h(const MlpParams& p, int a, int warp, int lane, const float (&tg)[4],
                                       const float (&tu)[4]) {
  const int gid = lane >> 2, tig = lane & 3;
  float hv[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int m = 2 * tig + (e & 1);
    const int row = a * kRowTile + warp * 16 + gid + (e >> 1) * 8;
    const float g = tg[e];
    const __nv_bfloat16 b = __float2bfloat16_rn(g / (1.f + expf(-g)) * tu[e]);
    hv[e] = m < p.M ? __bfloat162float(b) : 0.f;
    if (m < p.M) p.h[static_cast<size_t>(m) * p.I + row] = b;
  }
  // tokens 2tig and 2tig+1: rows gid and gid+8, then the 8 row groups (fixed order)
  float s0 = hv[0] + hv[2], s1 = hv[1] + hv[3];
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    s0 += __shfl_xor_sync(0xffffffffu, s0, o);
    s1 += __shfl_xor_sync(0xffffffffu, s1, o);
  }
  if (gid == 0) *reinterpret_cast<float2*>(p.hsum + (static_cast<size_t>(a) * kCW + warp) * kMp + 2 * tig) =
      make_float2(s0, s1);
}

// Phase A: a tile pair computed whole by this CTA is emitted; otherwise its
// partial sums go to slot c + a and a ticket is owed (returns true).
__device__ __forceinline__ bool store_a(const MlpParams& p, int a, int c, int u0, int u1, int warp, int lane,
                                        const float (&tg)[4], const float (&tu)[4]) {
  if (a * p.GA >= u0 && (a + 1) * p.GA <= u1) {
    emit_h(p, a, warp, lane, tg, tu);
    return false;
  }
  const int gid = lane >> 2, tig = lane & 3;
  float* sp = p.partA + (static_cast<size_t>(c + a) * kRowTile + warp * 16) * kMp * 2;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh)
    __stcg(reinterpret_cast<float4*>(sp + ((gid + 8 * hh) * kMp + 2 * tig) * 2),
           make_float4(tg[2 * hh], tu[2 * hh], tg[2 * hh + 1], tu[2 * hh + 1]));
  return true;
}

__device__ __forceinline__ void ticket_a(const MlpParams& p, int a, int warp, int lane) {
  __syncwarp();
  const int cf = cta_of(a * p.GA, p.UA, p.PA), cl = cta_of((a + 1) * p.GA - 1, p.UA, p.PA);
  int last = 0;
  if (lane == 0) {
    last = atom_add_release_gpu(&p.cntA[a * kCW + warp], 1) == cl - cf;
    if (last) fence_acq_rel_gpu();
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  const int gid = lane >> 2, tig = lane & 3;
  float tg[4] = {0.f, 0.f, 0.f, 0.f}, tu[4] = {0.f, 0.f, 0.f, 0.f};
  // CTA order (deterministic); four slots' loads in flight at a time
  const size_t kSlot = static_cast<size_t>(kRowTile) * kMp * 2;
  const float* base = p.partA + (static_cast<size_t>(cf + a) * kRowTile + warp * 16) * kMp * 2;
  const int np = cl - cf + 1;
  for (int j0 = 0; j0 < np; j0 += 4) {
    float4 v[4][2];
#pragma unroll
    for (int t = 0; t < 4; ++t)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
        v[t][hh] = j0 + t < np ? __ldcg(reinterpret_cast<const float4*>(base + (j0 + t) * kSlot +
                                                                        ((gid + 8 * hh) * kMp + 2 * tig) * 2))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int t = 0; t < 4; ++t)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
        tg[2 * hh] += v[t][hh].x, tu[2 * hh] += v[t][hh].y, tg[2 * hh + 1] += v[t][hh].z, tu[2 * hh + 1] += v[t][hh].w;
  }
  emit_h(p, a, warp, lane, tg, tu);
  if (lane == 0) p.cntA[a * kCW + warp] = 0;
}

// Phase B: y rows of tile t (bf16), or partial sums to slot c + t.
__device__ __forceinline__ void emit_y(const MlpParams& p, int t, int warp, int lane, const float (&tot)[4]) {
  const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int n = t * kRowTile + warp * 16 + gid + (e >> 1) * 8;
    const int m = 2 * tig + (e & 1);
    if (m < p.M) p.y[static_cast<size_t>(m) * p.H + n] = __float2bfloat16_rn(tot[e]);
  }
}

__device__ __forceinline__ bool store_b(const MlpParams& p, int t, int c, int u0, int u1, int warp, int lane,
                                        const float (&tot)[4]) {
  if (t * p.GB >= u0 && (t + 1) * p.GB <= u1) {
    emit_y(p, t, warp, lane, tot);
    return false;
  }
  const int gid = lane >> 2, tig = lane & 3;
  float* sp = p.partB + (static_cast<size_t>(c + t) * kRowTile + warp * 16) * kMp;
  __stcg(reinterpret_cast<float2*>(sp + gid * kMp + 2 * tig), make_float2(tot[0], tot[1]));
  __stcg(reinterpret_cast<float2*>(sp + (gid + 8) * kMp + 2 * tig), make_float2(tot[2], tot[3]));
  return true;
}

__device__ __forceinline__ void ticket_b(const MlpParams& p, int t, int warp, int lane) {
  __syncwarp();
  const int cf = cta_of(t * p.GB, p.UB, p.PB), cl = cta_of((t + 1) * p.GB - 1, p.UB, p.PB);
  int last = 0;
  if (lane == 0) {
    last = atom_add_release_gpu(&p.cntB[t * kCW + warp], 1) == cl - cf;
    if (last) fence_acq_rel_gpu();
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  const int gid = lane >> 2, tig = lane & 3;
  float tot[4] = {0.f, 0.f, 0.f, 0.f};
  // CTA order (deterministic); four slots' loads in flight at a time
  const size_t kSlot = static_cast<size_t>(kRowTile) * kMp;
  const float* base = p.partB + (static_cast<size_t>(cf + t) * kRowTile + warp * 16) * kMp;
  const int np = cl - cf + 1;
  for (int j0 = 0; j0 < np; j0 += 4) {
    float2 v[4][2];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float* sp = base + (j0 + q) * kSlot;
      const bool in = j0 + q < np;
      v[q][0] = in ? __ldcg(reinterpret_cast<const float2*>(sp + gid * kMp + 2 * tig)) : make_float2(0.f, 0.f);
      v[q][1] = in ? __ldcg(reinterpret_cast<const float2*>(sp + (gid + 8) * kMp + 2 * tig)) : make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) tot[0] += v[q][0].x, tot[1] += v[q][0].y, tot[2] += v[q][1].x, tot[3] += v[q][1].y;
  }
  emit_y(p, t, warp, lane, tot);
  if (lane == 0) p.cntB[t * kCW + warp] = 0;
}

// One fp32 group sum folded into a running total: v = acc - (128 + z) * sum_k x,
// tot += s16 * v.  128 + z as a float: z in the mantissa of 128.0.
__device__ __forceinline__ void fold_add(float (&tot)[4], const float (&acc)[1][4], float s0, float s1, uint32_t z0,
                                         uint32_t z1, float2 xs) {
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const uint32_t z = (e >> 1) ? z1 : z0;
    const float v = fmaf(-__uint_as_float(0x43000000u + (z << 16)), (e & 1) ? xs.y : xs.x, acc[0][e]);
    tot[e] = fmaf((e >> 1) ? s1 : s0, v, tot[e]);
  }
}

__global__ void __launch_bounds__(kThreads, 2) k_mlp_block(const MlpParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  uint64_t* empty = full + p.stages;
  uint64_t* passed = empty + p.stages;                     // the producer saw the hand-off complete
  volatile int32_t* hand_fail = reinterpret_cast<volatile int32_t*>(passed + 1);   // ... or gave up
  volatile int32_t* cfail = hand_fail + 1;                 // a consumer warp gave up (shared decision)
  float* xsum = reinterpret_cast<float*>(smem + p.xsum_off);   // [group slot][kMp]
  const uint8_t* xzero = smem + p.zrow_off;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const uint32_t xoff = 2 * kSbBytes;   // activations follow the two super-blocks of a stage

  // this CTA's ranges: phase A one unit per stage, phase B two
  const bool inA = c < p.PA, inB = c < p.PB;
  const int uA0 = inA ? ubegin(c, p.UA, p.PA) : 0, uA1 = inA ? ubegin(c + 1, p.UA, p.PA) : 0;
  const int uB0 = inB ? ubegin(c, p.UB, p.PB) : 0, uB1 = inB ? ubegin(c + 1, p.UB, p.PB) : 0;
  const int nA = uA1 - uA0, nBu = uB1 - uB0, nB = (nBu + 1) / 2;
  const int total = nA + nB;
  const int g0A = inA ? uA0 % p.GA : 0, g0B = inB ? uB0 % p.GB : 0;
  const int nslotA = nA < p.GA ? nA : p.GA, nslotB = nBu < p.GB ? nBu : p.GB;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCW);
    }
    mbar_init(passed, 1);
    *hand_fail = 0;
    *cfail = 0;
    fence_mbar_init();
  }
  if (threadIdx.x < 16) reinterpret_cast<uint4*>(smem + p.zrow_off)[threadIdx.x] = make_uint4(0u, 0u, 0u, 0u);
  cta_sync();

  if (warp == kCW) {
    // ------------------------------------------------ producer warp
    const uint64_t pol = policy_evict_first();
    bool ok = true, have = nB == 0;   // have: the hand-off is complete (phase-B activations may be read)
    auto issue_w = [&](int k, int slot) {
      uint8_t* st = smem + static_cast<size_t>(slot) * p.stage_bytes;
      if (lane != 0) return;
      if (k < nA) {
        const int u = uA0 + k, a = u / p.GA, g = u - a * p.GA;
        mbar_arrive_expect_tx(&full[slot], 2u * kSbBytes + p.M * 256u);
        bulk_g2s_hint(st, p.wg + (static_cast<size_t>(a) * p.GA + g) * kSbBytes, kSbBytes, &full[slot], pol);
        bulk_g2s_hint(st + kSbBytes, p.wu + (static_cast<size_t>(a) * p.GA + g) * kSbBytes, kSbBytes, &full[slot],
                      pol);
      } else {
        const int ub = uB0 + 2 * (k - nA), n = min(2, uB1 - ub);
        mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(n) * (kSbBytes + p.M * 256u));
        bulk_g2s_hint(st, p.wd + static_cast<size_t>(ub) * kSbBytes, static_cast<uint32_t>(n) * kSbBytes,
                      &full[slot], pol);
      }
    };
    auto issue_act = [&](int k) {
      uint8_t* st = smem + static_cast<size_t>(k % p.stages) * p.stage_bytes + xoff;
      uint64_t* fb = &full[k % p.stages];
      if (k < nA) {
        const int g = (uA0 + k) % p.GA;
        for (int m = lane; m < p.M; m += 32)
          bulk_g2s(st + m * kXRowStride, p.x + static_cast<size_t>(m) * p.H + g * kGroup, 256u, fb);
      } else {
        const int ub = uB0 + 2 * (k - nA), n = min(2, uB1 - ub);
        for (int idx = lane; idx < n * p.M; idx += 32) {
          const int i = idx / p.M, m = idx - i * p.M;
          const int g = (ub + i) % p.GB;
          bulk_g2s(st + (i * p.M + m) * kXRowStride, p.h + static_cast<size_t>(m) * p.I + g * kGroup, 256u, fb);
        }
      }
    };
    // Phase-B activations need every CTA's phase A: wait for the grid counter.
    auto probe = [&](bool block) -> bool {
      int done = 0;
      if (lane == 0) {
        const unsigned long long t0 = globaltimer();
        for (;;) {
          if (ld_acquire_gpu(p.bar) >= p.P) { done = 1; break; }
          if (!block) break;
          if (globaltimer() - t0 > p.wait_ns) { done = -1; break; }
          __nanosleep(64);
        }
      }
      done = __shfl_sync(0xffffffffu, done, 0);
      __syncwarp();   // orders lane 0's acquire before every lane's copies of h
      if (done == 1) {
        fence_proxy_async_global();   // h, written by other CTAs' generic stores, is read by bulk copies
        if (lane == 0) mbar_arrive(passed);
      } else if (done < 0 && lane == 0) {
        set_status(p.status, FL_ERR_TIMEOUT, 21);
        *hand_fail = 1;
        mbar_arrive(passed);
      }
      if (done < 0) ok = false;
      return done == 1;
    };
    int kx = 0;
    for (int kw = 0; kw < total && ok; ++kw) {
      const int slot = kw % p.stages;
      if (kw >= p.stages) {
        // the stage to recycle (kw - stages) must have its activations issued
        while (ok && kx <= kw - p.stages) {
          if (kx >= nA && !have) have = probe(true);
          if (!ok) break;
          issue_act(kx++);
        }
        if (!ok) break;
        if (!mbar_wait(&empty[slot], ((kw / p.stages) & 1u) ^ 1u)) {
          if (lane == 0) set_status(p.status, FL_ERR_TIMEOUT, 22);
          ok = false;
          break;
        }
      }
      issue_w(kw, slot);
      __syncwarp();
      // activations right behind the weights; phase B's only once the
      // hand-off is known complete (no probe here: each costs an L2 round
      // trip, and the weights keep filling the ring meanwhile)
      while (kx <= kw && (kx < nA || have)) issue_act(kx++);
    }
    while (ok && kx < total) {
      if (kx >= nA && !have) have = probe(true);
      if (!ok) break;
      issue_act(kx++);
    }
    if (!ok) {
      // let the copies already issued land before the CTA retires (a stage
      // still waiting for its activations gives up after the normal bound)
      if (lane == 0 && !have && nB > 0 && *hand_fail == 0) {
        *hand_fail = 1;
        mbar_arrive(passed);
      }
      for (int j = 0; j < p.stages; ++j) {
        const int nf = kx / p.stages + (j < kx % p.stages ? 1 : 0);
        if (nf > 0) mbar_wait(&full[j], static_cast<uint32_t>(nf - 1) & 1u);
      }
    }
  } else {
    // ------------------------------------------------ consumer warps
    const int gid = lane >> 2, tig = lane & 3;
    const int r0 = warp * 16 + gid;
    bool ok = true;
    // Σx per (phase-A group slot, token): four threads per item, fixed order
    {
      const int items = nslotA * p.M;
      const int nthr = (items * 4 + 31) & ~31;
      for (int idx = threadIdx.x; idx < nthr; idx += kCW * 32) {
        const int it = idx >> 2, part = idx & 3;
        float v = 0.f;
        if (it < items) {
          const int i = it / p.M, m = it - i * p.M;
          int g = g0A + i;
          if (g >= p.GA) g -= p.GA;
          const uint4* src = reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(m) * p.H + g * kGroup) + part * 4;
          float a4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const uint4 q = __ldg(src + t);
            const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int hh = 0; hh < 4; ++hh) {
              a4[hh] += __uint_as_float(w4[hh] << 16);
              a4[hh] += __uint_as_float(w4[hh] & 0xffff0000u);
            }
          }
          v = (a4[0] + a4[1]) + (a4[2] + a4[3]);
        }
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        if (part == 0 && it < items) xsum[(it / p.M) * kMp + it % p.M] = v;
      }
      for (int idx = threadIdx.x; idx < nslotA * (kMp - p.M); idx += kCW * 32) {
        const int i = idx / (kMp - p.M), m = p.M + idx - i * (kMp - p.M);
        xsum[i * kMp + m] = 0.f;
      }
      named_bar(1, kCW * 32);
    }
    int s = 0;
    uint32_t ph = 0;
    // ---------------- phase A
    {
      float tg[4] = {0.f, 0.f, 0.f, 0.f}, tu[4] = {0.f, 0.f, 0.f, 0.f};
      int a = nA > 0 ? uA0 / p.GA : 0, g = g0A, owed0 = -1, slot = 0;
      for (int k = 0; k < nA; ++k) {
        if (!mbar_wait(&full[s], ph)) {
          if (lane == 0) set_status(p.status, FL_ERR_TIMEOUT, 23);
          ok = false;
          break;
        }
        const uint8_t* st = smem + static_cast<size_t>(s) * p.stage_bytes;
        float ag[1][4], au[1][4];
        float sg0, sg1, su0, su1;
        uint32_t zg0, zg1, zu0, zu1;
        unit_dot<1, true, true>(st, st + xoff, p.M, r0, gid, tig, ag, sg0, sg1, zg0, zg1, 1, xzero);
        unit_dot<1, true, true>(st + kSbBytes, st + xoff, p.M, r0, gid, tig, au, su0, su1, zu0, zu1, 1, xzero);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        const float2 xs = *reinterpret_cast<const float2*>(xsum + slot * kMp + 2 * tig);
        if (++slot == nslotA) slot = 0;
        fold_add(tg, ag, sg0, sg1, zg0, zg1, xs);
        fold_add(tu, au, su0, su1, zu0, zu1, xs);
        if (++s == p.stages) s = 0, ph ^= 1u;
        if (++g == p.GA && k + 1 < nA) {
          g = 0;
          if (store_a(p, a, c, uA0, uA1, warp, lane, tg, tu)) owed0 = a;
#pragma unroll
          for (int e = 0; e < 4; ++e) tg[e] = 0.f, tu[e] = 0.f;
          ++a;
        } else if (g == p.GA) {
          g = 0;
        }
      }
      if (ok && nA > 0) {
        const bool owed1 = store_a(p, a, c, uA0, uA1, warp, lane, tg, tu);
        if (owed0 >= 0) ticket_a(p, owed0, warp, lane);
        if (owed1) ticket_a(p, a, warp, lane);
      }
    }
    // ---------------- hand-off: this CTA's h is written (tickets included).
    // Decisions that lead to named barriers are taken by all consumer warps
    // together, through cfail read after a barrier.
    if (!ok) *cfail = 1;
    fence_proxy_async_global();
    named_bar(1, kCW * 32);
    ok = *cfail == 0;
    if (threadIdx.x == 0) atom_add_release_gpu(p.bar, 1);
    if (ok && nB > 0) {
      if (!mbar_wait(passed, 0) || *hand_fail) {
        if (lane == 0 && !*hand_fail) set_status(p.status, FL_ERR_TIMEOUT, 24);
        *cfail = 1;
      }
    }
    named_bar(1, kCW * 32);
    ok = ok && *cfail == 0;
    if (ok && nB > 0) {
      fence_acq_rel_gpu();
      // Σh per (phase-B group slot, token): the 8 warp sums of the group's h tile, in warp order
      for (int idx = threadIdx.x; idx < nslotB * kMp; idx += kCW * 32) {
        const int i = idx / kMp, m = idx - i * kMp;
        int g = g0B + i;
        if (g >= p.GB) g -= p.GB;
        float v = 0.f;
        if (m < p.M)
          for (int w = 0; w < kCW; ++w) v += __ldcg(p.hsum + (static_cast<size_t>(g) * kCW + w) * kMp + m);
        xsum[idx] = v;
      }
      named_bar(1, kCW * 32);
      // ---------------- phase B (two units per stage)
      float tot[4] = {0.f, 0.f, 0.f, 0.f};
      int t = uB0 / p.GB, g = g0B, slot = 0, owed0 = -1;
      for (int k = 0; k < nB; ++k) {
        const int ub = uB0 + 2 * k, n = min(2, uB1 - ub);
        if (!mbar_wait(&full[s], ph)) {
          if (lane == 0) set_status(p.status, FL_ERR_TIMEOUT, 25);
          ok = false;
          break;
        }
        const uint8_t* st = smem + static_cast<size_t>(s) * p.stage_bytes;
        float acc[2][1][4];
        float sc[2][2];
        uint32_t zr[2][2];
        // both slots in one basic block (two independent MMA chains); a slot
        // past the end of the range holds stale data and its result is dropped
#pragma unroll
        for (int i = 0; i < 2; ++i)
          unit_dot<1, true, true>(st + i * kSbBytes, st + xoff + i * p.M * kXRowStride, p.M, r0, gid, tig, acc[i],
                                  sc[i][0], sc[i][1], zr[i][0], zr[i][1], 1, xzero);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (++s == p.stages) s = 0, ph ^= 1u;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (i < n) {
            const float2 xs = *reinterpret_cast<const float2*>(xsum + slot * kMp + 2 * tig);
            if (++slot == nslotB) slot = 0;
            fold_add(tot, acc[i], sc[i][0], sc[i][1], zr[i][0], zr[i][1], xs);
            if (++g == p.GB) {
              g = 0;
              if (ub + i + 1 < uB1) {
                if (store_b(p, t, c, uB0, uB1, warp, lane, tot)) owed0 = t;
#pragma unroll
                for (int e = 0; e < 4; ++e) tot[e] = 0.f;
                ++t;
              }
            }
          }
        }
      }
      if (ok) {
        const bool owed1 = store_b(p, t, c, uB0, uB1, warp, lane, tot);
        if (owed0 >= 0) ticket_b(p, owed0, warp, lane);
        if (owed1) ticket_b(p, t, warp, lane);
      }
    }
  }
  // ---------------- the last CTA to finish resets the grid counters
  cta_sync();
  if (threadIdx.x == 0) {
    fence_acq_rel_gpu();
    if (atomicAdd(p.bar + 1, 1) == p.P - 1) {
      p.bar[0] = 0;
      p.bar[1] = 0;
    }
  }
}

// ------------------------------------------------------------------ host
struct MlpPlan {
  int TA, GA, UA, PA, TB, GB, UB, PB, P, stages;
  uint32_t stage_bytes, bar_off, xsum_off, zrow_off;
  size_t smem;
  size_t o_bar, o_cntA, o_cntB, o_hsum, o_h, o_partA, o_partB, total;
};

size_t al256(size_t v) { return (v + 255) / 256 * 256; }
size_t al16(size_t v) { return (v + 15) / 16 * 16; }

// CTAs per SM the kernel may keep resident with `smem` bytes (cached per
// device and size); 0 when the query fails.
int mlp_blocks_per_sm(size_t smem) {
  struct Entry { int dev; size_t smem; int nb; };
  static Entry cache[64];
  static int n = 0;
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (cache[i].dev == dev && cache[i].smem == smem) return cache[i].nb;
  if (cudaFuncSetAttribute(k_mlp_block, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, k_mlp_block, kThreads, smem) != cudaSuccess) {
    cudaGetLastError();
    nb = 0;
  }
  if (n < 64) cache[n++] = Entry{dev, smem, nb};
  return nb;
}

// ctas: grid size (2 per SM).  The workspace layout depends on it.
bool make_mlp_plan(int M, int H, int I, int ctas, MlpPlan* pl) {
  if (M < 1 || M > kMaxTok || H < kGroup || I < kGroup || H % kGroup || I % kGroup || ctas < 1) return false;
  if (static_cast<long long>(H) * I > (1LL << 34)) return false;
  pl->TA = I / kRowTile;
  pl->GA = H / kGroup;
  pl->UA = pl->TA * pl->GA;
  pl->TB = H / kRowTile;
  pl->GB = I / kGroup;
  pl->UB = pl->TB * pl->GB;
  pl->P = ctas;
  pl->PA = pl->UA < ctas ? pl->UA : ctas;
  pl->PB = pl->UB < ctas ? pl->UB : ctas;
  const int maxA = (pl->UA + pl->PA - 1) / pl->PA, maxB = (pl->UB + pl->PB - 1) / pl->PB;
  const int nslot = std::max(std::min(maxA, pl->GA), std::min(maxB, pl->GB));
  pl->stage_bytes = static_cast<uint32_t>((2 * kSbBytes + 2 * M * kXRowStride + 127) / 128 * 128);
  const size_t extras = 16 * 12 + 16 + static_cast<size_t>(nslot) * kMp * 4 + 256 + 64;
  int stages = static_cast<int>((100u * 1024u - extras) / pl->stage_bytes);
  pl->stages = stages > 12 ? 12 : (stages < 2 ? 2 : stages);
  pl->bar_off = static_cast<uint32_t>(pl->stages) * pl->stage_bytes;
  pl->xsum_off = static_cast<uint32_t>(al16(pl->bar_off + (2 * pl->stages + 1) * 8 + 8));
  pl->zrow_off = static_cast<uint32_t>(al16(pl->xsum_off + static_cast<size_t>(nslot) * kMp * 4));
  pl->smem = pl->zrow_off + 256;
  // counters (zero between calls) in the shared counter region, scratch after it
  if (16 + 4ull * (pl->TA + pl->TB) * kCW > kScratchOff - kTicketOff) return false;
  size_t o = kTicketOff;
  pl->o_bar = o; o += 16;
  pl->o_cntA = o; o += 4ull * pl->TA * kCW;
  pl->o_cntB = o;
  o = kScratchOff;
  pl->o_hsum = o; o = al256(o + 4ull * pl->GB * kCW * kMp);
  pl->o_h = o; o = al256(o + 2ull * M * I);
  pl->o_partA = o; o = al256(o + 4ull * (pl->PA + pl->TA) * kRowTile * kMp * 2);
  pl->o_partB = o; o = al256(o + 4ull * (pl->PB + pl->TB) * kRowTile * kMp);
  pl->total = o;
  return true;
}

}  // namespace

int fl_linear_rows_workspace(int M, int N, int K, size_t* out);
int fl_linear_decode_workspace(int M, int N, int K, size_t* out);
int fl_linear_decode(const void* x, int M, int K, const void* w, int N, void* y, void* ws, size_t ws_bytes,
                     cudaStream_t s);
int fl_linear_glu(const void* x, int M, int H, const void* w_gate, const void* w_up, int I, void* h, void* ws,
                  size_t ws_bytes, cudaStream_t stream);

// Two-launch form: its workspace is the two decode linears' (shared, used in
// turn) and h after it.
static bool two_launch_layout(int M, int H, int I, size_t* h_off, size_t* total) {
  size_t a = 0, b = 0;
  if (fl_linear_rows_workspace(M, I, H, &a) != FL_OK || fl_linear_decode_workspace(M, H, I, &b) != FL_OK)
    return false;
  *h_off = (std::max(a, b) + 255) / 256 * 256;
  *total = *h_off + 2ull * M * I;
  return true;
}

extern "C" int fl_int4g_mlp_workspace(int M, int H, int I, size_t* out) {
  MlpPlan pl;
  size_t h_off = 0, two = 0;
  if (!out || !make_mlp_plan(M, H, I, 2 * flh::sm_count(), &pl) || !two_launch_layout(M, H, I, &h_off, &two))
    return FL_ERR_ARG;
  *out = std::max(pl.total, two);
  return FL_OK;
}

extern "C" int fl_int4g_mlp_fused(const void* x, int M, int H, int I, const void* w_gate, const void* w_up,
                                  const void* w_down, void* y, void* ws, size_t ws_bytes, fl_stream_t stream);

extern "C" int fl_int4g_mlp(const void* x, int M, int H, int I, const void* w_gate, const void* w_up,
                            const void* w_down, void* y, void* ws, size_t ws_bytes, fl_stream_t stream) {
  if (!x || !w_gate || !w_up || !w_down || !y || !ws) return FL_ERR_ARG;
  if (!flh::aligned16(x) || !flh::aligned16(w_gate) || !flh::aligned16(w_up) || !flh::aligned16(w_down) ||
      !flh::aligned16(y) || !flh::aligned16(ws))
    return FL_ERR_ARG;
  if (M > kMaxTok && M >= 1) return FL_ERR_UNSUPPORTED;
  size_t need = 0, h_off = 0, two = 0;
  if (fl_int4g_mlp_workspace(M, H, I, &need) != FL_OK || !two_launch_layout(M, H, I, &h_off, &two))
    return FL_ERR_ARG;
  if (ws_bytes < need) return FL_ERR_WORKSPACE;
  // gate/up with SwiGLU, then down, chained by programmatic launch; shapes
  // without the cluster split take the one-launch kernel
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  void* h = static_cast<uint8_t*>(ws) + h_off;
  const int rc = fl_linear_glu(x, M, H, w_gate, w_up, I, h, ws, h_off, s);
  if (rc == FL_ERR_UNSUPPORTED) return fl_int4g_mlp_fused(x, M, H, I, w_gate, w_up, w_down, y, ws, ws_bytes, stream);
  if (rc != FL_OK) return rc;
  return fl_linear_decode(h, M, I, w_down, H, y, ws, h_off, s);
}

extern "C" int fl_int4g_mlp_fused(const void* x, int M, int H, int I, const void* w_gate, const void* w_up,
                                  const void* w_down, void* y, void* ws, size_t ws_bytes, fl_stream_t stream) {
  if (!x || !w_gate || !w_up || !w_down || !y || !ws) return FL_ERR_ARG;
  if (!flh::aligned16(x) || !flh::aligned16(w_gate) || !flh::aligned16(w_up) || !flh::aligned16(w_down) ||
      !flh::aligned16(y) || !flh::aligned16(ws))
    return FL_ERR_ARG;
  if (M > kMaxTok && M >= 1) return FL_ERR_UNSUPPORTED;
  MlpPlan pl;
  const int sms = flh::sm_count();
  if (!make_mlp_plan(M, H, I, 2 * sms, &pl)) return FL_ERR_ARG;
  if (ws_bytes < pl.total) return FL_ERR_WORKSPACE;
  // every CTA must be resident at once (they wait on one another)
  if (mlp_blocks_per_sm(pl.smem) < 2) return FL_ERR_UNSUPPORTED;
  uint8_t* W = static_cast<uint8_t*>(ws);
  MlpParams p;
  p.wg = static_cast<const uint8_t*>(w_gate);
  p.wu = static_cast<const uint8_t*>(w_up);
  p.wd = static_cast<const uint8_t*>(w_down);
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.h = reinterpret_cast<__nv_bfloat16*>(W + pl.o_h);
  p.y = static_cast<__nv_bfloat16*>(y);
  p.hsum = reinterpret_cast<float*>(W + pl.o_hsum);
  p.partA = reinterpret_cast<float*>(W + pl.o_partA);
  p.partB = reinterpret_cast<float*>(W + pl.o_partB);
  p.cntA = reinterpret_cast<int32_t*>(W + pl.o_cntA);
  p.cntB = reinterpret_cast<int32_t*>(W + pl.o_cntB);
  p.bar = reinterpret_cast<int32_t*>(W + pl.o_bar);
  p.status = reinterpret_cast<int32_t*>(W);
  p.M = M;
  p.H = H;
  p.I = I;
  p.TA = pl.TA;
  p.GA = pl.GA;
  p.UA = pl.UA;
  p.PA = pl.PA;
  p.TB = pl.TB;
  p.GB = pl.GB;
  p.UB = pl.UB;
  p.PB = pl.PB;
  p.P = pl.P;
  p.stages = pl.stages;
  p.stage_bytes = pl.stage_bytes;
  p.bar_off = pl.bar_off;
  p.xsum_off = pl.xsum_off;
  p.zrow_off = pl.zrow_off;
  p.wait_ns = kWaitLimitNs;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.P);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, k_mlp_block, p) != cudaSuccess) {
    cudaGetLastError();
    return FL_ERR_CUDA;
  }
  return FL_OK;
}
