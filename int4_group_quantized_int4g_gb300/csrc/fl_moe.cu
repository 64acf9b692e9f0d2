// a5-a7: routed MoE layer with int4g experts.
//
// fastllm README (gittoolsai mirror), "2. 如何设定推理精度" (--moe_dtype int4g)
// and "5. 其它参数" (--moe_experts = top-k, --cuda_se = shared expert on the
// GPU): the expert FFNs hold int4g weights; each token runs through its top-k
// experts and an always-on shared expert.
//
// Pipeline, one stream, no host synchronisation:
//   k_moe_route    one warp per token: top-k of the fp32 logits, gate weights
//   k_moe_permute  one CTA: stable counting sort of the M*k assignments by
//                  expert, token segments of <= 8 rows per expert (the shared
//                  expert is one more expert holding every token with weight
//                  1), the device-side work plan, and (for the grouped
//                  rows kernels) zeroed ticket counters
//   k_moe_rows<0>  grouped gate/up: h = silu(G x) * (U x), bf16 [pos, I]
//   k_moe_rows<1>  grouped down: out = w_pos * (W2 h), fp32 [pos, H]
//   k_moe_combine  y[t] = sum_j out[slot (t,j)] + shared out[t], bf16
// The grouped kernels stream each active expert's super-blocks once per
// segment, with the same register-dequant mma.sync consumer as the decode
// linear, split over K across all SMs with a ticket hand-off, two CTAs per
// SM.  For M <= 8 with plain routing, k_moe_rows routes the tokens itself in
// every CTA and neither k_moe_route nor k_moe_permute is launched.
//
// With many tokens per expert (see moe_uses_gemm) the two grouped steps run on the
// tensor-memory GEMM instead (fl_moe_gemm, segments of up to 128 positions):
//   k_moe_gather   x rows in position order, bf16 [pos, H]
//   fl_moe_gemm    gate/up rows, fp32 [pos, 2I]
//   k_moe_swiglu   h = silu(gate) * up, bf16 [pos, I]
//   fl_moe_gemm    out = w_pos * (W2 h), fp32 [pos, H]
#include <climits>

#include "fl_common.cuh"
#include "fl_rows.cuh"

using namespace fl;

namespace {

constexpr int kNT = 1;                // token tiles of 8 per segment: segments of 8 positions
constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxE = 1024;
constexpr int kMaxAssign = 16384;     // M * k handled by the one-CTA permute

struct MoePlan {
  int nseg;   // segments (routed + shared)
  int U;      // units of each grouped kernel: nseg * tiles * groups
  int pad[14];
};

// ------------------------------------------------------------------ route
// Order used by the selection: larger logit first, equal logits -> lower index.

// A float's order as a signed integer (NaN excluded; -0 taken as +0).
__device__ __forceinline__ int order_key(float x) {
  const int b = __float_as_int(x == 0.f ? 0.f : x);
  return b ^ ((b >> 31) & 0x7fffffff);
}

// The routing of one token by one warp: the top k of the E logits at l
// (E <= 32 * kPer; a NaN counts as -inf and is reported through the return
// value), then the gate weights in fp32.  Lane j < k ends with slot j:
// expert `mye`, weight `myw`.  Each pick takes the warp maximum of the
// untaken keys and, among the lanes holding it, the lowest expert index.
template <int kPer>
__device__ __forceinline__ bool route_token(const float* __restrict__ l, int E, int k, int scoring, int renorm,
                                            float scale, int lane, int& mye, float& myw) {
  float v[kPer];
  int key[kPer];
  int bad = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = lane + 32 * i;
    float x = -INFINITY;
    if (e < E) {
      x = l[e];
      if (isnan(x)) bad = 1, x = -INFINITY;
    }
    v[i] = x;
    key[i] = e < E ? order_key(x) : INT_MIN;   // a real -inf still beats an absent slot
  }
  uint32_t taken = 0;
  float myv = -INFINITY, v0 = -INFINITY;
  mye = 0;
  for (int j = 0; j < k; ++j) {
    int lk = INT_MIN, li = 0;
    float lv = -INFINITY;
#pragma unroll
    for (int i = 0; i < kPer; ++i)
      if (!((taken >> i) & 1u) && key[i] > lk) lk = key[i], li = i, lv = v[i];
    const int m = __reduce_max_sync(0xffffffffu, lk);
    const int be = __reduce_min_sync(0xffffffffu, lk == m ? li * 32 + lane : INT_MAX);
    const float bv = __shfl_sync(0xffffffffu, lv, be & 31);
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == j) myv = bv, mye = be;
    if (j == 0) v0 = bv;
  }
  // gate weights in fp32; sums over the slots in slot order
  float den = 0.f, num = 0.f;
  if (scoring == FL_SOFTMAX) {
    const float lmax = v0;
    num = expf(myv - lmax);
    if (renorm) {
      for (int j = 0; j < k; ++j) den += __shfl_sync(0xffffffffu, num, j);
    } else {
      float part = 0.f;
#pragma unroll
      for (int i = 0; i < kPer; ++i)
        if (lane + 32 * i < E) part += expf(v[i] - lmax);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      den = part;
    }
  } else {
    num = 1.f / (1.f + expf(-myv));
    if (renorm)
      for (int j = 0; j < k; ++j) den += __shfl_sync(0xffffffffu, num, j);
    else
      den = 1.f;
  }
  myw = num / den * scale;
  return __any_sync(0xffffffffu, bad) != 0;
}

template <int kPer>
__global__ void k_moe_route(const float* __restrict__ logits, int M, int E, int k, int scoring, int renorm,
                            float scale, int32_t* __restrict__ ids, float* __restrict__ wts,
                            int32_t* __restrict__ status) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= M) return;
  int mye;
  float myw;
  const bool bad = route_token<kPer>(logits + static_cast<size_t>(t) * E, E, k, scoring, renorm, scale, lane, mye, myw);
  if (bad && lane == 0) set_status(status, FL_ERR_DEVICE_CHECK, t);
  if (lane < k) {
    ids[static_cast<size_t>(t) * k + lane] = mye;
    wts[static_cast<size_t>(t) * k + lane] = myw;
  }
}

__device__ __forceinline__ bool better_d(double v, int e, double bv, int be) {
  return v > bv || (v == bv && e < be);
}

// Warp-wide argmax under better_d: every lane ends with the winner.
__device__ __forceinline__ void warp_best(double& bv, int& be) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const double ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oe = __shfl_xor_sync(0xffffffffu, be, o);
    if (better_d(ov, oe, bv, be)) bv = ov, be = oe;
  }
}

// DeepSeek-V3 style routing, one warp per token (kRouteWarps per block): the
// affinities s_e = sigma(l_e) plus the selection bias b_e give the keys; the
// experts come in n_group runs of E/n_group, a group scores the sum of its
// two largest keys, the topk_group best groups are kept, and the top-k keys
// among their experts are chosen (ties: lower index; slots by descending
// key).  Weights use the unbiased s_e, renormalised if asked, times scale.
// Keys and group scores are doubles in shared memory, [warp][E + n_group],
// so that the choice is taken in double precision.
constexpr int kRouteWarps = 2;
__global__ void k_moe_route_keyed(const float* __restrict__ logits, const float* __restrict__ bias, int M, int E,
                                  int k, int renorm, int n_group, int topk_group, float scale,
                                  int32_t* __restrict__ ids, float* __restrict__ wts,
                                  int32_t* __restrict__ status) {
  extern __shared__ double rk_smem[];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int t = blockIdx.x * kRouteWarps + wib;
  if (t >= M) return;   // whole warps leave; the kernel has no block-wide barrier
  double* key = rk_smem + static_cast<size_t>(wib) * (E + n_group);
  double* gsc = key + E;
  const float* l = logits + static_cast<size_t>(t) * E;
  int bad = 0;
  for (int e = lane; e < E; e += 32) {
    float x = l[e];
    if (isnan(x)) bad = 1, x = -INFINITY;
    double kv = 1.0 / (1.0 + exp(-static_cast<double>(x))) + (bias ? static_cast<double>(bias[e]) : 0.0);
    if (isnan(kv)) bad = 1, kv = -INFINITY;   // a NaN bias: never chosen before a number
    key[e] = kv;
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(status, FL_ERR_DEVICE_CHECK, t);
  __syncwarp();
  const int gsz = E / n_group;
  for (int g = lane; g < n_group; g += 32) {
    double b1 = -INFINITY, b2 = -INFINITY;
    for (int i = 0; i < gsz; ++i) {
      const double v = key[g * gsz + i];
      if (v > b1) {
        b2 = b1;
        b1 = v;
      } else if (v > b2) {
        b2 = v;
      }
    }
    const double gs = gsz >= 2 ? b1 + b2 : b1;
    gsc[g] = isnan(gs) ? -INFINITY : gs;   // inf + -inf from infinite biases
  }
  __syncwarp();
  // kept groups: bit i of lane's mask = group lane + 32 i
  uint32_t kept = 0;
  for (int j = 0; j < topk_group; ++j) {
    double bv = -INFINITY;
    int bg = 0x7fffffff;
    for (int i = 0; i < 32 && lane + 32 * i < n_group; ++i) {
      const int g = lane + 32 * i;
      if (!((kept >> i) & 1u) && better_d(gsc[g], g, bv, bg)) bv = gsc[g], bg = g;
    }
    warp_best(bv, bg);
    if ((bg & 31) == lane) kept |= 1u << (bg >> 5);
  }
  __syncwarp();
  for (int i = 0; i < 32 && lane + 32 * i < n_group; ++i) gsc[lane + 32 * i] = ((kept >> i) & 1u) ? 1.0 : 0.0;
  __syncwarp();
  // experts: bit i of lane's mask = expert lane + 32 i
  uint32_t taken = 0;
  int sele[32];   // k <= 32 (checked on the host)
  for (int j = 0; j < k; ++j) {
    double bv = -INFINITY;
    int be = 0x7fffffff;
    for (int i = 0; i < 32 && lane + 32 * i < E; ++i) {
      const int e = lane + 32 * i;
      if (((taken >> i) & 1u) || gsc[e / gsz] == 0.0) continue;
      if (better_d(key[e], e, bv, be)) bv = key[e], be = e;
    }
    warp_best(bv, be);
    // the host checked k <= topk_group * E / n_group, so an untaken eligible
    // expert always exists; be stays in range whatever the keys are
    if (be >= E) be = 0;
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    sele[j] = be;
  }
  if (lane == 0) {
    double sg[32], den = 0.0;
    for (int j = 0; j < k; ++j) {
      float x = l[sele[j]];
      if (isnan(x)) x = -INFINITY;
      sg[j] = 1.0 / (1.0 + exp(-static_cast<double>(x)));
      den += sg[j];
    }
    for (int j = 0; j < k; ++j) {
      ids[static_cast<size_t>(t) * k + j] = sele[j];
      wts[static_cast<size_t>(t) * k + j] = static_cast<float>((renorm ? sg[j] / den : sg[j]) * scale);
    }
  }
}

// ------------------------------------------------------------------ permute
struct PermuteArgs {
  const int32_t* ids;
  const float* wts;
  int M, E, k, TT13, TT2;       // TT: row tiles of the grouped kernels' outputs
  int G13, G2;                  // groups along K of the two grouped kernels
  int has_shared;
  int seg_rows;                 // positions per segment (32: grouped rows kernels, 128: grouped GEMM)
  int32_t* offsets;             // [E+1]
  int32_t* perm;                // [M*k]
  int32_t* inv;                 // [M*k]
  int32_t* tok_of_pos;          // [M*k + M]
  float* wpos;                  // [M*k + M]
  int32_t* seg_e;               // [nseg_max]
  int32_t* seg_pos;
  int32_t* seg_n;
  MoePlan* plan;
  int32_t* cnt13;               // counters to zero: [nseg_max * TT13 * 8]
  int32_t* cnt2;                // [nseg_max * TT2 * 8]
  int32_t* user_offsets;        // optional copies
  int32_t* user_perm;
};

__global__ void __launch_bounds__(1024, 1) k_moe_permute(const PermuteArgs a) {
  extern __shared__ int32_t psm[];
  pdl_wait();   // ids / weights come from k_moe_route
  const int E = a.E, n = a.M * a.k;
  int32_t* counts = psm;                       // [32][E]
  int32_t* local = counts + 32 * E;            // [n]
  int32_t* tot = local + n;                    // [E + 1]
  int32_t* nch = tot + (E + 1);                // [E + 1] segment starts
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < 32 * E; i += blockDim.x) counts[i] = 0;
  cta_sync();
  // per-warp stable ranks: warp w owns assignments [w*C, (w+1)*C)
  const int C = (n + 31) / 32;
  const int i0 = warp * C, i1 = min(n, i0 + C);
  for (int base = i0; base < i1; base += 32) {
    const int i = base + lane;
    const bool act = i < i1;
    const unsigned am = __ballot_sync(0xffffffffu, act);
    if (act) {
      const int e = a.ids[i];
      const unsigned mask = __match_any_sync(am, e);
      const int rank = __popc(mask & ((1u << lane) - 1u));
      const int before = counts[warp * E + e];
      local[i] = before + rank;
      __syncwarp(am);
      if (lane == __ffs(mask) - 1) counts[warp * E + e] = before + __popc(mask);
    }
    __syncwarp();
  }
  cta_sync();
  // totals, then per-expert base offsets for every warp
  for (int e = tid; e < E; e += blockDim.x) {
    int s = 0;
    for (int w = 0; w < 32; ++w) s += counts[w * E + e];
    tot[e] = s;
  }
  cta_sync();
  if (warp == 0) {
    // exclusive scans of the counts (-> offsets) and of the segment counts
    // (-> first segment of each expert): lane l takes experts [l*per, (l+1)*per)
    const int per = (E + 31) / 32, e0 = lane * per, e1 = min(E, e0 + per);
    int run = 0, seg = 0;
    for (int e = e0; e < e1; ++e) run += tot[e], seg += (tot[e] + a.seg_rows - 1) / a.seg_rows;
    int xr = run, xs = seg;   // inclusive warp scan, then shifted to exclusive
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int yr = __shfl_up_sync(0xffffffffu, xr, o), ys = __shfl_up_sync(0xffffffffu, xs, o);
      if (lane >= o) xr += yr, xs += ys;
    }
    int rbase = xr - run, sbase = xs - seg;
    for (int e = e0; e < e1; ++e) {
      const int c = tot[e];
      tot[e] = rbase;
      nch[e] = sbase;
      rbase += c;
      sbase += (c + a.seg_rows - 1) / a.seg_rows;
    }
    const int all_r = __shfl_sync(0xffffffffu, xr, 31), all_s = __shfl_sync(0xffffffffu, xs, 31);
    if (lane == 0) {
      tot[E] = all_r;
      nch[E] = all_s;
      const int nshared = a.has_shared ? (a.M + a.seg_rows - 1) / a.seg_rows : 0;
      a.plan->nseg = all_s + nshared;
      a.plan->U = (all_s + nshared) * a.TT13 * a.G13;   // == (all_s + nshared) * TT2 * G2
    }
  }
  cta_sync();
  for (int e = tid; e < E; e += blockDim.x) {
    int run = tot[e];
    for (int w = 0; w < 32; ++w) {
      const int c = counts[w * E + e];
      counts[w * E + e] = run;
      run += c;
    }
  }
  for (int e = tid; e <= E; e += blockDim.x) {
    a.offsets[e] = tot[e];
    if (a.user_offsets) a.user_offsets[e] = tot[e];
  }
  cta_sync();
  for (int i = tid; i < n; i += blockDim.x) {
    const int w = i / C;
    const int e = a.ids[i];
    const int pos = counts[w * E + e] + local[i];
    a.perm[pos] = i;
    a.inv[i] = pos;
    a.tok_of_pos[pos] = i / a.k;
    a.wpos[pos] = a.wts[i];
    if (a.user_perm) a.user_perm[pos] = i;
  }
  // shared expert: positions n + t hold token t with weight 1
  for (int t = tid; t < (a.has_shared ? a.M : 0); t += blockDim.x) {
    a.tok_of_pos[n + t] = t;
    a.wpos[n + t] = 1.f;
  }
  // segments
  for (int e = tid; e < E; e += blockDim.x) {
    const int c = tot[e + 1] - tot[e];
    for (int s = 0; s * a.seg_rows < c; ++s) {
      const int si = nch[e] + s;
      a.seg_e[si] = e;
      a.seg_pos[si] = tot[e] + s * a.seg_rows;
      a.seg_n[si] = min(a.seg_rows, c - s * a.seg_rows);
    }
  }
  if (a.has_shared) {
    const int ns = (a.M + a.seg_rows - 1) / a.seg_rows;
    for (int s = tid; s < ns; s += blockDim.x) {
      const int si = nch[E] + s;
      a.seg_e[si] = E;   // E denotes the shared expert
      a.seg_pos[si] = n + s * a.seg_rows;
      a.seg_n[si] = min(a.seg_rows, a.M - s * a.seg_rows);
    }
  }
  // zero the ticket counters the grouped rows kernels will use (the grouped
  // GEMM takes none: null)
  const int nseg = nch[E] + (a.has_shared ? (a.M + a.seg_rows - 1) / a.seg_rows : 0);
  if (a.cnt13) {
    for (int i = tid; i < nseg * a.TT13 * kConsumerWarps; i += blockDim.x) a.cnt13[i] = 0;
    for (int i = tid; i < nseg * a.TT2 * kConsumerWarps; i += blockDim.x) a.cnt2[i] = 0;
  }
}

// ------------------------------------------------------------------ grouped rows
// MODE 0: gate/up.  A unit is (segment, tile pair a, group g): super-blocks of
//         gate tile a and up tile a + I/128 of the segment's expert; the
//         segment's token rows of x.  Output h = silu(gate) * up, bf16.
// MODE 1: down.  A unit is (segment, tile, group) of W2; x rows = h rows of
//         the segment's positions.  Output out = w_pos * sum, fp32.
struct MoeRowsParams {
  const uint8_t* w;            // routed experts back to back (when wtab is null)
  const uint8_t* const* wtab;  // device table of E expert pointers, or null
  const uint8_t* w_shared;     // shared expert (or null)
  size_t wbytes;               // bytes of one expert's matrix
  size_t side_off;             // groups of 64: offset of an expert's side array from its base (0: none)
  const __nv_bfloat16* x;      // MODE 0: x [M, K]; MODE 1: h [pos, K]
  int K, G, TT;                // K = reduction length, G = K/128, TT = output tiles
  int up_off;                  // MODE 0: I/128
  int E, Nout;                 // Nout = output row length (I or H)
  const int32_t* seg_e;
  const int32_t* seg_pos;
  const int32_t* seg_n;
  const int32_t* tok_of_pos;
  const float* wpos;
  const MoePlan* plan;
  __nv_bfloat16* h;            // MODE 0 output [pos, I]
  float* out;                  // MODE 1 output [pos, H]
  float* part;                 // [2P][128][32][VALS] partial sums
  int32_t* cnt;                // [nseg * TT][8] tickets
  int32_t* status;
  int P, stages;
  uint32_t stage_bytes;
  // Decode (segments of 8) with plain routing: `logits` non-null.  Every CTA
  // then routes the M <= 8 tokens and builds the plan itself, in shared
  // memory at `sr_off` (no route or permute launch); the gate/up kernel's
  // CTAs also write the routing outputs below, each a slice of them.
  const float* logits;
  int M, k, scoring, renorm, has_shared;
  float scale;
  uint32_t sr_off;
  int32_t* ids;
  float* wts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv;
  int32_t* user_offsets;
  int32_t* user_perm;
  MoePlan* plan_out;
};

// Shared-memory words of the self-routed plan for n = M*k assignments.
__host__ __device__ constexpr int sr_words(int M, int k) { return 4 * (M * k) + 3 * (M * k + 1) + 2 * (M * k + M) + 4; }

// The plan of the decode build computed in every CTA (see MoeRowsParams):
// the routing of each token (one warp per token, the route kernel's
// arithmetic), then what the permute kernel builds for segments of 8.  An
// expert holds at most M <= 8 positions, so each chosen expert is one
// segment of its positions in assignment order, ascending by expert, and
// the shared expert's M positions are the last segment.  Returns the
// number of segments; `pv` receives the plan's arrays in shared memory.
struct PlanView {
  const int32_t* seg_e;
  const int32_t* seg_pos;
  const int32_t* seg_n;
  const int32_t* tok_of_pos;
  const float* wpos;
};

template <int kPer>
__device__ __forceinline__ int self_plan(const MoeRowsParams& p, int32_t* sm, bool write_outputs, PlanView& pv) {
  const int M = p.M, k = p.k, n = M * k, npos = n + (p.has_shared ? M : 0);
  const int tid = threadIdx.x, nth = blockDim.x, warp = tid >> 5, lane = tid & 31;
  int32_t* sids = sm;
  float* swts = reinterpret_cast<float*>(sids + n);
  int32_t* sexp = reinterpret_cast<int32_t*>(swts + n);   // expert of each position
  int32_t* spos = sexp + n;                              // position of each assignment
  int32_t* seg_e = spos + n;
  int32_t* seg_pos = seg_e + (n + 1);
  int32_t* seg_n = seg_pos + (n + 1);
  int32_t* tok = seg_n + (n + 1);
  float* wpos = reinterpret_cast<float*>(tok + (n + M));
  int32_t* misc = reinterpret_cast<int32_t*>(wpos + (n + M));
  int mye = 0;
  float myw = 0.f;
  if (warp < M) {
    const bool bad = route_token<kPer>(p.logits + static_cast<size_t>(warp) * p.E, p.E, k, p.scoring, p.renorm,
                                       p.scale, lane, mye, myw);
    if (bad && lane == 0 && blockIdx.x == 0) set_status(p.status, FL_ERR_DEVICE_CHECK, warp);
    if (lane < k) sids[warp * k + lane] = mye, swts[warp * k + lane] = myw;
  }
  // n <= 32: warp 0 sorts and cuts the segments in registers (for M = 1 from
  // its own picks, without waiting for the block); otherwise the block does
  // it through shared memory
  const bool one_warp = n <= 32;
  if (!(one_warp && M == 1)) cta_sync();
  if (one_warp) {
    if (warp == 0) {
      const bool act = lane < n;
      const int e = act ? (M == 1 ? mye : sids[lane]) : INT_MAX;
      const float w = act ? (M == 1 ? myw : swts[lane]) : 0.f;
      // stable counting sort: position = assignments of smaller experts +
      // earlier assignments of the same expert; segment = the number of
      // smaller chosen experts (each expert's first assignment counts them)
      const unsigned same = __match_any_sync(0xffffffffu, e);
      const int rank = __popc(same & ((1u << lane) - 1u));
      const bool first = act && rank == 0;
      const unsigned firsts = __ballot_sync(0xffffffffu, first);
      int less = 0, si = 0;
      for (int j = 0; j < n; ++j) {
        const int ej = __shfl_sync(0xffffffffu, e, j);
        less += ej < e;
        si += ((firsts >> j) & 1u) && ej < e;
      }
      const int pos = less + rank;
      if (act) {
        sids[lane] = e;
        swts[lane] = w;
        spos[lane] = pos;
        sexp[pos] = e;
        tok[pos] = lane / k;
        wpos[pos] = w;
        if (first) seg_e[si] = e, seg_pos[si] = pos, seg_n[si] = __popc(same);
      }
      if (lane < (p.has_shared ? M : 0)) tok[n + lane] = lane, wpos[n + lane] = 1.f;
      if (lane == 0) {
        const int nr = __popc(firsts);
        if (p.has_shared) seg_e[nr] = p.E, seg_pos[nr] = n, seg_n[nr] = M;
        misc[0] = nr + (p.has_shared ? 1 : 0);
      }
    }
    cta_sync();
  } else {
    // stable counting sort by expert: position = assignments of smaller
    // experts + earlier assignments of the same expert
    for (int i = tid; i < n; i += nth) {
      const int e = sids[i];
      int pos = 0;
      for (int j = 0; j < n; ++j) {
        const int ej = sids[j];
        pos += (ej < e) | ((ej == e) & (j < i));
      }
      spos[i] = pos;
      sexp[pos] = e;
      tok[pos] = i / k;
      wpos[pos] = swts[i];
    }
    for (int t = tid; t < (p.has_shared ? M : 0); t += nth) tok[n + t] = t, wpos[n + t] = 1.f;
    cta_sync();
    for (int q = tid; q < n; q += nth) {
      if (q > 0 && sexp[q] == sexp[q - 1]) continue;
      int si = 0;
      for (int r = 1; r <= q; ++r) si += sexp[r] != sexp[r - 1];
      int cnt = 1;
      while (q + cnt < n && sexp[q + cnt] == sexp[q]) ++cnt;
      seg_e[si] = sexp[q];
      seg_pos[si] = q;
      seg_n[si] = cnt;
    }
    if (tid == 0) {
      int nr = n > 0 ? 1 : 0;
      for (int r = 1; r < n; ++r) nr += sexp[r] != sexp[r - 1];
      if (p.has_shared) seg_e[nr] = p.E, seg_pos[nr] = n, seg_n[nr] = M;
      misc[0] = nr + (p.has_shared ? 1 : 0);
    }
  }
  if (write_outputs) {
    // each CTA writes a slice of the routing outputs
    const int g0 = blockIdx.x * nth + tid, gs = gridDim.x * nth;
    for (int i = g0; i < n; i += gs) {
      p.ids[i] = sids[i];
      p.wts[i] = swts[i];
      p.inv[i] = spos[i];
      p.perm[spos[i]] = i;
      if (p.user_perm) p.user_perm[spos[i]] = i;
    }
    for (int e = g0; e <= p.E; e += gs) {
      int off = 0;
      for (int j = 0; j < n; ++j) off += sids[j] < e;
      p.offsets[e] = off;
      if (p.user_offsets) p.user_offsets[e] = off;
    }
  }
  if (!one_warp) cta_sync();   // (the one-warp plan was published by its barrier)
  const int nseg = misc[0];
  if (write_outputs && blockIdx.x == 0 && tid == 0) {
    p.plan_out->nseg = nseg;
    p.plan_out->U = nseg * p.TT * p.G;
  }
  pv.seg_e = seg_e;
  pv.seg_pos = seg_pos;
  pv.seg_n = seg_n;
  pv.tok_of_pos = tok;
  pv.wpos = wpos;
  (void)npos;
  return nseg;
}

template <int MODE>
struct MoeIO {
  static constexpr int kSB = MODE == 0 ? 2 : 1;     // super-blocks per unit
  static constexpr int kVals = MODE == 0 ? 2 : 1;   // partial values per element
};

__device__ __forceinline__ int unit_begin_d(int c, int U, int P) {
  return static_cast<int>(static_cast<long long>(c) * U / P);
}
__device__ __forceinline__ int cta_of_unit_d(int u, int U, int P) {
  return static_cast<int>((static_cast<long long>(u + 1) * P - 1) / U);
}

// Output of one finished (segment, tile) for the warp's 16 rows.
template <int MODE, int kNT>
__device__ __forceinline__ void emit(const MoeRowsParams& p, int seg, int tile, int warp, int lane,
                                     const float (&tg)[kNT][4], const float (&tu)[kNT][4]) {
  const int gid = lane >> 2, tig = lane & 3;
  const int pos0 = p.seg_pos[seg], nt_ok = p.seg_n[seg];
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int m = nt * 8 + 2 * tig + (e & 1);
      const int row = tile * kRowTile + warp * 16 + gid + (e >> 1) * 8;
      if (m >= nt_ok) continue;
      const size_t o = static_cast<size_t>(pos0 + m) * p.Nout + row;
      if (MODE == 0) {
        const float g = tg[nt][e];
        p.h[o] = __float2bfloat16_rn(g / (1.f + expf(-g)) * tu[nt][e]);
      } else {
        p.out[o] = p.wpos[pos0 + m] * tg[nt][e];
      }
    }
}

template <int MODE, int kNT>
__device__ __forceinline__ float* slot_ptr(const MoeRowsParams& p, int c, bool second, int warp) {
  constexpr size_t kSlot = static_cast<size_t>(kRowTile) * (8 * kNT) * MoeIO<MODE>::kVals;
  return p.part + (static_cast<size_t>(2 * c + (second ? 1 : 0))) * kSlot +
         static_cast<size_t>(warp) * 16 * (8 * kNT) * MoeIO<MODE>::kVals;
}

template <int MODE, int kNT>
__device__ __forceinline__ void ticket(const MoeRowsParams& p, int U, int Pe, int gt, int warp, int lane) {
  constexpr int Mp = 8 * kNT;
  constexpr int V = MoeIO<MODE>::kVals;
  const int tu0 = gt * p.G, tu1 = (gt + 1) * p.G;
  __syncwarp();
  const int cf = cta_of_unit_d(tu0, U, Pe), cl = cta_of_unit_d(tu1 - 1, U, Pe);
  int last = 0;
  if (lane == 0) {
    // one acq_rel atomic: release of the warp's partials (ordered before it
    // by the __syncwarp), acquire of everyone else's by the last arriver
    last = atom_add_acq_rel_gpu(&p.cnt[gt * kConsumerWarps + warp], 1) == cl - cf;
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  const int seg = gt / p.TT, tile = gt - seg * p.TT;
  const int gid = lane >> 2, tig = lane & 3;
  float tg[kNT][4], tu[kNT][4];
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) tg[nt][e] = 0.f, tu[nt][e] = 0.f;
  // the sharers' partials, added in CTA order (deterministic); the loads of
  // a batch of kB sharers are all issued before the first add, so the last
  // arriver pays about one L2 round trip per batch, not one per sharer
  constexpr int kB = 4;
  for (int cb = cf; cb <= cl; cb += kB) {
    float4 buf[kB][kNT][2];
#pragma unroll
    for (int b = 0; b < kB; ++b) {
      const int cc = cb + b;
      if (cc > cl) break;
      const bool second = gt != unit_begin_d(cc, U, Pe) / p.G;
      const float* sp = slot_ptr<MODE, kNT>(p, cc, second, warp);
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const float* q = sp + ((gid + 8 * hh) * Mp + nt * 8 + 2 * tig) * V;
          if (V == 2) {
            buf[b][nt][hh] = __ldcg(reinterpret_cast<const float4*>(q));
          } else {
            const float2 v = __ldcg(reinterpret_cast<const float2*>(q));
            buf[b][nt][hh] = make_float4(v.x, v.y, 0.f, 0.f);
          }
        }
    }
#pragma unroll
    for (int b = 0; b < kB; ++b) {
      if (cb + b > cl) break;
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const float4 v = buf[b][nt][hh];
          if (V == 2) {
            tg[nt][2 * hh] += v.x, tu[nt][2 * hh] += v.y, tg[nt][2 * hh + 1] += v.z, tu[nt][2 * hh + 1] += v.w;
          } else {
            tg[nt][2 * hh] += v.x, tg[nt][2 * hh + 1] += v.y;
          }
        }
    }
  }
  emit<MODE, kNT>(p, seg, tile, warp, lane, tg, tu);
  if (lane == 0) p.cnt[gt * kConsumerWarps + warp] = 0;
}

template <int MODE, int kNT>
__device__ __forceinline__ bool store(const MoeRowsParams& p, int gt, int c, int u0, int u1, int warp,
                                      int lane, const float (&tg)[kNT][4], const float (&tu)[kNT][4]) {
  constexpr int Mp = 8 * kNT;
  constexpr int V = MoeIO<MODE>::kVals;
  const int tu0 = gt * p.G, tu1 = (gt + 1) * p.G;
  if (tu0 >= u0 && tu1 <= u1) {
    const int seg = gt / p.TT;
    emit<MODE, kNT>(p, seg, gt - seg * p.TT, warp, lane, tg, tu);
    return false;
  }
  const int gid = lane >> 2, tig = lane & 3;
  float* sp = slot_ptr<MODE, kNT>(p, c, gt != u0 / p.G, warp);
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float* q = sp + ((gid + 8 * hh) * Mp + nt * 8 + 2 * tig) * V;
      if (V == 2)
        __stcg(reinterpret_cast<float4*>(q),
               make_float4(tg[nt][2 * hh], tu[nt][2 * hh], tg[nt][2 * hh + 1], tu[nt][2 * hh + 1]));
      else
        __stcg(reinterpret_cast<float2*>(q), make_float2(tg[nt][2 * hh], tg[nt][2 * hh + 1]));
    }
  return true;
}

// Everything after the plan: the unit range of this CTA, the producer warp
// and the consumer warps.
template <int MODE, bool G64, int kNT>
__device__ __forceinline__ void rows_run(const MoeRowsParams& p, const int U, uint8_t* smem, uint64_t* full,
                                         uint64_t* empty) {
  constexpr int SB = MoeIO<MODE>::kSB;
  constexpr int kSegRowsK = 8 * kNT;
  constexpr int XS = G64 ? 2 : 1;   // accumulator chains per super-block: one per 64-column group
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  // the work is split over min(P, U) CTAs, so that every working CTA owns at
  // least one unit (the ticket hand-off counts on it); the rest retire
  const int Pe = U < p.P ? U : p.P;
  if (c >= Pe) return;
  const int u0 = unit_begin_d(c, U, Pe), u1 = unit_begin_d(c + 1, U, Pe);
  const int TG = p.TT * p.G;
  const uint32_t xoff = SB * kSbBytes;

  if (warp == kConsumerWarps) {
    // ---------------- producer: super-block(s) + the segment's x rows
    const uint64_t pol = policy_evict_first();
    // MODE 1: the weights of the first stages before the wait (see rows_kernel)
    const int npre = MODE == 1 ? min(u1 - u0, p.stages) : 0;
    int s = 0, fills = 0;
    uint32_t ph = 0;
    // weights of (row tile, group) of expert e into stage `slot`, by lane 0
    auto issue_w = [&](int e, int tile, int g, int nt_ok, int slot) {
      // a bad table entry (recorded) skips the weight copy: the stage then
      // completes on its activations alone and its result is garbage
      const uint8_t* base = e == p.E ? p.w_shared : expert_base(p.w, p.wtab, p.wbytes, e, p.status);
      uint8_t* st = smem + static_cast<size_t>(slot) * p.stage_bytes;
      mbar_arrive_expect_tx(&full[slot],
                            static_cast<uint32_t>((base ? SB * (kSbBytes + (G64 ? kSbSide : 0)) : 0) + nt_ok * 256));
      if (base) {
        const size_t u_a = static_cast<size_t>(tile) * p.G + g, u_b = static_cast<size_t>(tile + p.up_off) * p.G + g;
        bulk_g2s_hint(st, base + u_a * kSbBytes, kSbBytes, &full[slot], pol);
        if (SB == 2) bulk_g2s_hint(st + kSbBytes, base + u_b * kSbBytes, kSbBytes, &full[slot], pol);
        if (G64) {   // side entries after the x rows
          uint8_t* sd = st + xoff + kSegRowsK * kXRowStride;
          bulk_g2s_hint(sd, base + p.side_off + u_a * kSbSide, kSbSide, &full[slot], pol);
          if (SB == 2) bulk_g2s_hint(sd + kSbSide, base + p.side_off + u_b * kSbSide, kSbSide, &full[slot], pol);
        }
      }
    };
    if (npre > 0) {
      if (lane == 0)
        for (int k = 0; k < npre; ++k) {
          const int u = u0 + k, seg = u / TG, rem = u - seg * TG, tile = rem / p.G;
          issue_w(p.seg_e[seg], tile, rem - tile * p.G, p.seg_n[seg], k);
        }
      __syncwarp();
    }
    if (MODE == 1) pdl_wait();   // h comes from the gate/up kernel
    for (int u = u0; u < u1; ++u) {
      if (fills >= p.stages && !mbar_wait(&empty[s], ph ^ 1u)) {
        if (lane == 0) set_status(p.status, FL_ERR_TIMEOUT, 11);
        for (int j = 0; j < p.stages; ++j) {
          const int nf = fills / p.stages + (j < fills % p.stages ? 1 : 0);
          if (nf > 0) mbar_wait(&full[j], static_cast<uint32_t>(nf - 1) & 1u);
        }
        return;
      }
      const int seg = u / TG, rem = u - seg * TG, tile = rem / p.G, g = rem - tile * p.G;
      const int e = p.seg_e[seg], pos0 = p.seg_pos[seg], nt_ok = p.seg_n[seg];
      uint8_t* st = smem + static_cast<size_t>(s) * p.stage_bytes;
      if (lane == 0 && fills >= npre) issue_w(e, tile, g, nt_ok, s);
      __syncwarp();
      if (lane < nt_ok) {
        const int row = MODE == 0 ? p.tok_of_pos[pos0 + lane] : pos0 + lane;
        bulk_g2s(st + xoff + lane * kXRowStride, p.x + static_cast<size_t>(row) * p.K + g * kGroup, 256u, &full[s]);
      }
      ++fills;
      if (++s == p.stages) s = 0, ph ^= 1u;
    }
    return;
  }
  if (MODE == 1) pdl_wait();   // the consumers write out[] and the tickets only after the gate/up kernel

  // ---------------- consumers
  const int gid = lane >> 2, tig = lane & 3;
  const int r0 = warp * 16 + gid;
  float tg[kNT][4], tu[kNT][4];
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) tg[nt][e] = 0.f, tu[nt][e] = 0.f;
  int s = 0, owed0 = -1;
  uint32_t ph = 0;
  int gt = u0 / p.G;
  for (int u = u0; u < u1; ++u) {
    const int seg = u / TG;
    const int nt_ok = p.seg_n[seg];
    if (!mbar_wait(&full[s], ph)) {
      if (lane == 0) set_status(p.status, FL_ERR_TIMEOUT, 12);
      return;
    }
    const uint8_t* sb = smem + static_cast<size_t>(s) * p.stage_bytes;
    float ag[XS][kNT][4], au[XS][kNT][4];
    float s0g[XS], s1g[XS], s0u[XS], s1u[XS];
    const int ntiles = (nt_ok + 7) / 8;
    if constexpr (G64) {
      const uint8_t* sd = sb + xoff + kSegRowsK * kXRowStride;
      uint32_t z0[2], z1[2];
      unit_dot64<kNT, false>(sb, sd, sb + xoff, nt_ok, r0, gid, tig, ag, s0g, s1g, z0, z1, ntiles);
      if (SB == 2)
        unit_dot64<kNT, false>(sb + kSbBytes, sd + kSbSide, sb + xoff, nt_ok, r0, gid, tig, au, s0u, s1u, z0, z1,
                               ntiles);
    } else {
      uint32_t z0, z1;
      unit_dot<kNT, false>(sb, sb + xoff, nt_ok, r0, gid, tig, ag[0], s0g[0], s1g[0], z0, z1, ntiles);
      if (SB == 2)
        unit_dot<kNT, false>(sb + kSbBytes, sb + xoff, nt_ok, r0, gid, tig, au[0], s0u[0], s1u[0], z0, z1, ntiles);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
#pragma unroll
    for (int hh = 0; hh < XS; ++hh)
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        tg[nt][e] = fmaf(e < 2 ? s0g[hh] : s1g[hh], ag[hh][nt][e], tg[nt][e]);
        if (SB == 2) tu[nt][e] = fmaf(e < 2 ? s0u[hh] : s1u[hh], au[hh][nt][e], tu[nt][e]);
      }
    if (++s == p.stages) s = 0, ph ^= 1u;
    if ((u + 1) % p.G == 0 && u + 1 < u1) {
      if (store<MODE, kNT>(p, gt, c, u0, u1, warp, lane, tg, tu)) owed0 = gt;
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) tg[nt][e] = 0.f, tu[nt][e] = 0.f;
      ++gt;
    }
  }
  const bool owed1 = store<MODE, kNT>(p, gt, c, u0, u1, warp, lane, tg, tu);
  if (owed0 >= 0) ticket<MODE, kNT>(p, U, Pe, owed0, warp, lane);
  if (owed1) ticket<MODE, kNT>(p, U, Pe, gt, warp, lane);
}

template <int MODE, bool G64, int kNT>
__device__ __forceinline__ void rows_kernel(const MoeRowsParams& p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(p.stages) * p.stage_bytes);
  uint64_t* empty = full + p.stages;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_mbar_init();
  }
  cta_sync();
  // MODE 0 (gate/up) gets its plan (or, self-routed, the logits), segments
  // and x from the kernels before it, and lets the next kernel start only
  // once that wait is over.  So MODE 1 (down) starts after those have
  // completed: it reads the plan or the logits at once (plain loads: written
  // by kernels that completed before this one started) and requests its
  // first weights before its own wait; only h (from MODE 0) waits for the
  // previous kernel.
  if (MODE == 0) {
    pdl_wait();
    pdl_launch_dependents();
  } else {
    pdl_launch_dependents();
  }
  if (p.logits) {
    PlanView pv;
    int32_t* sm = reinterpret_cast<int32_t*>(smem + p.sr_off);
    const int nseg = p.E <= 128 ? self_plan<4>(p, sm, MODE == 0, pv) : self_plan<8>(p, sm, MODE == 0, pv);
    MoeRowsParams q = p;   // the plan arrays in shared memory
    q.seg_e = pv.seg_e;
    q.seg_pos = pv.seg_pos;
    q.seg_n = pv.seg_n;
    q.tok_of_pos = pv.tok_of_pos;
    q.wpos = pv.wpos;
    rows_run<MODE, G64, kNT>(q, nseg * p.TT * p.G, smem, full, empty);
    return;
  }
  rows_run<MODE, G64, kNT>(p, p.plan->U, smem, full, empty);
}

// Two CTAs per SM.
template <int MODE, bool G64>
__global__ void __launch_bounds__(kThreads, 2) k_moe_rows(const MoeRowsParams p) {
  rows_kernel<MODE, G64, kNT>(p);
}

// ------------------------------------------------------------------ combine
// Four columns per thread; each output sums its slots in slot order.
__global__ void k_moe_combine(const float* __restrict__ out, const int32_t* __restrict__ inv, int M, int k, int H,
                              int has_shared, __nv_bfloat16* __restrict__ y) {
  const int t = blockIdx.y;
  const int n = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (t >= M || n >= H) return;
  pdl_wait();
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < k; ++j) {
    const float4 v = *reinterpret_cast<const float4*>(out + static_cast<size_t>(inv[t * k + j]) * H + n);
    acc.x += v.x, acc.y += v.y, acc.z += v.z, acc.w += v.w;
  }
  if (has_shared) {
    const float4 v = *reinterpret_cast<const float4*>(out + static_cast<size_t>(M * k + t) * H + n);
    acc.x += v.x, acc.y += v.y, acc.z += v.z, acc.w += v.w;
  }
  const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 st;
  st.x = *reinterpret_cast<const uint32_t*>(&lo);
  st.y = *reinterpret_cast<const uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(y + static_cast<size_t>(t) * H + n) = st;
}

// ------------------------------------------------------------------ gather / SwiGLU (grouped-GEMM path)
// xp[pos] = x[token of pos], 16 bytes per thread (32-bit indices: the host
// checks npos * H / 8 < 2^31).
__global__ void k_moe_gather(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ tok_of_pos, int npos,
                             int H, __nv_bfloat16* __restrict__ xp) {
  pdl_wait();
  const int per_row = H / 8;
  const int total = npos * per_row;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const int pos = i / per_row, c = i - pos * per_row;
    const int t = tok_of_pos[pos];
    reinterpret_cast<uint4*>(xp + static_cast<size_t>(pos) * H)[c] =
        reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H)[c];
  }
}

// h[pos, i] = bf16(silu(gu[pos, i]) * gu[pos, I + i]), gate rows first; four
// columns per thread (32-bit indices: the host checks npos * I / 4 < 2^31).
__global__ void k_moe_swiglu(const float* __restrict__ gu, int npos, int I, __nv_bfloat16* __restrict__ h) {
  pdl_wait();
  const int q4 = I / 4;
  const int total = npos * q4;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const int pos = i / q4, c = (i - pos * q4) * 4;
    const float* row = gu + static_cast<size_t>(pos) * 2 * I;
    const float4 g = *reinterpret_cast<const float4*>(row + c);
    const float4 u = *reinterpret_cast<const float4*>(row + I + c);
    const __nv_bfloat162 lo = __floats2bfloat162_rn(g.x / (1.f + expf(-g.x)) * u.x, g.y / (1.f + expf(-g.y)) * u.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(g.z / (1.f + expf(-g.z)) * u.z, g.w / (1.f + expf(-g.w)) * u.w);
    uint2 st;
    st.x = *reinterpret_cast<const uint32_t*>(&lo);
    st.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(h + static_cast<size_t>(pos) * I + c) = st;
  }
}

// ------------------------------------------------------------------ host plan
size_t al(size_t v) { return (v + 255) / 256 * 256; }

struct MoeLayout {
  size_t plan, ids, wts, offsets, perm, inv, tok, wpos, sege, segp, segn, h, out, cnt13, cnt2, part13, part2, xp, gu,
      total;
  int nseg_max, P, stages13, stages2, gemm;
  uint32_t stage13, stage2;
};

// Many tokens per expert: the grouped steps run on the tensor-memory GEMM
// above 8 positions per expert on average, or from 4 when the hidden size is
// at least 4096.  Below that the rows kernels win, although an expert with
// more than 8 positions streams its weights once per segment of 8 (measured:
// at 4 positions per expert the GEMM takes 0.95 of the rows kernels' time on
// the DeepSeek-V3-shaped layer, H = 7168, and 1.28 times it on the
// Qwen3-shaped one, H = 2048).
bool moe_uses_gemm(int M, int E, int k, int H) {
  const long long n = static_cast<long long>(M) * k;
  return n > 8LL * E || (H >= 4096 && n >= 4LL * E);
}

bool moe_layout(int M, int E, int k, int H, int I, int has_shared, int sms, MoeLayout* L, bool g64 = false) {
  if (M < 1 || E < 1 || E > kMaxE || k < 1 || k > E || k > 32 || H < kGroup || I < kGroup || H % kGroup ||
      I % kGroup || sms < 1)
    return false;
  if (static_cast<long long>(M) * k > kMaxAssign) return false;
  const int n = M * k, npos = n + (has_shared ? M : 0);
  // segments of 8 positions (an expert with more streams its weights once
  // per segment)
  const int seg_rows = 8 * kNT;
  L->nseg_max = std::min(E, n) + (n + seg_rows - 1) / seg_rows + (has_shared ? (M + seg_rows - 1) / seg_rows : 0);
  L->P = 2 * sms;   // two CTAs per SM
  const int TT13 = I / kRowTile, TT2 = H / kRowTile;
  // everything after the counter region that the linear kernels keep zero
  // between calls: one workspace can serve calls of every entry point
  size_t o = kScratchOff;
  L->plan = o; o = al(o + sizeof(MoePlan));
  L->ids = o; o = al(o + 4ull * n);
  L->wts = o; o = al(o + 4ull * n);
  L->offsets = o; o = al(o + 4ull * (E + 1));
  L->perm = o; o = al(o + 4ull * n);
  L->inv = o; o = al(o + 4ull * n);
  L->tok = o; o = al(o + 4ull * npos);
  L->wpos = o; o = al(o + 4ull * npos);
  L->sege = o; o = al(o + 4ull * L->nseg_max);
  L->segp = o; o = al(o + 4ull * L->nseg_max);
  L->segn = o; o = al(o + 4ull * L->nseg_max);
  L->h = o; o = al(o + 2ull * npos * I);
  L->out = o; o = al(o + 4ull * npos * H);
  L->cnt13 = o; o = al(o + 4ull * L->nseg_max * TT13 * kConsumerWarps);
  L->cnt2 = o; o = al(o + 4ull * L->nseg_max * TT2 * kConsumerWarps);
  L->part13 = o; o = al(o + 4ull * 2 * L->P * kRowTile * 8 * kNT * 2);
  L->part2 = o; o = al(o + 4ull * 2 * L->P * kRowTile * 8 * kNT);
  L->gemm = moe_uses_gemm(M, E, k, H) ? 1 : 0;
  L->xp = o; o = al(o + (L->gemm ? 2ull * npos * H : 0));
  L->gu = o; o = al(o + (L->gemm ? 4ull * npos * 2 * I : 0));
  L->total = o;
  const int side = g64 ? kSbSide : 0;
  L->stage13 = static_cast<uint32_t>((2 * (kSbBytes + side) + seg_rows * kXRowStride + 127) / 128 * 128);
  L->stage2 = static_cast<uint32_t>((kSbBytes + side + seg_rows * kXRowStride + 127) / 128 * 128);
  const unsigned budget = 100u * 1024u;   // two CTAs per SM
  L->stages13 = std::min(8, static_cast<int>(budget / L->stage13));
  L->stages2 = std::min(12, static_cast<int>(budget / L->stage2));
  return true;
}

// Launch with programmatic dependent launch: the kernel may start while the
// previous one in the stream finishes and must griddepcontrol.wait before
// touching what that kernel writes or reads.
template <typename K, typename... Args>
cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace

int fl_moe_gemm(const void* x, int npos, int K, const void* w, const void* const* wtab, const void* w_shared,
                size_t wbytes, size_t side_off, int E, int Nout, const int32_t* seg_e, const int32_t* seg_pos,
                const int32_t* seg_n, const int32_t* nseg, const float* wpos, float* out, int32_t* status,
                cudaStream_t s);

extern "C" int fl_moe_int4g_workspace(int M, int E, int k, int H, int I, int has_shared, size_t* out) {
  if (!out) return FL_ERR_ARG;
  MoeLayout L;
  if (!moe_layout(M, E, k, H, I, has_shared, flh::sm_count(), &L)) return FL_ERR_ARG;
  *out = L.total;
  return FL_OK;
}

// The routed layer; the experts are either back to back (w13, w2) or given
// by device tables of E pointers (w13tab, w2tab).
static int moe_layer(const void* x, const float* logits, int M, int H, int E, int k, int I,
                     const fl_moe_routing* routing, const void* w13, const void* w2, const void* const* w13tab,
                     const void* const* w2tab, const void* shared_w13, const void* shared_w2, void* y,
                     int32_t* topk_ids, float* topk_w, int32_t* expert_offsets, int32_t* perm, void* ws,
                     size_t ws_bytes, fl_stream_t stream, int group = kGroup) {
  if (!x || !logits || !y || !ws || !routing) return FL_ERR_ARG;
  if (group != kGroup && group != 2 * kGroup && group != kGroup / 2) return FL_ERR_UNSUPPORTED;
  const bool g64 = group == kGroup / 2;
  if ((shared_w13 == nullptr) != (shared_w2 == nullptr)) return FL_ERR_ARG;
  const int scoring = routing->scoring, renorm = routing->renorm;
  if (scoring != FL_SOFTMAX && scoring != FL_SIGMOID) return FL_ERR_ARG;
  const float scale = routing->routed_scale;
  if (!(scale > 0.f) || !(scale < INFINITY)) return FL_ERR_ARG;
  const int n_group = routing->n_group > 1 ? routing->n_group : 1;
  const int topk_group = routing->n_group > 1 ? routing->topk_group : 1;
  const bool keyed = routing->score_bias != nullptr || n_group > 1;
  if (keyed) {
    if (scoring != FL_SIGMOID || E < 1 || E % n_group || topk_group < 1 || topk_group > n_group) return FL_ERR_ARG;
    if (k > topk_group * (E / n_group)) return FL_ERR_ARG;
    if (routing->score_bias && !flh::aligned16(routing->score_bias)) return FL_ERR_ARG;
  }
  if (!flh::aligned16(x) || !flh::aligned16(w13) || !flh::aligned16(w2) || !flh::aligned16(y) ||
      (reinterpret_cast<uintptr_t>(w13tab) & 7u) || (reinterpret_cast<uintptr_t>(w2tab) & 7u) ||
      !flh::aligned16(ws) || (shared_w13 && (!flh::aligned16(shared_w13) || !flh::aligned16(shared_w2))))
    return FL_ERR_ARG;
  const int has_shared = shared_w13 != nullptr;
  MoeLayout L;
  if (!moe_layout(M, E, k, H, I, has_shared, flh::sm_count(), &L, g64)) return FL_ERR_ARG;
  if (ws_bytes < L.total) return FL_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* W = static_cast<uint8_t*>(ws);
  int32_t* status = reinterpret_cast<int32_t*>(W);
  int32_t* ids = topk_ids ? topk_ids : reinterpret_cast<int32_t*>(W + L.ids);
  float* wts = topk_w ? topk_w : reinterpret_cast<float*>(W + L.wts);
  MoePlan* plan = reinterpret_cast<MoePlan*>(W + L.plan);
  // one expert's matrices: super-blocks, then (groups of 64) their side entries
  const size_t n13 = static_cast<size_t>(2 * I / kRowTile) * (H / kGroup), n2 = static_cast<size_t>(H / kRowTile) * (I / kGroup);
  const size_t side13 = g64 ? n13 * kSbBytes : 0, side2 = g64 ? n2 * kSbBytes : 0;
  const size_t b13 = n13 * (kSbBytes + (g64 ? kSbSide : 0));
  const size_t b2 = n2 * (kSbBytes + (g64 ? kSbSide : 0));

  // Decode with plain routing (segments of 8, E <= 256): the grouped kernels
  // route the tokens themselves, so neither route nor permute is launched.
  // Their ticket counters then live in the counter region, which is zero
  // between calls, since no kernel before them can clear them.
  const size_t sr_cnt13 = 4ull * L.nseg_max * (I / kRowTile) * kConsumerWarps;
  const size_t sr_cnt2 = 4ull * L.nseg_max * (H / kRowTile) * kConsumerWarps;
  const bool sr = !keyed && !L.gemm && E <= 256 && M <= 8 &&
                  kTicketOff + sr_cnt13 + sr_cnt2 <= kScratchOff;
  // route
  if (!sr) {
    // plain launches: the logits come from whatever ran before this call
    if (keyed) {
      const size_t smem = static_cast<size_t>(kRouteWarps) * (E + n_group) * sizeof(double);
      k_moe_route_keyed<<<dim3((M + kRouteWarps - 1) / kRouteWarps), dim3(32 * kRouteWarps), smem, s>>>(
          logits, routing->score_bias, M, E, k, renorm, n_group, topk_group, scale, ids, wts, status);
    } else {
      const int warps = 8;
      const dim3 grid((M + warps - 1) / warps), block(32 * warps);
      if (E <= 128)
        k_moe_route<4><<<grid, block, 0, s>>>(logits, M, E, k, scoring, renorm, scale, ids, wts, status);
      else if (E <= 256)
        k_moe_route<8><<<grid, block, 0, s>>>(logits, M, E, k, scoring, renorm, scale, ids, wts, status);
      else if (E <= 512)
        k_moe_route<16><<<grid, block, 0, s>>>(logits, M, E, k, scoring, renorm, scale, ids, wts, status);
      else
        k_moe_route<32><<<grid, block, 0, s>>>(logits, M, E, k, scoring, renorm, scale, ids, wts, status);
    }
    if (cudaGetLastError() != cudaSuccess) return FL_ERR_CUDA;
  }
  // permute
  if (!sr) {
    PermuteArgs a;
    a.ids = ids;
    a.wts = wts;
    a.M = M;
    a.E = E;
    a.k = k;
    a.TT13 = I / kRowTile;
    a.TT2 = H / kRowTile;
    a.G13 = H / kGroup;
    a.G2 = I / kGroup;
    a.has_shared = has_shared;
    a.seg_rows = L.gemm ? 128 : 8 * kNT;
    a.offsets = reinterpret_cast<int32_t*>(W + L.offsets);
    a.perm = reinterpret_cast<int32_t*>(W + L.perm);
    a.inv = reinterpret_cast<int32_t*>(W + L.inv);
    a.tok_of_pos = reinterpret_cast<int32_t*>(W + L.tok);
    a.wpos = reinterpret_cast<float*>(W + L.wpos);
    a.seg_e = reinterpret_cast<int32_t*>(W + L.sege);
    a.seg_pos = reinterpret_cast<int32_t*>(W + L.segp);
    a.seg_n = reinterpret_cast<int32_t*>(W + L.segn);
    a.plan = plan;
    a.cnt13 = L.gemm ? nullptr : reinterpret_cast<int32_t*>(W + L.cnt13);
    a.cnt2 = L.gemm ? nullptr : reinterpret_cast<int32_t*>(W + L.cnt2);
    a.user_offsets = expert_offsets;
    a.user_perm = perm;
    const size_t smem = 4ull * (32 * E + M * k + 2 * (E + 1));
    static bool attr_done[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
      if (cudaFuncSetAttribute(k_moe_permute, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) !=
          cudaSuccess)
        return FL_ERR_CUDA;
      attr_done[dev] = true;
    }
    if (smem > 227 * 1024) return FL_ERR_UNSUPPORTED;
    if (launch_pdl(k_moe_permute, dim3(1), dim3(1024), smem, s, a) != cudaSuccess) return FL_ERR_CUDA;
  }
  const int n = M * k, npos = n + (has_shared ? M : 0);
  if (L.gemm) {
    // the element-wise kernels index with 32 bits
    if (static_cast<long long>(npos) * (H / 8) >= (1LL << 31) || static_cast<long long>(npos) * (I / 4) >= (1LL << 31))
      return FL_ERR_UNSUPPORTED;
    const int32_t* sege = reinterpret_cast<const int32_t*>(W + L.sege);
    const int32_t* segp = reinterpret_cast<const int32_t*>(W + L.segp);
    const int32_t* segn = reinterpret_cast<const int32_t*>(W + L.segn);
    const int32_t* nseg = reinterpret_cast<const int32_t*>(W + L.plan);   // MoePlan::nseg
    __nv_bfloat16* xp = reinterpret_cast<__nv_bfloat16*>(W + L.xp);
    float* gu = reinterpret_cast<float*>(W + L.gu);
    __nv_bfloat16* h = reinterpret_cast<__nv_bfloat16*>(W + L.h);
    const int sms = flh::sm_count();
    if (launch_pdl(k_moe_gather, dim3(4 * sms), dim3(256), 0, s, static_cast<const __nv_bfloat16*>(x),
                   reinterpret_cast<const int32_t*>(W + L.tok), npos, H, xp) != cudaSuccess)
      return FL_ERR_CUDA;
    int rc = fl_moe_gemm(xp, npos, H, w13, w13tab, shared_w13, b13, side13, E, 2 * I, sege, segp, segn, nseg,
                         nullptr, gu, status, s);
    if (rc != FL_OK) return rc;
    if (launch_pdl(k_moe_swiglu, dim3(4 * sms), dim3(256), 0, s, static_cast<const float*>(gu), npos, I, h) !=
        cudaSuccess)
      return FL_ERR_CUDA;
    rc = fl_moe_gemm(h, npos, I, w2, w2tab, shared_w2, b2, side2, E, H, sege, segp, segn, nseg,
                     reinterpret_cast<const float*>(W + L.wpos), reinterpret_cast<float*>(W + L.out), status, s);
    if (rc != FL_OK) return rc;
  }
  // grouped gate/up + SwiGLU, then grouped down
  for (int mode = 0; mode < 2 && !L.gemm; ++mode) {
    MoeRowsParams p;
    p.w = static_cast<const uint8_t*>(mode == 0 ? w13 : w2);
    p.wtab = reinterpret_cast<const uint8_t* const*>(mode == 0 ? w13tab : w2tab);
    p.w_shared = static_cast<const uint8_t*>(mode == 0 ? shared_w13 : shared_w2);
    p.wbytes = mode == 0 ? b13 : b2;
    p.side_off = mode == 0 ? side13 : side2;
    p.x = mode == 0 ? static_cast<const __nv_bfloat16*>(x) : reinterpret_cast<const __nv_bfloat16*>(W + L.h);
    p.K = mode == 0 ? H : I;
    p.G = p.K / kGroup;
    p.TT = mode == 0 ? I / kRowTile : H / kRowTile;
    p.up_off = I / kRowTile;
    p.E = E;
    p.Nout = mode == 0 ? I : H;
    p.seg_e = reinterpret_cast<const int32_t*>(W + L.sege);
    p.seg_pos = reinterpret_cast<const int32_t*>(W + L.segp);
    p.seg_n = reinterpret_cast<const int32_t*>(W + L.segn);
    p.tok_of_pos = reinterpret_cast<const int32_t*>(W + L.tok);
    p.wpos = reinterpret_cast<const float*>(W + L.wpos);
    p.plan = plan;
    p.h = reinterpret_cast<__nv_bfloat16*>(W + L.h);
    p.out = reinterpret_cast<float*>(W + L.out);
    p.part = reinterpret_cast<float*>(W + (mode == 0 ? L.part13 : L.part2));
    p.cnt = reinterpret_cast<int32_t*>(sr ? W + kTicketOff + (mode == 0 ? 0 : sr_cnt13)
                                          : W + (mode == 0 ? L.cnt13 : L.cnt2));
    p.status = status;
    p.P = L.P;
    p.stages = mode == 0 ? L.stages13 : L.stages2;
    p.stage_bytes = mode == 0 ? L.stage13 : L.stage2;
    size_t smem = static_cast<size_t>(p.stages) * p.stage_bytes + 2 * p.stages * sizeof(uint64_t);
    p.logits = sr ? logits : nullptr;
    p.M = M;
    p.k = k;
    p.scoring = scoring;
    p.renorm = renorm;
    p.has_shared = has_shared;
    p.scale = scale;
    p.sr_off = static_cast<uint32_t>((smem + 15) / 16 * 16);
    p.ids = ids;
    p.wts = wts;
    p.offsets = reinterpret_cast<int32_t*>(W + L.offsets);
    p.perm = reinterpret_cast<int32_t*>(W + L.perm);
    p.inv = reinterpret_cast<int32_t*>(W + L.inv);
    p.user_offsets = expert_offsets;
    p.user_perm = perm;
    p.plan_out = plan;
    if (sr) smem = p.sr_off + 4ull * sr_words(M, k);
    static bool attr_done[4][64] = {{false}};
    int dev = 0;
    cudaGetDevice(&dev);
    using KFn = void (*)(MoeRowsParams);
    static const KFn kerns[4] = {k_moe_rows<0, false>, k_moe_rows<1, false>, k_moe_rows<0, true>,
                                 k_moe_rows<1, true>};
    const int ki = 2 * (g64 ? 1 : 0) + mode;
    const KFn kern = kerns[ki];
    if (dev >= 0 && dev < 64 && !attr_done[ki][dev]) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) != cudaSuccess)
        return FL_ERR_CUDA;
      attr_done[ki][dev] = true;
    }
    if (launch_pdl(kern, dim3(L.P), dim3(kThreads), smem, s, p) != cudaSuccess) return FL_ERR_CUDA;
  }
  // combine
  if (launch_pdl(k_moe_combine, dim3((H / 4 + 255) / 256, M), dim3(256), 0, s,
                 reinterpret_cast<const float*>(W + L.out), reinterpret_cast<const int32_t*>(W + L.inv), M, k, H,
                 has_shared, static_cast<__nv_bfloat16*>(y)) != cudaSuccess)
    return FL_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? FL_OK : FL_ERR_CUDA;
}

extern "C" int fl_moe_int4g_ex(const void* x, const float* logits, int M, int H, int E, int k, int I,
                               const fl_moe_routing* routing, const void* w13, const void* w2,
                               const void* shared_w13, const void* shared_w2, void* y, int32_t* topk_ids,
                               float* topk_w, int32_t* expert_offsets, int32_t* perm, void* ws, size_t ws_bytes,
                               fl_stream_t stream) {
  if (!w13 || !w2) return FL_ERR_ARG;
  return moe_layer(x, logits, M, H, E, k, I, routing, w13, w2, nullptr, nullptr, shared_w13, shared_w2, y, topk_ids,
                   topk_w, expert_offsets, perm, ws, ws_bytes, stream);
}

extern "C" int fl_moe_int4g_g(const void* x, const float* logits, int M, int H, int E, int k, int I,
                              const fl_moe_routing* routing, int group, const void* w13, const void* w2,
                              const void* shared_w13, const void* shared_w2, void* y, int32_t* topk_ids,
                              float* topk_w, int32_t* expert_offsets, int32_t* perm, void* ws, size_t ws_bytes,
                              fl_stream_t stream) {
  if (!w13 || !w2) return FL_ERR_ARG;
  return moe_layer(x, logits, M, H, E, k, I, routing, w13, w2, nullptr, nullptr, shared_w13, shared_w2, y, topk_ids,
                   topk_w, expert_offsets, perm, ws, ws_bytes, stream, group);
}

extern "C" int fl_moe_int4g_ptrs(const void* x, const float* logits, int M, int H, int E, int k, int I,
                                 const fl_moe_routing* routing, const void* const* w13, const void* const* w2,
                                 const void* shared_w13, const void* shared_w2, void* y, int32_t* topk_ids,
                                 float* topk_w, int32_t* expert_offsets, int32_t* perm, void* ws, size_t ws_bytes,
                                 fl_stream_t stream) {
  if (!w13 || !w2) return FL_ERR_ARG;
  return moe_layer(x, logits, M, H, E, k, I, routing, nullptr, nullptr, w13, w2, shared_w13, shared_w2, y, topk_ids,
                   topk_w, expert_offsets, perm, ws, ws_bytes, stream);
}

extern "C" int fl_moe_int4g(const void* x, const float* logits, int M, int H, int E, int k, int I, int scoring,
                            int renorm, const void* w13, const void* w2, const void* shared_w13,
                            const void* shared_w2, void* y, int32_t* topk_ids, float* topk_w,
                            int32_t* expert_offsets, int32_t* perm, void* ws, size_t ws_bytes,
                            fl_stream_t stream) {
  fl_moe_routing r;
  r.scoring = scoring;
  r.renorm = renorm;
  r.score_bias = nullptr;
  r.n_group = 1;
  r.topk_group = 1;
  r.routed_scale = 1.0f;
  return fl_moe_int4g_ex(x, logits, M, H, E, k, I, &r, w13, w2, shared_w13, shared_w2, y, topk_ids, topk_w,
                         expert_offsets, perm, ws, ws_bytes, stream);
}
