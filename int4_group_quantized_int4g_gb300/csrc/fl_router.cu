// f2: router projection of the routed MoE layer, logits = x . Wr^T.
//
// x bf16 [M, H] (the layer input), Wr bf16 [E, H] (one row per routed
// expert), logits fp32 [M, E], fp32 accumulation.  The router is the gate
// linear in front of the top-k choice of the MoE layers the fastllm README
// runs with --moe_experts (section "5. 其它参数"); in DeepSeek-V3-style models
// it projects the hidden state onto the E expert centroids.  The pages give
// no detail of it; the plain dense reading is taken.
//
// A dense contraction, so it runs on the tensor cores (mma.sync m16n8k16,
// bf16 in, fp32 accumulate): CTA tiles of 64 tokens x 64 experts, K in steps
// of 32 staged in shared memory with cp.async (double buffered) and read
// with ldmatrix.  Few tiles (decode: M small) split K over several CTAs so
// the whole GPU streams Wr; each split writes an fp32 partial tile and the
// last split of a tile to take its ticket adds them in split order
// (deterministic) and writes the logits.
#include "fl_common.cuh"

using namespace fl;

namespace {

constexpr int kBM = 64, kBN = 64, kBK = 32;
constexpr int kLd = kBK + 8;            // smem row stride (elements): conflict-free ldmatrix
constexpr int kThreads = 128;           // 4 warps, 2 x 2, each 32 tokens x 32 experts

struct RouterParams {
  const __nv_bfloat16* x;
  const __nv_bfloat16* w;
  float* logits;
  float* part;        // [tile][split][kBM][kBN]
  int32_t* cnt;       // [tile]
  int M, H, E, tilesN, S, ksteps;   // ksteps: kBK-steps per split
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  const uint32_t s = smem_u32(smem);
  const int n = valid ? 16 : 0;   // 0: zero-fill, nothing read
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

__global__ void __launch_bounds__(kThreads) k_router(const RouterParams p) {
  __shared__ __align__(128) __nv_bfloat16 sa[2][kBM * kLd];
  __shared__ __align__(128) __nv_bfloat16 sb[2][kBN * kLd];
  __shared__ int last_flag;
  const int tn = blockIdx.x, tm = blockIdx.y, split = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int m0 = tm * kBM, n0 = tn * kBN;
  const int kbeg = split * p.ksteps * kBK;
  const int kend = min(p.H, kbeg + p.ksteps * kBK);
  const int nsteps = (kend - kbeg + kBK - 1) / kBK;

  // tile loads: 64 rows x 32 k of x and of Wr, 16 bytes per cp.async, 2 + 2 per thread
  auto load = [&](int buf, int k0) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int c = tid + i * kThreads, r = c >> 2, kc = (c & 3) * 8;
      const int m = m0 + r, e = n0 + r;
      const bool km = k0 + kc < kend;
      cp_async16(&sa[buf][r * kLd + kc], p.x + static_cast<size_t>(m < p.M ? m : 0) * p.H + (km ? k0 + kc : 0),
                 m < p.M && km);
      cp_async16(&sb[buf][r * kLd + kc], p.w + static_cast<size_t>(e < p.E ? e : 0) * p.H + (km ? k0 + kc : 0),
                 e < p.E && km);
    }
    cp_async_commit();
  };

  float acc[2][4][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][j][e] = 0.f;

  const int wm = (warp >> 1) * 32, wn = (warp & 1) * 32;
  if (nsteps > 0) load(0, kbeg);
  for (int st = 0; st < nsteps; ++st) {
    const int buf = st & 1;
    if (st + 1 < nsteps) {
      load(buf ^ 1, kbeg + (st + 1) * kBK);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kBK; kk += 16) {
      uint32_t a[2][4], b[2][4];
#pragma unroll
      for (int i = 0; i < 2; ++i)   // A: rows wm + 16i + (lane % 16), k kk + 8 (lane / 16)
        ldmatrix_x4(a[i], &sa[buf][(wm + 16 * i + (lane & 15)) * kLd + kk + 8 * (lane >> 4)]);
#pragma unroll
      for (int j = 0; j < 2; ++j)   // B: two n8 tiles per load: rows wn + 16j + (lane & 7) + 8 (lane >> 4), k kk + 8 ((lane >> 3) & 1)
        ldmatrix_x4(b[j], &sb[buf][(wn + 16 * j + (lane & 7) + 8 * (lane >> 4)) * kLd + kk + 8 * ((lane >> 3) & 1)]);
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          mma_bf16_16816(acc[i][j], a[i][0], a[i][1], a[i][2], a[i][3], b[j >> 1][2 * (j & 1)],
                         b[j >> 1][2 * (j & 1) + 1]);
    }
    __syncthreads();
  }

  // accumulator element (i, j, e): token wm + 16i + gid + 8(e >> 1), expert wn + 8j + 2tig + (e & 1)
  const int gid = lane >> 2, tig = lane & 3;
  if (p.S == 1) {
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int m = m0 + wm + 16 * i + gid + 8 * (e >> 1), n = n0 + wn + 8 * j + 2 * tig + (e & 1);
          if (m < p.M && n < p.E) p.logits[static_cast<size_t>(m) * p.E + n] = acc[i][j][e];
        }
    return;
  }
  const int tile = tm * p.tilesN + tn;
  float* mine = p.part + (static_cast<size_t>(tile) * p.S + split) * kBM * kBN;
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = wm + 16 * i + gid + 8 * h, c = wn + 8 * j + 2 * tig;
        __stcg(reinterpret_cast<float2*>(mine + r * kBN + c), make_float2(acc[i][j][2 * h], acc[i][j][2 * h + 1]));
      }
  __syncthreads();
  if (tid == 0) {
    fence_acq_rel_gpu();
    const int done = atomicAdd(&p.cnt[tile], 1);
    last_flag = done == p.S - 1;
    if (last_flag) fence_acq_rel_gpu();
  }
  __syncthreads();
  if (!last_flag) return;
  // last split of the tile: sum the partials in split order
  const float* base = p.part + static_cast<size_t>(tile) * p.S * kBM * kBN;
  for (int idx = tid; idx < kBM * kBN / 4; idx += kThreads) {
    float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sp = 0; sp < p.S; ++sp) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(base + static_cast<size_t>(sp) * kBM * kBN) + idx);
      s4.x += v.x, s4.y += v.y, s4.z += v.z, s4.w += v.w;
    }
    const int r = (4 * idx) / kBN, c = (4 * idx) % kBN;
    const int m = m0 + r;
    if (m < p.M) {
      const float vv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (n0 + c + q < p.E) p.logits[static_cast<size_t>(m) * p.E + n0 + c + q] = vv[q];
    }
  }
  if (tid == 0) p.cnt[tile] = 0;
}

struct RouterPlan {
  int tilesM, tilesN, S, ksteps;
  size_t cnt_off, part_off, total;
};

bool router_plan(int M, int H, int E, int sms, RouterPlan* pl) {
  if (M < 1 || H < 64 || H % 64 || E < 1 || E > 65536 || sms < 1) return false;
  pl->tilesM = (M + kBM - 1) / kBM;
  pl->tilesN = (E + kBN - 1) / kBN;
  if (pl->tilesM > 65535) return false;
  const int tiles = pl->tilesM * pl->tilesN;
  const int kst = H / kBK;
  int S = (2 * sms + tiles - 1) / tiles;   // about two CTAs per SM
  if (S < 1) S = 1;
  if (S > kst) S = kst;
  pl->ksteps = (kst + S - 1) / S;
  pl->S = (kst + pl->ksteps - 1) / pl->ksteps;   // every split has work
  // tickets in the shared counter region (zero between calls), partials after it
  if (static_cast<size_t>(tiles) * 4 > kScratchOff - kTicketOff) return false;
  pl->cnt_off = kTicketOff;
  pl->part_off = kScratchOff;
  pl->total = pl->S > 1 ? pl->part_off + 4ull * tiles * pl->S * kBM * kBN : pl->part_off;
  return true;
}

}  // namespace

extern "C" int fl_moe_router_logits_workspace(int M, int H, int E, size_t* out) {
  RouterPlan pl;
  if (!out || !router_plan(M, H, E, flh::sm_count(), &pl)) return FL_ERR_ARG;
  *out = pl.total;
  return FL_OK;
}

extern "C" int fl_moe_router_logits(const void* x, int M, int H, const void* w_router, int E, float* logits,
                                    void* ws, size_t ws_bytes, fl_stream_t stream) {
  if (!x || !w_router || !logits || !ws) return FL_ERR_ARG;
  if (!flh::aligned16(x) || !flh::aligned16(w_router) || !flh::aligned16(logits) || !flh::aligned16(ws))
    return FL_ERR_ARG;
  RouterPlan pl;
  if (!router_plan(M, H, E, flh::sm_count(), &pl)) return FL_ERR_ARG;
  if (ws_bytes < pl.total) return FL_ERR_WORKSPACE;
  RouterParams p;
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.w = static_cast<const __nv_bfloat16*>(w_router);
  p.logits = logits;
  p.part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + pl.part_off);
  p.cnt = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + pl.cnt_off);
  p.M = M;
  p.H = H;
  p.E = E;
  p.tilesN = pl.tilesN;
  p.S = pl.S;
  p.ksteps = pl.ksteps;
  k_router<<<dim3(pl.tilesN, pl.tilesM, pl.S), dim3(kThreads), 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError() == cudaSuccess ? FL_OK : FL_ERR_CUDA;
}
