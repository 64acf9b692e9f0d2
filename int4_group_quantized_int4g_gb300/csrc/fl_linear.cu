// a3: int4g decode linear, y = x . deq(W)^T for M <= 32 tokens.
//
// The weights (the interleaved layout, one 8512-byte super-block per 128 rows
// x one group) stream from HBM once.  FastLLM page, section 3.1: decode is
// memory-bound, so the 4-bit codes are read once and dequantized on the fly
// inside the matmul.  GB300 design:
//  * work = the T*G super-blocks.  Few row tiles: one thread-block cluster
//    per tile, its CTAs splitting the tile's groups (K), partial sums added
//    in rank 0's shared memory through distributed shared memory.  Many row
//    tiles: equal contiguous ranges of super-blocks, one per CTA (stream-K),
//    a tile shared by several CTAs finished by the last one to take its
//    ticket (no waiting; partials summed in CTA order, deterministic);
//  * one producer warp moves super-blocks into a ring of shared-memory stages
//    with 1-D bulk copies completing on mbarriers; the weights of the first
//    stages are requested before the wait on the previous kernel
//    (programmatic launch).  x: in cluster mode (M <= 8) the consumer warps
//    load the x rows of their CTA's K slice once, into an x region, while
//    they form the per-group token sums; otherwise the producer also copies
//    the matching 256-byte slices of every token row of x into each stage;
//  * 8 consumer warps each own 16 rows: 16 bytes of codes per lane and row
//    become 8 bf16 pairs (128 + q) with one LOP3 each, the A operand of
//    mma.sync m16n8k16 (the K order inside a group is permuted consistently
//    for A and B, which leaves the dot product unchanged); (128 + z) times
//    the group's sum of x is subtracted afterwards and the fp16 scale
//    applied to the fp32 group sum (M <= 16; larger M subtracts z per pair).
#include <atomic>
#include <mutex>

#include "fl_common.cuh"
#include "fl_rows.cuh"

using namespace fl;

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxTokens = 32;
constexpr size_t kMaxDynSmem = 227u * 1024u;   // the kernel's dynamic shared-memory limit
// Ticket counters live at a fixed offset with room for kMaxRowTiles row tiles,
// so that a workspace reused across shapes never finds another shape's
// scratch partial sums where its counters are (they must be zero on entry).
constexpr int kMaxRowTiles = 8192;  // N <= 1,048,576
static_assert(kMaxRowTiles == kTicketTiles && kConsumerWarps == kTicketWarps,
              "the decode counters are the shared ticket region");

struct RowsParams {
  const uint8_t* w;
  const uint8_t* side;   // groups of 64: the side array (the odd groups' scales and zeros), else null
  const __nv_bfloat16* x;
  __nv_bfloat16* y;
  float* part;       // [P + T][128][Mp] fp32 partial sums (slot = CTA + tile)
  int32_t* cnt;      // [T][8] tickets (zero between calls)
  int32_t* status;   // 16-byte status block
  int U;             // units = T * G
  int M, K, N, T, G, P;
  int stages;
  uint32_t stage_bytes;
  int csize;         // > 1: clusters of csize CTAs split one row tile over K (DSMEM reduction)
  uint32_t red_off;  // shared-memory offset of the cluster reduction barrier and buffer
  uint32_t zrow_off; // shared-memory offset of 256 zero bytes (x rows of absent tokens)
  unsigned long long red_wait_ns;  // bound of rank 0's wait for its peers' partial sums
  int withhold;      // test hook: the reduction barrier expects one arrival nobody makes
  const uint8_t* w_up;   // GLU: the up matrix (w is the gate); y receives h = silu(gate) * up
  // > 0 (cluster mode, M <= 8): the x rows of the CTA's whole K slice sit at
  // shared-memory offset xr_off, token m's at m * xr_stride, filled once by
  // the consumer warps; the stages then hold weights only.  0: each stage
  // carries its groups' x rows (kXRowStride apart), copied by the producer.
  int xr_stride;
  uint32_t xr_off;
};

// CTA c owns units [unit_begin(c), unit_begin(c+1)); cta_of_unit inverts it.
__host__ __device__ __forceinline__ int unit_begin(int c, int U, int P) {
  return static_cast<int>(static_cast<long long>(c) * U / P);
}
__host__ __device__ __forceinline__ int cta_of_unit(int u, int U, int P) {
  return static_cast<int>((static_cast<long long>(u + 1) * P - 1) / U);
}

// Partial sums of row tile T from CTA c go to slot c + T.  The slots are
// unique (the CTAs covering tile T precede those covering tile T+1) and those
// of one tile are contiguous, so its last CTA reads them as one block.
//
// store_tile: a row tile computed whole by this CTA is written to y as bf16;
// otherwise the warp's 16 x Mp partial sums go to the tile's slot and the
// function returns true (a ticket is owed, taken by ticket_tile after the
// main loop so that no warp waits on an atomic in the middle of its stream).
template <int NT>
__device__ __forceinline__ bool store_tile(const RowsParams& p, int T, int c, int u0, int u1, int warp, int lane,
                                           float (&tot)[NT][4]) {
  constexpr int Mp = 8 * NT;
  const int gid = lane >> 2, tig = lane & 3;
  const int tu0 = T * p.G, tu1 = (T + 1) * p.G;
  const int rbase = T * kRowTile + warp * 16;
  if (tu0 >= u0 && tu1 <= u1) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int n = rbase + gid + (e >> 1) * 8;
        const int m = nt * 8 + 2 * tig + (e & 1);
        if (n < p.N && m < p.M) p.y[static_cast<size_t>(m) * p.N + n] = __float2bfloat16_rn(tot[nt][e]);
      }
    }
    return false;
  }
  constexpr size_t kSlot = static_cast<size_t>(kRowTile) * Mp;   // floats per slot
  float* pp = p.part + static_cast<size_t>(c + T) * kSlot + warp * 16 * Mp;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    __stcg(reinterpret_cast<float2*>(pp + gid * Mp + nt * 8 + 2 * tig), make_float2(tot[nt][0], tot[nt][1]));
    __stcg(reinterpret_cast<float2*>(pp + (gid + 8) * Mp + nt * 8 + 2 * tig), make_float2(tot[nt][2], tot[nt][3]));
  }
  return true;
}

// Ticket for a row tile whose partials this warp stored; the last of the
// tile's CTAs to arrive sums all partials in CTA order and writes y.
template <int NT>
__device__ __forceinline__ void ticket_tile(const RowsParams& p, int T, int warp, int lane) {
  constexpr int Mp = 8 * NT;
  constexpr size_t kSlot = static_cast<size_t>(kRowTile) * Mp;
  const int tu0 = T * p.G, tu1 = (T + 1) * p.G;
  // the warp's partial stores are ordered before lane 0's ticket by the warp
  // barrier and published at GPU scope by the release half of lane 0's
  // acq_rel atomic; its acquire half gives the last arriver everyone else's
  __syncwarp();
  const int cf = cta_of_unit(tu0, p.U, p.P), cl = cta_of_unit(tu1 - 1, p.U, p.P);
  int last = 0;
  if (lane == 0) last = atom_add_acq_rel_gpu(&p.cnt[T * kConsumerWarps + warp], 1) == cl - cf;
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  const int np = cl - cf + 1;
  const int rbase = T * kRowTile + warp * 16;
  const float* base = p.part + static_cast<size_t>(cf + T) * kSlot + warp * 16 * Mp;
#pragma unroll
  for (int e4 = lane; e4 < 4 * Mp; e4 += 32) {
    // fixed summation order (CTA order) whatever order the loads complete in
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int j = 0;
    for (; j + 4 <= np; j += 4) {
      float4 v[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) v[t] = __ldcg(reinterpret_cast<const float4*>(base + (j + t) * kSlot) + e4);
#pragma unroll
      for (int t = 0; t < 4; ++t) acc.x += v[t].x, acc.y += v[t].y, acc.z += v[t].z, acc.w += v[t].w;
    }
    for (; j < np; ++j) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(base + j * kSlot) + e4);
      acc.x += v.x, acc.y += v.y, acc.z += v.z, acc.w += v.w;
    }
    const int row = (4 * e4) / Mp, m0 = (4 * e4) % Mp;
    const int n = rbase + row;
    if (n < p.N) {
      const float r[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
      for (int t = 0; t < 4; ++t)
        if (m0 + t < p.M) p.y[static_cast<size_t>(m0 + t) * p.N + n] = __float2bfloat16_rn(r[t]);
    }
  }
  if (lane == 0) p.cnt[T * kConsumerWarps + warp] = 0;
}

// Cluster reduction of row tile T: ranks 1..csize-1 write their warps' sums
// into rank 0's shared memory (distributed shared memory) and arrive on its
// barrier; rank 0 adds them to its own in rank order (= K order,
// deterministic) and writes y.  No global round trip, no ticket.
template <int NT>
__device__ __forceinline__ void cluster_reduce(const RowsParams& p, int T, int rank, int warp, int lane,
                                               const float (&tot)[NT][4], uint64_t* red_bar, float* red_buf) {
  constexpr int V = 4 * NT;   // values per lane
  if (rank > 0) {
    float* dst = cluster_map_rank0(red_buf) + ((static_cast<size_t>(rank - 1) * kConsumerWarps + warp) * 32 + lane) * V;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      *reinterpret_cast<float4*>(dst + 4 * nt) = make_float4(tot[nt][0], tot[nt][1], tot[nt][2], tot[nt][3]);
    __syncwarp();
    if (lane == 0) mbar_arrive_remote_rank0(red_bar);
    return;
  }
  if (!mbar_wait_cluster(red_bar, 0, p.red_wait_ns)) {
    if (lane == 0) set_status(p.status, FL_ERR_TIMEOUT, 4);
    // (test hook) the withheld arrival, made once the wait has run out
    if (p.withhold && warp == 0 && lane == 0) mbar_arrive(red_bar);
    // the peers write into this CTA's shared memory: it stays until they are
    // done (normal bound), then leaves without writing its rows of y
    mbar_wait_cluster(red_bar, 0);
    return;
  }
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[nt][e] = tot[nt][e];
  for (int rr = 1; rr < p.csize; ++rr) {
    const float* src = red_buf + ((static_cast<size_t>(rr - 1) * kConsumerWarps + warp) * 32 + lane) * V;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float4 v = *reinterpret_cast<const float4*>(src + 4 * nt);
      acc[nt][0] += v.x, acc[nt][1] += v.y, acc[nt][2] += v.z, acc[nt][3] += v.w;
    }
  }
  const int gid = lane >> 2, tig = lane & 3;
  const int rbase = T * kRowTile + warp * 16;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int n = rbase + gid + (e >> 1) * 8;
      const int m = nt * 8 + 2 * tig + (e & 1);
      if (n < p.N && m < p.M) p.y[static_cast<size_t>(m) * p.N + n] = __float2bfloat16_rn(acc[nt][e]);
    }
  }
}

// The consumer warps' stream over their stages.  CL: the CTA is one rank of
// a cluster sharing a row tile (its range lies inside that tile, group slot
// = unit index in the range, no tile boundaries); otherwise a stream-K range
// that may cross row tiles, finished through the ticket hand-off.
// GLU (the gate/up half of a decode MLP block, M <= 8, cluster mode): each
// stage holds the gate and the up super-block of one (row tile, group) (and
// that group's x rows when there is no x region); two folded sums per row;
// rank 0 of the cluster adds the ranks' gate and up sums in rank order and
// stores h = silu(gate) * up.
__device__ __forceinline__ void glu_reduce(const RowsParams& p, int T, int rank, int warp, int lane,
                                           const float (&tg)[4], const float (&tu)[4], uint64_t* red_bar,
                                           float* red_buf) {
  constexpr int V = 8;
  if (rank > 0) {
    float* dst = cluster_map_rank0(red_buf) + ((static_cast<size_t>(rank - 1) * kConsumerWarps + warp) * 32 + lane) * V;
    *reinterpret_cast<float4*>(dst) = make_float4(tg[0], tg[1], tg[2], tg[3]);
    *reinterpret_cast<float4*>(dst + 4) = make_float4(tu[0], tu[1], tu[2], tu[3]);
    __syncwarp();
    if (lane == 0) mbar_arrive_remote_rank0(red_bar);
    return;
  }
  if (!mbar_wait_cluster(red_bar, 0, p.red_wait_ns)) {
    if (lane == 0) set_status(p.status, FL_ERR_TIMEOUT, 6);
    if (p.withhold && warp == 0 && lane == 0) mbar_arrive(red_bar);
    mbar_wait_cluster(red_bar, 0);
    return;
  }
  float g[4], u[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) g[e] = tg[e], u[e] = tu[e];
  for (int rr = 1; rr < p.csize; ++rr) {
    const float* src = red_buf + ((static_cast<size_t>(rr - 1) * kConsumerWarps + warp) * 32 + lane) * V;
    const float4 a = *reinterpret_cast<const float4*>(src);
    const float4 b = *reinterpret_cast<const float4*>(src + 4);
    g[0] += a.x, g[1] += a.y, g[2] += a.z, g[3] += a.w;
    u[0] += b.x, u[1] += b.y, u[2] += b.z, u[3] += b.w;
  }
  const int gid = lane >> 2, tig = lane & 3;
  const int rbase = T * kRowTile + warp * 16;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int n = rbase + gid + (e >> 1) * 8;
    const int m = 2 * tig + (e & 1);
    if (n < p.N && m < p.M) p.y[static_cast<size_t>(m) * p.N + n] = __float2bfloat16_rn(g[e] / (1.f + expf(-g[e])) * u[e]);
  }
}

__device__ __forceinline__ void rows_consume_glu(const RowsParams& p, uint8_t* smem, uint64_t* full, uint64_t* empty,
                                                 const float* xsum, int u0, int nstage, int rank, int warp, int lane,
                                                 uint64_t* red_bar, float* red_buf) {
  constexpr int Mp = 8;
  const uint32_t xoff = 2 * kSbBytes;
  const int gid = lane >> 2, tig = lane & 3;
  const int r0 = warp * 16 + gid;
  const uint8_t* xzero = smem + p.zrow_off;
  float tg[4] = {0.f, 0.f, 0.f, 0.f}, tu[4] = {0.f, 0.f, 0.f, 0.f};
  int s = 0;
  uint32_t ph = 0;
  for (int k = 0; k < nstage; ++k) {
    if (!mbar_wait(&full[s], ph)) {
      if (lane == 0) set_status(p.status, FL_ERR_TIMEOUT, 2);
      if (rank == 0) mbar_wait_cluster(red_bar, 0);
      return;
    }
    const uint8_t* sb = smem + static_cast<size_t>(s) * p.stage_bytes;
    // unit k's x rows: the x region (slot k) or the stage
    const uint8_t* sx = p.xr_stride > 0 ? smem + p.xr_off + k * 256 : sb + xoff;
    const int xstride = p.xr_stride > 0 ? p.xr_stride : kXRowStride;
    float ag[1][4], au[1][4];
    float sg0, sg1, su0, su1;
    uint32_t zg0, zg1, zu0, zu1;
    unit_dot<1, true, true>(sb, sx, p.M, r0, gid, tig, ag, sg0, sg1, zg0, zg1, 1, xzero, xstride);
    unit_dot<1, true, true>(sb + kSbBytes, sx, p.M, r0, gid, tig, au, su0, su1, zu0, zu1, 1, xzero, xstride);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    const float2 xs = *reinterpret_cast<const float2*>(xsum + k * Mp + 2 * tig);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float xv = (e & 1) ? xs.y : xs.x;
      const uint32_t zg = (e >> 1) ? zg1 : zg0, zu = (e >> 1) ? zu1 : zu0;
      tg[e] = fmaf((e >> 1) ? sg1 : sg0, fmaf(-__uint_as_float(0x43000000u + (zg << 16)), xv, ag[0][e]), tg[e]);
      tu[e] = fmaf((e >> 1) ? su1 : su0, fmaf(-__uint_as_float(0x43000000u + (zu << 16)), xv, au[0][e]), tu[e]);
    }
    if (++s == p.stages) s = 0, ph ^= 1u;
  }
  glu_reduce(p, u0 / p.G, rank, warp, lane, tg, tu, red_bar, red_buf);
}

template <int NT, int UPS, bool CL, bool G64>
__device__ __forceinline__ void rows_consume(const RowsParams& p, uint8_t* smem, uint64_t* full, uint64_t* empty,
                                             const float* xsum, int u0, int u1, int g0, int nslot, int nstage,
                                             int c, int rank, int warp, int lane, uint64_t* red_bar,
                                             float* red_buf) {
  constexpr bool FOLD = NT <= 2;
  constexpr int Mp = 8 * NT;
  constexpr int XS = G64 ? 2 : 1;          // token sums per group slot: one per 64-column group
  const uint32_t xoff = UPS * kSbBytes;
  const bool xr = CL && p.xr_stride > 0;   // x from the CTA's x region, not from the stage
  const uint32_t soff = xoff + (xr ? 0 : UPS * p.M * kXRowStride);   // G64: the stage's side entries
  const int xstride = xr ? p.xr_stride : kXRowStride;
  const int gid = lane >> 2, tig = lane & 3;
  const int r0 = warp * 16 + gid;
  const uint8_t* xzero = smem + p.zrow_off;
  float tot[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) tot[nt][e] = 0.f;
  int curT = u0 / p.G, g = g0, slot = 0, s = 0, owed0 = -1;
  uint32_t ph = 0;
  for (int k = 0; k < nstage; ++k) {
    const int ua = u0 + k * UPS, n = min(UPS, u1 - ua);
    if (!mbar_wait(&full[s], ph)) {
      if (lane == 0) set_status(p.status, FL_ERR_TIMEOUT, 2);
      // rank 0 of a cluster stays until its peers' DSMEM writes have landed
      if (CL && rank == 0) mbar_wait_cluster(red_bar, 0);
      return;
    }
    const uint8_t* sb = smem + static_cast<size_t>(s) * p.stage_bytes;
    // G64: index [half] = the 64-column group (0: columns 0..63 of the super-block)
    float acc[UPS][XS][NT][4];
    float sc[UPS][XS][2];
    uint32_t zr[UPS][XS][2];
    // Every slot of the stage is computed, in one basic block so that the
    // compiler interleaves the independent MMA chains; a slot past the end
    // of the range holds stale shared memory and its result is dropped.
#pragma unroll
    for (int i = 0; i < UPS; ++i) {
      // cluster mode: group slot = unit index in the range (a slot past its
      // end reads the last group's x: in bounds, and its result is dropped)
      const uint8_t* sx = xr ? smem + p.xr_off + min(k * UPS + i, nslot - 1) * 256
                             : sb + xoff + i * p.M * kXRowStride;
      if constexpr (G64) {
        float s0[2], s1[2];
        uint32_t z0[2], z1[2];
        unit_dot64<NT, FOLD, true>(sb + i * kSbBytes, sb + soff + i * kSbSide, sx, p.M, r0, gid, tig, acc[i], s0, s1,
                                   z0, z1, NT, xzero, xstride);
#pragma unroll
        for (int hh = 0; hh < XS; ++hh) sc[i][hh][0] = s0[hh], sc[i][hh][1] = s1[hh], zr[i][hh][0] = z0[hh], zr[i][hh][1] = z1[hh];
      } else {
        unit_dot<NT, FOLD, true>(sb + i * kSbBytes, sx, p.M, r0, gid, tig, acc[i][0], sc[i][0][0], sc[i][0][1],
                                 zr[i][0][0], zr[i][0][1], NT, xzero, xstride);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
#pragma unroll
    for (int i = 0; i < UPS; ++i) {
      if (i < n) {
        const int sl = CL ? k * UPS + i : (slot < nslot ? slot : 0);
#pragma unroll
        for (int hh = 0; hh < XS; ++hh)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float2 xs = make_float2(0.f, 0.f);
          if (FOLD) xs = *reinterpret_cast<const float2*>(xsum + (sl * XS + hh) * Mp + nt * 8 + 2 * tig);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float v = acc[i][hh][nt][e];
            // 128 + z as a float without a conversion: z in the mantissa of 128.0
            if (FOLD) v = fmaf(-__uint_as_float(0x43000000u + (zr[i][hh][e >> 1] << 16)), (e & 1) ? xs.y : xs.x, v);
            tot[nt][e] = fmaf(sc[i][hh][e >> 1], v, tot[nt][e]);
          }
        }
        if (!CL) {
          ++slot;
          if (++g == p.G) {
            g = 0;
            if (ua + i + 1 < u1) {
              // row tile finished inside this CTA's range: store it now,
              // take its ticket after the stream
              if (store_tile<NT>(p, curT, c, u0, u1, warp, lane, tot)) owed0 = curT;
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) tot[nt][e] = 0.f;
              ++curT;
            }
          }
          if (slot == nslot) slot = 0;
        }
      }
    }
    if (++s == p.stages) s = 0, ph ^= 1u;
  }
  if (CL) {
    cluster_reduce<NT>(p, curT, rank, warp, lane, tot, red_bar, red_buf);
    return;
  }
  const bool owed1 = store_tile<NT>(p, curT, c, u0, u1, warp, lane, tot);
  // only the first and the last row tile of a CTA's range can be partial
  if (owed0 >= 0) ticket_tile<NT>(p, owed0, warp, lane);
  if (owed1) ticket_tile<NT>(p, curT, warp, lane);
}

// NT token tiles of 8; UPS super-blocks per pipeline stage (2 gives each
// warp two independent MMA chains and 17 KB bulk copies).  MINB CTAs per SM:
// 2 (M <= 8, up to 113 KB of shared memory each), 3 (M <= 8 when the row
// tiles' clusters would fill the GPU's cluster capacity at 2: smaller
// stages, fewer registers, so that every cluster is resident in one wave)
// or 1 (M > 8).
template <int NT, int UPS, int MINB, bool G64, bool GLU = false>
__global__ void __launch_bounds__(kThreads, MINB) k_linear_rows(const RowsParams p) {
  static_assert(!GLU || (NT == 1 && UPS == 2 && !G64), "GLU: one token tile, the gate and up super-blocks per stage");
  constexpr bool FOLD = NT <= 2;
  constexpr int Mp = 8 * NT;
  constexpr int XS = G64 ? 2 : 1;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(p.stages) * p.stage_bytes);
  uint64_t* empty = full + p.stages;
  float* xsum = reinterpret_cast<float*>(empty + p.stages);   // [group slot][XS][Mp]: sum_k x over each group
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  // stream-K ranges, or (clusters) K slice `rank` of row tile c / csize
  const int rank = p.csize > 1 ? c % p.csize : 0;
  int u0, u1;
  if (p.csize > 1) {
    const int t = c / p.csize;
    u0 = t * p.G + rank * p.G / p.csize;
    u1 = t * p.G + (rank + 1) * p.G / p.csize;
  } else {
    u0 = unit_begin(c, p.U, p.P);
    u1 = unit_begin(c + 1, p.U, p.P);
  }
  uint64_t* red_bar = reinterpret_cast<uint64_t*>(smem + p.red_off);
  float* red_buf = reinterpret_cast<float*>(smem + p.red_off + 16);   // [csize-1][warp][lane][4*NT]
  const int nstage = GLU ? u1 - u0 : (u1 - u0 + UPS - 1) / UPS;   // stages this CTA fills, in order
  const uint32_t xoff = UPS * kSbBytes;           // x slices follow the super-blocks
  const int g0 = u0 % p.G;
  const int nslot = (u1 - u0) < p.G ? (u1 - u0) : p.G;   // distinct groups, from g0 on (mod G)
  const bool xr = p.csize > 1 && p.xr_stride > 0;   // x region (cluster mode): no x in the stages

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    if (p.csize > 1) mbar_init(red_bar, (p.csize - 1) * kConsumerWarps + (p.withhold ? 1 : 0));
    fence_mbar_init();
  }
  if (threadIdx.x < 16) reinterpret_cast<uint4*>(smem + p.zrow_off)[threadIdx.x] = make_uint4(0u, 0u, 0u, 0u);
  cta_sync();
  // rank 0's reduction barrier is initialised before any peer can arrive on it
  if (p.csize > 1) cluster_sync_all();
  // the next kernel in the stream may start prefetching its weights now
  pdl_launch_dependents();

  if (warp == kConsumerWarps) {
    // ---------------- producer warp
    const uint64_t pol = policy_evict_first();
    auto issue_w = [&](int k, int slot) {   // weights of stage k (contiguous super-blocks, and side entries)
      if (GLU) {   // the gate and the up super-block of unit u0 + k
        if (lane == 0) {
          uint8_t* st = smem + static_cast<size_t>(slot) * p.stage_bytes;
          const size_t off = static_cast<size_t>(u0 + k) * kSbBytes;
          mbar_arrive_expect_tx(&full[slot], 2u * kSbBytes + (xr ? 0u : p.M * 256u));
          bulk_g2s_hint(st, p.w + off, kSbBytes, &full[slot], pol);
          bulk_g2s_hint(st + kSbBytes, p.w_up + off, kSbBytes, &full[slot], pol);
        }
        return;
      }
      const int ua = u0 + k * UPS, n = min(UPS, u1 - ua);
      if (lane == 0) {
        uint8_t* st = smem + static_cast<size_t>(slot) * p.stage_bytes;
        mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(n) * (kSbBytes + (xr ? 0u : p.M * 256u) +
                                                                      (G64 ? kSbSide : 0)));
        bulk_g2s_hint(st, p.w + static_cast<size_t>(ua) * kSbBytes, static_cast<uint32_t>(n) * kSbBytes, &full[slot],
                      pol);
        if (G64)
          bulk_g2s_hint(st + xoff + (xr ? 0 : UPS * p.M * kXRowStride), p.side + static_cast<size_t>(ua) * kSbSide,
                        static_cast<uint32_t>(n) * kSbSide, &full[slot], pol);
      }
    };
    auto issue_x = [&](int k, int slot) {   // the M token rows' slices of stage k's groups
      if (xr) return;   // the consumers fill the x region instead
      const int ua = GLU ? u0 + k : u0 + k * UPS, n = GLU ? 1 : min(UPS, u1 - ua);
      uint8_t* st = smem + static_cast<size_t>(slot) * p.stage_bytes + xoff;
      for (int idx = lane; idx < n * p.M; idx += 32) {
        const int i = idx / p.M, m = idx - i * p.M;
        const int g = (ua + i) % p.G;
        bulk_g2s(st + (i * p.M + m) * kXRowStride, p.x + static_cast<size_t>(m) * p.K + g * kGroup, 256u,
                 &full[slot]);
      }
    };
    // Weights do not depend on the previous kernel: fill the first stages
    // before waiting for it; x (its output) is copied after.
    const int pre = nstage < p.stages ? nstage : p.stages;
    for (int k = 0; k < pre; ++k) issue_w(k, k);
    __syncwarp();
    pdl_wait();
    for (int k = 0; k < pre; ++k) issue_x(k, k);
    int s = pre % p.stages;
    uint32_t ph = pre == p.stages ? 1u : 0u;
    for (int k = pre; k < nstage; ++k) {
      if (!mbar_wait(&empty[s], ph ^ 1u)) {
        if (lane == 0) set_status(p.status, FL_ERR_TIMEOUT, 1);
        // let the copies already issued land before the CTA retires
        for (int j = 0; j < p.stages; ++j) {
          const int nf = k / p.stages + (j < k % p.stages ? 1 : 0);
          if (nf > 0) mbar_wait(&full[j], static_cast<uint32_t>(nf - 1) & 1u);
        }
        return;
      }
      issue_w(k, s);
      __syncwarp();
      issue_x(k, s);
      if (++s == p.stages) s = 0, ph ^= 1u;
    }
    return;
  }

  // ---------------- consumer warps: rows warp*16 .. warp*16+15 of each tile
  // (they read x and write y and the workspace: only once the previous kernel is done)
  pdl_wait();
  if (FOLD) {
    // Per-group token sums of x for this CTA's groups, [slot][Mp]: four
    // neighbouring threads per (group slot, token < M), 32 values each in
    // four independent chains, then two shuffles (a fixed order:
    // deterministic).  The thread count is rounded up to whole warps so
    // that every lane of a warp runs the shuffles; tokens M..Mp-1 get 0.
    const int items = nslot * p.M;
    const int nthr = (items * 4 + 31) & ~31;
    for (int idx = threadIdx.x; idx < nthr; idx += kConsumerWarps * 32) {
      const int it = idx >> 2, part = idx & 3;
      float v = 0.f;
      if (it < items) {
        const int i = it / p.M, m = it - i * p.M;
        int g = g0 + i;
        if (g >= p.G) g -= p.G;
        // the thread's four 16-byte chunks of the group's 256 bytes: part + 4t
        // (the four threads of a token read 64 contiguous bytes per load, and
        // the eight threads of a store phase hit distinct bank groups); with
        // groups of 64, 4 part + t (parts 0, 1: columns 0..63)
        constexpr int kCs = G64 ? 1 : 4;   // chunk stride
        const int c0 = G64 ? part * 4 : part;
        const uint4* src = reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(m) * p.K + g * kGroup) + c0;
        uint4 q[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) q[t] = __ldg(src + kCs * t);
        if (xr) {   // these 64 bytes of x into the region: token m, group slot i
          uint4* dst = reinterpret_cast<uint4*>(smem + p.xr_off + static_cast<size_t>(m) * p.xr_stride + i * 256) + c0;
#pragma unroll
          for (int t = 0; t < 4; ++t) dst[kCs * t] = q[t];
        }
        float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const uint32_t w4[4] = {q[t].x, q[t].y, q[t].z, q[t].w};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            a[h] += __uint_as_float(w4[h] << 16);
            a[h] += __uint_as_float(w4[h] & 0xffff0000u);
          }
        }
        v = (a[0] + a[1]) + (a[2] + a[3]);
      }
      // G64: part 0, 1 summed columns 0..63 of the group, 2, 3 columns 64..127
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      if (G64) {
        if ((part & 1) == 0 && it < items) xsum[((it / p.M) * XS + (part >> 1)) * Mp + it % p.M] = v;
      } else {
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        if (part == 0 && it < items) xsum[(it / p.M) * Mp + it % p.M] = v;
      }
    }
    for (int idx = threadIdx.x; idx < nslot * XS * (Mp - p.M); idx += kConsumerWarps * 32) {
      const int i = idx / (Mp - p.M), m = p.M + idx - i * (Mp - p.M);
      xsum[i * Mp + m] = 0.f;
    }
    named_bar(1, kConsumerWarps * 32);
  }
  if constexpr (GLU) {
    rows_consume_glu(p, smem, full, empty, xsum, u0, nstage, rank, warp, lane, red_bar, red_buf);
    return;
  }
  if (p.csize > 1)
    rows_consume<NT, UPS, true, G64>(p, smem, full, empty, xsum, u0, u1, g0, nslot, nstage, c, rank, warp, lane,
                                     red_bar, red_buf);
  else
    rows_consume<NT, UPS, false, G64>(p, smem, full, empty, xsum, u0, u1, g0, nslot, nstage, c, rank, warp, lane,
                                      red_bar, red_buf);
}

// ------------------------------------------------------------------ plan
struct RowsPlan {
  int T, G, P, NT, ups, stages, U, csize, minb, xr_stride;
  uint32_t stage_bytes, red_off, zrow_off, xr_off;
  size_t smem, cnt_off, part_off, ws_bytes;
};

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// minb: CTAs per SM the kernel is built for (0 = the default for M); g64:
// groups of 64 (side entries in the stages, two token sums per group).
bool make_rows_plan(int M, int N, int K, int sms, RowsPlan* pl, int minb = 0, bool g64 = false, bool glu = false,
                    int max_cs = 8) {
  if (M < 1 || M > kMaxTokens || N < 1 || K < kGroup || K % kGroup || sms < 1) return false;
  if ((N + kRowTile - 1) / kRowTile > kMaxRowTiles) return false;
  pl->T = (N + kRowTile - 1) / kRowTile;
  pl->G = K / kGroup;
  const long long U = static_cast<long long>(pl->T) * pl->G;
  if (U > (1LL << 30)) return false;
  pl->U = static_cast<int>(U);
  pl->NT = (M + 7) / 8;
  pl->ups = pl->NT <= 2 ? 2 : 1;
  pl->minb = minb > 0 ? minb : (pl->NT == 1 ? 2 : 1);
  if (pl->NT > 1) pl->minb = 1;
  // M <= 8: two CTAs per SM (four consumer warps per scheduler)
  const long long slots = static_cast<long long>(sms) * (pl->NT == 1 ? 2 : 1);
  // Few row tiles: clusters of csize CTAs share each tile, split over K, and
  // reduce through distributed shared memory.  Otherwise contiguous unit
  // ranges over all tiles (stream-K) with the global ticket hand-off.
  pl->csize = 1;
  if (2LL * pl->T <= slots) {
    long long cs = slots / pl->T;
    if (cs > max_cs) cs = max_cs;
    // every rank streams at least one full stage (ups super-blocks): with a
    // single super-block a rank, the reduction over more ranks costs more
    // than the split saves (K=1024, N=3072, M=1: 4.04 us at 8 ranks, 3.28 us
    // at 4)
    if (cs > pl->G / pl->ups) cs = pl->G / pl->ups;
    if (cs < 1) cs = 1;
    pl->csize = static_cast<int>(cs);
  }
  if (pl->csize > 1)
    pl->P = pl->T * pl->csize;
  else
    pl->P = static_cast<int>(U < slots ? U : slots);
  if (glu && (pl->NT != 1 || pl->csize < 2 || g64)) return false;   // GLU: cluster mode, M <= 8
  const size_t red_bytes =
      pl->csize > 1
          ? 16 + static_cast<size_t>(pl->csize - 1) * kConsumerWarps * 32 * 4 * pl->NT * (glu ? 2 : 1) * sizeof(float)
          : 0;
  const int units_max = pl->csize > 1 ? (pl->G + pl->csize - 1) / pl->csize : (pl->U + pl->P - 1) / pl->P;
  const int nslot = units_max < pl->G ? units_max : pl->G;
  const size_t xsum_bytes = static_cast<size_t>(nslot) * (g64 ? 2 : 1) * 8 * pl->NT * sizeof(float);
  // Cluster mode with one token tile: the x rows of a rank's K slice (one
  // contiguous run of groups) are loaded once, by the token-sum prologue,
  // into an x region; the stages then carry weights only and the producer
  // issues one weight copy per stage instead of one more 256-byte copy per
  // token and group (chained launches at M=8: fused QKV 12.9 to 11.5 us; the
  // decode MLP block's gate/up half, M=8: its block 26.7 to 24.3 us).  Rows
  // are an odd multiple of 64 bytes apart: conflict-free B-fragment loads.
  for (int xr = (pl->csize > 1 && pl->NT == 1) ? 1 : 0; xr >= 0; --xr) {
    pl->xr_stride = xr ? nslot * 256 + 64 : 0;
    const size_t xr_bytes = static_cast<size_t>(M) * pl->xr_stride;
    pl->stage_bytes = static_cast<uint32_t>(align_up(
        glu ? 2 * static_cast<size_t>(kSbBytes) + (xr ? 0 : static_cast<size_t>(M) * kXRowStride)
            : static_cast<size_t>(pl->ups) *
                  (kSbBytes + (xr ? 0 : static_cast<size_t>(M) * kXRowStride) + (g64 ? kSbSide : 0)),
        128));
    long long stages;
    if (pl->minb == 2) {
      // two CTAs per SM: 113 KB each, of which the ring takes the rest (256
      // bytes of zero row, 256 of alignment slack)
      const long long fixed = static_cast<long long>(xsum_bytes + 256 + 256 + xr_bytes + red_bytes);
      stages = (113LL * 1024 - fixed) / static_cast<long long>(pl->stage_bytes + 2 * sizeof(uint64_t));
    } else {
      stages = (static_cast<long long>(pl->minb == 3 ? 66u * 1024u : 200u * 1024u) -
                static_cast<long long>(red_bytes + xr_bytes)) /
               static_cast<long long>(pl->stage_bytes);
    }
    if (xr && stages < 3) continue;   // too little room left for the ring: x in the stages
    pl->stages = stages > 12 ? 12 : (stages < 2 ? 2 : static_cast<int>(stages));
    break;
  }
  // The layout; a launch takes at most 227 KB of dynamic shared memory, so a
  // plan above that (long K with many tokens, whose group sums take room)
  // sheds stages, down to two.  A plan still above it is kept (its workspace
  // offsets serve the tcgen05 decode too); the launchers refuse it.
  for (;;) {
    pl->smem = static_cast<size_t>(pl->stages) * pl->stage_bytes + 2 * pl->stages * sizeof(uint64_t) + xsum_bytes;
    pl->zrow_off = static_cast<uint32_t>(align_up(pl->smem, 16));
    pl->smem = pl->zrow_off + 256;
    pl->xr_off = static_cast<uint32_t>(align_up(pl->smem, 128));
    if (pl->xr_stride) pl->smem = pl->xr_off + static_cast<size_t>(M) * pl->xr_stride;
    pl->red_off = static_cast<uint32_t>(align_up(pl->smem, 16));
    if (red_bytes) pl->smem = pl->red_off + red_bytes;
    if (pl->smem <= kMaxDynSmem || pl->stages <= 2) break;
    --pl->stages;
  }
  pl->cnt_off = kTicketOff;
  pl->part_off = kScratchOff;
  pl->ws_bytes = pl->part_off + static_cast<size_t>(pl->P + pl->T) * kRowTile * (8 * pl->NT) * 4;
  return true;
}

template <int NT, int UPS, int MINB, bool G64, bool GLU = false>
bool rows_attr(int dev) {
  static bool attr_done[64] = {false};
  if (dev < 0 || dev >= 64) return false;
  if (!attr_done[dev]) {
    if (cudaFuncSetAttribute(k_linear_rows<NT, UPS, MINB, G64, GLU>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kMaxDynSmem)) != cudaSuccess)
      return false;
    attr_done[dev] = true;
  }
  return true;
}

// How many clusters of pl.csize CTAs of the two-per-SM kernel (with pl.smem
// bytes each) the GPU holds at once; cached per device, cluster size and
// shared-memory size.  -1 when the query fails.
int rows_cluster_capacity(const RowsPlan& pl) {
  struct Entry { int dev, csize; size_t smem; int cap; };
  static Entry cache[64];
  static int n = 0;
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (cache[i].dev == dev && cache[i].csize == pl.csize && cache[i].smem == pl.smem) return cache[i].cap;
  if (!rows_attr<1, 2, 2, false>(dev)) return -1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.P);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = pl.smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(pl.csize);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int cap = -1;
  if (cudaOccupancyMaxActiveClusters(&cap, k_linear_rows<1, 2, 2, false>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    cap = -1;
  }
  if (n < 64) cache[n++] = Entry{dev, pl.csize, pl.smem, cap};
  return cap;
}

template <int NT, int UPS, int MINB, bool G64, bool GLU = false>
int launch_rows(const RowsPlan& pl, const RowsParams& prm, cudaStream_t s) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (!rows_attr<NT, UPS, MINB, G64, GLU>(dev)) return FL_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.P);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(pl.csize);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pl.csize > 1 ? 2 : 1;
  if (cudaLaunchKernelEx(&cfg, k_linear_rows<NT, UPS, MINB, G64, GLU>, prm) != cudaSuccess) return FL_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? FL_OK : FL_ERR_CUDA;
}

}  // namespace

// Test hook of the failure path (fl_int4g_test_withhold_cluster_arrival):
// < 0 off; otherwise the wait bound in ns of the cluster reductions of the
// following decode launches, which withhold one arrival.
static std::atomic<long long> g_withhold_ns{-1};

extern "C" int fl_int4g_test_withhold_cluster_arrival(long long ns) {
  g_withhold_ns.store(ns < 0 ? -1 : ns);
  return FL_OK;
}

// Test hook: the decode kernel's plan for a shape, without a GPU.
// out[0..10] = T, G, P, csize, stages, stage_bytes, dynamic shared memory,
// x-region stride (0: x in the stages), x-region offset, reduction offset,
// zero-row offset.
extern "C" int fl_int4g_test_decode_plan(int M, int N, int K, int sms, int group, int glu, int minb, int max_cs,
                                         long long* out) {
  if (!out || (group != kGroup && group != kGroup / 2) || max_cs < 1) return FL_ERR_ARG;
  RowsPlan pl;
  if (!make_rows_plan(M, N, K, sms, &pl, minb, group == kGroup / 2, glu != 0, max_cs)) return FL_ERR_ARG;
  const long long v[11] = {pl.T, pl.G, pl.P, pl.csize, pl.stages, pl.stage_bytes, static_cast<long long>(pl.smem),
                           pl.xr_stride, pl.xr_off, pl.red_off, pl.zrow_off};
  for (int i = 0; i < 11; ++i) out[i] = v[i];
  return FL_OK;
}

// Shared with the MoE and prefill launchers.
int fl_linear_rows_workspace(int M, int N, int K, size_t* out) {
  RowsPlan pl;
  if (!make_rows_plan(M, N, K, flh::sm_count(), &pl)) return FL_ERR_ARG;
  *out = pl.ws_bytes;
  return FL_OK;
}

// group: 128 (or 256: the same layout) or 64 (side array after the super-blocks).
int fl_linear_rows(const void* x, int M, int K, const void* w, int N, void* y, void* ws, size_t ws_bytes,
                   cudaStream_t stream, int group = kGroup) {
  const bool g64 = group == kGroup / 2;
  RowsPlan pl;
  if (!make_rows_plan(M, N, K, flh::sm_count(), &pl, 0, g64)) return FL_ERR_ARG;
  if (ws_bytes < pl.ws_bytes) return FL_ERR_WORKSPACE;
  // Clusters that would fill the GPU's cluster capacity leave some of them
  // waiting for a second wave whenever the previous kernel's exits fragment
  // the free slots.  Such shapes take smaller clusters first (fused QKV,
  // K=4096 N=12288 at M=1: 9.7 us with clusters of 2 against 11.2 us for the
  // three-per-SM build), and three smaller CTAs per SM (same grid, same
  // workspace) only if that is not enough.
  if (pl.NT == 1 && pl.csize > 1) {
    int cap = rows_cluster_capacity(pl);
    while (cap > 0 && pl.T > cap - 2 && pl.csize > 2) {
      if (!make_rows_plan(M, N, K, flh::sm_count(), &pl, 0, g64, false, pl.csize - 1)) return FL_ERR_ARG;
      cap = rows_cluster_capacity(pl);
    }
    if (cap > 0 && pl.T > cap - 2 && !make_rows_plan(M, N, K, flh::sm_count(), &pl, 3, g64)) return FL_ERR_ARG;
  }
  if (pl.smem > kMaxDynSmem) return FL_ERR_UNSUPPORTED;   // even two stages do not fit
  RowsParams prm;
  prm.w = static_cast<const uint8_t*>(w);
  prm.side = g64 ? static_cast<const uint8_t*>(w) + static_cast<size_t>(pl.U) * kSbBytes : nullptr;
  prm.w_up = nullptr;
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
  prm.stages = pl.stages;
  prm.stage_bytes = pl.stage_bytes;
  prm.csize = pl.csize;
  prm.red_off = pl.red_off;
  prm.zrow_off = pl.zrow_off;
  prm.xr_stride = pl.xr_stride;
  prm.xr_off = pl.xr_off;
  const long long hook = g_withhold_ns.load();
  prm.withhold = (hook >= 0 && pl.csize > 1) ? 1 : 0;
  prm.red_wait_ns = prm.withhold ? static_cast<unsigned long long>(hook) : kWaitLimitNs;
  if (g64) {
    switch (pl.NT) {
      case 1:
        return pl.minb == 3 ? launch_rows<1, 2, 3, true>(pl, prm, stream) : launch_rows<1, 2, 2, true>(pl, prm, stream);
      case 2: return launch_rows<2, 2, 1, true>(pl, prm, stream);
      case 3: return launch_rows<3, 1, 1, true>(pl, prm, stream);
      default: return launch_rows<4, 1, 1, true>(pl, prm, stream);
    }
  }
  switch (pl.NT) {
    case 1:
      return pl.minb == 3 ? launch_rows<1, 2, 3, false>(pl, prm, stream) : launch_rows<1, 2, 2, false>(pl, prm, stream);
    case 2: return launch_rows<2, 2, 1, false>(pl, prm, stream);
    case 3: return launch_rows<3, 1, 1, false>(pl, prm, stream);
    default: return launch_rows<4, 1, 1, false>(pl, prm, stream);
  }
}

// Gate/up half of a decode MLP block (M <= 8): h[m, i] = silu(G x)[m, i] *
// (U x)[m, i] as bf16, G and U interleaved [I, H].  Returns FL_ERR_UNSUPPORTED
// when the shape does not take the cluster split (the caller then uses
// another path).  ws: the linear workspace of (M, I, H).
int fl_linear_glu(const void* x, int M, int H, const void* w_gate, const void* w_up, int I, void* h, void* ws,
                  size_t ws_bytes, cudaStream_t stream) {
  RowsPlan pl;
  if (!make_rows_plan(M, I, H, flh::sm_count(), &pl, 0, false, true)) return FL_ERR_UNSUPPORTED;
  if (ws_bytes < pl.ws_bytes) return FL_ERR_WORKSPACE;
  if (pl.smem > kMaxDynSmem) return FL_ERR_UNSUPPORTED;
  const int cap = rows_cluster_capacity(pl);
  if (cap > 0 && pl.T > cap - 2) return FL_ERR_UNSUPPORTED;   // a second wave of clusters: not worth it
  RowsParams prm;
  prm.w = static_cast<const uint8_t*>(w_gate);
  prm.w_up = static_cast<const uint8_t*>(w_up);
  prm.side = nullptr;
  prm.x = static_cast<const __nv_bfloat16*>(x);
  prm.y = static_cast<__nv_bfloat16*>(h);
  prm.status = static_cast<int32_t*>(ws);
  prm.cnt = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + pl.cnt_off);
  prm.part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + pl.part_off);
  prm.U = pl.U;
  prm.M = M;
  prm.K = H;
  prm.N = I;
  prm.T = pl.T;
  prm.G = pl.G;
  prm.P = pl.P;
  prm.stages = pl.stages;
  prm.stage_bytes = pl.stage_bytes;
  prm.csize = pl.csize;
  prm.red_off = pl.red_off;
  prm.zrow_off = pl.zrow_off;
  prm.xr_stride = pl.xr_stride;
  prm.xr_off = pl.xr_off;
  const long long hook = g_withhold_ns.load();
  prm.withhold = hook >= 0 ? 1 : 0;
  prm.red_wait_ns = prm.withhold ? static_cast<unsigned long long>(hook) : kWaitLimitNs;
  return launch_rows<1, 2, 2, false, true>(pl, prm, stream);
}

static bool linear_args_ok(const void* x, int M, int K, const void* w, int N, const void* y, const void* ws) {
  if (!x || !w || !y || !ws) return false;
  if (M < 1 || N < 1 || K < kGroup || K % kGroup) return false;
  return flh::aligned16(x) && flh::aligned16(w) && flh::aligned16(y) && flh::aligned16(ws);
}

size_t fl_linear_tc_workspace(int M);
int fl_linear_tc(const void* x, int M, int K, const void* w, int N, void* y, void* ws, cudaStream_t s,
                 const void* side);
int fl_linear_tcdec(const void* x, int M, int K, const void* w, int N, void* y, void* ws, size_t cnt_off,
                    size_t part_off, cudaStream_t s);

// Workspace of the tcgen05 decode kernel: the decode layout (status, fixed
// counter region) with (min(U, SMs) + T) partial slots of 128 rows x NB floats,
// NB = 16 for M <= 16, else 32.
static bool tcdec_plan(int M, int N, int K, size_t* cnt_off, size_t* part_off, size_t* total) {
  RowsPlan pl;
  if (!make_rows_plan(M, N, K, flh::sm_count(), &pl)) return false;
  const int NB = M <= 16 ? 16 : 32;
  const long long sms = flh::sm_count();
  const long long P = pl.U < sms ? pl.U : sms;
  *cnt_off = pl.cnt_off;
  *part_off = pl.part_off;
  *total = pl.part_off + static_cast<size_t>(P + pl.T) * kRowTile * NB * 4;
  if (*total < pl.ws_bytes) *total = pl.ws_bytes;
  return true;
}

// Decode part of the linear (1 <= M <= 32), shared by fl_int4g_linear and
// the variant that allocates nothing: workspace bytes, and the dispatch.
int fl_linear_decode_workspace(int M, int N, int K, size_t* out) {
  size_t a, b;
  return tcdec_plan(M, N, K, &a, &b, out) ? FL_OK : FL_ERR_ARG;
}

int fl_linear_decode(const void* x, int M, int K, const void* w, int N, void* y, void* ws, size_t ws_bytes,
                     cudaStream_t s) {
  size_t cnt_off, part_off, need;
  if (!tcdec_plan(M, N, K, &cnt_off, &part_off, &need)) return FL_ERR_ARG;
  if (ws_bytes < need) return FL_ERR_WORKSPACE;
  // M <= 8: the register-dequant mma.sync stream is faster (one warp hand-off
  // per two super-blocks); 8 < M <= 32: tcgen05 (mma.sync issue-bound there)
  if (M <= 8) return fl_linear_rows(x, M, K, w, N, y, ws, ws_bytes, s);
  return fl_linear_tcdec(x, M, K, w, N, y, ws, cnt_off, part_off, s);
}

extern "C" int fl_int4g_linear_workspace(int M, int N, int K, size_t* out) {
  if (!out || M < 1 || N < 1 || K < kGroup || K % kGroup) return FL_ERR_ARG;
  if (M > kMaxTokens) {
    *out = fl_linear_tc_workspace(M);
    return FL_OK;
  }
  return fl_linear_decode_workspace(M, N, K, out);
}

extern "C" int fl_int4g_linear(const void* x, int M, int K, const void* w, int N, void* y, void* ws,
                               size_t ws_bytes, fl_stream_t stream) {
  if (!linear_args_ok(x, M, K, w, N, y, ws)) return FL_ERR_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (M > kMaxTokens) {
    if (ws_bytes < fl_linear_tc_workspace(M)) return FL_ERR_WORKSPACE;
    return fl_linear_tc(x, M, K, w, N, y, ws, s, nullptr);
  }
  return fl_linear_decode(x, M, K, w, N, y, ws, ws_bytes, s);
}

extern "C" int fl_int4g_linear_g(const void* x, int M, int K, const void* w, int N, int group, void* y, void* ws,
                                 size_t ws_bytes, fl_stream_t stream) {
  if (group == kGroup || group == 2 * kGroup) return fl_int4g_linear(x, M, K, w, N, y, ws, ws_bytes, stream);
  if (group != kGroup / 2) return FL_ERR_UNSUPPORTED;
  if (!linear_args_ok(x, M, K, w, N, y, ws)) return FL_ERR_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t nsb = static_cast<size_t>((N + kRowTile - 1) / kRowTile) * (K / kGroup);
  const uint8_t* side = static_cast<const uint8_t*>(w) + nsb * kSbBytes;
  if (M > kMaxTokens) {
    if (ws_bytes < fl_linear_tc_workspace(M)) return FL_ERR_WORKSPACE;
    return fl_linear_tc(x, M, K, w, N, y, ws, s, side);
  }
  // decode: the mma.sync kernel for every M <= 32 (the tcgen05 decode kernel
  // keeps one accumulator per 128 columns)
  size_t need = 0;
  if (fl_linear_decode_workspace(M, N, K, &need) != FL_OK) return FL_ERR_ARG;
  if (ws_bytes < need) return FL_ERR_WORKSPACE;
  return fl_linear_rows(x, M, K, w, N, y, ws, ws_bytes, s, kGroup / 2);
}
