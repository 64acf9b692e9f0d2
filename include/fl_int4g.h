/*
 * fl_int4g.h -- C ABI of the int4g (weight-only INT4, group-quantized) library
 * for NVIDIA GB300 (sm_103a).
 *
 * The method: weights are stored as 4-bit codes in groups of 128 along K,
 * each group sharing one scale and one zero point, and are dequantized inside
 * the matrix product ("FastLLM: zero-dependency CPU inference framework",
 * pgsm.cn, section 3.1 "4-bit quantization and weight reordering").  The
 * linear and MoE layers that use it are selected in fastllm by
 * `--dtype int4g` / `--moe_dtype int4g`, with `--moe_experts` (top-k) and
 * `--cuda_se` (shared expert) (fastllm README, gittoolsai mirror, sections
 * "2. 如何设定推理精度" and "5. 其它参数").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - W is [N, K] in nn.Linear order; y = x . deq(W)^T; x is [M, K] bf16,
 *    row-major, y is [M, N] bf16, row-major.
 *  - group is 128 or 256 (FastLLM page, section 4.2: --group-size 128 by
 *    default, 256 allowed) or 64 (section 5.4: 64 for more precision),
 *    K % group == 0 and K % 128 == 0.  The quantizer, the repack and the
 *    unrepack take it; the matmul entry points read the interleaved layout,
 *    whose super-blocks span 128 columns whatever the group size, and take
 *    a group argument only where groups of 64 are supported
 *    (fl_int4g_linear_g, fl_moe_int4g_g).
 *  - Canonical int4g triple (the storage the quantizer produces), G = K/group:
 *      q      uint8  [N, K/2]        codes 0..15, low nibble = even k
 *      scales uint16 [N, G]          IEEE fp16 bit patterns
 *      zeros  uint8  [N, ceil(G/2)]  zero points 0..15, low nibble = even g
 *    Dequantized weight: w' = s16 * (q - z).
 *  - Interleaved ("tiled") layout used by the matmul kernels, produced by
 *    fl_int4g_repack: rows are padded to a multiple of 128; super-block
 *    (T, g) -- rows 128T..128T+127, group g -- is 8512 contiguous bytes at
 *    offset (T * G + g) * 8512:
 *      [0, 8192)     codes, row r at r*64: logical column kk (0..127) goes to
 *                    32-bit word slot p = 4*(wl%4) + wl/4 (wl = kk/8) and
 *                    nibble e = 4*(o%2) + o/2 (o = kk%8) inside it; slot p
 *                    is word p%4 of 16-byte chunk c = p/4, and chunk c of
 *                    row r is stored at 16-byte position (c + (r/2)%4) % 4,
 *                    i.e. byte 16*pos + 4*(p%4) + e/2, high nibble iff e odd
 *                    (the rotation makes lanes that read one chunk of
 *                    consecutive rows hit distinct shared-memory banks);
 *      [8192, 8448)  128 fp16 scales, row r at 8192 + 2r (little endian);
 *      [8448, 8512)  128 zero points, row r in byte 8448 + r/2, low nibble
 *                    for even r.
 *    With groups of 256, super-blocks (T, 2j) and (T, 2j+1) both carry the
 *    scales and zero points of group j.  With groups of 64, super-block
 *    (T, g) carries those of group 2g (its columns 0..63), and a side array
 *    after all super-blocks, one 320-byte entry per super-block in the same
 *    order at offset (#super-blocks * 8512) + (T * G + g) * 320, carries
 *    those of group 2g+1: 128 fp16 scales (row r at 2r), then 128 zero
 *    points (row r in byte 256 + r/2, low nibble for even r).
 *    Size: 0.51953125 bytes per weight (the same as the canonical triple),
 *    plus padding rows.  Each super-block is one contiguous bulk copy.
 *  - All device pointers must be 16-byte aligned.
 *  - Every call is asynchronous on `stream` (0 = legacy default stream) and
 *    allocates no memory: the caller owns all buffers, including the
 *    workspaces whose sizes the *_workspace queries return.
 *  - Workspaces must be zero-filled before their first use.  Every entry
 *    point lays its workspace out the same way: a 16-byte status block, a
 *    counter region (up to byte 262,400) that a successful call leaves
 *    zero-filled again, and scratch after it.  So one workspace, sized for
 *    the largest query, can be reused by consecutive calls of any entry
 *    points on one stream.  Calls that run concurrently must not share a
 *    workspace; after a call reports a device-side error, zero the
 *    workspace again before reusing it.
 *  - The first 16 bytes of every workspace are a device status block; kernels
 *    OR error bits into it instead of trapping.  fl_int4g_status reads and
 *    clears it.
 *
 * Return values: FL_OK (0) or one of the FL_ERR_* codes below.  Argument
 * errors are detected on the host before anything is launched.
 */
#ifndef FL_INT4G_H
#define FL_INT4G_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fl_stream_t; /* same object as cudaStream_t */

#define FL_OK               0
#define FL_ERR_ARG          1  /* null/misaligned pointer, bad size, K % 128 != 0, ... */
#define FL_ERR_WORKSPACE    2  /* workspace smaller than the *_workspace query */
#define FL_ERR_UNSUPPORTED  3  /* group not 128 or 256, shape beyond a kernel limit */
#define FL_ERR_CUDA         4  /* a CUDA launch or query failed */
#define FL_ERR_TIMEOUT      5  /* a device-side bounded wait ran out (status word) */
#define FL_ERR_DEVICE_CHECK 6  /* a device-side check failed (status word) */
#define FL_ERR_RANGE        7  /* a group scale overflowed fp16 while quantizing (status word) */

#define FL_SOFTMAX 0
#define FL_SIGMOID 1

/* Human-readable name of a status code. Never NULL. */
const char* fl_strerror(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int fl_int4g_version(void);

/* ---------------------------------------------------------------- status */

/* Reads the device status block at `ws` (any workspace of this library, or
 * the status buffer given to fl_int4g_quantize), clears it, and stores in
 * *out FL_OK or the first device-side error recorded (FL_ERR_TIMEOUT,
 * FL_ERR_DEVICE_CHECK, FL_ERR_RANGE).  Synchronizes `stream`. */
int fl_int4g_status(void* ws, fl_stream_t stream, int* out);

/* --------------------------------------------------------- a1: quantize */

/* Online int4g quantization of fp32 weights w [N, K] (device) into the
 * canonical triple (device buffers q, scales, zeros as above).  Per group of
 * `group` (128 or 256) weights along K, in double precision:
 *   s = (max - min)/15, s16 = fp16(s) (nearest even),
 *   z = clamp(round(-min/s16), 0, 15), q = clamp(round(w/s16) + z, 0, 15),
 * round = half away from zero; a constant group c uses the range
 * [min(c,0), max(c,0)]; a zero group or s16 == 0 gives s16 = z = q = 0.
 * (FastLLM page, section 3.1: one scale and one zero point per group of
 * 128.)  A group whose s16 overflows fp16 is written as zeros and
 * FL_ERR_RANGE is recorded in the 16-byte device status block `status`
 * (zero-filled before first use; read it with fl_int4g_status). */
int fl_int4g_quantize(const float* w, int N, int K, int group,
                      uint8_t* q, uint16_t* scales, uint8_t* zeros,
                      void* status, fl_stream_t stream);

/* ------------------------------------------------------------ a2: repack */

/* Bytes of the interleaved layout for an [N, K] matrix (the same for groups
 * of 128 and 256: 8512 bytes per 128 rows x 128 columns). */
int fl_int4g_repacked_bytes(int N, int K, int group, size_t* out);

/* Canonical triple -> interleaved layout (FastLLM page, section 3.1:
 * weights reordered by group so that the matmul reads one contiguous span).
 * A pure, invertible permutation; bit-exact.  w_out must hold
 * fl_int4g_repacked_bytes(N, K) bytes; padding rows are written as zero. */
int fl_int4g_repack(const uint8_t* q, const uint16_t* scales, const uint8_t* zeros,
                    int N, int K, int group, void* w_out, size_t w_out_bytes,
                    fl_stream_t stream);

/* Inverse of fl_int4g_repack (for bit-exact round trips). */
int fl_int4g_unrepack(const void* w, size_t w_bytes, int N, int K, int group,
                      uint8_t* q, uint16_t* scales, uint8_t* zeros, fl_stream_t stream);

/* -------------------------------------------------- a3/a4: int4g linear */

/* Workspace bytes needed by fl_int4g_linear for this shape. */
int fl_int4g_linear_workspace(int M, int N, int K, size_t* out);

/* y[m, n] = sum_g s16[n,g] * sum_{k in g} x[m,k] * (q[n,k] - z[n,g]),
 * fp32 accumulation, bf16 output (FastLLM page, section 3.1: the 4-bit
 * weights are read, dequantized and multiplied in one pass).
 *   x  bf16 [M, K] device, row-major     w  interleaved layout of W [N, K]
 *   y  bf16 [M, N] device, row-major     ws workspace (see conventions)
 * M >= 1.  M <= 8: mma.sync decode kernel (HBM streaming, register-level
 * dequantization, split over K across the SMs, or per row tile across a
 * thread-block cluster reduced in distributed shared memory when the row
 * tiles are few); 8 < M <= 32: tcgen05 decode kernel (dequantized weights in
 * tensor memory); larger M: persistent tcgen05 prefill GEMM.  Reduction
 * order is fixed, so results are deterministic. */
int fl_int4g_linear(const void* x, int M, int K, const void* w, int N,
                    void* y, void* ws, size_t ws_bytes, fl_stream_t stream);

/* fl_int4g_linear for weights in the layout of any group size: group 128
 * or 256 (the same layout) is fl_int4g_linear; group 64 (FastLLM page,
 * section 5.4: groups of 64 for more precision) reads the side array of
 * the layout as well (fl_int4g_repack with group 64), each 64-column group
 * with its own scale and zero point.  The workspace is the one
 * fl_int4g_linear_workspace returns.  Group 64 runs the mma.sync decode
 * kernel for every M <= 32 and the tcgen05 prefill GEMM above.  Its ring
 * of stages sheds stages to fit 227 KB of shared memory; a shape that does
 * not fit even with two (many tokens, very long K and many row tiles, as
 * M = 32, K = 131072, N = 18432) returns FL_ERR_UNSUPPORTED before
 * launching anything.
 * FL_ERR_UNSUPPORTED for other group sizes. */
int fl_int4g_linear_g(const void* x, int M, int K, const void* w, int N, int group,
                      void* y, void* ws, size_t ws_bytes, fl_stream_t stream);

/* Decode linear (M <= 32) that allocates nothing and takes no workspace.
 * Not a step of the method: the pages have no counterpart; it exists for
 * callers that cannot allocate device memory where they call (cudaMalloc can
 * synchronize the device or fail under memory pressure, so latency-critical
 * loops and code inside frameworks that own all allocations avoid it).
 * Same arguments, same kernels and the same result, bit for bit, as
 * fl_int4g_linear for M <= 32; the split-K scratch lives in a 16 MiB array
 * inside the library that every GPU loading the library holds until exit.
 *  - The first call on a device looks up that array's device address
 *    (cudaGetSymbolAddress) with the device current: make it before any
 *    stream capture.  The address is cached per device and is not refreshed
 *    after a device reset: do not use this variant across one.
 *  - Every call shares the array, which keeps the last call's contents:
 *    calls whose executions overlap on the GPU (different streams, or graphs
 *    launched concurrently) race and must be serialized by the caller.  A
 *    successful call leaves the array's counters zero for the next one.
 *  - Device-side conditions (FL_ERR_TIMEOUT) are recorded in the array's
 *    status block: read them with fl_int4g_linear_noalloc_status before the
 *    next call on the device if they matter.
 *  - FL_ERR_UNSUPPORTED for M > 32; FL_ERR_WORKSPACE when the shape needs more
 *    scratch than the 16 MiB array (large N at M = 32); FL_ERR_ARG as for
 *    fl_int4g_linear. */
int fl_int4g_linear_noalloc(const void* x, int M, int K, const void* w, int N, void* y, fl_stream_t stream);

/* Reads and clears the device status block of fl_int4g_linear_noalloc's
 * array on the current device (as fl_int4g_status does for a workspace);
 * when an error was recorded it also clears the array's ticket counters, so
 * that the next call starts clean.  Synchronizes `stream`. */
int fl_int4g_linear_noalloc_status(fl_stream_t stream, int* out);

/* --------------------------------------- f3: fused decode MLP block */

/* Workspace bytes needed by fl_int4g_mlp. */
int fl_int4g_mlp_workspace(int M, int H, int I, size_t* out);

/* Decode MLP block, for 1 <= M <= 8 tokens:
 *   h = silu(G x) * (U x)  (h stored as bf16),   y = D h,
 * every product an int4g linear as in fl_int4g_linear (FastLLM page,
 * section 3.1; fastllm README, section 2: --dtype int4g applies to every
 * linear of the model).
 *   x       bf16 [M, H] device          y  bf16 [M, H] device
 *   w_gate  interleaved layout of G [I, H]     w_up  of U [I, H]
 *   w_down  interleaved layout of D [H, I]     ws    workspace (conventions)
 * H % 128 == 0, I % 128 == 0.  Two launches chained by programmatic launch:
 * the gate and up super-blocks stream through one decode kernel whose
 * thread-block clusters reduce each row tile and store h = silu(gate) * up,
 * then the down projection; shapes whose row tiles do not take that
 * cluster split run fl_int4g_mlp_fused.  Reduction order is fixed: results
 * are deterministic (both forms give the same h rounding, not the same
 * bits).  FL_ERR_UNSUPPORTED for M > 8. */
int fl_int4g_mlp(const void* x, int M, int H, int I, const void* w_gate, const void* w_up,
                 const void* w_down, void* y, void* ws, size_t ws_bytes, fl_stream_t stream);

/* The same block in ONE launch: a cooperative grid (two CTAs per SM) runs
 * gate/up with SwiGLU (split over K across the CTAs, ticketed partial sums),
 * hands h over through a grid-wide counter (a bounded wait: FL_ERR_TIMEOUT
 * in the status block if it runs out) and runs the down projection, while
 * the down weights already stream into the CTAs' rings.  Workspace as for
 * fl_int4g_mlp.  FL_ERR_UNSUPPORTED for M > 8 or when two CTAs per SM do not
 * fit. */
int fl_int4g_mlp_fused(const void* x, int M, int H, int I, const void* w_gate, const void* w_up,
                       const void* w_down, void* y, void* ws, size_t ws_bytes, fl_stream_t stream);

/* Test hook of the device-side failure path (no counterpart on the pages:
 * the library never traps or faults; a wait that runs out is reported).
 * ns >= 0: every later decode launch of fl_int4g_linear /
 * fl_int4g_linear_noalloc that reduces its row tiles across a thread-block
 * cluster withholds one arrival from each tile's reduction barrier, so the
 * bounded wait of the tile's first CTA runs out after ns nanoseconds.  That
 * CTA records FL_ERR_TIMEOUT in the status block, makes the missing arrival
 * itself, waits (normal bound) until its peers' partial sums have landed in
 * its shared memory, and exits without writing its rows of y.  ns < 0 (the
 * default) turns the hook off.  Process-wide; for tests only.  Always
 * FL_OK. */
int fl_int4g_test_withhold_cluster_arrival(long long ns);

/* Test hook: the plan of the decode kernel (M <= 8 mma.sync stream, and the
 * gate/up half of the decode MLP block when glu != 0) for one shape, computed
 * on the host without touching a GPU.  sms: the SM count to plan for; group:
 * 128 or 64; minb: CTAs per SM the kernel build holds (0: the default for M,
 * 3: the three-per-SM build); max_cs: the largest cluster to consider (the
 * launcher lowers it while clusters would crowd the GPU's capacity).
 * out[0..10] receives T (row tiles), G (groups), P (CTAs), csize (cluster
 * size, 1: stream-K), stages, stage bytes, dynamic shared memory bytes,
 * x-region stride (0: x travels in the stages), x-region offset, reduction
 * offset and zero-row offset.  FL_ERR_ARG for a shape the decode kernel
 * does not take or a bad argument; for tests only. */
int fl_int4g_test_decode_plan(int M, int N, int K, int sms, int group, int glu, int minb, int max_cs,
                              long long* out);

/* ------------------------------------------------------- a5-a7: MoE layer */

/* Workspace bytes needed by fl_moe_int4g. */
int fl_moe_int4g_workspace(int M, int E, int k, int H, int I, int has_shared, size_t* out);

/* Routed MoE expert FFN with int4g experts (fastllm README, sections
 * "2. 如何设定推理精度" --moe_dtype int4g and "5. 其它参数" --moe_experts,
 * --cuda_se):
 *   route:   top-k of the fp32 router logits [M, E] per token (ties to the
 *            lower expert index; slots ordered by descending logit, then
 *            ascending index); weights softmax over the selected k
 *            (FL_SOFTMAX, renorm=1), softmax over all E (renorm=0), or
 *            sigmoid of the selected, divided by their sum when renorm=1;
 *   permute: stable counting sort of assignments t*k+j by expert;
 *   experts: h = silu(G x) * (U x) with [G; U] = deq(W13_e) [2I, H]
 *            (gate rows first), h stored as bf16; out = deq(W2_e) h;
 *   combine: y[t] = sum_j w_{t,j} out_{t,j} (+ shared(x[t]) with weight 1).
 *   x       bf16 [M, H] device          logits fp32 [M, E] device
 *   w13     E interleaved [2I, H] matrices, back to back (stride
 *           fl_int4g_repacked_bytes(2I, H))
 *   w2      E interleaved [H, I] matrices, back to back
 *   shared_w13 / shared_w2   interleaved [2I, H] / [H, I] or both NULL
 *   y       bf16 [M, H] device
 *   topk_ids int32 [M, k], topk_w fp32 [M, k], expert_offsets int32 [E+1],
 *   perm int32 [M*k] -- optional device outputs (NULL = not written).
 * H % 128 == 0, I % 128 == 0, 1 <= k <= min(E, 32), E <= 1024, and
 * M * k <= 16384 (the permutation is one CTA's counting sort): larger
 * batches are split by the caller.  FL_ERR_ARG otherwise. */
int fl_moe_int4g(const void* x, const float* logits, int M, int H, int E, int k, int I,
                 int scoring, int renorm,
                 const void* w13, const void* w2,
                 const void* shared_w13, const void* shared_w2,
                 void* y, int32_t* topk_ids, float* topk_w,
                 int32_t* expert_offsets, int32_t* perm,
                 void* ws, size_t ws_bytes, fl_stream_t stream);

/* Routing options of fl_moe_int4g_ex.  fl_moe_int4g is this call with
 * score_bias = NULL, n_group = 1, topk_group = 1, routed_scale = 1.
 * score_bias / n_group > 1 select DeepSeek-V3 style (not on the FastLLM
 * pages, whose MoE options fix only top-k and the shared expert), with
 * scoring = FL_SIGMOID:
 *   s_e = sigmoid(l_e), key_e = s_e + score_bias[e] (the bias steers the
 *   choice only); experts form n_group runs of E/n_group, a group scores the
 *   sum of its two largest keys, the topk_group best groups are kept (ties:
 *   lower group index), and the top-k keys among their experts are chosen
 *   (ties: lower index; slots by descending key).  Keys are compared in
 *   double precision.  Weights: s_e of the chosen, divided by their sum when
 *   renorm.  In every mode the final weights are multiplied by routed_scale.
 * Errors (FL_ERR_ARG): a bias or n_group > 1 with softmax scoring,
 * E % n_group != 0, topk_group outside 1..n_group, k > topk_group * E /
 * n_group, routed_scale not positive and finite, a misaligned bias. */
typedef struct fl_moe_routing {
  int scoring;               /* FL_SOFTMAX or FL_SIGMOID */
  int renorm;                /* as in fl_moe_int4g */
  const float* score_bias;   /* fp32 [E] device, 16-byte aligned, or NULL */
  int n_group;               /* <= 1: no group limit */
  int topk_group;            /* groups kept per token when n_group > 1 */
  float routed_scale;        /* multiplies the final weights (1: none) */
} fl_moe_routing;

int fl_moe_int4g_ex(const void* x, const float* logits, int M, int H, int E, int k, int I,
                    const fl_moe_routing* routing,
                    const void* w13, const void* w2,
                    const void* shared_w13, const void* shared_w2,
                    void* y, int32_t* topk_ids, float* topk_w,
                    int32_t* expert_offsets, int32_t* perm,
                    void* ws, size_t ws_bytes, fl_stream_t stream);

/* ------------------------------------------- f2: router projection */

/* Workspace bytes needed by fl_moe_router_logits. */
int fl_moe_router_logits_workspace(int M, int H, int E, size_t* out);

/* Router logits of the routed MoE layer, logits = x . Wr^T, fp32
 * accumulation (the input of the top-k choice of fl_moe_int4g; the fastllm
 * README, section "5. 其它参数", sets only top-k; the dense projection is the
 * plain reading).
 *   x       bf16 [M, H] device, row-major     w_router bf16 [E, H] device, row-major
 *   logits  fp32 [M, E] device, row-major     ws       workspace (conventions)
 * H % 64 == 0, 1 <= E <= 65536.  Tensor cores (bf16 in, fp32 accumulate);
 * few output tiles split K over several CTAs, whose partials are summed in a
 * fixed order: deterministic. */
int fl_moe_router_logits(const void* x, int M, int H, const void* w_router, int E, float* logits,
                         void* ws, size_t ws_bytes, fl_stream_t stream);

/* fl_moe_int4g_ex for experts in the layout of any group size: group 128
 * or 256 is fl_moe_int4g_ex; group 64 (FastLLM page, section 5.4) reads
 * each expert matrix's side array as well.  Experts back to back with the
 * stride fl_int4g_repacked_bytes(rows, cols, group) (for group 64 that
 * includes the side array); the shared expert likewise.  The workspace is
 * the one fl_moe_int4g_workspace returns.  FL_ERR_UNSUPPORTED for other
 * group sizes. */
int fl_moe_int4g_g(const void* x, const float* logits, int M, int H, int E, int k, int I,
                   const fl_moe_routing* routing, int group,
                   const void* w13, const void* w2,
                   const void* shared_w13, const void* shared_w2,
                   void* y, int32_t* topk_ids, float* topk_w,
                   int32_t* expert_offsets, int32_t* perm,
                   void* ws, size_t ws_bytes, fl_stream_t stream);

/* fl_moe_int4g_ex with each expert's matrices at its own address: w13 and
 * w2 are DEVICE arrays of E device pointers (w13[e]: interleaved [2I, H] of
 * expert e, w2[e]: interleaved [H, I]), each 16-byte aligned, for callers
 * whose experts were loaded into separate allocations.  The tables are read
 * on the device, so a call can be captured in a CUDA graph and the caller
 * may update the tables between calls (stream order).  A null or misaligned
 * entry is detected on the device: FL_ERR_DEVICE_CHECK in the status block,
 * that expert's weight copies are skipped and the outputs of its tokens are
 * undefined.  The tables themselves must be 8-byte aligned (FL_ERR_ARG).
 * Everything else as fl_moe_int4g_ex. */
int fl_moe_int4g_ptrs(const void* x, const float* logits, int M, int H, int E, int k, int I,
                      const fl_moe_routing* routing,
                      const void* const* w13, const void* const* w2,
                      const void* shared_w13, const void* shared_w2,
                      void* y, int32_t* topk_ids, float* topk_w,
                      int32_t* expert_offsets, int32_t* perm,
                      void* ws, size_t ws_bytes, fl_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FL_INT4G_H */
