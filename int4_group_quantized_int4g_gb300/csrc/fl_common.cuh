// Shared device helpers for the int4g kernels (sm_103a): status block,
// mbarrier + bulk-copy pipeline primitives, mma.sync, nibble -> bf16 unpack.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fl_int4g.h"

namespace fl {

constexpr int kGroup = 128;     // weights per group along K
constexpr int kRowTile = 128;   // rows per super-block
constexpr int kSbNib = 8192;    // 128 rows x 64 B of codes
constexpr int kSbScale = 256;   // 128 fp16 scales
constexpr int kSbZero = 64;     // 128 4-bit zero points
constexpr int kSbBytes = kSbNib + kSbScale + kSbZero;  // 8512
constexpr int kSbSide = kSbScale + kSbZero;             // 320: groups of 64, the odd group's scales and zeros
constexpr int kStatusBytes = 16;
// Workspace layout shared by every split kernel of the linear: the status
// block, then ticket counters for up to kTicketTiles tiles x 8 warps at a fixed
// offset (a workspace reused across shapes always finds them zero: each last
// arriver resets its counter), then scratch from kScratchOff.
constexpr int kTicketTiles = 8192;
constexpr int kTicketWarps = 8;
constexpr size_t kTicketOff = kStatusBytes;
constexpr size_t kScratchOff = (kTicketOff + static_cast<size_t>(kTicketTiles) * kTicketWarps * 4 + 255) / 256 * 256;

// Upper bound for any device-side wait (ns).  A wait that runs out records
// FL_ERR_TIMEOUT in the status block and the kernel winds down.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// ----------------------------------------------------------------- status
// Status block: int32 [0] first error code, [1] OR of (1 << code), [2] detail.
__device__ __forceinline__ void set_status(int32_t* st, int code, int detail) {
  atomicCAS(st, 0, code);
  atomicOr(st + 1, 1 << code);
  st[2] = detail;
}

// Base of expert e's interleaved matrix: entry e of a device table of
// expert pointers when one is given, else w + e * wbytes (experts back to
// back).  A null or misaligned table entry is recorded in the status block
// (FL_ERR_DEVICE_CHECK) and returned as null: the caller skips its copy.
__device__ __forceinline__ const uint8_t* expert_base(const uint8_t* w, const uint8_t* const* wtab, size_t wbytes,
                                                      int e, int32_t* status) {
  if (!wtab) return w + static_cast<size_t>(e) * wbytes;
  const uint8_t* b = wtab[e];
  if (b == nullptr || (reinterpret_cast<uintptr_t>(b) & 15u) != 0) {
    set_status(status, FL_ERR_DEVICE_CHECK, 30);
    return nullptr;
  }
  return b;
}

// ----------------------------------------------------------------- smem/ptx
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// One try of a phase wait.  The suspend-time hint lets the hardware park the
// thread until the phase completes (or ~0.5 ms pass) instead of polling, so
// waiting warps leave their issue slots to the warps doing the work.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(500000u)
      : "memory");
  return ok != 0;
}

// Non-blocking probe of phase `parity` of `bar`.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for phase `parity` of `bar`; false when the limit ran out.
// A phase that has already completed is seen by the cheap probe.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_test(bar, parity)) return true;
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// L2 policy for data read exactly once (streamed weights).
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.
// dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// GPU-scope acquire/release fence (lighter than the sequentially consistent
// fence behind __threadfence) for ticket hand-offs between CTAs.
// Block barrier after code in which the lanes of a warp took different paths
// (a lane-0 producer or MMA loop, a thread-0 setup block): each warp first
// reconverges, so that the aligned barrier is always reached by whole warps.
__device__ __forceinline__ void cta_sync() {
  __syncwarp();
  __syncthreads();
}

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
// atomic add at GPU scope with acquire-release semantics; returns the old value
__device__ __forceinline__ int atom_add_acq_rel_gpu(int32_t* p, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ int ld_acquire_gpu(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Programmatic dependent launch: let the next kernel in the stream start its
// CTAs now / wait until the previous kernel has completed and its memory
// operations are visible.  Both are no-ops without the launch attribute.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Thread-block clusters: full barrier of every thread of the cluster (all
// CTAs of a cluster are resident together, so it cannot wait on a CTA that
// has not started).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Generic address of the same shared-memory object in cluster rank 0.
template <typename T>
__device__ __forceinline__ T* cluster_map_rank0(T* p) {
  uint64_t out;
  asm volatile("mapa.u64 %0, %1, 0;" : "=l"(out) : "l"(reinterpret_cast<uint64_t>(p)));
  return reinterpret_cast<T*>(out);
}
// Bounded wait, acquire at cluster scope (for arrivals made by other CTAs of
// the cluster with release.cluster); false when the limit ran out.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait_cluster(bar, parity)) {
    if (globaltimer() - t0 > limit_ns) return false;
  }
  return true;
}
// Arrive (release, cluster scope) on the same mbarrier in cluster rank 0.
__device__ __forceinline__ void mbar_arrive_remote_rank0(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b32 ra;\n\t"
      "mapa.shared::cluster.u32 ra, %0, 0;\n\t"
      "mbarrier.arrive.release.cluster.shared::cluster.b64 _, [ra];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

// Named barrier over `nthreads` threads (multiple of 32).
__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ----------------------------------------------------------------- math
// D += A(16x16, bf16, row) * B(16x8, bf16, col), fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// (a & b) | c in one LOP3.
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Nibbles i and i+4 of a 32-bit word as a bf16 pair (128 + q_i, 128 + q_{i+4}):
// OR-ing a 4-bit code into the mantissa of bf16 128.0 (0x4300) gives 128 + q
// exactly, because the bf16 spacing at 128 is 1.
__device__ __forceinline__ uint32_t nib_pair_bf16(uint32_t word, int i) {
  return lop3_and_or(word >> (4 * i), 0x000F000Fu, 0x43004300u);
}

// Exact (q - z) for both halves: (128 + q) - (128 + z), |q - z| <= 15.
__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  __nv_bfloat162 r = __hsub2(*reinterpret_cast<__nv_bfloat162*>(&a), *reinterpret_cast<__nv_bfloat162*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t bf16_bias_pair(uint32_t z) { return (0x4300u + z) * 0x00010001u; }

}  // namespace fl

// Host-side helpers shared by the launchers.
namespace flh {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int sm_count();  // cached per device (fl_abi.cu)

}  // namespace flh
