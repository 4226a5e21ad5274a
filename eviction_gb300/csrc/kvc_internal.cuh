// kvc_internal.cuh -- shared internals of the sm_103a compression-event library:
// the handle, kernel launch declarations, and thin inline-PTX wrappers for
// mbarrier, TMA (cp.async.bulk.tensor) and the 5th-generation tensor core
// (tcgen05: TMEM allocation, MMA, commit, TMEM loads).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "kvc.h"

namespace kvc {

// ---------------------------------------------------------------- handle ----

struct Workspace {
  float* negb = nullptr;        // [U][Rp] -log2 row normaliser (Rp = R rounded to 4)
  float* pmax = nullptr;        // [U][Rp] largest probability of each row
  float* usage = nullptr;       // [U][max_T] raw usage (no fill)
  float* mass = nullptr;        // [U][max_T]   (event intermediates)
  float* score = nullptr;       // [U][max_T]
  float* credit_post = nullptr; // [U][max_T]
  int32_t* seg_start = nullptr; // [U][S_max(max_T)]
  int32_t* seg_len = nullptr;
  int32_t* quota = nullptr;
  int32_t* n_seg = nullptr;     // [U]
  uint32_t* status = nullptr;   // device status bits; status[1] = the error word of
                                // the running paged compaction
  void* base = nullptr;         // single allocation
  size_t bytes = 0;
};

struct Dims {
  int L, B, H, G, W, d, R, U;  // R = G*W query rows per unit, U = L*B*H units
};

}  // namespace kvc

namespace kvc {

enum KernelId {
  kKernelUsagePass1 = 0,
  kKernelUsagePass2,
  kKernelMass,
  kKernelSegmentQuota,
  kKernelSelect,
  kKernelCompact,
  kKernelRefresh,
  kKernelCompactPaged,
  kKernelRedundancy,
  kKernelUnitPost,
  kNumKernels
};

// Per-kernel CUDA-event tracing (see kvc_profile in kvc.h).
struct Profiler {
  bool enabled = false;
  struct Mark {
    int kernel;
    cudaEvent_t begin, end;
  };
  std::vector<cudaEvent_t> pool;
  std::vector<Mark> pending;
  cudaEvent_t last = nullptr;  // most recent event on the traced stream
  int launches[kNumKernels] = {};
  double total_ms[kNumKernels] = {};
};

}  // namespace kvc

namespace kvc {
// Copy streams and events of kvc_event_host (created with the handle).
constexpr int kMaxHostStages = 64;
struct HostIO {
  cudaStream_t in = nullptr, out[2] = {nullptr, nullptr};  // device -> host on two streams:
  cudaEvent_t start = nullptr, end[2] = {nullptr, nullptr};  // one alone reaches ~1/3 of the link
  cudaEvent_t landed[kMaxHostStages] = {};  // a stage's inputs are on the device
  cudaEvent_t done[kMaxHostStages] = {};    // a stage's outputs are written
};
}  // namespace kvc

struct kvc_handle {
  kvc_config cfg;
  kvc::Dims dims;
  kvc::Workspace ws;
  int device = 0;
  int num_sms = 0;
  size_t smem_optin = 0;  // shared memory a block may opt in to
  std::string last_error;
  kvc::Profiler prof;
  kvc::HostIO io;
};

namespace kvc {

// ------------------------------------------------------------ launchers ----
// All return cudaSuccess or the launch error.  Defined next to their kernels.

struct UsageArgs {
  const uint16_t* q;
  const uint16_t* k;
  const int32_t* pad;
  int T;
  float scale_log2;  // softmax scale * log2(e)
};

// One pass (1 or 2) of the window attention usage (tcgen05 kernels).
cudaError_t launch_attention_usage(const kvc_handle* h, const UsageArgs& a,
                                   int pass, cudaStream_t s, std::string* err);

// The same pass on CTA pairs (cta_group::2, M256 x N128), attn_usage_pair.cu.
cudaError_t launch_attention_usage_pair(const kvc_handle* h, const UsageArgs& a,
                                        int pass, cudaStream_t s, std::string* err);

cudaError_t launch_mass_post(const kvc_handle* h, int T, const int32_t* pad,
                             const int32_t* n_carry, const float* credit_in,
                             float* credit_post, float* mass, float* score,
                             cudaStream_t s);

cudaError_t launch_segment_quota(const kvc_handle* h, const float* mass, int T,
                                 const int32_t* pad, int32_t* seg_start,
                                 int32_t* seg_len, int32_t* quota,
                                 int32_t* n_seg, cudaStream_t s);

cudaError_t launch_select(const kvc_handle* h, const float* score, int T,
                          const int32_t* pad, const int32_t* seg_start,
                          const int32_t* seg_len, const int32_t* quota,
                          const int32_t* n_seg, int32_t* kept_idx,
                          int32_t* n_kept, cudaStream_t s);

// Mass, segmentation with quotas and selection fused in one launch (one CTA
// per unit, unit_post.cu); for units of up to 4096 slots.  Same outputs, bit
// for bit, as launch_mass_post + launch_segment_quota + launch_select.
cudaError_t launch_unit_post(const kvc_handle* h, int T, const int32_t* pad,
                             const int32_t* n_carry, const float* credit_in,
                             float* credit_post, float* mass, float* score, int32_t* seg_start,
                             int32_t* seg_len, int32_t* quota, int32_t* n_seg,
                             int32_t* kept_idx, int32_t* n_kept, cudaStream_t s);

// Shared memory of the fused kernel for units of T slots (0: T too long for it).
size_t unit_post_smem_bytes(const kvc_config& c, int T);

// Host validation of a configuration (every field, and the unit and row counts
// in 64-bit arithmetic); KVC_OK or a negative code with the reason in *why.
int validate_config(const kvc_config* c, std::string* why);

cudaError_t launch_compact(const kvc_handle* h, const uint16_t* k,
                           const uint16_t* v, const float* credit_post, int T,
                           const int32_t* kept_idx, const int32_t* n_kept,
                           uint16_t* k_out, uint16_t* v_out,
                           float* credit_out, cudaStream_t s);

struct PagedArgs {
  uint16_t* k_pool;
  uint16_t* v_pool;
  int n_blocks, block_size, max_blocks, T;
  const int32_t* seq_len;
  const int32_t* pad;
  const int32_t* kept_idx;
  const int32_t* n_kept;
  const float* credit_post;
  float* credit_out;
  const int32_t* table_old;
  int32_t* table_new;
  int32_t* free_list;
  int32_t* free_top;
};

// Paged compaction (validate, allocate, copy, free); errors land in the word
// after the status word and are OR-ed into the status at the end.
cudaError_t launch_compact_paged(const kvc_handle* h, const PagedArgs& a, cudaStream_t s);

cudaError_t launch_refresh(const kvc_handle* h, const uint16_t* q, float* q_ref,
                           float threshold, int32_t* flag, float* sim, cudaStream_t s);

// SkipKV key-redundancy score mixed into the selection score (sel may alias
// score); red (optional) receives the softmax-normalised redundancy.
cudaError_t launch_redundancy(const kvc_handle* h, const uint16_t* k, const float* score, int T,
                              const int32_t* pad, float* sel, float* red, cudaStream_t s);
size_t redundancy_smem_bytes(int D, int T);

// One thread waits (bounded) on a barrier nothing completes: the timeout path.
cudaError_t launch_wait_self_test(const kvc_handle* h, cudaStream_t s);

inline int s_max_of(const kvc_config& c, int T) {
  int s = T / c.seg_min;
  return s > 1 ? s : 1;
}

// ------------------------------------------------------ device helpers ----

#if defined(__CUDACC__)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bound on any single wait of a pipeline role (ns).  Correct code waits
// microseconds; the bound only exists so that a broken pipeline reports an
// error instead of hanging the GPU.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar,
                                                      uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_test, but a thread whose phase is not complete yet is suspended
// until it completes or about `hint_ns` have passed (it does not spin and so
// leaves the issue slots of its SM sub-partition to the other warps).
__device__ __forceinline__ bool mbar_test_sleep(uint64_t* bar, uint32_t parity,
                                                uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Suspension hint of one wait step: short enough that the abort flag and the
// time limit are checked often.
constexpr uint32_t kWaitSleepNs = 20000;

// Wait for the phase of `bar` with the given parity to complete.  Gives up
// after kWaitLimitNs or as soon as *abort becomes non-zero; returns false then
// (and on its own time-out raises *abort and the device status bit).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          volatile int* abort,
                                          uint32_t* status) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_test_sleep(bar, parity, kWaitSleepNs)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      atomicOr(status, KVC_STATUS_WAIT_TIMEOUT);
      return false;
    }
  }
}

// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_now(uint64_t* bar, uint32_t parity) {
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

// As mbar_wait, but polling without suspending the thread, with the same time
// limit and abort flag (checked every 256 polls).
__device__ __forceinline__ bool mbar_wait_poll(uint64_t* bar, uint32_t parity,
                                               volatile int* abort, uint32_t* status) {
  if (mbar_test_now(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_test_now(bar, parity)) return true;
    if ((i & 255u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        *abort = 1;
        atomicOr(status, KVC_STATUS_WAIT_TIMEOUT);
        return false;
      }
    }
  }
}

// 2-D tiled TMA load global -> shared, completion on `bar` (transaction bytes).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map,
                                            int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_"
      "tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y),
      "r"(smem_u32(bar))
      : "memory");
}

// Hint: bring a 2-D tile of `map` into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

// Hint: bring `bytes` (a multiple of 16) at 16-byte aligned `src` into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                   reinterpret_cast<uint64_t>(src)),
               "r"(bytes)
               : "memory");
}

// 3-D tiled TMA load (x, y, z), completion on `bar` (transaction bytes).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y,
                                            int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map))
               : "memory");
}

// ---- tcgen05 ----

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile(
      "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
          smem_u32(slot)),
      "r"(ncols)
      : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile(
      "tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
      "r"(ncols)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row core-matrix groups 1024 bytes apart.  `addr` must lie in a
// 1024-byte aligned tile (plus the K-slice byte offset within the row).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
  uint64_t desc = 0;
  desc |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);  // start address
  desc |= static_cast<uint64_t>(1) << 16;                  // LBO (unused)
  desc |= static_cast<uint64_t>(1024 >> 4) << 32;          // SBO
  desc |= static_cast<uint64_t>(1) << 46;                  // descriptor version
  desc |= static_cast<uint64_t>(2) << 61;                  // SWIZZLE_128B
  return desc;
}

// Instruction descriptor, kind::f16: A = B = bf16, D = f32, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4)                                   // D format f32
         | (1u << 7)                                 // A format bf16
         | (1u << 10)                                // B format bf16
         | (static_cast<uint32_t>(N >> 3) << 17)     // N
         | (static_cast<uint32_t>(M >> 4) << 24);    // M
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc,
                                         uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 op issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 "
      "[%0];" ::"r"(smem_u32(bar))
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane
// (warp's lane quarter)*32 + i, columns col..col+31.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, "
      "[%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]),
        "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]),
        "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// As tmem_ld32, and also the maximum of the 32 loaded fp32 values of the lane
// (computed by the TMEM load path itself).
__device__ __forceinline__ void tmem_ld32_max(uint32_t taddr, uint32_t (&r)[32],
                                              float& mx) {
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, "
      "%32, [%33];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]),
        "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]),
        "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31]), "=f"(mx)
      : "r"(taddr)
      : "memory");
}

// ---- CTA pairs (cluster of two CTAs sharing one MMA: tcgen05 .cta_group::2) ----
// Every tcgen05 instruction of a kernel uses the same .cta_group, so a paired
// kernel allocates, issues and commits with these forms only.

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Shared::cluster address of the object at local shared address `local` in
// the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

// All threads of both CTAs: release this CTA's prior shared-memory writes
// (barrier inits included) to the cluster, then wait for the peer.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

// Arrive once on an mbarrier given by its shared::cluster address (this CTA's
// or the peer's).  Default semantics (release at CTA scope): a cluster-scope
// release would be a full memory barrier on every call, and the hazard it
// guards here -- this warp's tensor-memory reads against the next MMA's
// writes -- is ordered by tcgen05.fence::before_thread_sync before the arrive.
#ifndef KVC_REMOTE_ARRIVE_RELAXED
#define KVC_REMOTE_ARRIVE_RELAXED 0
#endif
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
#if KVC_REMOTE_ARRIVE_RELAXED
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
#else
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
#endif
}

// 3-D tiled TMA load into this CTA's shared memory whose completion (bytes)
// is counted on the mbarrier at shared::cluster address `bar` -- the pair's
// leading CTA's barrier, for the operands its MMA reads from both CTAs.
__device__ __forceinline__ void tma_load_3d_pair(void* dst, const CUtensorMap* map, int x, int y,
                                                 int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// One warp of EACH CTA of the pair executes these together: the columns are
// allocated at the same address in both CTAs' tensor memory.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// D[M x N] (+)= A * B^T over both CTAs: each CTA holds M/2 rows of A and N/2
// rows of B at the same shared-memory offsets and receives its M/2 rows of D
// at the same tensor-memory address.  Issued by one thread of the leading CTA.
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the mbarrier at local offset `bar` in every CTA of `cta_mask`
// when all tcgen05 ops this thread issued so far are done.
__device__ __forceinline__ void mma_commit_pair_multicast(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// As above, on this CTA's own barrier only.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Packed pair arithmetic (two fp32 lanes per instruction, FFMA2 / FADD2).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Hardware base-2 exponential (MUFU), flush-to-zero.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Order-preserving map of a float to uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t float_order_key(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

#endif  // __CUDACC__

}  // namespace kvc
