// attn_common.cuh -- epilogue arithmetic and small helpers shared by the two
// tensor-core kernels of the window attention usage (the single-SM kernel in
// attn_usage.cu and the CTA-pair kernel in attn_usage_pair.cu).
//
// What they compute ("Adaptive Mass-Segmented KV Compression for Long-Form
// Reasoning", Method, Key design 1): pass 1 keeps, per query row, an online
// maximum and the sum of exp2(scale*log2e*(z - max)) over the slots the row
// sees; pass 2 sums exp2(scale*log2e*z - b_r) over the query rows that see a
// slot, with b_r the row's log2 normaliser from pass 1.
#pragma once

#include <cmath>

#include "kvc_internal.cuh"

namespace kvc {
namespace attn {

constexpr int kChunkRows = 256;  // B-operand rows of one pass-2 row-constant block

// Row constants one pass-2 buffer holds: all chunks' rows (padding = -inf).
__host__ __device__ inline int rowb_floats(int R) { return ((R + kChunkRows - 1) / kChunkRows) * kChunkRows; }
__host__ __device__ inline int round4(int R) { return (R + 3) & ~3; }

// Warp-uniform wait, used by every role of the kernels: all 32 lanes wait on
// the barrier converged and vote on the outcome, so that what follows (the
// collective TMEM loads of the epilogue, or one lane's copy or MMA issue in
// the producer roles) runs converged.  A wait by lane 0 alone, with the other
// lanes parked at a shuffle or at the end of the role, issued about a tenth
// more instructions and took 8% longer on the 28-layer batch-32 event.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity,
                                          volatile int* abort, uint32_t* status) {
  const bool ok = mbar_wait(bar, parity, abort, status);
  return __all_sync(0xffffffffu, ok);
}

// Bounded wait that ignores the abort flag (used to drain in-flight work).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity,
                                           uint32_t* status) {
  volatile int never = 0;
  mbar_wait(bar, parity, &never, status);
}

__device__ __forceinline__ float4 lds128(const float* ptr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(smem_u32(ptr)));
  return v;
}

// 1-D bulk copy global -> shared (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
      "[%3];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Pass-1 row statistics of one 32-column block: online max (rescaling the
// running sum when it grows) and the sum of exp2(c*z - c*max) over the block's
// valid columns [lo, hi] (all of them when FULL; the masked form is a separate
// instantiation so that its selects never run on full blocks).
template <bool FULL>
__device__ __forceinline__ void row_block(const uint32_t (&v)[32], float bmx, int p0, int lo,
                                          int hi, float c, float& mz, float& sum) {
  // valid columns of the block as a bit mask (bit i = column p0 + i)
  uint32_t valid = 0xffffffffu;
  if constexpr (!FULL) {
    const int a = max(lo - p0, 0), b = min(hi - p0, 31);
    valid = (b < a) ? 0u : ((0xffffffffu >> (31 - b)) & (0xffffffffu << a));
  }
  float bm = bmx;
  if constexpr (!FULL) {
    bm = -INFINITY;
#pragma unroll
    for (int i = 0; i < 32; ++i)
      bm = (valid & (1u << i)) ? fmaxf(bm, __uint_as_float(v[i])) : bm;
  }
  // rescale only when some row's maximum grew (warp-uniform test)
  if (__any_sync(0xffffffffu, bm > mz)) {
    const float sc = bm > mz ? ex2((mz - bm) * c) : 1.f;
    sum *= sc;
    mz = fmaxf(mz, bm);
  }
  const float neg = -mz * c;
  const float2 cc = make_float2(c, c), nn = make_float2(neg, neg);
  float2 e[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    e[i] = fma2(make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])), cc, nn);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    e[i].x = ex2(e[i].x);
    e[i].y = ex2(e[i].y);
  }
  if constexpr (!FULL) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      e[i].x = (valid & (1u << (2 * i))) ? e[i].x : 0.f;
      e[i].y = (valid & (2u << (2 * i))) ? e[i].y : 0.f;
    }
  }
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) e[i] = add2(e[i], e[i + w]);
  sum += e[0].x + e[0].y;
}

// Pass-2 slot usage of one 32-row block (query rows r0 .. r0+31): sum of
// exp2(c*z - b_r) with the negated row constants from shared memory; rows of
// window index j < jmin do not see the slot (dropped unless FULL).
template <bool FULL>
__device__ __forceinline__ void slot_block(const uint32_t (&v)[32], const float* rbb, int r0,
                                           int W, int jmin, float c,
                                           float2& acc) {
  const float2 cc = make_float2(c, c);
  float2 e[16];
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    const float4 nb = lds128(rbb + 2 * i);  // negated row constants (-inf past R)
    e[i] = fma2(make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])), cc,
                make_float2(nb.x, nb.y));
    e[i + 1] = fma2(make_float2(__uint_as_float(v[2 * i + 2]), __uint_as_float(v[2 * i + 3])),
                    cc, make_float2(nb.z, nb.w));
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    e[i].x = ex2(e[i].x);
    e[i].y = ex2(e[i].y);
  }
  if constexpr (!FULL) {
    const int j0 = r0 % W;
    if (W % 32 == 0) {
      // the block's rows are window indices j0 .. j0+31 (no wrap)
      const int first = jmin - j0;  // rows i >= first see the slot
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        e[i].x = 2 * i >= first ? e[i].x : 0.f;
        e[i].y = 2 * i + 1 >= first ? e[i].y : 0.f;
      }
    } else {
      int j = j0;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        e[i].x = j >= jmin ? e[i].x : 0.f;
        j = (j + 1 == W) ? 0 : j + 1;
        e[i].y = j >= jmin ? e[i].y : 0.f;
        j = (j + 1 == W) ? 0 : j + 1;
      }
    }
  }
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) e[i] = add2(e[i], e[i + w]);
  acc = add2(acc, e[0]);
}

// Both blocks of a fully visible 64-column step at once (pass 1): one rescale
// decision for the pair, then 64 independent exponentials and one sum tree.
__device__ __forceinline__ void row_pair(const uint32_t (&v)[2][32], const float (&bmx)[2],
                                         float c, float& mz, float& sum) {
  const float bm = fmaxf(bmx[0], bmx[1]);
  if (__any_sync(0xffffffffu, bm > mz)) {
    const float sc = bm > mz ? ex2((mz - bm) * c) : 1.f;
    sum *= sc;
    mz = fmaxf(mz, bm);
  }
  const float neg = -mz * c;
  const float2 cc = make_float2(c, c), nn = make_float2(neg, neg);
  float2 e[32];
#pragma unroll
  for (int b = 0; b < 2; ++b)
#pragma unroll
    for (int i = 0; i < 16; ++i)
      e[16 * b + i] = fma2(make_float2(__uint_as_float(v[b][2 * i]),
                                       __uint_as_float(v[b][2 * i + 1])), cc, nn);
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    e[i].x = ex2(e[i].x);
    e[i].y = ex2(e[i].y);
  }
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) e[i] = add2(e[i], e[i + w]);
  sum += e[0].x + e[0].y;
}

// Both blocks of a 64-row step seen by every query row (pass 2).
__device__ __forceinline__ void slot_pair(const uint32_t (&v)[2][32], const float* rbb, float c,
                                          float2& acc) {
  const float2 cc = make_float2(c, c);
  float2 e[32];
#pragma unroll
  for (int b = 0; b < 2; ++b)
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      const float4 nb = lds128(rbb + 32 * b + 2 * i);  // negated row constants (-inf past R)
      e[16 * b + i] = fma2(make_float2(__uint_as_float(v[b][2 * i]),
                                       __uint_as_float(v[b][2 * i + 1])), cc,
                           make_float2(nb.x, nb.y));
      e[16 * b + i + 1] = fma2(make_float2(__uint_as_float(v[b][2 * i + 2]),
                                           __uint_as_float(v[b][2 * i + 3])), cc,
                               make_float2(nb.z, nb.w));
    }
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    e[i].x = ex2(e[i].x);
    e[i].y = ex2(e[i].y);
  }
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) e[i] = add2(e[i], e[i + w]);
  acc = add2(acc, e[0]);
}

// Copy two 32-column blocks of this warp's accumulator rows to registers,
// with the per-block maxima from the load path when `with_max` (warp-uniform).
__device__ __forceinline__ void load2(uint32_t taddr, bool with_max, uint32_t (&v)[2][32],
                                      float (&bmx)[2]) {
  if (with_max) {
    tmem_ld32_max(taddr, v[0], bmx[0]);
    tmem_ld32_max(taddr + 32, v[1], bmx[1]);
  } else {
    tmem_ld32(taddr, v[0]);
    tmem_ld32(taddr + 32, v[1]);
    bmx[0] = bmx[1] = -INFINITY;
  }
}

}  // namespace attn
}  // namespace kvc
