// paged.cu -- compaction into a paged KV pool: allocate new blocks, copy each
// head's kept rows into them, hand the old blocks back.
//
// "Adaptive Mass-Segmented KV Compression for Long-Form Reasoning", Appendix E:
// selection is separate from the paged storage layout.  From the per-head
// kept indices the runtime allocates new blocks, copies each head's KV from
// its original positions into the new physical slots, replaces the request's
// block table and frees the old blocks; the same compacted slot may hold
// different original positions in different heads.
//
// Layout: pools [L][n_blocks][H][bs][d] bf16 (a head's rows of a block are
// contiguous), one block table per sequence shared by every layer (logical
// token t lives in block table[b][t / bs], row t % bs).  The free blocks are a
// stack (free_list[0, *free_top)).  Four launches on one stream:
//   1. validate every kept index against the old table (any failure sets the
//      call's error word; nothing below changes anything then);
//   2. allocate (one CTA): a block scan of ceil(n_kept_b / bs) over sequences
//      takes the top entries of the stack in sequence order -- deterministic;
//   3. copy kept rows (row offsets resolved once into shared memory, then
//      16-byte vectors with several loads in flight), plus the dense credit gather;
//   4. free (one CTA): push each sequence's old blocks in sequence order.
// Old and new blocks coexist between 2 and 4, as the appendix notes.
#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kScanThreads = 1024;

struct PagedParams {
  int L, B, H, d, bs, n_blocks, max_blocks, budget, T;
  int unit0;  // first unit of a copy launch (units go in chunks of gridDim.y <= 65535)
  uint16_t* k_pool;
  uint16_t* v_pool;
  const int32_t* seq_len;
  const int32_t* pad;
  const int32_t* kept;
  const int32_t* n_kept;
  const float* credit_post;
  float* credit_out;
  const int32_t* table_old;
  int32_t* table_new;
  int32_t* free_list;
  int32_t* free_top;
  uint32_t* err;     // this call's error word (0 = fine)
  uint32_t* status;  // the handle's sticky status bits
};

__global__ void paged_validate_kernel(PagedParams p) {
  const int u = blockIdx.x;  // (l, b, h)
  const int b = (u / p.H) % p.B;
  const int nk = p.n_kept[u];
  const int nk0 = p.n_kept[static_cast<size_t>(b) * p.H];  // layer 0, head 0
  bool bad = nk != nk0 || nk < 0 || nk > p.budget ||
             (nk + p.bs - 1) / p.bs > p.max_blocks;
  for (int j = threadIdx.x; !bad && j < nk; j += blockDim.x) {
    const int t = p.kept[static_cast<size_t>(u) * p.budget + j] - p.pad[b];
    if (t < 0 || t >= p.seq_len[b]) {
      bad = true;
    } else {
      const int blk = p.table_old[static_cast<size_t>(b) * p.max_blocks + t / p.bs];
      bad = blk < 0 || blk >= p.n_blocks;
    }
  }
  if (u == 0 && threadIdx.x == 0 && (*p.free_top < 0 || *p.free_top > p.n_blocks)) bad = true;
  if (bad) atomicOr(p.err, KVC_STATUS_BAD_INDEX);
}

// Exclusive block scan of one value per thread (kScanThreads threads); *total
// receives the sum.
__device__ int block_exclusive_scan(int v, int* total) {
  __shared__ int warp_sums[kScanThreads / 32];
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kScanThreads / 32 ? warp_sums[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    if (lane < kScanThreads / 32) warp_sums[lane] = wi - w;
    if (lane == 31) *total = wi;
  }
  __syncthreads();
  const int r = warp_sums[warp] + incl - v;
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kScanThreads) paged_alloc_kernel(PagedParams p) {
  __shared__ int s_total, s_need, s_err, s_bad;
  if (threadIdx.x == 0) {
    s_need = 0;
    s_bad = 0;
    s_err = *p.err != 0;
  }
  __syncthreads();
  if (s_err) return;  // CTA-uniform
  // total need first (a pass over all sequences), then allocate chunk by chunk
  for (int b0 = 0; b0 < p.B; b0 += kScanThreads) {
    const int b = b0 + threadIdx.x;
    const int need = b < p.B ? (p.n_kept[static_cast<size_t>(b) * p.H] + p.bs - 1) / p.bs : 0;
    int total;
    block_exclusive_scan(need, &s_total);
    __syncthreads();
    total = s_total;
    if (threadIdx.x == 0) s_need += total;
    __syncthreads();
  }
  const int top = *p.free_top;
  if (s_need > top) {
    if (threadIdx.x == 0) atomicOr(p.err, KVC_STATUS_POOL_EXHAUSTED);
    return;  // CTA-uniform
  }
  int base = top - s_need;
  for (int b0 = 0; b0 < p.B; b0 += kScanThreads) {
    const int b = b0 + threadIdx.x;
    const int need = b < p.B ? (p.n_kept[static_cast<size_t>(b) * p.H] + p.bs - 1) / p.bs : 0;
    const int off = block_exclusive_scan(need, &s_total);
    if (b < p.B) {
      int32_t* row = p.table_new + static_cast<size_t>(b) * p.max_blocks;
      for (int i = 0; i < p.max_blocks; ++i) {
        const int blk = i < need ? p.free_list[base + off + i] : -1;
        if (i < need && (blk < 0 || blk >= p.n_blocks)) s_bad = 1;  // a corrupt free list
        row[i] = blk;
      }
    }
    __syncthreads();
    base += s_total;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    if (s_bad)
      atomicOr(p.err, KVC_STATUS_BAD_INDEX);
    else
      *p.free_top = top - s_need;
  }
}

// grid (ceil(budget / rows_per_cta), L*B*H); 16-byte vectors, rows_per_cta rows
constexpr int kCopyRows = 64;      // kept rows per CTA
constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;     // 16-byte loads in flight per thread

// Copy kept rows into the new blocks.  The row offsets (source position in an
// old block, destination row of a new block) and the credit are resolved once
// per row into shared memory; the rows then move as 16-byte vectors with
// several loads in flight per thread.  Old and new blocks are disjoint (new
// blocks come off the free stack), so reads and writes never overlap.
__global__ void __launch_bounds__(kCopyThreads) paged_copy_kernel(PagedParams p, int vpr_log2) {
  __shared__ long long s_src[kCopyRows], s_dst[kCopyRows];  // 16-byte units; -1 = no row
  if (*p.err) return;  // the same value for every thread: written by the validation launch
  const int u = p.unit0 + static_cast<int>(blockIdx.y);
  const int h = u % p.H;
  const int b = (u / p.H) % p.B;
  const int l = u / (p.H * p.B);
  const int nk = p.n_kept[u];
  const int j0 = blockIdx.x * kCopyRows;
  const int rows = min(kCopyRows, p.budget - j0);
  for (int r = threadIdx.x; r < rows; r += kCopyThreads) {
    const int j = j0 + r;
    const size_t cj = static_cast<size_t>(u) * p.budget + j;
    if (j < nk) {
      const int slot = p.kept[cj];
      const int t = slot - p.pad[b];
      const int src_blk = p.table_old[static_cast<size_t>(b) * p.max_blocks + t / p.bs];
      const int dst_blk = p.table_new[static_cast<size_t>(b) * p.max_blocks + j / p.bs];
      s_src[r] = static_cast<long long>(
                     ((static_cast<size_t>(l) * p.n_blocks + src_blk) * p.H + h) * p.bs + t % p.bs)
                 << vpr_log2;
      s_dst[r] = static_cast<long long>(
                     ((static_cast<size_t>(l) * p.n_blocks + dst_blk) * p.H + h) * p.bs + j % p.bs)
                 << vpr_log2;
      p.credit_out[cj] = p.credit_post[static_cast<size_t>(u) * p.T + slot];
    } else {
      s_src[r] = -1;
      p.credit_out[cj] = 0.f;  // slots past n_kept are zero, as in the dense compaction
    }
  }
  __syncthreads();
  const uint4* kin = reinterpret_cast<const uint4*>(p.k_pool);
  const uint4* vin = reinterpret_cast<const uint4*>(p.v_pool);
  uint4* kout = reinterpret_cast<uint4*>(p.k_pool);
  uint4* vout = reinterpret_cast<uint4*>(p.v_pool);
  const int vmask = (1 << vpr_log2) - 1;
  const int total = rows << vpr_log2;
  for (int x0 = threadIdx.x; x0 < total; x0 += kCopyThreads * kCopyUnroll) {
    uint4 kv[kCopyUnroll], vv[kCopyUnroll];
#pragma unroll
    for (int i = 0; i < kCopyUnroll; ++i) {
      const int x = x0 + i * kCopyThreads;
      const long long src = x < total ? s_src[x >> vpr_log2] : -1;
      if (src >= 0) {
        kv[i] = kin[src + (x & vmask)];
        vv[i] = vin[src + (x & vmask)];
      }
    }
#pragma unroll
    for (int i = 0; i < kCopyUnroll; ++i) {
      const int x = x0 + i * kCopyThreads;
      if (x < total && s_src[x >> vpr_log2] >= 0) {
        const long long dst = s_dst[x >> vpr_log2] + (x & vmask);
        kout[dst] = kv[i];
        vout[dst] = vv[i];
      }
    }
  }
}

__global__ void __launch_bounds__(kScanThreads) paged_free_kernel(PagedParams p) {
  __shared__ int s_total, s_err;
  if (threadIdx.x == 0) s_err = *p.err != 0;
  __syncthreads();
  if (s_err) {
    if (threadIdx.x == 0) atomicOr(p.status, *p.err);
    return;
  }
  int base = *p.free_top;
  for (int b0 = 0; b0 < p.B; b0 += kScanThreads) {
    const int b = b0 + threadIdx.x;
    const int need = b < p.B ? (p.seq_len[b] + p.bs - 1) / p.bs : 0;
    const int off = block_exclusive_scan(need, &s_total);
    for (int i = 0; i < need; ++i) {
      if (base + off + i < p.n_blocks)  // a consistent pool never overflows the stack
        p.free_list[base + off + i] = p.table_old[static_cast<size_t>(b) * p.max_blocks + i];
      else
        atomicOr(p.status, KVC_STATUS_BAD_INDEX);
    }
    __syncthreads();
    base += s_total;
    __syncthreads();
  }
  if (threadIdx.x == 0) *p.free_top = min(base, p.n_blocks);
}

}  // namespace

cudaError_t launch_compact_paged(const kvc_handle* h, const PagedArgs& a, cudaStream_t s) {
  PagedParams p;
  p.L = h->dims.L;
  p.B = h->dims.B;
  p.H = h->dims.H;
  p.d = h->dims.d;
  p.bs = a.block_size;
  p.n_blocks = a.n_blocks;
  p.max_blocks = a.max_blocks;
  p.budget = h->cfg.budget;
  p.T = a.T;
  p.k_pool = a.k_pool;
  p.v_pool = a.v_pool;
  p.seq_len = a.seq_len;
  p.pad = a.pad;
  p.kept = a.kept_idx;
  p.n_kept = a.n_kept;
  p.credit_post = a.credit_post;
  p.credit_out = a.credit_out;
  p.table_old = a.table_old;
  p.table_new = a.table_new;
  p.free_list = a.free_list;
  p.free_top = a.free_top;
  p.err = h->ws.status + 1;
  p.status = h->ws.status;
  const int U = h->dims.U;
  cudaError_t e = cudaMemsetAsync(p.err, 0, sizeof(uint32_t), s);
  if (e != cudaSuccess) return e;
  paged_validate_kernel<<<U, 128, 0, s>>>(p);
  paged_alloc_kernel<<<1, kScanThreads, 0, s>>>(p);
  for (int u0 = 0; u0 < U; u0 += 65535) {  // gridDim.y is at most 65535
    p.unit0 = u0;
    dim3 grid((p.budget + kCopyRows - 1) / kCopyRows, min(65535, U - u0));
    paged_copy_kernel<<<grid, kCopyThreads, 0, s>>>(p, p.d == 64 ? 3 : 4);  // d / 8 vectors per row
  }
  paged_free_kernel<<<1, kScanThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace kvc
