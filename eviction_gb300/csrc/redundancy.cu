// redundancy.cu -- SkipKV key-redundancy score mixed into the selection score.
//
// "SkipKV: ...", A2 token redundancy score (after R-KV) and the final eviction
// score: per KV head, r_i = the mean cosine similarity of key i to the other
// valid keys, R = softmax of r over the valid slots, I = score / (sum of the
// score over the valid slots), and selection runs on f = sigma*I - (1-sigma)*R
// (more redundant -> evicted earlier).  Padding slots never count and get
// f = -inf.
//
// The mean cosine needs no n x n similarity matrix.  With k^_j = k_j / |k_j|
// (the zero vector for a zero key) and S = sum over the valid j of k^_j,
//     sum over j != i of cos(k_i, k_j) = k^_i . S - [k_i != 0]
// exactly, so a unit costs O(n d) and the kernel is bound by reading K once.
//
// Work layout.  One thread-block cluster of C CTAs (C = 1, 2, 4 or 8) per unit;
// CTA c owns a contiguous slice of the unit's valid rows.  The slice arrives in
// shared memory by 1-D bulk async copies in 16 KB chunks.  When the slice fits
// (up to 96 KB; two CTAs per SM), every chunk has its own buffer and stays
// resident, so K crosses HBM exactly once; a longer slice is streamed twice
// through a ring of chunk buffers.  The CTAs combine their partial S, and later
// their partial sums of e^r and of the score, by reading each other's shared
// memory (DSMEM) in rank order, so every CTA holds bit-identical totals and
// repeated calls give the same bits.  Every mbarrier wait is bounded; all CTAs
// of a cluster pass the same cluster barriers whatever happens.
#include <cmath>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChunkBytes = 16384;
constexpr int kMaxCluster = 8;
constexpr int kResidentChunks = 6;  // 96 KB: the slice stays in shared memory
constexpr int kStreamStages = 6;    // ring depth when it does not

struct RedArgs {
  const uint16_t* k;
  const float* score;
  const int32_t* pad;
  float* sel;    // may alias score
  float* red;    // optional R output
  int T, B, H, C;
  int slice_cap;  // rows of the longest slice any unit can have
  int n_stages;
  int resident;
  float sigma;
  uint32_t* status;
};

// Shared-memory carve-up, identical on host and device.
struct RedLayout {
  size_t stages, sacc, spart, stot, ebuf, sbuf, xs, bars, abort_flag, bytes;
  __host__ __device__ RedLayout(int D, int n_stages, int slice_cap) {
    size_t o = 0;
    stages = o;
    o += static_cast<size_t>(n_stages) * kChunkBytes;
    sacc = o;                                        // [kWarps][D] per-warp partial S
    o += static_cast<size_t>(kWarps) * D * 4;
    spart = o;                                       // [D] this CTA's partial S
    o += static_cast<size_t>(D) * 4;
    stot = o;                                        // [D] S of the unit
    o += static_cast<size_t>(D) * 4;
    ebuf = o;                                        // [slice_cap] e^{r}
    o += (static_cast<size_t>(slice_cap) * 4 + 15) & ~size_t(15);
    sbuf = o;                                        // [slice_cap] score
    o += (static_cast<size_t>(slice_cap) * 4 + 15) & ~size_t(15);
    xs = o;                                          // [2] partial sums; [2*kWarps] warp sums
    o += (2 + 2 * kWarps) * 4;
    o = (o + 7) & ~size_t(7);
    bars = o;
    o += static_cast<size_t>(n_stages) * 8;
    abort_flag = o;
    o += 16;
    bytes = o;
  }
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of every CTA of the cluster arrives, then waits (release /
// acquire: shared-memory writes before the barrier are visible to the peers'
// DSMEM reads after it).
__device__ __forceinline__ void cluster_sync_all() {
  __syncwarp();  // the .aligned forms need a converged warp
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// fp32 at the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ float ld_peer(const float* p, uint32_t rank) {
  uint32_t addr;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(addr) : "r"(smem_u32(p)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// 1-D bulk copy global -> shared (both 16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
      "[%3];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void unpack8(const uint4 raw, float (&x)[8]) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads) redundancy_kernel(const RedArgs a) {
  constexpr int kLpr = D / 8;                  // lanes per key row (8 bf16 each)
  constexpr int kRpw = 32 / kLpr;              // rows per warp and step
  constexpr int kRowsStep = kWarps * kRpw;     // rows per CTA step
  constexpr int kChunkRows = kChunkBytes / (D * 2);

  extern __shared__ __align__(128) unsigned char smem[];
  const RedLayout lay(D, a.n_stages, a.slice_cap);
  unsigned char* stage_base = smem + lay.stages;
  float* sacc = reinterpret_cast<float*>(smem + lay.sacc);
  float* spart = reinterpret_cast<float*>(smem + lay.spart);
  float* stot = reinterpret_cast<float*>(smem + lay.stot);
  float* ebuf = reinterpret_cast<float*>(smem + lay.ebuf);
  float* sbuf = reinterpret_cast<float*>(smem + lay.sbuf);
  float* xs = reinterpret_cast<float*>(smem + lay.xs);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.bars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + lay.abort_flag);

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int grp = warp * kRpw + lane / kLpr;   // row group within a step
  const int sub = lane % kLpr;                 // dims [8 sub, 8 sub + 8)
  const int C = a.C, T = a.T;
  const int u = blockIdx.x / C;
  const uint32_t rank = cluster_rank();
  const int b = (u / a.H) % a.B;
  const int pad = min(max(a.pad[b], 0), T);
  const int n = T - pad;
  const int slice = (n + C - 1) / C;
  const int r0 = min(n, static_cast<int>(rank) * slice);
  const int my = min(n, r0 + slice) - r0;
  const int nch = (my + kChunkRows - 1) / kChunkRows;
  const int NS = a.n_stages;
  const int total_seq = a.resident ? nch : 2 * nch;
  const uint16_t* krow0 = a.k + (static_cast<size_t>(u) * T + pad + r0) * D;

  auto chunk_rows = [&](int c) { return min(kChunkRows, my - c * kChunkRows); };
  auto stage_ptr = [&](int s) {
    return reinterpret_cast<const uint16_t*>(stage_base + static_cast<size_t>(s) * kChunkBytes);
  };
  // Issue the copy of sequence item g (chunk g, or chunk g - nch on the second
  // streamed pass) into its ring slot; thread 0 only, in order g = 0, 1, ...
  int n_issued = 0;
  auto issue = [&](int g) {
    n_issued = g + 1;
    const int c = g < nch ? g : g - nch;
    const int s = g % NS;
    const uint32_t bytes = static_cast<uint32_t>(chunk_rows(c)) * D * 2;
    mbar_arrive_expect_tx(&bars[s], bytes);
    bulk_copy(stage_base + static_cast<size_t>(s) * kChunkBytes,
              krow0 + static_cast<size_t>(c) * kChunkRows * D, bytes, &bars[s]);
  };

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&bars[s], 1);
    // A wait that already timed out in this launch (or an unread earlier
    // failure) stops the CTA before it issues any copy: the result is invalid
    // anyway, and the error stays in the status word.
    *abort_flag = (*reinterpret_cast<volatile uint32_t*>(a.status) & KVC_STATUS_WAIT_TIMEOUT) ? 1 : 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (tid == 0 && !*abort_flag)
    for (int g = 0; g < min(NS, total_seq); ++g) issue(g);

  // ---- pass A: S = sum of the unit-normalised keys ---------------------------
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  for (int c = 0; c < nch; ++c) {
    const int g = c, s = g % NS;
    mbar_wait(&bars[s], (g / NS) & 1, abort_flag, a.status);
    const uint16_t* buf = stage_ptr(s);
    const int rows = chunk_rows(c);
    for (int base = 0; base < rows; base += kRowsStep) {
      const int r = base + grp;
      const uint4 raw = r < rows ? *reinterpret_cast<const uint4*>(buf + r * D + sub * 8)
                                 : make_uint4(0u, 0u, 0u, 0u);
      float x[8];
      unpack8(raw, x);
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
      for (int o = kLpr / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float inv = ss > 0.f ? 1.0f / sqrtf(ss) : 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = fmaf(x[e], inv, acc[e]);
    }
    if (!a.resident) {
      __syncthreads();  // every thread is done with slot s
      if (tid == 0 && g + NS < total_seq && !*abort_flag) issue(g + NS);
    }
  }
  // Combine the row groups of a warp (lanes with the same dims), then warps.
#pragma unroll
  for (int o = kLpr; o < 32; o <<= 1)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
  if (lane < kLpr) {
#pragma unroll
    for (int e = 0; e < 8; ++e) sacc[warp * D + sub * 8 + e] = acc[e];
  }
  __syncthreads();
  for (int t = tid; t < D; t += kThreads) {
    float v = 0.f;
    for (int w = 0; w < kWarps; ++w) v += sacc[w * D + t];
    spart[t] = v;
  }
  cluster_sync_all();
  for (int t = tid; t < D; t += kThreads) {
    float v = 0.f;
    for (int c = 0; c < C; ++c) v += ld_peer(spart + t, static_cast<uint32_t>(c));
    stot[t] = v;
  }
  __syncthreads();

  // ---- pass B: e^{r_i}, r_i = (k^_i . S - 1) / (n - 1) ---------------------------
  float sv[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) sv[e] = stot[sub * 8 + e];
  const float inv_nm1 = n >= 2 ? 1.0f / static_cast<float>(n - 1) : 0.f;
  for (int c = 0; c < nch; ++c) {
    const int g = a.resident ? c : nch + c, s = g % NS;
    if (!a.resident) mbar_wait(&bars[s], (g / NS) & 1, abort_flag, a.status);
    const uint16_t* buf = stage_ptr(s);
    const int rows = chunk_rows(c);
    for (int base = 0; base < rows; base += kRowsStep) {
      const int r = base + grp;
      const uint4 raw = r < rows ? *reinterpret_cast<const uint4*>(buf + r * D + sub * 8)
                                 : make_uint4(0u, 0u, 0u, 0u);
      float x[8];
      unpack8(raw, x);
      float ss = 0.f, dot = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        ss = fmaf(x[e], x[e], ss);
        dot = fmaf(x[e], sv[e], dot);
      }
#pragma unroll
      for (int o = kLpr / 2; o > 0; o >>= 1) {
        ss += __shfl_xor_sync(0xffffffffu, ss, o);
        dot += __shfl_xor_sync(0xffffffffu, dot, o);
      }
      if (r < rows && sub == 0) {
        const float rr = ss > 0.f ? (dot / sqrtf(ss) - 1.0f) * inv_nm1 : 0.f;
        ebuf[c * kChunkRows + r] = expf(rr);
      }
    }
    if (!a.resident) {
      __syncthreads();
      if (tid == 0 && g + NS < total_seq && !*abort_flag) issue(g + NS);
    }
  }
  __syncthreads();

  // ---- sums of e^r and of the score over the unit, then f ------------------------
  const float* srow = a.score + static_cast<size_t>(u) * T + pad + r0;
  float pe = 0.f, ps = 0.f;
  for (int i = tid; i < my; i += kThreads) {
    const float sc = srow[i];
    sbuf[i] = sc;
    ps += sc;
    pe += ebuf[i];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    pe += __shfl_xor_sync(0xffffffffu, pe, o);
    ps += __shfl_xor_sync(0xffffffffu, ps, o);
  }
  float* wsum = xs + 2;
  if (lane == 0) {
    wsum[2 * warp] = pe;
    wsum[2 * warp + 1] = ps;
  }
  __syncthreads();
  if (tid == 0) {
    float e = 0.f, sc = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      e += wsum[2 * w];
      sc += wsum[2 * w + 1];
    }
    xs[0] = e;
    xs[1] = sc;
  }
  cluster_sync_all();
  float z = 0.f, s_tot = 0.f;
  for (int c = 0; c < C; ++c) {
    z += ld_peer(xs, static_cast<uint32_t>(c));
    s_tot += ld_peer(xs + 1, static_cast<uint32_t>(c));
  }
  const float inv_z = z > 0.f ? 1.0f / z : 0.f;
  const float inv_s = s_tot > 0.f ? 1.0f / s_tot : 0.f;
  const float w_i = a.sigma * inv_s;
  const float w_r = (1.0f - a.sigma) * inv_z;
  float* sel = a.sel + static_cast<size_t>(u) * T;
  float* red = a.red ? a.red + static_cast<size_t>(u) * T : nullptr;
  for (int i = tid; i < my; i += kThreads) {
    const float e = ebuf[i];
    sel[pad + r0 + i] = fmaf(w_i, sbuf[i], -(w_r * e));
    if (red) red[pad + r0 + i] = e * inv_z;
  }
  if (rank == 0) {
    for (int i = tid; i < pad; i += kThreads) {
      sel[i] = -INFINITY;
      if (red) red[i] = 0.f;
    }
  }

  // A wait that gave up may leave copies in flight: let them land (bounded)
  // before the shared memory is released.  Only the last copy issued into a
  // slot can be outstanding: a slot is refilled only after all threads saw
  // its previous copy complete, and nothing is issued after an abort.
  if (tid == 0 && *abort_flag) {
    const uint64_t t0 = global_timer_ns();
    for (int s = 0; s < NS && s < n_issued; ++s) {
      const int last = s + NS * ((n_issued - 1 - s) / NS);
      while (!mbar_test_sleep(&bars[s], (last / NS) & 1, kWaitSleepNs) &&
             global_timer_ns() - t0 < kWaitLimitNs) {
      }
    }
  }
  cluster_sync_all();  // no peer reads this CTA's shared memory any more
}

int cdiv(int a, int b) { return (a + b - 1) / b; }

}  // namespace

cudaError_t launch_redundancy(const kvc_handle* h, const uint16_t* k, const float* score, int T,
                              const int32_t* pad, float* sel, float* red, cudaStream_t s) {
  const int D = h->dims.d;
  const int chunk_rows = kChunkBytes / (D * 2);
  int C = 1;
  while (C < kMaxCluster && cdiv(cdiv(T, C), chunk_rows) > kResidentChunks) C *= 2;
  const int slice_cap = cdiv(T, C);
  const int nch = cdiv(slice_cap, chunk_rows);
  const bool resident = nch <= kResidentChunks;
  RedArgs a{k, score, pad, sel, red, T, h->dims.B, h->dims.H, C, slice_cap,
            resident ? (nch > 0 ? nch : 1) : kStreamStages, resident ? 1 : 0,
            h->cfg.redundancy_sigma, h->ws.status};
  const RedLayout lay(D, a.n_stages, slice_cap);
  const int smem = static_cast<int>(lay.bytes);
  void (*kern)(const RedArgs) = D == 64 ? redundancy_kernel<64> : redundancy_kernel<128>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(C) * static_cast<unsigned>(h->dims.U), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, a);
  return e;
}

size_t redundancy_smem_bytes(int D, int T) {
  const int chunk_rows = kChunkBytes / (D * 2);
  int C = 1;
  while (C < kMaxCluster && cdiv(cdiv(T, C), chunk_rows) > kResidentChunks) C *= 2;
  const int slice_cap = cdiv(T, C);
  const int nch = cdiv(slice_cap, chunk_rows);
  const int ns = nch <= kResidentChunks ? (nch > 0 ? nch : 1) : kStreamStages;
  return RedLayout(D, ns, slice_cap).bytes;
}

}  // namespace kvc
