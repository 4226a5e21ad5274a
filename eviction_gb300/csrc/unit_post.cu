// unit_post.cu -- the fused per-unit kernel of the event: mass, segmentation
// with quotas, and selection in one CTA per unit, for units of up to 4096 slots.
//
// "Adaptive Mass-Segmented KV Compression for Long-Form Reasoning", Method,
// Key designs 1-4, and its overhead statement: after the attention usage, mass
// processing and the prefix sum are O(H_kv * T) work per layer.  That work is a
// chain of short dependent steps per unit (block reductions, a scan, a serial
// segment build, searches), so the three steps share one launch, and the
// unit's mass, score and segments stay in shared memory between them instead
// of making a round trip through global memory between three launches.  With
// 15 CTAs per SM the schedulers are busy most of the time: the kernel's time
// follows its instruction count.
//
// The steps are the functions of unit_phases.cuh that the stand-alone kernels
// run, with the CTA shape of the stand-alone mass kernel (unit::mass_shape; the
// mass step is the only one whose floating-point summation order depends on
// it), so every output is bit-identical to the three-launch sequence.  Score,
// mass, credit, segments, quotas, kept indices and counts are all still written
// to global memory.
//
// Shared memory (dynamic, 16-byte aligned offsets), reused from step to step so
// that many units fit on an SM at once:
//   score [T] f32                mass -> selection
//   A                            mass: filled usage [kEpt*NT] f32, then the
//                                mass [T] f32 (written after its last read);
//                                selection: flags [T] u8, then the radix
//                                histograms [NT/32][256] i32 of the picks, reused
//                                by the pick keys [budget] u32 of the excess
//                                search (units past 8*NT slots)
//   b [K] i32                    segmentation (cut points)
//   segments [S_cap] x 32 B      segmentation: mass u64 | rem i64 | start | len | q | floor;
//                                selection: start [S_cap] | want [S_cap] over mass
#include "unit_phases.cuh"

namespace kvc {
int attention_row_stride(int R);
int segment_threshold_count(double delta);
void segment_delta_parts(float delta, uint64_t* m, int* e);
int segment_capacity(const kvc_config& c, int T);

namespace {

constexpr int kMaxFusedT = unit::kSmemT;

__host__ __device__ inline int round16(int x) { return (x + 15) & ~15; }

struct FusedLayout {
  int off_a, off_b, off_seg, total;
  int off_key, off_hist;  // within A, selection step
};

__host__ inline FusedLayout fused_layout(int T, int NT, int kEpt, int K, int S_cap, int budget) {
  FusedLayout l;
  l.off_a = round16(4 * T);
  // the pick keys of the excess search and the radix histograms of the picks
  // are never live together (a barrier separates them): one region
  l.off_key = round16(T);
  l.off_hist = l.off_key;
  const int keys = T > unit::kRegPer * NT ? 4 * budget : 0;
  const int hist = 1024 * (NT / 32);
  int a = 4 * kEpt * NT;                              // filled usage (>= the mass)
  const int sel = l.off_key + (keys > hist ? keys : hist);  // flags + (keys | histograms)
  a = a > sel ? a : sel;
  l.off_b = l.off_a + round16(a);
  l.off_seg = l.off_b + round16(4 * K);
  l.total = l.off_seg + 32 * S_cap;
  return l;
}

struct FusedParams {
  unit::PostParams post;
  unit::SegParams seg;
  unit::SelParams sel;
  FusedLayout ly;
};

// NT threads, kEpt = slots per thread of the mass step (unit::mass_shape).
// Latency-bound, one CTA per unit, held to 32 registers (some spilled) so that
// 16 CTAs of 128 threads (or 8 of 256) share an SM: with 40 registers and 6
// CTAs of 256 threads the 28-layer batch-32 event took 0.131 ms, 0.118 now.
template <int NT, int kEpt>
__global__ void __launch_bounds__(NT, NT == 128 ? 16 : (kEpt <= 8 ? 8 : 4))
    unit_post_kernel(FusedParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ float red[3 * (NT / 32 + 1)];
  __shared__ uint64_t part[NT / 32];
  __shared__ uint64_t pre[NT];
  __shared__ uint64_t total;
  __shared__ int nseg;
  __shared__ int sred[NT / 32];
  __shared__ int sred2[2 * NT / 32];
  __shared__ int sscan[NT / 32];
  float* score_sm = reinterpret_cast<float*>(smem);
  uint8_t* A = smem + p.ly.off_a;
  float* mass_sm = reinterpret_cast<float*>(A);
  uint8_t* segb = smem + p.ly.off_seg;
  const int u = blockIdx.x;

  // Key design 1: mass, credit, score (also kept in shared memory)
  unit::mass_phase<kEpt, NT>(p.post, u, reinterpret_cast<float*>(A), red, mass_sm, score_sm);
  __syncthreads();  // mass_sm / score_sm complete

  // Key designs 2-3: segments and quotas from the mass in shared memory
  const int T = p.post.T;
  const int b = (u / p.post.H) % p.post.B;
  const int pad = min(max(p.post.pad[b], 0), T);
  const int n = T - pad;
  const int S_cap = p.seg.S_cap;
  unit::SegSmem ss;
  ss.mass = reinterpret_cast<uint64_t*>(segb);
  ss.rem = reinterpret_cast<int64_t*>(ss.mass + S_cap);
  ss.start = reinterpret_cast<int32_t*>(ss.rem + S_cap);
  ss.len = ss.start + S_cap;
  ss.q = ss.len + S_cap;
  ss.floor = ss.q + S_cap;
  ss.b = reinterpret_cast<int32_t*>(smem + p.ly.off_b);
  ss.part = part;
  ss.pre = pre;
  ss.sub = nullptr;
  ss.total = &total;
  ss.nseg = &nseg;
  unit::segment_phase<NT>(p.seg, u, mass_sm + pad, pad, n, ss, true);
  __syncthreads();  // segments final (warp 0 wrote them); the mass is dead

  // Key designs 3-4: selection on the score in shared memory
  const int ns = (n > 0) ? min(nseg, p.sel.S_max) : 0;
  unit::SelSmem sl;
  sl.start = reinterpret_cast<int32_t*>(segb);  // over the segment masses (dead)
  sl.want = sl.start + S_cap;
  sl.flag = A;
  sl.key = reinterpret_cast<uint32_t*>(A + p.ly.off_key);
  sl.hist = reinterpret_cast<int*>(A + p.ly.off_hist);
  sl.xhist = nullptr;  // (1024-thread CTAs only)
  sl.red = sred;
  sl.red2 = sred2;
  sl.scan = sscan;
  const unit::SegsShared segs{ss.start, ss.len, ss.q};
  unit::select_phase<NT, false>(p.sel, u, score_sm + pad, pad, n, ns, segs, sl);
}

}  // namespace

// Shared memory of the fused kernel for units of T slots; 0 when T is too long
// for it (the three stand-alone kernels run instead).
size_t unit_post_smem_bytes(const kvc_config& c, int T) {
  if (T > kMaxFusedT) return 0;
  int nt, ept;
  unit::mass_shape(T, &nt, &ept);
  const int K = segment_threshold_count(static_cast<double>(c.delta));
  return static_cast<size_t>(
      fused_layout(T, nt, ept, K, segment_capacity(c, T), c.budget).total);
}

cudaError_t launch_unit_post(const kvc_handle* h, int T, const int32_t* pad,
                             const int32_t* n_carry, const float* credit_in,
                             float* credit_post, float* mass, float* score, int32_t* seg_start,
                             int32_t* seg_len, int32_t* quota, int32_t* n_seg,
                             int32_t* kept_idx, int32_t* n_kept, cudaStream_t s) {
  const Dims& dm = h->dims;
  const kvc_config& c = h->cfg;
  if (T > kMaxFusedT) return cudaErrorInvalidValue;
  FusedParams p;
  unit::PostParams& q = p.post;
  q.T = T;
  q.R = dm.R;
  q.W = dm.W;
  q.G = dm.G;
  q.B = dm.B;
  q.H = dm.H;
  q.avg_pool = c.avg_pool;
  q.max_pool = c.max_pool;
  q.eps = c.eps;
  q.lambda = c.lambda;
  q.beta = c.beta;
  q.Rp = attention_row_stride(dm.R);
  q.pmax = h->ws.pmax;
  q.usage = h->ws.usage;
  q.pad = pad;
  q.n_carry = n_carry;
  q.credit_in = credit_in;
  q.credit_post = credit_post;
  q.mass = mass;
  q.score = score;
  unit::SegParams& g = p.seg;
  g.T = T;
  g.B = dm.B;
  g.H = dm.H;
  g.S_max = s_max_of(c, T);
  g.S_cap = segment_capacity(c, T);
  g.budget = c.budget;
  g.q_min = c.q_min;
  g.seg_min = c.seg_min;
  g.seg_max = c.seg_max;
  g.seg_fixed = c.seg_fixed;
  g.quota_by_len = c.quota_by_len;
  g.global_topk = c.global_topk;
  segment_delta_parts(c.delta, &g.delta_m, &g.delta_e);
  g.K = segment_threshold_count(static_cast<double>(c.delta));
  g.mass = mass;
  g.pad = pad;
  g.seg_start = seg_start;
  g.seg_len = seg_len;
  g.quota = quota;
  g.n_seg = n_seg;
  unit::SelParams& e = p.sel;
  e.T = T;
  e.B = dm.B;
  e.H = dm.H;
  e.S_max = g.S_max;
  e.budget = c.budget;
  e.n_sink = c.n_sink;
  e.n_recent = c.n_recent;
  e.score = score;
  e.pad = pad;
  e.seg_start = seg_start;
  e.seg_len = seg_len;
  e.quota = quota;
  e.n_seg = n_seg;
  e.kept_idx = kept_idx;
  e.n_kept = n_kept;
  int nt, ept;
  unit::mass_shape(T, &nt, &ept);
  p.ly = fused_layout(T, nt, ept, g.K, g.S_cap, c.budget);
  auto kern = nt == 256    ? unit_post_kernel<256, 16>
              : ept == 4  ? unit_post_kernel<128, 4>
              : ept == 6  ? unit_post_kernel<128, 6>
              : ept == 8  ? unit_post_kernel<128, 8>
              : ept == 12 ? unit_post_kernel<128, 12>
                          : unit_post_kernel<128, 16>;
  const size_t smem = static_cast<size_t>(p.ly.total);
  if (smem > 48 * 1024) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
  }
  kern<<<dm.U, nt, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace kvc
