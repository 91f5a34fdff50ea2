// C ABI of the gated delta rule prefill library (declared in include/gdn.h):
// host-side validation, workspace layout, the prep kernel (device checks of
// cu_seqlens / state_index and the longest-first sequence order) and dispatch
// to the chunk kernels.
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "gdn_internal.cuh"
#include "gdn_ops.cuh"

namespace gdn {

constexpr int kPrepThreads = 1024;
constexpr int kBins = 4096;  // sequences are ordered by chunk count, capped here

// One block. Resets the status word, checks what only the device can see, and
// writes the sequence order (most chunks first) by a counting sort on the
// chunk count. The order only steers scheduling; results do not depend on it.
//
// A tree launch (p.parent set) also checks parent[n] in [-1, n), clears the
// ready flags and the work counter, and orders the roots (parent -1) longest
// first followed by every other sequence in index order: a parent then always
// precedes its children, as the tree kernel's in-order unit counter needs.
__global__ void __launch_bounds__(kPrepThreads) gdn_prep_kernel(Params p, int32_t* order) {
  __shared__ int hist[kBins];
  __shared__ int warp_tot[kPrepThreads / 32];
  __shared__ int n_roots;
  const int tid = threadIdx.x;
  const bool tree = p.parent != nullptr;
  // The chunk kernel, launched as a programmatic dependent of this one, may start its
  // set-up now; it waits for this grid to complete before it reads anything written here.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    if (!p.keep_status) {
      p.status->code = 0u;
      p.status->detail = 0u;
    }
    p.status->units_done = 0u;
    p.status->next_unit = 0u;
    n_roots = 0;
  }
  if (tree)
    for (int64_t u = tid; u < (int64_t)p.num_seqs * p.h_v; u += kPrepThreads) p.ready[u] = 0u;
  for (int b = tid; b < kBins; b += kPrepThreads) hist[b] = 0;
  __syncthreads();

  const int N = p.num_seqs;
  for (int n = tid; n < N; n += kPrepThreads) {
    if (!p.seq_rows) {  // (a segment launch's rows were checked by its set-up kernel)
      const int64_t b = p.cu_seqlens[n], e = p.cu_seqlens[n + 1];
      if ((n == 0 && b != 0) || e < b || (n == N - 1 && e != p.total_tokens) ||
          (p.max_seqlen > 0 && e - b > p.max_seqlen))
        report(p.status, GDN_ERR_SEQLENS, (uint32_t)n);
    }
    if (p.initial_state && p.state_index) {
      const int32_t s = p.state_index[n];
      if (s < -1 || s >= p.num_state_slots) report(p.status, GDN_ERR_STATE_INDEX, (uint32_t)n);
    }
    if (tree) {
      const int32_t pa = p.parent[n];
      if (pa < -1 || pa >= n) report(p.status, GDN_ERR_PARENT, (uint32_t)n);
      if (tree_parent(p, n) >= 0) continue;  // ordered after the roots, below
      atomicAdd(&n_roots, 1);
    }
    int64_t bos, eos;
    seq_bounds(p, n, bos, eos);
    int64_t nc = (eos - bos + kChunk - 1) / kChunk;
    const int bin = (int)(nc < kBins - 1 ? nc : kBins - 1);
    atomicAdd(&hist[bin], 1);
  }
  __syncthreads();

  // Exclusive prefix sum over bins taken from the top: start[b] = #seqs in bins > b.
  constexpr int per = kBins / kPrepThreads;
  int local[per];
  int sum = 0;
#pragma unroll
  for (int j = 0; j < per; ++j) {
    local[j] = hist[kBins - 1 - (tid * per + j)];
    sum += local[j];
  }
  const int lane = tid & 31, warp = tid >> 5;
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_tot[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    warp_tot[lane] = wi - w;  // exclusive
  }
  __syncthreads();
  int run = warp_tot[warp] + incl - sum;
#pragma unroll
  for (int j = 0; j < per; ++j) {
    hist[kBins - 1 - (tid * per + j)] = run;
    run += local[j];
  }
  __syncthreads();
  for (int n = tid; n < N; n += kPrepThreads) {
    if (tree && tree_parent(p, n) >= 0) continue;
    int64_t bos, eos;
    seq_bounds(p, n, bos, eos);
    int64_t nc = (eos - bos + kChunk - 1) / kChunk;
    const int bin = (int)(nc < kBins - 1 ? nc : kBins - 1);
    const int pos = atomicAdd(&hist[bin], 1);
    if (GDN_IN_BOUNDS(p.status, pos >= 0 && pos < N, 0x201u)) order[pos] = n;
  }
  if (!tree) return;
  // the other sequences after the roots, in index order (a block-wide scan per pass)
  int base = n_roots;
  for (int n0 = 0; n0 < N; n0 += kPrepThreads) {
    const int n = n0 + tid;
    const int f = (n < N && tree_parent(p, n) >= 0) ? 1 : 0;
    int incl = f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    __syncthreads();  // warp_tot is free again
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < kPrepThreads / 32; ++w) {
      if (w < warp) before += warp_tot[w];
      total += warp_tot[w];
    }
    if (f && GDN_IN_BOUNDS(p.status, base + before + incl - 1 < N, 0x202u)) order[base + before + incl - 1] = n;
    base += total;
  }
}

// The prep kernel for a batch of at most 32 sequences outside a tree launch: one warp,
// lane n checks sequence n and places it by rank (more chunks first, then lower index).
// The same checks and the same kind of order as gdn_prep_kernel, without its 4096-bin
// histogram and block-wide scans, which set a small batch's latency.
__global__ void __launch_bounds__(32) gdn_prep_small_kernel(Params p, int32_t* order) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int n = threadIdx.x, N = p.num_seqs;
  if (n == 0) {
    if (!p.keep_status) {
      p.status->code = 0u;
      p.status->detail = 0u;
    }
    p.status->units_done = 0u;
    p.status->next_unit = 0u;
  }
  __syncwarp();
  int64_t nc = -1;  // lanes past N rank last and write nothing
  if (n < N) {
    if (!p.seq_rows) {
      const int64_t b = p.cu_seqlens[n], e = p.cu_seqlens[n + 1];
      if ((n == 0 && b != 0) || e < b || (n == N - 1 && e != p.total_tokens) ||
          (p.max_seqlen > 0 && e - b > p.max_seqlen))
        report(p.status, GDN_ERR_SEQLENS, (uint32_t)n);
    }
    if (p.initial_state && p.state_index) {
      const int32_t si = p.state_index[n];
      if (si < -1 || si >= p.num_state_slots) report(p.status, GDN_ERR_STATE_INDEX, (uint32_t)n);
    }
    int64_t bos, eos;
    seq_bounds(p, n, bos, eos);
    nc = (eos - bos + kChunk - 1) / kChunk;
  }
  int rank = 0;
#pragma unroll 1
  for (int m = 0; m < 32; ++m) {
    const int64_t o = __shfl_sync(0xffffffffu, nc, m);
    rank += (o > nc || (o == nc && m < n)) ? 1 : 0;
  }
  if (n < N && GDN_IN_BOUNDS(p.status, rank < N, 0x203u)) order[rank] = n;
}

cudaError_t launch_prep(const Params& p, cudaStream_t stream) {
  if (!p.parent && p.num_seqs <= 32)
    gdn_prep_small_kernel<<<1, 32, 0, stream>>>(p, const_cast<int32_t*>(p.order));
  else
    gdn_prep_kernel<<<1, kPrepThreads, 0, stream>>>(p, const_cast<int32_t*>(p.order));
  return cudaGetLastError();
}

cudaError_t set_smem_once(const void* kernel, int bytes) {
  static std::mutex mu;
  static const void* done_kernel[256];
  static int done_dev[256];
  static int n_done = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_done; ++i)
    if (done_kernel[i] == kernel && done_dev[i] == dev) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  if (n_done < 256) {
    done_kernel[n_done] = kernel;
    done_dev[n_done] = dev;
    ++n_done;
  }
  return cudaSuccess;
}

// Streaming multiprocessors of the current device (cached per device).
cudaError_t device_sm_count(int* out) {
  static std::mutex mu;
  static int cached[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    cached[dev] = n > 0 ? n : 1;
  }
  *out = cached[dev];
  return cudaSuccess;
}

// ---------------------------------------------------------------- host checks

static bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
  if (!a || !b || an == 0 || bn == 0) return false;
  const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
  return a0 < b0 + bn && b0 < a0 + an;
}

static bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

// sm_103 check, cached per device.
static gdn_status check_arch() {
  static std::mutex mu;
  static int cached[64];  // 0 unknown, 1 ok, 2 not sm_103
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
  if (dev < 0 || dev >= 64) return GDN_ERR_ARCH;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return GDN_ERR_CUDA;
    cached[dev] = (major == 10 && minor == 3) ? 1 : 2;
  }
  return cached[dev] == 1 ? GDN_OK : GDN_ERR_ARCH;
}

}  // namespace gdn

using namespace gdn;

extern "C" int gdn_abi_version(void) { return GDN_ABI_VERSION; }

extern "C" size_t gdn_workspace_bytes(const gdn_desc* desc) {
  if (!desc || desc->num_seqs < 0) return 0;
  const size_t base = gdn::workspace_bytes(desc->num_seqs);
  if (!gdn::seg_eligible(desc)) return base;
  const size_t seg = gdn::seg_layout(desc->h_v, desc->d_k, desc->d_v).end;
  return seg > base ? seg : base;
}

extern "C" gdn_status gdn_segment_plan(const gdn_desc* desc, int32_t sms, int32_t* segments, int64_t* rows0,
                                       int64_t* rows) {
  if (!desc || !segments || !rows0 || !rows) return GDN_ERR_NULL;
  if (sms < 1) return GDN_ERR_VALUE;
  *segments = 0;
  *rows0 = desc->total_tokens;
  *rows = 0;
  if (!gdn::seg_eligible(desc) || desc->workspace_bytes < gdn::seg_layout(desc->h_v, desc->d_k, desc->d_v).end)
    return GDN_OK;
  const gdn::SegPlan plan = gdn::seg_plan(desc->total_tokens, desc->h_v, sms);
  if (plan.G >= 3) {
    *segments = plan.G;
    *rows0 = plan.a;
    *rows = plan.b;
  }
  return GDN_OK;
}

extern "C" size_t gdn_tree_workspace_bytes(const gdn_desc* desc) {
  if (!desc || desc->num_seqs < 0 || desc->h_v < 1) return 0;
  return gdn::tree_workspace_bytes(desc->num_seqs, desc->h_v);
}

extern "C" const char* gdn_status_string(gdn_status s) {
  switch (s) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_NULL: return "GDN_ERR_NULL: a required pointer is NULL";
    case GDN_ERR_SHAPE: return "GDN_ERR_SHAPE: unsupported or inconsistent sizes";
    case GDN_ERR_DTYPE: return "GDN_ERR_DTYPE: unsupported storage type";
    case GDN_ERR_ALIGN: return "GDN_ERR_ALIGN: misaligned pointer";
    case GDN_ERR_SEQLENS: return "GDN_ERR_SEQLENS: cu_seqlens inconsistent (device check)";
    case GDN_ERR_STATE_INDEX: return "GDN_ERR_STATE_INDEX: state_index out of range (device check)";
    case GDN_ERR_ALIAS: return "GDN_ERR_ALIAS: an output overlaps an input";
    case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case GDN_ERR_ARCH: return "GDN_ERR_ARCH: the current device is not sm_103";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA: a CUDA runtime call failed";
    case GDN_ERR_DEVICE_TIMEOUT: return "GDN_ERR_DEVICE_TIMEOUT: a bounded device wait gave up";
    case GDN_ERR_PARENT: return "GDN_ERR_PARENT: a parent index outside [-1, n) (device check)";
    case GDN_ERR_VALUE: return "GDN_ERR_VALUE: an argument outside its range";
    case GDN_ERR_BOUNDS: return "GDN_ERR_BOUNDS: an index outside its buffer (bounds-checked build)";
  }
  return "unknown gdn_status";
}

// Host-side validation shared by every entry point that launches. Fills `p`.
static gdn_status validate(const void* q, const void* k, const void* v, const void* g,
                           const void* beta, const int32_t* cu_seqlens,
                           const float* initial_state, const int32_t* state_index, void* out,
                           float* final_state, const gdn_desc* d, Params& p,
                           const int32_t* parent = nullptr) {
  if (!d) return GDN_ERR_NULL;
  const int64_t T = d->total_tokens;
  const int N = d->num_seqs;
  if (N < 0 || T < 0 || d->max_seqlen < 0) return GDN_ERR_SHAPE;
  if (d->h_qk < 1 || d->h_v < 1 || d->h_v % d->h_qk != 0) return GDN_ERR_SHAPE;
  if (!((d->d_k == 64 || d->d_k == 128) && (d->d_v == 64 || d->d_v == 128))) return GDN_ERR_SHAPE;
  if (d->qkv_dtype != GDN_BF16) return GDN_ERR_DTYPE;
  if (d->gate_dtype != GDN_BF16 && d->gate_dtype != GDN_F32) return GDN_ERR_DTYPE;
  if (d->out_dtype != GDN_BF16 && d->out_dtype != GDN_F32) return GDN_ERR_DTYPE;
  if (!cu_seqlens) return GDN_ERR_NULL;
  if (T > 0 && (!q || !k || !v || !g || !beta || !out)) return GDN_ERR_NULL;
  if (initial_state && d->num_state_slots < 1) return GDN_ERR_SHAPE;
  if (initial_state && !state_index && d->num_state_slots < N) return GDN_ERR_SHAPE;
  if (!d->workspace) return GDN_ERR_WORKSPACE;
  if (!aligned(d->workspace, 256) || d->workspace_bytes < gdn::workspace_bytes(N))
    return GDN_ERR_WORKSPACE;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(initial_state, 16) || !aligned(final_state, 16) || !aligned(g, 4) ||
      !aligned(beta, 4) || !aligned(cu_seqlens, 4) || !aligned(state_index, 4) || !aligned(parent, 4))
    return GDN_ERR_ALIGN;

  const size_t gsz = d->gate_dtype == GDN_F32 ? 4 : 2;
  const size_t osz = d->out_dtype == GDN_F32 ? 4 : 2;
  const size_t qb = (size_t)T * d->h_qk * d->d_k * 2, vb = (size_t)T * d->h_v * d->d_v * 2;
  const size_t gb = (size_t)T * d->h_v * gsz, ob = (size_t)T * d->h_v * d->d_v * osz;
  const size_t sb = (size_t)d->h_v * d->d_k * d->d_v * 4;
  const size_t isb = initial_state ? sb * (size_t)d->num_state_slots : 0;
  const size_t fsb = final_state ? sb * (size_t)N : 0;
  const size_t cub = sizeof(int32_t) * (size_t)(N + 1);
  const size_t sib = state_index ? sizeof(int32_t) * (size_t)N : 0;
  const size_t pab = parent ? sizeof(int32_t) * (size_t)N : 0;
  const size_t wsb = d->workspace_bytes;
  struct R { const void* p; size_t n; } ins[] = {{q, qb}, {k, qb}, {v, vb}, {g, gb}, {beta, gb},
                                                 {cu_seqlens, cub}, {initial_state, isb},
                                                 {state_index, sib}, {d->workspace, wsb},
                                                 {parent, pab}};
  for (const R& r : ins) {
    if (overlaps(out, ob, r.p, r.n)) return GDN_ERR_ALIAS;
    if (overlaps(final_state, fsb, r.p, r.n)) return GDN_ERR_ALIAS;
  }
  if (overlaps(out, ob, final_state, fsb)) return GDN_ERR_ALIAS;

  const gdn_status arch = check_arch();
  if (arch != GDN_OK) return arch;

  memset(&p, 0, sizeof(p));
  p.q = (const __nv_bfloat16*)q;
  p.k = (const __nv_bfloat16*)k;
  p.v = (const __nv_bfloat16*)v;
  p.g = g;
  p.beta = beta;
  p.cu_seqlens = cu_seqlens;
  p.initial_state = initial_state;
  p.state_index = state_index;
  p.out = out;
  p.final_state = final_state;
  p.status = (Status*)d->workspace;
  p.order = (const int32_t*)((char*)d->workspace + kOrderOffset);
  p.total_tokens = T;
  p.num_seqs = N;
  p.max_seqlen = d->max_seqlen;
  p.h_qk = d->h_qk;
  p.h_v = d->h_v;
  p.d_k = d->d_k;
  p.d_v = d->d_v;
  p.num_state_slots = initial_state ? d->num_state_slots : 0;
  p.gate_f32 = d->gate_dtype == GDN_F32;
  p.out_f32 = d->out_dtype == GDN_F32;
  p.l2norm = (d->flags & GDN_FLAG_NO_L2NORM) ? 0 : 1;
  p.scale = d->scale != 0.0f ? d->scale : 1.0f / sqrtf((float)d->d_k);
  p.vzero_from = N;
  p.out_upto = N;
  return GDN_OK;
}

namespace gdn {

// The segment scan of one sequence (the plan has G >= 3): set-up, launch A, the
// composition, launch C, and the final state copied out of the workspace. Every step
// is stream-ordered; the status word collects the first error of any of them.
static gdn_status run_segmented(const Params& p0, const SegPlan& plan, char* ws, cudaStream_t s) {
  const SegLayout L = seg_layout(p0.h_v, p0.d_k, p0.d_v);
  const int G = plan.G;
  const size_t sb = (size_t)p0.h_v * p0.d_k * p0.d_v * 4;
  if (launch_seg_setup(p0, plan, L, ws, s) != cudaSuccess) return GDN_ERR_CUDA;
  Params pa = p0;
  pa.num_seqs = 2 * G - 3;
  pa.max_seqlen = 0;
  pa.seq_rows = reinterpret_cast<const int64_t*>(ws + L.rows_a);
  pa.initial_state = reinterpret_cast<const float*>(ws + L.slots);
  pa.num_state_slots = 2;
  pa.state_index = reinterpret_cast<const int32_t*>(ws + L.sidx_a);
  pa.final_state = reinterpret_cast<float*>(ws + L.fin_a);
  pa.vzero_from = G - 1;
  pa.out_upto = 1;
  pa.keep_status = 1;
  if (launch_prep(pa, s) != cudaSuccess || launch_tc(pa, s) != cudaSuccess) return GDN_ERR_CUDA;
  if (launch_seg_combine(p0, plan, L, ws, s) != cudaSuccess) return GDN_ERR_CUDA;
  Params pc = p0;
  pc.num_seqs = G - 1;
  pc.max_seqlen = 0;
  pc.seq_rows = reinterpret_cast<const int64_t*>(ws + L.rows_c);
  pc.initial_state = reinterpret_cast<const float*>(ws + L.s_c);
  pc.num_state_slots = G - 1;
  pc.state_index = nullptr;                              // segment n starts from S_{n+1}
  pc.final_state = reinterpret_cast<float*>(ws + L.fin_a);  // launch A's states are spent
  pc.vzero_from = G - 1;
  pc.out_upto = G - 1;
  pc.keep_status = 1;
  if (launch_prep(pc, s) != cudaSuccess || launch_tc(pc, s) != cudaSuccess) return GDN_ERR_CUDA;
  if (p0.final_state &&
      cudaMemcpyAsync(p0.final_state, ws + L.fin_a + (size_t)(G - 2) * sb, sb, cudaMemcpyDeviceToDevice, s) !=
          cudaSuccess)
    return GDN_ERR_CUDA;
  return GDN_OK;
}

}  // namespace gdn

extern "C" gdn_status gdn_prefill_varlen(const void* q, const void* k, const void* v,
                                         const void* g, const void* beta,
                                         const int32_t* cu_seqlens, const float* initial_state,
                                         const int32_t* state_index, void* out,
                                         float* final_state, const gdn_desc* desc, void* stream) {
  Params p;
  const gdn_status st = validate(q, k, v, g, beta, cu_seqlens, initial_state, state_index, out,
                                 final_state, desc, p);
  if (st != GDN_OK) return st;
  if (p.num_seqs == 0) return GDN_OK;
  cudaStream_t s = (cudaStream_t)stream;
  if (gdn::seg_eligible(desc) &&
      desc->workspace_bytes >= gdn::seg_layout(desc->h_v, desc->d_k, desc->d_v).end) {
    int sms = 0;
    if (gdn::device_sm_count(&sms) != cudaSuccess) return GDN_ERR_CUDA;
    const gdn::SegPlan plan = gdn::seg_plan(p.total_tokens, p.h_v, sms);
    if (plan.G >= 3) return gdn::run_segmented(p, plan, (char*)desc->workspace, s);
  }
  if (!(desc->flags & GDN_FLAG_SIMT) && p.total_tokens > 0 && p.num_seqs <= 32 && p.d_k == p.d_v) {
    // A batch with at most one (sequence, value head) unit per SM needs no work list:
    // CTA b takes unit b and checks its own sequence, and a memset of the status block
    // replaces the prep kernel (one launch less on the latency of a small call).
    int sms = 0;
    if (gdn::device_sm_count(&sms) != cudaSuccess) return GDN_ERR_CUDA;
    if ((long long)p.num_seqs * p.h_v <= sms) {
      if (cudaMemsetAsync(p.status, 0, 4 * sizeof(uint32_t), s) != cudaSuccess) return GDN_ERR_CUDA;
      p.direct = 1;
      return gdn::launch_tc(p, s) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
    }
  }
  if (launch_prep(p, s) != cudaSuccess) return GDN_ERR_CUDA;
  const cudaError_t e = (desc->flags & GDN_FLAG_SIMT) ? launch_simt(p, s) : launch_tc(p, s);
  if (e != cudaSuccess) return GDN_ERR_CUDA;
  return GDN_OK;
}

namespace gdn {

// GDN_FLAG_TEST_CHILD_FIRST: reverses the work list (one block), so that children
// precede their parents (fault injection for the bounded waits).
__global__ void gdn_reverse_order_kernel(int32_t* order, int n) {
  for (int i = threadIdx.x; i < n / 2; i += blockDim.x) {
    const int32_t a = order[i];
    order[i] = order[n - 1 - i];
    order[n - 1 - i] = a;
  }
}

// Tree launch with no tokens at all: every sequence ends where it starts, so
// final_state[n] is its root's starting state (one block per (sequence, head)).
__global__ void gdn_tree_copy_kernel(Params p) {
  const int n = blockIdx.x / p.h_v, h = blockIdx.x % p.h_v;
  int r = n;
  for (int steps = 0; steps <= n; ++steps) {  // parents have smaller indices: the walk ends
    const int pa = tree_parent(p, r);
    if (pa < 0) break;
    r = pa;
  }
  const int64_t slot = state_slot(p, r);
  const size_t sz = (size_t)p.d_k * p.d_v;
  const float* src = slot >= 0 ? p.initial_state + ((size_t)slot * p.h_v + h) * sz : nullptr;
  float* dst = p.final_state + ((size_t)n * p.h_v + h) * sz;
  for (size_t i = threadIdx.x; i < sz; i += blockDim.x) dst[i] = src ? src[i] : 0.f;
}

}  // namespace gdn

extern "C" gdn_status gdn_prefill_tree(const void* q, const void* k, const void* v, const void* g,
                                       const void* beta, const int32_t* cu_seqlens,
                                       const int32_t* parent, const float* initial_state,
                                       const int32_t* state_index, void* out, float* final_state,
                                       const gdn_desc* desc, void* stream) {
  if (!desc) return GDN_ERR_NULL;
  if (!parent || !final_state) return GDN_ERR_NULL;
  if (desc->flags & GDN_FLAG_SIMT) return GDN_ERR_SHAPE;
  if (desc->num_seqs > 0 && desc->h_v >= 1 && desc->workspace &&
      desc->workspace_bytes < gdn::tree_workspace_bytes(desc->num_seqs, desc->h_v))
    return GDN_ERR_WORKSPACE;
  Params p;
  const gdn_status st = validate(q, k, v, g, beta, cu_seqlens, initial_state, state_index, out,
                                 final_state, desc, p, parent);
  if (st != GDN_OK) return st;
  if (p.num_seqs == 0) return GDN_OK;
  p.parent = parent;
  p.ready = (uint32_t*)((char*)desc->workspace + gdn::tree_flags_offset(p.num_seqs));
  cudaStream_t s = (cudaStream_t)stream;
  if (launch_prep(p, s) != cudaSuccess) return GDN_ERR_CUDA;
  if (desc->flags & GDN_FLAG_TEST_CHILD_FIRST) {
    gdn::gdn_reverse_order_kernel<<<1, 256, 0, s>>>(const_cast<int32_t*>(p.order), p.num_seqs);
    if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
  }
  if (p.total_tokens == 0) {
    const long long units = (long long)p.num_seqs * p.h_v;
    if (units > 0x7fffffffLL) return GDN_ERR_SHAPE;
    gdn::gdn_tree_copy_kernel<<<(unsigned)units, 256, 0, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
  }
  return launch_tc(p, s) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

extern "C" gdn_status gdn_get_device_status(const gdn_desc* desc, void* stream) {
  if (!desc || !desc->workspace) return GDN_ERR_NULL;
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t code = 0;
  if (cudaMemcpyAsync(&code, desc->workspace, sizeof(code), cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return GDN_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return GDN_ERR_CUDA;
  return (gdn_status)code;
}

// ------------------------------------------------ variant without a workspace
//
// The workspace of gdn_prefill_varlen_noalloc: a status block and a work list
// for GDN_NOALLOC_MAX_SEQS sequences, compiled in as static device memory (one
// copy per device). The prep kernel of every call resets the status word and
// rewrites the work list, so nothing here needs clearing between calls.
namespace gdn {

constexpr size_t kNoallocBytes = kOrderOffset + sizeof(int32_t) * (size_t)GDN_NOALLOC_MAX_SEQS;
static_assert(kNoallocBytes % 256 == 0, "the work list ends on a 256-byte boundary");

static __device__ __align__(256) unsigned char g_noalloc_workspace[kNoallocBytes];

// The device address of g_noalloc_workspace on the current device, looked up
// once per device and kept. Calls after the first on a device read the kept
// address without taking the lock.
static gdn_status noalloc_workspace(void** addr) {
  static std::mutex mu;
  static std::atomic<void*> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
  if (dev < 0 || dev >= 64) return GDN_ERR_ARCH;
  void* a = cached[dev].load(std::memory_order_acquire);
  if (!a) {
    std::lock_guard<std::mutex> lock(mu);
    a = cached[dev].load(std::memory_order_relaxed);
    if (!a) {
      if (cudaGetSymbolAddress(&a, g_noalloc_workspace) != cudaSuccess || !a) return GDN_ERR_CUDA;
      cached[dev].store(a, std::memory_order_release);
    }
  }
  *addr = a;
  return GDN_OK;
}

}  // namespace gdn

extern "C" gdn_status gdn_prefill_varlen_noalloc(const void* q, const void* k, const void* v,
                                                 const void* g, const void* beta,
                                                 const int32_t* cu_seqlens,
                                                 const float* initial_state,
                                                 const int32_t* state_index, void* out,
                                                 float* final_state, const gdn_desc* desc,
                                                 void* stream) {
  if (!desc) return GDN_ERR_NULL;
  if (desc->num_seqs > GDN_NOALLOC_MAX_SEQS) return GDN_ERR_WORKSPACE;
  const gdn_status arch = check_arch();
  if (arch != GDN_OK) return arch;
  void* ws = nullptr;
  const gdn_status st = noalloc_workspace(&ws);
  if (st != GDN_OK) return st;
  gdn_desc d = *desc;
  d.workspace = ws;
  d.workspace_bytes = kNoallocBytes;
  return gdn_prefill_varlen(q, k, v, g, beta, cu_seqlens, initial_state, state_index, out,
                            final_state, &d, stream);
}

extern "C" gdn_status gdn_gated_rmsnorm(const void* o, const void* z, const float* weight, void* y,
                                        int64_t rows, int32_t d_v, gdn_dtype x_dtype, gdn_dtype z_dtype,
                                        float eps, void* stream) {
  if (rows < 0 || (d_v != 64 && d_v != 128 && d_v != 256)) return GDN_ERR_SHAPE;
  if ((x_dtype != GDN_BF16 && x_dtype != GDN_F32) || (z_dtype != GDN_BF16 && z_dtype != GDN_F32))
    return GDN_ERR_DTYPE;
  if (!(eps > 0.f) || !(eps < 3.0e38f)) return GDN_ERR_VALUE;
  if (rows == 0) return GDN_OK;
  if (!o || !z || !weight || !y) return GDN_ERR_NULL;
  if (!aligned(o, 16) || !aligned(z, 16) || !aligned(weight, 16) || !aligned(y, 16)) return GDN_ERR_ALIGN;
  const size_t xb = (size_t)rows * (size_t)d_v * (x_dtype == GDN_F32 ? 4 : 2);
  const size_t zb = (size_t)rows * (size_t)d_v * (z_dtype == GDN_F32 ? 4 : 2);
  // y may be o itself (each entry is read before the same thread writes it), not a
  // shifted view of it, and may not overlap z or the weights
  if (y != o && overlaps(y, xb, o, xb)) return GDN_ERR_ALIAS;
  if (overlaps(y, xb, z, zb) || overlaps(y, xb, weight, (size_t)d_v * 4)) return GDN_ERR_ALIAS;
  const gdn_status arch = check_arch();
  if (arch != GDN_OK) return arch;
  const cudaError_t e = launch_gated_rmsnorm(o, z, weight, y, rows, d_v, x_dtype == GDN_F32, z_dtype == GDN_F32,
                                             eps, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

static gdn_status input_prep(const void* x, const float* conv_w, const float* conv_bias,
                             const int32_t* cu_seqlens, const int32_t* parent, const void* conv_state_in,
                             const int32_t* state_index, const void* a, const void* b, const float* A_log,
                             const float* dt_bias, void* q, void* k, void* v, float* g, float* beta,
                             void* conv_state_out, const gdn_prep_desc* desc, void* stream, bool tree) {
  if (!desc) return GDN_ERR_NULL;
  if (tree && desc->num_seqs > 0 && !parent) return GDN_ERR_NULL;
  const gdn_prep_desc& d = *desc;
  if (d.num_seqs < 0 || d.total_tokens < 0 || d.h_qk < 1 || d.h_v < 1 || d.d_k < 8 || d.d_v < 8 ||
      d.d_k % 8 || d.d_v % 8 || d.conv_width < 2 || d.conv_width > 4 || d.num_state_slots < 0)
    return GDN_ERR_SHAPE;
  const int64_t Cq = (int64_t)d.h_qk * d.d_k, Cv = (int64_t)d.h_v * d.d_v, C = 2 * Cq + Cv;
  if (C > (int64_t)1 << 24) return GDN_ERR_SHAPE;
  if (d.num_seqs == 0 && d.total_tokens > 0) return GDN_ERR_SHAPE;  // rows but no sequence
  if (conv_state_in && (d.num_state_slots == 0 || (!state_index && d.num_state_slots < d.num_seqs)))
    return GDN_ERR_SHAPE;
  if (d.num_seqs == 0) return GDN_OK;
  const int64_t T = d.total_tokens;
  const int K = d.conv_width;
  if (!cu_seqlens) return GDN_ERR_NULL;
  if (T > 0 && (!x || !conv_w || !q || !k || !v)) return GDN_ERR_NULL;
  if (a && (!b || !A_log || !dt_bias || !g || !beta)) return GDN_ERR_NULL;
  const void* v16[] = {x, conv_w, q, k, v, conv_state_in, conv_state_out};
  for (const void* ptr : v16)
    if (!aligned(ptr, 16)) return GDN_ERR_ALIGN;
  const void* v4[] = {conv_bias, cu_seqlens, parent, state_index, A_log, dt_bias, g, beta};
  for (const void* ptr : v4)
    if (!aligned(ptr, 4)) return GDN_ERR_ALIGN;
  if (!aligned(a, 2) || !aligned(b, 2)) return GDN_ERR_ALIGN;
  // outputs overlap no input and no other output
  const bool gates = a != nullptr;
  const size_t gb = gates ? (size_t)T * d.h_v * 4 : 0, ab = gates ? (size_t)T * d.h_v * 2 : 0;
  struct R { const void* p; size_t n; };
  const R ins[] = {{x, (size_t)T * C * 2},
                   {conv_w, (size_t)C * K * 4},
                   {conv_bias, conv_bias ? (size_t)C * 4 : 0},
                   {cu_seqlens, (size_t)(d.num_seqs + 1) * 4},
                   {conv_state_in, conv_state_in ? (size_t)d.num_state_slots * (K - 1) * C * 2 : 0},
                   {state_index, state_index ? (size_t)d.num_seqs * 4 : 0},
                   {parent, tree ? (size_t)d.num_seqs * 4 : 0},
                   {a, ab},
                   {b, ab},
                   {A_log, gates ? (size_t)d.h_v * 4 : 0},
                   {dt_bias, gates ? (size_t)d.h_v * 4 : 0}};
  const R outs[] = {{q, (size_t)T * Cq * 2},
                    {k, (size_t)T * Cq * 2},
                    {v, (size_t)T * Cv * 2},
                    {g, gb},
                    {beta, gb},
                    {conv_state_out, conv_state_out ? (size_t)d.num_seqs * (K - 1) * C * 2 : 0}};
  for (size_t i = 0; i < sizeof(outs) / sizeof(outs[0]); ++i) {
    for (const R& r : ins)
      if (overlaps(outs[i].p, outs[i].n, r.p, r.n)) return GDN_ERR_ALIAS;
    for (size_t j = i + 1; j < sizeof(outs) / sizeof(outs[0]); ++j)
      if (overlaps(outs[i].p, outs[i].n, outs[j].p, outs[j].n)) return GDN_ERR_ALIAS;
  }
  const gdn_status arch = check_arch();
  if (arch != GDN_OK) return arch;
  InputPrepArgs p;
  p.x = x;
  p.conv_w = conv_w;
  p.conv_bias = conv_bias;
  p.cu_seqlens = cu_seqlens;
  p.conv_state_in = conv_state_in;
  p.state_index = state_index;
  p.parent = tree ? parent : nullptr;
  p.a = a;
  p.b = b;
  p.A_log = A_log;
  p.dt_bias = dt_bias;
  p.q = q;
  p.k = k;
  p.v = v;
  p.g = g;
  p.beta = beta;
  p.conv_state_out = conv_state_out;
  p.T = T;
  p.N = d.num_seqs;
  p.C = (int)C;
  p.Cq = (int)Cq;
  p.h_v = d.h_v;
  p.K = K;
  p.slots = conv_state_in ? d.num_state_slots : 0;
  const cudaError_t e = launch_input_prep(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

extern "C" gdn_status gdn_input_prep(const void* x, const float* conv_w, const float* conv_bias,
                                     const int32_t* cu_seqlens, const void* conv_state_in,
                                     const int32_t* state_index, const void* a, const void* b,
                                     const float* A_log, const float* dt_bias, void* q, void* k, void* v,
                                     float* g, float* beta, void* conv_state_out, const gdn_prep_desc* desc,
                                     void* stream) {
  return input_prep(x, conv_w, conv_bias, cu_seqlens, nullptr, conv_state_in, state_index, a, b, A_log, dt_bias,
                    q, k, v, g, beta, conv_state_out, desc, stream, false);
}

extern "C" gdn_status gdn_input_prep_tree(const void* x, const float* conv_w, const float* conv_bias,
                                          const int32_t* cu_seqlens, const int32_t* parent,
                                          const void* conv_state_in, const int32_t* state_index, const void* a,
                                          const void* b, const float* A_log, const float* dt_bias, void* q,
                                          void* k, void* v, float* g, float* beta, void* conv_state_out,
                                          const gdn_prep_desc* desc, void* stream) {
  return input_prep(x, conv_w, conv_bias, cu_seqlens, parent, conv_state_in, state_index, a, b, A_log, dt_bias,
                    q, k, v, g, beta, conv_state_out, desc, stream, true);
}
