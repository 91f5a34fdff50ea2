// GDN input prep (gdn_input_prep in include/gdn.h): the steps in front of the
// gated delta rule that the open-jev-fast README fuses into one kernel (Phase 2
// item 1): causal depthwise convolution and SiLU over the packed projection rows,
// the q / k / v split, and the gate parameters.
//
//   u[t, c]  = silu(bias[c] + sum_j w[c, j] x[t - (K-1) + j, c])     (per sequence;
//              rows before a sequence's start read its carried window)
//   q | k | v = u[:, 0:Cq] | u[:, Cq:2Cq] | u[:, 2Cq:]                (Cq = h_qk d_k)
//   g[t, h]  = -exp(A_log[h]) softplus(a[t, h] + dt_bias[h]),  beta = sigmoid(b)
//
// Head expansion is not materialised: the prefill maps value head h to q/k head
// h / (h_v / h_qk) itself. The L2 norm of q and k also stays in the prefill (fp32,
// before the values are rounded).
//
// Both kernels are bound by HBM. The convolution gives each thread 8 consecutive
// channels (one 16-byte bf16 vector) over a run of kRows rows: partial sums of the
// open outputs stay in registers, rows stream through a per-thread ring in shared
// memory (cp.async) so that many loads are in flight, and a warp's loads and stores
// cover 512 contiguous bytes of a row. A run that starts inside a sequence re-reads its K-1 halo rows (3 of 128
// rows for K = 4). Consecutive blocks take the channel blocks of one run.
#include <cuda_bf16.h>
#include <stdint.h>

#include "gdn_internal.cuh"
#include "gdn_ops.cuh"

namespace gdn {
namespace {

constexpr int kConvThreads = 128;
constexpr int kRows = 128;   // rows per thread
constexpr int kStages = 16;  // rows in flight per thread (a ring of 16-byte slots in shared memory)
static_assert((kStages & (kStages - 1)) == 0, "ring slots are indexed with a mask");
constexpr int kConvBlocks = 5;  // resident blocks per SM the register budget allows (<= 102 registers)
constexpr int kAuxThreads = 256;

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// 16 bytes global -> shared without a register (cached in L2 only), and its group
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// silu(y) = y / (1 + e^-y), with e^-y capped at e^80 so that the fast division stays
// in range (below y = -80 the result is y e^-80 instead of y e^y: both round to a
// bf16 far below the row's other entries).
__device__ __forceinline__ float silu(float y) { return __fdividef(y, 1.0f + __expf(fminf(-y, 80.0f))); }

// The sequence holding row t: the largest n with cu[n] <= t (empty sequences are
// never chosen), clamped to [0, N-1].
__device__ __forceinline__ int seq_of(const int32_t* cu, int N, int64_t t) {
  int lo = 0, hi = N;  // answer in [lo, hi)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if ((int64_t)cu[mid] <= t) lo = mid; else hi = mid;
  }
  return lo;
}

struct PrepArgs {
  const __nv_bfloat16* x;
  const float* w;     // [C, K]
  const float* bias;  // [C] or null
  const int32_t* cu;
  const __nv_bfloat16* state_in;  // [slots, K-1, C] or null
  const int32_t* state_index;     // [N] or null
  const int32_t* parent;          // [N] or null: a prefix tree (parent[n] in [-1, n))
  __nv_bfloat16* q;
  __nv_bfloat16* k;
  __nv_bfloat16* v;
  __nv_bfloat16* state_out;  // [N, K-1, C] or null
  const __nv_bfloat16* a;    // [T, h_v] or null (no gates)
  const __nv_bfloat16* b;
  const float* A_log;
  const float* dt_bias;
  float* g;
  float* beta;
  int64_t T;
  int N, C, Cq, h_v, slots;
};

// the carried window's row r (0 = oldest) of sequence n, 8 channels from c8 * 8,
// as loaded (packed bf16). In a tree the window is the last rows of the ancestors'
// path: the walk goes up parent by parent (indices fall, so it ends) until the row
// is inside one, else the root's carried window supplies it. A parent outside
// [-1, n) counts as none.
__device__ __forceinline__ uint4 carried_row(const PrepArgs& p, int K, int n, int r, int c8) {
  if (p.parent) {
    int64_t need = (K - 1) - r;  // rows before sequence n's first row
#pragma unroll 1
    for (int steps = 0; steps < p.N; ++steps) {
      const int32_t pa = p.parent[n];
      if (pa < 0 || pa >= n) break;
      const int64_t pb = p.cu[pa] > 0 ? (int64_t)p.cu[pa] : 0;
      const int64_t pe = (int64_t)p.cu[pa + 1] < p.T ? (int64_t)p.cu[pa + 1] : p.T;
      const int64_t len = pe > pb ? pe - pb : 0;
      if (need <= len)
        return __ldg(reinterpret_cast<const uint4*>(p.x + (pe - need) * p.C) + c8);
      need -= len;
      n = pa;
    }
    r = (K - 1) - (int)need;
  }
  int64_t slot = -1;
  if (p.state_in) {
    slot = p.state_index ? (int64_t)p.state_index[n] : (int64_t)n;
    if (slot >= p.slots) slot = -1;
  }
  if (slot < 0) return make_uint4(0u, 0u, 0u, 0u);
  return __ldg(reinterpret_cast<const uint4*>(p.state_in + ((size_t)slot * (K - 1) + r) * p.C) + c8);
}

// x row r or, before the sequence's first row bos, row r - bos + (K-1) of its
// carried window (as loaded, packed bf16)
template <int K>
__device__ __forceinline__ uint4 row_or_carried(const PrepArgs& p, int64_t r, int64_t bos, int n, int c8) {
  if (r >= bos) return __ldcs(reinterpret_cast<const uint4*>(p.x + r * p.C) + c8);
  return carried_row(p, K, n, (K - 1) - (int)(bos - r), c8);
}

// The convolution runs as a scatter: when row t arrives (unpacked once) it completes
// output t and adds its term to the K-2 outputs still open after it, whose partial
// sums acc[0..K-2] (bias first, then the taps in order) stay in registers as channel
// pairs for the packed fp32 multiply-add. Starting a run (or a sequence) feeds the
// K-1 rows before it through the same update without emitting anything. A
// sequence's final window is read again at its last row (once per sequence).
template <int K, bool BIAS>
__global__ void __launch_bounds__(kConvThreads, kConvBlocks) conv_silu_kernel(PrepArgs p) {
  const int nvec = p.C / 8;
  const int cblocks = (nvec + kConvThreads - 1) / kConvThreads;
  const int c8 = (int)(blockIdx.x % cblocks) * kConvThreads + threadIdx.x;
  const int64_t t0 = (int64_t)(blockIdx.x / cblocks) * kRows;
  if (c8 >= nvec || t0 >= p.T) return;
  const int64_t t1 = t0 + kRows < p.T ? t0 + kRows : p.T;
  const int c = 8 * c8;

  float2 wt[K][4], bs[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float a_[K], b_[K];
    if constexpr (K == 4) {
      const float4 wa = __ldg(reinterpret_cast<const float4*>(p.w + (size_t)(c + 2 * e) * 4));
      const float4 wb = __ldg(reinterpret_cast<const float4*>(p.w + (size_t)(c + 2 * e + 1) * 4));
      a_[0] = wa.x; a_[1] = wa.y; a_[2] = wa.z; a_[3] = wa.w;
      b_[0] = wb.x; b_[1] = wb.y; b_[2] = wb.z; b_[3] = wb.w;
    } else {
#pragma unroll
      for (int j = 0; j < K; ++j) {
        a_[j] = __ldg(p.w + (size_t)(c + 2 * e) * K + j);
        b_[j] = __ldg(p.w + (size_t)(c + 2 * e + 1) * K + j);
      }
    }
#pragma unroll
    for (int j = 0; j < K; ++j) wt[j][e] = make_float2(a_[j], b_[j]);
    bs[e] = BIAS ? make_float2(__ldg(p.bias + c + 2 * e), __ldg(p.bias + c + 2 * e + 1)) : make_float2(0.f, 0.f);
  }
  // where this thread's outputs go: q, k or v, and the channel offset inside it
  __nv_bfloat16* dst;
  int ldd, cd;
  if (c < p.Cq) { dst = p.q; ldd = p.Cq; cd = c; }
  else if (c < 2 * p.Cq) { dst = p.k; ldd = p.Cq; cd = c - p.Cq; }
  else { dst = p.v; ldd = p.C - 2 * p.Cq; cd = c - 2 * p.Cq; }

  float2 acc[K - 1][4];
  // row xr enters: returns nothing, completes output (acc[0] + w_{K-1} x) into `out`
  auto feed = [&](const uint4& xr, float2 (&out)[4]) {
    const uint32_t xw[4] = {xr.x, xr.y, xr.z, xr.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 xv = make_float2(__uint_as_float(xw[e] << 16), __uint_as_float(xw[e] & 0xffff0000u));
      out[e] = __ffma2_rn(wt[K - 1][e], xv, acc[0][e]);
#pragma unroll
      for (int j = 0; j < K - 2; ++j) acc[j][e] = __ffma2_rn(wt[K - 2 - j][e], xv, acc[j + 1][e]);
      acc[K - 2][e] = __ffma2_rn(wt[0][e], xv, bs[e]);
    }
  };
  // the K-1 rows before row t of sequence n (which starts at bos) prime the sums
  auto prime = [&](int64_t t, int64_t bos, int n) {
#pragma unroll
    for (int j = 0; j < K - 1; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[j][e] = bs[e];
#pragma unroll
    for (int j = 0; j < K - 1; ++j) {
      float2 unused[4];
      feed(row_or_carried<K>(p, t - (K - 1) + j, bos, n, c8), unused);
    }
  };

  int n = seq_of(p.cu, p.N, t0);
  int64_t bos = p.cu[n] > 0 ? (int64_t)p.cu[n] : 0;
  int64_t eos = p.cu[n + 1];
  prime(t0, bos > t0 ? t0 : bos, n);
  // Rows stream through a ring of kStages 16-byte slots per thread: the copy of row
  // t + kStages - 1 is issued before row t is used, so kStages - 1 rows are in flight
  // without holding registers. A thread reads only its own slots (no block barrier).
  __shared__ uint4 ring[kStages][kConvThreads];
  const uint32_t slot0 = (uint32_t)__cvta_generic_to_shared(&ring[0][threadIdx.x]);
  auto issue = [&](int64_t r) {  // an empty group past the run keeps the group count uniform
    if (r < t1) cp_async16(slot0 + (uint32_t)((r - t0) & (kStages - 1)) * (kConvThreads * 16u), p.x + r * p.C + 8 * c8);
    cp_async_commit();
  };
#pragma unroll
  for (int s_ = 0; s_ < kStages - 1; ++s_) issue(t0 + s_);
#pragma unroll 1
  for (int64_t t = t0; t < t1; ++t) {
    issue(t + kStages - 1);
    cp_async_wait<kStages - 1>();  // row t's group has landed
    const uint4 xr = ring[(t - t0) & (kStages - 1)][threadIdx.x];
    if (t >= eos) {  // a new sequence starts at row t (skipping empty ones)
      while (n + 1 < p.N && (int64_t)p.cu[n + 1] <= t) ++n;
      bos = t;
      eos = p.cu[n + 1];
      prime(t, bos, n);
    }
    float2 y[4];
    feed(xr, y);
    float out[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      out[2 * e] = silu(y[e].x);
      out[2 * e + 1] = silu(y[e].y);
    }
    __stcs(reinterpret_cast<uint4*>(dst + t * ldd + cd), pack8(out));
    if (t == eos - 1 && p.state_out) {  // the sequence's last row: its final window
#pragma unroll
      for (int j = 0; j < K - 1; ++j)
        *(reinterpret_cast<uint4*>(p.state_out + ((size_t)n * (K - 1) + j) * p.C) + c8) =
            row_or_carried<K>(p, t - (K - 2) + j, bos, n, c8);
    }
  }
  cp_async_wait<0>();  // no copy outlives the thread
}

// Gate parameters over every (row, value head), and the final windows of empty
// sequences (their carried window, or zeros), which no row of the convolution visits.
template <int K>
__global__ void __launch_bounds__(kAuxThreads) gates_kernel(PrepArgs p) {
  const int64_t stride = (int64_t)gridDim.x * kAuxThreads;
  const int64_t id0 = (int64_t)blockIdx.x * kAuxThreads + threadIdx.x;
  if (p.a) {
    const int64_t total = p.T * p.h_v;
    for (int64_t i = id0; i < total; i += stride) {
      const int h = (int)(i % p.h_v);
      const float s = __bfloat162float(p.a[i]) + __ldg(p.dt_bias + h);
      const float sp = s > 20.f ? s + log1pf(expf(-s)) : log1pf(expf(s));  // ln(1 + e^s)
      p.g[i] = -expf(__ldg(p.A_log + h)) * sp;
      p.beta[i] = 1.0f / (1.0f + expf(-__bfloat162float(p.b[i])));
    }
  }
  if (p.state_out) {
    const int nvec = p.C / 8;
    const int64_t total = (int64_t)p.N * nvec;
    for (int64_t i = id0; i < total; i += stride) {
      const int n = (int)(i / nvec), c8 = (int)(i % nvec);
      if (p.cu[n + 1] != p.cu[n]) continue;
      for (int j = 0; j < K - 1; ++j)
        *(reinterpret_cast<uint4*>(p.state_out + ((size_t)n * (K - 1) + j) * p.C) + c8) = carried_row(p, K, n, j, c8);
    }
  }
}

template <int K>
cudaError_t launch_k(const PrepArgs& p, cudaStream_t stream) {
  const int nvec = p.C / 8;
  const int64_t cblocks = (nvec + kConvThreads - 1) / kConvThreads;
  const int64_t tiles = (p.T + kRows - 1) / kRows;
  if (tiles > 0) {
    if (p.bias)
      conv_silu_kernel<K, true><<<(unsigned)(tiles * cblocks), kConvThreads, 0, stream>>>(p);
    else
      conv_silu_kernel<K, false><<<(unsigned)(tiles * cblocks), kConvThreads, 0, stream>>>(p);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int64_t work = (p.a ? p.T * p.h_v : 0) > (p.state_out ? (int64_t)p.N * nvec : 0)
                           ? (p.a ? p.T * p.h_v : 0)
                           : (p.state_out ? (int64_t)p.N * nvec : 0);
  if (work > 0) {
    int64_t blocks = (work + kAuxThreads - 1) / kAuxThreads;
    if (blocks > 4096) blocks = 4096;
    gates_kernel<K><<<(unsigned)blocks, kAuxThreads, 0, stream>>>(p);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_input_prep(const InputPrepArgs& a, cudaStream_t stream) {
  PrepArgs p;
  p.x = static_cast<const __nv_bfloat16*>(a.x);
  p.w = a.conv_w;
  p.bias = a.conv_bias;
  p.cu = a.cu_seqlens;
  p.state_in = static_cast<const __nv_bfloat16*>(a.conv_state_in);
  p.state_index = a.state_index;
  p.parent = a.parent;
  p.q = static_cast<__nv_bfloat16*>(a.q);
  p.k = static_cast<__nv_bfloat16*>(a.k);
  p.v = static_cast<__nv_bfloat16*>(a.v);
  p.state_out = static_cast<__nv_bfloat16*>(a.conv_state_out);
  p.a = static_cast<const __nv_bfloat16*>(a.a);
  p.b = static_cast<const __nv_bfloat16*>(a.b);
  p.A_log = a.A_log;
  p.dt_bias = a.dt_bias;
  p.g = a.g;
  p.beta = a.beta;
  p.T = a.T;
  p.N = a.N;
  p.C = a.C;
  p.Cq = a.Cq;
  p.h_v = a.h_v;
  p.slots = a.slots;
  switch (a.K) {
    case 2: return launch_k<2>(p, stream);
    case 3: return launch_k<3>(p, stream);
    default: return launch_k<4>(p, stream);
  }
}

}  // namespace gdn
