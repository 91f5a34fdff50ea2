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
// channels (one 16-byte bf16 vector) over a run of kRows rows: the window of the
// K-1 previous rows stays in registers, rows are loaded kBatch at a time so that
// several loads are in flight, and a warp's loads and stores cover 512 contiguous
// bytes of a row. A run that starts inside a sequence re-reads its K-1 halo rows
// (3 of 32 rows for K = 4).
#include <cuda_bf16.h>
#include <stdint.h>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kConvThreads = 128;
constexpr int kRows = 32;   // rows per thread
constexpr int kBatch = 8;   // rows loaded at once
constexpr int kAuxThreads = 256;

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
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

// the carried window's row r (0 = oldest) of sequence n, 8 channels from c8 * 8
__device__ __forceinline__ void carried_row(const PrepArgs& p, int K, int n, int r, int c8, float (&f)[8]) {
  int64_t slot = -1;
  if (p.state_in) {
    slot = p.state_index ? (int64_t)p.state_index[n] : (int64_t)n;
    if (slot >= p.slots) slot = -1;
  }
  if (slot < 0) {
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = 0.f;
    return;
  }
  unpack8(__ldg(reinterpret_cast<const uint4*>(p.state_in + ((size_t)slot * (K - 1) + r) * p.C) + c8), f);
}

template <int K>
__global__ void __launch_bounds__(kConvThreads) conv_silu_kernel(PrepArgs p) {
  const int nvec = p.C / 8;
  const int cblocks = (nvec + kConvThreads - 1) / kConvThreads;
  const int c8 = (int)(blockIdx.x % cblocks) * kConvThreads + threadIdx.x;
  const int64_t t0 = (int64_t)(blockIdx.x / cblocks) * kRows;
  if (c8 >= nvec || t0 >= p.T) return;
  const int64_t t1 = t0 + kRows < p.T ? t0 + kRows : p.T;
  const int c = 8 * c8;

  float wt[K][8], bs[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
#pragma unroll
    for (int j = 0; j < K; ++j) wt[j][e] = __ldg(p.w + (size_t)(c + e) * K + j);
    bs[e] = p.bias ? __ldg(p.bias + c + e) : 0.f;
  }
  // where this thread's outputs go: q, k or v, and the channel offset inside it
  __nv_bfloat16* dst;
  int ldd, cd;
  if (c < p.Cq) { dst = p.q; ldd = p.Cq; cd = c; }
  else if (c < 2 * p.Cq) { dst = p.k; ldd = p.Cq; cd = c - p.Cq; }
  else { dst = p.v; ldd = p.C - 2 * p.Cq; cd = c - 2 * p.Cq; }

  int n = seq_of(p.cu, p.N, t0);
  int64_t bos = p.cu[n] > 0 ? (int64_t)p.cu[n] : 0;
  int64_t eos = p.cu[n + 1];
  // the window: rows t0-(K-1) .. t0-1, from x inside the sequence, else carried
  float win[K - 1][8];
#pragma unroll
  for (int j = 0; j < K - 1; ++j) {
    const int64_t r = t0 - (K - 1) + j;
    if (r >= bos && r >= 0) unpack8(__ldcs(reinterpret_cast<const uint4*>(p.x + r * p.C) + c8), win[j]);
    else if (bos - r <= K - 1) carried_row(p, K, n, (K - 1) - (int)(bos - r), c8, win[j]);
    else {
#pragma unroll
      for (int e = 0; e < 8; ++e) win[j][e] = 0.f;
    }
  }
#pragma unroll 1
  for (int64_t tb = t0; tb < t1; tb += kBatch) {
    uint4 raw[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i)
      if (tb + i < t1) raw[i] = __ldcs(reinterpret_cast<const uint4*>(p.x + (tb + i) * p.C) + c8);
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int64_t t = tb + i;
      if (t >= t1) break;
      if (t >= eos) {  // a new sequence starts at row t (skipping empty ones)
        while (n + 1 < p.N && (int64_t)p.cu[n + 1] <= t) ++n;
        bos = t;
        eos = p.cu[n + 1];
#pragma unroll
        for (int j = 0; j < K - 1; ++j) carried_row(p, K, n, j, c8, win[j]);
      }
      float xt[8], out[8];
      unpack8(raw[i], xt);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float y = bs[e];
#pragma unroll
        for (int j = 0; j < K - 1; ++j) y = fmaf(wt[j][e], win[j][e], y);
        y = fmaf(wt[K - 1][e], xt[e], y);
        out[e] = silu(y);
      }
      __stcs(reinterpret_cast<uint4*>(dst + t * ldd + cd), pack8(out));
#pragma unroll
      for (int j = 0; j < K - 2; ++j)
#pragma unroll
        for (int e = 0; e < 8; ++e) win[j][e] = win[j + 1][e];
#pragma unroll
      for (int e = 0; e < 8; ++e) win[K - 2][e] = xt[e];
      if (t == eos - 1 && p.state_out) {  // the sequence's last row: its final window
#pragma unroll
        for (int j = 0; j < K - 1; ++j)
          *(reinterpret_cast<uint4*>(p.state_out + ((size_t)n * (K - 1) + j) * p.C) + c8) = pack8(win[j]);
      }
    }
  }
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
      for (int j = 0; j < K - 1; ++j) {
        float f[8];
        carried_row(p, K, n, j, c8, f);
        *(reinterpret_cast<uint4*>(p.state_out + ((size_t)n * (K - 1) + j) * p.C) + c8) = pack8(f);
      }
    }
  }
}

template <int K>
cudaError_t launch_k(const PrepArgs& p, cudaStream_t stream) {
  const int nvec = p.C / 8;
  const int64_t cblocks = (nvec + kConvThreads - 1) / kConvThreads;
  const int64_t tiles = (p.T + kRows - 1) / kRows;
  if (tiles > 0) {
    conv_silu_kernel<K><<<(unsigned)(tiles * cblocks), kConvThreads, 0, stream>>>(p);
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
