// Gated RMSNorm of the prefill output (gdn_gated_rmsnorm in include/gdn.h):
//
//     y_j = w_j * x_j / sqrt(mean_j(x_j^2) + eps) * silu(z_j),  silu(z) = z / (1 + e^-z)
//
// over every row x of d_v entries (one token and value head). The open-jev-fast
// README lists the gated RMSNorm among the six fused element-wise kernels that
// follow its Gated DeltaNet core (Phase 2 item 1) and reports fusing it into that
// core as measured and rejected (item 4); it is kept as its own kernel here too.
//
// The kernel is bound by HBM: one read of o and z and one write of y, nothing
// reused. Each thread owns 8 consecutive entries of a row (one 16-byte bf16
// vector, two for fp32), a row is d_v / 8 consecutive lanes, so every load and
// store is coalesced and 16 bytes wide; the row's sum of squares is a butterfly
// over its lanes. The grid is persistent (blocks resident on every SM) and each
// warp has kGroups row groups in flight. y may be o itself (each entry is read by the
// thread that later writes it), so o is not declared restrict.
#include <cuda_bf16.h>
#include <stdint.h>

#include <mutex>

#include "gdn_internal.cuh"
#include "gdn_ops.cuh"

namespace gdn {
namespace {

constexpr int kNormThreads = 256;
constexpr int kGroups = 2;  // row groups in flight per warp

// 8 entries as loaded: bf16 stays packed (4 registers) until the arithmetic, so
// that more loads fit in flight per thread
template <typename T> struct Raw8;
template <> struct Raw8<__nv_bfloat16> { uint4 u; };
template <> struct Raw8<float> { float4 a, b; };

__device__ __forceinline__ void load8(const __nv_bfloat16* p, Raw8<__nv_bfloat16>& r) {
  r.u = __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void load8(const float* p, Raw8<float>& r) {
  r.a = __ldcs(reinterpret_cast<const float4*>(p));
  r.b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
}
__device__ __forceinline__ void zero8(Raw8<__nv_bfloat16>& r) { r.u = make_uint4(0u, 0u, 0u, 0u); }
__device__ __forceinline__ void zero8(Raw8<float>& r) { r.a = r.b = make_float4(0.f, 0.f, 0.f, 0.f); }

__device__ __forceinline__ void unpack8(const Raw8<__nv_bfloat16>& r, float (&f)[8]) {
  const uint32_t w[4] = {r.u.x, r.u.y, r.u.z, r.u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ void unpack8(const Raw8<float>& r, float (&f)[8]) {
  f[0] = r.a.x; f[1] = r.a.y; f[2] = r.a.z; f[3] = r.a.w;
  f[4] = r.b.x; f[5] = r.b.y; f[6] = r.b.z; f[7] = r.b.w;
}

__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&f)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  __stcs(reinterpret_cast<uint4*>(p), make_uint4(w[0], w[1], w[2], w[3]));
}

__device__ __forceinline__ void store8(float* p, const float (&f)[8]) {
  __stcs(reinterpret_cast<float4*>(p), make_float4(f[0], f[1], f[2], f[3]));
  __stcs(reinterpret_cast<float4*>(p) + 1, make_float4(f[4], f[5], f[6], f[7]));
}

// silu(z) = z / (1 + e^-z). e^-z is capped at e^80, so the fast division
// never sees a divisor near its 2^126 limit; below z = -80 the result is z e^-80
// instead of z e^z, both far below anything a bf16 or fp32 output resolves next to
// the row's other entries.
__device__ __forceinline__ float silu(float z) {
  return __fdividef(z, 1.0f + __expf(fminf(-z, 80.0f)));
}

template <typename TX, typename TZ, int DV>
__global__ void __launch_bounds__(kNormThreads)
    gated_rmsnorm_kernel(const TX* o, const TZ* __restrict__ z, const float* __restrict__ w, TX* y, int64_t rows,
                         float eps) {
  constexpr int LPR = DV / 8;    // lanes per row
  constexpr int RPW = 32 / LPR;  // rows per warp and row group
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPR, part = lane % LPR;
  float wv[8];
  {
    const float4 a = __ldg(reinterpret_cast<const float4*>(w + 8 * part));
    const float4 b = __ldg(reinterpret_cast<const float4*>(w + 8 * part) + 1);
    wv[0] = a.x; wv[1] = a.y; wv[2] = a.z; wv[3] = a.w;
    wv[4] = b.x; wv[5] = b.y; wv[6] = b.z; wv[7] = b.w;
  }
  const int64_t nwarps = (int64_t)gridDim.x * (kNormThreads / 32);
  const int64_t groups = (rows + RPW - 1) / RPW;
#pragma unroll 1
  for (int64_t gidx = (int64_t)blockIdx.x * (kNormThreads / 32) + threadIdx.x / 32; gidx < groups;
       gidx += kGroups * nwarps) {
    Raw8<TX> xr[kGroups];
    Raw8<TZ> zr[kGroups];
    int64_t r[kGroups];
#pragma unroll
    for (int s = 0; s < kGroups; ++s) {
      r[s] = (gidx + s * nwarps) * RPW + sub;
      if (r[s] < rows) {
        load8(o + r[s] * DV + 8 * part, xr[s]);
        load8(z + r[s] * DV + 8 * part, zr[s]);
      } else {
        zero8(xr[s]);
        zero8(zr[s]);
      }
    }
#pragma unroll
    for (int s = 0; s < kGroups; ++s) {
      float x[8], zz[8];
      unpack8(xr[s], x);
      unpack8(zr[s], zz);
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
      for (int off = LPR / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      const float inv = rsqrtf(ss * (1.0f / DV) + eps);
      float out[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) out[e] = (x[e] * inv) * wv[e] * silu(zz[e]);
      if (r[s] < rows) store8(y + r[s] * DV + 8 * part, out);
    }
  }
}

template <typename TX, typename TZ, int DV>
cudaError_t launch_dv(const void* o, const void* z, const float* w, void* y, int64_t rows, float eps,
                      cudaStream_t stream) {
  auto kernel = gated_rmsnorm_kernel<TX, TZ, DV>;
  // resident blocks per SM of this instantiation, queried once per device
  static std::mutex mu;
  static int per_sm[64];
  int dev = 0, cap_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  e = device_sm_count(&cap_sm);
  if (e != cudaSuccess) return e;
  int cap_blocks = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (per_sm[dev] == 0) {
      int b = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, kNormThreads, 0);
      if (e != cudaSuccess) return e;
      per_sm[dev] = b > 0 ? b : 1;
    }
    cap_blocks = per_sm[dev];
  }
  constexpr int RPW = 32 / (DV / 8);
  const int64_t groups = (rows + RPW - 1) / RPW;
  const int64_t want = (groups + kGroups * (kNormThreads / 32) - 1) / (kGroups * (kNormThreads / 32));
  const int64_t cap = (int64_t)cap_sm * cap_blocks;
  const int blocks = (int)(want < cap ? want : cap);
  kernel<<<blocks, kNormThreads, 0, stream>>>(static_cast<const TX*>(o), static_cast<const TZ*>(z), w,
                                              static_cast<TX*>(y), rows, eps);
  return cudaGetLastError();
}

template <typename TX, typename TZ>
cudaError_t launch_xz(const void* o, const void* z, const float* w, void* y, int64_t rows, int d_v, float eps,
                      cudaStream_t stream) {
  switch (d_v) {
    case 64: return launch_dv<TX, TZ, 64>(o, z, w, y, rows, eps, stream);
    case 128: return launch_dv<TX, TZ, 128>(o, z, w, y, rows, eps, stream);
    default: return launch_dv<TX, TZ, 256>(o, z, w, y, rows, eps, stream);
  }
}

}  // namespace

cudaError_t launch_gated_rmsnorm(const void* o, const void* z, const float* w, void* y, int64_t rows, int d_v,
                                 bool x_f32, bool z_f32, float eps, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  if (x_f32)
    return z_f32 ? launch_xz<float, float>(o, z, w, y, rows, d_v, eps, stream)
                 : launch_xz<float, __nv_bfloat16>(o, z, w, y, rows, d_v, eps, stream);
  return z_f32 ? launch_xz<__nv_bfloat16, float>(o, z, w, y, rows, d_v, eps, stream)
               : launch_xz<__nv_bfloat16, __nv_bfloat16>(o, z, w, y, rows, d_v, eps, stream);
}

}  // namespace gdn
