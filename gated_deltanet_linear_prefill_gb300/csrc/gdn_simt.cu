// CUDA-core (SIMT) kernel for the chunked gated delta rule.
//
// The plain fp32 version of the chunked form (open-jev-fast README, Phase 3
// item 1: per 64-token chunk, gate cumsum, K K^T, the (I + A)^-1 solve, u and
// w, the chunk output and the state update), one thread block per
// (sequence, value head, 64-column slice of d_v). It is the correctness
// baseline the tensor-core kernel is measured against and a debugging
// fallback selected by GDN_FLAG_SIMT; every product runs in fp32 FMA.
//
// Per chunk of m <= 64 rows (rows past the sequence end are zero with
// beta = g = 0, which makes them inert):
//   r_i = 1/sqrt(|k_i|^2 + eps) (same for q); G = cumsum(g)
//   A_ij = beta_i e^{G_i-G_j} k_i.k_j (j < i);  T = (I + A)^-1
//   W = T diag(beta e^G) K;  U = T diag(beta) V;  U' = U - W S
//   O = scale (diag(e^G) Q S + (Q K^T o e^{G_i-G_j}, j <= i) U')
//   S <- e^{G_last} S + sum_j e^{G_last-G_j} k_j u'_j^T
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kDVB = 64;  // d_v columns per block

template <int DK>
struct SimtSmem {
  static constexpr int LDK = DK + 1, LDC = kChunk + 1, LDV = kDVB + 1;
  float K[kChunk * LDK];
  float Q[kChunk * LDK];
  float W[kChunk * LDK];
  float S[DK * LDV];
  float V[kChunk * LDV];
  float U[kChunk * LDV];  // U, then U'
  float T[kChunk * LDC];  // A, then T, then T diag(beta)
  float P[kChunk * LDC];  // masked decayed Q K^T
  float G[kChunk], eG[kChunk], B[kChunk];
};

// acc[r][c] = sum_x A(i, x) B(x, j) for i = ty + 16 r, j = tx + 16 c, with
// element (i, x) of A at A[i*sai + x*sax] and (x, j) of B at B[x*sbx + j*sbj].
template <int M, int N>
__device__ __forceinline__ void mm(int K, const float* A, int sai, int sax, const float* B,
                                   int sbx, int sbj, float (&acc)[M / 16][N / 16]) {
  constexpr int TM = M / 16, TN = N / 16;
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
#pragma unroll
  for (int r = 0; r < TM; ++r)
#pragma unroll
    for (int c = 0; c < TN; ++c) acc[r][c] = 0.f;
#pragma unroll 4
  for (int x = 0; x < K; ++x) {
    float a[TM], b[TN];
#pragma unroll
    for (int r = 0; r < TM; ++r) a[r] = A[(ty + 16 * r) * sai + x * sax];
#pragma unroll
    for (int c = 0; c < TN; ++c) b[c] = B[x * sbx + (tx + 16 * c) * sbj];
#pragma unroll
    for (int r = 0; r < TM; ++r)
#pragma unroll
      for (int c = 0; c < TN; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
  }
}

template <int DK>
__global__ void __launch_bounds__(kThreads) gdn_simt_kernel(Params p, int n_col_blocks) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SimtSmem<DK>& sm = *reinterpret_cast<SimtSmem<DK>*>(smem_raw);
  constexpr int LDK = SimtSmem<DK>::LDK, LDC = SimtSmem<DK>::LDC, LDV = SimtSmem<DK>::LDV;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ty = tid >> 4, tx = tid & 15;

  // unit -> (sequence in longest-first order, value head, column block)
  const int unit = blockIdx.x;
  const int per_seq = p.h_v * n_col_blocks;
  const int n = p.order[unit / per_seq];
  if (n < 0 || n >= p.num_seqs) {  // never expected: the prep kernel writes a permutation
    if (threadIdx.x == 0) report(p.status, GDN_ERR_SEQLENS, (uint32_t)unit);
    return;
  }
  const int h = (unit % per_seq) / n_col_blocks;
  const int cb = unit % n_col_blocks;
  const int hq = h / (p.h_v / p.h_qk);
  const int c0 = cb * kDVB;
  int64_t bos, eos;
  seq_bounds(p, n, bos, eos);

  // initial state slice S[x][c] = S0[x][c0 + c]
  const int64_t slot = state_slot(p, n);
  for (int e = tid; e < DK * kDVB; e += kThreads) {
    const int x = e / kDVB, c = e % kDVB;
    sm.S[x * LDV + c] =
        slot >= 0 ? p.initial_state[(((size_t)slot * p.h_v + h) * DK + x) * p.d_v + c0 + c] : 0.f;
  }

  for (int64_t t0 = bos; t0 < eos; t0 += kChunk) {
    const int m = (int)((eos - t0) < kChunk ? (eos - t0) : kChunk);
    __syncthreads();  // previous chunk finished with every buffer
    // ---- load (rows >= m are zero)
    for (int e = tid; e < kChunk * DK; e += kThreads) {
      const int i = e / DK, x = e % DK;
      float kv = 0.f, qv = 0.f;
      if (i < m) {
        const size_t off = ((size_t)(t0 + i) * p.h_qk + hq) * DK + x;
        kv = __bfloat162float(p.k[off]);
        qv = __bfloat162float(p.q[off]);
      }
      sm.K[i * LDK + x] = kv;
      sm.Q[i * LDK + x] = qv;
    }
    for (int e = tid; e < kChunk * kDVB; e += kThreads) {
      const int i = e / kDVB, c = e % kDVB;
      sm.V[i * LDV + c] =
          i < m ? __bfloat162float(p.v[((size_t)(t0 + i) * p.h_v + h) * p.d_v + c0 + c]) : 0.f;
    }
    if (tid < kChunk) {
      const int i = tid;
      sm.G[i] = i < m ? load_gate(p.g, (t0 + i) * p.h_v + h, p.gate_f32) : 0.f;
      sm.B[i] = i < m ? load_gate(p.beta, (t0 + i) * p.h_v + h, p.gate_f32) : 0.f;
    }
    __syncthreads();
    // ---- L2 norm of k and q rows (one warp per row) and the gate cumsum
    if (p.l2norm) {
      for (int i = warp; i < 2 * kChunk; i += kThreads / 32) {
        float* row = (i < kChunk ? sm.K : sm.Q) + (i % kChunk) * LDK;
        float ss = 0.f;
        for (int x = lane; x < DK; x += 32) ss = fmaf(row[x], row[x], ss);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float r = 1.0f / sqrtf(ss + 1e-6f);
        for (int x = lane; x < DK; x += 32) row[x] *= r;
      }
    }
    if (warp == 0) {  // inclusive scan of 64 gates, two per lane
      float a = sm.G[2 * lane], b = sm.G[2 * lane + 1];
      float s = a + b, incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const float base = incl - s;
      sm.G[2 * lane] = base + a;
      sm.G[2 * lane + 1] = base + a + b;
    }
    __syncthreads();
    if (tid < kChunk) sm.eG[tid] = expf(sm.G[tid]);
    // ---- A = strictly lower beta_i e^{G_i-G_j} k_i.k_j  (held in the W buffer until the solve)
    //      P = lower incl. e^{G_i-G_j} q_i.k_j
    float* Abuf = sm.W;
    {
      float acc[4][4];
      mm<64, 64>(DK, sm.K, LDK, 1, sm.K, 1, LDK, acc);
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int i = ty + 16 * r, j = tx + 16 * c;
          Abuf[i * LDC + j] = j < i ? sm.B[i] * expf(sm.G[i] - sm.G[j]) * acc[r][c] : 0.f;
        }
      mm<64, 64>(DK, sm.Q, LDK, 1, sm.K, 1, LDK, acc);
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int i = ty + 16 * r, j = tx + 16 * c;
          sm.P[i * LDC + j] = j <= i ? expf(sm.G[i] - sm.G[j]) * acc[r][c] : 0.f;
        }
    }
    __syncthreads();
    // ---- T = (I + A)^-1 by forward substitution; thread j owns column j and
    // reads only its own earlier rows of T plus row i of A.
    if (tid < kChunk) {
      const int j = tid;
      for (int i = 0; i < kChunk; ++i) {
        float s = (i == j) ? 1.f : 0.f;
        for (int x = j; x < i; ++x) s = fmaf(-Abuf[i * LDC + x], sm.T[x * LDC + j], s);
        sm.T[i * LDC + j] = s;
      }
    }
    __syncthreads();
    // ---- T <- T diag(beta)
    for (int e = tid; e < kChunk * kChunk; e += kThreads) {
      const int i = e / kChunk, j = e % kChunk;
      sm.T[i * LDC + j] *= sm.B[j];
    }
    __syncthreads();
    // ---- W = (T diag(beta)) diag(e^G) K   [64 x DK];  U = (T diag(beta)) V   [64 x 64]
    {
      // e^{G_j} is folded into the A operand, (T diag(beta))_ij e^{G_j}, so K stays unscaled
      float acc[4][DK / 16];
      {
        constexpr int TN = DK / 16;
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int c = 0; c < TN; ++c) acc[r][c] = 0.f;
#pragma unroll 4
        for (int x = 0; x < kChunk; ++x) {
          const float ex = sm.eG[x];
          float a[4], b[TN];
#pragma unroll
          for (int r = 0; r < 4; ++r) a[r] = sm.T[(ty + 16 * r) * LDC + x] * ex;
#pragma unroll
          for (int c = 0; c < TN; ++c) b[c] = sm.K[x * LDK + tx + 16 * c];
#pragma unroll
          for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < TN; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
        }
      }
      float accu[4][4];
      mm<64, 64>(kChunk, sm.T, LDC, 1, sm.V, LDV, 1, accu);
      __syncthreads();  // A (kept in the W buffer) is no longer read: W may be written
#pragma unroll
      for (int r = 0; r < 4; ++r) {
#pragma unroll
        for (int c = 0; c < DK / 16; ++c) sm.W[(ty + 16 * r) * LDK + tx + 16 * c] = acc[r][c];
#pragma unroll
        for (int c = 0; c < 4; ++c) sm.U[(ty + 16 * r) * LDV + tx + 16 * c] = accu[r][c];
      }
    }
    __syncthreads();
    // ---- U' = U - W S ;  O = scale (e^G o (Q S) + P U')
    {
      float acc[4][4];
      mm<64, 64>(DK, sm.W, LDK, 1, sm.S, LDV, 1, acc);
      float qs[4][4];
      mm<64, 64>(DK, sm.Q, LDK, 1, sm.S, LDV, 1, qs);
      __syncthreads();  // everyone has read S and W before U is overwritten
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int i = ty + 16 * r, j = tx + 16 * c;
          sm.U[i * LDV + j] -= acc[r][c];
        }
      __syncthreads();
      float pu[4][4];
      mm<64, 64>(kChunk, sm.P, LDC, 1, sm.U, LDV, 1, pu);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int i = ty + 16 * r;
        if (i < m) {
          const size_t row = ((size_t)(t0 + i) * p.h_v + h) * p.d_v + c0;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int j = tx + 16 * c;
            const float o = p.scale * fmaf(sm.eG[i], qs[r][c], pu[r][c]);
            if (p.out_f32)
              reinterpret_cast<float*>(p.out)[row + j] = o;
            else
              reinterpret_cast<__nv_bfloat16*>(p.out)[row + j] = __float2bfloat16_rn(o);
          }
        }
      }
    }
    // ---- S <- e^{G_last} S + sum_j (e^{G_last-G_j} k_j) u'_j^T
    {
      const float gl = sm.G[kChunk - 1];
      constexpr int TM = DK / 16;
      float acc[TM][4];
#pragma unroll
      for (int r = 0; r < TM; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
#pragma unroll 4
      for (int j = 0; j < kChunk; ++j) {
        const float d = expf(gl - sm.G[j]);
        float a[TM], b[4];
#pragma unroll
        for (int r = 0; r < TM; ++r) a[r] = sm.K[j * LDK + ty + 16 * r] * d;
#pragma unroll
        for (int c = 0; c < 4; ++c) b[c] = sm.U[j * LDV + tx + 16 * c];
#pragma unroll
        for (int r = 0; r < TM; ++r)
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
      }
      const float el = expf(gl);
#pragma unroll
      for (int r = 0; r < TM; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float* s = &sm.S[(ty + 16 * r) * LDV + tx + 16 * c];
          *s = fmaf(el, *s, acc[r][c]);
        }
    }
  }
  __syncthreads();
  if (p.final_state) {
    for (int e = tid; e < DK * kDVB; e += kThreads) {
      const int x = e / kDVB, c = e % kDVB;
      p.final_state[(((size_t)n * p.h_v + h) * DK + x) * p.d_v + c0 + c] = sm.S[x * LDV + c];
    }
  }
}

template <int DK>
cudaError_t launch_simt_dk(const Params& p, cudaStream_t stream) {
  const size_t smem = sizeof(SimtSmem<DK>);
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(&gdn_simt_kernel<DK>), (int)smem);
  if (e != cudaSuccess) return e;
  const int ncb = p.d_v / kDVB;
  const long long units = (long long)p.num_seqs * p.h_v * ncb;
  if (units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  gdn_simt_kernel<DK><<<(unsigned)units, kThreads, smem, stream>>>(p, ncb);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_simt(const Params& p, cudaStream_t stream) {
  return p.d_k == 128 ? launch_simt_dk<128>(p, stream) : launch_simt_dk<64>(p, stream);
}

}  // namespace gdn
