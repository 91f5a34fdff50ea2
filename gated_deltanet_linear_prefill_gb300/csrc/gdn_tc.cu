// Tensor-core (tcgen05 / TMEM / TMA) kernel for the chunked gated delta rule.
//
// Chunked form (open-jev-fast README, Phase 3 item 1: per 64-token chunk the
// gate cumsum, K K^T, the (I + A)^-1 solve, u and w, the chunk output and the
// state update; the cost is per chunk). With S the d_k x d_v state entering a
// chunk of m <= 64 rows, G_i = sum_{s<=i} g_s, r^k_i / r^q_i the L2-norm
// scales of k_i / q_i:
//
//   A_ij = beta_i r^k_i r^k_j e^{G_i-G_j} k_i.k_j   (j < i)     T = (I + A)^-1
//   U  = T diag(beta) V               W = T diag(beta e^G r^k) K
//   U' = U - W S
//   o_i = scale r^q_i ( e^{G_i} S^T q_i + sum_{j<=i} e^{G_i-G_j} r^k_j (q_i.k_j) u'_j )
//   S  <- e^{G_m} S + sum_j (e^{G_m-G_j} r^k_j) k_j u'_j^T
//
// One CTA owns one (sequence, value head) chain and walks its chunks in order.
// All dense products run on tcgen05 in the "d-major" orientation, where the
// 128 TMEM lanes index d_v (or d_k) so every MMA has M = 128:
//   [K;Q] K^T          -> KK^T (lanes 0-63), QK^T (lanes 64-127)       (per chunk)
//   W^T  = K^T T_w^T    (T_w = T diag(beta e^G r^k), bf16)
//   U'^T = V^T T_b^T (T_b = T diag(beta) as bf16 hi + lo) - S^T W^T
//   O^T  = S^T Qh^T + U'^T P^T      (Qh_i = e^{G_i} q_i, P_ij = e^{G_i-G_j} r^k_j q_i.k_j)
//   S^T += (U' diag(s))^T K         (s_j = e^{G_m-G_j} r^k_j; U' diag(s) as bf16 hi + lo,
//                                    read by the MMA straight from TMEM)
// Operand precision: the products feeding the fp32 state carry T and U' as
// bf16 hi + lo pairs (about 16 significant bits); S and W enter as bf16; every
// accumulation is fp32 in TMEM. The triangular solve, decays and norms run on
// CUDA cores in fp32.
//
// Warp roles (384 threads): warp 0 loads K/Q/V tiles by TMA (128-byte swizzle)
// and the gates; warp 1 allocates TMEM and issues the state-independent MMAs;
// warp 2 issues the state-dependent MMAs; warps 4-7 (WG-A) prepare chunk c+1
// (norms, A and P, the solve, T_b / T_w / Qh, W^T) while warps 8-11 (WG-B) run
// chunk c's state step (S -> bf16 operand, U' split, output epilogue). Every
// mbarrier wait is bounded: on timeout the CTA reports GDN_ERR_DEVICE_TIMEOUT
// and unwinds.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace {

using namespace ptx;

constexpr int kTcThreads = 384;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait: far above any legal wait

// TMEM columns (fp32 unless noted)
constexpr uint32_t TM_S = 0;     // S^T: lanes d_v, columns d_k            (128)
constexpr uint32_t TM_R = 128;   // U^T, then U'^T: lanes d_v, columns j    (64)
constexpr uint32_t TM_O = 192;   // O^T: lanes d_v, columns i               (64)
constexpr uint32_t TM_KQ = 256;  // [K;Q] K^T, then W^T                     (64)
constexpr uint32_t TM_UH = 320;  // (U' diag(s))^T hi, packed bf16 pairs    (32)
constexpr uint32_t TM_UL = 352;  // (U' diag(s))^T lo                       (32)
constexpr uint32_t TM_UU = 384;  // U'^T as bf16                            (32)
constexpr uint32_t kTmemCols = 512;

// Barrier indices
enum {
  B_FULL0 = 0, B_FULL1, B_EMPTY0, B_EMPTY1, B_KQ_READY, B_KQ_DONE, B_P1_MID, B_W_DONE,
  B_P1_DONE0, B_P1_DONE1, B_BUF_FREE0, B_BUF_FREE1, B_S_READY, B_UP_DONE, B_UOPS_READY,
  B_O_DONE, B_DRAIN1, B_DRAIN2, kNumBars
};

// Per-chunk scalars shared by WG-A (writer) and WG-B (reader).
struct ChunkScalars {
  float rk[64], rq[64], G[64], beta[64], eG[64], s[64], tw[64];
  float eGC;
  int pad[15];
};

// Shared-memory layout, byte offsets from a 1024-aligned base.
template <int DK, int DV>
struct TcLayout {
  static constexpr int NKA = DK / 64;  // 64-element atom columns of K / Q
  static constexpr int NVA = DV / 64;
  static constexpr uint32_t KQ_BYTES = NKA * 16384u;  // [K ac][Q ac] per atom column
  static constexpr uint32_t V_BYTES = NVA * 8192u;
  static constexpr uint32_t GATE_BYTES = 1024u;  // G[64], beta[64] fp32
  static constexpr uint32_t STAGE_BYTES = KQ_BYTES + V_BYTES + GATE_BYTES;
  static constexpr uint32_t STAGE0 = 0;
  static constexpr uint32_t P0 = 2 * STAGE_BYTES;         // P (bf16 64x64) x2
  static constexpr uint32_t TB0 = P0 + 2 * 8192u;         // T_b hi/lo (or fp32 T) x2
  static constexpr uint32_t TW = TB0 + 2 * 16384u;        // T_w bf16
  static constexpr uint32_t WT0 = TW + 8192u;             // W^T bf16 128x64 (or fp32 A) x2
  static constexpr uint32_t SOP = WT0 + 2 * 16384u;       // -S^T bf16 [128][DK]
  static constexpr uint32_t SOP_BYTES = NKA * 16384u;
  static constexpr bool NEED_ZERO = (DK == 64) || (DV == 64);
  static constexpr uint32_t ZERO = SOP + SOP_BYTES;       // 8 KB of zeros (M padding)
  static constexpr uint32_t SC0 = ZERO + (NEED_ZERO ? 8192u : 0u);
  static constexpr uint32_t BARS = SC0 + 2 * (uint32_t)sizeof(ChunkScalars);
  static constexpr uint32_t MISC = BARS + kNumBars * 8u;  // tmem base, abort flag
  static constexpr uint32_t TOTAL = MISC + 64u;
  static constexpr uint32_t DYN_SMEM = TOTAL + 1024u;     // alignment slack
  static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
  static_assert(DYN_SMEM <= 232448u, "shared memory budget");
};

struct Tmaps {
  CUtensorMap q, k, v;
};

// Swizzled fp32 64x64 scratch (A and T of the solve): element (r, c).
__device__ __forceinline__ int fidx(int r, int c) { return r * 64 + (c ^ (r & 31)); }

// ---------------------------------------------------------------- the solve
// T = (I + A)^-1 for the 64x64 strictly-lower A, by 16x16 blocks: invert the
// diagonal blocks by forward substitution, then T_ij = -D_i sum_{k=j}^{i-1}
// A_ik T_kj level by level. 128 threads (4 warps).
__device__ __forceinline__ void solve_unit_lower(const float* __restrict__ A, float* __restrict__ T,
                                                 int wa) {
  const int wq = wa >> 5, ln = wa & 31;
  // diagonal blocks: warp wq owns block wq, lane l < 16 owns column l
  {
    const int b = wq * 16;
    if (ln < 16) {
      const int l = ln;
      float t[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) t[i] = (i == l) ? 1.f : 0.f;
#pragma unroll
      for (int i = 1; i < 16; ++i) {
        float s = 0.f;
#pragma unroll
        for (int x = 0; x < i; ++x) s = fmaf(A[fidx(b + i, b + x)], t[x], s);
        if (i > l) t[i] = -s;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) T[fidx(b + i, b + l)] = t[i];
    }
  }
  named_bar_sync(1, 128);
  // level 1: T_{i,i-1}, warp wq -> block (wq+1, wq)
  if (wq < 3) {
    const int bi = (wq + 1) * 16, bj = wq * 16;
    const int r = ln >> 1, c0 = (ln & 1) * 8;
    float x[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float a = A[fidx(bi + r, bj + k)];
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = fmaf(a, T[fidx(bj + k, bj + c0 + e)], x[e]);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) T[fidx(bi + r, bj + c0 + e)] = x[e];
    __syncwarp();
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) y[e] = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float d = T[fidx(bi + r, bi + k)];
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = fmaf(d, T[fidx(bi + k, bj + c0 + e)], y[e]);
    }
    __syncwarp();
#pragma unroll
    for (int e = 0; e < 8; ++e) T[fidx(bi + r, bj + c0 + e)] = -y[e];
  }
  named_bar_sync(1, 128);
  // level 2: T_20 (warps 0, 1) and T_31 (warps 2, 3), 8 columns per warp
  {
    const int bi = (wq < 2 ? 2 : 3) * 16, bj = (wq < 2 ? 0 : 1) * 16;
    const int r = ln >> 1, c0 = (wq & 1) * 8 + (ln & 1) * 4;
    float x[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) {
      const int bk = bj + kb * 16;
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float a = A[fidx(bi + r, bk + k)];
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = fmaf(a, T[fidx(bk + k, bj + c0 + e)], x[e]);
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) T[fidx(bi + r, bj + c0 + e)] = x[e];
    __syncwarp();
    float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float d = T[fidx(bi + r, bi + k)];
#pragma unroll
      for (int e = 0; e < 4; ++e) y[e] = fmaf(d, T[fidx(bi + k, bj + c0 + e)], y[e]);
    }
    __syncwarp();
#pragma unroll
    for (int e = 0; e < 4; ++e) T[fidx(bi + r, bj + c0 + e)] = -y[e];
  }
  named_bar_sync(1, 128);
  // level 3: T_30, 4 columns per warp
  {
    const int bi = 48;
    const int r = ln >> 1, c0 = wq * 4 + (ln & 1) * 2;
    float x[2] = {0.f, 0.f};
#pragma unroll
    for (int kb = 0; kb < 3; ++kb) {
      const int bk = kb * 16;
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float a = A[fidx(bi + r, bk + k)];
#pragma unroll
        for (int e = 0; e < 2; ++e) x[e] = fmaf(a, T[fidx(bk + k, c0 + e)], x[e]);
      }
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) T[fidx(bi + r, c0 + e)] = x[e];
    __syncwarp();
    float y[2] = {0.f, 0.f};
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float d = T[fidx(bi + r, bi + k)];
#pragma unroll
      for (int e = 0; e < 2; ++e) y[e] = fmaf(d, T[fidx(bi + k, c0 + e)], y[e]);
    }
    __syncwarp();
#pragma unroll
    for (int e = 0; e < 2; ++e) T[fidx(bi + r, c0 + e)] = -y[e];
  }
  named_bar_sync(1, 128);
}

// ---------------------------------------------------------------- the kernel
template <int DK, int DV>
__global__ void __launch_bounds__(kTcThreads, 1)
    gdn_tc_kernel(const Params p, const __grid_constant__ Tmaps tm) {
  using L = TcLayout<DK, DV>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(sm);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BARS);
  uint32_t* tmem_base_ptr = reinterpret_cast<uint32_t*>(sm + L::MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::MISC + 4);
  ChunkScalars* scal = reinterpret_cast<ChunkScalars*>(sm + L::SC0);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int unit = blockIdx.x;
  const int n = p.order[unit / p.h_v];
  const int h = unit % p.h_v;
  if (n < 0 || n >= p.num_seqs) {  // never expected: the prep kernel writes a permutation
    if (tid == 0) report(p.status, GDN_ERR_SEQLENS, (uint32_t)unit);
    return;
  }
  const int hq = h / (p.h_v / p.h_qk);
  int64_t bos, eos;
  seq_bounds(p, n, bos, eos);
  const int nchunks = (int)((eos - bos + kChunk - 1) / kChunk);

  // ---- setup
  if (tid == 0) {
    for (int b = 0; b < kNumBars; ++b) {
      uint32_t cnt = 1;
      if (b == B_FULL0 || b == B_FULL1) cnt = 32;
      mbar_init(&bars[b], cnt);
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (L::NEED_ZERO) {
    for (int i = tid; i < 8192 / 16; i += kTcThreads) st_shared_v4(sbase + L::ZERO + i * 16, 0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm.q);
    tma_prefetch_desc(&tm.k);
    tma_prefetch_desc(&tm.v);
  }
  if (warp == 1) tmem_alloc(tmem_base_ptr, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_ptr;

  auto fail = [&](int where) {
    if (!*abort_flag) {
      *abort_flag = 1;
      report(p.status, GDN_ERR_DEVICE_TIMEOUT, (uint32_t)(unit * 16 + where));
    }
  };

  auto stage_kq = [&](int s) { return sbase + L::STAGE0 + (uint32_t)s * L::STAGE_BYTES; };
  auto stage_v = [&](int s) { return stage_kq(s) + L::KQ_BYTES; };
  auto stage_gates = [&](int s) {
    return reinterpret_cast<float*>(sm + L::STAGE0 + (uint32_t)s * L::STAGE_BYTES + L::KQ_BYTES +
                                    L::V_BYTES);
  };

  if (warp == 0) {
    // ================================================================ producer
    const uint32_t tx_bytes = (uint32_t)(2 * L::NKA + L::NVA) * 8192u;
    int issued[2] = {-1, -1};  // last chunk whose tiles were requested into each stage
    for (int c = 0; c < nchunks; ++c) {
      const int s = c & 1;
      if (c >= 2 && !mbar_wait(&bars[B_EMPTY0 + s], ((c >> 1) + 1) & 1, abort_flag, kWaitLimitNs)) {
        fail(0);
        break;
      }
      const int64_t t0 = bos + (int64_t)c * kChunk;
      const int m = (int)((eos - t0) < kChunk ? (eos - t0) : kChunk);
      if (lane == 0) {
        mbar_expect_tx(&bars[B_FULL0 + s], tx_bytes);
        uint8_t* kq = sm + L::STAGE0 + s * L::STAGE_BYTES;
        for (int a = 0; a < L::NKA; ++a) {
          tma_load_3d(kq + a * 16384, &tm.k, &bars[B_FULL0 + s], 64 * a, hq, (int)t0);
          tma_load_3d(kq + a * 16384 + 8192, &tm.q, &bars[B_FULL0 + s], 64 * a, hq, (int)t0);
        }
        for (int a = 0; a < L::NVA; ++a)
          tma_load_3d(kq + L::KQ_BYTES + a * 8192, &tm.v, &bars[B_FULL0 + s], 64 * a, h, (int)t0);
      }
      issued[s] = c;
      // gates: rows lane and lane + 32, masked past the sequence end
      float g0 = 0.f, g1 = 0.f, b0 = 0.f, b1 = 0.f;
      if (lane < m) {
        g0 = load_gate(p.g, (t0 + lane) * p.h_v + h, p.gate_f32);
        b0 = load_gate(p.beta, (t0 + lane) * p.h_v + h, p.gate_f32);
      }
      if (lane + 32 < m) {
        g1 = load_gate(p.g, (t0 + lane + 32) * p.h_v + h, p.gate_f32);
        b1 = load_gate(p.beta, (t0 + lane + 32) * p.h_v + h, p.gate_f32);
      }
      float c0v = g0, c1v = g1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float u0 = __shfl_up_sync(0xffffffffu, c0v, o);
        const float u1 = __shfl_up_sync(0xffffffffu, c1v, o);
        if (lane >= o) {
          c0v += u0;
          c1v += u1;
        }
      }
      c1v += __shfl_sync(0xffffffffu, c0v, 31);
      float* gt = stage_gates(s);
      gt[lane] = c0v;
      gt[lane + 32] = c1v;
      gt[64 + lane] = b0;
      gt[64 + lane + 32] = b1;
      mbar_arrive(&bars[B_FULL0 + s]);
    }
    // on abort, let the loads already issued land before the CTA can exit
    // (in the normal path their stages were consumed and these return at once)
    if (*abort_flag) {
      for (int s = 0; s < 2; ++s)
        if (issued[s] >= 0) mbar_wait(&bars[B_FULL0 + s], (issued[s] >> 1) & 1, nullptr, 100000000ull);
    }
  } else if (warp == 1) {
    // ================================================================ state-independent MMAs
    if (lane == 0) {
      constexpr uint32_t id_kq = idesc_bf16(128, 64, 0, 0);
      constexpr uint32_t id_w = idesc_bf16(128, 64, 1, 0);
      for (int c = 0; c < nchunks; ++c) {
        const int s = c & 1;
        if (!mbar_wait(&bars[B_KQ_READY], c & 1, abort_flag, kWaitLimitNs)) {
          fail(1);
          break;
        }
        tc_fence_after();
        const uint32_t kq = stage_kq(s);
        // [K;Q] K^T : A = rows of K then Q (K-major), B = K (K-major, N = 64)
#pragma unroll
        for (int a = 0; a < L::NKA; ++a)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t off = a * 16384u + k * 32u;
            mma_ss(tmem + TM_KQ, sdesc(kq + off, 16, 1024), sdesc(kq + off, 16, 1024), id_kq,
                   (a | k) != 0);
          }
        mma_commit(&bars[B_KQ_DONE]);
        if (!mbar_wait(&bars[B_P1_MID], c & 1, abort_flag, kWaitLimitNs)) {
          fail(2);
          break;
        }
        tc_fence_after();
        // W^T = K^T T_w^T : A = K^T (MN-major, d_k atoms 16 KB apart or the zero page)
        const uint32_t lbo_k = (L::NKA == 2) ? 16384u : (sbase + L::ZERO - kq);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ss(tmem + TM_KQ, sdesc(kq + k * 2048u, lbo_k, 1024),
                 sdesc(sbase + L::TW + k * 32u, 16, 1024), id_w, k != 0);
        mma_commit(&bars[B_W_DONE]);
      }
      mma_commit(&bars[B_DRAIN1]);  // every MMA this thread issued has finished before exit
      mbar_wait(&bars[B_DRAIN1], 0, nullptr, 100000000ull);
    }
  } else if (warp == 2) {
    // ================================================================ state-dependent MMAs
    if (lane == 0) {
      constexpr uint32_t id_u = idesc_bf16(128, 64, 1, 0);
      constexpr uint32_t id_sw = idesc_bf16(128, 64, 0, 1);
      constexpr uint32_t id_qs = idesc_bf16(128, 64, 0, 0);
      constexpr uint32_t id_st = idesc_bf16(128, DK, 0, 1);
      constexpr uint32_t id_pu = idesc_bf16(128, 64, 0, 0);
      for (int c = 0; c < nchunks; ++c) {
        const int s = c & 1, par = c & 1;
        if (!mbar_wait(&bars[B_P1_DONE0 + par], (c >> 1) & 1, abort_flag, kWaitLimitNs) ||
            !mbar_wait(&bars[B_S_READY], c & 1, abort_flag, kWaitLimitNs)) {
          fail(3);
          break;
        }
        tc_fence_after();
        const uint32_t kq = stage_kq(s), vv = stage_v(s);
        const uint32_t tb = sbase + L::TB0 + par * 16384u;
        const uint32_t wt = sbase + L::WT0 + par * 16384u;
        const uint32_t sop = sbase + L::SOP;
        // U^T = V^T (T_b hi + lo)^T : A = V^T MN-major (d_v atoms 8 KB apart or the zero page)
        const uint32_t lbo_v = (L::NVA == 2) ? 8192u : (sbase + L::ZERO - vv);
#pragma unroll
        for (int half = 0; half < 2; ++half)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(tmem + TM_R, sdesc(vv + k * 2048u, lbo_v, 1024),
                   sdesc(tb + half * 8192u + k * 32u, 16, 1024), id_u, (half | k) != 0);
        // U'^T += (-S^T) W^T : A = -S^T K-major, B = W^T MN-major [d_k][j]
#pragma unroll
        for (int a = 0; a < L::NKA; ++a)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(tmem + TM_R, sdesc(sop + a * 16384u + k * 32u, 16, 1024),
                   sdesc(wt + (a * 4 + k) * 2048u, 16, 1024), id_sw, 1);
        // O^T = (-S^T) (-Qh)^T : B = Qh in place of Q (K-major)
#pragma unroll
        for (int a = 0; a < L::NKA; ++a)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(tmem + TM_O, sdesc(sop + a * 16384u + k * 32u, 16, 1024),
                   sdesc(kq + a * 16384u + 8192u + k * 32u, 16, 1024), id_qs, (a | k) != 0);
        mma_commit(&bars[B_UP_DONE]);
        if (!mbar_wait(&bars[B_UOPS_READY], c & 1, abort_flag, kWaitLimitNs)) {
          fail(4);
          break;
        }
        tc_fence_after();
        // S^T += (U' diag(s))^T K : A from TMEM (hi, then lo), B = K MN-major (N = d_k)
        const uint32_t lbo_kn = (L::NKA == 2) ? 16384u : 16u;
#pragma unroll
        for (int half = 0; half < 2; ++half)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ts(tmem + TM_S, tmem + (half ? TM_UL : TM_UH) + k * 8u,
                   sdesc(kq + k * 2048u, lbo_kn, 1024), id_st, 1);
        // O^T += U'^T P^T : A from TMEM (bf16 U'), B = P K-major [i][j]
        const uint32_t pp = sbase + L::P0 + par * 8192u;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ts(tmem + TM_O, tmem + TM_UU + k * 8u, sdesc(pp + k * 32u, 16, 1024), id_pu, 1);
        mma_commit(&bars[B_O_DONE]);
        mma_commit(&bars[B_EMPTY0 + s]);
      }
      mma_commit(&bars[B_DRAIN2]);
      mbar_wait(&bars[B_DRAIN2], 0, nullptr, 100000000ull);
    }
  } else if (warp >= 4 && warp < 8) {
    // ================================================================ WG-A: chunk preparation
    const int wa = tid - 128;  // == TMEM lane
    const uint32_t lane_off = (uint32_t)((wa & ~31) << 16);
    for (int c = 0; c < nchunks; ++c) {
      const int s = c & 1, par = c & 1;
      bool ok = mbar_wait(&bars[B_FULL0 + s], (c >> 1) & 1, abort_flag, kWaitLimitNs);
      if (ok && c >= 2)
        ok = mbar_wait(&bars[B_BUF_FREE0 + par], ((c >> 1) + 1) & 1, abort_flag, kWaitLimitNs);
      if (!ok) fail(5);
      named_bar_sync(1, 128);
      if (*abort_flag) break;
      const int64_t t0 = bos + (int64_t)c * kChunk;
      const int m = (int)((eos - t0) < kChunk ? (eos - t0) : kChunk);
      const uint32_t kq = stage_kq(s), vv = stage_v(s);
      const float* gt = stage_gates(s);
      ChunkScalars& sc = scal[par];
      // rows past the sequence end belong to another sequence (or are TMA zero
      // fill): clear them so that only exact zeros enter the products
      if (m < kChunk) {
        const int rows = kChunk - m;
        const int per_row = 8;  // 16-byte chunks in a 128-byte row
        const int nreg = 2 * L::NKA + L::NVA;
        for (int idx = wa; idx < rows * per_row * nreg; idx += 128) {
          const int reg = idx / (rows * per_row), rem = idx % (rows * per_row);
          const int r = m + rem / per_row, ch = rem % per_row;
          uint32_t base;
          if (reg < 2 * L::NKA)
            base = kq + (reg >> 1) * 16384u + (reg & 1) * 8192u;
          else
            base = vv + (reg - 2 * L::NKA) * 8192u;
          st_shared_v4(base + r * 128u + ch * 16u, 0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
      }
      // L2-norm scales: thread wa < 64 -> k row wa, else q row wa - 64
      {
        const int row = wa & 63;
        const uint32_t rbase = kq + (wa >= 64 ? 8192u : 0u) + row * 128u;
        float ss = 0.f;
#pragma unroll
        for (int a = 0; a < L::NKA; ++a)
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            uint32_t x0, x1, x2, x3;
            ld_shared_v4(rbase + a * 16384u + ch * 16u, x0, x1, x2, x3);
            const uint32_t xs[4] = {x0, x1, x2, x3};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float lo = bf16_lo_f(xs[e]), hi = bf16_hi_f(xs[e]);
              ss = fmaf(lo, lo, ss);
              ss = fmaf(hi, hi, ss);
            }
          }
        const float r = p.l2norm ? 1.0f / sqrtf(ss + 1e-6f) : 1.0f;
        if (wa < 64)
          sc.rk[row] = r;
        else
          sc.rq[row] = r;
      }
      named_bar_sync(1, 128);
      if (wa < 64) {
        const int j = wa;
        const float G = gt[j], GC = gt[63], bj = gt[64 + j];
        const float eg = expf(G);
        sc.G[j] = G;
        sc.beta[j] = bj;
        sc.eG[j] = eg;
        sc.s[j] = expf(GC - G) * sc.rk[j];
        sc.tw[j] = bj * eg * sc.rk[j];
        if (j == 0) sc.eGC = expf(GC);
      }
      named_bar_sync(1, 128);
      if (wa == 0) mbar_arrive(&bars[B_KQ_READY]);
      // ---- A and P from [K;Q] K^T
      ok = mbar_wait(&bars[B_KQ_DONE], c & 1, abort_flag, kWaitLimitNs);
      if (!ok) fail(6);
      named_bar_sync(1, 128);
      if (*abort_flag) break;
      tc_fence_after();
      float* Abuf = reinterpret_cast<float*>(sm + L::WT0 + par * 16384u);
      float* Tbuf = reinterpret_cast<float*>(sm + L::TB0 + par * 16384u);
      {
        uint32_t v0[32], v1[32];
        tmem_ld32(tmem + lane_off + TM_KQ, v0);
        tmem_ld32(tmem + lane_off + TM_KQ + 32, v1);
        tmem_ld_wait();
        if (wa < 64) {
          const int i = wa;
          const float ci = sc.beta[i] * sc.rk[i], Gi = sc.G[i];
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const float kk = __uint_as_float(j < 32 ? v0[j] : v1[j - 32]);
            Abuf[fidx(i, j)] = (j < i) ? ci * sc.rk[j] * expf(Gi - sc.G[j]) * kk : 0.f;
          }
        } else {
          const int i = wa - 64;
          const float Gi = sc.G[i];
          const uint32_t prow = sbase + L::P0 + par * 8192u;
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float pv[2];
#pragma unroll
              for (int q = 0; q < 2; ++q) {
                const int j = ch * 8 + e * 2 + q;
                const float qk = __uint_as_float(j < 32 ? v0[j] : v1[j - 32]);
                pv[q] = (j <= i) ? expf(Gi - sc.G[j]) * sc.rk[j] * qk : 0.f;
              }
              w4[e] = pack_bf16(pv[0], pv[1]);
            }
            st_shared_v4(prow + sw128(i, ch), w4[0], w4[1], w4[2], w4[3]);
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(1, 128);
      // ---- T = (I + A)^-1
      solve_unit_lower(Abuf, Tbuf, wa);
      // ---- T_b = T diag(beta) as bf16 hi + lo; T_w = T diag(beta e^G r^k)
      {
        const int i = wa >> 1, hh = wa & 1;
        float t[32];
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const int j = hh * 32 + jj;
          t[jj] = ((j >> 4) > (i >> 4)) ? 0.f : Tbuf[fidx(i, j)];
        }
        named_bar_sync(1, 128);  // every thread has read T before it is overwritten
        const uint32_t tb = sbase + L::TB0 + par * 16384u;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t hi4[4], lo4[4], w4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j0 = hh * 32 + q * 8 + e * 2;
            const float x0 = t[q * 8 + e * 2] * sc.beta[j0];
            const float x1 = t[q * 8 + e * 2 + 1] * sc.beta[j0 + 1];
            hi4[e] = pack_bf16(x0, x1);
            lo4[e] = pack_bf16(x0 - bf16_lo_f(hi4[e]), x1 - bf16_hi_f(hi4[e]));
            w4[e] = pack_bf16(t[q * 8 + e * 2] * sc.tw[j0], t[q * 8 + e * 2 + 1] * sc.tw[j0 + 1]);
          }
          const uint32_t off = sw128(i, hh * 4 + q);
          st_shared_v4(tb + off, hi4[0], hi4[1], hi4[2], hi4[3]);
          st_shared_v4(tb + 8192u + off, lo4[0], lo4[1], lo4[2], lo4[3]);
          st_shared_v4(sbase + L::TW + off, w4[0], w4[1], w4[2], w4[3]);
        }
      }
      // ---- Qh = -e^{G_i} q_i, in place over the q tile (row-wise scale ignores the swizzle)
      {
        const int row = wa >> 1;
        const float f = -sc.eG[row];
        for (int idx = (wa & 1); idx < 8 * L::NKA; idx += 2) {
          const int a = idx >> 3, ch = idx & 7;
          const uint32_t addr = kq + a * 16384u + 8192u + row * 128u + ch * 16u;
          uint32_t x[4];
          ld_shared_v4(addr, x[0], x[1], x[2], x[3]);
#pragma unroll
          for (int e = 0; e < 4; ++e) x[e] = pack_bf16(bf16_lo_f(x[e]) * f, bf16_hi_f(x[e]) * f);
          st_shared_v4(addr, x[0], x[1], x[2], x[3]);
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (wa == 0) mbar_arrive(&bars[B_P1_MID]);
      // ---- W^T: TMEM -> bf16 MN-major [d_k][j]
      ok = mbar_wait(&bars[B_W_DONE], c & 1, abort_flag, kWaitLimitNs);
      if (!ok) fail(7);
      named_bar_sync(1, 128);
      if (*abort_flag) break;
      tc_fence_after();
      {
        uint32_t v0[32], v1[32];
        tmem_ld32(tmem + lane_off + TM_KQ, v0);
        tmem_ld32(tmem + lane_off + TM_KQ + 32, v1);
        tmem_ld_wait();
        const uint32_t wt = sbase + L::WT0 + par * 16384u;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          uint32_t w4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = ch * 8 + e * 2;
            const float a0 = __uint_as_float(j < 32 ? v0[j] : v1[j - 32]);
            const float a1 = __uint_as_float(j + 1 < 32 ? v0[j + 1] : v1[j + 1 - 32]);
            w4[e] = pack_bf16(a0, a1);
          }
          st_shared_v4(wt + sw128(wa, ch), w4[0], w4[1], w4[2], w4[3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(1, 128);
      if (wa == 0) mbar_arrive(&bars[B_P1_DONE0 + par]);
    }
  } else if (warp >= 8) {
    // ================================================================ WG-B: state step + epilogue
    const int wb = tid - 256;  // == TMEM lane == d_v index
    const uint32_t lane_off = (uint32_t)((wb & ~31) << 16);
    const bool live = wb < DV;
    // initial state -> S^T in TMEM (lane d_v, column d_k)
    {
      const int64_t slot = state_slot(p, n);
      const float* s0 = slot >= 0 ? p.initial_state + ((size_t)slot * p.h_v + h) * DK * DV : nullptr;
#pragma unroll
      for (int xb = 0; xb < DK / 32; ++xb) {
        uint32_t v[32];
#pragma unroll
        for (int x = 0; x < 32; ++x)
          v[x] = (s0 && live) ? __float_as_uint(s0[(size_t)(xb * 32 + x) * DV + wb]) : 0u;
        tmem_st32(tmem + lane_off + TM_S + xb * 32, v);
      }
      tmem_st_wait();
    }
    for (int c = 0; c < nchunks; ++c) {
      const int par = c & 1;
      // ---- S -> -S^T (bf16 operand); S *= e^{G_m}
      bool ok = mbar_wait(&bars[B_P1_DONE0 + par], (c >> 1) & 1, abort_flag, kWaitLimitNs);
      if (!ok) fail(8);
      named_bar_sync(2, 128);
      if (*abort_flag) break;
      tc_fence_after();
      const ChunkScalars& sc = scal[par];
      const float eGC = sc.eGC;
#pragma unroll
      for (int xb = 0; xb < DK / 32; ++xb) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + TM_S + xb * 32, v);
        tmem_ld_wait();
        const uint32_t row = sbase + L::SOP + (xb >> 1) * 16384u;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t w4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w4[e] = pack_bf16(-__uint_as_float(v[q * 8 + e * 2]), -__uint_as_float(v[q * 8 + e * 2 + 1]));
          st_shared_v4(row + sw128(wb, (xb & 1) * 4 + q), w4[0], w4[1], w4[2], w4[3]);
        }
#pragma unroll
        for (int x = 0; x < 32; ++x) v[x] = __float_as_uint(__uint_as_float(v[x]) * eGC);
        tmem_st32(tmem + lane_off + TM_S + xb * 32, v);
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(2, 128);
      if (wb == 0) mbar_arrive(&bars[B_S_READY]);
      // ---- U' -> (U' s) hi / lo and U' as bf16, into TMEM A operands
      ok = mbar_wait(&bars[B_UP_DONE], c & 1, abort_flag, kWaitLimitNs);
      if (!ok) fail(9);
      named_bar_sync(2, 128);
      if (*abort_flag) break;
      tc_fence_after();
      {
        uint32_t u0[32], u1[32];
        tmem_ld32(tmem + lane_off + TM_R, u0);
        tmem_ld32(tmem + lane_off + TM_R + 32, u1);
        tmem_ld_wait();
        uint32_t w[32];
#pragma unroll
        for (int pass = 0; pass < 3; ++pass) {
#pragma unroll
          for (int cc = 0; cc < 32; ++cc) {
            const int j = 2 * cc;
            const float a0 = __uint_as_float(j < 32 ? u0[j] : u1[j - 32]);
            const float a1 = __uint_as_float(j + 1 < 32 ? u0[j + 1] : u1[j + 1 - 32]);
            if (pass == 2) {
              w[cc] = pack_bf16(a0, a1);
            } else {
              const float x0 = a0 * sc.s[j], x1 = a1 * sc.s[j + 1];
              const uint32_t hi = pack_bf16(x0, x1);
              w[cc] = pass == 0 ? hi : pack_bf16(x0 - bf16_lo_f(hi), x1 - bf16_hi_f(hi));
            }
          }
          tmem_st32(tmem + lane_off + (pass == 0 ? TM_UH : pass == 1 ? TM_UL : TM_UU), w);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      named_bar_sync(2, 128);
      if (wb == 0) mbar_arrive(&bars[B_UOPS_READY]);
      // ---- epilogue: o_i = scale r^q_i O^T[:, i]
      ok = mbar_wait(&bars[B_O_DONE], c & 1, abort_flag, kWaitLimitNs);
      if (!ok) fail(10);
      named_bar_sync(2, 128);
      if (*abort_flag) break;
      tc_fence_after();
      {
        const int64_t t0 = bos + (int64_t)c * kChunk;
        const int m = (int)((eos - t0) < kChunk ? (eos - t0) : kChunk);
        uint32_t o0[32], o1[32];
        tmem_ld32(tmem + lane_off + TM_O, o0);
        tmem_ld32(tmem + lane_off + TM_O + 32, o1);
        tmem_ld_wait();
        if (live) {
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            if (i < m) {
              const float o = p.scale * sc.rq[i] * __uint_as_float(i < 32 ? o0[i] : o1[i - 32]);
              const size_t idx = ((size_t)(t0 + i) * p.h_v + h) * DV + wb;
              if (p.out_f32)
                reinterpret_cast<float*>(p.out)[idx] = o;
              else
                reinterpret_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(o);
            }
          }
        }
      }
      tc_fence_before();
      named_bar_sync(2, 128);
      if (wb == 0) mbar_arrive(&bars[B_BUF_FREE0 + par]);
    }
    // final state
    if (!*abort_flag && p.final_state) {
      tc_fence_after();
      float* fs = p.final_state + ((size_t)n * p.h_v + h) * DK * DV;
#pragma unroll
      for (int xb = 0; xb < DK / 32; ++xb) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + TM_S + xb * 32, v);
        tmem_ld_wait();
        if (live) {
#pragma unroll
          for (int x = 0; x < 32; ++x) fs[(size_t)(xb * 32 + x) * DV + wb] = __uint_as_float(v[x]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                        &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// [T, H, D] bf16 viewed as a 3-D tensor (D innermost); box = 64 elements x 1 head x 64 rows.
bool encode_rows(CUtensorMap* m, const void* base, int64_t T, int H, int D) {
  auto fn = get_encode();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int DK, int DV>
cudaError_t launch_tc_dk(const Params& p, cudaStream_t stream) {
  using L = TcLayout<DK, DV>;
  Tmaps tm;
  if (!encode_rows(&tm.q, p.q, p.total_tokens, p.h_qk, DK) ||
      !encode_rows(&tm.k, p.k, p.total_tokens, p.h_qk, DK) ||
      !encode_rows(&tm.v, p.v, p.total_tokens, p.h_v, DV))
    return cudaErrorInvalidValue;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(&gdn_tc_kernel<DK, DV>), (int)L::DYN_SMEM);
  if (e != cudaSuccess) return e;
  const long long units = (long long)p.num_seqs * p.h_v;
  if (units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  gdn_tc_kernel<DK, DV><<<(unsigned)units, kTcThreads, L::DYN_SMEM, stream>>>(p, tm);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc(const Params& p, cudaStream_t stream) {
  if (p.total_tokens <= 0) return launch_simt(p, stream);  // only empty sequences: state copy
  if (p.total_tokens > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (p.d_k == 128 && p.d_v == 128) return launch_tc_dk<128, 128>(p, stream);
  if (p.d_k == 64 && p.d_v == 64) return launch_tc_dk<64, 64>(p, stream);
  if (p.d_k == 128 && p.d_v == 64) return launch_tc_dk<128, 64>(p, stream);
  return launch_tc_dk<64, 128>(p, stream);
}

}  // namespace gdn
