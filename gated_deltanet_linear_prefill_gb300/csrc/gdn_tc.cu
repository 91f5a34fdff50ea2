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
//   QS^T = -S^T Q^T                 (the inter-chunk term, weighted by e^{G_i} at the end)
//   O^T  = U'^T P^T                 (P_ij = e^{G_i-G_j} r^k_j q_i.k_j, j <= i)
//   S^T += (U' diag(s))^T K         (s_j = e^{G_m-G_j} r^k_j; U' diag(s) as bf16 hi + lo,
//                                    read by the MMA straight from TMEM)
// Operand precision: the products feeding the fp32 state carry T and U' as
// bf16 hi + lo pairs (about 16 significant bits); S and W enter as bf16; every
// accumulation is fp32 in TMEM. Decays, norms and the 64x64 unit-lower-
// triangular inverse (16x16 blocks merged level by level, the blocked order
// the open-jev-fast README's GDN kernel also uses) run on CUDA cores in fp32.
//
// Warp roles (512 threads): warp 0 loads K/Q/V tiles by TMA (128-byte swizzle),
// clears rows past the sequence end and scans the gates; warp 1 allocates TMEM and issues the state-independent MMAs;
// warp 2 issues the state-dependent MMAs; warps 4-11 (WG-A) prepare chunk c+1
// (norms, A and P, the solve, T_b / T_w, W^T) while warps 12-15 (WG-B) run
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

constexpr int kTcThreads = 512;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait: far above any legal wait

// TMEM columns (fp32 unless noted)
constexpr uint32_t TM_S = 0;     // S^T: lanes d_v, columns d_k            (128)
constexpr uint32_t TM_R = 128;   // U^T, then U'^T: lanes d_v, columns j    (64)
constexpr uint32_t TM_O = 192;   // O^T: lanes d_v, columns i               (64)
constexpr uint32_t TM_KQ = 256;  // [K;Q] K^T, then W^T                     (64)
constexpr uint32_t TM_UH = 320;  // (U' diag(s))^T hi, packed bf16 pairs    (32)
constexpr uint32_t TM_UL = 352;  // (U' diag(s))^T lo                       (32)
constexpr uint32_t TM_UU = 384;  // U'^T as bf16                            (32)
constexpr uint32_t TM_QS = 448;  // -S^T Q^T: lanes d_v, columns i          (64)
constexpr uint32_t kTmemCols = 512;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kMaxDecaySpan = 80.0f;  // chunks whose log-decay spans more use exact exps

// Barrier indices
enum {
  B_TMA0 = 0, B_TMA1, B_READY0, B_READY1, B_EMPTY0, B_EMPTY1, B_KQ_DONE, B_P1_MID, B_W_DONE,
  B_KQ_FREE, B_P1_DONE0, B_P1_DONE1, B_CS_FREE0, B_CS_FREE1, B_CS_FREE2, B_S_READY, B_UP_DONE,
  B_UOPS_READY, B_O_DONE, B_STATE_DONE, B_EPI_DONE, B_DRAIN1, B_DRAIN2, kNumBars
};

// Per-chunk values WG-A hands to WG-B (three buffers, indexed by chunk % 3).
struct ChunkScalars {
  float cq[64];  // -scale r^q_i e^{G_i}: weight of the (-S^T q_i) column
  float co[64];  // scale r^q_i: weight of the intra-chunk column
  float s[64];   // e^{G_m - G_j} r^k_j: state-update weight of row j
  float eGC;     // e^{G_m}: decay of the whole chunk
  int pad[31];
};
// WG-A private per-chunk values.
struct PrepScalars {
  float d[64];     // r^k_j e^{Gmax - G_j}
  float r[64];     // r^k_j
  float tw[64];    // beta_j e^{G_j} r^k_j: column scale of T_w
  float beta[64];
};
// Stage scalars: G[64], beta[64], Gmax, Gmin written by the producer; WG-A
// parks half-row partial sums of |q_i|^2 in [SC_QSS, SC_QSS + 64).
constexpr int SC_G = 0, SC_B = 64, SC_QSS = 128, SC_GMAX = 192, SC_GMIN = 193;

constexpr int LDF = 68;  // row stride (floats) of the fp32 64x64 scratch of the solve

// Shared-memory layout, byte offsets from a 1024-aligned base.
template <int DK, int DV>
struct TcLayout {
  static constexpr int NKA = DK / 64;  // 64-element atom columns of K / Q
  static constexpr int NVA = DV / 64;
  static constexpr uint32_t KQ_BYTES = NKA * 16384u;  // [K ac][Q ac] per atom column
  static constexpr uint32_t V_BYTES = NVA * 8192u;
  static constexpr uint32_t SCAL_BYTES = 1024u;
  static constexpr uint32_t STAGE_BYTES = KQ_BYTES + V_BYTES + SCAL_BYTES;
  static constexpr uint32_t STAGE0 = 0;
  static constexpr uint32_t SCR_BYTES = 17408u;           // 64 x 68 fp32, 1024-aligned size
  static constexpr uint32_t P0 = 2 * STAGE_BYTES;         // P (bf16 64x64) x2
  static constexpr uint32_t TB0 = P0 + 2 * 8192u;         // T_b hi/lo (or fp32 T) x2
  static constexpr uint32_t TW = TB0 + 2 * SCR_BYTES;     // T_w bf16
  static constexpr uint32_t WT0 = TW + 8192u;             // W^T bf16 128x64 (or fp32 A) x2
  static constexpr uint32_t SOP = WT0 + 2 * SCR_BYTES;    // -S^T bf16 [128][DK]; output staging
  static constexpr uint32_t SOP_BYTES =
      (NKA * 16384u > 64u * DV * 4u) ? NKA * 16384u : 64u * DV * 4u;
  static constexpr bool NEED_ZERO = (DK == 64) || (DV == 64);
  static constexpr uint32_t ZERO = SOP + SOP_BYTES;       // 8 KB of zeros (M padding)
  static constexpr uint32_t CS0 = ZERO + (NEED_ZERO ? 8192u : 0u);
  static constexpr uint32_t PS = CS0 + 3 * (uint32_t)sizeof(ChunkScalars);
  static constexpr uint32_t BARS = PS + (uint32_t)sizeof(PrepScalars);
  static constexpr uint32_t MISC = BARS + kNumBars * 8u;  // tmem base, abort flag
  static constexpr uint32_t TOTAL = MISC + 64u;
  static constexpr uint32_t DYN_SMEM = TOTAL + 1024u;     // alignment slack
  static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
  static_assert(DYN_SMEM <= 232448u, "shared memory budget");
};

struct Tmaps {
  CUtensorMap q, k, v;
};

// Exact-decay fallback for a chunk whose log-decay spans more than
// kMaxDecaySpan (the factorised e^{G_i - G_j} = a_i b_j could leave fp32
// range): the 32 weights of one A row (krow) or P row, each decay by its own
// exp; the caller multiplies them by the K K^T / Q K^T entries. Kept out of
// line: it is rare and its code would crowd the hot loop. It sees only its
// own output array, so the caller's TMEM values stay in registers.
__device__ __noinline__ void exact_row(float* out, const float* r, const float* G, float Gl2i,
                                       float ci, int j0, int i, int krow) {
  for (int e = 0; e < 32; ++e) {
    const int j = j0 + e;
    const float x = r[j] * exp2f(Gl2i - G[j] * 1.4426950408889634f);
    out[e] = krow ? ((j < i) ? ci * x : 0.f) : ((j <= i) ? x : 0.f);
  }
}

// ---------------------------------------------------------------- the solve
// Warp-level tensor-core tiles for the block merges: mma.sync m16n8k8 with
// tf32 operands, each fp32 operand split as hi + lo (both tf32) and the
// product taken as hi*hi + hi*lo + lo*hi, which keeps close to fp32 accuracy.
// Fragment layout (lane = 4 g + t): A rows g, g+8 x columns t, t+4; B rows
// t, t+4 x column g; C rows g, g+8 x columns 2t, 2t+1.
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(hi) : "f"(x));
  const float r = x - __uint_as_float(hi);
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(lo) : "f"(r));
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// c[16 x 8] += X[xr.., xc + k) * Y[yr + k, yc..) over k in [0, 8 nk8), fp32 smem with row
// stride LDF.
__device__ __forceinline__ void mma_tile(const float* X, int xr, int xc, const float* Y, int yr,
                                         int yc, int nk8, float (&c)[4], int lane) {
  const int g = lane >> 2, t = lane & 3;
  const float* x0 = X + (xr + g) * LDF + xc + t;
  const float* x1 = x0 + 8 * LDF;
  const float* y0 = Y + (yr + t) * LDF + yc + g;
  for (int k = 0; k < nk8; ++k) {
    uint32_t ah[4], al[4], bh[2], bl[2];
    split_tf32(x0[8 * k], ah[0], al[0]);
    split_tf32(x1[8 * k], ah[1], al[1]);
    split_tf32(x0[8 * k + 4], ah[2], al[2]);
    split_tf32(x1[8 * k + 4], ah[3], al[3]);
    split_tf32(y0[8 * k * LDF], bh[0], bl[0]);
    split_tf32(y0[(8 * k + 4) * LDF], bh[1], bl[1]);
    mma_tf32(c, ah[0], ah[1], ah[2], ah[3], bh[0], bh[1]);
    mma_tf32(c, ah[0], ah[1], ah[2], ah[3], bl[0], bl[1]);
    mma_tf32(c, al[0], al[1], al[2], al[3], bh[0], bh[1]);
  }
}
__device__ __forceinline__ void store_tile(float* M, int r0, int c0, const float (&c)[4], float sgn,
                                           int lane) {
  const int g = lane >> 2, t = lane & 3;
  *reinterpret_cast<float2*>(&M[(r0 + g) * LDF + c0 + 2 * t]) = make_float2(sgn * c[0], sgn * c[1]);
  *reinterpret_cast<float2*>(&M[(r0 + g + 8) * LDF + c0 + 2 * t]) = make_float2(sgn * c[2], sgn * c[3]);
}

// T = (I + A)^-1 for the strictly-lower 64x64 A (fp32, stride LDF), in 16x16
// blocks (the blocked order of the open-jev-fast README's GDN kernel):
//  1. the four diagonal blocks D_b by forward substitution, one column per
//     lane, each row of A read as float4 broadcasts;
//  2. T_{b+1,b} = -D_{b+1} (A_{b+1,b} D_b) inside both 32x32 diagonal blocks;
//  3. T_21 = -T_22 (A_21 T_11) for the lower-left 32x32 block.
// Steps 2 and 3 run on the warp-level tensor cores (three-term tf32). Their
// intermediate products are parked in T's upper triangle, which nothing reads
// as T. Blocks above the diagonal are not otherwise written. 256 threads
// (8 warps); ends with every T entry visible to all of them.
__device__ __forceinline__ void solve_unit_lower(const float* __restrict__ A, float* __restrict__ T,
                                                 int wa) {
  const int wq = wa >> 5, ln = wa & 31;
  if (wq < 4 && ln < 16) {
    const int b = 16 * wq, l = ln;  // lane l owns column l of D_wq
    float t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float* row = A + (b + i) * LDF + b;
      float acc = (i == l) ? 1.f : 0.f;
#pragma unroll
      for (int x4 = 0; x4 < i; x4 += 4) {
        const float4 a4 = *reinterpret_cast<const float4*>(row + x4);
        acc = fmaf(-a4.x, t[x4], acc);
        if (x4 + 1 < i) acc = fmaf(-a4.y, t[x4 + 1], acc);
        if (x4 + 2 < i) acc = fmaf(-a4.z, t[x4 + 2], acc);
        if (x4 + 3 < i) acc = fmaf(-a4.w, t[x4 + 3], acc);
      }
      t[i] = acc;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) T[(b + i) * LDF + b + l] = t[i];
  }
  named_bar_sync(1, 256);
  // step 2: warp wq < 4 takes pair p = wq >> 1 (b = 32 p), columns 8 h of the 16-wide block
  const int h = wq & 1;
  if (wq < 4) {
    const int b = 32 * (wq >> 1);
    float c[4] = {};
    mma_tile(A, b + 16, b, T, b, b + 8 * h, 2, c, ln);  // A_{b+1,b} D_b
    store_tile(T, b, b + 16 + 8 * h, c, 1.f, ln);       // parked in block (b, b+1)
  }
  named_bar_sync(1, 256);
  if (wq < 4) {
    const int b = 32 * (wq >> 1);
    float c[4] = {};
    mma_tile(T, b + 16, b + 16, T, b, b + 16 + 8 * h, 2, c, ln);  // D_{b+1} X
    store_tile(T, b + 16, b + 8 * h, c, -1.f, ln);
  }
  named_bar_sync(1, 256);
  // step 3: warp wq -> output block (rb, cb) = (2 + (wq >> 2), (wq >> 1) & 1), columns 8 h
  const int rb = 2 + (wq >> 2), cb = (wq >> 1) & 1;
  {
    float c[4] = {};
    // X = A_{rb, cb..1} T_{cb..1, cb}  (T_11 is lower triangular)
    mma_tile(A, 16 * rb, 16 * cb, T, 16 * cb, 16 * cb + 8 * h, 2 * (2 - cb), c, ln);
    store_tile(T, 16 * (rb - 2), 32 + 16 * cb + 8 * h, c, 1.f, ln);  // parked in the upper right
  }
  named_bar_sync(1, 256);
  {
    float c[4] = {};
    // T_{rb,cb} = -T_{rb, 2..rb} X_{2..rb, cb}
    mma_tile(T, 16 * rb, 32, T, 0, 32 + 16 * cb + 8 * h, 2 * (rb - 1), c, ln);
    store_tile(T, 16 * rb, 16 * cb + 8 * h, c, -1.f, ln);
  }
  named_bar_sync(1, 256);
}

// ---------------------------------------------------------------- the kernel
template <int DK, int DV>
__global__ void __launch_bounds__(kTcThreads, 1)
    gdn_tc_kernel(const Params p, const __grid_constant__ Tmaps tm) {
  using L = TcLayout<DK, DV>;
  using L_ = L;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(sm);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BARS);
  uint32_t* tmem_base_ptr = reinterpret_cast<uint32_t*>(sm + L::MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::MISC + 4);
  ChunkScalars* cscal = reinterpret_cast<ChunkScalars*>(sm + L::CS0);
  PrepScalars* ps = reinterpret_cast<PrepScalars*>(sm + L::PS);

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
    for (int b = 0; b < kNumBars; ++b) mbar_init(&bars[b], (b == B_READY0 || b == B_READY1) ? 32u : 1u);
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
  auto stage_scal = [&](int s) {
    return reinterpret_cast<float*>(sm + L::STAGE0 + (uint32_t)s * L::STAGE_BYTES + L::KQ_BYTES +
                                    L::V_BYTES);
  };
  auto chunk_rows = [&](int c) {
    const int64_t t0 = bos + (int64_t)c * kChunk;
    return (int)((eos - t0) < kChunk ? (eos - t0) : kChunk);
  };

  if (warp == 0) {
    // ================================================================ producer
    // TMA tiles for chunk c+1 are requested before chunk c is finished here;
    // then chunk c's tail rows are cleared, its gates scanned and its q norms
    // taken, and the stage is published to WG-A and the MMA issuer.
    const uint32_t tx_bytes = (uint32_t)(2 * L::NKA + L::NVA) * 8192u;
    int issued[2] = {-1, -1};
    auto issue = [&](int c) {
      const int s = c & 1;
      const int t0 = (int)(bos + (int64_t)c * kChunk);
      uint8_t* kq = sm + L::STAGE0 + s * L::STAGE_BYTES;
      mbar_arrive_expect_tx(&bars[B_TMA0 + s], tx_bytes);
      for (int a = 0; a < L::NKA; ++a) {
        tma_load_3d(kq + a * 16384, &tm.k, &bars[B_TMA0 + s], 64 * a, hq, t0);
        tma_load_3d(kq + a * 16384 + 8192, &tm.q, &bars[B_TMA0 + s], 64 * a, hq, t0);
      }
      for (int a = 0; a < L::NVA; ++a)
        tma_load_3d(kq + L::KQ_BYTES + a * 8192, &tm.v, &bars[B_TMA0 + s], 64 * a, h, t0);
    };
    auto load_gates = [&](int c, float& g0, float& g1, float& b0, float& b1) {
      const int64_t t0 = bos + (int64_t)c * kChunk;
      const int m = chunk_rows(c);
      g0 = g1 = b0 = b1 = 0.f;
      if (lane < m) {
        g0 = load_gate(p.g, (t0 + lane) * p.h_v + h, p.gate_f32);
        b0 = load_gate(p.beta, (t0 + lane) * p.h_v + h, p.gate_f32);
      }
      if (lane + 32 < m) {
        g1 = load_gate(p.g, (t0 + lane + 32) * p.h_v + h, p.gate_f32);
        b1 = load_gate(p.beta, (t0 + lane + 32) * p.h_v + h, p.gate_f32);
      }
    };
    float g0 = 0.f, g1 = 0.f, b0 = 0.f, b1 = 0.f;
    if (nchunks > 0) {
      if (lane == 0) issue(0);
      issued[0] = 0;
      load_gates(0, g0, g1, b0, b1);
    }
    for (int c = 0; c < nchunks; ++c) {
      const int s = c & 1;
      if (!mbar_wait(&bars[B_TMA0 + s], (c >> 1) & 1, abort_flag, kWaitLimitNs)) {
        fail(1);
        break;
      }
      const int m = chunk_rows(c);
      const uint32_t kq = stage_kq(s), vv = stage_v(s);
      if (m < kChunk) {  // rows of the next sequence (or TMA zero fill): clear them
        const int rows = kChunk - m, nreg = 2 * L::NKA + L::NVA;
        for (int idx = lane; idx < rows * 8 * nreg; idx += 32) {
          const int reg = idx / (rows * 8), rem = idx % (rows * 8);
          const int r = m + (rem >> 3), ch = rem & 7;
          const uint32_t base = reg < 2 * L::NKA ? kq + (reg >> 1) * 16384u + (reg & 1) * 8192u
                                                 : vv + (reg - 2 * L::NKA) * 8192u;
          st_shared_v4(base + r * 128u + ch * 16u, 0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      // gate cumsum over the chunk and its span
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
      float gmax = fmaxf(c0v, c1v), gmin = fminf(c0v, c1v);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, o));
        gmin = fminf(gmin, __shfl_xor_sync(0xffffffffu, gmin, o));
      }
      float* sc = stage_scal(s);
      sc[SC_G + lane] = c0v;
      sc[SC_G + lane + 32] = c1v;
      sc[SC_B + lane] = b0;
      sc[SC_B + lane + 32] = b1;
      if (lane == 0) {
        sc[SC_GMAX] = gmax;
        sc[SC_GMIN] = gmin;
      }
      mbar_arrive(&bars[B_READY0 + s]);
      // next chunk: gates into registers, then its tiles once the stage is free
      if (c + 1 < nchunks) {
        load_gates(c + 1, g0, g1, b0, b1);
        const int s1 = (c + 1) & 1;
        if (c + 1 >= 2 &&
            !mbar_wait(&bars[B_EMPTY0 + s1], (((c + 1) >> 1) + 1) & 1, abort_flag, kWaitLimitNs)) {
          fail(0);
          break;
        }
        if (lane == 0) issue(c + 1);
        issued[s1] = c + 1;
      }
    }
    // on abort, let the loads already issued land before the CTA can exit
    // (in the normal path they were all consumed and these return at once)
    for (int s = 0; s < 2; ++s)
      if (issued[s] >= 0)
        mbar_wait(&bars[B_TMA0 + s], (issued[s] >> 1) & 1, nullptr, 100000000ull);
  } else if (warp == 1) {
    // ================================================================ state-independent MMAs
    if (lane == 0) {
      constexpr uint32_t id_kq = idesc_bf16(128, 64, 0, 0);
      constexpr uint32_t id_w = idesc_bf16(128, 64, 1, 0);
      for (int c = 0; c < nchunks; ++c) {
        const int s = c & 1;
        if (!mbar_wait(&bars[B_READY0 + s], (c >> 1) & 1, abort_flag, kWaitLimitNs) ||
            (c >= 1 && !mbar_wait(&bars[B_KQ_FREE], (c - 1) & 1, abort_flag, kWaitLimitNs))) {
          fail(2);
          break;
        }
        tc_fence_after();
        const uint32_t kq = stage_kq(s);
        // [K;Q] K^T : A = rows of K then Q (K-major), B = K (K-major, N = 64)
        const uint64_t dkq = sdesc(kq, 16, 1024);
#pragma unroll
        for (int a = 0; a < L::NKA; ++a)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t d = sdesc_add(dkq, a * 16384u + k * 32u);
            mma_ss(tmem + TM_KQ, d, d, id_kq, (a | k) != 0);
          }
        mma_commit(&bars[B_KQ_DONE]);
        if (!mbar_wait(&bars[B_P1_MID], c & 1, abort_flag, kWaitLimitNs)) {
          fail(3);
          break;
        }
        tc_fence_after();
        // W^T = K^T T_w^T : A = K^T (MN-major, d_k atoms 16 KB apart or the zero page)
        const uint32_t lbo_k = (L::NKA == 2) ? 16384u : (sbase + L::ZERO - kq);
        const uint64_t dka = sdesc(kq, lbo_k, 1024), dtw = sdesc(sbase + L::TW, 16, 1024);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ss(tmem + TM_KQ, sdesc_add(dka, k * 2048u), sdesc_add(dtw, k * 32u), id_w, k != 0);
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
        if (!mbar_wait(&bars[B_P1_DONE0 + par], (c >> 1) & 1, abort_flag, kWaitLimitNs)) {
          fail(4);
          break;
        }
        tc_fence_after();
        const uint32_t kq = stage_kq(s), vv = stage_v(s);
        const uint32_t tb = sbase + L::TB0 + par * L::SCR_BYTES;
        const uint32_t wt = sbase + L::WT0 + par * L::SCR_BYTES;
        const uint32_t sop = sbase + L::SOP;
        // U^T = V^T (T_b hi + lo)^T : A = V^T MN-major (d_v atoms 8 KB apart or the zero page).
        // State-independent: issued as soon as the chunk is prepared.
        const uint32_t lbo_v = (L::NVA == 2) ? 8192u : (sbase + L::ZERO - vv);
        const uint64_t dva = sdesc(vv, lbo_v, 1024), dtb = sdesc(tb, 16, 1024);
#pragma unroll
        for (int half = 0; half < 2; ++half)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(tmem + TM_R, sdesc_add(dva, k * 2048u), sdesc_add(dtb, half * 8192u + k * 32u), id_u,
                   (half | k) != 0);
        if (!mbar_wait(&bars[B_S_READY], c & 1, abort_flag, kWaitLimitNs)) {
          fail(5);
          break;
        }
        tc_fence_after();
        // U'^T += (-S^T) W^T : A = -S^T K-major, B = W^T MN-major [d_k][j]
        const uint64_t dsop = sdesc(sop, 16, 1024), dwt = sdesc(wt, 16, 1024);
#pragma unroll
        for (int a = 0; a < L::NKA; ++a)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(tmem + TM_R, sdesc_add(dsop, a * 16384u + k * 32u), sdesc_add(dwt, (a * 4 + k) * 2048u),
                   id_sw, 1);
        mma_commit(&bars[B_UP_DONE]);
        // QS^T = (-S^T) Q^T (raw q tile, K-major), once the last epilogue has read its block
        if (c >= 1 && !mbar_wait(&bars[B_EPI_DONE], (c - 1) & 1, abort_flag, kWaitLimitNs)) {
          fail(6);
          break;
        }
        tc_fence_after();
        const uint64_t dq = sdesc(kq + 8192u, 16, 1024);
#pragma unroll
        for (int a = 0; a < L::NKA; ++a)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(tmem + TM_QS, sdesc_add(dsop, a * 16384u + k * 32u), sdesc_add(dq, a * 16384u + k * 32u),
                   id_qs, (a | k) != 0);
        if (!mbar_wait(&bars[B_UOPS_READY], c & 1, abort_flag, kWaitLimitNs)) {
          fail(7);
          break;
        }
        tc_fence_after();
        // S^T += (U' diag(s))^T K : A from TMEM (hi, then lo), B = K MN-major (N = d_k)
        const uint32_t lbo_kn = (L::NKA == 2) ? 16384u : 16u;
        const uint64_t dkn = sdesc(kq, lbo_kn, 1024);
#pragma unroll
        for (int half = 0; half < 2; ++half)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ts(tmem + TM_S, tmem + (half ? TM_UL : TM_UH) + k * 8u, sdesc_add(dkn, k * 2048u), id_st, 1);
        mma_commit(&bars[B_STATE_DONE]);
        // O^T = U'^T P^T : A from TMEM (bf16 U'), B = P K-major [i][j]
        const uint64_t dpp = sdesc(sbase + L::P0 + par * 8192u, 16, 1024);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ts(tmem + TM_O, tmem + TM_UU + k * 8u, sdesc_add(dpp, k * 32u), id_pu, k != 0);
        mma_commit(&bars[B_O_DONE]);
        mma_commit(&bars[B_EMPTY0 + s]);
      }
      mma_commit(&bars[B_DRAIN2]);
      mbar_wait(&bars[B_DRAIN2], 0, nullptr, 100000000ull);
    }
  } else if (warp >= 4 && warp < 12) {
    // ================================================================ WG-A: chunk preparation
    const int wa = tid - 128;         // 0..255
    const int L = wa & 127;           // TMEM lane
    const int hf = wa >> 7;           // which 32-column half of a 64-wide block
    const uint32_t lane_off = (uint32_t)((L & ~31) << 16);
    const bool krow = L < 64;
    const int i = L & 63;
    for (int c = 0; c < nchunks; ++c) {
      const int s = c & 1, par = c & 1;
      bool ok = mbar_wait(&bars[B_READY0 + s], (c >> 1) & 1, abort_flag, kWaitLimitNs);
      // P, T_b and W^T of this parity were last read by chunk c-2's MMAs
      if (ok && c >= 2)
        ok = mbar_wait(&bars[B_EMPTY0 + s], ((c >> 1) + 1) & 1, abort_flag, kWaitLimitNs);
      // chunk scalars c % 3 were last read by chunk c-3's epilogue
      if (ok && c >= 3)
        ok = mbar_wait(&bars[B_CS_FREE0 + c % 3], ((c / 3) + 1) & 1, abort_flag, kWaitLimitNs);
      if (!ok) fail(8);
      named_bar_sync(1, 256);
      if (*abort_flag) break;
      const float* sc = stage_scal(s);
      ChunkScalars& cs = cscal[c % 3];
      const float gmax = sc[SC_GMAX];
      const bool exact = (gmax - sc[SC_GMIN]) > kMaxDecaySpan;
      const float Gi = sc[SC_G + i], Gl2i = Gi * kLog2e, GCl2 = sc[SC_G + 63] * kLog2e;
      const float ai = exp2f((Gi - gmax) * kLog2e);
      ok = mbar_wait(&bars[B_KQ_DONE], c & 1, abort_flag, kWaitLimitNs);
      if (!ok) fail(9);
      named_bar_sync(1, 256);
      if (*abort_flag) break;
      tc_fence_after();
      float qss_own = 0.f;
      uint32_t v[32];  // row L of [K;Q] K^T, columns [32 hf, 32 hf + 32)
      tmem_ld32(tmem + lane_off + TM_KQ + 32 * hf, v);
      tmem_ld_wait();
      float* Abuf = reinterpret_cast<float*>(sm + L_::WT0 + par * L_::SCR_BYTES);
      float* Tbuf = reinterpret_cast<float*>(sm + L_::TB0 + par * L_::SCR_BYTES);
      if (krow && (i >> 5) == hf) {
        // r^k_i from the diagonal of K K^T (fp32 sum of exact bf16 products)
        float diag = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j == (i & 31)) diag = __uint_as_float(v[j]);
        const float ri = p.l2norm ? 1.0f / sqrtf(diag + 1e-6f) : 1.f;
        const float bi = sc[SC_B + i];
        ps->d[i] = ri * exp2f((gmax - Gi) * kLog2e);
        ps->r[i] = ri;
        ps->beta[i] = bi;
        ps->tw[i] = bi * exp2f(Gl2i) * ri;
        cs.s[i] = exp2f(GCl2 - Gl2i) * ri;
      } else if (!krow) {
        // |q_i|^2 over this thread's half of the raw q row (r^q only scales the output)
        float ss0 = 0.f, ss1 = 0.f;
        const uint32_t rbase = stage_kq(s) + 8192u + i * 128u;
#pragma unroll
        for (int k = 0; k < 4 * L_::NKA; ++k) {
          const int idx = hf * 4 * L_::NKA + k;
          uint32_t x[4];
          ld_shared_v4(rbase + (idx >> 3) * 16384u + (idx & 7) * 16u, x[0], x[1], x[2], x[3]);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float lo = bf16_lo_f(x[e]), hi = bf16_hi_f(x[e]);
            ss0 = fmaf(lo, lo, ss0);
            ss1 = fmaf(hi, hi, ss1);
          }
        }
        if (hf == 1) const_cast<float*>(sc)[SC_QSS + i] = ss0 + ss1;
        else qss_own = ss0 + ss1;
      }
      named_bar_sync(1, 256);
      if (!krow && hf == 0) {
        const float rq = p.l2norm ? 1.0f / sqrtf(qss_own + sc[SC_QSS + i] + 1e-6f) : 1.f;
        const float co = p.scale * rq;
        cs.co[i] = co;
        cs.cq[i] = -co * exp2f(Gl2i);
        if (i == 0) cs.eGC = exp2f(GCl2);
      }
      if (exact) {
        // rare: every decay by its own exp (A and P rows into registers first)
        float row[32];
        {
          float wgt[32];
          exact_row(wgt, ps->r, sc + SC_G, Gl2i, ps->beta[i] * ps->r[i], 32 * hf, i, krow);
#pragma unroll
          for (int e = 0; e < 32; ++e) row[e] = wgt[e] * __uint_as_float(v[e]);
        }
        if (krow) {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4*>(&Abuf[i * LDF + 32 * hf + 4 * q]) =
                make_float4(row[4 * q], row[4 * q + 1], row[4 * q + 2], row[4 * q + 3]);
        } else {
          const uint32_t prow = sbase + L_::P0 + par * 8192u;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            st_shared_v4(prow + sw128(i, 4 * hf + q), pack_bf16(row[8 * q], row[8 * q + 1]),
                         pack_bf16(row[8 * q + 2], row[8 * q + 3]), pack_bf16(row[8 * q + 4], row[8 * q + 5]),
                         pack_bf16(row[8 * q + 6], row[8 * q + 7]));
        }
      } else if (krow) {
        // A_ij = beta_i r_i r_j e^{G_i - G_j} k_i.k_j  (j < i), fp32 into the scratch
        const float cia = ps->beta[i] * ps->r[i] * ai;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int j0 = 32 * hf + 4 * q;
          const float4 d4 = *reinterpret_cast<const float4*>(&ps->d[j0]);
          const float dd[4] = {d4.x, d4.y, d4.z, d4.w};
          float a4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            a4[e] = (j0 + e < i) ? (cia * __uint_as_float(v[4 * q + e])) * dd[e] : 0.f;
          *reinterpret_cast<float4*>(&Abuf[i * LDF + j0]) = make_float4(a4[0], a4[1], a4[2], a4[3]);
        }
      } else {
        // P_ij = e^{G_i - G_j} r^k_j q_i.k_j  (j <= i), bf16 K-major [i][j]
        const uint32_t prow = sbase + L_::P0 + par * 8192u;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int j0 = 32 * hf + 8 * q;
          const float4 da = *reinterpret_cast<const float4*>(&ps->d[j0]);
          const float4 db = *reinterpret_cast<const float4*>(&ps->d[j0 + 4]);
          const float dd[8] = {da.x, da.y, da.z, da.w, db.x, db.y, db.z, db.w};
          float pv[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            pv[e] = (j0 + e <= i) ? (ai * __uint_as_float(v[8 * q + e])) * dd[e] : 0.f;
          st_shared_v4(prow + sw128(i, 4 * hf + q), pack_bf16(pv[0], pv[1]), pack_bf16(pv[2], pv[3]),
                       pack_bf16(pv[4], pv[5]), pack_bf16(pv[6], pv[7]));
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(1, 256);
      // ---- T = (I + A)^-1
      solve_unit_lower(Abuf, Tbuf, wa);
      // ---- T_b = T diag(beta) as bf16 hi + lo; T_w = T diag(beta e^G r^k)
      {
        const int ti = wa & 63, qq = wa >> 6;  // row ti, columns [16 qq, 16 qq + 16)
        float t[16];
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const float4 x = *reinterpret_cast<const float4*>(&Tbuf[ti * LDF + 16 * qq + 4 * k4]);
          const bool zero = qq > (ti >> 4);  // block above the diagonal
          t[4 * k4 + 0] = zero ? 0.f : x.x;
          t[4 * k4 + 1] = zero ? 0.f : x.y;
          t[4 * k4 + 2] = zero ? 0.f : x.z;
          t[4 * k4 + 3] = zero ? 0.f : x.w;
        }
        named_bar_sync(1, 256);  // every thread has read T before it is overwritten
        const uint32_t tb = sbase + L_::TB0 + par * L_::SCR_BYTES;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int j0 = 16 * qq + 8 * q;
          const float4 ba = *reinterpret_cast<const float4*>(&ps->beta[j0]);
          const float4 bb = *reinterpret_cast<const float4*>(&ps->beta[j0 + 4]);
          const float4 wa4 = *reinterpret_cast<const float4*>(&ps->tw[j0]);
          const float4 wb4 = *reinterpret_cast<const float4*>(&ps->tw[j0 + 4]);
          const float bt[8] = {ba.x, ba.y, ba.z, ba.w, bb.x, bb.y, bb.z, bb.w};
          const float wt8[8] = {wa4.x, wa4.y, wa4.z, wa4.w, wb4.x, wb4.y, wb4.z, wb4.w};
          uint32_t hi4[4], lo4[4], w4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float x0 = t[8 * q + 2 * e] * bt[2 * e], x1 = t[8 * q + 2 * e + 1] * bt[2 * e + 1];
            hi4[e] = pack_bf16(x0, x1);
            lo4[e] = pack_bf16(x0 - bf16_lo_f(hi4[e]), x1 - bf16_hi_f(hi4[e]));
            w4[e] = pack_bf16(t[8 * q + 2 * e] * wt8[2 * e], t[8 * q + 2 * e + 1] * wt8[2 * e + 1]);
          }
          const uint32_t off = sw128(ti, 2 * qq + q);
          st_shared_v4(tb + off, hi4[0], hi4[1], hi4[2], hi4[3]);
          st_shared_v4(tb + 8192u + off, lo4[0], lo4[1], lo4[2], lo4[3]);
          st_shared_v4(sbase + L_::TW + off, w4[0], w4[1], w4[2], w4[3]);
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 256);
      if (wa == 0) mbar_arrive(&bars[B_P1_MID]);
      // ---- W^T: TMEM -> bf16 MN-major [d_k][j]
      ok = mbar_wait(&bars[B_W_DONE], c & 1, abort_flag, kWaitLimitNs);
      if (!ok) fail(10);
      named_bar_sync(1, 256);
      if (*abort_flag) break;
      tc_fence_after();
      {
        tmem_ld32(tmem + lane_off + TM_KQ + 32 * hf, v);
        tmem_ld_wait();
        const uint32_t wt = sbase + L_::WT0 + par * L_::SCR_BYTES;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          st_shared_v4(wt + sw128(L, 4 * hf + q),
                       pack_bf16(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1])),
                       pack_bf16(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                       pack_bf16(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                       pack_bf16(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(1, 256);
      if (wa == 0) {
        mbar_arrive(&bars[B_P1_DONE0 + par]);
        mbar_arrive(&bars[B_KQ_FREE]);
      }
    }
  } else if (warp >= 12) {
    // ================================================================ WG-B: state step + epilogue
    const int wb = tid - 384;  // == TMEM lane == d_v index
    const uint32_t lane_off = (uint32_t)((wb & ~31) << 16);
    const bool live = wb < DV;
    // initial state -> S^T in TMEM (lane d_v, column d_k)
    {
      const int64_t slot = state_slot(p, n);
      const float* s0 = slot >= 0 ? p.initial_state + ((size_t)slot * p.h_v + h) * DK * DV : nullptr;
#pragma unroll 1
      for (int xb = 0; xb < DK / 32; ++xb) {
        uint32_t v[32];
#pragma unroll
        for (int x = 0; x < 32; ++x)
          v[x] = (s0 && live) ? __float_as_uint(s0[(size_t)(xb * 32 + x) * DV + wb]) : 0u;
        tmem_st32(tmem + lane_off + TM_S + xb * 32, v);
      }
      tmem_st_wait();
    }
    // S -> -S^T (bf16 operand of chunk c's MMAs); S *= e^{G_m} of chunk c
    auto s_convert = [&](int c) -> bool {
      const int par = c & 1;
      bool ok = mbar_wait(&bars[B_P1_DONE0 + par], (c >> 1) & 1, abort_flag, kWaitLimitNs);
      if (ok && c >= 1) ok = mbar_wait(&bars[B_STATE_DONE], (c - 1) & 1, abort_flag, kWaitLimitNs);
      if (!ok) fail(11);
      named_bar_sync(2, 128);
      if (*abort_flag) return false;
      tc_fence_after();
      const float eGC = cscal[c % 3].eGC;
#pragma unroll 1
      for (int xb = 0; xb < DK / 32; ++xb) {
        uint32_t va[32];
        tmem_ld32(tmem + lane_off + TM_S + xb * 32, va);
        tmem_ld_wait();
        const uint32_t row = sbase + L_::SOP + (xb >> 1) * 16384u;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          st_shared_v4(row + sw128(wb, (xb & 1) * 4 + q),
                       pack_bf16(-__uint_as_float(va[8 * q + 0]), -__uint_as_float(va[8 * q + 1])),
                       pack_bf16(-__uint_as_float(va[8 * q + 2]), -__uint_as_float(va[8 * q + 3])),
                       pack_bf16(-__uint_as_float(va[8 * q + 4]), -__uint_as_float(va[8 * q + 5])),
                       pack_bf16(-__uint_as_float(va[8 * q + 6]), -__uint_as_float(va[8 * q + 7])));
#pragma unroll
        for (int x = 0; x < 32; ++x) va[x] = __float_as_uint(__uint_as_float(va[x]) * eGC);
        tmem_st32(tmem + lane_off + TM_S + xb * 32, va);
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(2, 128);
      if (wb == 0) mbar_arrive(&bars[B_S_READY]);
      return true;
    };
    bool run = nchunks == 0 || s_convert(0);
    for (int c = 0; run && c < nchunks; ++c) {
      const ChunkScalars& cs = cscal[c % 3];
      // ---- U' -> (U' s) hi / lo and U' as bf16, into TMEM A operands
      bool ok = mbar_wait(&bars[B_UP_DONE], c & 1, abort_flag, kWaitLimitNs);
      if (!ok) fail(12);
      named_bar_sync(2, 128);
      if (*abort_flag) break;
      tc_fence_after();
#pragma unroll 1
      for (int hb = 0; hb < 2; ++hb) {  // tokens [32 hb, 32 hb + 32)
        uint32_t u[32];
        tmem_ld32(tmem + lane_off + TM_R + hb * 32, u);
        tmem_ld_wait();
        uint32_t hi[16], lo[16], uu[16];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 s4 = *reinterpret_cast<const float4*>(&cs.s[hb * 32 + q * 4]);
          const float sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float a0 = __uint_as_float(u[q * 4 + 2 * e]), a1 = __uint_as_float(u[q * 4 + 2 * e + 1]);
            const float x0 = a0 * sv[2 * e], x1 = a1 * sv[2 * e + 1];
            const uint32_t hh = pack_bf16(x0, x1);
            hi[q * 2 + e] = hh;
            lo[q * 2 + e] = pack_bf16(x0 - bf16_lo_f(hh), x1 - bf16_hi_f(hh));
            uu[q * 2 + e] = pack_bf16(a0, a1);
          }
        }
        tmem_st16(tmem + lane_off + TM_UH + hb * 16, hi);
        tmem_st16(tmem + lane_off + TM_UL + hb * 16, lo);
        tmem_st16(tmem + lane_off + TM_UU + hb * 16, uu);
      }
      tmem_st_wait();
      tc_fence_before();
      named_bar_sync(2, 128);
      if (wb == 0) mbar_arrive(&bars[B_UOPS_READY]);
      // ---- the next chunk's state operand first: it is on the serial path
      if (c + 1 < nchunks && !s_convert(c + 1)) break;
      // ---- epilogue: o_i = cq_i (-S^T q_i) + co_i (U'^T P^T)_i, stored straight to out
      ok = mbar_wait(&bars[B_O_DONE], c & 1, abort_flag, kWaitLimitNs);
      if (!ok) fail(13);
      named_bar_sync(2, 128);
      if (*abort_flag) break;
      tc_fence_after();
      {
        const int64_t t0 = bos + (int64_t)c * kChunk;
        const int m = chunk_rows(c);
        const bool odd = wb & 1;
#pragma unroll 1
        for (int hb = 0; hb < 2; ++hb) {  // tokens [32 hb, 32 hb + 32)
          uint32_t oq[32], oi[32];
          tmem_ld32(tmem + lane_off + TM_QS + hb * 32, oq);
          tmem_ld32(tmem + lane_off + TM_O + hb * 32, oi);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 a4 = *reinterpret_cast<const float4*>(&cs.cq[hb * 32 + q * 4]);
            const float4 b4 = *reinterpret_cast<const float4*>(&cs.co[hb * 32 + q * 4]);
            const float av[4] = {a4.x, a4.y, a4.z, a4.w}, bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              oq[q * 4 + e] = __float_as_uint(fmaf(av[e], __uint_as_float(oq[q * 4 + e]),
                                                   bv[e] * __uint_as_float(oi[q * 4 + e])));
          }
          if (p.out_f32) {
            if (live) {
#pragma unroll
              for (int ii = 0; ii < 32; ++ii)
                if (hb * 32 + ii < m)
                  reinterpret_cast<float*>(p.out)[((size_t)(t0 + hb * 32 + ii) * p.h_v + h) * DV + wb] =
                      __uint_as_float(oq[ii]);
            }
          } else {
            // lanes 2k and 2k+1 swap values so each stores a bf16 pair (d_v 2k, 2k+1)
            // of one token: a warp writes two 64-byte row segments per store
#pragma unroll
            for (int tp = 0; tp < 16; ++tp) {
              const float x0 = __uint_as_float(oq[2 * tp]), x1 = __uint_as_float(oq[2 * tp + 1]);
              const float got = __shfl_xor_sync(0xffffffffu, odd ? x0 : x1, 1);
              const int row = hb * 32 + 2 * tp + (odd ? 1 : 0);
              const uint32_t word = odd ? pack_bf16(got, x1) : pack_bf16(x0, got);
              if (live && row < m)
                reinterpret_cast<uint32_t*>(p.out)[(((size_t)(t0 + row) * p.h_v + h) * DV + (wb & ~1)) >> 1] = word;
            }
          }
        }
      }
      tc_fence_before();
      named_bar_sync(2, 128);
      if (wb == 0) {
        mbar_arrive(&bars[B_EPI_DONE]);
        mbar_arrive(&bars[B_CS_FREE0 + c % 3]);
      }
    }
    // final state
    if (!*abort_flag && p.final_state) {
      tc_fence_after();
      float* fs = p.final_state + ((size_t)n * p.h_v + h) * DK * DV;
#pragma unroll 1
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
