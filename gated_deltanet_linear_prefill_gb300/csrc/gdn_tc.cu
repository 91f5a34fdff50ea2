// Tensor-core (tcgen05 / TMEM / TMA) kernel for the chunked gated delta rule.
//
// Chunked form (open-jev-fast README, Phase 3 item 1: per chunk the gate
// cumsum, K K^T, the (I + A)^-1 solve, u and w, the chunk output and the state
// update). With S the d_k x d_v state entering a chunk of m <= 64 rows,
// G_i = sum_{s<=i} g_s (G_m: the whole chunk), r^k_i / r^q_i the L2-norm
// scales of k_i / q_i, and M_ij = q_i.k_j for j <= i (0 above):
//
//   A_ij = beta_i r^k_i r^k_j e^{G_i-G_j} k_i.k_j   (j < i)     T = (I + A)^-1
//   U  = T diag(beta) V               W = T diag(beta e^G r^k) K
//   U' = U - W S                      s_j = e^{G_m-G_j} r^k_j
//   o_i = scale r^q_i e^{G_i-G_m} ( e^{G_m} S^T q_i + sum_j s_j u'_j M_ij )
//   S  <- e^{G_m} S + sum_j s_j k_j u'_j^T
//
// The stored state is S~ = S / mu. A chunk's decay e^{G_m} is folded into the
// operand scalars (lambda = mu e^{G_m} becomes the new mu) and only applied to
// the stored state when |log lambda| would pass kMaxLogScale, so the state is
// not rewritten every chunk. A chunk ends early when the log-decay inside it
// spans more than kMaxSpan, which keeps every factorised exponential in fp32
// range for any finite gate.
//
// One CTA per SM stays resident and takes (sequence, value head) units in turn
// from a counter (longest first), walking each unit's chunks in order; the
// chunks of successive units form one stream through the pipeline, so it does
// not drain between units.
// All dense products run on tcgen05 in the "d-major" orientation, where the
// 128 TMEM lanes index d_v (or d_k) so every MMA has M = 128:
//   [K;Q] K^T                    KK^T (lanes 0-63) and QK^T (lanes 64-127)
//   W'^T  = K^T T_w^T            T_w = -nu T diag(beta e^G r^k), bf16
//   U'^T  = V^T T_b^T + S~^T W'^T   T_b = T diag(beta) as bf16 hi + lo
//   O^T   = S~^T Q^T + (U' diag(s/lambda))^T M^T
//   S~^T += (U' diag(s/lambda))^T K
// S~^T and U' diag(s/lambda) (bf16 hi + lo) are A operands read straight from
// TMEM. Operand precision: T_b and U' s carry about 16 significant bits (hi +
// lo) where they feed the state; S~, W, M and the U' s of the intra-chunk
// output term enter as bf16; every accumulation is fp32. Decays, norms and
// the 64x64 unit-lower-triangular inverse run on CUDA cores in fp32, the
// inverse's block merges on the warp-level tensor cores (tf32 operands, fp32
// accumulation; the merged blocks carry about 11 significant bits).
//
// Warp roles (512 threads): warp 0 scans the gates, sizes the chunks and loads
// K/Q/V tiles by TMA (128-byte swizzle) into a 3-deep K/Q ring and a 2-deep V
// ring; warp 1 allocates TMEM and issues [K;Q] K^T; warp 2 issues the
// state-dependent MMAs; warp 3 takes the q norms; warps 4-11 (WG-A) prepare
// chunk c+1 (k norms, A and M, the solve, T_b / T_w, the W and U products)
// while warps 12-15 (WG-B) run chunk c's state step (U' split, S~ -> bf16
// operand, output epilogue). Every mbarrier wait is bounded: on timeout the
// CTA reports GDN_ERR_DEVICE_TIMEOUT and unwinds.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {
#ifdef GDN_TC_TRACE
// [16 warps][256 chunks][8 points] clock64 stamps, then {clock, globaltimer} at the
// traced CTA's start and end (for the clock rate)
__device__ unsigned long long g_gdn_trace[16 * 2048 + 4];
__device__ int g_gdn_trace_cta = 0;
#endif
namespace {

using namespace ptx;

constexpr int kTcThreads = 512;

// Per-role clock trace, compiled only into the tracing build (-DGDN_TC_TRACE, the
// separate libgdn_trace.so): lane 0 of warp `role` in CTA g_gdn_trace_cta records
// clock64() at point `pt` (0-7) of chunk `chunk` (< 256); gdn_trace_* read it back.
#ifdef GDN_TC_TRACE
#define GDN_TRACE(role, chunk, pt)                                                                   \
  do {                                                                                               \
    const int gt_c = (chunk);                                                                        \
    if ((int)blockIdx.x == g_gdn_trace_cta && gt_c >= 0 && gt_c < 256 && (threadIdx.x & 31) == 0 &&  \
        (int)(threadIdx.x >> 5) == (role))                                                           \
      g_gdn_trace[(role) * 2048 + gt_c * 8 + (pt)] = clock64();                                      \
  } while (0)
#else
#define GDN_TRACE(role, chunk, pt) \
  do {                             \
  } while (0)
#endif
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait: far above any legal wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kMaxSpan = 30.0f;      // largest log-decay span inside one chunk
constexpr float kMaxLogScale = 50.0f;  // largest |log mu| of the stored state

// TMEM columns (fp32 unless noted)
constexpr uint32_t TM_S = 0;     // S~^T: lanes d_v, columns d_k             (128)
constexpr uint32_t TM_KQ = 128;  // [K;Q] K^T                                 (64)
constexpr uint32_t TM_W = 192;   // W'^T: lanes d_k, columns j                (64)
constexpr uint32_t TM_R = 256;   // U^T, then U'^T: lanes d_v, columns j      (64)
constexpr uint32_t TM_O = 320;   // O^T: lanes d_v, columns i                 (64)
constexpr uint32_t TM_UH = 384;  // (U' diag(s/lambda))^T hi, packed bf16     (32)
constexpr uint32_t TM_UL = 416;  // (U' diag(s/lambda))^T lo                  (32)
constexpr uint32_t TM_SB = 448;  // S~^T as packed bf16                       (64)
constexpr uint32_t kTmemCols = 512;

// Barrier indices (arrival count 1 each)
enum {
  B_FULL0 = 0, B_FULL1, B_FULL2,  // chunk K/Q tiles + gate scalars landed (slot c % 3)
  B_VFULL0, B_VFULL1,             // chunk V tile landed (slot c % 2)
  B_KQE0, B_KQE1, B_KQE2,         // K/Q slot released (chunk c's output staged out)
  B_VE0, B_VE1,                   // V slot released (slot c % 2)
  B_RQ0, B_RQ1, B_RQ2,            // q norms of slot c % 3 written
  B_KQ_DONE, B_KQ_FREE, B_W_DONE, B_R_FREE, B_W_FREE,
  B_WCONV0, B_WCONV1,             // W'^T of chunk c converted to bf16 (c % 2)
  B_P1_DONE0, B_P1_DONE1,         // chunk prepared (c % 2)
  B_T_READY0, B_T_READY1,         // T_b / T_w of chunk c written (c % 2)
  B_U_DONE, B_S_READY, B_UP_DONE, B_UOPS_READY, B_STATE_DONE, B_O_DONE, B_EPI_DONE,
  B_MFREE0, B_MFREE1, B_CSF0, B_CSF1, B_CSF2,
  B_DRAIN1, B_DRAIN2, B_DRAIN3, kNumBars
};
static_assert(kNumBars <= 127, "barrier indices fit the seven bits of a wait-list entry");

// Gate scalars the producer writes next to each K/Q slot (floats).
constexpr int SC_G = 0;        // G_i (rows past m repeat G_{m-1})
constexpr int SC_B = 64;       // beta_i (0 past m)
constexpr int SC_RQ = 128;     // r^q_i (written by warp 3)
constexpr int SC_GMAX = 192;   // max / min of G over the chunk's rows
constexpr int SC_GMIN = 193;
constexpr int SC_GM = 194;     // G_m
constexpr int SC_LAMLOG = 195; // log lambda used by s and the output weights (0 when eager)
constexpr int SC_NULOG = 196;  // log of the W' weight applied to e^{G_j}
constexpr int SC_RMW = 197;    // factor applied to the stored state first (1 unless eager)
constexpr int SC_MUNEXT = 198; // mu after this chunk
constexpr int SC_M = 199;      // rows (int)
constexpr int SC_FLAGS = 200;  // F_* bits below
constexpr int SC_T0 = 202;     // first row (int64, two words)
constexpr int SC_N = 204;      // the chunk's sequence (int)
constexpr int SC_H = 205;      // the chunk's value head (int)
// chunk flags
constexpr int F_ULAST = 1;     // last chunk of its (sequence, head) unit
constexpr int F_EAGER = 2;     // the stored state is rescaled before this chunk
constexpr int F_UFIRST = 4;    // first chunk of its unit: the state starts over
constexpr int F_SLAST = 8;     // last chunk this CTA processes
constexpr int F_ZFIRST = 16;   // first chunk of a unit whose starting state is zero: the
                               // state-dependent products (W' S~, S~^T Q^T) vanish
constexpr int F_VZERO = 32;    // the unit reads V as zero (a segment's state map Phi)
constexpr int F_NOOUT = 64;    // the unit writes no output (only its final state is used)
// (the last two occur only in a segment launch, the kernel's SEG instance: every test of
// them is written SEG && ..., so that the other instances carry none of their code)

// Per-chunk values WG-A hands to WG-B (three buffers, chunk % 3).
struct ChunkScalars {
  float co[64];  // scale e^{G_i - G_m} lambda: output weight of row i without r^q_i (0 past m)
  long long t0;  // first row of the chunk
  float mu_next; // mu after the chunk
  int m;         // rows
  int slast;     // the last chunk this CTA processes
  int n, h;      // the chunk's (sequence, value head) unit
  int pad;
};
// WG-A private per-chunk values.
struct PrepScalars {
  float d[64];     // r^k_j e^{Gmax - G_j}
  float r[64];     // r^k_j
  float tw[64];    // column scale of T_w
  float beta[64];
  float s[64];     // e^{G_m - G_j} r^k_j / lambda: weight of u'_j (0 past m), the row scale of T_b, T_w
};

constexpr int LDF = 68;  // row stride (floats) of the fp32 64x64 scratch of the solve

// Shared-memory layout, byte offsets from a 1024-aligned base.
template <int DK, int DV>
struct TcLayout {
  static constexpr int NKA = DK / 64;  // 64-element atom columns of K / Q
  static constexpr int NVA = DV / 64;
  static constexpr uint32_t KQ_BYTES = NKA * 16384u;  // [K atom][Q atom] per atom column
  static constexpr uint32_t SCAL_BYTES = 1024u;
  static constexpr uint32_t SLOT_BYTES = KQ_BYTES + SCAL_BYTES;
  static constexpr uint32_t V_BYTES = NVA * 8192u;
  static constexpr uint32_t SCR_BYTES = 17408u;           // 64 x 68 fp32, 1024-aligned size
  static constexpr uint32_t WP_BYTES = DK * 64u * 4u;      // W' fp32 [64 rows j][DK], K-major
  // K/Q slots x3; once a chunk's products have read its K/Q tiles, the first 16 KB of
  // its slot stage that chunk's output tiles
  static constexpr uint32_t RING0 = 0;
  static constexpr uint32_t V0 = 3 * SLOT_BYTES;           // V slots x2
  static constexpr uint32_t M0 = V0 + 2 * V_BYTES;         // M (bf16 64x64) x2
  static constexpr uint32_t TB = M0 + 2 * 8192u;           // fp32 T, then T_b hi / lo
  static constexpr uint32_t TW = TB + SCR_BYTES;           // T_w bf16
  static constexpr uint32_t AS = TW + 8192u;               // fp32 A (WG-A's own chunk only)
  static constexpr uint32_t WP = AS + SCR_BYTES;           // W' fp32 (one chunk at a time)
  static constexpr bool NEED_ZERO = (DK == 64) || (DV == 64);
  static constexpr uint32_t ZERO = WP + WP_BYTES;          // 8 KB of zeros (M padding)
  static constexpr uint32_t CS0 = ZERO + (NEED_ZERO ? 8192u : 0u);
  static constexpr uint32_t PS = CS0 + 3 * (uint32_t)sizeof(ChunkScalars);
  static constexpr uint32_t BARS = PS + (uint32_t)sizeof(PrepScalars);
  static constexpr uint32_t MISC = BARS + kNumBars * 8u;  // tmem base, abort flag
  static constexpr uint32_t TOTAL = MISC + 64u;
  static constexpr uint32_t DYN_SMEM = TOTAL + 1024u;     // alignment slack
  static_assert(SLOT_BYTES % 1024 == 0 && WP_BYTES % 1024 == 0, "slot alignment");
  static_assert(KQ_BYTES >= 16384u, "a K/Q slot holds a chunk's output staging tiles");
  static_assert(sizeof(ChunkScalars) % 16 == 0, "chunk scalars alignment");
  static_assert(DYN_SMEM <= 232448u, "shared memory budget");
};

struct Tmaps {
  CUtensorMap q, k, v;
  CUtensorMap o;  // out [T, h_v, d_v]: box d_v x 1 head x 32 rows (bf16) or 16 rows (fp32)
};

// v, or 0 when `zero` (a block above the diagonal, whose T entries are parked products).
__device__ __forceinline__ float zero_row(float v, bool zero) { return zero ? 0.f : v; }

// ---------------------------------------------------------------- the solve
// Warp-level tensor-core tiles for the block merges: mma.sync m16n8k8 with
// tf32 operands taken straight from the fp32 values in shared memory (the
// tensor cores read the top 19 bits), fp32 accumulation. Every T entry itself
// stays fp32. Fragment layout (lane = 4 g + t): A rows g, g+8 x columns t, t+4;
// B rows t, t+4 x column g; C rows g, g+8 x columns 2t, 2t+1.
__device__ __forceinline__ void mma_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// c[16 x 8] += X[xr.., xc + k) * Y[yr + k, yc..) over k in [0, 8 nk8), nk8 <= 4, fp32 smem
// with row stride LDF (xc a multiple of 4). Every operand is loaded before the first
// product. The A fragments come from one ldmatrix per k step: read as 16-bit pairs, an
// 8 x 8 b16 matrix is an 8 x 4 block of fp32 words and lane 4 g + t gets word (g, t), so
// the four blocks (rows 0-7 / 8-15 by columns 0-3 / 4-7 of the step) are a0 .. a3; lane
// l gives the address of row (l & 7) + 8 ((l >> 3) & 1), columns 4 (l >> 4) on.
__device__ __forceinline__ void mma_tile(const float* X, int xr, int xc, const float* Y, int yr,
                                         int yc, int nk8, float (&c)[4], int lane) {
  const int g = lane >> 2, t = lane & 3;
  const uint32_t xrow = smem_u32(X + (xr + (lane & 7) + 8 * ((lane >> 3) & 1)) * LDF + xc + 4 * (lane >> 4));
  const float* y0 = Y + (yr + t) * LDF + yc + g;
  uint32_t xa[4][4], yb[4][2];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (k < nk8) {
      ldmatrix_x4(xrow + 32u * k, xa[k][0], xa[k][1], xa[k][2], xa[k][3]);
      yb[k][0] = __float_as_uint(y0[8 * k * LDF]);
      yb[k][1] = __float_as_uint(y0[(8 * k + 4) * LDF]);
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k)
    if (k < nk8) mma_tf32(c, xa[k][0], xa[k][1], xa[k][2], xa[k][3], yb[k][0], yb[k][1]);
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
//     lane (two blocks per warp), each row of A read as float4 broadcasts;
//  2. T_{b+1,b} = -D_{b+1} (A_{b+1,b} D_b) inside both 32x32 diagonal blocks;
//  3. T_21 = -T_22 (A_21 T_11) for the lower-left 32x32 block.
// Steps 2 and 3 run on the warp-level tensor cores (tf32 operands, fp32
// accumulation), one 16x8 tile per warp and product. Their intermediate products are parked in
// T's upper triangle, which nothing reads as T; blocks above the diagonal are
// not otherwise written. A warp that reads a parked tile either wrote it
// itself or waits for its writer on a pair barrier (ids 3-6), so only three
// barriers span all 256 threads (8 warps). Ends with every T entry visible to
// all of them.
__device__ __forceinline__ void solve_unit_lower(const float* __restrict__ A, float* __restrict__ T,
                                                 int wa) {
  const int wq = wa >> 5, ln = wa & 31;
  if (wq < 2) {
    // warp wq inverts blocks 2 wq (lanes 0-15) and 2 wq + 1 (lanes 16-31)
    const int b = 32 * wq + 16 * (ln >> 4), l = ln & 15;  // lane owns column l of its block
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
  const int h8 = 8 * (wq & 1);  // which 8 columns of a 16-wide block this warp takes
  if (wq < 4) {
    // step 2 in the 32x32 diagonal block at b: P = A_{b+1,b} D_b (parked at block (b, b+1)),
    // then T_{b+1,b} = -D_{b+1} P; the warp reads back only its own P columns
    const int b = 32 * (wq >> 1);
    float c[4] = {}, d[4] = {};
    mma_tile(A, b + 16, b, T, b, b + h8, 2, c, ln);
    store_tile(T, b, b + 16 + h8, c, 1.f, ln);
    __syncwarp();
    mma_tile(T, b + 16, b + 16, T, b, b + 16 + h8, 2, d, ln);
    store_tile(T, b + 16, b + h8, d, -1.f, ln);
  }
  named_bar_sync(1, 256);
  {
    // step 3 for row block rb in {2, 3}, column block cb in {0, 1}:
    // Z_rb = A_{rb, cb..1} T_{cb..1, cb} (parked in row block rb - 2 of the upper right),
    // then T_{rb,cb} = -T_{rb, 2..rb} Z_{2..rb}; row block 3 also needs row block 2's Z
    const int rb = 2 + (wq >> 2), cb = (wq >> 1) & 1;
    float c[4] = {}, d[4] = {};
    mma_tile(A, 16 * rb, 16 * cb, T, 16 * cb, 16 * cb + h8, 2 * (2 - cb), c, ln);
    store_tile(T, 16 * (rb - 2), 32 + 16 * cb + h8, c, 1.f, ln);
    if (rb == 2)
      named_bar_arrive(3 + (wq & 3), 64);
    else
      named_bar_sync(3 + (wq & 3), 64);
    __syncwarp();
    mma_tile(T, 16 * rb, 32, T, 0, 32 + 16 * cb + h8, 2 * (rb - 1), d, ln);
    store_tile(T, 16 * rb, 16 * cb + h8, d, -1.f, ln);
  }
  named_bar_sync(1, 256);
}

// Shared words of the MISC block: the TMEM base, the abort flag, the status
// pointer and the unit, so that the slow path of a wait needs only addresses.
constexpr uint32_t MISC_TMEM = 0, MISC_ABORT = 4, MISC_STATUS = 8, MISC_UNIT = 16, MISC_WORK = 20;
constexpr uint32_t kDrainWait = 0x8000u;  // site flag: a drain (ignores abort, shorter limit)

// Slow path of every mbarrier wait: polls (each poll may park the thread until
// the phase completes) until the phase is done, another role has aborted, or
// the time limit passes. On timeout the CTA reports GDN_ERR_DEVICE_TIMEOUT
// once (detail: unit * 16 + site) and raises the abort flag so that every role
// unwinds. Out of line: a wait rarely gets here.
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, uint32_t misc, uint32_t site) {
  const bool drain = (site & kDrainWait) != 0;
  const uint64_t limit = drain ? 100000000ull : kWaitLimitNs;
  const uint64_t t0 = globaltimer();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (!drain && ld_shared_volatile_u32(misc + MISC_ABORT)) return false;
    if (globaltimer() - t0 > limit) {
      if (!drain && !ld_shared_volatile_u32(misc + MISC_ABORT)) {
        st_shared_volatile_u32(misc + MISC_ABORT, 1u);
        Status* st;
        asm volatile("ld.shared.u64 %0, [%1];" : "=l"(st) : "r"(misc + MISC_STATUS));
        report(st, GDN_ERR_DEVICE_TIMEOUT, ld_shared_volatile_u32(misc + MISC_UNIT) * 16u + (site & 15u));
      }
      return false;
    }
  }
}

// A group of bounded waits through one call: `list` holds one byte per barrier (its
// index from `bars` in the low seven bits, the parity in the top bit), 0xff after the
// last. False when a wait gave up (see wait_slow).
__device__ __noinline__ bool wait_list(uint64_t list, uint32_t bars, uint32_t misc, uint32_t site) {
#pragma unroll 1
  for (; (list & 0xffu) != 0xffu; list >>= 8) {
    const uint32_t e = (uint32_t)list & 0xffu;
    const uint32_t bar = bars + 8u * (e & 0x7fu);
    if (!mbar_try_wait(bar, e >> 7) && !wait_slow(bar, e >> 7, misc, site)) return false;
  }
  return true;
}

// The rows of a chunk whose gates span more than kMaxSpan in log-decay: the window
// of m rows is halved until the span of {0, G_0 .. G_{m-1}} fits (one row always
// does). s0 / s1: the inclusive prefix sums G of rows lane and lane + 32. Returns
// (m as int bits, max and min of G over the chosen rows). Out of line: only
// decays far outside the usual range get here.
__device__ __noinline__ float3 span_fit(float s0, float s1, int m, int lane) {
#pragma unroll 1
  for (;;) {
    m = (m + 1) >> 1;
    const float wmax = warp_max(fmaxf(lane < m ? s0 : -3.0e38f, lane + 32 < m ? s1 : -3.0e38f));
    const float wmin = warp_min(fminf(lane < m ? s0 : 3.0e38f, lane + 32 < m ? s1 : 3.0e38f));
    if (m <= 1 || fmaxf(wmax, 0.f) - fminf(wmin, 0.f) <= kMaxSpan) return make_float3(__int_as_float(m), wmax, wmin);
  }
}

// Waits (bounded) until the K / Q loads of the last three chunks and the V loads
// of the last two that the producer requested have landed, before the CTA exits.
__device__ __noinline__ void drain_loads(uint32_t bars, int kq_issued, int v_issued, uint32_t misc) {
#pragma unroll 1
  for (int c = kq_issued - 3 < 0 ? 0 : kq_issued - 3; c < kq_issued; ++c) {
    const uint32_t bar = bars + 8u * (uint32_t)(B_FULL0 + c % 3), par = (uint32_t)((c / 3) & 1);
    if (!mbar_try_wait(bar, par)) wait_slow(bar, par, misc, kDrainWait);
  }
#pragma unroll 1
  for (int c = v_issued - 2 < 0 ? 0 : v_issued - 2; c < v_issued; ++c) {
    const uint32_t bar = bars + 8u * (uint32_t)(B_VFULL0 + (c & 1)), par = (uint32_t)((c >> 1) & 1);
    if (!mbar_try_wait(bar, par)) wait_slow(bar, par, misc, kDrainWait);
  }
}

// ---------------------------------------------------------------- the kernel
// OF32: fp32 output (else bf16); GF32: fp32 gates (else bf16). Template parameters,
// so that each kernel holds only its own epilogue and gate loads.
template <int DK, int DV, bool OF32, bool GF32, int MODE>
__global__ void __launch_bounds__(kTcThreads, 1)
    gdn_tc_kernel(const Params p, const __grid_constant__ Tmaps tm) {
  // instance: 0 the regular launch, 1 a segment launch (V-zero and no-output units), 2 a
  // direct launch of a small batch (CTA b takes unit b, no work list)
  constexpr bool SEG = MODE == 1, DIRECT = MODE == 2;
  using L = TcLayout<DK, DV>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(sm);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BARS);
  uint32_t* tmem_base_ptr = reinterpret_cast<uint32_t*>(sm + L::MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::MISC + MISC_ABORT);
  ChunkScalars* cscal = reinterpret_cast<ChunkScalars*>(sm + L::CS0);
  PrepScalars* ps = reinterpret_cast<PrepScalars*>(sm + L::PS);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
#ifdef GDN_TC_TRACE
  if (tid == 0 && (int)blockIdx.x == g_gdn_trace_cta) {
    g_gdn_trace[16 * 2048] = clock64();
    g_gdn_trace[16 * 2048 + 1] = globaltimer();
  }
#endif
  // The CTA stays resident and takes (sequence, head) units in order from a counter
  // (the work list is longest first; in a tree launch parents come before children),
  // running their chunks as one stream so that the pipeline does not drain between
  // units. Thread 0 takes the first unit here; the producer takes the rest.
  const int total_units = p.num_seqs * p.h_v;
  int* first_unit = reinterpret_cast<int*>(sm + L::MISC + MISC_WORK);

  // ---- setup
  if (tid == 0) {
    for (int b = 0; b < kNumBars; ++b) mbar_init(&bars[b], 1u);
    *abort_flag = 0;
    *reinterpret_cast<Status**>(sm + L::MISC + MISC_STATUS) = p.status;
    *reinterpret_cast<uint32_t*>(sm + L::MISC + MISC_UNIT) = (uint32_t)blockIdx.x;
    mbar_init_fence();
  }
  if (L::NEED_ZERO)
    for (int i = tid; i < 8192 / 16; i += kTcThreads) st_shared_v4(sbase + L::ZERO + i * 16, 0, 0, 0, 0);
  for (int i = tid; i < 2 * 8192 / 16; i += kTcThreads) st_shared_v4(sbase + L::M0 + i * 16, 0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm.q);
    tma_prefetch_desc(&tm.k);
    tma_prefetch_desc(&tm.v);
    tma_prefetch_desc(&tm.o);
  }
  if (warp == 1) tmem_alloc(tmem_base_ptr, kTmemCols);
  // The launch may overlap the prep kernel (programmatic dependent launch): everything
  // above touches only this CTA's own memory; the status block, the work counter and the
  // work list are read only after the prep grid has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid == 0) *first_unit = DIRECT ? (int)blockIdx.x : (int)atomicAdd(&p.status->next_unit, 1u);
  if (DIRECT && tid == 32 && (int)blockIdx.x < total_units && blockIdx.x % p.h_v == 0) {
    // a direct launch checks what the prep kernel would: this CTA's own sequence
    const int n = (int)blockIdx.x / p.h_v;
    const int64_t b = p.cu_seqlens[n], e = p.cu_seqlens[n + 1];
    if ((n == 0 && b != 0) || e < b || (n == p.num_seqs - 1 && e != p.total_tokens) ||
        (p.max_seqlen > 0 && e - b > p.max_seqlen))
      report(p.status, GDN_ERR_SEQLENS, (uint32_t)n);
    if (p.initial_state && p.state_index) {
      const int32_t si = p.state_index[n];
      if (si < -1 || si >= p.num_state_slots) report(p.status, GDN_ERR_STATE_INDEX, (uint32_t)n);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_ptr;
  const bool any = *first_unit < total_units;  // this CTA has at least one unit

  auto slot_kq = [&](int c) { return sbase + L::RING0 + (uint32_t)(c % 3) * L::SLOT_BYTES; };
  auto slot_v = [&](int c) { return sbase + L::V0 + (uint32_t)(c & 1) * L::V_BYTES; };
  auto slot_sc = [&](int c) {
    return reinterpret_cast<float*>(sm + L::RING0 + (uint32_t)(c % 3) * L::SLOT_BYTES + L::KQ_BYTES);
  };
  auto sc_int = [](const float* sc, int k) { return __float_as_int(sc[k]); };
  // bounded wait on barrier b; `site` names the wait in a timeout report
  auto wait = [&](int b, uint32_t parity, uint32_t site) {
    const uint32_t bar = sbase + L::BARS + 8u * (uint32_t)b;
    return mbar_try_wait(bar, parity) || wait_slow(bar, parity, sbase + L::MISC, site);
  };
  // a group of waits (see wait_list); the order of the entries does not matter
  auto wait_all = [&](uint64_t list, uint32_t site) {
    return wait_list(list, sbase + L::BARS, sbase + L::MISC, site);
  };
  // list entry for barrier b at parity `parity`, prepended to `list`
  auto with = [](uint64_t list, int b, uint32_t parity) {
    return (list << 8) | (uint64_t)((uint32_t)b | ((parity & 1u) << 7));
  };
  constexpr uint64_t kNone = 0xffu;  // an empty list

  if (warp == 0) {
    // ================================================================ producer
    // Scans the gates of the next 64 rows, ends the chunk early if the log-decay
    // span would pass kMaxSpan, keeps the state-scale bookkeeping, and requests
    // the chunk's tiles once its ring slots are free. It never waits for data.
    const uint32_t kq_bytes = (uint32_t)(2 * L::NKA) * 8192u, v_bytes = (uint32_t)L::NVA * 8192u;
    int kq_issued = 0, v_issued = 0;  // chunks whose K / Q and V loads were requested
    int cur = *first_unit, g = 0;     // the unit in hand; chunks emitted so far
    // the next unit is taken when the last chunk of the current one is emitted (so that
    // this chunk knows whether it is the CTA's last), not earlier: a CTA then holds a
    // second unit only briefly, and the work list keeps its longest-first order
    auto take_unit = [&]() {
      if (DIRECT) return total_units;  // one unit per CTA
      int u = 0;
      if (lane == 0) u = (int)atomicAdd(&p.status->next_unit, 1u);
      return __shfl_sync(0xffffffffu, u, 0);
    };
    int nxt = -1;
    bool ok = true;
#pragma unroll 1
    while (ok && cur < total_units) {
      int n = !GDN_IN_BOUNDS(p.status, cur / p.h_v < p.num_seqs, 0x101u) ? 0
              : DIRECT ? cur / p.h_v : p.order[cur / p.h_v];
      if (n < 0 || n >= p.num_seqs) {  // never expected: the prep kernel writes a permutation
        if (lane == 0) report(p.status, GDN_ERR_SEQLENS, (uint32_t)cur);
        n = 0;
      }
      const int h = cur % p.h_v, hq = h / (p.h_v / p.h_qk);
      const bool vzero = SEG && n >= p.vzero_from, noout = SEG && n >= p.out_upto;
      const bool zstart = tree_parent(p, n) < 0 && state_slot(p, n) < 0 && !vzero;
      int64_t bos, eos;
      seq_bounds(p, n, bos, eos);
      const int64_t len = eos - bos;  // 0: one chunk of no rows carries the unit's state through
      int64_t start = 0;
      float logmu = 0.f;
#pragma unroll 1
      for (int cu = 0;; ++cu, ++g) {
        // the gates of the chunk's rows (0 past the sequence)
        float g0 = 0.f, g1 = 0.f, b0 = 0.f, b1 = 0.f;
        {
          const int64_t avail = len - start;
          const int64_t i0 = (bos + start + lane) * p.h_v + h, i1 = i0 + 32 * (int64_t)p.h_v;
          const bool in0 = lane < avail && GDN_IN_BOUNDS(p.status, bos + start + lane < p.total_tokens, 0x102u);
          const bool in1 =
              lane + 32 < avail && GDN_IN_BOUNDS(p.status, bos + start + lane + 32 < p.total_tokens, 0x102u);
          if constexpr (GF32) {
            const float* gg = reinterpret_cast<const float*>(p.g);
            const float* bb = reinterpret_cast<const float*>(p.beta);
            if (in0) { g0 = gg[i0]; b0 = bb[i0]; }
            if (in1) { g1 = gg[i1]; b1 = bb[i1]; }
          } else {
            const __nv_bfloat16* gg = reinterpret_cast<const __nv_bfloat16*>(p.g);
            const __nv_bfloat16* bb = reinterpret_cast<const __nv_bfloat16*>(p.beta);
            if (in0) { g0 = __bfloat162float(gg[i0]); b0 = __bfloat162float(bb[i0]); }
            if (in1) { g1 = __bfloat162float(gg[i1]); b1 = __bfloat162float(bb[i1]); }
          }
        }
        const int mv = (int)(len - start < kChunk ? len - start : kChunk);
        // inclusive prefix sums and prefix max / min (the chunk start, 0, included)
        float s0 = g0, s1 = g1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float u0 = __shfl_up_sync(0xffffffffu, s0, o), u1 = __shfl_up_sync(0xffffffffu, s1, o);
          if (lane >= o) { s0 += u0; s1 += u1; }
        }
        s1 += __shfl_sync(0xffffffffu, s0, 31);
        // rows of the chunk: the window, halved (out of line, only for decays far outside
        // the usual range) while the span of {0, G_0 .. G_{m-1}} passes kMaxSpan
        int m = mv;
        float gmax = warp_max(fmaxf(lane < m ? s0 : -3.0e38f, lane + 32 < m ? s1 : -3.0e38f));
        float gmin = warp_min(fminf(lane < m ? s0 : 3.0e38f, lane + 32 < m ? s1 : 3.0e38f));
        if (m > 1 && fmaxf(gmax, 0.f) - fminf(gmin, 0.f) > kMaxSpan) {
          const float3 f = span_fit(s0, s1, m, lane);
          m = __float_as_int(f.x);
          gmax = f.y;
          gmin = f.z;
        }
        // rows past m: no decay, no write
        const float Gm = m > 0 ? __shfl_sync(0xffffffffu, (m - 1) < 32 ? s0 : s1, (m - 1) & 31) : 0.f;
        if (lane >= m) { s0 = Gm; b0 = 0.f; }
        if (lane + 32 >= m) { s1 = Gm; b1 = 0.f; }
        const float loglam = logmu + Gm;
        const bool eager = fabsf(loglam) > kMaxLogScale;
        const bool ulast = start + m >= len;
        if (ulast && nxt < 0) nxt = take_unit();
        const bool slast = ulast && nxt >= total_units;
        const float b0c = b0, b1c = b1;
        // the K / Q ring slot of chunk g-3 was released
        if (g >= 3) ok = wait(B_KQE0 + g % 3, ((g / 3) + 1) & 1, 0);
        GDN_TRACE(0, g, 0);
        if (!ok) break;
        float* sc = slot_sc(g);
        sc[SC_G + lane] = s0;
        sc[SC_G + lane + 32] = s1;
        sc[SC_B + lane] = b0c;
        sc[SC_B + lane + 32] = b1c;
        __syncwarp();  // every lane's scalars before lane 0's arrive publishes them
        const int row = (int)(bos + start);
        if (lane == 0) {
          sc[SC_GMAX] = gmax;
          sc[SC_GMIN] = gmin;
          sc[SC_GM] = Gm;
          sc[SC_LAMLOG] = eager ? 0.f : loglam;
          sc[SC_NULOG] = eager ? -Gm : logmu;
          const float lam = exp2f(loglam * kLog2e);
          sc[SC_RMW] = eager ? lam : 1.f;
          sc[SC_MUNEXT] = eager ? 1.f : lam;
          sc[SC_M] = __int_as_float(m);
          sc[SC_FLAGS] = __int_as_float((ulast ? F_ULAST : 0) | (eager ? F_EAGER : 0) |
                                        (cu == 0 ? F_UFIRST : 0) | (slast ? F_SLAST : 0) |
                                        (cu == 0 && zstart ? F_ZFIRST : 0) | (vzero ? F_VZERO : 0) |
                                        (noout ? F_NOOUT : 0));
          *reinterpret_cast<long long*>(&sc[SC_T0]) = (long long)(bos + start);
          sc[SC_N] = __int_as_float(n);
          sc[SC_H] = __int_as_float(h);
          // the arrive publishes the scalars; the K / Q tiles complete the phase (a chunk of
          // no rows at the end of the tensor reads zeros)
          uint64_t* full = &bars[B_FULL0 + g % 3];
          mbar_arrive_expect_tx(full, kq_bytes);
          const uint32_t kq = slot_kq(g);
#pragma unroll 1
          for (int a = 0; a < 2 * L::NKA; ++a)  // K, Q per atom column
            tma_load_3d(sm + (kq - sbase) + (a >> 1) * 16384 + (a & 1) * 8192, (a & 1) ? &tm.q : &tm.k, full,
                        64 * (a >> 1), hq, row);
        }
        __syncwarp();
        kq_issued = g + 1;
        GDN_TRACE(0, g, 1);
        // V has its own ring (two slots, released by chunk g-2's U product) and barrier, so
        // the K / Q tiles above never wait for it
        if (g >= 2) ok = wait(B_VE0 + (g & 1), ((g >> 1) + 1) & 1, 0);
        if (!ok) break;
        if (lane == 0) {
          uint64_t* vfull = &bars[B_VFULL0 + (g & 1)];
          if (vzero) {
            mbar_arrive(vfull);  // no tile: the U product is skipped
          } else {
            mbar_arrive_expect_tx(vfull, v_bytes);
            const uint32_t vv = slot_v(g);
#pragma unroll 1
            for (int a = 0; a < L::NVA; ++a) tma_load_3d(sm + (vv - sbase) + a * 8192, &tm.v, vfull, 64 * a, h, row);
          }
        }
        __syncwarp();
        v_issued = g + 1;
        GDN_TRACE(0, g, 2);
        if (ulast) {
          ++g;
          break;
        }
        start += m;
        logmu = eager ? 0.f : loglam;
      }
      if (nxt >= total_units) break;
      cur = nxt;
      nxt = -1;
    }
    // let every requested tile land before the CTA can exit (on the normal path
    // they were all consumed and these return at once)
    if (lane == 0) drain_loads(sbase + L::BARS, kq_issued, v_issued, sbase + L::MISC);
  } else if (warp == 1) {
    // ================================================================ state-independent MMAs
    // W'^T = K^T T_w^T and U^T = V^T T_b^T of chunk c once WG-A has written T_b / T_w
    // (warp 3 issues the chunks' [K;Q] K^T, so these never wait for later tiles).
    if (lane == 0 && any) {
      constexpr uint32_t id_w = idesc_bf16(128, 64, 1, 0);
#pragma unroll 1
      for (int c = 0;; ++c) {
        GDN_TRACE(1, c, 0);
        const int par = c & 1;
        // R and the W' accumulator were read by WG-B for chunk c-1
        uint64_t wl = with(kNone, B_T_READY0 + par, (c >> 1) & 1);
        if (c >= 1) wl = with(with(wl, B_R_FREE, (c - 1) & 1), B_W_FREE, (c - 1) & 1);
        if (!wait_all(wl, 10)) break;
        GDN_TRACE(1, c, 1);
        tc_fence_after();
        const uint32_t kq = slot_kq(c), vv = slot_v(c);
        const uint32_t lbo_k = (L::NKA == 2) ? 16384u : (sbase + L::ZERO - kq);
        const uint64_t dka = sdesc(kq, lbo_k, 1024), dtw = sdesc(sbase + L::TW, 16, 1024);
        const int fl = sc_int(slot_sc(c), SC_FLAGS);
        if (!(fl & F_ZFIRST)) {  // W' only meets a nonzero state
#pragma unroll 1
          for (int k = 0; k < 4; ++k)
            mma_ss(tmem + TM_W, sdesc_add(dka, k * 2048u), sdesc_add(dtw, k * 32u), id_w, k != 0);
        }
        mma_commit(&bars[B_W_DONE]);  // W'^T may be converted while U is still running
        GDN_TRACE(1, c, 2);
        if (!wait(B_VFULL0 + par, (c >> 1) & 1, 10)) break;
        GDN_TRACE(1, c, 3);
        tc_fence_after();
        const uint32_t lbo_v = (L::NVA == 2) ? 8192u : (sbase + L::ZERO - vv);
        const uint64_t dva = sdesc(vv, lbo_v, 1024), dtb = sdesc(sbase + L::TB, 16, 1024);
        if (!(SEG && (fl & F_VZERO))) {  // V = 0: U = 0, and U' starts from -W' S~
#pragma unroll 1
          for (int kk = 0; kk < 8; ++kk)  // T_b hi, then lo
            mma_ss(tmem + TM_R, sdesc_add(dva, (kk & 3) * 2048u), sdesc_add(dtb, (kk >> 2) * 8192u + (kk & 3) * 32u),
                   id_w, kk != 0);
        }
        mma_commit(&bars[B_U_DONE]);
        mma_commit(&bars[B_VE0 + par]);
        GDN_TRACE(1, c, 4);
        if (fl & F_SLAST) break;
      }
      mma_commit(&bars[B_DRAIN1]);  // every MMA this thread issued has finished before exit
      wait(B_DRAIN1, 0, kDrainWait);
    }
  } else if (warp == 2) {
    // ================================================================ state-dependent MMAs
    if (lane == 0 && any) {
      constexpr uint32_t id_sw = idesc_tf32(128, 64);
      constexpr uint32_t id_qs = idesc_bf16(128, 64, 0, 0);
      constexpr uint32_t id_st = idesc_bf16(128, DK, 0, 1);
      constexpr uint32_t id_pu = idesc_bf16(128, 64, 0, 0);
#pragma unroll 1
      for (int c = 0;; ++c) {
        const int par = c & 1;
        if (!wait_all(with(with(with(kNone, B_P1_DONE0 + par, (c >> 1) & 1), B_WCONV0 + par, (c >> 1) & 1),
                           B_U_DONE, c & 1), 4)) {
          break;
        }
        // U' reads the fp32 state itself: it needs chunk c-1's state update, or, when the
        // state starts over or is rescaled before this chunk, WG-B's write of it
        const int fl = sc_int(slot_sc(c), SC_FLAGS);
        GDN_TRACE(2, c, 0);
        const bool s_written = (fl & (F_UFIRST | F_EAGER)) != 0;
        if (!(s_written ? wait(B_S_READY, c & 1, 4) : wait(B_STATE_DONE, (c - 1) & 1, 4))) break;
        GDN_TRACE(2, c, 1);
        tc_fence_after();
        const bool last = cscal[c % 3].slast;  // read now: the buffer is reused after this chunk
        const uint32_t kq = slot_kq(c);
        // a zero starting state: U' = U, no S~^T Q^T term, and the state update and the
        // output product start their accumulators afresh
        const uint32_t zf = (fl & F_ZFIRST) ? 0u : 1u;
        const uint32_t vz = (SEG && (fl & F_VZERO)) ? 1u : 0u;  // R holds no U: the first product overwrites it
        const bool want_o = !(SEG && (fl & F_NOOUT));           // no output: no output products
        if (zf) {
          // U'^T += S~^T W'^T in tf32: A = S~^T (fp32, TMEM), B = W' fp32 K-major [j][d_k]
          const uint64_t dwt = sdesc(sbase + L::WP, 16, 1024);
#pragma unroll 1
          for (int kk = 0; kk < DK / 8; ++kk)
            mma_ts_tf32(tmem + TM_R, tmem + TM_S + kk * 8u, sdesc_add(dwt, (kk >> 2) * 8192u + (kk & 3) * 32u), id_sw,
                        kk != 0 || !vz);
        }
        mma_commit(&bars[B_UP_DONE]);
        GDN_TRACE(2, c, 2);
        // O^T = S~^T Q^T (raw q tile, K-major) from the bf16 copy of the state, once the
        // last epilogue has read O
        uint64_t ol = with(kNone, B_S_READY, c & 1);
        if (c >= 1) ol = with(ol, B_EPI_DONE, (c - 1) & 1);
        if (!wait_all(ol, 4)) break;
        GDN_TRACE(2, c, 3);
        tc_fence_after();
        if (zf && want_o) {
          const uint64_t dq = sdesc(kq + 8192u, 16, 1024);
#pragma unroll 1
          for (int kk = 0; kk < 4 * L::NKA; ++kk)
            mma_ts(tmem + TM_O, tmem + TM_SB + kk * 8u, sdesc_add(dq, (kk >> 2) * 16384u + (kk & 3) * 32u),
                   id_qs, kk != 0);
        }
        if (!wait(B_UOPS_READY, c & 1, 7)) {
          break;
        }
        GDN_TRACE(2, c, 4);
        tc_fence_after();
        // S~^T += (U' s)^T K : A from TMEM (hi, then lo), B = K MN-major (N = d_k)
        const uint64_t dkn = sdesc(kq, (L::NKA == 2) ? 16384u : 16u, 1024);
#pragma unroll 1
        for (int kk = 0; kk < 8; ++kk)  // hi (kk < 4), then lo
          mma_ts(tmem + TM_S, tmem + TM_UH + kk * 8u, sdesc_add(dkn, (kk & 3) * 2048u), id_st, kk != 0 || zf);
        mma_commit(&bars[B_STATE_DONE]);
        GDN_TRACE(2, c, 5);
        // O^T += (U' s)^T M^T : B = M K-major [i][j]; the hi part of U' s only, since
        // this term reaches the output alone (M itself is bf16)
        const uint64_t dm = sdesc(sbase + L::M0 + par * 8192u, 16, 1024);
        if (want_o) {
#pragma unroll 1
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(tmem + TM_O, tmem + TM_UH + kk * 8u, sdesc_add(dm, kk * 32u), id_pu, kk != 0 || zf);
        }
        mma_commit(&bars[B_O_DONE]);
        mma_commit(&bars[B_MFREE0 + par]);
        GDN_TRACE(2, c, 6);
        if (last) break;
      }
      mma_commit(&bars[B_DRAIN2]);
      wait(B_DRAIN2, 0, kDrainWait);
    }
  } else if (warp == 3) {
    // ================================================================ q norms
    // Lane 0 issues [K;Q] K^T of each chunk (tcgen05) as soon as its tiles are in and
    // WG-A has read the previous chunk's. Then r^q_i from the diagonal of Q Q^T, 16 rows
    // at a time on the warp-level tensor cores (bf16 products are exact in fp32), straight
    // from the swizzled tile and off the path of the chunk preparation (r^q only weights
    // the output rows).
    if (any) {
      const int g = lane >> 2, t = lane & 3;
      // ldmatrix rows: matrices 0 / 1 are rows 0-7 / 8-15 of k 0-7, 2 / 3 the same of k 8-15
      const uint32_t lr = (uint32_t)((lane & 7) + 8 * ((lane >> 3) & 1)), lk = (uint32_t)(lane >> 4);
      constexpr uint32_t id_kq = idesc_bf16(128, 64, 0, 0);
#pragma unroll 1
      for (int c = 0;; ++c) {
        bool ok = true;
        if (lane == 0) {
          ok = wait(B_FULL0 + c % 3, (c / 3) & 1, 14) && (c == 0 || wait(B_KQ_FREE, (c - 1) & 1, 14));
          if (ok) {
            tc_fence_after();
            const uint64_t dkq = sdesc(slot_kq(c), 16, 1024);
#pragma unroll 1
            for (int kk = 0; kk < 4 * L::NKA; ++kk) {
              const uint64_t d = sdesc_add(dkq, (kk >> 2) * 16384u + (kk & 3) * 32u);
              mma_ss(tmem + TM_KQ, d, d, id_kq, kk != 0);
            }
            mma_commit(&bars[B_KQ_DONE]);
            GDN_TRACE(3, c, 0);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        float* sc = slot_sc(c);
        const uint32_t qa = slot_kq(c) + 8192u;  // Q atom 0 (atom a at + 16384 a)
        const int nrb = (SEG && (sc_int(sc, SC_FLAGS) & F_NOOUT)) ? 0 : 4;  // r^q only weights outputs
#pragma unroll 1
        for (int rb = 0; rb < nrb; ++rb) {
          const uint32_t r = 16u * rb + lr;
          float d0[4] = {}, d1[4] = {};  // columns 0-7 and 8-15 of the 16 x 16 block
#pragma unroll
          for (int s = 0; s < 4 * L::NKA; ++s) {
            uint32_t a0, a1, a2, a3;
            ldmatrix_x4(qa + (uint32_t)(s >> 2) * 16384u + sw128(r, 2u * (s & 3) + lk), a0, a1, a2, a3);
            mma_bf16_16816(d0, a0, a1, a2, a3, a0, a2);  // B = rows 0-7 of the block
            mma_bf16_16816(d1, a0, a1, a2, a3, a1, a3);  // B = rows 8-15
          }
          if (t == (g >> 1)) {  // this lane holds (g, g) and (g + 8, g + 8)
            const float q0 = (g & 1) ? d0[1] : d0[0], q1 = (g & 1) ? d1[3] : d1[2];
            sc[SC_RQ + 16 * rb + g] = p.l2norm ? 1.0f / sqrtf(q0 + 1e-6f) : 1.f;
            sc[SC_RQ + 16 * rb + g + 8] = p.l2norm ? 1.0f / sqrtf(q1 + 1e-6f) : 1.f;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_RQ0 + c % 3]);
        GDN_TRACE(3, c, 1);
        if (sc_int(sc, SC_FLAGS) & F_SLAST) break;
      }
      if (lane == 0) {  // every MMA this thread issued has finished before exit
        mma_commit(&bars[B_DRAIN3]);
        wait(B_DRAIN3, 0, kDrainWait);
      }
    }
  } else if (warp < 12) {
    // ================================================================ WG-A: chunk preparation
    const int wa = tid - 128;         // 0..255
    const int Ln = wa & 127;          // TMEM lane
    const int hf = wa >> 7;           // which 32-column half of a 64-wide block
    const uint32_t lane_off = (uint32_t)((Ln & ~31) << 16);
    const bool krow = Ln < 64;
    const int i = Ln & 63;
    if (any) {
#pragma unroll 1
      for (int c = 0;; ++c) {
        const int par = c & 1;
        // the chunk's tiles and [K;Q] K^T; M, W'^T / A and the chunk scalars of this parity
        // released by chunk c-2 / c-3 (the q norms only weight the output rows: the
        // epilogue applies them)
        uint64_t wl = with(with(kNone, B_FULL0 + c % 3, (c / 3) & 1), B_KQ_DONE, c & 1);
        if (c >= 2) wl = with(wl, B_MFREE0 + par, ((c >> 1) + 1) & 1);
        if (c >= 3) wl = with(wl, B_CSF0 + c % 3, ((c / 3) + 1) & 1);
        bool ok = wait_all(wl, 8);
        GDN_TRACE(4, c, 0);
        if (named_bar_or(1, 256, !ok || *abort_flag)) break;
        tc_fence_after();
        const float* sc = slot_sc(c);
        ChunkScalars& cs = cscal[c % 3];
        const int m = sc_int(sc, SC_M);
        const bool last = sc_int(sc, SC_FLAGS) & F_SLAST;
        const float gmax = sc[SC_GMAX], Gm = sc[SC_GM], lamlog = sc[SC_LAMLOG];
        const float Gi = sc[SC_G + i];
        uint32_t v[32];  // row Ln of [K;Q] K^T, columns [32 hf, 32 hf + 32)
        tmem_ld32(tmem + lane_off + TM_KQ + 32 * hf, v);
        tmem_ld_wait();
        tc_fence_before();
        float* Abuf = reinterpret_cast<float*>(sm + L::AS);
        float* Tbuf = reinterpret_cast<float*>(sm + L::TB);
        if (krow && (i >> 5) == hf) {
          // r^k_i from the diagonal of K K^T (fp32 sum of exact bf16 products), then the
          // per-row scalars of the A / T_w / state-update weights
          float diag = 0.f;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j == (i & 31)) diag = __uint_as_float(v[j]);
          const float ri = p.l2norm ? 1.0f / sqrtf(diag + 1e-6f) : 1.f;
          const float bi = sc[SC_B + i];
          const bool live = i < m;
          ps->d[i] = live ? ri * exp2f((gmax - Gi) * kLog2e) : 0.f;
          ps->r[i] = ri;
          ps->beta[i] = bi;
          ps->tw[i] = live ? -bi * ri * exp2f((Gi + sc[SC_NULOG]) * kLog2e) : 0.f;
          ps->s[i] = live ? ri * exp2f((Gm - Gi - lamlog) * kLog2e) : 0.f;
        } else if (!krow && hf == 0) {
          // output weights
          cs.co[i] = i < m ? p.scale * exp2f((Gi - Gm + lamlog) * kLog2e) : 0.f;
          if (i == 0) {
            cs.t0 = *reinterpret_cast<const long long*>(&sc[SC_T0]);
            cs.mu_next = sc[SC_MUNEXT];
            cs.m = m;
            cs.slast = last ? 1 : 0;
            cs.n = sc_int(sc, SC_N);
            cs.h = sc_int(sc, SC_H);
          }
        }
        named_bar_sync(1, 256);
        if (wa == 0) mbar_arrive(&bars[B_KQ_FREE]);  // [K;Q] K^T is in registers
        GDN_TRACE(4, c, 1);
        // A above the block diagonal (rows 0-31, columns 32-63) is never read, and M there is
        // always zero (cleared once at the start): those two warps have nothing to write
        const bool upper = hf == 1 && (Ln & 63) < 32;
        if (krow && !upper) {
          // A_ij = beta_i r_i r_j e^{G_i - G_j} k_i.k_j, fp32 into the scratch (0 in rows and
          // columns past m). The solve reads only j < i, so entries on and above the diagonal
          // are stored as computed, unmasked.
          const float cia = i < m ? ps->beta[i] * ps->r[i] * exp2f((Gi - gmax) * kLog2e) : 0.f;
          const float2 ci2 = make_float2(cia, cia);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int j0 = 32 * hf + 4 * q;
            const float4 d4 = *reinterpret_cast<const float4*>(&ps->d[j0]);
            const float2 a01 = __fmul2_rn(__fmul2_rn(ci2, make_float2(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]))),
                                          make_float2(d4.x, d4.y));
            const float2 a23 = __fmul2_rn(__fmul2_rn(ci2, make_float2(__uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]))),
                                          make_float2(d4.z, d4.w));
            *reinterpret_cast<float4*>(&Abuf[i * LDF + j0]) = make_float4(a01.x, a01.y, a23.x, a23.y);
          }
        } else if (!krow && !upper && !(SEG && (sc_int(sc, SC_FLAGS) & F_NOOUT))) {
          // M_ij = q_i.k_j  (j <= i), bf16 K-major [i][j]
          const uint32_t mrow = sbase + L::M0 + par * 8192u;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int j0 = 32 * hf + 8 * q;
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w4[e] = pack_bf16(j0 + 2 * e <= i ? __uint_as_float(v[8 * q + 2 * e]) : 0.f,
                                j0 + 2 * e + 1 <= i ? __uint_as_float(v[8 * q + 2 * e + 1]) : 0.f);
            st_shared_v4(mrow + sw128(i, 4 * hf + q), w4[0], w4[1], w4[2], w4[3]);
          }
        }
        fence_proxy_async_smem();
        GDN_TRACE(4, c, 2);
        // T_b / T_w of chunk c-1 have been read by its W and U products (the solve
        // overwrites them); A is complete once every thread passes this barrier
        ok = c < 1 || wait(B_U_DONE, (c - 1) & 1, 9);
        if (named_bar_or(1, 256, !ok || *abort_flag)) break;
        GDN_TRACE(4, c, 3);
        // ---- T = (I + A)^-1
        solve_unit_lower(Abuf, Tbuf, wa);
        GDN_TRACE(4, c, 4);
        // ---- T_b = T diag(beta) as bf16 hi + lo; T_w = T diag(tw)
        {
          const int ti = wa & 63, qq = wa >> 6;  // row ti, columns [16 qq, 16 qq + 16)
          // row ti carries the state-update weight s_ti (so U' and W' come out of their
          // products already multiplied by diag(s / lambda))
          const float si = zero_row(ps->s[ti], qq > (ti >> 4));
          const float2 si2 = make_float2(si, si);
          float2 t[8];
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const float4 x = *reinterpret_cast<const float4*>(&Tbuf[ti * LDF + 16 * qq + 4 * k4]);
            t[2 * k4] = __fmul2_rn(si2, make_float2(x.x, x.y));
            t[2 * k4 + 1] = __fmul2_rn(si2, make_float2(x.z, x.w));
          }
          named_bar_sync(1, 256);  // every thread has read T before it is overwritten
          const uint32_t tb = sbase + L::TB;
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int j0 = 16 * qq + 8 * q;
            const float4 ba = *reinterpret_cast<const float4*>(&ps->beta[j0]);
            const float4 bb = *reinterpret_cast<const float4*>(&ps->beta[j0 + 4]);
            const float4 wa4 = *reinterpret_cast<const float4*>(&ps->tw[j0]);
            const float4 wb4 = *reinterpret_cast<const float4*>(&ps->tw[j0 + 4]);
            const float2 bt[4] = {make_float2(ba.x, ba.y), make_float2(ba.z, ba.w), make_float2(bb.x, bb.y),
                                  make_float2(bb.z, bb.w)};
            const float2 wt[4] = {make_float2(wa4.x, wa4.y), make_float2(wa4.z, wa4.w), make_float2(wb4.x, wb4.y),
                                  make_float2(wb4.z, wb4.w)};
            uint32_t hi4[4], lo4[4], w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 x = __fmul2_rn(t[4 * q + e], bt[e]);
              hi4[e] = pack_bf16(x.x, x.y);
              lo4[e] = pack_bf16_2(bf16_residual(x, hi4[e]));
              const float2 w = __fmul2_rn(t[4 * q + e], wt[e]);
              w4[e] = pack_bf16(w.x, w.y);
            }
            const uint32_t off = sw128(ti, 2 * qq + q);
            st_shared_v4(tb + off, hi4[0], hi4[1], hi4[2], hi4[3]);
            st_shared_v4(tb + 8192u + off, lo4[0], lo4[1], lo4[2], lo4[3]);
            st_shared_v4(sbase + L::TW + off, w4[0], w4[1], w4[2], w4[3]);
          }
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 256);
        // ---- W'^T = K^T T_w^T and U^T = V^T T_b^T, issued from here
        // T_b / T_w go to warp 1's W and U products; the chunk's scalars and M to the
        // state step (WG-B converts W'^T)
        if (wa == 0) {
          mbar_arrive(&bars[B_T_READY0 + par]);
          mbar_arrive(&bars[B_P1_DONE0 + par]);
          GDN_TRACE(4, c, 5);
        }
        if (last) break;
      }
    }
  } else {
    // ================================================================ WG-B: state step + epilogue
    const int wb = tid - 384;  // == TMEM lane == d_v index
    const uint32_t lane_off = (uint32_t)((wb & ~31) << 16);
    const bool live = wb < DV;
    // A unit's final state S = mu S~, once its last S~ update has finished; in a tree
    // launch the unit's children may then start from it.
    auto store_final = [&](int un, int uh, float umu) {
      if (!p.final_state) return;
      if (!GDN_IN_BOUNDS(p.status, un >= 0 && un < p.num_seqs && uh >= 0 && uh < p.h_v, 0x103u)) return;
      float* fs = p.final_state + ((size_t)un * p.h_v + uh) * DK * DV;
#pragma unroll 1
      for (int xb = 0; xb < DK / 32; ++xb) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + TM_S + xb * 32, v);
        tmem_ld_wait();
        if (live) {
#pragma unroll
          for (int x = 0; x < 32; ++x) fs[(size_t)(xb * 32 + x) * DV + wb] = umu * __uint_as_float(v[x]);
        }
      }
      if (p.parent) {
        named_bar_sync(2, 128);  // every thread's stores before the release
        if (wb == 0) release_flag(&p.ready[(size_t)un * p.h_v + uh]);  // (un, uh checked above)
      }
    };
    // A unit's starting state -> S~^T in TMEM (lane d_v, column d_k), mu = 1: an
    // initial-state slot or zero, or in a tree launch a child's parent's final state once
    // the parent's unit has released it. False if that wait gave up.
    auto load_initial = [&](int un, int uh) {
      const int par = tree_parent(p, un);
      if (par >= 0) {
        bool ok = true;
        if (wb == 0) {
          ok = wait_flag(&p.ready[(size_t)par * p.h_v + uh], kWaitLimitNs);
          if (!ok && !*abort_flag) {
            *abort_flag = 1;
            report(p.status, GDN_ERR_DEVICE_TIMEOUT, blockIdx.x * 16u + 5u);
          }
        }
        if (named_bar_or(2, 128, !ok)) return false;
      }
      const int64_t slot = state_slot(p, un);
      const float* s0 = par >= 0 ? p.final_state + ((size_t)par * p.h_v + uh) * DK * DV
                                 : (slot >= 0 ? p.initial_state + ((size_t)slot * p.h_v + uh) * DK * DV : nullptr);
      if (s0 && !GDN_IN_BOUNDS(p.status,
                               uh >= 0 && uh < p.h_v && (par >= 0 ? par < p.num_seqs : slot < p.num_state_slots),
                               0x104u))
        s0 = nullptr;
      if (!s0) return true;  // a zero state: the first state update overwrites S~ outright
#pragma unroll 1
      for (int xb = 0; xb < DK / 32; ++xb) {
        uint32_t v[32];
#pragma unroll
        for (int x = 0; x < 32; ++x)
          v[x] = (s0 && live) ? __float_as_uint(s0[(size_t)(xb * 32 + x) * DV + wb]) : 0u;
        tmem_st32(tmem + lane_off + TM_S + xb * 32, v);
      }
      tmem_st_wait();
      return true;
    };
    int un_c = 0, uh_c = 0;  // the unit of the chunk whose state step ran last,
    float mu_c = 1.f;        // and mu after it
    constexpr size_t osz = OF32 ? 4 : 2;
    const int pieces = (int)(DV * osz / 16);  // 16-byte pieces of one output row
    const int pshift = __ffs(pieces) - 1;
    uint32_t npass = 0;  // epilogue passes so far (selects the staging tile)
    // The K/Q slot whose staged output tiles a tensor store may still be reading (thread
    // 0 of the group issued the store): it goes back to the producer at the next wait
    // for a U' product, where the group waits anyway.
    int slot_pending = -1;
    auto release_slot = [&]() {
      if (wb == 0 && slot_pending >= 0) {
        bulk_wait_read();
        mbar_arrive(&bars[B_KQE0 + slot_pending % 3]);
      }
      slot_pending = -1;
    };
#pragma unroll 1
    for (int c = -1;; ++c) {
      bool more = any && c < 0;
      if (c >= 0) {
        // ---- (U' diag(s/lambda))^T -> bf16 hi / lo A operands
        const ChunkScalars& cs = cscal[c % 3];
        release_slot();
        bool ok = wait_all(with(with(kNone, B_P1_DONE0 + (c & 1), (c >> 1) & 1), B_UP_DONE, c & 1), 12);
        if (named_bar_or(2, 128, !ok || *abort_flag)) break;
        tc_fence_after();
        GDN_TRACE(12, c, 0);
#pragma unroll 1
        for (int hb = 0; hb < 2; ++hb) {  // columns j in [32 hb, 32 hb + 32)
          uint32_t u[32];
          tmem_ld32(tmem + lane_off + TM_R + hb * 32, u);
          tmem_ld_wait();
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            const float2 x2 = make_float2(__uint_as_float(u[2 * x]), __uint_as_float(u[2 * x + 1]));
            hi[x] = pack_bf16(x2.x, x2.y);
            lo[x] = pack_bf16_2(bf16_residual(x2, hi[x]));
          }
          tmem_st16(tmem + lane_off + TM_UH + hb * 16, hi);
          tmem_st16(tmem + lane_off + TM_UL + hb * 16, lo);
        }
        tmem_st_wait();
        tc_fence_before();
        named_bar_sync(2, 128);
        if (wb == 0) {
          mbar_arrive(&bars[B_R_FREE]);
          mbar_arrive(&bars[B_UOPS_READY]);
          GDN_TRACE(12, c, 1);
        }
        more = !cs.slast;
        un_c = cs.n;
        uh_c = cs.h;
        mu_c = cs.mu_next;
      }
      if (more) {
        // ---- W'^T of chunk c+1: TMEM -> fp32 K-major [j][d_k] with the 128-byte swizzle
        // (32 fp32 per row of an atom), the B operand of warp 2's tf32 U' product. Right
        // after the split: it does not depend on the state, and the U' product of chunk
        // c+1 needs it as soon as chunk c's state update is done. Thread d_k writes column
        // d_k of every row j: a warp fills one 128-byte atom row per store, in 32 banks.
        const int cn = c + 1, pn = cn & 1;
        bool ok = wait(B_W_DONE, cn & 1, 15);
        if (named_bar_or(2, 128, !ok || *abort_flag)) break;
        tc_fence_after();
        GDN_TRACE(12, c + 1, 2);
        // (chunk c's U' product, the buffer's last reader, finished before the split above)
        const uint32_t wcol = sbase + L::WP + (uint32_t)(wb >> 5) * 8192u + (uint32_t)(wb & 3) * 4u;
        const uint32_t wch = (uint32_t)((wb >> 2) & 7);  // 16-byte chunk of the row before the swizzle
        const bool wz = sc_int(slot_sc(cn), SC_FLAGS) & F_ZFIRST;  // no U' product reads it
#pragma unroll 1
        for (int hb = 0; hb < (wz ? 0 : 2); ++hb) {
          uint32_t w[32];
          tmem_ld32(tmem + lane_off + TM_W + 32 * hb, w);
          tmem_ld_wait();
          if (wb < DK) {
#pragma unroll
            for (int x = 0; x < 32; ++x)
              asm volatile("st.shared.b32 [%0], %1;" ::"r"(wcol + (uint32_t)(32 * hb + x) * 128u +
                                                            ((wch ^ (uint32_t)(x & 7)) << 4)),
                           "r"(w[x])
                           : "memory");
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        named_bar_sync(2, 128);
        if (wb == 0) {
          mbar_arrive(&bars[B_W_FREE]);
          mbar_arrive(&bars[B_WCONV0 + pn]);
          GDN_TRACE(12, c + 1, 3);
        }
      }
      if (more || c >= 0) {
        // ---- S~ -> bf16 A operand for chunk c+1 (first applying its decay when eager).
        // After the CTA's last chunk (no chunk c+1) only the final state of its unit is
        // stored here, once chunk c's S~ update has finished.
        const int cn = c + 1;
        const float* sc = slot_sc(cn);
        uint64_t wl = more ? with(kNone, B_FULL0 + cn % 3, (cn / 3) & 1) : kNone;
        if (c >= 0) wl = with(wl, B_STATE_DONE, c & 1);
        bool ok = wait_all(wl, 11);
        if (named_bar_or(2, 128, !ok || *abort_flag)) break;
        tc_fence_after();
        GDN_TRACE(12, c + 1, 4);
        if (!more || (sc_int(sc, SC_FLAGS) & F_UFIRST)) {
          // chunk cn starts a unit (or there is none): the one that ended with chunk c is complete
          if (c >= 0) store_final(un_c, uh_c, mu_c);
          if (more && !load_initial(sc_int(sc, SC_N), sc_int(sc, SC_H))) break;
        }
      }
      if (more) {
        const int cn = c + 1;
        const float* sc = slot_sc(cn);
        const bool eager = sc_int(sc, SC_FLAGS) & F_EAGER;
        const float rmw = sc[SC_RMW];
        // the bf16 copy only feeds S~^T Q^T, which a zero state or a unit without output skips;
        // the decay of an eager chunk is applied all the same
        const bool sb = !(sc_int(sc, SC_FLAGS) & (F_ZFIRST | (SEG ? F_NOOUT : 0)));
#pragma unroll 1
        for (int xb = 0; xb < (sb || eager ? DK / 32 : 0); ++xb) {
          uint32_t va[32];
          tmem_ld32(tmem + lane_off + TM_S + xb * 32, va);
          tmem_ld_wait();
          if (eager) {
#pragma unroll
            for (int x = 0; x < 32; ++x) va[x] = __float_as_uint(__uint_as_float(va[x]) * rmw);
            tmem_st32(tmem + lane_off + TM_S + xb * 32, va);
          }
          if (sb) {
            uint32_t pk[16];
#pragma unroll
            for (int x = 0; x < 16; ++x) pk[x] = pack_bf16(__uint_as_float(va[2 * x]), __uint_as_float(va[2 * x + 1]));
            tmem_st16(tmem + lane_off + TM_SB + xb * 16, pk);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        named_bar_sync(2, 128);
        if (wb == 0) mbar_arrive(&bars[B_S_READY]);
        GDN_TRACE(12, c + 1, 5);
      }
      if (c >= 0) {
        // ---- epilogue: out_i = co_i O^T_i, staged in shared memory and written by tensor
        // stores. bf16: the whole chunk at once, as two 64-column tiles of 64 rows (128-byte
        // swizzle), one store each; fp32: passes of 16 rows alternating between two tiles.
        // A chunk (or pass) shorter than the tile is copied out row by row instead, since a
        // store of the full tile would run into the next sequence's rows. The tiles sit in
        // the chunk's own K/Q slot: once O is complete, every product that reads the chunk's
        // K and Q tiles has finished; the slot goes back to the producer when the stores
        // have read the tiles.
        // The q norms of the chunk (warp 3) complete the row weights here; once they are
        // written, warp 3 has also finished reading the chunk's Q tile.
        const ChunkScalars& cs = cscal[c % 3];
        bool ok = wait_all(with(with(kNone, B_O_DONE, c & 1), B_RQ0 + c % 3, (c / 3) & 1), 13);
        if (named_bar_or(2, 128, !ok || *abort_flag)) break;
        tc_fence_after();
        GDN_TRACE(12, c, 6);
        const int m = cs.m;
        const long long t0 = cs.t0;
        const uint32_t stg = slot_kq(c);
        const float* rq = slot_sc(c) + SC_RQ;
        if (SEG && (sc_int(slot_sc(c), SC_FLAGS) & F_NOOUT)) {
          // nothing to write: the chunk's buffers go straight back
          if (wb == 0) {
            mbar_arrive(&bars[B_EPI_DONE]);
            mbar_arrive(&bars[B_CSF0 + c % 3]);
            mbar_arrive(&bars[B_KQE0 + c % 3]);
          }
        } else if constexpr (!OF32) {
          // each thread takes consecutive row pairs of its 16-lane blocks (16 x 256b loads)
          // and writes 8x8 blocks transposed into the row-major tiles (the eight rows of a
          // block hit distinct banks under the swizzle); a tile row is 32 half + lane
          const int qd = wb >> 5, t = lane & 3;
          const uint32_t tile = stg + (uint32_t)(qd >> 1) * 8192u;
#pragma unroll 1
          for (int half = 0; half < 2 && 32 * half < m; ++half) {
            const int p0 = 32 * half;
            uint32_t a[16], b[16];
            tmem_ld16x256b_x4(tmem + ((uint32_t)(32 * qd) << 16) + TM_O + p0, a);
            tmem_ld16x256b_x4(tmem + ((uint32_t)(32 * qd + 16) << 16) + TM_O + p0, b);
            tmem_ld_wait();
            if (32 * qd < DV) {
              float2 co2[4];
#pragma unroll
              for (int r = 0; r < 4; ++r)
                co2[r] = __fmul2_rn(*reinterpret_cast<const float2*>(&cs.co[p0 + 8 * r + 2 * t]),
                                    *reinterpret_cast<const float2*>(&rq[p0 + 8 * r + 2 * t]));
#pragma unroll
              for (int hs = 0; hs < 4; ++hs) {  // lane half (hs >> 1) and 8-lane block (hs & 1)
                const uint32_t* x = (hs >> 1) ? b : a;
                const int o = 2 * (hs & 1);
                uint32_t pk[4];
#pragma unroll
                for (int r = 0; r < 4; ++r)
                  pk[r] = pack_bf16_2(__fmul2_rn(co2[r], make_float2(__uint_as_float(x[4 * r + o]),
                                                                      __uint_as_float(x[4 * r + o + 1]))));
                stmatrix_x4_trans(tile + sw128((uint32_t)(p0 + lane), (uint32_t)(4 * (qd & 1) + hs)), pk[0], pk[1],
                                  pk[2], pk[3]);
              }
            }
          }
          tc_fence_before();
          fence_proxy_async_smem();
          named_bar_sync(2, 128);  // tiles written, O and the chunk's scalars read
          if (wb == 0) {
            mbar_arrive(&bars[B_EPI_DONE]);
            mbar_arrive(&bars[B_CSF0 + c % 3]);
          }
          GDN_TRACE(12, c, 7);
          if (m == 64) {
            if (wb == 0) {
#pragma unroll
              for (int tl = 0; tl < DV / 64; ++tl)
                tma_store_3d(&tm.o, sm + (stg - sbase) + tl * 8192, 64 * tl, cs.h, (int)t0);
              bulk_commit();
            }
            slot_pending = c;
          } else {
            for (int idx = wb; idx < (m << pshift); idx += 128) {
              const int r = idx >> pshift, pc = idx & (pieces - 1);
              const uint4 x = *reinterpret_cast<const uint4*>(
                  sm + (stg - sbase) + (pc >> 3) * 8192 + sw128((uint32_t)r, (uint32_t)(pc & 7)));
              char* dst = reinterpret_cast<char*>(p.out) + (((size_t)(t0 + r) * p.h_v + cs.h) * DV) * osz;
              if (GDN_IN_BOUNDS(p.status, t0 + r < p.total_tokens && cs.h < p.h_v, 0x105u))
                *reinterpret_cast<uint4*>(dst + pc * 16) = x;
            }
            named_bar_sync(2, 128);  // every thread has read the tiles
            if (wb == 0) mbar_arrive(&bars[B_KQE0 + c % 3]);
          }
        } else {
#pragma unroll 1
          for (int p0 = 0; p0 < m; p0 += 16, ++npass) {
            uint8_t* stage = sm + (stg - sbase) + (npass & 1) * 8192u;
            // the store that last used this tile has read it (one store group per pass)
            if (wb == 0) bulk_wait_read_1();
            named_bar_sync(2, 128);
            uint32_t oa[16];
            tmem_ld16(tmem + lane_off + TM_O + p0, oa);
            tmem_ld_wait();
            if (live) {
#pragma unroll
              for (int t4 = 0; t4 < 4; ++t4) {
                const float4 c4w = *reinterpret_cast<const float4*>(&cs.co[p0 + 4 * t4]);
                const float4 r4 = *reinterpret_cast<const float4*>(&rq[p0 + 4 * t4]);
                const float4 c4 = make_float4(c4w.x * r4.x, c4w.y * r4.y, c4w.z * r4.z, c4w.w * r4.w);
                float* st = reinterpret_cast<float*>(stage) + (4 * t4) * DV + wb;
                st[0] = c4.x * __uint_as_float(oa[4 * t4]);
                st[DV] = c4.y * __uint_as_float(oa[4 * t4 + 1]);
                st[2 * DV] = c4.z * __uint_as_float(oa[4 * t4 + 2]);
                st[3 * DV] = c4.w * __uint_as_float(oa[4 * t4 + 3]);
              }
            }
            fence_proxy_async_smem();
            named_bar_sync(2, 128);
            const int rows = m - p0 < 16 ? m - p0 : 16;
            if (rows == 16) {
              if (wb == 0) tma_store_3d(&tm.o, stage, 0, cs.h, (int)(t0 + p0));
            } else {
              for (int idx = wb; idx < (rows << pshift); idx += 128) {
                const int r = idx >> pshift, pc = idx & (pieces - 1);
                const uint4 x = *reinterpret_cast<const uint4*>(stage + r * DV * 4 + pc * 16);
                char* dst = reinterpret_cast<char*>(p.out) + (((size_t)(t0 + p0 + r) * p.h_v + cs.h) * DV) * osz;
                if (GDN_IN_BOUNDS(p.status, t0 + p0 + r < p.total_tokens && cs.h < p.h_v, 0x106u))
                  *reinterpret_cast<uint4*>(dst + pc * 16) = x;
              }
            }
            if (wb == 0) bulk_commit();  // empty for a copied pass
          }
          tc_fence_before();
          named_bar_sync(2, 128);
          if (wb == 0) {
            mbar_arrive(&bars[B_EPI_DONE]);
            mbar_arrive(&bars[B_CSF0 + c % 3]);
          }
          slot_pending = c;  // released once the stores have read the tiles
        }
      }
      if (!more) break;
    }
    release_slot();
    if (wb == 0) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
#ifdef GDN_TC_TRACE
  if (tid == 0 && (int)blockIdx.x == g_gdn_trace_cta) {
    g_gdn_trace[16 * 2048 + 2] = clock64();
    g_gdn_trace[16 * 2048 + 3] = globaltimer();
  }
#endif
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

// out [T, H, D] for tensor stores: bf16 as 64 columns x 1 head x 64 rows with 128-byte swizzle
// (one staging tile per 64 columns of a chunk); fp32 as D x 1 x 16 rows, unswizzled.
bool encode_out(CUtensorMap* m, void* base, int64_t T, int H, int D, bool f32) {
  auto fn = get_encode();
  if (!fn) return false;
  const cuuint64_t es = f32 ? 4 : 2;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)D * es, (cuuint64_t)H * D * es};
  cuuint32_t box[3] = {f32 ? (cuuint32_t)D : 64u, 1, f32 ? 16u : 64u};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims,
            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            f32 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


template <int DK, int DV, bool OF32, bool GF32, int MODE>
cudaError_t launch_tc_dk(const Params& p, cudaStream_t stream) {
  using L = TcLayout<DK, DV>;
  Tmaps tm;
  if (!encode_rows(&tm.q, p.q, p.total_tokens, p.h_qk, DK) ||
      !encode_rows(&tm.k, p.k, p.total_tokens, p.h_qk, DK) ||
      !encode_rows(&tm.v, p.v, p.total_tokens, p.h_v, DV) ||
      !encode_out(&tm.o, p.out, p.total_tokens, p.h_v, DV, p.out_f32 != 0))
    return cudaErrorInvalidValue;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(&gdn_tc_kernel<DK, DV, OF32, GF32, MODE>), (int)L::DYN_SMEM);
  if (e != cudaSuccess) return e;
  const long long units = (long long)p.num_seqs * p.h_v;
  if (units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  // one resident CTA per SM (the kernel's shared memory and TMEM fill an SM), each
  // taking units until the work list is exhausted
  int sms = 0;
  e = device_sm_count(&sms);
  if (e != cudaSuccess) return e;
  const long long grid = units < sms ? units : sms;
  // launched as a programmatic dependent of the prep kernel, so that its set-up overlaps it
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = L::DYN_SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = MODE == 2 ? 0 : 1;  // a direct launch follows a memset, not the prep kernel
  e = cudaLaunchKernelEx(&cfg, gdn_tc_kernel<DK, DV, OF32, GF32, MODE>, p, tm);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc(const Params& p, cudaStream_t stream) {
  if (p.total_tokens <= 0) return launch_simt(p, stream);  // only empty sequences: state copy
  if (p.total_tokens > 0x7fffffffLL) return cudaErrorInvalidValue;
  // output and gate storage types are template parameters, so that each kernel carries
  // only the code of its own types
  const int t = (p.out_f32 ? 2 : 0) + (p.gate_f32 ? 1 : 0);
  auto by_types = [&](auto dk, auto dv) {
    constexpr int K_ = decltype(dk)::value, V_ = decltype(dv)::value;
    // segment and direct launches (square states only) take their own instances
    constexpr bool SQ = K_ == V_;
    constexpr int SEGM = SQ ? 1 : 0, DIRM = SQ ? 2 : 0;
    if (SQ && p.seq_rows) {
      switch (t) {
        case 0: return launch_tc_dk<K_, V_, false, false, SEGM>(p, stream);
        case 1: return launch_tc_dk<K_, V_, false, true, SEGM>(p, stream);
        case 2: return launch_tc_dk<K_, V_, true, false, SEGM>(p, stream);
        default: return launch_tc_dk<K_, V_, true, true, SEGM>(p, stream);
      }
    }
    if (SQ && p.direct) {
      switch (t) {
        case 0: return launch_tc_dk<K_, V_, false, false, DIRM>(p, stream);
        case 1: return launch_tc_dk<K_, V_, false, true, DIRM>(p, stream);
        case 2: return launch_tc_dk<K_, V_, true, false, DIRM>(p, stream);
        default: return launch_tc_dk<K_, V_, true, true, DIRM>(p, stream);
      }
    }
    switch (t) {
      case 0: return launch_tc_dk<K_, V_, false, false, 0>(p, stream);
      case 1: return launch_tc_dk<K_, V_, false, true, 0>(p, stream);
      case 2: return launch_tc_dk<K_, V_, true, false, 0>(p, stream);
      default: return launch_tc_dk<K_, V_, true, true, 0>(p, stream);
    }
  };
  using I64 = std::integral_constant<int, 64>;
  using I128 = std::integral_constant<int, 128>;
  if (p.d_k == 128 && p.d_v == 128) return by_types(I128{}, I128{});
  if (p.d_k == 64 && p.d_v == 64) return by_types(I64{}, I64{});
  if (p.d_k == 128 && p.d_v == 64) return by_types(I128{}, I64{});
  return by_types(I64{}, I128{});
}

}  // namespace gdn

#ifdef GDN_TC_TRACE
// Accessors of the tracing build (declared in include/gdn_trace.h).
extern "C" int gdn_trace_set_cta(int cta) {
  return (int)cudaMemcpyToSymbol(gdn::g_gdn_trace_cta, &cta, sizeof(int));
}
extern "C" int gdn_trace_clear(void) {
  static unsigned long long zeros[16 * 2048 + 4];
  return (int)cudaMemcpyToSymbol(gdn::g_gdn_trace, zeros, sizeof(zeros));
}
extern "C" int gdn_trace_read(unsigned long long* host) {
  if (cudaDeviceSynchronize() != cudaSuccess) return 1;
  return (int)cudaMemcpyFromSymbol(host, gdn::g_gdn_trace, sizeof(unsigned long long) * (16 * 2048 + 4));
}
#endif
