// Segment scan of one long sequence: the plan, the set-up kernel and the
// composition of the segments' state maps.
//
// The gated delta rule S_t = exp(g_t) (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
// (S is d_k x d_v; "Gated Delta Networks", reference [5] of the open-jev-fast README)
// is affine in the starting state: over a run of rows it maps S to Phi S + Delta, where Phi
// (d_k x d_k) is what the run makes of S = I with every v_t = 0, and Delta is
// what it makes of S = 0 with the true v_t. The chunk kernel computes both as
// ordinary runs, and S_{j+1} = Phi_j S_j + Delta_j chains them.
#include <algorithm>
#include <functional>
#include <mutex>
#include <queue>
#include <vector>

#include "gdn_internal.cuh"

namespace gdn {

namespace {

// Longest-first list scheduling of whole units (sizes in chunks) on `sms` SMs: the
// makespan the persistent chunk kernel's work list gives, in chunk periods.
int64_t lpt_makespan(std::vector<int64_t> units, int sms) {
  std::sort(units.begin(), units.end(), [](int64_t x, int64_t y) { return x > y; });
  std::priority_queue<int64_t, std::vector<int64_t>, std::greater<int64_t>> load;
  for (int i = 0; i < (sms > 0 ? sms : 1); ++i) load.push(0);
  int64_t span = 0;
  for (int64_t u : units) {
    const int64_t t = load.top() + u;
    load.pop();
    load.push(t);
    span = t > span ? t : span;
  }
  return span;
}

int64_t chunks_of(int64_t rows) { return (rows + kChunk - 1) / kChunk; }

}  // namespace

static SegPlan seg_plan_search(int64_t T, int h_v, int sms) {
  SegPlan best{0, T, 0};
  const int64_t serial = chunks_of(T);
  // the extra launches (set-up, a second prep + chunk launch, the composition) cost
  // about four chunk periods
  constexpr int64_t kOverhead = 4;
  int64_t best_cost = serial * 85 / 100 - kOverhead;
  for (int G = 3; G <= kSegMaxG; ++G) {
    for (int ratio = 2; ratio <= 4; ++ratio) {  // a = b * ratio / 4
      // a + (G - 1) b = T with b a multiple of the chunk: segment 0 takes the rest
      const double bf = (double)T / ((double)(G - 1) + ratio / 4.0);
      const int64_t b = ((int64_t)bf + kChunk - 1) / kChunk * kChunk;
      const int64_t a = T - (int64_t)(G - 1) * b;
      const int64_t a_rows = a > 0 ? a : 0;
      if (a_rows < kChunk) continue;
      const int64_t last = T - a_rows - (int64_t)(G - 2) * b;
      if (last < 1) continue;
      std::vector<int64_t> ua, uc;
      for (int h = 0; h < h_v; ++h) {
        ua.push_back(chunks_of(a_rows));
        for (int j = 1; j <= G - 2; ++j) {
          ua.push_back(chunks_of(b));  // Delta_j
          ua.push_back(chunks_of(b));  // Phi_j
        }
        for (int j = 1; j <= G - 2; ++j) uc.push_back(chunks_of(b));
        uc.push_back(chunks_of(last));
      }
      const int64_t cost = lpt_makespan(ua, sms) + lpt_makespan(uc, sms);
      if (cost < best_cost) {
        best_cost = cost;
        best = SegPlan{G, a_rows, b};
      }
    }
  }
  return best;
}

SegPlan seg_plan(int64_t T, int h_v, int sms) {
  // the last plan is kept: a caller usually repeats one shape (one call per layer)
  static std::mutex mu;
  static int64_t kT = -1;
  static int kh = -1, ks = -1;
  static SegPlan kp{0, 0, 0};
  std::lock_guard<std::mutex> lock(mu);
  if (T != kT || h_v != kh || sms != ks) {
    kp = seg_plan_search(T, h_v, sms);
    kT = T;
    kh = h_v;
    ks = sms;
  }
  return kp;
}

namespace {

// Block 0 resets the status word, checks the caller's cu_seqlens and state_index and
// writes the row and slot tables of both launches. The other blocks write the two state
// slots, kSetupSplit blocks per (slot, head): slot 0 the caller's starting state of the
// sequence (or nothing, when it starts from zero), slot 1 the identity.
constexpr int kSetupSplit = 8;
__global__ void gdn_seg_setup_kernel(Params p, SegPlan plan, float* slots, int64_t* rows_a, int64_t* rows_c,
                                     int32_t* sidx_a) {
  const int G = plan.G;
  const int64_t a = plan.a, b = plan.b, T = p.total_tokens;
  // the caller's slot for sequence 0 (-1: zero state; -2: out of range, reported below)
  int32_t slot = -1;
  if (p.initial_state) {
    slot = p.state_index ? p.state_index[0] : 0;
    if (slot < -1 || slot >= p.num_state_slots) slot = -2;
  }
  if (blockIdx.x == 0) {
    if (threadIdx.x == 0) {
      p.status->code = 0u;
      p.status->detail = 0u;
      p.status->units_done = 0u;
      p.status->next_unit = 0u;
      if (p.cu_seqlens[0] != 0 || p.cu_seqlens[1] != T || (p.max_seqlen > 0 && T > p.max_seqlen))
        report(p.status, GDN_ERR_SEQLENS, 0u);
      if (slot == -2) report(p.status, GDN_ERR_STATE_INDEX, 0u);
    }
    // launch A: segment 0 (true state), Delta_1 .. Delta_{G-2}, Phi_1 .. Phi_{G-2}
    for (int n = threadIdx.x; n < 2 * G - 3; n += blockDim.x) {
      int64_t r0, r1;
      int32_t si;
      if (n == 0) {
        r0 = 0;
        r1 = a;
        si = slot >= 0 ? 0 : -1;
      } else {
        const int j = n <= G - 2 ? n : n - (G - 2);
        r0 = a + (int64_t)(j - 1) * b;
        r1 = r0 + b;
        si = n <= G - 2 ? -1 : 1;
      }
      rows_a[2 * n] = r0;
      rows_a[2 * n + 1] = r1;
      sidx_a[n] = si;
    }
    // launch C: segments 1 .. G-1 (b rows each; the last ends at T)
    for (int n = threadIdx.x; n < G - 1; n += blockDim.x) {
      const int64_t r0 = a + (int64_t)n * b;
      rows_c[2 * n] = r0;
      rows_c[2 * n + 1] = n == G - 2 ? T : r0 + b;
    }
    return;
  }
  const int blk = blockIdx.x - 1, part = blk % kSetupSplit, sh = blk / kSetupSplit;
  const int s = sh / p.h_v, h = sh % p.h_v;
  if (s == 0 && slot < 0) return;
  const int rows = p.d_k / kSetupSplit, v4 = p.d_v / 4;  // float4 per row
  const size_t sz = (size_t)p.d_k * p.d_v;
  float4* dst = reinterpret_cast<float4*>(slots + ((size_t)s * p.h_v + h) * sz) + (size_t)part * rows * v4;
  const float4* src = s == 0 ? reinterpret_cast<const float4*>(p.initial_state + ((size_t)slot * p.h_v + h) * sz) +
                                   (size_t)part * rows * v4
                             : nullptr;
  for (int i = threadIdx.x; i < rows * v4; i += blockDim.x) {
    if (src) {
      dst[i] = src[i];
    } else {
      const int r = part * rows + i / v4, c = 4 * (i % v4);  // the identity: 1 where c == r
      dst[i] = make_float4(r == c ? 1.f : 0.f, r == c + 1 ? 1.f : 0.f, r == c + 2 ? 1.f : 0.f, r == c + 3 ? 1.f : 0.f);
    }
  }
}

// Block (h, slice): S_1 = fin_a[0] and S_{j+1} = Phi_j S_j + Delta_j on the 32 columns
// [32 slice, 32 slice + 32) of head h (a column slice of S depends only on the same slice
// of the previous S). Phi_j is staged transposed in shared memory; thread (rg, cg) keeps
// rows [4 rg, 4 rg + 4) of columns [4 cg, 4 cg + 4) (2 DK threads). fp32 throughout.
constexpr int kCombCols = 32;
template <int DK>
__global__ void __launch_bounds__(2 * DK) gdn_seg_combine_kernel(Params p, SegPlan plan, const float* fin_a,
                                                                 float* s_c) {
  constexpr int kCombThreads = 2 * DK, R = 4, LDT = DK + 4;
  extern __shared__ float4 comb_smem4[];
  float* pht = reinterpret_cast<float*>(comb_smem4);  // Phi_j^T [DK][LDT]: pht[m][r] = Phi_j[r][m]
  float* sj = pht + DK * LDT;                          // S_j slice [DK][32]
  const int G = plan.G, dv = p.d_v;
  const int nsl = dv / kCombCols;
  const int h = blockIdx.x / nsl, c0 = (blockIdx.x % nsl) * kCombCols;
  const size_t sz = (size_t)DK * dv, hs = (size_t)p.h_v * sz;
  const int tid = threadIdx.x, cg = tid % 8, rg = tid / 8;
  const float* s1 = fin_a + (size_t)h * sz;
  constexpr int NS = DK * 8 / kCombThreads;      // float4 pieces of the slice per thread
  constexpr int NP = DK * DK / 4 / kCombThreads;  // float4 pieces of Phi_j per thread
  // Phi_j and Delta_j of the next step are loaded into registers while the current
  // step computes (all of a step's loads in flight at once). Piece u of Phi_j holds
  // Phi_j[r][m .. m+3] with r = i % DK, i = tid + u * threads: a warp covers 32 rows,
  // so that its transposed stores fill 32 banks.
  float4 pf[NP], pd[R];
  auto load_step = [&](int j) {
    const float* phi = fin_a + (size_t)(G - 2 + j) * hs + (size_t)h * sz;  // Phi_j [DK][DK]
    const float* del = fin_a + (size_t)j * hs + (size_t)h * sz;             // Delta_j [DK][d_v]
#pragma unroll
    for (int u = 0; u < NP; ++u) {
      const int i = tid + u * kCombThreads;
      pf[u] = *reinterpret_cast<const float4*>(&phi[(size_t)(i % DK) * DK + 4 * (i / DK)]);
    }
#pragma unroll
    for (int i = 0; i < R; ++i)
      pd[i] = *reinterpret_cast<const float4*>(&del[(size_t)(R * rg + i) * dv + c0 + 4 * cg]);
  };
  float4 xs[NS];
#pragma unroll
  for (int u = 0; u < NS; ++u) {
    const int i = tid + u * kCombThreads, r = i / 8, q = i % 8;
    xs[u] = *reinterpret_cast<const float4*>(&s1[(size_t)r * dv + c0 + 4 * q]);
  }
  if (G >= 3) load_step(1);
#pragma unroll
  for (int u = 0; u < NS; ++u) {
    const int i = tid + u * kCombThreads, r = i / 8, q = i % 8;
    *reinterpret_cast<float4*>(&sj[r * kCombCols + 4 * q]) = xs[u];
    *reinterpret_cast<float4*>(&s_c[(size_t)h * sz + (size_t)r * dv + c0 + 4 * q]) = xs[u];
  }
  for (int j = 1; j <= G - 2; ++j) {
    __syncthreads();  // the previous Phi is no longer read; S_j is in place
#pragma unroll
    for (int u = 0; u < NP; ++u) {
      const int i = tid + u * kCombThreads, r = i % DK, m = 4 * (i / DK);
      pht[(m + 0) * LDT + r] = pf[u].x;
      pht[(m + 1) * LDT + r] = pf[u].y;
      pht[(m + 2) * LDT + r] = pf[u].z;
      pht[(m + 3) * LDT + r] = pf[u].w;
    }
    float acc[R][4];
#pragma unroll
    for (int i = 0; i < R; ++i) {
      acc[i][0] = pd[i].x;
      acc[i][1] = pd[i].y;
      acc[i][2] = pd[i].z;
      acc[i][3] = pd[i].w;
    }
    __syncthreads();
    if (j + 1 <= G - 2) load_step(j + 1);
#pragma unroll 8
    for (int m = 0; m < DK; ++m) {
      const float4 x = *reinterpret_cast<const float4*>(&sj[m * kCombCols + 4 * cg]);
      const float4 f = *reinterpret_cast<const float4*>(&pht[m * LDT + R * rg]);
      const float fr[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc[k][0] = fmaf(fr[k], x.x, acc[k][0]);
        acc[k][1] = fmaf(fr[k], x.y, acc[k][1]);
        acc[k][2] = fmaf(fr[k], x.z, acc[k][2]);
        acc[k][3] = fmaf(fr[k], x.w, acc[k][3]);
      }
    }
    __syncthreads();  // every thread has read S_j
    float* out = s_c + (size_t)j * hs + (size_t)h * sz;
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const float4 y = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
      *reinterpret_cast<float4*>(&sj[(R * rg + i) * kCombCols + 4 * cg]) = y;
      *reinterpret_cast<float4*>(&out[(size_t)(R * rg + i) * dv + c0 + 4 * cg]) = y;
    }
  }
}

}  // namespace

cudaError_t launch_seg_setup(const Params& p, const SegPlan& plan, const SegLayout& L, char* ws,
                             cudaStream_t stream) {
  if (p.d_k % kSetupSplit != 0 || p.d_v % 4 != 0) return cudaErrorInvalidValue;
  const long long blocks = 1 + 2LL * p.h_v * kSetupSplit;
  gdn_seg_setup_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
      p, plan, reinterpret_cast<float*>(ws + L.slots), reinterpret_cast<int64_t*>(ws + L.rows_a),
      reinterpret_cast<int64_t*>(ws + L.rows_c), reinterpret_cast<int32_t*>(ws + L.sidx_a));
  return cudaGetLastError();
}

cudaError_t launch_seg_combine(const Params& p, const SegPlan& plan, const SegLayout& L, char* ws,
                               cudaStream_t stream) {
  if (p.d_k != p.d_v || p.d_v % kCombCols != 0 || (p.d_k != 64 && p.d_k != 128)) return cudaErrorInvalidValue;
  const long long blocks = (long long)p.h_v * (p.d_v / kCombCols);
  const float* fin = reinterpret_cast<const float*>(ws + L.fin_a);
  float* sc = reinterpret_cast<float*>(ws + L.s_c);
  auto go = [&](auto kern, int dk) {
    const int smem = (int)sizeof(float) * (dk * (dk + 4) + dk * kCombCols);
    const cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)blocks, 2 * dk, smem, stream>>>(p, plan, fin, sc);
    return cudaGetLastError();
  };
  return p.d_k == 128 ? go(gdn_seg_combine_kernel<128>, 128) : go(gdn_seg_combine_kernel<64>, 64);
}

}  // namespace gdn
