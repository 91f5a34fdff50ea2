// Internal declarations shared by the C ABI (gdn_api.cu) and the kernels.
// Not part of the public interface (include/gdn.h is).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

// Chunk length of the chunked form (open-jev-fast README, Phase 3 item 1 and
// "Limits": the cost is per 64-token chunk).
constexpr int kChunk = 64;

// Workspace layout (all offsets 256-byte aligned):
//   [0, 256)           Status: the device status word and diagnostics
//   [256, 256 + 4*N)   the sequence order, longest first (int32)
struct Status {
  uint32_t code;       // first gdn_status a kernel reported (0 = none)
  uint32_t detail;     // the sequence or unit it concerns
  uint32_t units_done;
  uint32_t next_unit;  // tree launches: work counter (units are taken in order)
  uint32_t pad[60];
};
static_assert(sizeof(Status) == 256, "status block is 256 bytes");

constexpr size_t kOrderOffset = 256;

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline size_t workspace_bytes(int num_seqs) {
  return kOrderOffset + round_up(sizeof(int32_t) * (size_t)(num_seqs > 0 ? num_seqs : 1), 256);
}

// A tree launch adds, after the work list, one ready flag (uint32) per
// (sequence, value head): set once that unit's final state is written.
inline size_t tree_flags_offset(int num_seqs) { return workspace_bytes(num_seqs); }
inline size_t tree_workspace_bytes(int num_seqs, int h_v) {
  const size_t units = (size_t)(num_seqs > 0 ? num_seqs : 1) * (size_t)(h_v > 0 ? h_v : 1);
  return tree_flags_offset(num_seqs) + round_up(sizeof(uint32_t) * units, 256);
}

// Everything a kernel needs, passed by value.
struct Params {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const void* g;
  const void* beta;
  const int32_t* cu_seqlens;
  const float* initial_state;
  const int32_t* state_index;
  void* out;
  float* final_state;
  Status* status;
  const int32_t* order;  // sequences, longest first (tree launches: parents before children)
  const int32_t* parent; // tree launches only (else NULL): parent[n] in [-1, n)
  uint32_t* ready;       // tree launches only: ready flag per (sequence, value head)
  // Segment launches of one long sequence (else NULL / num_seqs / num_seqs / 0): the rows
  // of virtual sequence n are [seq_rows[2n], seq_rows[2n+1]) (sequences may share rows);
  // sequences n >= vzero_from read V as zero; only sequences n < out_upto write out;
  // keep_status leaves the status word to the launch that set it up.
  const int64_t* seq_rows;
  int vzero_from;
  int out_upto;
  int keep_status;
  // Direct launch (a small batch, no prep kernel): CTA b takes unit b (grid = units), the
  // units in index order, and checks its own sequence's cu_seqlens / state_index entries;
  // the host has zeroed the status word.
  int direct;
  int64_t total_tokens;
  int num_seqs;
  int max_seqlen;
  int h_qk, h_v, d_k, d_v;
  int num_state_slots;
  int gate_f32;
  int out_f32;
  int l2norm;
  float scale;
};

__device__ __forceinline__ void report(Status* st, uint32_t code, uint32_t detail) {
  if (atomicCAS(&st->code, 0u, code) == 0u) st->detail = detail;
}

// Bounds checks of the bounds-checked build (-DGDN_CHECKED, libgdn_checked.so, the
// stand-in for a memory checker): a failed check reports GDN_ERR_BOUNDS with the site
// as detail, and the access it guards is skipped. The regular build compiles the
// checks away: there every index is in range by construction (clamped bounds, guards).
__device__ __forceinline__ bool check_bounds(Status* st, bool ok, uint32_t site) {
  if (!ok) report(st, GDN_ERR_BOUNDS, site);
  return ok;
}
#ifdef GDN_CHECKED
#define GDN_IN_BOUNDS(status, cond, site) ::gdn::check_bounds((status), (cond), (site))
#else
#define GDN_IN_BOUNDS(status, cond, site) true
#endif

__device__ __forceinline__ float load_gate(const void* p, int64_t idx, int is_f32) {
  return is_f32 ? reinterpret_cast<const float*>(p)[idx]
                : __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[idx]);
}

// Rows [bos, eos) of sequence n, clamped into [0, T] so that a malformed
// cu_seqlens (reported by the prep kernel) can never send a load out of bounds.
__device__ __forceinline__ void seq_bounds(const Params& p, int n, int64_t& bos, int64_t& eos) {
  int64_t b = p.seq_rows ? p.seq_rows[2 * n] : p.cu_seqlens[n];
  int64_t e = p.seq_rows ? p.seq_rows[2 * n + 1] : p.cu_seqlens[n + 1];
  b = b < 0 ? 0 : (b > p.total_tokens ? p.total_tokens : b);
  e = e < b ? b : (e > p.total_tokens ? p.total_tokens : e);
  bos = b;
  eos = e;
}

// Parent of sequence n in a tree launch, or -1 (no parent, not a tree launch, or
// an index outside [-1, n), which the prep kernel reports).
__device__ __forceinline__ int tree_parent(const Params& p, int n) {
  if (!p.parent) return -1;
  const int32_t pa = p.parent[n];
  return (pa >= 0 && pa < n) ? pa : -1;
}

// Initial-state slot of sequence n, or -1 for a zero state (an out-of-range
// index was reported by the prep kernel and reads as zero here).
__device__ __forceinline__ int64_t state_slot(const Params& p, int n) {
  if (!p.initial_state) return -1;
  int64_t s = p.state_index ? (int64_t)p.state_index[n] : (int64_t)n;
  return (s >= 0 && s < p.num_state_slots) ? s : -1;
}

// Raises a kernel's dynamic shared-memory limit once per (kernel, device), so
// that a launch made during stream capture issues no attribute calls.
cudaError_t set_smem_once(const void* kernel, int bytes);

// Streaming multiprocessors of the current device (cached per device).
cudaError_t device_sm_count(int* out);

// Launchers (each returns the launch's cudaError_t).
cudaError_t launch_prep(const Params& p, cudaStream_t stream);
cudaError_t launch_simt(const Params& p, cudaStream_t stream);
cudaError_t launch_tc(const Params& p, cudaStream_t stream);

// ---- segment scan of one long sequence
//
// A single sequence of T rows leaves most SMs idle (one chain of chunks per value
// head). The state after each segment is an affine map of the state before it,
// S -> Phi_j S + Delta_j, so the sequence is cut into G segments (segments 1 .. G-1 of
// b rows each, segment 0 the a = T - (G-1) b before them) and run in two chunk-kernel
// launches:
//   A: segment 0 from the true starting state (its outputs are final), Delta_j (segments
//      1 .. G-2 from a zero state) and Phi_j (the same segments with V = 0 from S = I);
//   combine: S_1 = state after segment 0, S_{j+1} = Phi_j S_j + Delta_j;
//   C: segments 1 .. G-1 from S_1 .. S_{G-1}: their outputs and the final state.
struct SegPlan {
  int G;       // segments (0: run the sequence in one launch)
  int64_t a;   // rows of segment 0
  int64_t b;   // rows of every later segment (a + (G-1) b = T)
};
constexpr int kSegMaxG = 8;
constexpr int64_t kSegMinTokens = 4096;

// Byte offsets of the segment buffers after the work list (256-byte aligned), sized for
// kSegMaxG segments: two state slots (the gathered starting state, the identity), the
// launch-A final states, the states S_1 .. S_{G-1}, and the row / slot tables.
struct SegLayout {
  size_t slots, fin_a, s_c, rows_a, rows_c, sidx_a, end;
};
inline SegLayout seg_layout(int h_v, int d_k, int d_v) {
  const size_t sb = (size_t)h_v * d_k * d_v * 4;
  SegLayout L;
  L.slots = workspace_bytes(1);
  L.fin_a = L.slots + 2 * sb;
  L.s_c = L.fin_a + (size_t)(2 * kSegMaxG - 3) * sb;
  L.rows_a = L.s_c + (size_t)(kSegMaxG - 1) * sb;
  L.rows_c = L.rows_a + round_up(sizeof(int64_t) * 2 * (2 * kSegMaxG - 3), 256);
  L.sidx_a = L.rows_c + round_up(sizeof(int64_t) * 2 * (kSegMaxG - 1), 256);
  L.end = L.sidx_a + round_up(sizeof(int32_t) * (2 * kSegMaxG - 3), 256);
  return L;
}
// Whether a descriptor of one sequence may take the segment scan (the workspace size
// then includes SegLayout): the tensor-core kernel, square states, a long sequence.
inline bool seg_eligible(const gdn_desc* d) {
  return d && d->num_seqs == 1 && !(d->flags & (GDN_FLAG_SIMT | GDN_FLAG_NO_SEGMENT)) && d->d_k == d->d_v &&
         d->total_tokens >= kSegMinTokens && d->h_v >= 1;
}
// The plan for one sequence of T rows on `sms` SMs: the segment count and lengths that
// minimise the two launches' makespan (longest-first list scheduling of whole units,
// in chunk periods), or G = 0 when one launch is as fast.
SegPlan seg_plan(int64_t T, int h_v, int sms);
// Launch set-up (one kernel): status reset, checks of the caller's cu_seqlens and
// state_index, the slot states, the row tables and slot table of both launches.
cudaError_t launch_seg_setup(const Params& p, const SegPlan& plan, const SegLayout& L, char* ws,
                             cudaStream_t stream);
// S_1 = fin_a[0]; S_{j+1} = Phi_j S_j + Delta_j for j = 1 .. G-2, into s_c[0 .. G-2].
cudaError_t launch_seg_combine(const Params& p, const SegPlan& plan, const SegLayout& L, char* ws,
                               cudaStream_t stream);

}  // namespace gdn
