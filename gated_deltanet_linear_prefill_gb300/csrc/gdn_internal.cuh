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

__device__ __forceinline__ float load_gate(const void* p, int64_t idx, int is_f32) {
  return is_f32 ? reinterpret_cast<const float*>(p)[idx]
                : __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[idx]);
}

// Rows [bos, eos) of sequence n, clamped into [0, T] so that a malformed
// cu_seqlens (reported by the prep kernel) can never send a load out of bounds.
__device__ __forceinline__ void seq_bounds(const Params& p, int n, int64_t& bos, int64_t& eos) {
  int64_t b = p.cu_seqlens[n], e = p.cu_seqlens[n + 1];
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

}  // namespace gdn
