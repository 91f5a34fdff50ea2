// Launchers of the kernels around the prefill (the input prep and the gated
// RMSNorm), kept apart from the chunk kernel's own declarations.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

// GDN input prep (causal depthwise conv + SiLU + q/k/v split, gate parameters);
// pointers and sizes as in gdn_input_prep, already validated.
struct InputPrepArgs {
  const void* x;
  const float* conv_w;
  const float* conv_bias;
  const int32_t* cu_seqlens;
  const void* conv_state_in;
  const int32_t* state_index;
  const int32_t* parent;  // null: independent sequences
  const void* a;
  const void* b;
  const float* A_log;
  const float* dt_bias;
  void* q;
  void* k;
  void* v;
  float* g;
  float* beta;
  void* conv_state_out;
  int64_t T;
  int N, C, Cq, h_v, K, slots;
};
cudaError_t launch_input_prep(const InputPrepArgs& a, cudaStream_t stream);
// Gated RMSNorm over `rows` rows of d_v (64, 128 or 256) entries; o and y bf16 or
// fp32 (x_f32), z bf16 or fp32 (z_f32), w fp32 [d_v]; nothing is launched for rows <= 0.
cudaError_t launch_gated_rmsnorm(const void* o, const void* z, const float* w, void* y, int64_t rows, int d_v,
                                 bool x_f32, bool z_f32, float eps, cudaStream_t stream);

}  // namespace gdn
