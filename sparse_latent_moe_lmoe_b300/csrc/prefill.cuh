// Argument block and launchers of the prefill-path kernels (many tokens).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "decode.cuh"

namespace lmoe {

struct PrefillArgs {
  int d, E, G, k, L, f, r, epg;
  const float* W_r;
  const float* b_r;
  const uint16_t* W_r_split;  // [3][E][d] bf16: W_r = hi + mid + lo
  const uint8_t* W_in_q;
  const uint16_t* W_in_s;
  const uint8_t* W_out_q;
  const uint16_t* W_out_s;
  const uint8_t* gate_q;
  const uint16_t* gate_s;
  const uint8_t* up_q;
  const uint16_t* up_s;
  const uint8_t* down_q;
  const uint16_t* down_s;
  const uint16_t* A_in;
  const uint16_t* B_in;
  const uint16_t* A_out;
  const uint16_t* B_out;
  // weight format (LMOE_WEIGHTS_*); NVFP4: E4M3 bytes behind the *_s pointers
  // and the per-tensor fp32 scales
  int wfmt;
  const float* W_in_gs;
  const float* W_out_gs;
  const float* gate_gs;
  const float* up_gs;
  const float* down_gs;
  unsigned* err;
  int num_sms;
  long long timeout;
  // the handle's second stream and its fork / join events (null: everything on the caller's stream)
  cudaStream_t aux;
  cudaEvent_t ev_fork, ev_join;
};

// W_r fp32 [E][d] -> three bf16 matrices whose sum is W_r (to fp32 rounding).
cudaError_t launch_split_router(const float* W_r, int E, int d, uint16_t* out, cudaStream_t st);

bool prefill_supported(const PrefillArgs& P);
cudaError_t prefill_set_attributes();
size_t prefill_workspace_bytes(const PrefillArgs& P, int T);
cudaError_t launch_prefill_route(const PrefillArgs& P, const uint16_t* x, int T, int32_t* idx, float* w,
                                 float* logits, void* ws, cudaStream_t st);
cudaError_t launch_prefill_experts(const PrefillArgs& P, const uint16_t* x, int T, const int32_t* idx, const float* w,
                                   const PermPtrs& perm, float* Yrows, const uint16_t* residual, uint16_t* y,
                                   void* ws, cudaStream_t st);
cudaError_t launch_prefill_layer(const PrefillArgs& P, const uint16_t* x, int T, const uint16_t* residual,
                                 uint16_t* y, void* ws, cudaStream_t st, const std::vector<cudaEvent_t>* events);
// The layer in token chunks sharing one dequantisation: the fp16 weights into
// a workspace laid out for layout_T tokens, then the layer on T <= layout_T
// tokens in that workspace (any number of times, in stream order)
cudaError_t launch_prefill_weights(const PrefillArgs& P, int layout_T, void* ws, cudaStream_t st);
cudaError_t launch_prefill_layer_chunk(const PrefillArgs& P, const uint16_t* x, int T, int layout_T,
                                       const uint16_t* residual, uint16_t* y, void* ws, cudaStream_t st);
const char* prefill_stage_name(const PrefillArgs& P, int T, int i, int* count);
// kernels launched by launch_prefill_layer
int prefill_launch_count(const PrefillArgs& P, int T);

}  // namespace lmoe
