// Prefill path of the latent MoE layer (many tokens): grouped int4-dequant
// GEMMs on the tcgen05 tensor cores.
#include "common.cuh"
#include "prefill.cuh"

namespace lmoe {

// W = hi + mid + lo with each term the bf16 rounding of what remains; the
// three terms carry 24 significant bits, so the split is exact for every
// fp32 value in bf16's normal range.
__global__ void split_router_kernel(const float* __restrict__ W, size_t n, uint16_t* __restrict__ out) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const float v = W[i];
    const uint16_t hi = f32_to_bf16_rne(v);
    const float r1 = v - bf16_to_f32(hi);
    const uint16_t mid = f32_to_bf16_rne(r1);
    const float r2 = r1 - bf16_to_f32(mid);
    out[i] = hi;
    out[n + i] = mid;
    out[2 * n + i] = f32_to_bf16_rne(r2);
  }
}

cudaError_t launch_split_router(const float* W_r, int E, int d, uint16_t* out, cudaStream_t st) {
  const size_t n = (size_t)E * d;
  split_router_kernel<<<296, 256, 0, st>>>(W_r, n, out);
  return cudaGetLastError();
}

bool prefill_available() { return false; }

size_t prefill_workspace_bytes(const PrefillArgs&, int) { return 0; }

cudaError_t launch_prefill_route(const PrefillArgs&, const uint16_t*, int, int32_t*, float*, float*, void*,
                                 cudaStream_t) {
  return cudaErrorNotSupported;
}

cudaError_t launch_prefill_experts(const PrefillArgs&, const uint16_t*, int, const int32_t*, const float*,
                                   const PermPtrs&, float*, const uint16_t*, uint16_t*, void*, cudaStream_t) {
  return cudaErrorNotSupported;
}

cudaError_t launch_prefill_layer(const PrefillArgs&, const uint16_t*, int, const uint16_t*, uint16_t*, void*,
                                 cudaStream_t, const std::vector<cudaEvent_t>*) {
  return cudaErrorNotSupported;
}

const char* prefill_stage_name(const PrefillArgs&, int, int, int* count) {
  if (count) *count = 0;
  return "";
}

}  // namespace lmoe
