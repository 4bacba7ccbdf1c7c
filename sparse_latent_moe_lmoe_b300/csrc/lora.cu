// The Recover-LoRA branch around the single-kernel decode pass ("Edge0-145B:
// Run a 145B Open-Source Model on Your Laptop", "The Three Pillars That Make
// It Fast", paragraph "Recover-LoRA": LoRA adapters run as a parallel branch
// beside the frozen 4-bit base). Per group g, with rank r:
//   h  += B_in[g]^T (A_in[g]^T x)      added to H before the expert SwiGLU
//   o  += B_out[g]^T (A_out[g]^T z)    added to the group's W_out output
// The expert work stays in the single kernel; three small kernels surround it:
//   lora_in   P = A_in^T x in row blocks of A_in (partial sums per block); the
//             last block of a group sums them in block order and writes
//             Hl[g][t] = B_in^T P, which the single kernel adds to H
//   lora_q    Q[g][t] = A_out[g]^T Z[g][t], Z as the single kernel wrote it
//             (fp32), for every routed group
//   lora_out  y_t = sum over routed groups in ascending order of
//             (Y[g][t] + B_out[g]^T Q[g][t]) (+ residual), rounded once
#include "common.cuh"
#include "decode.cuh"

namespace lmoe {

namespace {
constexpr int LI_ROWS = 256;  // rows of A_in per lora_in block
constexpr int LQ_COLS = 8;    // columns of Q per lora_q block
constexpr int LO_ROWS = 32;   // output rows per lora_out block
}  // namespace

// grid (G, d / LI_ROWS), 256 threads. Ppart [G][d/LI_ROWS][16][r], P [G][16][r],
// Hl [G][16][L]; tickets[g] zero between calls.
__global__ void __launch_bounds__(256) lora_in_kernel(DecodeArgs A, float* __restrict__ Ppart, float* __restrict__ P,
                                                      float* __restrict__ Hl, unsigned* __restrict__ tickets) {
  extern __shared__ __align__(16) unsigned char lsm[];
  const int g = blockIdx.x, kb = blockIdx.y, nkb = gridDim.y, T = A.T, r = A.r, d = A.d, L = A.L;
  const int tid = threadIdx.x;
  float* xs = reinterpret_cast<float*>(lsm);           // [16][LI_ROWS]
  float* as = xs + 16 * LI_ROWS;                         // [LI_ROWS][r]
  const int k0 = kb * LI_ROWS;
  for (int i = tid; i < 16 * LI_ROWS; i += 256) {
    const int t = i / LI_ROWS, kk = i % LI_ROWS;
    xs[i] = t < T ? bf16_to_f32(A.x[(size_t)t * d + k0 + kk]) : 0.f;
  }
  const uint16_t* Ain = A.A_in + ((size_t)g * d + k0) * r;
  for (int i = tid; i < LI_ROWS * r; i += 256) as[i] = bf16_to_f32(Ain[i]);
  __syncthreads();
  // thread -> (token t, column j) pairs; sums over the block's rows in order
  for (int o = tid; o < 16 * r; o += 256) {
    const int t = o / r, j = o % r;
    float s = 0.f;
    if (t < T)
      for (int kk = 0; kk < LI_ROWS; ++kk) s = fmaf(xs[t * LI_ROWS + kk], as[kk * r + j], s);
    Ppart[(((size_t)g * nkb + kb) * 16 + t) * r + j] = s;
  }
  __threadfence();
  __syncthreads();
  __shared__ int last;
  if (tid == 0) {
    last = atomicAdd(&tickets[g], 1u) == (unsigned)(nkb - 1);
    if (last) tickets[g] = 0;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  // P = sum of the blocks in order, then Hl = B_in^T P
  float* ps = xs;  // [16][r]
  for (int o = tid; o < 16 * r; o += 256) {
    const int t = o / r, j = o % r;
    float s = 0.f;
    for (int b = 0; b < nkb; ++b) s += __ldcg(Ppart + (((size_t)g * nkb + b) * 16 + t) * r + j);
    ps[o] = s;
    P[((size_t)g * 16 + t) * r + j] = s;
  }
  __syncthreads();
  const uint16_t* Bin = A.B_in + (size_t)g * r * L;
  for (int l = tid; l < L; l += 256) {
    float acc[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) acc[t] = 0.f;
    for (int j = 0; j < r; ++j) {
      const float b = bf16_to_f32(Bin[(size_t)j * L + l]);
#pragma unroll
      for (int t = 0; t < 16; ++t) acc[t] = fmaf(b, ps[t * r + j], acc[t]);
    }
#pragma unroll
    for (int t = 0; t < 16; ++t)
      if (t < T) Hl[((size_t)g * 16 + t) * L + l] = acc[t];
  }
}

// bit g: some token routes into group g
LMOE_DEV unsigned long long routed_groups(const DecodeArgs& A) {
  unsigned long long m = 0;
  for (int a = 0; a < A.T * A.k; ++a) m |= 1ull << (A.idx[a] / A.epg);
  return m;
}

// grid (G, r / LQ_COLS), 256 threads. Zlin [G][16][L] (written for routed
// groups), Q [G][16][r].
__global__ void __launch_bounds__(256) lora_q_kernel(DecodeArgs A, const float* __restrict__ Zlin, float* __restrict__ Q) {
  __shared__ float red[8][16][LQ_COLS];
  const int g = blockIdx.x, j0 = blockIdx.y * LQ_COLS, T = A.T, r = A.r, L = A.L;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool routed = (routed_groups(A) >> g) & 1ull;
  // warp w sums rows l = w, w + 8, ...; lane = (token t, column pair)
  float acc[LQ_COLS / 2] = {};
  const int t = lane >> 1, jh = (lane & 1) * (LQ_COLS / 2);
  if (routed && t < T) {
    const uint16_t* Ao = A.A_out + (size_t)g * L * r;
    for (int l = warp; l < L; l += 8) {
      const float z = __ldcg(Zlin + ((size_t)g * 16 + t) * L + l);
#pragma unroll
      for (int q = 0; q < LQ_COLS / 2; ++q) acc[q] = fmaf(z, bf16_to_f32(Ao[(size_t)l * r + j0 + jh + q]), acc[q]);
    }
  }
#pragma unroll
  for (int q = 0; q < LQ_COLS / 2; ++q) red[warp][t][jh + q] = acc[q];
  __syncthreads();
  if (threadIdx.x < 16 * LQ_COLS) {
    const int tt = threadIdx.x / LQ_COLS, j = threadIdx.x % LQ_COLS;
    float s = 0.f;
    for (int w = 0; w < 8; ++w) s += red[w][tt][j];
    if (tt < T) Q[((size_t)g * 16 + tt) * r + j0 + j] = s;
  }
}

// grid d / LO_ROWS, 256 threads: thread (token t, row) of the block.
__global__ void __launch_bounds__(256) lora_out_kernel(DecodeArgs A, const float* __restrict__ Yp,
                                                       const float* __restrict__ Q) {
  __shared__ float qs[16][128];
  const int T = A.T, r = A.r, d = A.d, G = A.G;
  const int row0 = blockIdx.x * LO_ROWS;
  const unsigned long long gm = routed_groups(A);
  float acc[2] = {0.f, 0.f};
  const int rl = threadIdx.x % LO_ROWS, t0 = threadIdx.x / LO_ROWS;  // tokens t0 and t0 + 8
  for (int g = 0; g < G; ++g) {
    if (!((gm >> g) & 1ull)) continue;
    __syncthreads();
    for (int i = threadIdx.x; i < 16 * r; i += 256) qs[i / r][i % r] = __ldcg(Q + (size_t)g * 16 * r + i);
    __syncthreads();
    const uint16_t* Bo = A.B_out + (size_t)g * r * d + row0 + rl;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = t0 + 8 * h;
      if (t >= T) continue;
      float s = __ldcg(Yp + ((size_t)g * 16 + t) * d + row0 + rl);
      for (int j = 0; j < r; ++j) s = fmaf(bf16_to_f32(Bo[(size_t)j * d]), qs[t][j], s);
      acc[h] += s;
    }
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int t = t0 + 8 * h;
    if (t >= T) continue;
    float v = acc[h];
    const size_t o = (size_t)t * d + row0 + rl;
    if (A.residual) v += bf16_to_f32(A.residual[o]);
    A.y[o] = f32_to_bf16_rne(v);
  }
}

size_t lora_in_smem(int r) { return (size_t)(16 * LI_ROWS + LI_ROWS * r) * 4; }

cudaError_t lora_set_attributes() {
  cudaFuncSetAttribute(lora_in_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lora_in_smem(128));
  return cudaGetLastError();
}

bool lora_fused_supported(const DecodeArgs& A) {
  return A.r > 0 && A.r <= 128 && A.r % LQ_COLS == 0 && A.d % LI_ROWS == 0 && A.d % LO_ROWS == 0 && A.G <= 64;
}

cudaError_t launch_lora_in(const DecodeArgs& A, float* Ppart, float* P, float* Hl, unsigned* tickets,
                           cudaStream_t st) {
  lora_in_kernel<<<dim3(A.G, A.d / LI_ROWS), 256, lora_in_smem(A.r), st>>>(A, Ppart, P, Hl, tickets);
  return cudaGetLastError();
}

cudaError_t launch_lora_q(const DecodeArgs& A, const float* Zlin, float* Q, cudaStream_t st) {
  lora_q_kernel<<<dim3(A.G, A.r / LQ_COLS), 256, 0, st>>>(A, Zlin, Q);
  return cudaGetLastError();
}

cudaError_t launch_lora_out(const DecodeArgs& A, const float* Yp, const float* Q, cudaStream_t st) {
  lora_out_kernel<<<A.d / LO_ROWS, 256, 0, st>>>(A, Yp, Q);
  return cudaGetLastError();
}

}  // namespace lmoe
