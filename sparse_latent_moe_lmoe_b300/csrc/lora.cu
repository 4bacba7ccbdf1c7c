// The Recover-LoRA branch around the single-kernel decode pass ("Edge0-145B:
// Run a 145B Open-Source Model on Your Laptop", "The Three Pillars That Make
// It Fast", paragraph "Recover-LoRA": LoRA adapters run as a parallel branch
// beside the frozen 4-bit base). Per group g, with rank r:
//   h  += B_in[g]^T (A_in[g]^T x)      added to H before the expert SwiGLU
//   o  += B_out[g]^T (A_out[g]^T z)    added to the group's W_out output
// The expert work stays in the single kernel; four small kernels surround it:
//   lora_p    P = A_in^T x: CTA (g, block of 256 rows of A_in) -> a partial;
//             the last CTA of a group sums the partials in block order
//   lora_hl   Hl[g][t] = B_in^T P[g][t] for a block of 128 latent columns,
//             which the single kernel adds to H
//   lora_q    Q[g][t] = A_out[g]^T Z[g][t] from the single kernel's fp32 Z,
//             like lora_p, for the routed groups
//   lora_out  Y[g] += B_out[g]^T Q[g] for (block of 256 output rows, group);
//             the last group of a row block writes y_t = sum over the routed
//             groups in ascending order (+ residual), rounded once
// Each streams its bf16 matrix in whole rows (a warp reads 128 contiguous
// bytes per load, eight loads in flight per lane) and reduces in a fixed order.
// Chained by programmatic dependent launch (unless stage events are being
// recorded between them): each kernel lets its successor launch as soon as
// it starts, the successor waits (griddepcontrol.wait) before it reads what
// the predecessor wrote, and the single kernel waits only where it adds Hl,
// so that its router and W_in work overlap lora_p and lora_hl. A successor
// launches only once every CTA of its predecessor has started, so each
// predecessor runs to completion whatever its successors occupy.
#include "common.cuh"
#include "decode.cuh"

namespace lmoe {

namespace {
constexpr int LP_ROWS = LORA_ROWS;  // rows of A_in / A_out per lora_p / lora_q CTA (8 warps x LP_ROWS / 8)
constexpr int LH_COLS = 128;   // latent columns per lora_hl CTA
constexpr int LO_ROWS = 128;   // output rows per lora_out CTA
constexpr int MAXR = 128;

// bit g: some token routes into group g (every thread of the CTA; the CTA's
// threads load the routing once between them)
LMOE_DEV unsigned long long routed_groups(const DecodeArgs& A) {
  __shared__ unsigned long long m;
  if (threadIdx.x == 0) m = 0ull;
  __syncthreads();
  for (int a = threadIdx.x; a < A.T * A.k; a += blockDim.x) atomicOr(&m, 1ull << (__ldg(A.idx + a) / A.epg));
  __syncthreads();
  return m;
}

LMOE_DEV float2 bf16x2(uint32_t u) { return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u)); }

// Partial of act^T M over rows k0 .. k0 + LP_ROWS of M ([K][r] bf16) for 16
// tokens, act (fp32 in shared memory, [16][LP_ROWS]) -> out [16][r] (fp32,
// global), the 8 warps summed in order. Lane l of a warp takes columns 2l,
// 2l + 1 (a 128-byte row per warp load when r = 64); a warp takes LP_ROWS / 8
// rows.
LMOE_DEV void rows_partial(const uint16_t* __restrict__ M, int r, const float* act, float (*red)[16][MAXR],
                           float* __restrict__ out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float acc[16][2];
#pragma unroll
  for (int t = 0; t < 16; ++t) acc[t][0] = acc[t][1] = 0.f;
  for (int c2 = lane; 2 * c2 < r; c2 += 32) {  // column pairs of this lane (one pass when r <= 64)
#pragma unroll
    for (int t = 0; t < 16; ++t) acc[t][0] = acc[t][1] = 0.f;
#pragma unroll 1
    for (int i0 = 0; i0 < LP_ROWS / 8; i0 += 8) {
      uint32_t w[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        w[u] = __ldg(reinterpret_cast<const uint32_t*>(M + (size_t)(warp * (LP_ROWS / 8) + i0 + u) * r) + c2);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float2 m = bf16x2(w[u]);
        const int i = warp * (LP_ROWS / 8) + i0 + u;
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          const float a = act[t * LP_ROWS + i];
          acc[t][0] = fmaf(a, m.x, acc[t][0]);
          acc[t][1] = fmaf(a, m.y, acc[t][1]);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      red[warp][t][2 * c2] = acc[t][0];
      red[warp][t][2 * c2 + 1] = acc[t][1];
    }
  }
  __syncthreads();
  for (int o = threadIdx.x; o < 16 * r; o += blockDim.x) {
    const int t = o / r, c = o % r;
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += red[w][t][c];
    out[o] = s;
  }
}

// The last of `n` CTAs to arrive on *ticket (which it resets); all threads learn it.
LMOE_DEV bool last_arrival(unsigned* ticket, unsigned n) {
  __shared__ int last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    last = atomicAdd(ticket, 1u) == n - 1;
    if (last) *ticket = 0;
  }
  __syncthreads();
  if (last) __threadfence();
  return last;
}
// out[o] = sum over b < n of part[b][o] in b order, o < len (a multiple of 4):
// four values per thread, eight partials' loads in flight
LMOE_DEV void sum_partials(const float* part, int n, int len, float* out) {
  for (int o = 4 * threadIdx.x; o < len; o += 4 * blockDim.x) {
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
    for (int b0 = 0; b0 < n; b0 += 8) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        v[u] = b0 + u < n ? __ldcg(reinterpret_cast<const float4*>(part + (size_t)(b0 + u) * len + o))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        s.x += v[u].x; s.y += v[u].y; s.z += v[u].z; s.w += v[u].w;
      }
    }
    *reinterpret_cast<float4*>(out + o) = s;
  }
}
}  // namespace

// grid (G, d / LP_ROWS). Ppart [G][d/LP_ROWS][16][r], P [G][16][r].
__global__ void __launch_bounds__(256) lora_p_kernel(DecodeArgs A, float* __restrict__ Ppart, float* __restrict__ P,
                                                     unsigned* __restrict__ tickets) {
  extern __shared__ __align__(16) unsigned char lsm[];
  float* act = reinterpret_cast<float*>(lsm);                               // [16][LP_ROWS]
  float (*red)[16][MAXR] = reinterpret_cast<float (*)[16][MAXR]>(act + 16 * LP_ROWS);  // [8][16][r]
  const int g = blockIdx.x, kb = blockIdx.y, nkb = gridDim.y, T = A.T, r = A.r, d = A.d;
  const int k0 = kb * LP_ROWS;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int i = threadIdx.x; i < 2 * LP_ROWS; i += blockDim.x) {  // 8 elements of x per thread
    const int t = i / (LP_ROWS / 8), kk = (i % (LP_ROWS / 8)) * 8;
    const uint4 v = t < T ? __ldg(reinterpret_cast<const uint4*>(A.x + (size_t)t * d + k0 + kk)) : make_uint4(0, 0, 0, 0);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = bf16x2(u[q]);
      act[t * LP_ROWS + kk + 2 * q] = f.x;
      act[t * LP_ROWS + kk + 2 * q + 1] = f.y;
    }
  }
  __syncthreads();
  rows_partial(A.A_in + ((size_t)g * d + k0) * r, r, act, red, Ppart + ((size_t)g * nkb + kb) * 16 * r);
  if (!last_arrival(tickets + g, (unsigned)nkb)) return;
  sum_partials(Ppart + (size_t)g * nkb * 16 * r, nkb, 16 * r, P + (size_t)g * 16 * r);
}

// grid (G, L / LH_COLS). Hl [G][16][L] = P[g]^T-contracted with B_in[g] ([r][L]).
// Thread (column pair cp of the block, quarter q of r); quarters summed in order.
__global__ void __launch_bounds__(256) lora_hl_kernel(DecodeArgs A, const float* __restrict__ P, float* __restrict__ Hl) {
  __shared__ float ps[16][MAXR];
  __shared__ float red[4][16][LH_COLS];
  const int g = blockIdx.x, l0 = blockIdx.y * LH_COLS, T = A.T, r = A.r, L = A.L;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");  // P (lora_p)
  for (int i = threadIdx.x; i < 16 * r; i += blockDim.x) ps[i / r][i % r] = __ldcg(P + (size_t)g * 16 * r + i);
  __syncthreads();
  const int cp = threadIdx.x & 63, q = threadIdx.x >> 6, rq = r / 4;
  const uint16_t* B = A.B_in + (size_t)g * r * L + l0 + 2 * cp;
  float acc[16][2];
#pragma unroll
  for (int t = 0; t < 16; ++t) acc[t][0] = acc[t][1] = 0.f;
#pragma unroll 1
  for (int j0 = q * rq; j0 < (q + 1) * rq; j0 += 8) {
    uint32_t w[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) w[u] = j0 + u < (q + 1) * rq ? __ldg(reinterpret_cast<const uint32_t*>(B + (size_t)(j0 + u) * L)) : 0u;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (j0 + u >= (q + 1) * rq) break;
      const float2 b = bf16x2(w[u]);
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        acc[t][0] = fmaf(ps[t][j0 + u], b.x, acc[t][0]);
        acc[t][1] = fmaf(ps[t][j0 + u], b.y, acc[t][1]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    red[q][t][2 * cp] = acc[t][0];
    red[q][t][2 * cp + 1] = acc[t][1];
  }
  __syncthreads();
  for (int o = threadIdx.x; o < 16 * LH_COLS; o += blockDim.x) {
    const int t = o / LH_COLS, c = o % LH_COLS;
    if (t < T) Hl[((size_t)g * 16 + t) * L + l0 + c] = red[0][t][c] + red[1][t][c] + red[2][t][c] + red[3][t][c];
  }
}

// grid (G, L / LP_ROWS). Zlin [G][16][L] (routed groups), Qpart [G][L/LP_ROWS][16][r], Q [G][16][r].
__global__ void __launch_bounds__(256) lora_q_kernel(DecodeArgs A, const float* __restrict__ Zlin,
                                                     float* __restrict__ Qpart, float* __restrict__ Q,
                                                     unsigned* __restrict__ tickets) {
  extern __shared__ __align__(16) unsigned char lsm[];
  float* act = reinterpret_cast<float*>(lsm);
  float (*red)[16][MAXR] = reinterpret_cast<float (*)[16][MAXR]>(act + 16 * LP_ROWS);
  const int g = blockIdx.x, kb = blockIdx.y, nkb = gridDim.y, T = A.T, r = A.r, L = A.L;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");  // Z and the routing (the single kernel)
  if (!((routed_groups(A) >> g) & 1ull)) return;  // the whole group's CTAs leave together
  const int k0 = kb * LP_ROWS;
  for (int i = threadIdx.x; i < 16 * LP_ROWS; i += blockDim.x) {
    const int t = i / LP_ROWS, kk = i % LP_ROWS;
    act[i] = t < T ? __ldcg(Zlin + ((size_t)g * 16 + t) * L + k0 + kk) : 0.f;
  }
  __syncthreads();
  rows_partial(A.A_out + ((size_t)g * L + k0) * r, r, act, red, Qpart + ((size_t)g * nkb + kb) * 16 * r);
  if (!last_arrival(tickets + g, (unsigned)nkb)) return;
  sum_partials(Qpart + (size_t)g * nkb * 16 * r, nkb, 16 * r, Q + (size_t)g * 16 * r);
}

// grid (d / LO_ROWS, G). Y[g][t][i] += sum_c Q[g][t][c] B_out[g][c][i] for the
// block's rows (routed groups); thread (row pair rp, quarter h of r), quarters
// summed in order. The last group CTA of a row block sums the routed groups in
// ascending order, adds the residual and writes y.
__global__ void __launch_bounds__(256) lora_out_kernel(DecodeArgs A, float* __restrict__ Yp,
                                                       const float* __restrict__ Q, unsigned* __restrict__ tickets) {
  __shared__ float qs[16][MAXR];
  __shared__ float red[4][16][LO_ROWS];
  const int rb = blockIdx.x, g = blockIdx.y, G = gridDim.y, T = A.T, r = A.r, d = A.d;
  const int row0 = rb * LO_ROWS;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // Q (lora_q), Y and the routing (the single kernel)
  const unsigned long long gm = routed_groups(A);
  if ((gm >> g) & 1ull) {
    for (int i = threadIdx.x; i < 16 * r; i += blockDim.x) qs[i / r][i % r] = __ldcg(Q + (size_t)g * 16 * r + i);
    __syncthreads();
    const int rp = threadIdx.x & (LO_ROWS / 2 - 1), h = threadIdx.x / (LO_ROWS / 2), rh = r / 4;
    const uint16_t* B = A.B_out + (size_t)g * r * d + row0 + 2 * rp;
    float acc[16][2];
#pragma unroll
    for (int t = 0; t < 16; ++t) acc[t][0] = acc[t][1] = 0.f;
#pragma unroll 1
    for (int j0 = h * rh; j0 < (h + 1) * rh; j0 += 8) {
      uint32_t w[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) w[u] = j0 + u < (h + 1) * rh ? __ldg(reinterpret_cast<const uint32_t*>(B + (size_t)(j0 + u) * d)) : 0u;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (j0 + u >= (h + 1) * rh) break;
        const float2 b = bf16x2(w[u]);
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          acc[t][0] = fmaf(qs[t][j0 + u], b.x, acc[t][0]);
          acc[t][1] = fmaf(qs[t][j0 + u], b.y, acc[t][1]);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      red[h][t][2 * rp] = acc[t][0];
      red[h][t][2 * rp + 1] = acc[t][1];
    }
    __syncthreads();
    for (int o = threadIdx.x; o < 16 * LO_ROWS; o += blockDim.x) {
      const int t = o / LO_ROWS, c = o % LO_ROWS;
      if (t < T) {
        float* yp = Yp + ((size_t)g * 16 + t) * d + row0 + c;
        *yp = __ldcg(yp) + (red[0][t][c] + red[1][t][c] + red[2][t][c] + red[3][t][c]);
      }
    }
  }
  if (!last_arrival(tickets + rb, (unsigned)G)) return;
  for (int o = threadIdx.x; o < T * LO_ROWS; o += blockDim.x) {
    const int t = o / LO_ROWS, i = row0 + o % LO_ROWS;
    float v = 0.f;
    for (int gg = 0; gg < G; ++gg)
      if ((gm >> gg) & 1ull) v += __ldcg(Yp + ((size_t)gg * 16 + t) * d + i);
    const size_t oi = (size_t)t * d + i;
    if (A.residual) v += bf16_to_f32(A.residual[oi]);
    A.y[oi] = f32_to_bf16_rne(v);
  }
}

size_t lora_rows_smem() { return (size_t)(16 * LP_ROWS + 8 * 16 * MAXR) * 4; }

cudaError_t lora_set_attributes() {
  cudaFuncSetAttribute(lora_p_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lora_rows_smem());
  cudaFuncSetAttribute(lora_q_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lora_rows_smem());
  return cudaGetLastError();
}

bool lora_fused_supported(const DecodeArgs& A) {
  return A.r > 0 && A.r <= MAXR && A.r % 8 == 0 && A.d % LP_ROWS == 0 && A.d % LO_ROWS == 0 &&
         A.L % LP_ROWS == 0 && A.L % LH_COLS == 0 && A.G <= 64;
}

// tickets: [0, G) lora_p, [G, 2G) lora_q, [2G, 2G + d/LO_ROWS) lora_out
size_t lora_ticket_words(int d, int G) { return (size_t)2 * G + d / LO_ROWS + 1; }

namespace {
// a launch that may start while its stream predecessor runs (pdl), or after it
template <typename... Params, typename... Args>
cudaError_t launch(void (*k)(Params...), dim3 grid, size_t smem, cudaStream_t st, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, args...);
}
}  // namespace

cudaError_t launch_lora_in(const DecodeArgs& A, float* Ppart, float* P, float* Hl, unsigned* tickets,
                           cudaStream_t st, StageHook* hook, bool pdl) {
  if (hook) hook->before(st);
  cudaError_t e = launch(lora_p_kernel, dim3(A.G, A.d / LP_ROWS), lora_rows_smem(), st, false, A, Ppart, P, tickets);
  if (hook) hook->after(st);
  if (e != cudaSuccess) return e;
  if (hook) hook->before(st);
  e = launch(lora_hl_kernel, dim3(A.G, A.L / LH_COLS), 0, st, pdl, A, (const float*)P, Hl);
  if (hook) hook->after(st);
  return e;
}

cudaError_t launch_lora_q(const DecodeArgs& A, const float* Zlin, float* Qpart, float* Q, unsigned* tickets,
                          cudaStream_t st, bool pdl) {
  return launch(lora_q_kernel, dim3(A.G, A.L / LP_ROWS), lora_rows_smem(), st, pdl, A, Zlin, Qpart, Q,
                tickets + A.G);
}

cudaError_t launch_lora_out(const DecodeArgs& A, float* Yp, const float* Q, unsigned* tickets, cudaStream_t st,
                            bool pdl) {
  return launch(lora_out_kernel, dim3(A.d / LO_ROWS, A.G), 0, st, pdl, A, Yp, Q, tickets + 2 * A.G);
}

}  // namespace lmoe
