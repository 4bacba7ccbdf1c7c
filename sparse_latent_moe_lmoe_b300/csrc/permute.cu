// Token permutation by group, then expert, for any number of tokens.
//
// Groups of 64 experts share the two large matrices ("Architecture: share
// large matrices across sparse experts"), so the layer gathers tokens per
// group for the shared projections and per expert for the expert's own
// parameters. Assignment a = t*k + j.
//
// Three deterministic passes (no result depends on the order of atomics):
//   count    per block of PERM_TB tokens: assignments per expert, tokens per group
//   scan     per expert / group: exclusive scan over blocks, then over experts / groups
//   scatter  per block: stable ranks (warp match + per-warp counts), then
//            sorted_assign / inv, group_tokens / assign_row
#include "common.cuh"
#include "decode.cuh"

namespace lmoe {

constexpr int PERM_TB = 256;     // tokens per block
constexpr int PERM_THREADS = 1024;

static int perm_blocks(int T) { return (T + PERM_TB - 1) / PERM_TB; }

size_t permute_scratch_bytes(int T, int E, int G) {
  const size_t nb = (size_t)perm_blocks(T);
  return (nb * (E + G) + 2 * (size_t)(E + G) + 64) * sizeof(int);
}

LMOE_DEV unsigned long long group_mask(const int32_t* idx_t, int k, int epg, int E, unsigned* err) {
  unsigned long long m = 0;
  for (int j = 0; j < k; ++j) {
    const int e = idx_t[j];
    if (e < 0 || e >= E) {
      set_error(err, ERRBIT_BAD_INDEX);
      continue;
    }
    m |= 1ull << (e / epg);
  }
  return m;
}

__global__ void __launch_bounds__(PERM_THREADS) perm_count_kernel(const int32_t* __restrict__ idx, int T, int E,
                                                                  int G, int k, int* cnt, int* gcnt, unsigned* err) {
  __shared__ int h[1024];
  __shared__ int gh[64];
  const int blk = blockIdx.x, epg = E / G;
  for (int i = threadIdx.x; i < E; i += blockDim.x) h[i] = 0;
  if (threadIdx.x < G) gh[threadIdx.x] = 0;
  __syncthreads();
  const int t0 = blk * PERM_TB, t1 = min(T, t0 + PERM_TB);
  for (int a = t0 * k + threadIdx.x; a < t1 * k; a += blockDim.x) {
    const int e = idx[a];
    if (e >= 0 && e < E) atomicAdd(&h[e], 1);
  }
  for (int t = t0 + threadIdx.x; t < t1; t += blockDim.x) {
    unsigned long long m = group_mask(idx + (size_t)t * k, k, epg, E, err);
    while (m) {
      const int g = __ffsll((long long)m) - 1;
      m &= m - 1;
      atomicAdd(&gh[g], 1);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += blockDim.x) cnt[(size_t)blk * E + i] = h[i];
  if (threadIdx.x < G) gcnt[(size_t)blk * G + threadIdx.x] = gh[threadIdx.x];
}

// block-wide exclusive scan of n <= 1024 values (one per thread), returns total
LMOE_DEV int block_exclusive_scan(int v, int* s_warp, int& excl) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int wv = lane < nw ? s_warp[lane] : 0;
    int wi = wv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    if (lane < nw) s_warp[lane] = wi - wv;
    if (lane == 31) s_warp[32] = wi;
  }
  __syncthreads();
  excl = s_warp[warp] + incl - v;
  const int total = s_warp[32];
  __syncthreads();
  return total;
}

// in-place exclusive scan of col[b * stride], b < n, by one thread; returns
// the total. Loads go out 16 at a time (the column is n dependent steps).
LMOE_DEV int column_exclusive_scan(int* col, size_t stride, int n) {
  int run = 0;
#pragma unroll 1
  for (int b0 = 0; b0 < n; b0 += 16) {
    int v[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) v[u] = b0 + u < n ? col[(size_t)(b0 + u) * stride] : 0;
#pragma unroll
    for (int u = 0; u < 16; ++u)
      if (b0 + u < n) {
        col[(size_t)(b0 + u) * stride] = run;
        run += v[u];
      }
  }
  return run;
}

__global__ void __launch_bounds__(PERM_THREADS) perm_scan_kernel(int nblk, int E, int G, int* cnt, int* gcnt,
                                                                 PermPtrs pm) {
  __shared__ int s_warp[33];
  const int epg = E / G;
  int tot = 0;
  const int e = threadIdx.x;
  if (e < E) tot = column_exclusive_scan(cnt + e, (size_t)E, nblk);
  int excl;
  const int total = block_exclusive_scan(e < E ? tot : 0, s_warp, excl);
  if (e < E) pm.expert_offsets[e] = excl;
  if (e == 0) pm.expert_offsets[E] = total;
  __syncthreads();
  if (e <= G) pm.group_offsets[e] = (e == G) ? total : pm.expert_offsets[e * epg];
  int gt = 0;
  if (e < G) gt = column_exclusive_scan(gcnt + e, (size_t)G, nblk);
  int gex;
  const int gtotal = block_exclusive_scan(e < G ? gt : 0, s_warp, gex);
  if (e < G) pm.group_tok_offsets[e] = gex;
  if (e == 0) pm.group_tok_offsets[G] = gtotal;
}

__global__ void __launch_bounds__(PERM_THREADS) perm_scatter_kernel(const int32_t* __restrict__ idx, int T, int E,
                                                                    int G, int k, const int* __restrict__ cnt,
                                                                    const int* __restrict__ gcnt, PermPtrs pm) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned short* wcnt = reinterpret_cast<unsigned short*>(smem_raw);  // [32 warps][E]
  int* run = reinterpret_cast<int*>(smem_raw + (size_t)32 * E * 2);    // [E]
  __shared__ int gw[32];
  __shared__ int gbase[64];
  const int blk = blockIdx.x, epg = E / G;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned lt = (1u << lane) - 1u;
  for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) wcnt[i] = 0;
  for (int i = threadIdx.x; i < E; i += blockDim.x) run[i] = pm.expert_offsets[i] + cnt[(size_t)blk * E + i];
  if (threadIdx.x < G) gbase[threadIdx.x] = pm.group_tok_offsets[threadIdx.x] + gcnt[(size_t)blk * G + threadIdx.x];
  __syncthreads();
  const int t0 = blk * PERM_TB, t1 = min(T, t0 + PERM_TB);
  const int a0 = t0 * k, a1 = t1 * k;
  for (int base = a0; base < a1; base += blockDim.x) {
    const int a = base + threadIdx.x;
    int e = (a < a1) ? idx[a] : -1;
    if (e >= E) e = -1;
    const unsigned m = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(m & lt), cw = __popc(m);
    const bool leader = (m & lt) == 0;
    if (e >= 0 && leader) wcnt[warp * E + e] = (unsigned short)cw;
    __syncthreads();
    if (e >= 0) {
      int bw = 0;
      for (int w = 0; w < warp; ++w) bw += wcnt[w * E + e];
      const int pos = run[e] + bw + rank;
      pm.sorted_assign[pos] = a;
      pm.inv[a] = pos;
    }
    __syncthreads();
    if (e >= 0 && leader) {
      atomicAdd(&run[e], cw);
      wcnt[warp * E + e] = 0;
    }
    __syncthreads();
  }
  // group token lists: tokens of this block in ascending order
  for (int tb = t0; tb < t1; tb += blockDim.x) {
    const int t = tb + threadIdx.x;
    unsigned long long msk = 0;
    if (t < t1) {
      for (int j = 0; j < k; ++j) {
        const int e = idx[(size_t)t * k + j];
        if (e >= 0 && e < E) msk |= 1ull << (e / epg);
      }
    }
    for (int g = 0; g < G; ++g) {
      const bool hit = (msk >> g) & 1ull;
      const unsigned bal = __ballot_sync(0xffffffffu, hit);
      if (lane == 0) gw[warp] = __popc(bal);
      __syncthreads();
      int bw = 0;
      for (int w = 0; w < warp; ++w) bw += gw[w];
      if (hit) {
        const int row = gbase[g] + bw + __popc(bal & lt);
        pm.group_tokens[row] = t;
        for (int j = 0; j < k; ++j)
          if (idx[(size_t)t * k + j] / epg == g) pm.assign_row[(size_t)t * k + j] = row;
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        int tot = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += gw[w];
        gbase[g] += tot;
      }
      __syncthreads();
    }
  }
}

cudaError_t permute_set_attributes() {
  cudaFuncSetAttribute(perm_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 100 * 1024);
  return cudaGetLastError();
}

cudaError_t launch_permute(const int32_t* idx, int T, int E, int G, int k, const PermPtrs& pm, void* scratch,
                           unsigned* err, cudaStream_t st) {
  const int nblk = perm_blocks(T);
  int* cnt = reinterpret_cast<int*>(scratch);
  int* gcnt = cnt + (size_t)nblk * E;
  if (nblk > 0) perm_count_kernel<<<nblk, PERM_THREADS, 0, st>>>(idx, T, E, G, k, cnt, gcnt, err);
  perm_scan_kernel<<<1, PERM_THREADS, 0, st>>>(nblk, E, G, cnt, gcnt, pm);
  if (nblk > 0) {
    const size_t smem = (size_t)32 * E * 2 + (size_t)E * 4;
    perm_scatter_kernel<<<nblk, PERM_THREADS, smem, st>>>(idx, T, E, G, k, cnt, gcnt, pm);
  }
  return cudaGetLastError();
}

}  // namespace lmoe
