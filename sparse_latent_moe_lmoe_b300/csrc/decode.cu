// Decode / speculative-verify path of the latent MoE layer: up to 16 tokens
// per pass. Every weight byte is read once per pass; the int4 matrices are
// streamed with 128-bit loads, dequantised in registers and multiplied on the
// tensor cores against the (at most 16) token columns.
//
// Kernels, in launch order (one pass = one chunk of <= 16 tokens):
//   route     router logits (FFMA, fp32), then in the last-arriving CTA the
//             top-k with softmax renormalisation and, optionally, the token
//             permutation by group then expert
//   lora_p    (LoRA only) P[g][t] = A_in[g]^T x_t
//   win       H[g][t] = Win[g] x_t for every active group (+ B_in^T P)
//   gateup    V[p] = silu(Gate_e h) * (Up_e h) for every routed assignment p
//   down      Z[g][t] = sum_{e in g} w Down_e V  (the weighted group reduce)
//   lora_q    (LoRA only) Q[g][t] = A_out[g]^T Z[g][t]
//   wout      Y[g][t] = Wout[g] Z[g][t] (+ B_out^T Q), then the weighted
//             combine y_t = sum_g Y[g][t] (+ residual) in ascending g by the
//             last CTA to finish each row block (a ticket, no waiting)
#include "common.cuh"
#include "decode.cuh"
#include "topk.cuh"

namespace lmoe {

// ---------------------------------------------------------------- helpers

__host__ __device__ __forceinline__ int n_chunks(int K) { return (K + 127) / 128; }

// Build activation fragments for chunks [c0, c1) of a K-long activation,
// for tokens n < 8*NT. src(n, k) returns the fp32 value (0 beyond T or K).
template <int NT, class Src>
LMOE_DEV void stage_frags(uint4* frag, int c0, int c1, int K, Src src) {
  const int nslots = (c1 - c0) * NT * 4 * 32;
  for (int sidx = threadIdx.x; sidx < nslots; sidx += blockDim.x) {
    const int lane = sidx & 31, mp = (sidx >> 5) & 3;
    const int rest = sidx >> 7;  // (c - c0) * NT + nt
    const int nt = rest % NT, cc = rest / NT;
    const int n = nt * 8 + (lane >> 2), tig = lane & 3;
    const int k0 = (c0 + cc) * 128 + tig * 32 + mp * 8;
    float e[8];
    src(n, k0, e);
    frag[sidx] = pack_frag8(e);
    (void)K;
  }
}

// ------------------------------------------------------------------ route

// logits[t][e] for a block of ROWS experts; 16 warps split d.
constexpr int ROUTE_ROWS = 4;
constexpr int ROUTE_WARPS = 16;

LMOE_DEV bool better(float v, int e, float bv, int be) { return v > bv || (v == bv && e < be); }

// top-k of one token by one warp (E <= 1024); writes idx/w.
LMOE_DEV void warp_topk(const float* __restrict__ lg, int E, int k, int32_t* idx_out, float* w_out, int32_t* s_idx,
                        unsigned* err) {
  const int lane = threadIdx.x & 31;
  float v[32];
  unsigned taken = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? __ldcg(lg + e) : -INFINITY;
    if (e < E && v[i] != v[i]) set_error(err, ERRBIT_BAD_DATA);
  }
  float sel = 0.f, l0 = 0.f;
  int sel_e = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && better(v[i], e, bv, be)) {
        bv = v[i];
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (better(ov, oe, bv, be)) {
        bv = ov;
        be = oe;
      }
    }
    if ((be & 31) == lane && be < E) taken |= 1u << (be >> 5);
    if (j == 0) l0 = bv;
    if (lane == j) {
      sel = bv;
      sel_e = be;
    }
  }
  const float ex = (lane < k) ? __expf(sel - l0) : 0.f;
  float z = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  if (lane < k) {
    idx_out[lane] = sel_e;
    w_out[lane] = ex / z;
    if (s_idx) s_idx[lane] = sel_e;
  }
}

// Permutation of T*k (<= 256) assignments by one CTA (see lmoe_perm).
LMOE_DEV void block_permute(const int32_t* s_idx, int T, int E, int G, int k, int* s_cnt, const PermPtrs& pm,
                            unsigned* err) {
  const int n = T * k, epg = E / G;
  for (int e = threadIdx.x; e <= E; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  for (int a = threadIdx.x; a < n; a += blockDim.x) {
    const int e = s_idx[a];
    if (e < 0 || e >= E) {
      set_error(err, ERRBIT_BAD_INDEX);
      continue;
    }
    atomicAdd(&s_cnt[e + 1], 1);
  }
  __syncthreads();
  if (threadIdx.x < 32) {  // inclusive scan of s_cnt[1..E] by one warp
    const int lane = threadIdx.x;
    const int per = (E + 31) / 32;
    int run = 0;
    for (int i = 0; i < per; ++i) {
      const int e = 1 + lane * per + i;
      if (e <= E) run += s_cnt[e];
    }
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    int base = incl - run;
    for (int i = 0; i < per; ++i) {
      const int e = 1 + lane * per + i;
      if (e <= E) {
        base += s_cnt[e];
        s_cnt[e] = base;
      }
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) pm.expert_offsets[e] = s_cnt[e];
  for (int g = threadIdx.x; g <= G; g += blockDim.x) pm.group_offsets[g] = s_cnt[g * epg];
  for (int a = threadIdx.x; a < n; a += blockDim.x) {
    const int e = s_idx[a];
    if (e < 0 || e >= E) continue;
    int rank = 0;
    for (int b = 0; b < a; ++b) rank += (s_idx[b] == e);
    const int pos = s_cnt[e] + rank;
    pm.sorted_assign[pos] = a;
    pm.inv[a] = pos;
  }
  // per-group distinct tokens, ascending; rows numbered group by group
  __shared__ int s_gcnt[65];
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    int c = 0;
    for (int t = 0; t < T; ++t) {
      bool hit = false;
      for (int j = 0; j < k; ++j) hit |= (s_idx[t * k + j] / epg == g);
      c += hit;
    }
    s_gcnt[g] = c;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int g = 0; g < G; ++g) {
      const int c = s_gcnt[g];
      s_gcnt[g] = run;
      run += c;
    }
    s_gcnt[G] = run;
  }
  __syncthreads();
  for (int g = threadIdx.x; g <= G; g += blockDim.x) pm.group_tok_offsets[g] = s_gcnt[g];
  for (int pr = threadIdx.x; pr < G * T; pr += blockDim.x) {
    const int g = pr / T, t = pr % T;
    bool hit = false;
    for (int j = 0; j < k; ++j) hit |= (s_idx[t * k + j] / epg == g);
    if (!hit) continue;
    int rank = 0;
    for (int t2 = 0; t2 < t; ++t2) {
      bool h2 = false;
      for (int j = 0; j < k; ++j) h2 |= (s_idx[t2 * k + j] / epg == g);
      rank += h2;
    }
    const int row = s_gcnt[g] + rank;
    pm.group_tokens[row] = t;
    for (int j = 0; j < k; ++j)
      if (s_idx[t * k + j] / epg == g) pm.assign_row[t * k + j] = row;
  }
}

__global__ void __launch_bounds__(ROUTE_WARPS * 32) route_kernel(DecodeArgs A, int do_perm, float* logits_out) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int T = A.T, d = A.d, E = A.E;
  uint16_t* s_x = reinterpret_cast<uint16_t*>(smem_raw);  // [T][d]
  float* s_red = reinterpret_cast<float*>(smem_raw + (size_t)T * d * 2);  // [warps][ROWS][16]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // stage x (bf16) in shared memory
  {
    const uint4* src = reinterpret_cast<const uint4*>(A.x);
    uint4* dst = reinterpret_cast<uint4*>(s_x);
    const int n16 = T * d / 8;
    for (int i = threadIdx.x; i < n16; i += blockDim.x) dst[i] = __ldg(src + i);
  }
  __syncthreads();
  const int row0 = blockIdx.x * ROUTE_ROWS;
  float acc[ROUTE_ROWS][16];
#pragma unroll
  for (int r = 0; r < ROUTE_ROWS; ++r)
#pragma unroll
    for (int t = 0; t < 16; ++t) acc[r][t] = 0.f;
  const int d4 = d / 4;
  const int p0 = warp * d4 / ROUTE_WARPS, p1 = (warp + 1) * d4 / ROUTE_WARPS;
  for (int pos = p0 + lane; pos < p1; pos += 32) {
    float4 wv[ROUTE_ROWS];
#pragma unroll
    for (int r = 0; r < ROUTE_ROWS; ++r)
      wv[r] = (row0 + r < E) ? __ldg(reinterpret_cast<const float4*>(A.W_r + (size_t)(row0 + r) * d) + pos)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      if (t < T) {
        const uint2 xb = *reinterpret_cast<const uint2*>(s_x + (size_t)t * d + pos * 4);
        const float x0 = __uint_as_float(xb.x << 16), x1 = __uint_as_float(xb.x & 0xffff0000u);
        const float x2 = __uint_as_float(xb.y << 16), x3 = __uint_as_float(xb.y & 0xffff0000u);
#pragma unroll
        for (int r = 0; r < ROUTE_ROWS; ++r)
          acc[r][t] = fmaf(wv[r].w, x3, fmaf(wv[r].z, x2, fmaf(wv[r].y, x1, fmaf(wv[r].x, x0, acc[r][t]))));
      }
    }
  }
  // reduce over lanes, then over warps
#pragma unroll
  for (int r = 0; r < ROUTE_ROWS; ++r)
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      float v = acc[r][t];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) s_red[(warp * ROUTE_ROWS + r) * 16 + t] = v;
    }
  __syncthreads();
  if (threadIdx.x < ROUTE_ROWS * 16) {
    const int r = threadIdx.x / 16, t = threadIdx.x % 16;
    if (t < T && row0 + r < E) {
      float v = 0.f;
      for (int w = 0; w < ROUTE_WARPS; ++w) v += s_red[(w * ROUTE_ROWS + r) * 16 + t];
      if (A.b_r) v += A.b_r[row0 + r];
      logits_out[(size_t)t * E + row0 + r] = v;
    }
  }
  // the last CTA to finish does top-k (+ permutation)
  __shared__ int s_last;
  __shared__ uint2 s_scr[ROUTE_WARPS * 32];  // top-k candidates, per warp
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned old = atomicAdd(&A.tickets[0], 1u);
    s_last = (old == gridDim.x - 1);
    if (s_last) A.tickets[0] = 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  int32_t* s_idx = reinterpret_cast<int32_t*>(smem_raw);        // [T*k] (reuses the x area)
  int* s_cnt = reinterpret_cast<int*>(smem_raw + 16 * 16 * 4);  // [E+1]
  if (warp < T) {
    if (E <= 512) {  // the threshold selector (topk.cuh): a few dependent steps per token instead of k rounds
      const float* row = logits_out + (size_t)warp * E;
      bool bad = false;
      for (int e = lane; e < E; e += 32) bad |= __ldcg(row + e) != __ldcg(row + e);
      if (__any_sync(0xffffffffu, bad) && lane == 0) set_error(A.err, ERRBIT_BAD_DATA);
      const float2 sw = topk_warp_thr(row, E, A.k, reinterpret_cast<uint2*>(s_scr) + warp * 32);
      if (lane < A.k) {
        const int e = __float_as_int(sw.x);
        A.idx[warp * A.k + lane] = e;
        A.w[warp * A.k + lane] = sw.y;
        s_idx[warp * A.k + lane] = e;
      }
    } else {
      warp_topk(logits_out + (size_t)warp * E, E, A.k, A.idx + warp * A.k, A.w + warp * A.k, s_idx + warp * A.k,
                A.err);
    }
  }
  __syncthreads();
  if (do_perm) block_permute(s_idx, T, E, A.G, A.k, s_cnt, A.pm, A.err);
}

// ------------------------------------------------------------------- LoRA
// P[g][t][c] = sum_i act(t, i) * M[g][i][c] (M = A_in over i < d with act = x,
// or A_out over i < L with act = Z): one CTA of 8 warps per (g, t). A row of M
// is r/8 16-byte chunks; lane l of a warp takes chunk l % (r/8) of row
// l / (r/8) of the warp's rows, and eight row passes are loaded before any is
// used, so a CTA keeps 32 KB of M in flight. Partial sums are added in a
// fixed order (warp, then row within the warp).
__global__ void __launch_bounds__(256) lora_proj_kernel(DecodeArgs A, int which) {
  __shared__ float red[256][8];
  const int g = blockIdx.x, t = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, r = A.r;
  const int cpr = r / 8, rpw = 32 / cpr;  // chunks per row (2..16), rows per warp pass
  const int rl = lane / cpr, cc = lane % cpr, step = 8 * rpw;
  const int K = which == 0 ? A.d : A.L;
  const uint16_t* M = which == 0 ? A.A_in + (size_t)g * A.d * r : A.A_out + (size_t)g * A.L * r;
  const uint16_t* xr = A.x + (size_t)t * A.d;
  const float* zr = A.Z + ((size_t)g * 16 + t) * A.L;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (rl < rpw) {
    for (int i0 = warp * rpw + rl; i0 < K; i0 += 8 * step) {
      uint4 m[8];
      float act[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * step;
        m[u] = i < K ? __ldg(reinterpret_cast<const uint4*>(M + (size_t)i * r + cc * 8)) : make_uint4(0u, 0u, 0u, 0u);
        act[u] = i < K ? (which == 0 ? bf16_to_f32(xr[i]) : zr[i]) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t w[4] = {m[u].x, m[u].y, m[u].z, m[u].w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          acc[2 * h] = fmaf(act[u], __uint_as_float(w[h] << 16), acc[2 * h]);
          acc[2 * h + 1] = fmaf(act[u], __uint_as_float(w[h] & 0xffff0000u), acc[2 * h + 1]);
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) red[tid][j] = acc[j];
  __syncthreads();
  for (int c = tid; c < r; c += blockDim.x) {
    const int chunk = c / 8, j = c % 8;
    float v = 0.f;
    for (int w = 0; w < 8; ++w)
      for (int q = 0; q < rpw; ++q) v += red[w * 32 + q * cpr + chunk][j];
    (which == 0 ? A.Pin : A.Qout)[((size_t)g * 16 + t) * r + c] = v;
  }
}

// -------------------------------------------------------------------- win
// grid (ceil(L / (16*8)), G, KS); 8 warps, one 16-row tile each, over the
// chunk range of split ks. Output Hp[ks][g][t][l].
template <int NT>
__global__ void __launch_bounds__(256) win_kernel(DecodeArgs A) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint4* frag = reinterpret_cast<uint4*>(smem_raw);
  const int g = blockIdx.y, ks = blockIdx.z;
  const int ng = A.pm.group_tok_offsets[g + 1] - A.pm.group_tok_offsets[g];
  if (ng == 0) return;
  const int nch = n_chunks(A.d), cps = (nch + A.ks_in - 1) / A.ks_in;
  const int c0 = ks * cps, c1 = min(nch, c0 + cps);
  if (c0 >= c1) return;
  const uint16_t* x = A.x;
  const int T = A.T, d = A.d;
  stage_frags<NT>(frag, c0, c1, d, [&](int n, int k0, float* e) {
    if (n < T && k0 < d) {
      const uint4 v = *reinterpret_cast<const uint4*>(x + (size_t)n * d + k0);
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        e[2 * i] = __uint_as_float(u[i] << 16);
        e[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) e[i] = 0.f;
    }
  });
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
  const int rt = blockIdx.x * 8 + warp;
  if (rt * 16 >= A.L) return;
  float acc[NT][4] = {};
  mma_rows<NT>(A.W_in_q + (size_t)g * A.L * (d / 2), A.W_in_s + (size_t)g * A.L * (d / 32), d, rt * 16, c0, c1, c0,
               frag, acc);
  float* Hp = A.Hp + ((size_t)ks * A.G + g) * 16 * A.L;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = rt * 16 + gid + ((i & 2) ? 8 : 0);
      const int t = nt * 8 + 2 * tig + (i & 1);
      float v = acc[nt][i];
      if (A.r > 0 && ks == 0 && t < T) {  // Recover-LoRA branch on the shared down-projection
        const float* P = A.Pin + ((size_t)g * 16 + t) * A.r;
        const uint16_t* B = A.B_in + (size_t)g * A.r * A.L + row;
        for (int c = 0; c < A.r; ++c) v = fmaf(P[c], bf16_to_f32(B[(size_t)c * A.L]), v);
      }
      if (t < T) Hp[(size_t)t * A.L + row] = v;
    }
}

// ----------------------------------------------------------------- gateup
// grid (ceil(f/64), E); 8 warps: 0..3 gate row tiles, 4..7 the same up rows.
template <int NT>
__global__ void __launch_bounds__(256) gateup_kernel(DecodeArgs A) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int e = blockIdx.y;
  const int p0 = A.pm.expert_offsets[e], p1 = A.pm.expert_offsets[e + 1];
  if (p0 == p1) return;
  const int g = e / A.epg, L = A.L, T = A.T, f = A.f;
  __shared__ int s_pos[16];
  __shared__ float s_gate[4][16][16];
  if (threadIdx.x < 16) s_pos[threadIdx.x] = -1;
  __syncthreads();
  if (threadIdx.x < p1 - p0) s_pos[A.pm.sorted_assign[p0 + threadIdx.x] / A.k] = p0 + threadIdx.x;
  uint4* frag = reinterpret_cast<uint4*>(smem_raw);
  const int nch = n_chunks(L), ks_in = A.ks_in;
  const float* Hg = A.Hp + (size_t)g * 16 * L;
  const size_t hstride = (size_t)A.G * 16 * L;
  stage_frags<NT>(frag, 0, nch, L, [&](int n, int k0, float* ev) {
#pragma unroll
    for (int i = 0; i < 8; ++i) ev[i] = 0.f;
    if (n < T && k0 < L) {
      for (int s = 0; s < ks_in; ++s) {
        const float4* h = reinterpret_cast<const float4*>(Hg + s * hstride + (size_t)n * L + k0);
        const float4 a = h[0], b = h[1];
        ev[0] += a.x; ev[1] += a.y; ev[2] += a.z; ev[3] += a.w;
        ev[4] += b.x; ev[5] += b.y; ev[6] += b.z; ev[7] += b.w;
      }
    }
  });
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
  const int which = warp >> 2;  // 0 gate, 1 up
  const int rt = blockIdx.x * 4 + (warp & 3);
  const bool active = rt * 16 < f;
  float acc[NT][4] = {};
  if (active) {
    const uint8_t* q = (which ? A.up_q : A.gate_q) + (size_t)e * f * (L / 2);
    const uint16_t* s = (which ? A.up_s : A.gate_s) + (size_t)e * f * (L / 32);
    mma_rows<NT>(q, s, L, rt * 16, 0, nch, 0, frag, acc);
  }
  if (which == 0 && active) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i)
        s_gate[warp & 3][gid + ((i & 2) ? 8 : 0)][nt * 8 + 2 * tig + (i & 1)] = acc[nt][i];
  }
  __syncthreads();
  if (which == 1 && active) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int rr = gid + ((i & 2) ? 8 : 0), t = nt * 8 + 2 * tig + (i & 1);
        if (t < T && s_pos[t] >= 0) {
          const float a = s_gate[warp & 3][rr][t];
          A.V[(size_t)s_pos[t] * f + rt * 16 + rr] = silu(a) * acc[nt][i];
        }
      }
  }
}

// ------------------------------------------------------------------- down
// grid (ceil(L / (16*4)), G); 8 warps = 4 row tiles x 2 expert splits. For
// every active expert e of group g the activation columns are w_p * V[p] at
// the tokens routed to e and zero elsewhere, so one accumulator sums the
// group's experts: Z[g][t] = sum_e Down_e (w V)[t].
constexpr int DOWN_BATCH = 8;
template <int NT>
__global__ void __launch_bounds__(256) down_kernel(DecodeArgs A) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint4* frag = reinterpret_cast<uint4*>(smem_raw);
  const int g = blockIdx.y, L = A.L, f = A.f, T = A.T, k = A.k;
  __shared__ int s_e[256];  // active experts of g: at most min(E/G, T*k) <= 256
  __shared__ int s_ne;
  __shared__ float s_red[4][16][16];
  if (threadIdx.x == 0) {
    int n = 0;
    for (int e = g * A.epg; e < (g + 1) * A.epg; ++e)
      if (A.pm.expert_offsets[e + 1] > A.pm.expert_offsets[e]) s_e[n++] = e;
    s_ne = n;
  }
  __syncthreads();
  const int ne = s_ne;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
  const int rt = blockIdx.x * 4 + (warp & 3), es = warp >> 2;
  const int nch = n_chunks(f);
  const int per_e = nch * NT * 4 * 32;  // uint4 per expert
  float acc[NT][4] = {};
  for (int b0 = 0; b0 < ne; b0 += DOWN_BATCH) {
    const int nb = min(DOWN_BATCH, ne - b0);
    __syncthreads();
    for (int bi = 0; bi < nb; ++bi) {
      const int e = s_e[b0 + bi];
      const int p0 = A.pm.expert_offsets[e], p1 = A.pm.expert_offsets[e + 1];
      stage_frags<NT>(frag + bi * per_e, 0, nch, f, [&](int n, int k0, float* ev) {
#pragma unroll
        for (int i = 0; i < 8; ++i) ev[i] = 0.f;
        if (n >= T || k0 >= f) return;
        for (int p = p0; p < p1; ++p) {
          const int a = A.pm.sorted_assign[p];
          if (a / k == n) {
            const float wt = A.w[a];
            const float4* v = reinterpret_cast<const float4*>(A.V + (size_t)p * f + k0);
            const float4 x0 = v[0], x1 = v[1];
            ev[0] = wt * x0.x; ev[1] = wt * x0.y; ev[2] = wt * x0.z; ev[3] = wt * x0.w;
            ev[4] = wt * x1.x; ev[5] = wt * x1.y; ev[6] = wt * x1.z; ev[7] = wt * x1.w;
          }
        }
      });
    }
    __syncthreads();
    if (rt * 16 < L) {
      for (int bi = es; bi < nb; bi += 2) {
        const int e = s_e[b0 + bi];
        mma_rows<NT>(A.down_q + (size_t)e * L * (f / 2), A.down_s + (size_t)e * L * (f / 32), f, rt * 16, 0, nch, 0,
                     frag + bi * per_e, acc);
      }
    }
  }
  if (es == 1) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) s_red[warp & 3][gid + ((i & 2) ? 8 : 0)][nt * 8 + 2 * tig + (i & 1)] = acc[nt][i];
  }
  __syncthreads();
  if (es == 0 && rt * 16 < L) {
    float* Z = A.Z + (size_t)g * 16 * L;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int rr = gid + ((i & 2) ? 8 : 0), t = nt * 8 + 2 * tig + (i & 1);
        if (t < T) Z[(size_t)t * L + rt * 16 + rr] = acc[nt][i] + s_red[warp][rr][t];
      }
  }
}

// ------------------------------------------------------------------- wout
// grid (ceil(d / (16*4)), G); 8 warps = 4 row tiles x 2 K splits.
// mode 0: combine -- Y partial per group, the last CTA of a row block sums
//         the active groups in ascending order (+ residual) into y (bf16).
// mode 1: rows   -- write Y[row(g, t)] (fp32) for the permutation's rows.
template <int NT>
__global__ void __launch_bounds__(256) wout_kernel(DecodeArgs A, int mode) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint4* frag = reinterpret_cast<uint4*>(smem_raw);
  const int g = blockIdx.y, L = A.L, d = A.d, T = A.T, G = A.G;
  const int ng = A.pm.group_tok_offsets[g + 1] - A.pm.group_tok_offsets[g];
  if (ng == 0) return;
  __shared__ float s_red[4][16][16];
  __shared__ int s_last;
  const int nch = n_chunks(L);
  const float* Zg = A.Z + (size_t)g * 16 * L;
  stage_frags<NT>(frag, 0, nch, L, [&](int n, int k0, float* ev) {
    if (n < T && k0 < L) {
      const float4* z = reinterpret_cast<const float4*>(Zg + (size_t)n * L + k0);
      const float4 a = z[0], b = z[1];
      ev[0] = a.x; ev[1] = a.y; ev[2] = a.z; ev[3] = a.w;
      ev[4] = b.x; ev[5] = b.y; ev[6] = b.z; ev[7] = b.w;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) ev[i] = 0.f;
    }
  });
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
  const int rt = blockIdx.x * 4 + (warp & 3), ks = warp >> 2;
  const int half = (nch + 1) / 2;
  const int c0 = ks * half, c1 = min(nch, c0 + half);
  float acc[NT][4] = {};
  if (rt * 16 < d && c0 < c1)
    mma_rows<NT>(A.W_out_q + (size_t)g * d * (L / 2), A.W_out_s + (size_t)g * d * (L / 32), L, rt * 16, c0, c1, 0,
                 frag, acc);
  if (ks == 1) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) s_red[warp & 3][gid + ((i & 2) ? 8 : 0)][nt * 8 + 2 * tig + (i & 1)] = acc[nt][i];
  }
  __syncthreads();
  if (ks == 0 && rt * 16 < d) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int rr = gid + ((i & 2) ? 8 : 0), t = nt * 8 + 2 * tig + (i & 1);
        if (t >= T) continue;
        const int row = rt * 16 + rr;
        float v = acc[nt][i] + s_red[warp][rr][t];
        if (A.r > 0) {  // Recover-LoRA branch on the shared up-projection
          const float* Q = A.Qout + ((size_t)g * 16 + t) * A.r;
          const uint16_t* B = A.B_out + (size_t)g * A.r * d + row;
          for (int c = 0; c < A.r; ++c) v = fmaf(Q[c], bf16_to_f32(B[(size_t)c * d]), v);
        }
        if (mode == 0) {
          A.Yp[((size_t)g * 16 + t) * d + row] = v;
        } else {
          // the (g, t) row of the permutation, if t routes into g
          const int tg = A.tok0 + t;
          for (int j = 0; j < A.k; ++j)
            if (A.idx_all[(size_t)tg * A.k + j] / A.epg == g) {
              A.Yrows[(size_t)A.assign_row_all[(size_t)tg * A.k + j] * d + row] = v;
              break;
            }
        }
      }
  }
  if (mode != 0) return;
  // ticketed combine: the last active group to finish this row block sums
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    int n_active = 0;
    for (int gg = 0; gg < G; ++gg) n_active += (A.pm.group_tok_offsets[gg + 1] > A.pm.group_tok_offsets[gg]);
    const unsigned old = atomicAdd(&A.tickets[1 + blockIdx.x], 1u);
    s_last = (old == (unsigned)n_active - 1u);
    if (s_last) A.tickets[1 + blockIdx.x] = 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int rows0 = blockIdx.x * 64;
  for (int i = threadIdx.x; i < 64 * T; i += blockDim.x) {
    const int t = i / 64, row = rows0 + (i % 64);
    if (row >= d) continue;
    float v = 0.f;
    for (int gg = 0; gg < G; ++gg)
      if (A.pm.group_tok_offsets[gg + 1] > A.pm.group_tok_offsets[gg])
        v += __ldcg(A.Yp + ((size_t)gg * 16 + t) * d + row);
    if (A.residual) v += bf16_to_f32(A.residual[(size_t)t * d + row]);
    A.y[(size_t)t * d + row] = f32_to_bf16_rne(v);
  }
}

// -------------------------------------------------------------- combine
// y_t = sum over t's groups (ascending) of Y[row(g, t)] (+ residual).
__global__ void combine_kernel(const float* __restrict__ Y, const int32_t* __restrict__ idx,
                               const int32_t* __restrict__ assign_row, int T, int d, int k, int epg,
                               const uint16_t* __restrict__ residual, uint16_t* __restrict__ y) {
  const int t = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= d) return;
  int rows[16];
  int gs[16];
  int n = 0;
  for (int j = 0; j < k; ++j) {
    const int g = idx[(size_t)t * k + j] / epg;
    bool seen = false;
    for (int i = 0; i < n; ++i) seen |= (gs[i] == g);
    if (!seen) {
      gs[n] = g;
      rows[n] = assign_row[(size_t)t * k + j];
      ++n;
    }
  }
  // ascending group order
  for (int i = 1; i < n; ++i)
    for (int m = i; m > 0 && gs[m] < gs[m - 1]; --m) {
      int tg = gs[m]; gs[m] = gs[m - 1]; gs[m - 1] = tg;
      int tr = rows[m]; rows[m] = rows[m - 1]; rows[m - 1] = tr;
    }
  float v = 0.f;
  for (int i = 0; i < n; ++i) v += Y[(size_t)rows[i] * d + c];
  if (residual) v += bf16_to_f32(residual[(size_t)t * d + c]);
  y[(size_t)t * d + c] = f32_to_bf16_rne(v);
}

// --------------------------------------------------------------- launchers

// Raise every decode kernel's dynamic shared-memory cap once per device.
cudaError_t decode_set_attributes() {
  const int cap = 200 * 1024;
  cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, cap);
  cudaFuncSetAttribute(win_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, cap);
  cudaFuncSetAttribute(win_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, cap);
  cudaFuncSetAttribute(gateup_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, cap);
  cudaFuncSetAttribute(gateup_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, cap);
  cudaFuncSetAttribute(down_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, cap);
  cudaFuncSetAttribute(down_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, cap);
  cudaFuncSetAttribute(wout_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, cap);
  cudaFuncSetAttribute(wout_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, cap);
  return cudaGetLastError();
}

static size_t frag_bytes(int nch, int NT) { return (size_t)nch * NT * 4 * 32 * 16; }

cudaError_t launch_route(const DecodeArgs& A, int do_perm, float* logits_out, cudaStream_t st) {
  const int grid = (A.E + ROUTE_ROWS - 1) / ROUTE_ROWS;
  size_t smem = (size_t)A.T * A.d * 2 + ROUTE_WARPS * ROUTE_ROWS * 16 * 4;
  const size_t need_tail = 16 * 16 * 4 + (size_t)(A.E + 1) * 4;
  if (smem < need_tail) smem = need_tail;
  route_kernel<<<grid, ROUTE_WARPS * 32, smem, st>>>(A, do_perm, logits_out);
  return cudaGetLastError();
}

cudaError_t launch_lora_proj(const DecodeArgs& A, int which, cudaStream_t st) {
  lora_proj_kernel<<<dim3(A.G, A.T), 256, 0, st>>>(A, which);
  return cudaGetLastError();
}

template <int NT>
static cudaError_t launch_experts_nt(const DecodeArgs& A, int mode, cudaStream_t st, StageHook* hook) {
  // win
  {
    const int nch = n_chunks(A.d), cps = (nch + A.ks_in - 1) / A.ks_in;
    const size_t smem = frag_bytes(cps, NT);
    if (hook) hook->before(st);
    win_kernel<NT><<<dim3((A.L + 127) / 128, A.G, A.ks_in), 256, smem, st>>>(A);
    if (hook) hook->after(st);
  }
  {
    const size_t smem = frag_bytes(n_chunks(A.L), NT);
    if (hook) hook->before(st);
    gateup_kernel<NT><<<dim3((A.f + 63) / 64, A.E), 256, smem, st>>>(A);
    if (hook) hook->after(st);
  }
  {
    const size_t smem = frag_bytes(n_chunks(A.f), NT) * DOWN_BATCH;
    if (hook) hook->before(st);
    down_kernel<NT><<<dim3((A.L + 63) / 64, A.G), 256, smem, st>>>(A);
    if (hook) hook->after(st);
  }
  if (A.r > 0) {
    if (hook) hook->before(st);
    lora_proj_kernel<<<dim3(A.G, A.T), 256, 0, st>>>(A, 1);
    if (hook) hook->after(st);
  }
  {
    const size_t smem = frag_bytes(n_chunks(A.L), NT);
    if (hook) hook->before(st);
    wout_kernel<NT><<<dim3((A.d + 63) / 64, A.G), 256, smem, st>>>(A, mode);
    if (hook) hook->after(st);
  }
  return cudaGetLastError();
}

cudaError_t launch_experts(const DecodeArgs& A, int mode, cudaStream_t st, StageHook* hook) {
  if (A.T <= 8) return launch_experts_nt<1>(A, mode, st, hook);
  return launch_experts_nt<2>(A, mode, st, hook);
}

// x_next = bf16(x + y) for bf16 x, y (the sum of two bf16 values is exact in
// fp32, so this is the single rounding of the residual step)
__global__ void residual_add_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ y, size_t n8,
                                    uint16_t* __restrict__ out) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
    const uint4 a = reinterpret_cast<const uint4*>(x)[i], b = reinterpret_cast<const uint4*>(y)[i];
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = __uint_as_float(av[j] << 16) + __uint_as_float(bv[j] << 16);
      const float hi = __uint_as_float(av[j] & 0xffff0000u) + __uint_as_float(bv[j] & 0xffff0000u);
      o[j] = (uint32_t)f32_to_bf16_rne(lo) | ((uint32_t)f32_to_bf16_rne(hi) << 16);
    }
    reinterpret_cast<uint4*>(out)[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

cudaError_t launch_residual_add(const uint16_t* x, const uint16_t* y, size_t n, uint16_t* out, cudaStream_t st) {
  const size_t n8 = n / 8;
  const int blocks = (int)((n8 + 255) / 256 < 1184 ? (n8 + 255) / 256 : 1184);
  residual_add_kernel<<<blocks > 0 ? blocks : 1, 256, 0, st>>>(x, y, n8, out);
  return cudaGetLastError();
}

cudaError_t launch_combine(const float* Y, const int32_t* idx, const int32_t* assign_row, int T, int d, int k,
                           int epg, const uint16_t* residual, uint16_t* y, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  combine_kernel<<<dim3((d + 255) / 256, T), 256, 0, st>>>(Y, idx, assign_row, T, d, k, epg, residual, y);
  return cudaGetLastError();
}

}  // namespace lmoe
