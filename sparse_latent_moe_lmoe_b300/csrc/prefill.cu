// Prefill path of the latent MoE layer (many tokens): the router and every
// projection are GEMMs on the tcgen05 tensor cores (tc_gemm.cuh), both
// operands fed by TMA wherever their rows are contiguous. The int4 matrices
// are dequantised to fp16 once per call (q*s is exact in fp16).
//
//   dequant  Win, Wout, Gate, Up, Down -> fp16, x -> fp16
//
//   route    logits = x . (W_hi + W_mid + W_lo)^T  (W_r split into three
//            bf16 terms at create time; x is exact in bf16; fp32 accumulate)
//            in 128-token x 256-expert tiles, then the top-k and softmax
//            renormalisation by one warp per token over its E logits
//   permute  the deterministic multi-CTA permutation (permute.cu)
//   tsort    (layer calls, G <= 8) tokens in a stable order of the set of
//            groups they route into, the union of those sets per 128-token
//            tile, and x in fp16 in that order: a token tile then reads only
//            the groups its tokens use, in W_in and in W_out
//   win      H[g][t] = Win[g] x_t for every token tile whose tokens use g
//            (rows of tokens of the tile with no expert in g are dropped),
//            stored once per assignment in the expert-sorted order
//   gateup   V[a] = silu(Gate_e h) * Up_e h   grouped by expert (128 gate
//            rows + the matching 128 up rows per tile, SwiGLU in the epilogue)
//   down     U[a] = w_a * Down_e V[a]     grouped by expert
//   zreduce  Z[(g,t)] = sum_{j: g(e_j) = g} U[(t,j)]  in ascending j
//   wout     y_t = sum_g Wout[g] Z[(g,t)] (+ residual): one GEMM per token
//            tile over K = the tile's groups x L (absent (g,t) rows read as
//            zero), so the weighted combine happens in the accumulator
// Intermediates H, V, U, Z are fp16 (fp32 accumulation everywhere).
#include <cuda.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "prefill.cuh"
#include "tc_gemm.cuh"
#include "tmap.cuh"
#include "topk.cuh"

namespace lmoe {

using tc::Tile;

// ------------------------------------------------------------- tile tables

// scratch[0..n] = exclusive prefix of per-problem tile counts (computed by
// the whole CTA); returns through scratch[n] the total.
template <class CountF>
LMOE_DEV void tile_prefix(int* scratch, int n, CountF count) {
  __shared__ int warp_tot[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nt = blockDim.x;
  int carry = 0;
  for (int b0 = 0; b0 < n; b0 += nt) {
    const int i = b0 + tid;
    const int v = i < n ? count(i) : 0;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    if (warp == 0) {
      const int nw = nt >> 5;
      int wv = lane < nw ? warp_tot[lane] : 0, wi = wv;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += t;
      }
      if (lane < nw) warp_tot[lane] = wi - wv;
    }
    __syncthreads();
    if (i < n) scratch[i] = carry + warp_tot[warp] + inc - v;
    if (tid == nt - 1) scratch[n] = carry + warp_tot[warp] + inc;  // running total
    __syncthreads();
    carry = scratch[n];
    __syncthreads();
  }
  if (n == 0 && tid == 0) scratch[0] = 0;
  __syncthreads();
}

// largest p with scratch[p] <= t (problems with zero tiles are skipped)
LMOE_DEV int find_prob(const int* scratch, int n, int t) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (scratch[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

struct ProbBase {
  static constexpr int EPI_SETS = 2;  // epilogue warp sets (TMA operands only)
  // the problem splits its copies into kprep (coordinates, before the stage
  // wait) and kissue (the copies), instead of load_a / load_b
  static constexpr bool KPREP = false;
  long long budget;
  unsigned* err;
};

LMOE_DEV void mma_k4(uint32_t d_tmem, uint64_t da, uint64_t db, uint32_t id, int kb) {
#pragma unroll
  for (int k = 0; k < 4; ++k) tc::mma_f16(d_tmem, da + (uint64_t)(2 * k), db + (uint64_t)(2 * k), id, (kb > 0 || k > 0) ? 1u : 0u);
}

LMOE_DEV void store_half16(__half* dst, const float v[16]) {
  uint32_t h[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) h[i] = pack_half2(v[2 * i], v[2 * i + 1]);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  d4[0] = make_uint4(h[0], h[1], h[2], h[3]);
  d4[1] = make_uint4(h[4], h[5], h[6], h[7]);
}

// the epilogue's column range of an n-column tile: every column (half < 0)
// or the first / second half (two epilogue warp sets)
LMOE_DEV void epi_cols(int half, int n, int& lo, int& hi) {
  lo = half < 0 ? 0 : half * (n / 2);
  hi = half < 0 ? n : lo + n / 2;
}

// ------------------------------------------------------------------ router
// logits[t][e] (+ bias) = x_t . (W_hi + W_mid + W_lo)[e] for 128 tokens x 256
// experts per output tile; the top-k runs afterwards (route_topk_kernel), one
// warp per token.
//
// Every product is exact (bf16 x bf16) but the tensor core's fp32
// accumulator loses up to an ulp of its running value at each accumulate
// step, so the error grows with the number of steps and with the size of the
// sum being accumulated. Each output tile is therefore computed as separate
// accumulations ("segments", each a tile of this problem with its own
// accumulator): KSEG_HI K blocks of x . W_hi per segment, then one segment
// for every K block of x . W_mid and x . W_lo (terms ~2^-8 the size of the
// logit, whose rounding stays far smaller). A CTA takes the segments of one
// output tile back to back; its epilogue adds each segment's result to a
// running fp32 sum in a fixed order (the W_hi segments in K order, then
// W_mid + W_lo, then the bias), so the result is deterministic. The running
// sum lives in the CTA's own 128 KB scratch tile (L2-resident), laid out
// [column / 4][row][4] so that a warp's 32 rows are one contiguous 512-byte
// run per access; the last segment writes the logits rows.
struct ProbRoute : ProbBase {
  static constexpr int BN = 256, ACC_COLS = 256, STAGES = 4;
  static constexpr int KSEG_HI = 16;
  CUtensorMap am;         // x as [T][d] bf16, box {64, 128}
  CUtensorMap bm;         // the split W_r as [3][E][d] bf16, box {64, 256, 1}
  const float* bias;      // [E] or null
  int T, d, E;
  float* logits;          // [T][E]
  float* part;            // [grid][64][128][4] running sums, one tile per CTA
  LMOE_DEV int ntn() const { return (E + 255) / 256; }
  LMOE_DEV int nmn() const { return ((T + 127) / 128) * ntn(); }
  LMOE_DEV int nhi() const { return (d / 64 + KSEG_HI - 1) / KSEG_HI; }
  LMOE_DEV int nseg() const { return nhi() + 1; }
  LMOE_DEV void init(int*) const {}
  // CTA c takes output tiles c, c + grid, ...; each as nseg() consecutive
  // tiles of this problem (tiles past the last output tile are empty)
  LMOE_DEV int num_tiles(const int*) const {
    const int g = (int)gridDim.x;
    return nseg() * g * ((nmn() + g - 1) / g);
  }
  LMOE_DEV Tile tile(const int*, int t) const {
    const int g = (int)gridDim.x, i = t / g;
    const int mn = (i / nseg()) * g + t % g;
    Tile tl;
    tl.prob = i % nseg();
    tl.gm = 0;
    tl.arow = 0;
    if (mn >= nmn()) {
      tl.m0 = tl.n0 = tl.rows = tl.nkb = 0;
      return tl;
    }
    tl.m0 = (mn / ntn()) * 128;  // both expert halves of a token tile run side by side (x shared in L2)
    tl.n0 = (mn % ntn()) * 256;
    tl.rows = min(128, T - tl.m0);
    const int kx = d / 64;
    tl.nkb = tl.prob < nhi() ? min(KSEG_HI, kx - tl.prob * KSEG_HI) : 2 * kx;
    return tl;
  }
  // K block kb of segment s: x block s*KSEG_HI + kb against W_hi, or (the
  // last segment) x block kb/2 against W_mid (kb even) and W_lo (kb odd);
  // rows beyond T or E read as zero
  LMOE_DEV void load_a(const Tile& tl, int kb, void* dst, uint64_t* bar) const {
    const int xb = tl.prob < nhi() ? tl.prob * KSEG_HI + kb : kb >> 1;
    tma_load_2d(dst, &am, xb * 64, tl.m0, bar);
  }
  LMOE_DEV void load_b(const Tile& tl, int kb, void* dst, uint64_t* bar) const {
    const bool hi = tl.prob < nhi();
    tma_load_3d(dst, &bm, (hi ? tl.prob * KSEG_HI + kb : kb >> 1) * 64, tl.n0, hi ? 0 : 1 + (kb & 1), bar);
  }
  LMOE_DEV void mma_stage(const Tile&, int kb, uint32_t d_tmem, uint64_t da, uint64_t db) const {
    mma_k4(d_tmem, da, db, tc::idesc(128, 256, 1), kb);
  }
  // one thread per token row: the segment's sums (this warp set's columns)
  // added to the row's running value (this thread's own from the previous
  // segment), 16 columns at a time with the next 16 columns' loads in flight
  LMOE_DEV void epilogue(const int*, const Tile& tl, int row, uint32_t tbase, int half) const {
    const bool valid = row < tl.rows, first = tl.prob == 0, last = tl.prob == nseg() - 1;
    float4* pp = reinterpret_cast<float4*>(part) + (size_t)blockIdx.x * (64 * 128) + row;  // + (c / 4) * 128
    const bool ld = valid && !first;
    int lo, hi;
    epi_cols(half, 256, lo, hi);
    float4 cur[4], nxt[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) cur[i] = ld ? __ldcg(pp + (lo / 4 + i) * 128) : make_float4(0.f, 0.f, 0.f, 0.f);
    float* out = logits + (size_t)(tl.m0 + row) * E + tl.n0;
    const int ne = min(256, E - tl.n0);
#pragma unroll 1
    for (int c0 = lo; c0 < hi; c0 += 16) {
      if (c0 + 16 < hi) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          nxt[i] = ld ? __ldcg(pp + ((c0 + 16) / 4 + i) * 128) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float v[16];
      tc::tmem_ld16(tbase + (uint32_t)c0, v);  // warp-collective: every lane loads
      if (valid) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v[4 * i] = cur[i].x + v[4 * i];
          v[4 * i + 1] = cur[i].y + v[4 * i + 1];
          v[4 * i + 2] = cur[i].z + v[4 * i + 2];
          v[4 * i + 3] = cur[i].w + v[4 * i + 3];
        }
        if (!last) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            __stcg(pp + (c0 / 4 + i) * 128, make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
        } else {
          if (bias) {
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] += c0 + i < ne ? bias[tl.n0 + c0 + i] : 0.f;
          }
          if (c0 + 16 <= ne) {
#pragma unroll
            for (int i = 0; i < 16; i += 4)
              *reinterpret_cast<float4*>(out + c0 + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (c0 + i < ne) out[c0 + i] = v[i];
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) cur[i] = nxt[i];
    }
  }
};

// top-k with softmax renormalisation, one warp per token
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                         int32_t* __restrict__ idx, float* __restrict__ w) {
  __shared__ uint2 scratch[8][32];
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= T) return;
  const float2 sw = topk_warp_thr(logits + (size_t)t * E, E, k, scratch[threadIdx.x >> 5]);
  if (lane < k) {
    idx[(size_t)t * k + lane] = __float_as_int(sw.x);
    w[(size_t)t * k + lane] = sw.y;
  }
}

// -------------------------------------------------------------------- W_in
struct ProbWin : ProbBase {
  // H for every (group, token): one dense GEMM per group, A = x by TMA. The
  // rows of tokens with no expert in a group are computed and dropped --
  // cheaper than gathering each group's tokens. The epilogue writes row
  // (g, t) once for each of the token's assignments in group g, at that
  // assignment's position in the expert-sorted order, so the expert GEMM
  // reads its A operand by plain TMA boxes.
  static constexpr int BN = 256, ACC_COLS = 256, STAGES = 4;
  CUtensorMap am;   // x in fp16 as [T][d] (in tsort order when sorted), box {64, 128}
  CUtensorMap bm;   // Win in fp16 as [G][L][d], box {64, 256, 1}
  int T, d, L, G, k, epg;
  const int32_t* idx;  // [T*k] routed experts
  const int32_t* inv;  // [T*k] assignment -> position in the expert-sorted order
  __half* H;           // [T*k][L] by sorted position
  // sorted: A row p is token tsort[p]; group g visits only the token tiles
  // gtl[g][0 .. gtc[g]) (the tiles whose union of groups holds g)
  const int32_t* tsort;
  const int* gtc;
  const int* gtl;
  // Recover-LoRA (rp > 0, the rank padded to 64): K blocks d/64 .. (d+rp)/64
  // read P = x . A_in (every group, [T][G*rp] fp16 in x16's row order) and
  // B_in[g]^T in fp16 as [G][L][rp], so H = [x | P_g] . [Win[g] ; B_in[g]]
  CUtensorMap pm;   // P, box {64, 128}
  CUtensorMap lbm;  // B_in^T, box {64, 256, 1}
  int rp;
  LMOE_DEV int ntn() const { return L / 256; }
  LMOE_DEV int ntm() const { return (T + 127) / 128; }
  LMOE_DEV void init(int* sc) const {
    if (tsort) tile_prefix(sc, G, [&](int g) { return gtc[g] * ntn(); });
  }
  LMOE_DEV int num_tiles(const int* sc) const { return tsort ? sc[G] : G * ntm() * ntn(); }
  LMOE_DEV Tile tile(const int* sc, int t) const {
    Tile tl;
    int loc;
    if (tsort) {
      tl.prob = find_prob(sc, G, t);
      loc = t - sc[tl.prob];
      tl.m0 = gtl[tl.prob * ntm() + loc / ntn()] * 128;
    } else {
      tl.prob = t / (ntm() * ntn());
      loc = t % (ntm() * ntn());
      tl.m0 = (loc / ntn()) * 128;
    }
    tl.n0 = (loc % ntn()) * 256;
    tl.rows = min(128, T - tl.m0);
    tl.nkb = (d + rp) / 64;
    tl.gm = 0;
    tl.arow = tl.m0;
    return tl;
  }
  LMOE_DEV void load_a(const Tile& tl, int kb, void* dst, uint64_t* bar) const {
    const int kx = d >> 6;
    if (rp == 0 || kb < kx) tma_load_2d(dst, &am, kb * 64, tl.m0, bar);
    else tma_load_2d(dst, &pm, tl.prob * rp + (kb - kx) * 64, tl.m0, bar);
  }
  LMOE_DEV void load_b(const Tile& tl, int kb, void* dst, uint64_t* bar) const {
    const int kx = d >> 6;
    if (rp == 0 || kb < kx) tma_load_3d(dst, &bm, kb * 64, tl.n0, tl.prob, bar);
    else tma_load_3d(dst, &lbm, (kb - kx) * 64, tl.n0, tl.prob, bar);
  }
  LMOE_DEV void mma_stage(const Tile&, int kb, uint32_t d_tmem, uint64_t da, uint64_t db) const {
    mma_k4(d_tmem, da, db, tc::idesc(128, 256, 0), kb);
  }
  LMOE_DEV void epilogue(const int*, const Tile& tl, int row, uint32_t tbase, int half) const {
    const int t = row < tl.rows ? (tsort ? tsort[tl.m0 + row] : tl.m0 + row) : 0;
    unsigned dest = 0;  // bit j: assignment j of token t is an expert of group tl.prob
    if (row < tl.rows)
      for (int j = 0; j < k; ++j)
        if (idx[(size_t)t * k + j] / epg == tl.prob) dest |= 1u << j;
    int lo, hi;
    epi_cols(half, 256, lo, hi);
    for (int c0 = lo; c0 < hi; c0 += 16) {
      float v[16];
      tc::tmem_ld16(tbase + (uint32_t)c0, v);  // warp-collective: every lane loads
      for (unsigned m = dest; m; m &= m - 1u)
        store_half16(H + (size_t)inv[(size_t)t * k + __ffs(m) - 1] * L + tl.n0 + c0, v);
    }
  }
};

// ---------------------------------------------------------------- gate/up
struct ProbGateUp : ProbBase {
  static constexpr int BN = 256, ACC_COLS = 256, STAGES = 4;
  CUtensorMap gm, um;  // gate / up in fp16 as [E*f][L], box {64, 128}
  CUtensorMap am;      // H by sorted position as [T*k][L] fp16, box {64, 128}
  int L, f, E;
  const int32_t* eo;
  __half* V;  // [T*k][f]
  LMOE_DEV int ntn() const { return f / 128; }
  LMOE_DEV void init(int* sc) const {
    tile_prefix(sc, E, [&](int e) { return ((eo[e + 1] - eo[e] + 127) / 128) * ntn(); });
  }
  LMOE_DEV int num_tiles(const int* sc) const { return sc[E]; }
  LMOE_DEV Tile tile(const int* sc, int t) const {
    Tile tl;
    const int e = find_prob(sc, E, t), loc = t - sc[e];
    tl.prob = e;
    tl.m0 = (loc / ntn()) * 128;
    tl.n0 = (loc % ntn()) * 128;
    tl.rows = min(128, eo[e + 1] - eo[e] - tl.m0);
    tl.nkb = L / 64;
    tl.gm = 0;
    tl.arow = eo[e] + tl.m0;
    return tl;
  }
  // A rows: the expert's assignments (rows past the expert's end belong to
  // the next expert or lie beyond T*k and read as zero; the epilogue drops them)
  LMOE_DEV void load_a(const Tile& tl, int kb, void* dst, uint64_t* bar) const {
    tma_load_2d(dst, &am, kb * 64, tl.arow, bar);
  }
  // B rows 0..127: gate rows n0.. of expert e; 128..255: the matching up rows
  LMOE_DEV void load_b(const Tile& tl, int kb, void* dst, uint64_t* bar) const {
    tma_load_2d(dst, &gm, kb * 64, tl.prob * f + tl.n0, bar);
    tma_load_2d(static_cast<char*>(dst) + 128 * 128, &um, kb * 64, tl.prob * f + tl.n0, bar);
  }
  LMOE_DEV void mma_stage(const Tile&, int kb, uint32_t d_tmem, uint64_t da, uint64_t db) const {
    mma_k4(d_tmem, da, db, tc::idesc(128, 256, 0), kb);
  }
  LMOE_DEV void epilogue(const int*, const Tile& tl, int row, uint32_t tbase, int half) const {
    int lo, hi;
    epi_cols(half, 128, lo, hi);
    for (int c0 = lo; c0 < hi; c0 += 16) {
      float g[16], u[16];
      tc::tmem_ld16(tbase + (uint32_t)c0, g);
      tc::tmem_ld16(tbase + (uint32_t)(128 + c0), u);
#pragma unroll
      for (int i = 0; i < 16; ++i) g[i] = silu(g[i]) * u[i];
      if (row < tl.rows) store_half16(V + (size_t)(tl.arow + row) * f + tl.n0 + c0, g);
    }
  }
};

// ------------------------------------------------------------------- down
struct ProbDown : ProbBase {
  static constexpr int BN = 256, ACC_COLS = 256, STAGES = 4;
  CUtensorMap am;  // V as [T*k][f] fp16, box {64, 128}
  CUtensorMap bm;  // down in fp16 as [E*L][f], box {64, 256}
  int L, f, E;
  const int32_t* eo;
  const int32_t* sa;
  const float* wts;  // [T*k]
  __half* U;  // [T*k][L] by sorted position
  LMOE_DEV int ntn() const { return L / 256; }
  LMOE_DEV void init(int* sc) const {
    tile_prefix(sc, E, [&](int e) { return ((eo[e + 1] - eo[e] + 127) / 128) * ntn(); });
  }
  LMOE_DEV int num_tiles(const int* sc) const { return sc[E]; }
  LMOE_DEV Tile tile(const int* sc, int t) const {
    Tile tl;
    const int e = find_prob(sc, E, t), loc = t - sc[e];
    tl.prob = e;
    tl.m0 = (loc / ntn()) * 128;
    tl.n0 = (loc % ntn()) * 256;
    tl.rows = min(128, eo[e + 1] - eo[e] - tl.m0);
    tl.nkb = f / 64;
    tl.gm = 0;
    tl.arow = eo[e] + tl.m0;
    return tl;
  }
  // A: the expert's rows of V (rows past its range belong to the next expert
  // or read as zero; their outputs are not stored)
  LMOE_DEV void load_a(const Tile& tl, int kb, void* dst, uint64_t* bar) const {
    tma_load_2d(dst, &am, kb * 64, tl.arow, bar);
  }
  LMOE_DEV void load_b(const Tile& tl, int kb, void* dst, uint64_t* bar) const {
    tma_load_2d(dst, &bm, kb * 64, tl.prob * L + tl.n0, bar);
  }
  LMOE_DEV void mma_stage(const Tile&, int kb, uint32_t d_tmem, uint64_t da, uint64_t db) const {
    mma_k4(d_tmem, da, db, tc::idesc(128, 256, 0), kb);
  }
  LMOE_DEV void epilogue(const int*, const Tile& tl, int row, uint32_t tbase, int half) const {
    const bool valid = row < tl.rows;
    const int p = tl.arow + row;
    const float wt = valid ? wts[sa[p]] : 0.f;
    int lo, hi;
    epi_cols(half, 256, lo, hi);
    for (int c0 = lo; c0 < hi; c0 += 16) {
      float v[16];
      tc::tmem_ld16(tbase + (uint32_t)c0, v);
      if (!valid) continue;
      uint4* dst = reinterpret_cast<uint4*>(U + (size_t)p * L + tl.n0 + c0);
#pragma unroll
      for (int i = 0; i < 2; ++i)
        dst[i] = make_uint4(pack_half2(wt * v[8 * i], wt * v[8 * i + 1]), pack_half2(wt * v[8 * i + 2], wt * v[8 * i + 3]),
                            pack_half2(wt * v[8 * i + 4], wt * v[8 * i + 5]), pack_half2(wt * v[8 * i + 6], wt * v[8 * i + 7]));
    }
  }
};

// ------------------------------------------------------------------- W_out
// mode 0: y_t = sum_g Wout[g] Z[(g,t)] (+ residual), tiles over tokens, K = G*L
// mode 1: Y[(g,t)] = Wout[g] Z[(g,t)] (fp32 rows), tiles over group rows
struct ProbWout : ProbBase {
  static constexpr int BN = 256, ACC_COLS = 256, STAGES = 4;
  CUtensorMap bm;         // Wout in fp16 as [G][d][L], box {64, 256, 1}
  CUtensorMap am;         // mode 0: Z by token as [T][G*L] (zero rows for absent (t, g));
                          // mode 1: Z by group rows as [rows][L]; box {64, 128}
  const int32_t* gto;
  int T, d, L, G, mode;
  const uint16_t* residual;
  uint16_t* y;  // [T][d] bf16 (mode 0)
  float* Y;     // [rows][d] (mode 1)
  // mode 0, sorted: A row p is token tsort[p], and token tile j reads only
  // the K blocks of the groups in tunion[j]
  const int32_t* tsort;
  const uint32_t* tunion;
  // Recover-LoRA (rp > 0): after a group's L/64 K blocks of Z come rp/64 K
  // blocks of Q = Z . A_out[g] against B_out[g]^T, so the accumulator takes
  // [Z | Q] . [Wout[g] ; B_out[g]] for each group
  CUtensorMap qm;   // mode 0: Q as [T][G*rp] (A's row order); mode 1: [rows][rp]; box {64, 128}
  CUtensorMap lbm;  // B_out^T in fp16 as [G][d][rp], box {64, 256, 1}
  int rp;
  LMOE_DEV int ntn() const { return d / 256; }
  // K blocks per group (LoRA included) and its multiply-high reciprocal:
  // kb / kpg2 = umulhi(kb, kdiv) for every kb < 2^32 / kpg2 (kdiv = ceil(2^32 / kpg2),
  // set on the host). The K-block split runs on the one TMA-issuing thread
  // for every K block, where a hardware-less integer division would cost
  // about as much as the block's MMAs.
  int kpg_, kpg2_, kshift;  // L/64, (L+rp)/64, log2(kpg2_) or -1 when kpg2_ is not a power of two
  unsigned kdiv;
  LMOE_DEV int kpg() const { return kpg_; }
  LMOE_DEV int kpg2() const { return kpg2_; }
  // K block kb -> (its group's index within the tile's set, K block within the group)
  LMOE_DEV void ksplit(int kb, int& i, int& w) const {
    if (kshift >= 0) {
      i = kb >> kshift;
      w = kb & (kpg2_ - 1);
    } else {
      i = (int)__umulhi((unsigned)kb, kdiv);
      w = kb - i * kpg2_;
    }
  }
  // the group of a mode-0 tile's K-block group index i: the i-th set bit of
  // its set, from the tile's packed list when G <= 16 and the set has at
  // most 8 groups
  LMOE_DEV int kgroup(const Tile& tl, int i) const {
    if (i < 8 && G <= 16) return (int)((tl.gl >> (4 * i)) & 15u);
    unsigned m = tl.gm;
#pragma unroll 1
    for (; i > 0; --i) m &= m - 1u;
    return __ffs(m) - 1;
  }
  LMOE_DEV void init(int* sc) const {
    if (mode == 1) tile_prefix(sc, G, [&](int g) { return ((gto[g + 1] - gto[g] + 127) / 128) * ntn(); });
  }
  LMOE_DEV int num_tiles(const int* sc) const { return mode == 0 ? ((T + 127) / 128) * ntn() : sc[G]; }
  LMOE_DEV Tile tile(const int* sc, int t) const {
    Tile tl;
    if (mode == 0) {
      tl.prob = 0;
      tl.m0 = (t / ntn()) * 128;
      tl.n0 = (t % ntn()) * 256;
      tl.rows = min(128, T - tl.m0);
      tl.gm = tsort ? tunion[t / ntn()] : (G >= 32 ? 0xffffffffu : (1u << G) - 1u);
      tl.nkb = __popc(tl.gm) * kpg2();
      tl.arow = tl.m0;
      tl.gl = 0;
      unsigned m = tl.gm;
      for (int i = 0; i < 8 && m; ++i, m &= m - 1u) tl.gl |= (unsigned)(__ffs(m) - 1) << (4 * i);
    } else {
      const int g = find_prob(sc, G, t), loc = t - sc[g];
      tl.prob = g;
      tl.m0 = (loc / ntn()) * 128;
      tl.n0 = (loc % ntn()) * 256;
      tl.rows = min(128, gto[g + 1] - gto[g] - tl.m0);
      tl.nkb = kpg2();
      tl.gm = 0;
      tl.arow = gto[g] + tl.m0;
    }
    return tl;
  }
  static constexpr bool KPREP = true;
  struct KC {
    const CUtensorMap* am;  // A: Z or Q
    const CUtensorMap* bm;  // B: Wout or B_out
    int ax, ay, bx, by, bz;
  };
  LMOE_DEV KC kprep(const Tile& tl, int kb) const {
    int i, w;
    ksplit(kb, i, w);
    const int g = mode == 0 ? kgroup(tl, i) : tl.prob;
    const bool z = rp == 0 || w < kpg();  // a K block of Z (else of Q)
    KC c;
    c.am = z ? &am : &qm;
    c.bm = z ? &bm : &lbm;
    const int wx = (z ? w : w - kpg()) * 64;
    c.ax = mode == 0 ? g * (z ? L : rp) + wx : wx;
    c.ay = tl.arow;
    c.bx = wx;
    c.by = tl.n0;
    c.bz = g;
    return c;
  }
  LMOE_DEV void kissue(const KC& c, void* da, void* db, uint64_t* bar) const {
    tma_load_2d(da, c.am, c.ax, c.ay, bar);
    tma_load_3d(db, c.bm, c.bx, c.by, c.bz, bar);
  }
  LMOE_DEV void load_a(const Tile& tl, int kb, void* dst, uint64_t* bar) const {
    int i, w;  // group index in the tile's set, K block within the group
    ksplit(kb, i, w);
    const bool z = rp == 0 || w < kpg();  // a K block of Z (else of Q)
    if (mode == 0) {
      const int g = kgroup(tl, i);
      if (z) tma_load_2d(dst, &am, g * L + w * 64, tl.arow, bar);
      else tma_load_2d(dst, &qm, g * rp + (w - kpg()) * 64, tl.arow, bar);
    } else {  // rows past the group's range belong to the next group or read as zero; not stored
      if (z) tma_load_2d(dst, &am, w * 64, tl.arow, bar);
      else tma_load_2d(dst, &qm, (w - kpg()) * 64, tl.arow, bar);
    }
  }
  LMOE_DEV void load_b(const Tile& tl, int kb, void* dst, uint64_t* bar) const {
    int i, w;
    ksplit(kb, i, w);
    const int g = mode == 0 ? kgroup(tl, i) : tl.prob;
    if (rp == 0 || w < kpg()) tma_load_3d(dst, &bm, w * 64, tl.n0, g, bar);
    else tma_load_3d(dst, &lbm, (w - kpg()) * 64, tl.n0, g, bar);
  }
  LMOE_DEV void mma_stage(const Tile&, int kb, uint32_t d_tmem, uint64_t da, uint64_t db) const {
    mma_k4(d_tmem, da, db, tc::idesc(128, 256, 0), kb);
  }
  LMOE_DEV void epilogue(const int*, const Tile& tl, int row, uint32_t tbase, int half) const {
    const bool valid = row < tl.rows;
    int lo, hi;
    epi_cols(half, 256, lo, hi);
    for (int c0 = lo; c0 < hi; c0 += 16) {
      float v[16];
      tc::tmem_ld16(tbase + (uint32_t)c0, v);
      if (!valid) continue;
      if (mode == 0) {
        const size_t o = (size_t)(tsort ? tsort[tl.m0 + row] : tl.m0 + row) * d + tl.n0 + c0;
        uint32_t h[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float a = v[2 * i], b = v[2 * i + 1];
          if (residual) {
            a += bf16_to_f32(residual[o + 2 * i]);
            b += bf16_to_f32(residual[o + 2 * i + 1]);
          }
          h[i] = (uint32_t)f32_to_bf16_rne(a) | ((uint32_t)f32_to_bf16_rne(b) << 16);
        }
        uint4* d4 = reinterpret_cast<uint4*>(y + o);
        d4[0] = make_uint4(h[0], h[1], h[2], h[3]);
        d4[1] = make_uint4(h[4], h[5], h[6], h[7]);
      } else {
        float4* dst = reinterpret_cast<float4*>(Y + (size_t)(tl.arow + row) * d + tl.n0 + c0);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      }
    }
  }
};

// ------------------------------------------------------------ Recover-LoRA
// P = x . A_in for every group at once: [T][d] x [d][G*rp] -> fp16 [T][G*rp]
// (rows in x16's order; the rank padded to rp with zero columns)
struct ProbLoraP : ProbBase {
  static constexpr int BN = 256, ACC_COLS = 256, STAGES = 4;
  CUtensorMap am;  // x in fp16 as [T][d], box {64, 128}
  CUtensorMap bm;  // A_in^T in fp16 as [G*rp][d] (rows past G*rp read as zero), box {64, 256}
  int T, d, N;     // N = G*rp
  __half* P;
  LMOE_DEV int ntn() const { return (N + 255) / 256; }
  LMOE_DEV void init(int*) const {}
  LMOE_DEV int num_tiles(const int*) const { return ((T + 127) / 128) * ntn(); }
  LMOE_DEV Tile tile(const int*, int t) const {
    Tile tl;
    tl.prob = 0;
    tl.m0 = (t / ntn()) * 128;
    tl.n0 = (t % ntn()) * 256;
    tl.rows = min(128, T - tl.m0);
    tl.nkb = d / 64;
    tl.gm = 0;
    tl.arow = tl.m0;
    return tl;
  }
  LMOE_DEV void load_a(const Tile& tl, int kb, void* dst, uint64_t* bar) const {
    tma_load_2d(dst, &am, kb * 64, tl.m0, bar);
  }
  LMOE_DEV void load_b(const Tile& tl, int kb, void* dst, uint64_t* bar) const {
    tma_load_2d(dst, &bm, kb * 64, tl.n0, bar);
  }
  LMOE_DEV void mma_stage(const Tile&, int kb, uint32_t d_tmem, uint64_t da, uint64_t db) const {
    mma_k4(d_tmem, da, db, tc::idesc(128, 256, 0), kb);
  }
  LMOE_DEV void epilogue(const int*, const Tile& tl, int row, uint32_t tbase, int half) const {
    int lo, hi;
    epi_cols(half, 256, lo, hi);
    for (int c0 = lo; c0 < hi; c0 += 16) {
      float v[16];
      tc::tmem_ld16(tbase + (uint32_t)c0, v);
      if (row < tl.rows && tl.n0 + c0 < N) store_half16(P + (size_t)(tl.m0 + row) * N + tl.n0 + c0, v);
    }
  }
};

// Q = Z . A_out[g] per group, 64 columns of the padded rank per tile:
// mode 0: Z by token ([T][G*L], A's row order), Q as [T][G*rp]; with the
//         group -> token-tile lists only the tiles whose groups hold g
// mode 1: Z by group rows ([rows][L]), Q as [rows][rp]
struct ProbLoraQ : ProbBase {
  static constexpr int BN = 64, ACC_COLS = 64, STAGES = 4;
  CUtensorMap am;  // Z, box {64, 128}
  CUtensorMap bm;  // A_out^T in fp16 as [G][rp][L], box {64, 64, 1}
  const int32_t* gto;
  const int* gtc;  // mode 0: null = every (token tile, group)
  const int* gtl;
  int T, L, G, rp, mode;
  __half* Q;
  LMOE_DEV int rpk() const { return rp / 64; }
  LMOE_DEV int ntm() const { return (T + 127) / 128; }
  LMOE_DEV void init(int* sc) const {
    if (mode == 1) tile_prefix(sc, G, [&](int g) { return ((gto[g + 1] - gto[g] + 127) / 128) * rpk(); });
    else if (gtc) tile_prefix(sc, G, [&](int g) { return gtc[g] * rpk(); });
  }
  LMOE_DEV int num_tiles(const int* sc) const { return (mode == 1 || gtc) ? sc[G] : G * ntm() * rpk(); }
  LMOE_DEV Tile tile(const int* sc, int t) const {
    Tile tl;
    int loc;
    if (mode == 1 || gtc) {
      tl.prob = find_prob(sc, G, t);
      loc = t - sc[tl.prob];
    } else {
      tl.prob = t / (ntm() * rpk());
      loc = t % (ntm() * rpk());
    }
    const int mi = loc / rpk();
    tl.n0 = (loc % rpk()) * 64;
    if (mode == 1) {
      tl.m0 = mi * 128;
      tl.rows = min(128, gto[tl.prob + 1] - gto[tl.prob] - tl.m0);
      tl.arow = gto[tl.prob] + tl.m0;
    } else {
      tl.m0 = (gtc ? gtl[tl.prob * ntm() + mi] : mi) * 128;
      tl.rows = min(128, T - tl.m0);
      tl.arow = tl.m0;
    }
    tl.nkb = L / 64;
    tl.gm = 0;
    return tl;
  }
  LMOE_DEV void load_a(const Tile& tl, int kb, void* dst, uint64_t* bar) const {
    if (mode == 0) tma_load_2d(dst, &am, tl.prob * L + kb * 64, tl.arow, bar);
    else tma_load_2d(dst, &am, kb * 64, tl.arow, bar);  // rows past the group: not stored
  }
  LMOE_DEV void load_b(const Tile& tl, int kb, void* dst, uint64_t* bar) const {
    tma_load_3d(dst, &bm, kb * 64, tl.n0, tl.prob, bar);
  }
  LMOE_DEV void mma_stage(const Tile&, int kb, uint32_t d_tmem, uint64_t da, uint64_t db) const {
    mma_k4(d_tmem, da, db, tc::idesc(128, 64, 0), kb);
  }
  LMOE_DEV void epilogue(const int*, const Tile& tl, int row, uint32_t tbase, int half) const {
    const bool valid = row < tl.rows;
    __half* out = mode == 0 ? Q + (size_t)(tl.m0 + row) * G * rp + tl.prob * rp + tl.n0
                            : Q + (size_t)(tl.arow + row) * rp + tl.n0;
    int lo, hi;
    epi_cols(half, 64, lo, hi);
    for (int c0 = lo; c0 < hi; c0 += 16) {
      float v[16];
      tc::tmem_ld16(tbase + (uint32_t)c0, v);
      if (valid) store_half16(out + c0, v);
    }
  }
};

// ----------------------------------------------------------------- zreduce
// One warp per (group, token) row: Z[row] = sum over the token's experts in
// that group, in ascending j, of U[inv[t*k + j]]; tokrow[t][g] = row.
// One warp: out[0 .. L) = sum over the set bits j of `mask`, ascending, of
// the fp16 rows U + r_j * L, in fp32, rounded to fp16; lane j holds r_j (the
// row indices come in one parallel load, not one dependent load per row).
// Each pass over j loads four 256-element runs of the row at once.
LMOE_DEV void sum_rows_f16(const __half* __restrict__ U, int my_row, unsigned mask, int L, __half* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  for (int c0 = 0; c0 < L; c0 += 1024) {
    float acc[4][8];
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int h = 0; h < 8; ++h) acc[q][h] = 0.f;
    unsigned m = mask;  // warp-uniform
    while (m) {
      const int rj = __shfl_sync(0xffffffffu, my_row, __ffs(m) - 1);
      m &= m - 1u;
      uint4 u[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int c = c0 + q * 256 + lane * 8;
        u[q] = c < L ? __ldcs(reinterpret_cast<const uint4*>(U + (size_t)rj * L + c)) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t w[4] = {u[q].x, u[q].y, u[q].z, u[q].w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[h]));
          acc[q][2 * h] += f.x;
          acc[q][2 * h + 1] += f.y;
        }
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int c = c0 + q * 256 + lane * 8;
      if (c < L)
        *reinterpret_cast<uint4*>(out + c) = make_uint4(pack_half2(acc[q][0], acc[q][1]), pack_half2(acc[q][2], acc[q][3]),
                                                        pack_half2(acc[q][4], acc[q][5]), pack_half2(acc[q][6], acc[q][7]));
    }
  }
}

// Mode-1 Z rows: Z[row] for row = (g, t) of the group-token lists, one warp
// per row (k <= 32).
__global__ void zreduce_kernel(const __half* __restrict__ U, const int32_t* __restrict__ idx,
                               const int32_t* __restrict__ inv, const int32_t* __restrict__ gto, const int32_t* __restrict__ gtok, int G, int k, int epg,
                               int L, __half* __restrict__ Z, int32_t* __restrict__ tokrow) {
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= gto[G]) return;
  int g = 0;
  while (g + 1 < G && gto[g + 1] <= row) ++g;
  const int t = gtok[row];
  if (lane == 0) tokrow[(size_t)t * G + g] = row;
  const bool mine = lane < k && idx[(size_t)t * k + lane] / epg == g;
  const unsigned mask = __ballot_sync(0xffffffffu, mine);
  sum_rows_f16(U, mine ? inv[(size_t)t * k + lane] : 0, mask, L, Z + (size_t)row * L);
}

// Mode-0 operand of W_out: Ztok[t][g][:] = sum over the token's experts in
// group g, in ascending j, of U[inv[t*k + j]], or zero when the token has no
// expert in g. One warp per (t, g) (k <= 32).
__global__ void zreduce_tok_kernel(const __half* __restrict__ U, const int32_t* __restrict__ idx,
                                   const int32_t* __restrict__ inv, int T, int G, int k, int epg, int L,
                                   const int32_t* __restrict__ tpos, __half* __restrict__ Ztok) {
  const int item = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (item >= T * G) return;
  const int t = item / G, g = item % G;
  const bool mine = lane < k && idx[(size_t)t * k + lane] / epg == g;
  const unsigned mask = __ballot_sync(0xffffffffu, mine);
  const int row = tpos ? tpos[t] : t;  // the token's row in the sorted order (or its own)
  sum_rows_f16(U, mine ? inv[(size_t)t * k + lane] : 0, mask, L, Ztok + ((size_t)row * G + g) * L);
}

// ------------------------------------------------------------- token order
// Tokens in a stable order of the set of groups they route into (G <= 8: an
// 8-bit mask), so that a 128-token tile of the order holds few distinct sets.
// Three passes (no result depends on the order of atomics): masks and
// per-block histograms; offsets; ranks within a block by warp match and
// per-warp counts. Then the union of the sets per tile and, per group, the
// tiles whose union holds it.
constexpr int TS_TB = 1024;

__global__ void __launch_bounds__(TS_TB) tsort_count_kernel(const int32_t* __restrict__ idx, int T, int k, int epg,
                                                            uint8_t* __restrict__ mask, int* __restrict__ bh) {
  __shared__ int h[256];
  if (threadIdx.x < 256) h[threadIdx.x] = 0;
  __syncthreads();
  const int t = blockIdx.x * TS_TB + threadIdx.x;
  if (t < T) {
    unsigned m = 0;
    for (int j = 0; j < k; ++j) m |= 1u << (idx[(size_t)t * k + j] / epg);
    mask[t] = (uint8_t)m;
    atomicAdd(&h[m & 255u], 1);
  }
  __syncthreads();
  if (threadIdx.x < 256) bh[blockIdx.x * 256 + threadIdx.x] = h[threadIdx.x];
}

// one block of 256 threads: bh[b][m] -> first position of block b's tokens of set m
__global__ void __launch_bounds__(256) tsort_scan_kernel(int* __restrict__ bh, int nb) {
  __shared__ int tot[256];
  const int m = threadIdx.x;
  int s = 0;
  for (int b = 0; b < nb; ++b) s += bh[b * 256 + m];
  tot[m] = s;
  __syncthreads();
  if (m == 0) {
    int run = 0;
    for (int i = 0; i < 256; ++i) {
      const int c = tot[i];
      tot[i] = run;
      run += c;
    }
  }
  __syncthreads();
  int run = tot[m];
  for (int b = 0; b < nb; ++b) {
    const int c = bh[b * 256 + m];
    bh[b * 256 + m] = run;
    run += c;
  }
}

__global__ void __launch_bounds__(TS_TB) tsort_scatter_kernel(const uint8_t* __restrict__ mask, int T,
                                                              const int* __restrict__ bh, int32_t* __restrict__ tsort,
                                                              int32_t* __restrict__ tpos) {
  __shared__ int wc[TS_TB / 32][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < (TS_TB / 32) * 256; i += TS_TB) (&wc[0][0])[i] = 0;
  __syncthreads();
  const int t = blockIdx.x * TS_TB + threadIdx.x;
  const unsigned m = t < T ? mask[t] : 256u;  // 256: no token
  const unsigned peers = __match_any_sync(0xffffffffu, m);
  const int rank = __popc(peers & ((1u << lane) - 1u));
  if (m < 256u && rank == 0) wc[warp][m] = __popc(peers);
  __syncthreads();
  if (m < 256u) {
    int pre = 0;
    for (int w = 0; w < warp; ++w) pre += wc[w][m];
    const int pos = bh[blockIdx.x * 256 + m] + pre + rank;
    tsort[pos] = t;
    tpos[t] = pos;
  }
}

// one block: tunion[j] = OR of the sets of tile j's tokens; per group g, the
// tiles whose union holds g, ascending: gtl[g][0 .. gtc[g])
__global__ void __launch_bounds__(1024) tsort_tiles_kernel(const uint8_t* __restrict__ mask,
                                                           const int32_t* __restrict__ tsort, int T, int G,
                                                           uint32_t* __restrict__ tunion, int* __restrict__ gtc,
                                                           int* __restrict__ gtl) {
  constexpr int SU = 4096;  // unions kept in shared memory (T <= 524288 tokens; beyond, read back from tunion)
  __shared__ uint32_t su[SU];
  const int nt = (T + 127) / 128, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int j = warp; j < nt; j += 32) {
    unsigned u = 0;
    for (int p = j * 128 + lane; p < min(T, j * 128 + 128); p += 32) u |= mask[tsort[p]];
    for (int o = 16; o > 0; o >>= 1) u |= __shfl_xor_sync(0xffffffffu, u, o);
    if (lane == 0) {
      tunion[j] = u;
      if (j < SU) su[j] = u;
    }
  }
  __syncthreads();
  // warp g: the tiles whose union holds group g, in order, 32 tiles per ballot
  if (warp < G) {
    const int g = warp;
    int c = 0;
    for (int j0 = 0; j0 < nt; j0 += 32) {
      const int j = j0 + lane;
      const bool in = j < nt && (((j < SU ? su[j] : __ldcg(tunion + j)) >> g) & 1u);
      const unsigned b = __ballot_sync(0xffffffffu, in);
      if (in) gtl[g * nt + c + __popc(b & ((1u << lane) - 1u))] = j;
      c += __popc(b);
    }
    if (lane == 0) gtc[g] = c;
  }
}

// x (bf16) to fp16 rows in the token order: x16[p] = x[tsort[p]]
__global__ void __launch_bounds__(256) x_sorted_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ tsort,
                                                       int T, int d8, uint4* __restrict__ x16) {
  const size_t n = (size_t)T * d8, stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += stride) {
    const size_t p = i / d8, c = i % d8;
    const uint4 v = __ldcs(x + (size_t)tsort[p] * d8 + c);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
    uint32_t h[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) h[j] = pack_half2(__uint_as_float(u[j] << 16), __uint_as_float(u[j] & 0xffff0000u));
    x16[i] = make_uint4(h[0], h[1], h[2], h[3]);
  }
}

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

// Every int4 matrix to fp16 and x to fp16, in one launch. An int4 matrix of
// rows [rows][K/2] with bf16 scales [rows][K/32] is a run of 32-bit words of
// 8 elements each, 4 words per scale group, and its fp16 copy the matching
// run of 16-byte words: a warp takes 32 consecutive words, so both its loads
// and its stores are contiguous.
struct DqSeg {
  const uint32_t* q;
  const uint16_t* s;
  uint4* out;
  size_t n;  // 32-bit words
  // NVFP4: E2M1 codes with one E4M3 byte per 2 words and a per-tensor scale
  // (tensor = wpt consecutive words); the fp16 copy holds e2m1 * e4m3 * gs,
  // rounded once
  int fp4;
  const float* gs;
  size_t wpt;
};
struct DqJob {
  DqSeg seg[5];
  int nseg;
  const uint4* x;  // bf16, 8 per 16-byte word
  uint4* x16;
  size_t nx;
};

__global__ void __launch_bounds__(256) dequant_all_kernel(const __grid_constant__ DqJob J) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x, base = 0;
#pragma unroll 1
  for (int g = 0; g < J.nseg; ++g) {
    const DqSeg S = J.seg[g];
#pragma unroll 4
    for (; i < base + S.n; i += stride) {
      const size_t w = i - base;
      uint32_t o[4];
      if (S.fp4) {
        const uint8_t sb = __ldg(reinterpret_cast<const uint8_t*>(S.s) + (w >> 1));
        const uint32_t sh = e4m3x2_to_h2(sb);
        const float sc = __low2float(*reinterpret_cast<const __half2*>(&sh)) * __ldg(S.gs + w / S.wpt);
        e2m1x8_to_h2x4(__ldcs(S.q + w), o);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&o[j]));
          const __half2 h = __floats2half2_rn(f.x * sc, f.y * sc);
          o[j] = *reinterpret_cast<const uint32_t*>(&h);
        }
      } else {
        tc::dequant_word_natural(__ldcs(S.q + w), scale_h2(__ldg(S.s + (w >> 2))), o);
      }
      __stcs(S.out + w, make_uint4(o[0], o[1], o[2], o[3]));
    }
    base += S.n;
  }
#pragma unroll 4
  for (; i < base + J.nx; i += stride) {
    const uint4 v = __ldcs(J.x + (i - base));
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
    uint32_t h[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) h[j] = pack_half2(__uint_as_float(u[j] << 16), __uint_as_float(u[j] & 0xffff0000u));
    J.x16[i - base] = make_uint4(h[0], h[1], h[2], h[3]);
  }
}

// The Recover-LoRA matrices, bf16 [G][R][C], to transposed fp16 copies
// [G][Cp][Rp] (out[g][c][q] = in[g][q][c]; zero for q >= R or c >= C, the
// rank's padding), 32 x 32 tiles through shared memory. bf16 -> fp16 is
// exact from 2^-14 up to 65504; below 2^-14 it rounds to the fp16 subnormal
// grid (error <= 2^-25); a finite value that overflows sets BAD_DATA.
struct LoraT16 {
  const uint16_t* in;
  __half* out;
  int R, C, Rp, Cp;
  LMOE_DEV int tiles() const { return ((Cp + 31) / 32) * ((Rp + 31) / 32); }
};
struct LoraT16Job {
  LoraT16 m[4];
  int G;
  unsigned* err;
};

__global__ void __launch_bounds__(256) lora_t16_kernel(const __grid_constant__ LoraT16Job J) {
  __shared__ float tile[32][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  int per[4], total = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) total += (per[i] = J.G * J.m[i].tiles());
#pragma unroll 1
  for (int b = blockIdx.x; b < total; b += gridDim.x) {
    int i = 0, loc = b;
    while (loc >= per[i]) loc -= per[i++];
    const LoraT16 M = J.m[i];
    const int ntq = (M.Rp + 31) / 32, per_g = M.tiles();
    const int g = loc / per_g, c0 = ((loc % per_g) / ntq) * 32, q0 = ((loc % per_g) % ntq) * 32;
    bool bad = false;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int q = q0 + ty + 8 * j, c = c0 + tx;
      float v = 0.f;
      if (q < M.R && c < M.C) {
        v = bf16_to_f32(M.in[((size_t)g * M.R + q) * M.C + c]);
        bad |= fabsf(v) < INFINITY && fabsf(__half2float(__float2half_rn(v))) == INFINITY;
      }
      tile[ty + 8 * j][tx] = v;
    }
    if (bad) set_error(J.err, ERRBIT_BAD_DATA);
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = c0 + ty + 8 * j, q = q0 + tx;
      if (c < M.Cp && q < M.Rp) M.out[((size_t)g * M.Cp + c) * M.Rp + q] = __float2half_rn(tile[tx][ty + 8 * j]);
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ host side

namespace {

constexpr size_t kAl = 256;
size_t al(size_t v) { return (v + kAl - 1) & ~(kAl - 1); }

struct PWs {
  size_t logits, rpart, idx, w, eo, sa, inv, go, gto, gt, ar, perm_scratch, H, V, U, Z, tokrow, x16, win16, wout16, gate16, up16,
      down16, ztok, tmask, tsort, tpos, tbh, tunion, gtc, gtl, ain16, bin16, aout16, bout16, lp, lq, end;
};

// the LoRA rank padded to whole K blocks of 64 (0: no branch)
int lora_rp(const PrefillArgs& P) { return (P.r + 63) / 64 * 64; }

PWs pws(const PrefillArgs& P, int T) {
  PWs m;
  size_t o = 0;
  auto take = [&](size_t b) {
    size_t at = o;
    o = al(o + b);
    return at;
  };
  const size_t n = (size_t)T * P.k, gk = (size_t)T * (P.G < P.k ? P.G : P.k);
  m.logits = take((size_t)T * P.E * 4);
  m.rpart = take((size_t)(P.num_sms > 0 ? P.num_sms : 1) * 128 * 256 * 4);  // the router's running sums
  m.idx = take(n * 4);
  m.w = take(n * 4);
  m.eo = take((size_t)(P.E + 1) * 4);
  m.sa = take(n * 4);
  m.inv = take(n * 4);
  m.go = take((size_t)(P.G + 1) * 4);
  m.gto = take((size_t)(P.G + 1) * 4);
  m.gt = take(gk * 4);
  m.ar = take(n * 4);
  m.perm_scratch = take(permute_scratch_bytes(T, P.E, P.G));
  m.H = take(n * P.L * 2);
  m.V = take(n * P.f * 2);
  m.U = take(n * P.L * 2);
  m.Z = take(gk * P.L * 2);
  m.tokrow = take((size_t)T * P.G * 4);
  m.x16 = take((size_t)T * P.d * 2);
  m.win16 = take((size_t)P.G * P.L * P.d * 2);
  m.wout16 = take((size_t)P.G * P.d * P.L * 2);
  m.gate16 = take((size_t)P.E * P.f * P.L * 2);
  m.up16 = take((size_t)P.E * P.f * P.L * 2);
  m.down16 = take((size_t)P.E * P.L * P.f * 2);
  m.ztok = take((size_t)T * P.G * P.L * 2);
  const size_t nt = (size_t)(T + 127) / 128, nb = (size_t)(T + TS_TB - 1) / TS_TB;
  m.tmask = take((size_t)T);
  m.tsort = take((size_t)T * 4);
  m.tpos = take((size_t)T * 4);
  m.tbh = take(nb * 256 * 4);
  m.tunion = take(nt * 4);
  m.gtc = take((size_t)P.G * 4);
  m.gtl = take((size_t)P.G * nt * 4);
  // Recover-LoRA: the transposed fp16 matrices, P = x . A_in and Q = Z . A_out
  const size_t rp = (size_t)lora_rp(P);
  m.ain16 = take((size_t)P.G * rp * P.d * 2);
  m.bin16 = take((size_t)P.G * P.L * rp * 2);
  m.aout16 = take((size_t)P.G * rp * P.L * 2);
  m.bout16 = take((size_t)P.G * P.d * rp * 2);
  m.lp = take((size_t)T * P.G * rp * 2);
  m.lq = take((size_t)T * P.G * rp * 2);  // mode 1: rows (<= T*G) x rp
  m.end = o;
  return m;
}

template <class Prob>
cudaError_t set_attr() {
  return cudaFuncSetAttribute(tc::gemm_kernel<Prob>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              tc::smem_bytes<Prob>());
}

template <class Prob>
cudaError_t run_gemm(const Prob& p, int grid, cudaStream_t st) {
  tc::gemm_kernel<Prob><<<grid, tc::THREADS, tc::smem_bytes<Prob>(), st>>>(p);
  return cudaGetLastError();
}

struct EvHook {
  const std::vector<cudaEvent_t>* ev;
  int i = 0;
  void rec(cudaEvent_t e, cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
      cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
    else
      cudaEventRecord(e, s);
  }
  void before(cudaStream_t s) {
    if (ev && 2 * i < (int)ev->size()) rec((*ev)[2 * i], s);
  }
  void after(cudaStream_t s) {
    if (ev && 2 * i + 1 < (int)ev->size()) rec((*ev)[2 * i + 1], s);
    ++i;
  }
};

PermPtrs perm_ptrs(char* b, const PWs& m) {
  PermPtrs pm;
  pm.expert_offsets = reinterpret_cast<int32_t*>(b + m.eo);
  pm.sorted_assign = reinterpret_cast<int32_t*>(b + m.sa);
  pm.inv = reinterpret_cast<int32_t*>(b + m.inv);
  pm.group_offsets = reinterpret_cast<int32_t*>(b + m.go);
  pm.group_tok_offsets = reinterpret_cast<int32_t*>(b + m.gto);
  pm.group_tokens = reinterpret_cast<int32_t*>(b + m.gt);
  pm.assign_row = reinterpret_cast<int32_t*>(b + m.ar);
  return pm;
}

ProbBase base(const PrefillArgs& P) {
  ProbBase b;
  b.budget = P.timeout;
  b.err = P.err;
  return b;
}

// the token order of a layer call (all null: tokens in their own order)
struct TokOrder {
  const int32_t* tsort;
  const int32_t* tpos;
  const uint32_t* tunion;
  const int* gtc;
  const int* gtl;
};

// expert part of the layer after routing and permutation: win, gateup, down,
// zreduce, then wout (mode 0 -> y, mode 1 -> Yrows)
cudaError_t dequant(const PrefillArgs& P, const uint16_t* x, int T, char* b, const PWs& m, cudaStream_t st,
                    EvHook* hook, bool with_x);

cudaError_t experts(const PrefillArgs& P, const uint16_t* x, int T, const int32_t* idx, const float* w,
                    const PermPtrs& pm, char* b, const PWs& m, int mode, float* Yrows, const uint16_t* residual,
                    uint16_t* y, cudaStream_t st, EvHook* hook, bool dequant_here, const TokOrder& to) {
  const int grid = P.num_sms;
  __half* H = reinterpret_cast<__half*>(b + m.H);
  __half* V = reinterpret_cast<__half*>(b + m.V);
  __half* U = reinterpret_cast<__half*>(b + m.U);
  __half* Z = reinterpret_cast<__half*>(b + m.Z);
  int32_t* tokrow = reinterpret_cast<int32_t*>(b + m.tokrow);
  __half* x16 = reinterpret_cast<__half*>(b + m.x16);
  __half* win16 = reinterpret_cast<__half*>(b + m.win16);
  __half* wout16 = reinterpret_cast<__half*>(b + m.wout16);
  __half* gate16 = reinterpret_cast<__half*>(b + m.gate16);
  __half* up16 = reinterpret_cast<__half*>(b + m.up16);
  __half* down16 = reinterpret_cast<__half*>(b + m.down16);
  __half* ztok = reinterpret_cast<__half*>(b + m.ztok);
  const int rp = lora_rp(P);
  __half* lp = reinterpret_cast<__half*>(b + m.lp);
  __half* lq = reinterpret_cast<__half*>(b + m.lq);
  cudaError_t e;
  if (dequant_here) {
    const int at = hook ? hook->i : 0;
    if (hook) hook->i = 2;  // the dequant stage's slot
    if ((e = dequant(P, x, T, b, m, st, hook, to.tsort == nullptr)) != cudaSuccess) return e;
    if (hook) hook->i = at;
  }
  if (rp > 0) {  // lora_p: P = x . A_in for every group
    ProbLoraP p;
    static_cast<ProbBase&>(p) = base(P);
    {
      const cuuint64_t ad[2] = {(cuuint64_t)P.d, (cuuint64_t)T}, as[1] = {(cuuint64_t)P.d * 2};
      const cuuint32_t ab[2] = {64, 128};
      const cuuint64_t bd[2] = {(cuuint64_t)P.d, (cuuint64_t)P.G * rp}, bs[1] = {(cuuint64_t)P.d * 2};
      const cuuint32_t bb[2] = {64, 256};
      if (!tmap_encode(&p.am, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, x16, ad, as, ab, CU_TENSOR_MAP_SWIZZLE_128B) ||
          !tmap_encode(&p.bm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, b + m.ain16, bd, bs, bb, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    }
    p.T = T; p.d = P.d; p.N = P.G * rp; p.P = lp;
    if (hook) hook->before(st);
    if ((e = run_gemm(p, grid, st)) != cudaSuccess) return e;
    if (hook) hook->after(st);
  }
  {
    ProbWin p;
    static_cast<ProbBase&>(p) = base(P);
    {
      const cuuint64_t ad[2] = {(cuuint64_t)P.d, (cuuint64_t)T}, as[1] = {(cuuint64_t)P.d * 2};
      const cuuint32_t ab[2] = {64, 128};
      const cuuint64_t bd[3] = {(cuuint64_t)P.d, (cuuint64_t)P.L, (cuuint64_t)P.G};
      const cuuint64_t bs[2] = {(cuuint64_t)P.d * 2, (cuuint64_t)P.L * P.d * 2};
      const cuuint32_t bb[3] = {64, 256, 1};
      if (!tmap_encode(&p.am, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, x16, ad, as, ab, CU_TENSOR_MAP_SWIZZLE_128B) ||
          !tmap_encode(&p.bm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, win16, bd, bs, bb, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    }
    p.rp = rp;
    if (rp > 0) {
      const cuuint64_t pd[2] = {(cuuint64_t)P.G * rp, (cuuint64_t)T}, ps[1] = {(cuuint64_t)P.G * rp * 2};
      const cuuint32_t pb[2] = {64, 128};
      const cuuint64_t ld[3] = {(cuuint64_t)rp, (cuuint64_t)P.L, (cuuint64_t)P.G};
      const cuuint64_t ls[2] = {(cuuint64_t)rp * 2, (cuuint64_t)P.L * rp * 2};
      const cuuint32_t lb[3] = {64, 256, 1};
      if (!tmap_encode(&p.pm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, lp, pd, ps, pb, CU_TENSOR_MAP_SWIZZLE_128B) ||
          !tmap_encode(&p.lbm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, b + m.bin16, ld, ls, lb, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    }
    p.T = T; p.d = P.d; p.L = P.L; p.G = P.G; p.k = P.k; p.epg = P.epg; p.idx = idx; p.inv = pm.inv; p.H = H;
    p.tsort = to.tsort; p.gtc = to.gtc; p.gtl = to.gtl;
    if (hook) hook->before(st);
    if ((e = run_gemm(p, grid, st)) != cudaSuccess) return e;
    if (hook) hook->after(st);
  }
  {
    ProbGateUp p;
    static_cast<ProbBase&>(p) = base(P);
    p.L = P.L; p.f = P.f; p.E = P.E; p.eo = pm.expert_offsets;
    {
      const cuuint64_t dims[2] = {(cuuint64_t)P.L, (cuuint64_t)P.E * P.f}, strides[1] = {(cuuint64_t)P.L * 2};
      const cuuint32_t box[2] = {64, 128};
      const cuuint64_t ad[2] = {(cuuint64_t)P.L, (cuuint64_t)T * P.k}, as[1] = {(cuuint64_t)P.L * 2};
      if (!tmap_encode(&p.gm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, gate16, dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
          !tmap_encode(&p.um, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, up16, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
          !tmap_encode(&p.am, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, H, ad, as, box, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    }
    p.V = V;
    if (hook) hook->before(st);
    if ((e = run_gemm(p, grid, st)) != cudaSuccess) return e;
    if (hook) hook->after(st);
  }
  {
    ProbDown p;
    static_cast<ProbBase&>(p) = base(P);
    p.L = P.L; p.f = P.f; p.E = P.E; p.eo = pm.expert_offsets; p.sa = pm.sorted_assign; p.wts = w;
    {
      const cuuint64_t ad[2] = {(cuuint64_t)P.f, (cuuint64_t)T * P.k}, as[1] = {(cuuint64_t)P.f * 2};
      const cuuint32_t ab[2] = {64, 128};
      const cuuint64_t bd[2] = {(cuuint64_t)P.f, (cuuint64_t)P.E * P.L}, bs[1] = {(cuuint64_t)P.f * 2};
      const cuuint32_t bb[2] = {64, 256};
      if (!tmap_encode(&p.am, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, V, ad, as, ab, CU_TENSOR_MAP_SWIZZLE_128B) ||
          !tmap_encode(&p.bm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, down16, bd, bs, bb, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    }
    p.U = U;
    if (hook) hook->before(st);
    if ((e = run_gemm(p, grid, st)) != cudaSuccess) return e;
    if (hook) hook->after(st);
  }
  {
    if (hook) hook->before(st);
    if (mode == 0) {
      zreduce_tok_kernel<<<(T * P.G + 7) / 8, 256, 0, st>>>(U, idx, pm.inv, T, P.G, P.k, P.epg, P.L, to.tpos, ztok);
    } else {
      cudaMemsetAsync(tokrow, 0xff, (size_t)T * P.G * 4, st);
      const int rows_cap = T * (P.G < P.k ? P.G : P.k);
      zreduce_kernel<<<(rows_cap + 7) / 8, 256, 0, st>>>(U, idx, pm.inv, pm.group_tok_offsets, pm.group_tokens, P.G,
                                                        P.k, P.epg, P.L, Z, tokrow);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (hook) hook->after(st);
  }
  const int rows_cap = T * (P.G < P.k ? P.G : P.k);
  if (rp > 0) {  // lora_q: Q = Z . A_out[g]
    ProbLoraQ p;
    static_cast<ProbBase&>(p) = base(P);
    {
      const cuuint64_t ad0[2] = {(cuuint64_t)P.G * P.L, (cuuint64_t)T}, as0[1] = {(cuuint64_t)P.G * P.L * 2};
      const cuuint64_t ad1[2] = {(cuuint64_t)P.L, (cuuint64_t)rows_cap}, as1[1] = {(cuuint64_t)P.L * 2};
      const cuuint32_t ab[2] = {64, 128};
      const cuuint64_t bd[3] = {(cuuint64_t)P.L, (cuuint64_t)rp, (cuuint64_t)P.G};
      const cuuint64_t bs[2] = {(cuuint64_t)P.L * 2, (cuuint64_t)rp * P.L * 2};
      const cuuint32_t bb[3] = {64, 64, 1};
      if (!tmap_encode(&p.am, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, mode == 0 ? (const void*)ztok : (const void*)Z,
                       mode == 0 ? ad0 : ad1, mode == 0 ? as0 : as1, ab, CU_TENSOR_MAP_SWIZZLE_128B) ||
          !tmap_encode(&p.bm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, b + m.aout16, bd, bs, bb, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    }
    p.gto = pm.group_tok_offsets;
    p.gtc = mode == 0 ? to.gtc : nullptr;
    p.gtl = mode == 0 ? to.gtl : nullptr;
    p.T = T; p.L = P.L; p.G = P.G; p.rp = rp; p.mode = mode; p.Q = lq;
    if (hook) hook->before(st);
    if ((e = run_gemm(p, grid, st)) != cudaSuccess) return e;
    if (hook) hook->after(st);
  }
  {
    ProbWout p;
    static_cast<ProbBase&>(p) = base(P);
    {
      const cuuint64_t dims[3] = {(cuuint64_t)P.L, (cuuint64_t)P.d, (cuuint64_t)P.G};
      const cuuint64_t strides[2] = {(cuuint64_t)P.L * 2, (cuuint64_t)P.d * P.L * 2};
      const cuuint32_t box[3] = {64, 256, 1};
      if (!tmap_encode(&p.bm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, wout16, dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    }
    {
      const cuuint64_t ad0[2] = {(cuuint64_t)P.G * P.L, (cuuint64_t)T}, as0[1] = {(cuuint64_t)P.G * P.L * 2};
      const cuuint64_t ad1[2] = {(cuuint64_t)P.L, (cuuint64_t)rows_cap}, as1[1] = {(cuuint64_t)P.L * 2};
      const cuuint32_t ab[2] = {64, 128};
      if (!tmap_encode(&p.am, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, mode == 0 ? (const void*)ztok : (const void*)Z,
                       mode == 0 ? ad0 : ad1, mode == 0 ? as0 : as1, ab, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    }
    p.rp = rp;
    if (rp > 0) {
      const cuuint64_t qd0[2] = {(cuuint64_t)P.G * rp, (cuuint64_t)T}, qs0[1] = {(cuuint64_t)P.G * rp * 2};
      const cuuint64_t qd1[2] = {(cuuint64_t)rp, (cuuint64_t)rows_cap}, qs1[1] = {(cuuint64_t)rp * 2};
      const cuuint32_t qb[2] = {64, 128};
      const cuuint64_t ld[3] = {(cuuint64_t)rp, (cuuint64_t)P.d, (cuuint64_t)P.G};
      const cuuint64_t ls[2] = {(cuuint64_t)rp * 2, (cuuint64_t)P.d * rp * 2};
      const cuuint32_t lb[3] = {64, 256, 1};
      if (!tmap_encode(&p.qm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, lq, mode == 0 ? qd0 : qd1, mode == 0 ? qs0 : qs1, qb,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
          !tmap_encode(&p.lbm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, b + m.bout16, ld, ls, lb, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    }
    p.kpg_ = P.L / 64;
    p.kpg2_ = (P.L + rp) / 64;
    p.kshift = (p.kpg2_ & (p.kpg2_ - 1)) == 0 ? __builtin_ctz((unsigned)p.kpg2_) : -1;
    p.kdiv = (unsigned)(((1ull << 32) + (unsigned long long)p.kpg2_ - 1) / (unsigned long long)p.kpg2_);
    p.gto = pm.group_tok_offsets; p.T = T; p.d = P.d; p.L = P.L; p.G = P.G; p.mode = mode;
    p.tsort = mode == 0 ? to.tsort : nullptr;
    p.tunion = to.tunion;
    p.residual = residual; p.y = y; p.Y = Yrows;
    if (hook) hook->before(st);
    if ((e = run_gemm(p, grid, st)) != cudaSuccess) return e;
    if (hook) hook->after(st);
  }
  return cudaSuccess;
}

// every int4 matrix and x in fp16 (x16 in the workspace); once per call
cudaError_t dequant(const PrefillArgs& P, const uint16_t* x, int T, char* b, const PWs& m, cudaStream_t st,
                    EvHook* hook, bool with_x) {
  const int grid = P.num_sms;
  __half* x16 = reinterpret_cast<__half*>(b + m.x16);
  __half* win16 = reinterpret_cast<__half*>(b + m.win16);
  __half* wout16 = reinterpret_cast<__half*>(b + m.wout16);
  __half* gate16 = reinterpret_cast<__half*>(b + m.gate16);
  __half* up16 = reinterpret_cast<__half*>(b + m.up16);
  __half* down16 = reinterpret_cast<__half*>(b + m.down16);
  cudaError_t e;
  {
    if (hook) hook->before(st);
    DqJob J;
    const size_t wwords = (size_t)P.G * P.L * P.d / 8, ewords = (size_t)P.E * P.f * P.L / 8;
    const void* q[5] = {P.W_in_q, P.W_out_q, P.gate_q, P.up_q, P.down_q};
    const uint16_t* sc[5] = {P.W_in_s, P.W_out_s, P.gate_s, P.up_s, P.down_s};
    __half* out[5] = {win16, wout16, gate16, up16, down16};
    const float* gsp[5] = {P.W_in_gs, P.W_out_gs, P.gate_gs, P.up_gs, P.down_gs};
    for (int i = 0; i < 5; ++i) {
      J.seg[i].q = static_cast<const uint32_t*>(q[i]);
      J.seg[i].s = sc[i];
      J.seg[i].out = reinterpret_cast<uint4*>(out[i]);
      J.seg[i].n = i < 2 ? wwords : ewords;
      J.seg[i].fp4 = P.wfmt != 0;
      J.seg[i].gs = gsp[i];
      J.seg[i].wpt = i < 2 ? wwords / P.G : ewords / P.E;  // one group's / one expert's matrix
    }
    J.nseg = 5;
    J.x = reinterpret_cast<const uint4*>(x);
    J.x16 = reinterpret_cast<uint4*>(x16);
    J.nx = with_x ? (size_t)T * P.d / 8 : 0;
    dequant_all_kernel<<<8 * grid, 256, 0, st>>>(J);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int rp = lora_rp(P);
    if (rp > 0) {  // A_in^T [G*rp][d], B_in^T [G][L][rp], A_out^T [G][rp][L], B_out^T [G][d][rp]
      LoraT16Job L;
      L.m[0] = LoraT16{P.A_in, reinterpret_cast<__half*>(b + m.ain16), P.d, P.r, P.d, rp};
      L.m[1] = LoraT16{P.B_in, reinterpret_cast<__half*>(b + m.bin16), P.r, P.L, rp, P.L};
      L.m[2] = LoraT16{P.A_out, reinterpret_cast<__half*>(b + m.aout16), P.L, P.r, P.L, rp};
      L.m[3] = LoraT16{P.B_out, reinterpret_cast<__half*>(b + m.bout16), P.r, P.d, rp, P.d};
      L.G = P.G;
      L.err = P.err;
      lora_t16_kernel<<<4 * grid, 256, 0, st>>>(L);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (hook) hook->after(st);
  }
  return cudaSuccess;
}

cudaError_t route(const PrefillArgs& P, const uint16_t* x, int T, int32_t* idx, float* w, float* logits,
                  float* part, cudaStream_t st) {
  ProbRoute p;
  static_cast<ProbBase&>(p) = base(P);
  {
    const cuuint64_t ad[2] = {(cuuint64_t)P.d, (cuuint64_t)T}, as[1] = {(cuuint64_t)P.d * 2};
    const cuuint32_t ab[2] = {64, 128};
    const cuuint64_t bd[3] = {(cuuint64_t)P.d, (cuuint64_t)P.E, 3},
                     bs[2] = {(cuuint64_t)P.d * 2, (cuuint64_t)P.E * P.d * 2};
    const cuuint32_t bb[3] = {64, 256, 1};
    if (!tmap_encode(&p.am, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, ad, as, ab, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !tmap_encode(&p.bm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, P.W_r_split, bd, bs, bb, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  p.bias = P.b_r; p.T = T; p.d = P.d; p.E = P.E;
  p.logits = logits;
  p.part = part;
  cudaError_t e = run_gemm(p, P.num_sms, st);
  if (e != cudaSuccess) return e;
  route_topk_kernel<<<(T + 7) / 8, 256, 0, st>>>(logits, T, P.E, P.k, idx, w);
  return cudaGetLastError();
}

}  // namespace

cudaError_t prefill_set_attributes() {
  cudaError_t e;
  if ((e = set_attr<ProbRoute>()) != cudaSuccess) return e;
  if ((e = set_attr<ProbWin>()) != cudaSuccess) return e;
  if ((e = set_attr<ProbGateUp>()) != cudaSuccess) return e;
  if ((e = set_attr<ProbDown>()) != cudaSuccess) return e;
  if ((e = set_attr<ProbLoraP>()) != cudaSuccess) return e;
  if ((e = set_attr<ProbLoraQ>()) != cudaSuccess) return e;
  return set_attr<ProbWout>();
}

bool prefill_supported(const PrefillArgs& P) {
  if (P.r < 0 || P.r > 128) return false;
  if (P.d % 256 != 0 || P.L % 256 != 0 || P.f % 128 != 0) return false;
  if (P.E > 512 || P.k > 16 || P.G > 32) return false;  // top-k: E <= 512 logits per warp; group masks: 32 bits
  if (P.E % 4 != 0) return false;                         // logits rows by 16-byte words
  return P.num_sms > 0;
}

size_t prefill_workspace_bytes(const PrefillArgs& P, int T) {
  if (!prefill_supported(P) || T <= 0) return 0;
  return pws(P, T).end;
}

cudaError_t launch_prefill_route(const PrefillArgs& P, const uint16_t* x, int T, int32_t* idx, float* w,
                                 float* logits, void* ws, cudaStream_t st) {
  if (!logits) logits = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + pws(P, T).logits);
  return route(P, x, T, idx, w, logits, reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + pws(P, T).rpart), st);
}

cudaError_t launch_prefill_experts(const PrefillArgs& P, const uint16_t* x, int T, const int32_t* idx, const float* w,
                                   const PermPtrs& perm, float* Yrows, const uint16_t*, uint16_t*, void* ws,
                                   cudaStream_t st) {
  char* b = reinterpret_cast<char*>(ws);
  const PWs m = pws(P, T);
  return experts(P, x, T, idx, w, perm, b, m, 1, Yrows, nullptr, nullptr, st, nullptr, true, TokOrder{});
}

namespace {
// the layer on T tokens in a workspace laid out for at least T tokens (m);
// weights_ready: the fp16 weights are already in the workspace (made by
// launch_prefill_weights), so only x is converted
cudaError_t prefill_layer_impl(const PrefillArgs& P, const uint16_t* x, int T, const uint16_t* residual, uint16_t* y,
                               char* b, const PWs& m, cudaStream_t st, const std::vector<cudaEvent_t>* events,
                               bool weights_ready) {
  int32_t* idx = reinterpret_cast<int32_t*>(b + m.idx);
  float* w = reinterpret_cast<float*>(b + m.w);
  const PermPtrs pm = perm_ptrs(b, m);
  EvHook hook;
  hook.ev = events;
  EvHook* hk = events ? &hook : nullptr;
  cudaError_t e;
  // The dequantisation needs neither the routing nor the permutation: it runs
  // on the handle's second stream, forked from and joined back into `st` by
  // events (so the whole call stays in `st`'s order and can be captured).
  const bool fork = !weights_ready && P.aux != nullptr && P.ev_fork != nullptr && P.ev_join != nullptr;
  const bool sorted = P.G <= 8;  // group sets fit the 8-bit keys of the token order
  if (fork) {
    if ((e = cudaEventRecord(P.ev_fork, st)) != cudaSuccess || (e = cudaStreamWaitEvent(P.aux, P.ev_fork, 0)) != cudaSuccess)
      return e;
    if (hk) hk->i = 2;  // stage order: route, permute, dequant, tsort, win, ...
    if ((e = dequant(P, x, T, b, m, P.aux, hk, !sorted)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(P.ev_join, P.aux)) != cudaSuccess) return e;
    if (hk) hk->i = 0;
  }
  if (hk) hk->before(st);
  if ((e = route(P, x, T, idx, w, reinterpret_cast<float*>(b + m.logits), reinterpret_cast<float*>(b + m.rpart), st)) !=
      cudaSuccess)
    return e;
  if (hk) hk->after(st);
  if (hk) hk->before(st);
  if ((e = launch_permute(idx, T, P.E, P.G, P.k, pm, b + m.perm_scratch, P.err, st)) != cudaSuccess) return e;
  if (hk) hk->after(st);
  TokOrder to{};
  if (sorted) {
    if (hk) hk->i = 3;
    if (hk) hk->before(st);
    uint8_t* tmask = reinterpret_cast<uint8_t*>(b + m.tmask);
    int32_t* tsort = reinterpret_cast<int32_t*>(b + m.tsort);
    int32_t* tpos = reinterpret_cast<int32_t*>(b + m.tpos);
    int* tbh = reinterpret_cast<int*>(b + m.tbh);
    uint32_t* tunion = reinterpret_cast<uint32_t*>(b + m.tunion);
    int* gtc = reinterpret_cast<int*>(b + m.gtc);
    int* gtl = reinterpret_cast<int*>(b + m.gtl);
    const int nb = (T + TS_TB - 1) / TS_TB;
    tsort_count_kernel<<<nb, TS_TB, 0, st>>>(idx, T, P.k, P.epg, tmask, tbh);
    tsort_scan_kernel<<<1, 256, 0, st>>>(tbh, nb);
    tsort_scatter_kernel<<<nb, TS_TB, 0, st>>>(tmask, T, tbh, tsort, tpos);
    tsort_tiles_kernel<<<1, 1024, 0, st>>>(tmask, tsort, T, P.G, tunion, gtc, gtl);
    x_sorted_kernel<<<4 * P.num_sms, 256, 0, st>>>(reinterpret_cast<const uint4*>(x), tsort, T, P.d / 8,
                                                   reinterpret_cast<uint4*>(b + m.x16));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (hk) hk->after(st);
    to = TokOrder{tsort, tpos, tunion, gtc, gtl};
  }
  if (weights_ready && !sorted) {  // x in fp16, token order unchanged
    DqJob J;
    J.nseg = 0;
    J.x = reinterpret_cast<const uint4*>(x);
    J.x16 = reinterpret_cast<uint4*>(b + m.x16);
    J.nx = (size_t)T * P.d / 8;
    dequant_all_kernel<<<8 * P.num_sms, 256, 0, st>>>(J);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (fork) {
    if ((e = cudaStreamWaitEvent(st, P.ev_join, 0)) != cudaSuccess) return e;
    if (hk) hk->i = sorted ? 4 : 3;  // the first stage after the dequantisation and the token order
  }
  return experts(P, x, T, idx, w, pm, b, m, 0, nullptr, residual, y, st, hk, !fork && !weights_ready, to);
}
}  // namespace

cudaError_t launch_prefill_layer(const PrefillArgs& P, const uint16_t* x, int T, const uint16_t* residual,
                                 uint16_t* y, void* ws, cudaStream_t st, const std::vector<cudaEvent_t>* events) {
  return prefill_layer_impl(P, x, T, residual, y, reinterpret_cast<char*>(ws), pws(P, T), st, events, false);
}

cudaError_t launch_prefill_weights(const PrefillArgs& P, int layout_T, void* ws, cudaStream_t st) {
  return dequant(P, nullptr, 0, reinterpret_cast<char*>(ws), pws(P, layout_T), st, nullptr, false);
}

cudaError_t launch_prefill_layer_chunk(const PrefillArgs& P, const uint16_t* x, int T, int layout_T,
                                       const uint16_t* residual, uint16_t* y, void* ws, cudaStream_t st) {
  if (T > layout_T) return cudaErrorInvalidValue;
  return prefill_layer_impl(P, x, T, residual, y, reinterpret_cast<char*>(ws), pws(P, layout_T), st, nullptr, true);
}

int prefill_launch_count(const PrefillArgs& P, int T) {
  // route: GEMM + top-k; permute: count, scan, scatter; dequant (+ the LoRA
  // matrices); tsort: count, scan, scatter, tiles, x in order (G <= 8);
  // [lora_p]; win; gateup; down; zreduce; [lora_q]; wout
  if (T <= 0) return 0;
  return (P.G <= 8 ? 16 : 11) + (P.r > 0 ? 3 : 0);
}

const char* prefill_stage_name(const PrefillArgs& P, int, int i, int* count) {
  static const char* names[] = {"route", "permute", "dequant", "tsort", "win", "gateup", "down", "zreduce", "wout"};
  static const char* names_l[] = {"route", "permute", "dequant", "tsort", "lora_p", "win",
                                  "gateup", "down", "zreduce", "lora_q", "wout"};
  const bool sorted = P.G <= 8, lora = P.r > 0;
  const char* const* list = lora ? names_l : names;
  const int n = (sorted ? 9 : 8) + (lora ? 2 : 0);
  if (count) *count = n;
  if (i < 0 || i >= n) return "";
  return list[sorted || i < 3 ? i : i + 1];  // without the token order, "tsort" is skipped
}

}  // namespace lmoe
