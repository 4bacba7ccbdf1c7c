// The decode-path layer as one persistent cooperative kernel (<= 16 tokens,
// no LoRA branch): one CTA per SM, phases separated by grid barriers.
//
//   P0  router logits, split along d; a ticket per expert pair sums the
//       partial sums in fixed order (deterministic)
//   P1  every CTA: top-k with softmax renormalisation for all tokens and the
//       routed-expert / routed-group tables (no serial single-CTA tail)
//   P2  H[g][t] = Win[g] x_t, split along d, reduced by a ticket per tile
//   P3  V[e][t] = silu(Gate_e h) * Up_e h for each routed (expert, token)
//   P4  Z[g][t] = sum_{e in g} w Down_e V: one CTA per (group, 64 rows),
//       all of the group's experts accumulated in registers
//   P5  Y[g][t] = Wout[g] Z[g][t]; the last group to finish a 16-row tile
//       sums the routed groups in ascending order (+ residual) into y
//
// Weights stream through a register prefetch ring (PFD chunks of 16 rows x
// 128 reduction elements in flight per warp).
//
// Every spin is bounded by the handle's cycle budget; running out sets the
// timeout bit of the device error word and the kernel carries on (the output
// is then invalid and lmoe_check reports LMOE_ERR_TIMEOUT).
#include "common.cuh"
#include "decode.cuh"

namespace lmoe {

constexpr int FW = 16;             // warps per CTA
constexpr int FT = FW * 32;        // threads per CTA
constexpr int SLOT_BYTES = 32768;  // one staged activation set
constexpr int NSLOT = 3;           // activation sets staged at once
constexpr int RED_BYTES = 3 * 4 * 16 * 16 * 4;
constexpr int DYN_SMEM = NSLOT * SLOT_BYTES;
constexpr int MAX_ACT = 256;       // routed experts per pass: <= 16 tokens * 16
constexpr int PFD = 6;             // register prefetch depth (chunks)

// Grid barrier on a monotonically increasing 64-bit arrival counter: the
// k-th barrier of a launch completes when the counter reaches the next
// multiple of the grid size. Nothing is ever reset, so a launch leaves the
// counter at a multiple of the grid size even when a wait ran out of budget
// (every CTA still arrives exactly once per barrier).
LMOE_DEV void grid_sync(unsigned long long* bar, long long budget, unsigned* err) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned long long n = gridDim.x;
    const unsigned long long arrived = atomicAdd(bar, 1ull);
    const unsigned long long target = (arrived / n + 1) * n;
    volatile unsigned long long* vb = bar;
    const long long t0 = clock64();
    while (*vb < target) {
      if (clock64() - t0 > budget) {
        set_error(err, ERRBIT_TIMEOUT);
        break;
      }
      __nanosleep(32);
    }
    __threadfence();
  }
  __syncthreads();
}

// The last of `n` arrivals on a ticket returns true (and resets it). Called
// by one lane after its writes; the caller fences before.
LMOE_DEV bool ticket_last(unsigned* t, unsigned n) {
  const unsigned old = atomicAdd(t, 1u);
  if (old == n - 1) {
    *t = 0;
    __threadfence();
    return true;
  }
  return false;
}

struct Tables {
  int32_t idx[16 * 16];
  float w[16 * 16];
  unsigned emask[1024];   // routed tokens per expert
  int16_t elist[MAX_ACT]; // routed experts, ascending
  int16_t glist[64];      // routed groups, ascending
  int16_t gslot0[65];     // first expert slot of each routed group
  int n_act, n_actg;
  // per-phase item ranges of this CTA
  int nq, per_q, lo2, hi2, lo3, hi3, N4, nblk, lo5, hi5;
  int slot_key[NSLOT];
};

LMOE_DEV float route_weight(const Tables& tb, int t, int e, int k) {
  for (int j = 0; j < k; ++j)
    if (tb.idx[t * 16 + j] == e) return tb.w[t * 16 + j];
  return 0.f;
}

// fp32 activations [T][K] (row stride K) -> frags for all chunks of K
template <int NT>
LMOE_DEV void stage_f32(uint4* fr, const float* src, int T, int K) {
  const int nslots = (K / 128) * NT * 128;
  for (int si = threadIdx.x; si < nslots; si += FT) {
    const int ln = si & 31, mp = (si >> 5) & 3, rest = si >> 7;
    const int nt = rest % NT, cc = rest / NT;
    const int n = nt * 8 + (ln >> 2), tg = ln & 3;
    const int k0 = cc * 128 + tg * 32 + mp * 8;
    float e[8];
    if (n < T) {
      const float4 a = __ldcg(reinterpret_cast<const float4*>(src + (size_t)n * K + k0));
      const float4 b = __ldcg(reinterpret_cast<const float4*>(src + (size_t)n * K + k0 + 4));
      e[0] = a.x; e[1] = a.y; e[2] = a.z; e[3] = a.w; e[4] = b.x; e[5] = b.y; e[6] = b.z; e[7] = b.w;
    } else {
#pragma unroll
      for (int h = 0; h < 8; ++h) e[h] = 0.f;
    }
    fr[si] = pack_frag8(e);
  }
}

// Stage the distinct keys (nondecreasing over items [lo, hi)) into the
// activation slots, at most NSLOT of them; tb.slot_key[s] = key or -1.
template <class KeyF, class StageF>
LMOE_DEV void stage_keys(Tables& tb, int lo, int hi, KeyF key, StageF stage, unsigned* err) {
  int n = 0, last = -1;
  for (int i = lo; i < hi; ++i) {
    const int kk = key(i);
    if (kk != last) {
      if (n == NSLOT) {
        if (threadIdx.x == 0) set_error(err, ERRBIT_BAD_DATA);
        break;
      }
      stage(n, kk);
      if (threadIdx.x == 0) tb.slot_key[n] = kk;
      ++n;
      last = kk;
    }
  }
  if (threadIdx.x == 0)
    for (int s = n; s < NSLOT; ++s) tb.slot_key[s] = -1;
  __syncthreads();
}

LMOE_DEV int slot_of(const Tables& tb, int kk) {
  for (int s = 0; s < NSLOT; ++s)
    if (tb.slot_key[s] == kk) return s;
  return 0;
}

template <int NT>
__global__ void __launch_bounds__(FT, 1) decode_fused_kernel(FusedArgs F) {
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ Tables tb;
  const DecodeArgs& A = F.A;
  const int T = A.T, d = A.d, E = A.E, G = A.G, k = A.k, L = A.L, f = A.f, epg = A.epg;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
  const int nC = gridDim.x, c = blockIdx.x;
  uint4* slot_base = reinterpret_cast<uint4*>(dsm);
  auto slot = [&](int s) { return slot_base + s * (SLOT_BYTES / 16); };

  // item -> weights of each phase
  auto win_item = [&](int i, const uint8_t*& q, const uint16_t*& sc, int& r0, int& c0, int& c1, int& g, int& q_) {
    const int ntile = L / 16, nch = d / 128;
    q_ = i / tb.per_q;
    const int rem = i % tb.per_q, gi = rem / ntile, rt = rem % ntile;
    g = tb.glist[gi];
    q = A.W_in_q + (size_t)g * L * (d / 2);
    sc = A.W_in_s + (size_t)g * L * (d / 32);
    r0 = rt * 16;
    c0 = q_ * nch / tb.nq;
    c1 = (q_ + 1) * nch / tb.nq;
  };
  // ---------------------------------------------------------------- P0 router
  {
    // The W_in and W_out tickets count arrivals that depend on the routing;
    // clearing them here (they are first used after the next barrier) keeps a
    // launch correct even after one whose waits ran out of budget. The
    // router's tickets always see exactly d/RS arrivals and reset themselves.
    for (int i = c * FT + threadIdx.x; i < G * (L / 16); i += nC * FT) F.tk_win[i] = 0u;
    for (int i = c * FT + threadIdx.x; i < d / 16; i += nC * FT) F.tk_wout[i] = 0u;
    const int RS = F.router_slice, nslice = d / RS, nrp = E / 2;
    const int N0 = nslice * nrp;
    const int lo = (int)((long long)c * N0 / nC), hi = (int)((long long)(c + 1) * N0 / nC);
    stage_keys(
        tb, lo, hi, [&](int i) { return i / nrp; },
        [&](int s, int sl) {  // x[:, sl*RS .. +RS] as bf16 [T][RS]
          uint4* dst = slot(s);
          const int per = RS / 8;
          for (int i = threadIdx.x; i < T * per; i += FT) {
            const int t = i / per, p = i % per;
            dst[i] = *reinterpret_cast<const uint4*>(A.x + (size_t)t * d + (size_t)sl * RS + p * 8);
          }
        },
        A.err);
    for (int i = lo + warp; i < hi; i += FW) {
      const int sl = i / nrp, rp = i % nrp, e0 = 2 * rp;
      const uint16_t* xs = reinterpret_cast<const uint16_t*>(slot(slot_of(tb, sl)));
      const float* w0 = A.W_r + (size_t)e0 * d + (size_t)sl * RS;
      const float* w1 = w0 + d;
      float4 wa[4], wb[4];  // RS <= 512: all of this lane's weights in flight at once
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int pos = lane * 4 + u * 128;
        wa[u] = pos < RS ? __ldg(reinterpret_cast<const float4*>(w0 + pos)) : make_float4(0.f, 0.f, 0.f, 0.f);
        wb[u] = pos < RS ? __ldg(reinterpret_cast<const float4*>(w1 + pos)) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float acc[2][16];
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int t = 0; t < 16; ++t) acc[r][t] = 0.f;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int pos = lane * 4 + u * 128;
        if (pos >= RS) continue;
        const float4 a = wa[u], b = wb[u];
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          if (t < T) {
            const uint2 xb = *reinterpret_cast<const uint2*>(xs + t * RS + pos);
            const float x0 = __uint_as_float(xb.x << 16), x1 = __uint_as_float(xb.x & 0xffff0000u);
            const float x2 = __uint_as_float(xb.y << 16), x3 = __uint_as_float(xb.y & 0xffff0000u);
            acc[0][t] = fmaf(a.w, x3, fmaf(a.z, x2, fmaf(a.y, x1, fmaf(a.x, x0, acc[0][t]))));
            acc[1][t] = fmaf(b.w, x3, fmaf(b.z, x2, fmaf(b.y, x1, fmaf(b.x, x0, acc[1][t]))));
          }
        }
      }
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          float v = acc[r][t];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          acc[r][t] = v;
        }
      {  // lane (t, r) writes its partial, the last of the slices sums them
        const int t = lane >> 1, r = lane & 1;
        float mine = 0.f;
#pragma unroll
        for (int tt = 0; tt < 16; ++tt)
          if (tt == t) mine = acc[r][tt];
        if (t < T) F.Lp[((size_t)sl * 16 + t) * E + e0 + r] = mine;
        __threadfence();
        __syncwarp();
        bool last = false;
        if (lane == 0) last = ticket_last(F.tk_router + rp, (unsigned)nslice);
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last && t < T) {
          float part[16];
#pragma unroll
          for (int s2 = 0; s2 < 16; ++s2)
            part[s2] = s2 < nslice ? __ldcg(F.Lp + ((size_t)s2 * 16 + t) * E + e0 + r) : 0.f;
          float v = 0.f;
#pragma unroll
          for (int s2 = 0; s2 < 16; ++s2) v += part[s2];
          if (A.b_r) v += A.b_r[e0 + r];
          F.logits[(size_t)t * E + e0 + r] = v;
        }
      }
    }
  }
  grid_sync(F.bar, F.timeout, A.err);

  // --------------------------------------------------------------- P1 routing
  {
    float* lg = reinterpret_cast<float*>(slot(0));  // [T][E] logits in shared memory
    for (int i = threadIdx.x; i < T * E / 4; i += FT)
      reinterpret_cast<float4*>(lg)[i] = __ldcg(reinterpret_cast<const float4*>(F.logits) + i);
    for (int e = threadIdx.x; e < E; e += FT) tb.emask[e] = 0u;
    __syncthreads();
    if (warp < T) {
      // top-k of token `warp`: lane holds logits lane, lane+32, ... (E <= 512)
      // in registers and its own best remaining one; each round the warp picks
      // the best lane head (ties -> lower index) and only the winner rescans
      const float* row = lg + (size_t)warp * E;
      float v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = (lane + 32 * i < E) ? row[lane + 32 * i] : -INFINITY;
      auto lane_best = [&](float& bv, int& be) {
        bv = -INFINITY;
        be = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int e = lane + 32 * i;
          if (e < E && (v[i] > bv || (v[i] == bv && e < be))) {
            bv = v[i];
            be = e;
          }
        }
      };
      float mv;
      int me;
      lane_best(mv, me);
      float sel = 0.f, l0 = 0.f;
      int sel_e = 0;
      for (int j = 0; j < k; ++j) {
        float bv = mv;
        int be = me;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oe = __shfl_xor_sync(0xffffffffu, be, o);
          if (ov > bv || (ov == bv && oe < be)) {
            bv = ov;
            be = oe;
          }
        }
        if (be >= E) be = 0;
        if (be == me) {  // the winning lane drops that logit and finds its next best
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (lane + 32 * i == be) v[i] = -INFINITY;
          lane_best(mv, me);
          if (mv == -INFINITY) me = 0x7fffffff;
        }
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
        tb.idx[warp * 16 + lane] = sel_e;
        tb.w[warp * 16 + lane] = ex / z;
        if (c == 0) {
          A.idx[warp * k + lane] = sel_e;
          A.w[warp * k + lane] = ex / z;
        }
      }
    }
    __syncthreads();
    if (threadIdx.x < T * k) {
      const int t = threadIdx.x / k, j = threadIdx.x % k;
      atomicOr(&tb.emask[tb.idx[t * 16 + j]], 1u << t);
    }
    __syncthreads();
    if (warp == 0) {  // ascending compaction of routed experts
      int base = 0;
      for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        const bool on = e < E && tb.emask[e] != 0u;
        const unsigned bal = __ballot_sync(0xffffffffu, on);
        const int pos = base + __popc(bal & ((1u << lane) - 1u));
        if (on) tb.elist[pos] = (int16_t)e;
        base += __popc(bal);
      }
      if (lane == 0) tb.n_act = base;
    }
    __syncthreads();
    if (warp == 1) {  // routed groups: per-group expert counts scanned by one warp
      int cnt0 = 0, cnt1 = 0;  // groups lane and lane + 32
      if (lane < G)
        for (int e = lane * epg; e < (lane + 1) * epg; ++e) cnt0 += tb.emask[e] != 0u;
      if (lane + 32 < G)
        for (int e = (lane + 32) * epg; e < (lane + 33) * epg; ++e) cnt1 += tb.emask[e] != 0u;
      int inc0 = cnt0, inc1 = cnt1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int a0 = __shfl_up_sync(0xffffffffu, inc0, o), a1 = __shfl_up_sync(0xffffffffu, inc1, o);
        if (lane >= o) {
          inc0 += a0;
          inc1 += a1;
        }
      }
      const int tot0 = __shfl_sync(0xffffffffu, inc0, 31);
      const unsigned b0 = __ballot_sync(0xffffffffu, cnt0 > 0), b1 = __ballot_sync(0xffffffffu, cnt1 > 0);
      const int n0 = __popc(b0);
      if (cnt0 > 0) {
        const int gi = __popc(b0 & ((1u << lane) - 1u));
        tb.glist[gi] = (int16_t)lane;
        tb.gslot0[gi] = (int16_t)(inc0 - cnt0);
      }
      if (cnt1 > 0) {
        const int gi = n0 + __popc(b1 & ((1u << lane) - 1u));
        tb.glist[gi] = (int16_t)(lane + 32);
        tb.gslot0[gi] = (int16_t)(tot0 + inc1 - cnt1);
      }
      const int ng = n0 + __popc(b1);
      if (lane == 0) {
        tb.gslot0[ng] = (int16_t)tb.n_act;
        tb.n_actg = ng;
        tb.nq = A.ks_in;
        tb.per_q = ng * (L / 16);
        const int N2 = tb.nq * tb.per_q, N3 = tb.n_act * (f / 16), N5 = ng * (d / 16);
        tb.lo2 = (int)((long long)c * N2 / nC); tb.hi2 = (int)((long long)(c + 1) * N2 / nC);
        tb.lo3 = (int)((long long)c * N3 / nC); tb.hi3 = (int)((long long)(c + 1) * N3 / nC);
        tb.nblk = L / 64; tb.N4 = ng * tb.nblk;
        tb.lo5 = (int)((long long)c * N5 / nC); tb.hi5 = (int)((long long)(c + 1) * N5 / nC);
      }
    }
    __syncthreads();
  }

  // ------------------------------------------------------------------ P2 W_in
  {
    const int nch = d / 128, ntile = L / 16;
    stage_keys(
        tb, tb.lo2, tb.hi2, [&](int i) { return i / tb.per_q; },
        [&](int s, int q) {
          const int c0 = q * nch / tb.nq, c1 = (q + 1) * nch / tb.nq;
          const int nslots = (c1 - c0) * NT * 128;
          uint4* fr = slot(s);
          for (int si = threadIdx.x; si < nslots; si += FT) {
            const int ln = si & 31, mp = (si >> 5) & 3, rest = si >> 7;
            const int nt = rest % NT, cc = rest / NT;
            const int n = nt * 8 + (ln >> 2), tg = ln & 3;
            const int k0 = (c0 + cc) * 128 + tg * 32 + mp * 8;
            float e[8];
            if (n < T) {
              const uint4 v = *reinterpret_cast<const uint4*>(A.x + (size_t)n * d + k0);
              const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                e[2 * h] = __uint_as_float(u[h] << 16);
                e[2 * h + 1] = __uint_as_float(u[h] & 0xffff0000u);
              }
            } else {
#pragma unroll
              for (int h = 0; h < 8; ++h) e[h] = 0.f;
            }
            fr[si] = pack_frag8(e);
          }
        },
        A.err);
    for (int i = tb.lo2 + warp; i < tb.hi2; i += FW) {
      const uint8_t* q; const uint16_t* sc; int r0, c0, c1, g, qq;
      win_item(i, q, sc, r0, c0, c1, g, qq);
      const int rt = r0 / 16, nq = tb.nq;
      float acc[NT][4] = {};
      mma_rows<NT, PFD>(q, sc, d, r0, c0, c1, c0, slot(slot_of(tb, qq)), acc);
      float* Hp = A.Hp + ((size_t)qq * G + g) * 16 * L;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const int row = r0 + gid + ((h & 2) ? 8 : 0), t = nt * 8 + 2 * tig + (h & 1);
          if (t < T) Hp[(size_t)t * L + row] = acc[nt][h];
        }
      __threadfence();
      __syncwarp();
      bool last = false;
      if (lane == 0) last = ticket_last(F.tk_win + g * ntile + rt, (unsigned)nq);
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {  // sum the K-split partials: each lane 8 outputs, loads issued together
        float part[8][8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int o = lane + 32 * u, row = r0 + (o & 15), t = o >> 4;
#pragma unroll
          for (int q2 = 0; q2 < 8; ++q2)
            part[u][q2] = (t < T && q2 < nq) ? __ldcg(A.Hp + (((size_t)q2 * G + g) * 16 + t) * L + row) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int o = lane + 32 * u, row = r0 + (o & 15), t = o >> 4;
          float v = 0.f;
#pragma unroll
          for (int q2 = 0; q2 < 8; ++q2) v += part[u][q2];
          if (t < T) F.H[((size_t)g * 16 + t) * L + row] = v;
        }
      }
    }
  }
  grid_sync(F.bar, F.timeout, A.err);

  // --------------------------------------------------------------- P3 gate/up
  {
    const int nch = L / 128, ntile = f / 16;
    stage_keys(
        tb, tb.lo3, tb.hi3, [&](int i) { return tb.elist[i / ntile] / epg; },
        [&](int s, int g) { stage_f32<NT>(slot(s), F.H + (size_t)g * 16 * L, T, L); }, A.err);
    for (int i = tb.lo3 + warp; i < tb.hi3; i += FW) {
      const int es = i / ntile, rt = i % ntile, e = tb.elist[es];
      const uint4* fr = slot(slot_of(tb, e / epg));
      float ag[NT][4] = {}, au[NT][4] = {};
      mma_rows<NT, PFD>(A.gate_q + (size_t)e * f * (L / 2), A.gate_s + (size_t)e * f * (L / 32), L, rt * 16, 0, nch, 0,
                        fr, ag);
      mma_rows<NT, PFD>(A.up_q + (size_t)e * f * (L / 2), A.up_s + (size_t)e * f * (L / 32), L, rt * 16, 0, nch, 0,
                        fr, au);
      const unsigned m = tb.emask[e];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const int row = rt * 16 + gid + ((h & 2) ? 8 : 0), t = nt * 8 + 2 * tig + (h & 1);
          if (t < T && ((m >> t) & 1u)) A.V[((size_t)es * 16 + t) * f + row] = silu(ag[nt][h]) * au[nt][h];
        }
    }
  }
  grid_sync(F.bar, F.timeout, A.err);

  // ------------------------------------------------------------------ P4 down
  {
    const int nch = f / 128;
    const int per_e = nch * NT * 128;  // uint4 per expert
    const int nb_max = (NSLOT * SLOT_BYTES - RED_BYTES) / (per_e * 16);
    float* red = reinterpret_cast<float*>(dsm + NSLOT * SLOT_BYTES - RED_BYTES);  // [3][4][16][16]
    const int rt = warp & 3, es = warp >> 2;
    for (int it = c; it < tb.N4; it += nC) {
      const int gi = it / tb.nblk, blk = it % tb.nblk, g = tb.glist[gi];
      const int s0 = tb.gslot0[gi], s1 = tb.gslot0[gi + 1];
      const int row0 = blk * 64 + rt * 16;
      float acc[NT][4] = {};
      for (int b0 = s0; b0 < s1; b0 += nb_max) {
        const int nb = min(nb_max, s1 - b0);
        __syncthreads();
        uint4* fr = slot_base;
        for (int si = threadIdx.x; si < nb * per_e; si += FT) {
          const int bi = si / per_e, sj = si % per_e;
          const int ln = sj & 31, mp = (sj >> 5) & 3, rest = sj >> 7;
          const int nt = rest % NT, cc = rest / NT;
          const int n = nt * 8 + (ln >> 2), tg = ln & 3;
          const int k0 = cc * 128 + tg * 32 + mp * 8;
          const int sl = b0 + bi, e = tb.elist[sl];
          float ev[8];
          if (n < T && ((tb.emask[e] >> n) & 1u)) {
            const float wt = route_weight(tb, n, e, k);
            const float* vp = A.V + ((size_t)sl * 16 + n) * f + k0;
            const float4 a = __ldcg(reinterpret_cast<const float4*>(vp));
            const float4 b = __ldcg(reinterpret_cast<const float4*>(vp + 4));
            ev[0] = wt * a.x; ev[1] = wt * a.y; ev[2] = wt * a.z; ev[3] = wt * a.w;
            ev[4] = wt * b.x; ev[5] = wt * b.y; ev[6] = wt * b.z; ev[7] = wt * b.w;
          } else {
#pragma unroll
            for (int h = 0; h < 8; ++h) ev[h] = 0.f;
          }
          fr[si] = pack_frag8(ev);
        }
        __syncthreads();
        for (int sl = s0 + es; sl < b0 + nb; sl += 4) {
          if (sl < b0) continue;
          const int e = tb.elist[sl];
          mma_rows<NT, PFD>(A.down_q + (size_t)e * L * (f / 2), A.down_s + (size_t)e * L * (f / 32), f, row0, 0, nch, 0,
                            fr + (sl - b0) * per_e, acc);
        }
      }
      if (es > 0) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int h = 0; h < 4; ++h)
            red[(((es - 1) * 4 + rt) * 16 + gid + ((h & 2) ? 8 : 0)) * 16 + nt * 8 + 2 * tig + (h & 1)] = acc[nt][h];
      }
      __syncthreads();
      if (es == 0) {
        float* Z = A.Z + (size_t)g * 16 * L;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const int rr = gid + ((h & 2) ? 8 : 0), t = nt * 8 + 2 * tig + (h & 1);
            float v = acc[nt][h];
            for (int s2 = 0; s2 < 3; ++s2) v += red[((s2 * 4 + rt) * 16 + rr) * 16 + t];
            if (t < T) Z[(size_t)t * L + row0 + rr] = v;
          }
      }
      __syncthreads();
    }
  }
  grid_sync(F.bar, F.timeout, A.err);

  // ------------------------------------------------------------------ P5 W_out
  {
    const int nch = L / 128, ntile = d / 16;
    stage_keys(
        tb, tb.lo5, tb.hi5, [&](int i) { return i / ntile; },
        [&](int s, int gi) { stage_f32<NT>(slot(s), A.Z + (size_t)tb.glist[gi] * 16 * L, T, L); }, A.err);
    for (int i = tb.lo5 + warp; i < tb.hi5; i += FW) {
      const int gi = i / ntile, rt = i % ntile, g = tb.glist[gi];
      float acc[NT][4] = {};
      mma_rows<NT, PFD>(A.W_out_q + (size_t)g * d * (L / 2), A.W_out_s + (size_t)g * d * (L / 32), L, rt * 16, 0, nch,
                        0, slot(slot_of(tb, gi)), acc);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const int row = rt * 16 + gid + ((h & 2) ? 8 : 0), t = nt * 8 + 2 * tig + (h & 1);
          if (t < T) A.Yp[((size_t)g * 16 + t) * d + row] = acc[nt][h];
        }
      __threadfence();
      __syncwarp();
      bool last = false;
      if (lane == 0) last = ticket_last(F.tk_wout + rt, (unsigned)tb.n_actg);
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {  // weighted combine in ascending group order, 8 groups' loads at a time
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = 0.f;
        for (int g0 = 0; g0 < tb.n_actg; g0 += 8) {
          float part[8][8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int o = lane + 32 * u, row = rt * 16 + (o & 15), t = o >> 4;
#pragma unroll
            for (int gg = 0; gg < 8; ++gg)
              part[u][gg] = (t < T && g0 + gg < tb.n_actg)
                                ? __ldcg(A.Yp + ((size_t)tb.glist[g0 + gg] * 16 + t) * d + row)
                                : 0.f;
          }
#pragma unroll
          for (int u = 0; u < 8; ++u)
#pragma unroll
            for (int gg = 0; gg < 8; ++gg) v[u] += part[u][gg];
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int o = lane + 32 * u, row = rt * 16 + (o & 15), t = o >> 4;
          if (t >= T) continue;
          float r = v[u];
          if (A.residual) r += bf16_to_f32(A.residual[(size_t)t * d + row]);
          A.y[(size_t)t * d + row] = f32_to_bf16_rne(r);
        }
      }
    }
  }
}

bool fused_decode_supported(const DecodeArgs& A) {
  if (A.r != 0 || A.T < 1 || A.T > 16) return false;
  if (A.E > 1024 || A.E % 2 != 0 || A.G > 64) return false;
  // every streamed matrix walks whole chunks of 128 (scale rows 8-byte aligned);
  // these bounds keep each CTA's activation sets within NSLOT slots
  if (A.d % 128 != 0 || A.L % 128 != 0 || A.f % 128 != 0) return false;
  if (A.L < 256 || A.L > 1024 || A.f < 128 || A.d < 128) return false;
  if ((A.d / 128 + A.ks_in - 1) / A.ks_in > 8 || A.ks_in > 8) return false;
  const int RS = A.d % 512 == 0 ? 512 : 128;
  if (A.d / RS > 16) return false;  // router partial sums reduced 16 at a time
  if ((long long)A.T * RS * 2 > SLOT_BYTES) return false;
  const int nchf = A.f / 128;
  if (nchf * 2 * 128 * 16 > NSLOT * SLOT_BYTES - RED_BYTES) return false;
  if ((long long)A.T * A.E * 4 > SLOT_BYTES || A.E > 512) return false;  // logits: one slot, 16 per lane
  return true;
}

cudaError_t fused_set_attributes() {
  cudaFuncSetAttribute(decode_fused_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, DYN_SMEM);
  cudaFuncSetAttribute(decode_fused_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, DYN_SMEM);
  return cudaGetLastError();
}

int fused_grid(int num_sms) {
  int per = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, decode_fused_kernel<2>, FT, DYN_SMEM) != cudaSuccess ||
      per < 1)
    return 0;
  return num_sms;  // one CTA per SM
}

cudaError_t launch_decode_fused(FusedArgs F, int grid, cudaStream_t st) {
  F.router_slice = F.A.d % 512 == 0 ? 512 : 128;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(FT);
  cfg.dynamicSmemBytes = DYN_SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (F.A.T <= 8) return cudaLaunchKernelEx(&cfg, decode_fused_kernel<1>, F);
  return cudaLaunchKernelEx(&cfg, decode_fused_kernel<2>, F);
}

}  // namespace lmoe
