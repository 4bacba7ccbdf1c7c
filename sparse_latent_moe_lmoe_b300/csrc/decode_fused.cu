// The decode-path layer (<= 16 tokens, no LoRA branch) as one persistent
// cooperative kernel built around a shared-memory weight ring.
//
// Per CTA (one per SM, 16 warps): warp 15 is the producer. Its lane 0 walks
// the CTA's list of weight chunks for the whole layer and loads each into the
// next ring slot with TMA tensor copies (one box of up to 8 KB of packed int4
// in 128-byte swizzle plus one box of bf16 scales, or 8 KB of fp32 router
// rows), as far ahead as the ring allows (weights with an evict-first L2
// policy; W_out also prefetched into L2 during the expert phases). Warps
// 0..14 consume the chunks with tensor-core MMAs (int4 dequantised in
// registers, fp16 operands, fp32 accumulation) against activation fragments
// staged in shared memory.
//
// Work, in ring order (KS = d/1024 reduction segments):
//   A1  router logits: (segment, expert pair) items, partial sums reduced in
//       segment order by the last arriver of each pair
//   A2  H[g] = W_in[g] x for every group: (segment, group, 16-row tile)
//       items, reduced in segment order by the last arriver of each tile
//   --  every CTA computes the routing itself (top-k, softmax, tables) on
//       the warps without a router item, while the others finish A2
//   B   V[e] = silu(Gate_e h) * Up_e h for each routed expert: (expert,
//       16-row tile) items, gate and up chunks back to back
//   C   Z[g] = sum_{e in g} Down_e (w V_e): (expert, 32-row block) items with
//       per-expert partials, summed in ascending expert order by the last
//       arriver of each (group, block)
//   D   Y[g] = W_out[g] Z[g]: (group, 16-row tile) items; the last group to
//       finish a tile sums the groups in ascending order (+ residual) into y
// Dependencies between CTAs are arrival counters (per group for H and Z, per
// expert for V, one for the logits) instead of grid barriers: a CTA waits
// only for the data it stages next, and the producer keeps streaming the next
// phase's weights meanwhile. The counters come in two copies used by
// alternate launches; each launch clears the copy the next one uses, so a
// launch that ran out of its wait budget leaves the next one correct.
//
// Every wait is bounded by the handle's cycle budget; running out sets the
// timeout bit of the device error word and the kernel carries on to the end
// (the output is then invalid and lmoe_check reports LMOE_ERR_TIMEOUT).
#include "common.cuh"
#include "decode.cuh"
#include "ring.cuh"
#include "tmap.cuh"
#include "topk.cuh"

namespace lmoe {

// cold, once-per-phase code is kept out of line: the kernel's instruction
// footprint, not its arithmetic, bounds how fast every SM gets through it
#define LMOE_COLD __device__ __noinline__

namespace {

constexpr int NWARP = 16, NTHR = NWARP * 32, NCW = NWARP - 1, PROD = NWARP - 1, NCT = NCW * 32;
constexpr int SLOT_BYTES = 10240;  // 8 KB of weights + 1 KB of scales, 1024-byte aligned
constexpr int KEYS = 3;            // activation sets staged at once
constexpr int KSEG = 1024;         // reduction segment of the router and W_in
constexpr int DR = 32;             // rows of a down chunk
constexpr int MAX_ACT = 256;       // routed experts per pass (16 tokens x k <= 16)

template <int NT>
__host__ __device__ constexpr int nslot() {
  return NT == 1 ? 16 : 12;
}
template <int NT>
__host__ __device__ constexpr int key_bytes() {
  return 16384 * NT;
}
template <int NT>
__host__ __device__ constexpr int dyn_smem() {
  return 1024 + nslot<NT>() * SLOT_BYTES + KEYS * key_bytes<NT>();
}

struct Tables {
  int32_t idx[16 * 16];
  float w[16 * 16];
  unsigned emask[16];        // bit e: expert e is routed by some token (E <= 512)
  int16_t elist[MAX_ACT];    // routed experts, ascending
  int16_t glist[64];         // routed groups, ascending
  int16_t gslot0[65];        // first expert slot of each routed group
  int n_act, n_actg, par;
  volatile int tables_ready;
  volatile int x_issued;     // the consumers' loads of x are in flight: weight copies may start
  int key[KEYS];              // activation sets of the B, C and D phases
  int keyA[KEYS];             // segments of x staged for the A phase
  uint2 tkscr[NCW][32];       // top-k candidates, per routing warp
  uint64_t full[16], empty[16];
  volatile int seq[16];
};

// Orders this thread's earlier memory accesses before its later ones at GPU
// scope. Every hand-off between CTAs here is a release/acquire pair (data,
// fence, counter atomic; counter seen, fence or acquire load, data), for
// which an acquire-release fence suffices: the sequentially consistent
// fence (__threadfence) also joins one total order of all such fences on
// the GPU, which thousands of hand-offs a pass would wait on.
LMOE_DEV void fence_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

LMOE_DEV unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Whole warp, no divergence: lane i waits until *p_i >= target (p_i null:
// nothing to wait for), polling with acquire loads.
LMOE_COLD void wait_counts(const unsigned* p, unsigned target, long long budget, unsigned* err) {
  const long long t0 = clock64();
  #pragma unroll 1
  while (!__all_sync(0xffffffffu, p == nullptr || ld_acquire(p) >= target)) {
    if (__any_sync(0xffffffffu, clock64() - t0 > budget)) {
      if ((threadIdx.x & 31) == 0) set_error(err, ERRBIT_TIMEOUT);
      return;
    }
    __nanosleep(32);
  }
}

// The routing warps (the last n consumer warps).
LMOE_DEV void route_sync(int n) {
  __syncwarp();
  asm volatile("barrier.sync 3, %0;" ::"r"(n * 32) : "memory");
}

// Every warp, once, at the end of the kernel.
LMOE_DEV void end_sync() { asm volatile("barrier.sync 2, %0;" ::"n"(NTHR) : "memory"); }

// Consumer warps only (the producer never joins). Callers often reach it from
// divergent code (a few lanes waiting on a counter), so the warp reconverges
// first and the barrier is the non-aligned form, which counts every thread.
LMOE_DEV void cons_sync() {
  __syncwarp();
  asm volatile("barrier.sync 1, %0;" ::"n"(NCT) : "memory");
}

// The last of n arrivals on a ticket returns true; called by one lane after a
// fence_gpu that publishes the caller's partial results.
LMOE_DEV bool ticket_last(unsigned* t, unsigned n) { return atomicAdd(t, 1u) == n - 1; }

LMOE_DEV float route_weight(const Tables& tb, int t, int e, int k) {
  #pragma unroll 1
  for (int j = 0; j < k; ++j)
    if (tb.idx[t * 16 + j] == e) return tb.w[t * 16 + j];
  return 0.f;
}

// Counter layout (one copy; two copies alternate between launches). Every
// counter sits on a 128-byte line of its own (CSTR words apart): the
// completion counters are polled by whole CTAs, and the tickets take up to
// a few hundred atomics each within microseconds, which one L2 line would
// serialise.
constexpr int CSTR = 32;
struct CtrMap {
  int tk_router, done_router, tk_win, done_in, done_gu, tk_down, done_down, tk_wout, n;
};
__host__ __device__ inline CtrMap ctr_map(int d, int E, int G, int L) {
  CtrMap m;
  int o = 0;
  m.tk_router = o; o += E / 2 * CSTR;
  m.done_router = o; o += CSTR;
  m.tk_win = o; o += G * (L / 16) * CSTR;
  m.done_in = o; o += G * CSTR;
  m.done_gu = o; o += MAX_ACT * CSTR;
  m.tk_down = o; o += G * (L / DR) * CSTR;
  m.done_down = o; o += G * CSTR;
  m.tk_wout = o; o += d / 16 * CSTR;
  m.n = (o + 31) & ~31;
  return m;
}

// index range of CTA c of nC over n items
LMOE_DEV void split(int n, int c, int nC, int& lo, int& hi) {
  lo = (int)((long long)c * n / nC);
  hi = (int)((long long)(c + 1) * n / nC);
}

// ------------------------------------------------------------ staging
// Fragment layout of an activation set over K elements: frag_index(chunk c of
// 128, token tile nt, m pair mp, lane) -> 8 consecutive elements of token
// 8*nt + lane/4 starting at 128 c + 32 (lane % 4) + 8 mp, as fp16 pairs
// (e0,e4) (e1,e5) (e2,e6) (e3,e7).
template <int NT>
LMOE_COLD void stage_x(Tables& tb, uint4* keyset, const uint16_t* x, int T, int d, int ctid) {
  constexpr int N = (KSEG / 128) * NT * 128, PER = (N + NCT - 1) / NCT;
  // every load first, then let the producer start the weight copies: x's
  // loads must not queue behind them
  uint4 v[KEYS][PER];
#pragma unroll
  for (int s = 0; s < KEYS; ++s) {
    const int ks = tb.keyA[s];
#pragma unroll
    for (int r = 0; r < PER; ++r) {
      const int si = ctid + r * NCT;
      const int ln = si & 31, mp = (si >> 5) & 3, rest = si >> 7;
      const int nt = rest % NT, cc = rest / NT;
      const int tok = nt * 8 + (ln >> 2), tg = ln & 3;
      const int k0 = ks * KSEG + cc * 128 + tg * 32 + mp * 8;
      v[s][r] = (ks >= 0 && si < N && tok < T) ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)tok * d + k0))
                                               : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  cons_sync();
  if (ctid == 0) tb.x_issued = 1;
#pragma unroll
  for (int s = 0; s < KEYS; ++s) {
    uint4* fr = keyset + s * (key_bytes<NT>() / 16);
#pragma unroll
    for (int r = 0; r < PER; ++r) {
      const int si = ctid + r * NCT;
      if (tb.keyA[s] < 0 || si >= N) continue;
      const uint32_t u[4] = {v[s][r].x, v[s][r].y, v[s][r].z, v[s][r].w};
      float e[8];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        e[2 * h] = __uint_as_float(u[h] << 16);
        e[2 * h + 1] = __uint_as_float(u[h] & 0xffff0000u);
      }
      fr[si] = pack_frag8(e);
    }
  }
}

// Index of the fragment entry holding elements k0 .. k0+7 (k0 a multiple of
// 8) of token n, in the layout above.
template <int NT>
LMOE_DEV int entry_index(int k0, int n) {
  return frag_index(k0 >> 7, n >> 3, (k0 & 31) >> 3, (n & 7) * 4 + ((k0 & 127) >> 5), NT);
}

// n fragment entries from global memory into shared memory (consumer threads)
LMOE_COLD void copy_frags(uint4* dst, const uint4* src, int n, int ctid) {
  #pragma unroll 1
  for (int i = ctid; i < n; i += 4 * NCT) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = (i + u * NCT < n) ? __ldcg(src + i + u * NCT) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (i + u * NCT < n) dst[i + u * NCT] = v[u];
  }
}

// Distinct keys of items [lo, hi) (nondecreasing) into the key table; returns
// false (and flags bad data) if more than KEYS are needed. Consumer thread 0.
template <class KeyF>
LMOE_COLD void collect_keys(int* keys, int lo, int hi, KeyF key, unsigned* err) {
  int n = 0, last = -1;
  #pragma unroll 1
  for (int i = lo; i < hi; ++i) {
    const int kk = key(i);
    if (kk != last) {
      if (n == KEYS) {
        set_error(err, ERRBIT_BAD_DATA);
        break;
      }
      keys[n++] = kk;
      last = kk;
    }
  }
  #pragma unroll 1
  for (int s = n; s < KEYS; ++s) keys[s] = -1;
}

LMOE_DEV int key_slot(const int* keys, int kk) {
  #pragma unroll 1
  for (int s = 0; s < KEYS; ++s)
    if (keys[s] == kk) return s;
  return 0;
}

// ------------------------------------------------------------ ring access
template <int NS>
LMOE_DEV const unsigned char* cons_wait(Tables& tb, unsigned char* ring, int j, long long budget, unsigned* err) {
  const int s = j % NS, u = j / NS;
  const long long t0 = clock64();
  #pragma unroll 1
  while (tb.seq[s] != j) {
    if (clock64() - t0 > budget) {
      set_error(err, ERRBIT_TIMEOUT);
      break;
    }
    __nanosleep(20);
  }
  mbar_wait(&tb.full[s], u & 1, budget, err);
  return ring + s * SLOT_BYTES;
}

template <int NS>
LMOE_DEV void cons_release(Tables& tb, int j) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&tb.empty[j % NS]);
}


}  // namespace

// ==================================================================== kernel
// Routed-expert and routed-group tables from the routed-expert bit mask (one
// warp): elist = routed experts ascending, glist = their groups, gslot0[gi] =
// first slot of group gi in elist (gslot0[n_actg] = n_act).
LMOE_COLD void build_tables(Tables& tb, int epg) {
  const int lane = threadIdx.x & 31;
  const unsigned m = lane < 16 ? tb.emask[lane] : 0u;  // experts 32 lane .. 32 lane + 31
  const int cnt = __popc(m);
  int pre = cnt;  // inclusive prefix over lanes
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, pre, o);
    if (lane >= o) pre += y;
  }
  const int n_act = __shfl_sync(0xffffffffu, pre, 31);
  int pos = pre - cnt;
  unsigned mm = m;
#pragma unroll 1
  while (mm) {
    tb.elist[pos++] = (int16_t)(32 * lane + __ffs(mm) - 1);
    mm &= mm - 1u;
  }
  __syncwarp();
  int ng = 0;
#pragma unroll 1
  for (int i0 = 0; i0 < n_act; i0 += 32) {
    const int i = i0 + lane;
    const int g = i < n_act ? tb.elist[i] / epg : -1;
    const int gp = (i > 0 && i < n_act) ? tb.elist[i - 1] / epg : -1;
    const bool first = i < n_act && g != gp;
    const unsigned bal = __ballot_sync(0xffffffffu, first);
    if (first) {
      const int gi = ng + __popc(bal & ((1u << lane) - 1u));
      tb.glist[gi] = (int16_t)g;
      tb.gslot0[gi] = (int16_t)i;
    }
    ng += __popc(bal);
  }
  if (lane == 0) {
    tb.n_act = n_act;
    tb.n_actg = ng;
    tb.gslot0[ng] = (int16_t)n_act;
  }
  __syncwarp();
}

template <int NT>
__global__ void __launch_bounds__(NTHR, 1) decode_fused_kernel(const __grid_constant__ FusedArgs F) {
  constexpr int NS = nslot<NT>();
  constexpr int FR = 128 * NT;  // fragment entries per 128 elements of an activation set
  extern __shared__ unsigned char dsm_raw[];
  __shared__ Tables tb;
  unsigned char* dsm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~(uintptr_t)1023);
  unsigned char* ring = dsm;
  uint4* keyset = reinterpret_cast<uint4*>(dsm + NS * SLOT_BYTES);
  auto kfr = [&](int s) { return keyset + s * (key_bytes<NT>() / 16); };

  const DecodeArgs& A = F.A;
  const int T = A.T, d = A.d, E = A.E, G = A.G, k = A.k, L = A.L, f = A.f, epg = A.epg;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
  const int nC = gridDim.x, c = blockIdx.x;
  const int KS = d / KSEG, NPAIR = E / 2, NRT_IN = L / 16, NRB = L / DR, NRT_OUT = d / 16;
  const long long budget = F.timeout;
  unsigned* err = A.err;
  const CtrMap cm = ctr_map(d, E, G, L);

  // ---------------------------------------------------------------- set-up
  if (threadIdx.x == 0) {
    const unsigned long long old = atomicAdd(F.launches, 1ull);
    tb.par = (int)((old / (unsigned long long)nC) & 1ull);
    tb.tables_ready = 0;
    tb.x_issued = 0;
    #pragma unroll 1
    for (int s = 0; s < NS; ++s) {
      mbar_init(&tb.full[s], 1);
      mbar_init(&tb.empty[s], 1);
      tb.seq[s] = -1;
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  unsigned* ctr = F.ctr + (size_t)tb.par * cm.n;
  {  // clear the copy of the counters the next launch uses
    unsigned* nxt = F.ctr + (size_t)(tb.par ^ 1) * cm.n;
    #pragma unroll 1
    for (int i = c * NTHR + threadIdx.x; i < cm.n; i += nC * NTHR) nxt[i] = 0u;
  }
  int a1lo, a1hi, a2lo, a2hi;
  split(KS * NPAIR, c, nC, a1lo, a1hi);
  split(KS * G * NRT_IN, c, nC, a2lo, a2hi);
  const int nA1 = a1hi - a1lo, nA2 = a2hi - a2lo;

  if (warp == PROD) {
    // ================================================== producer
    // Lane 0 issues every chunk. Its loop is kept short (no divisions, no
    // calls): it shares an SM sub-partition with three consumer warps, and
    // its issue rate bounds how fast weights reach the ring.
    int j = 0, slot = 0, use = 0;
    bool ok = true;
    auto claim = [&](uint32_t bytes) -> unsigned char* {  // next chunk's slot, armed for `bytes`
      if (use > 0) {
        const long long t0 = clock64();
        while (!mbar_test(&tb.full[slot], (use - 1) & 1) || !mbar_test(&tb.empty[slot], (use - 1) & 1)) {
          if (clock64() - t0 > budget) {
            set_error(err, ERRBIT_TIMEOUT);
            ok = false;
            return nullptr;
          }
        }
      }
      tb.seq[slot] = j;
      mbar_expect_tx(&tb.full[slot], bytes);
      return ring + slot * SLOT_BYTES;
    };
    auto advance = [&]() {
      ++j;
      if (++slot == NS) {
        slot = 0;
        ++use;
      }
    };
    if (lane == 0) {
      const uint64_t pol = l2_evict_first();  // weights are read once per pass
      {  // x first: its loads are small and every CTA waits on them
        const long long t0 = clock64();
#pragma unroll 1
        while (tb.x_issued == 0) {
          if (clock64() - t0 > budget) {
            set_error(err, ERRBIT_TIMEOUT);
            ok = false;
            break;
          }
          __nanosleep(32);
        }
      }
      {  // router: (segment, expert pair)
        int ks = a1lo / NPAIR, pr = a1lo % NPAIR;
#pragma unroll 1
        for (int i = a1lo; ok && i < a1hi; ++i) {
          unsigned char* dst = claim(2 * KSEG * 4);
          if (!dst) break;
          tma_load_3d_hint(dst, &F.maps.wr, 0, ks * (KSEG / 256), 2 * pr, &tb.full[slot], pol);
          advance();
          if (++pr == NPAIR) { pr = 0; ++ks; }
        }
      }
      {  // W_in: (segment, group, 16-row tile)
        const int per_ks = G * NRT_IN;
        int ks = a2lo / per_ks, row = a2lo % per_ks;  // row tile index g * NRT_IN + rt
#pragma unroll 1
        for (int i = a2lo; ok && i < a2hi; ++i) {
          unsigned char* dst = claim(16 * KSEG / 2 + 16 * KSEG / 16);
          if (!dst) break;
          tma_load_3d_hint(dst, &F.maps.win_q, 0, ks * (KSEG / 256), row * 16, &tb.full[slot], pol);
          tma_load_2d_hint(dst + 16 * KSEG / 2, &F.maps.win_s, ks * (KSEG / 32), row * 16, &tb.full[slot], pol);
          advance();
          if (++row == per_ks) { row = 0; ++ks; }
        }
      }
      if (ok) {  // the routing tables (built by the consumers)
        const long long t0 = clock64();
#pragma unroll 1
        while (tb.tables_ready == 0) {
          if (clock64() - t0 > budget) {
            set_error(err, ERRBIT_TIMEOUT);
            ok = false;
            break;
          }
          __nanosleep(64);
        }
        __threadfence_block();
      }
      const int n_act = tb.n_act, n_actg = tb.n_actg, FT = f / 16;
      int lo = 0, hi = 0;
      if (ok) split(n_act * FT, c, nC, lo, hi);
      {  // gate/up: (expert slot, 16-row tile), gate then up
        int es = lo / FT, rt = lo % FT;
        int e = es < n_act ? tb.elist[es] : 0;
#pragma unroll 1
        for (int i = lo; ok && i < hi; ++i) {
          const int row = e * f + rt * 16;
          unsigned char* dst = claim(16 * L / 2 + 16 * L / 16);
          if (!dst) break;
          tma_load_3d_hint(dst, &F.maps.gate_q, 0, 0, row, &tb.full[slot], pol);
          tma_load_2d_hint(dst + 16 * L / 2, &F.maps.gate_s, 0, row, &tb.full[slot], pol);
          advance();
          dst = claim(16 * L / 2 + 16 * L / 16);
          if (!dst) break;
          tma_load_3d_hint(dst, &F.maps.up_q, 0, 0, row, &tb.full[slot], pol);
          tma_load_2d_hint(dst + 16 * L / 2, &F.maps.up_s, 0, row, &tb.full[slot], pol);
          advance();
          if (++rt == FT) {
            rt = 0;
            if (++es < n_act) e = tb.elist[es];
          }
        }
      }
      if (ok) {  // this CTA's W_out chunks into L2 now, while the experts are computed:
                 // fetched in a burst at the end they would slow the Z reductions
        int plo, phi;
        split(n_actg * NRT_OUT, c, nC, plo, phi);
        int gi = plo / NRT_OUT, rt = plo % NRT_OUT;
#pragma unroll 1
        for (int i = plo; i < phi; ++i) {
          const int row = tb.glist[gi] * d + rt * 16;
          tma_prefetch_3d(&F.maps.wout_q, 0, 0, row);
          tma_prefetch_2d(&F.maps.wout_s, 0, row);
          if (++rt == NRT_OUT) { rt = 0; ++gi; }
        }
      }
      if (ok) split(n_act * NRB, c, nC, lo, hi);
      {  // down: (expert slot, 32-row block)
        int es = lo / NRB, rb = lo % NRB;
        int e = es < n_act ? tb.elist[es] : 0;
#pragma unroll 1
        for (int i = lo; ok && i < hi; ++i) {
          const int row = e * L + rb * DR;
          unsigned char* dst = claim(DR * f / 2 + DR * f / 16);
          if (!dst) break;
          tma_load_3d_hint(dst, &F.maps.down_q, 0, 0, row, &tb.full[slot], pol);
          tma_load_2d_hint(dst + DR * f / 2, &F.maps.down_s, 0, row, &tb.full[slot], pol);
          advance();
          if (++rb == NRB) {
            rb = 0;
            if (++es < n_act) e = tb.elist[es];
          }
        }
      }
      if (ok) split(n_actg * NRT_OUT, c, nC, lo, hi);
      {  // W_out: (group slot, 16-row tile)
        int gi = lo / NRT_OUT, rt = lo % NRT_OUT;
        int g = gi < n_actg ? tb.glist[gi] : 0;
#pragma unroll 1
        for (int i = lo; ok && i < hi; ++i) {
          const int row = g * d + rt * 16;
          unsigned char* dst = claim(16 * L / 2 + 16 * L / 16);
          if (!dst) break;
          tma_load_3d_hint(dst, &F.maps.wout_q, 0, 0, row, &tb.full[slot], pol);
          tma_load_2d_hint(dst + 16 * L / 2, &F.maps.wout_s, 0, row, &tb.full[slot], pol);
          advance();
          if (++rt == NRT_OUT) {
            rt = 0;
            if (++gi < n_actg) g = tb.glist[gi];
          }
        }
      }
      // Wait for the copies still in flight before the CTA may exit. They do
      // not depend on other CTAs, so this drain gets a budget of its own.
      const long long drain = budget > (1ll << 28) ? budget : (1ll << 28);
#pragma unroll 1
      for (int jj = (j > NS ? j - NS : 0); jj < j; ++jj) mbar_wait(&tb.full[jj % NS], (jj / NS) & 1, drain, err);
    }
    // The whole producer warp stays resident until every consumer is done: a
    // warp that exits changes what the consumers' named barrier counts.
    __syncwarp();
    end_sync();
    return;
  }

  // ================================================================ consumers
  const int ctid = threadIdx.x;  // 0 .. NCT-1
  int jbase = 0;

  // ------------------------------------------------- segments of x (A1, A2)
  if (ctid == 0) {
    const int k1lo = a1lo / NPAIR, k1hi = (a1hi - 1) / NPAIR, k2lo = a2lo / (G * NRT_IN),
              k2hi = (a2hi - 1) / (G * NRT_IN);
    int n = 0;
    #pragma unroll 1
    for (int ks = 0; ks < KS; ++ks) {
      const bool need = (nA1 > 0 && ks >= k1lo && ks <= k1hi) || (nA2 > 0 && ks >= k2lo && ks <= k2hi);
      if (!need) continue;
      if (n == KEYS) {
        set_error(err, ERRBIT_BAD_DATA);
        break;
      }
      tb.keyA[n++] = ks;
    }
    #pragma unroll 1
    for (int s = n; s < KEYS; ++s) tb.keyA[s] = -1;
  }
  cons_sync();
  stage_x<NT>(tb, keyset, A.x, T, d, ctid);
  cons_sync();

  // ------------------------------------------------------------ A1 router
  #pragma unroll 1
  for (int li = warp; li < nA1; li += NCW) {
    const int i = a1lo + li, ks = i / NPAIR, pr = i % NPAIR, e0 = 2 * pr;
    const float* wr = reinterpret_cast<const float*>(cons_wait<NS>(tb, ring, jbase + li, budget, err));
    const uint4* fr = kfr(key_slot(tb.keyA, ks));
    // lane covers elements u*256 + 8*lane .. +7 (u < 4) of both experts; for
    // each half of u the 32 weights stay in registers while the tokens stream
    // past, 16 independent sums per lane
#pragma unroll 1
    for (int nt = 0; nt < NT; ++nt) {
      float v[16];  // v[2 t + r]: token 8 nt + t, expert e0 + r
#pragma unroll
      for (int q = 0; q < 16; ++q) v[q] = 0.f;
#pragma unroll 1
      for (int uh = 0; uh < 2; ++uh) {
        float4 w0[2][2], w1[2][2];
#pragma unroll
        for (int u2 = 0; u2 < 2; ++u2) {
          const int kk = (2 * uh + u2) * 256 + lane * 8;
          w0[u2][0] = *reinterpret_cast<const float4*>(wr + kk);
          w0[u2][1] = *reinterpret_cast<const float4*>(wr + kk + 4);
          w1[u2][0] = *reinterpret_cast<const float4*>(wr + KSEG + kk);
          w1[u2][1] = *reinterpret_cast<const float4*>(wr + KSEG + kk + 4);
        }
        if (uh == 1 && nt == NT - 1) cons_release<NS>(tb, jbase + li);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          float s0 = v[2 * t], s1 = v[2 * t + 1];
#pragma unroll
          for (int u2 = 0; u2 < 2; ++u2) {
            const int kk = (2 * uh + u2) * 256 + lane * 8;
            const int cc = kk >> 7, tg = (kk & 127) >> 5, mp = (kk & 31) >> 3;
            const uint4 xv = fr[((cc * NT + nt) * 4 + mp) * 32 + t * 4 + tg];
            const float2 p0 = __half22float2(*reinterpret_cast<const __half2*>(&xv.x));  // e0, e4
            const float2 p1 = __half22float2(*reinterpret_cast<const __half2*>(&xv.y));  // e1, e5
            const float2 p2 = __half22float2(*reinterpret_cast<const __half2*>(&xv.z));  // e2, e6
            const float2 p3 = __half22float2(*reinterpret_cast<const __half2*>(&xv.w));  // e3, e7
            const float4 a0 = w0[u2][0], a1 = w0[u2][1], b0 = w1[u2][0], b1 = w1[u2][1];
            s0 = fmaf(a0.x, p0.x, s0); s0 = fmaf(a0.y, p1.x, s0); s0 = fmaf(a0.z, p2.x, s0); s0 = fmaf(a0.w, p3.x, s0);
            s0 = fmaf(a1.x, p0.y, s0); s0 = fmaf(a1.y, p1.y, s0); s0 = fmaf(a1.z, p2.y, s0); s0 = fmaf(a1.w, p3.y, s0);
            s1 = fmaf(b0.x, p0.x, s1); s1 = fmaf(b0.y, p1.x, s1); s1 = fmaf(b0.z, p2.x, s1); s1 = fmaf(b0.w, p3.x, s1);
            s1 = fmaf(b1.x, p0.y, s1); s1 = fmaf(b1.y, p1.y, s1); s1 = fmaf(b1.z, p2.y, s1); s1 = fmaf(b1.w, p3.y, s1);
          }
          v[2 * t] = s0;
          v[2 * t + 1] = s1;
        }
      }
      // butterfly reduce-scatter over the warp: lanes 2q, 2q + 1 end with the
      // sum of v[q] over all lanes
#pragma unroll
      for (int h = 8; h >= 1; h >>= 1) {
        const bool hi = lane & (2 * h);
#pragma unroll
        for (int j = 0; j < h; ++j) {
          const float keep = hi ? v[j + h] : v[j], send = hi ? v[j] : v[j + h];
          v[j] = keep + __shfl_xor_sync(0xffffffffu, send, 2 * h);
        }
      }
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
      const int t = nt * 8 + (lane >> 2), r = (lane >> 1) & 1;
      if ((lane & 1) == 0 && t < T) F.Lp[((size_t)ks * 16 + t) * E + e0 + r] = v[0];
    }
    fence_gpu();
    __syncwarp();
    bool last = false;
    if (lane == 0) last = ticket_last(ctr + cm.tk_router + pr * CSTR, (unsigned)KS);
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) {
      fence_gpu();
      const int t = lane >> 1, r = lane & 1;
      if (t < T) {
        float part[8];
#pragma unroll
        for (int s2 = 0; s2 < 8; ++s2) part[s2] = s2 < KS ? __ldcg(F.Lp + ((size_t)s2 * 16 + t) * E + e0 + r) : 0.f;
        float v = 0.f;
#pragma unroll
        for (int s2 = 0; s2 < 8; ++s2) v += part[s2];
        if (A.b_r) v += A.b_r[e0 + r];
        F.logits[(size_t)t * E + e0 + r] = v;
      }
      fence_gpu();
      __syncwarp();
      if (lane == 0) atomicAdd(ctr + cm.done_router, 1u);
    }
  }
  jbase += nA1;

  // ------------------------------------------------------------ A2 W_in
  #pragma unroll 1
  for (int li = warp; li < nA2; li += NCW) {
    const int i = a2lo + li, ks = i / (G * NRT_IN), rem = i % (G * NRT_IN), g = rem / NRT_IN, rt = rem % NRT_IN;
    const unsigned char* sl = cons_wait<NS>(tb, ring, jbase + li, budget, err);
    float acc[NT][4] = {};
    mma_ring_rows_swz<NT>(sl, KSEG / 256, 0, reinterpret_cast<const uint16_t*>(sl + 16 * KSEG / 2), KSEG / 32,
                          KSEG / 128, kfr(key_slot(tb.keyA, ks)), acc);
    cons_release<NS>(tb, jbase + li);
    float* Hp = A.Hp + ((size_t)ks * G + g) * 16 * L;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const int row = rt * 16 + gid + ((h & 2) ? 8 : 0), t = nt * 8 + 2 * tig + (h & 1);
        if (t < T) Hp[(size_t)t * L + row] = acc[nt][h];
      }
    fence_gpu();
    __syncwarp();
    bool last = false;
    if (lane == 0) last = ticket_last(ctr + cm.tk_win + (g * NRT_IN + rt) * CSTR, (unsigned)KS);
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) {  // sum the segment partials in order, straight into fp16 fragments
      fence_gpu();
      const int run = lane & 1, n = lane >> 1, k0 = rt * 16 + run * 8;
      float e[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (n < T) {
        float4 p[8][2];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float* src = A.Hp + (((size_t)q * G + g) * 16 + n) * L + k0;
          p[q][0] = q < KS ? __ldcg(reinterpret_cast<const float4*>(src)) : make_float4(0.f, 0.f, 0.f, 0.f);
          p[q][1] = q < KS ? __ldcg(reinterpret_cast<const float4*>(src + 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          e[0] += p[q][0].x; e[1] += p[q][0].y; e[2] += p[q][0].z; e[3] += p[q][0].w;
          e[4] += p[q][1].x; e[5] += p[q][1].y; e[6] += p[q][1].z; e[7] += p[q][1].w;
        }
      }
      if (n < 8 * NT) F.Hf[(size_t)g * (L / 128) * FR + entry_index<NT>(k0, n)] = pack_frag8(e);
      fence_gpu();
      __syncwarp();
      if (lane == 0) atomicAdd(ctr + cm.done_in + g * CSTR, 1u);
    }
  }
  jbase += nA2;

  // ------------------------------------------------------------ routing
  // Every CTA routes all tokens itself: top-k of each token (a warp per
  // token), then the tables. The warps without a router item finish the A
  // phase first; they route while the others finish their W_in items.
  const int rw0 = nA1 < NCW - 1 ? nA1 : NCW - 1, nrw = NCW - rw0;
  if (warp >= rw0) {
    const int rt = (warp - rw0) * 32 + lane;
    if (rt < 16) tb.emask[rt] = 0u;
    if (warp == rw0) wait_counts(lane == 0 ? ctr + cm.done_router : nullptr, (unsigned)NPAIR, budget, err);
    route_sync(nrw);
#pragma unroll 1
    for (int tw = warp - rw0; tw < T; tw += nrw) {
      const float2 sw = topk_warp_thr(F.logits + (size_t)tw * E, E, k, tb.tkscr[warp]);
      if (lane < k) {
        const int e = __float_as_int(sw.x);
        tb.idx[tw * 16 + lane] = e;
        tb.w[tw * 16 + lane] = sw.y;
        atomicOr(&tb.emask[e >> 5], 1u << (e & 31));
        if (c == 0) {
          A.idx[tw * k + lane] = e;
          A.w[tw * k + lane] = sw.y;
        }
      }
    }
    route_sync(nrw);
    if (warp == rw0) {
      build_tables(tb, epg);
      if (lane == 0) {
        __threadfence_block();
        tb.tables_ready = 1;  // the producer may issue the expert weights
      }
      // the B phase's groups and the completion of their H, while the other
      // warps finish the A phase
      int lo, hi;
      split(tb.n_act * (f / 16), c, nC, lo, hi);
      if (lane == 0) collect_keys(tb.key, lo, hi, [&](int i) { return tb.elist[i / (f / 16)] / epg; }, err);
      __syncwarp();
      wait_counts(lane < KEYS && tb.key[lane] >= 0 ? ctr + cm.done_in + tb.key[lane] * CSTR : nullptr, (unsigned)NRT_IN,
                  budget, err);
    }
  }
  cons_sync();
  const int n_act = tb.n_act, n_actg = tb.n_actg;

  // ------------------------------------------------------------ B gate/up
  {
    int lo, hi;
    split(n_act * (f / 16), c, nC, lo, hi);  // keys collected, H completion awaited by the routing
    #pragma unroll 1
    for (int s = 0; s < KEYS; ++s)
      if (tb.key[s] >= 0) copy_frags(kfr(s), F.Hf + (size_t)tb.key[s] * (L / 128) * FR, (L / 128) * FR, ctid);
    cons_sync();
    #pragma unroll 1
    for (int li = warp; li < hi - lo; li += NCW) {
      const int i = lo + li, es = i / (f / 16), rt = i % (f / 16), e = tb.elist[es];
      const uint4* fr = kfr(key_slot(tb.key, e / epg));
      float ag[NT][4] = {}, au[NT][4] = {};
      const unsigned char* sg = cons_wait<NS>(tb, ring, jbase + 2 * li, budget, err);
      const unsigned char* su = cons_wait<NS>(tb, ring, jbase + 2 * li + 1, budget, err);
      mma_ring_rows_swz2<NT>(sg, reinterpret_cast<const uint16_t*>(sg + 16 * L / 2), su,
                             reinterpret_cast<const uint16_t*>(su + 16 * L / 2), L / 256, L / 32, L / 128, fr, ag, au);
      cons_release<NS>(tb, jbase + 2 * li);
      cons_release<NS>(tb, jbase + 2 * li + 1);
      // v = w(t, e) * silu(gate) * up, as the down projection's fragments;
      // lane t < T looks up w(t, e), the other lanes take it by shuffle
      const float wl = lane < T ? route_weight(tb, lane, e, k) : 0.f;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int t = nt * 8 + 2 * tig + h2;
          const float wt = __shfl_sync(0xffffffffu, wl, t);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const float a = ag[nt][hh * 2 + h2];
            ag[nt][hh * 2 + h2] = wt != 0.f ? wt * a * __frcp_rn(1.f + __expf(-a)) * au[nt][hh * 2 + h2] : 0.f;
          }
        }
      float ev[8];
      acc_to_entry<NT>(ag, ev);
      const int run = lane & 1, n = lane >> 1;
      if (n < 8 * NT) F.Vf[(size_t)es * (f / 128) * FR + entry_index<NT>(rt * 16 + run * 8, n)] = pack_frag8(ev);
      fence_gpu();
      __syncwarp();
      if (lane == 0) atomicAdd(ctr + cm.done_gu + es * CSTR, 1u);
    }
    jbase += 2 * (hi - lo);
  }

  // ------------------------------------------------------------ C down
  {
    int lo, hi;
    split(n_act * NRB, c, nC, lo, hi);
    cons_sync();
    if (ctid == 0) collect_keys(tb.key, lo, hi, [&](int i) { return i / NRB; }, err);
    cons_sync();
    if (warp == 0)
      wait_counts(lane < KEYS && tb.key[lane] >= 0 ? ctr + cm.done_gu + tb.key[lane] * CSTR : nullptr, (unsigned)(f / 16), budget,
                  err);
    cons_sync();
    #pragma unroll 1
    for (int s = 0; s < KEYS; ++s)
      if (tb.key[s] >= 0) copy_frags(kfr(s), F.Vf + (size_t)tb.key[s] * (f / 128) * FR, (f / 128) * FR, ctid);
    cons_sync();
    // A warp's items are contracted back to back, then their partials are
    // published with one fence: the second item does not wait on the first
    // one's ticket and reduction
    auto c_compute = [&](int li) {
      const int i = lo + li, es = i / NRB, rb = i % NRB;
      const uint4* fr = kfr(key_slot(tb.key, es));
      const unsigned char* sl = cons_wait<NS>(tb, ring, jbase + li, budget, err);
      float* Zp = F.Zp + (size_t)es * 16 * L;
#pragma unroll 1
      for (int mt = 0; mt < DR / 16; ++mt) {
        float acc[NT][4] = {};
        mma_ring_rows_swz<NT>(sl, f / 256, mt * 16, reinterpret_cast<const uint16_t*>(sl + DR * f / 2), f / 32, f / 128,
                              fr, acc);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const int row = rb * DR + mt * 16 + gid + ((h & 2) ? 8 : 0), t = nt * 8 + 2 * tig + (h & 1);
            if (t < T) Zp[(size_t)t * L + row] = acc[nt][h];
          }
      }
      cons_release<NS>(tb, jbase + li);
    };
    // block (group, row block) of item li: its ticket and its group's expert slots
    auto c_block = [&](int li, int& g, int& rb, int& s0, int& s1) {
      const int i = lo + li, es = i / NRB;
      rb = i % NRB;
      g = tb.elist[es] / epg;
      int gi = 0;
      #pragma unroll 1
      while (gi < n_actg && tb.glist[gi] != g) ++gi;
      s0 = tb.gslot0[gi];
      s1 = tb.gslot0[gi + 1];
    };
    // Z rows of a block: the group's experts in ascending order, into fragments
    auto c_reduce = [&](int g, int rb, int s0, int s1) {
        // fragment entries per lane: DR/8 runs x 8 NT tokens over 32 lanes;
        // the experts' partials are loaded QB at a time, all loads first
        constexpr int PE = DR / 8 * 8 * NT / 32, QB = NT == 1 ? 12 : 4;
        float ev[PE][8];
#pragma unroll
        for (int u = 0; u < PE; ++u)
#pragma unroll
          for (int h = 0; h < 8; ++h) ev[u][h] = 0.f;
#pragma unroll 1
        for (int sl2 = s0; sl2 < s1; sl2 += QB) {
          float4 p[QB][PE][2];
#pragma unroll
          for (int q = 0; q < QB; ++q)
#pragma unroll
            for (int u = 0; u < PE; ++u) {
              const int en = lane + 32 * u, run = en % (DR / 8), n = en / (DR / 8);
              const float* src = F.Zp + ((size_t)(sl2 + q) * 16 + n) * L + rb * DR + run * 8;
              const bool v = n < T && sl2 + q < s1;
              p[q][u][0] = v ? __ldcg(reinterpret_cast<const float4*>(src)) : make_float4(0.f, 0.f, 0.f, 0.f);
              p[q][u][1] = v ? __ldcg(reinterpret_cast<const float4*>(src + 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
          for (int q = 0; q < QB; ++q)
#pragma unroll
            for (int u = 0; u < PE; ++u) {
              ev[u][0] += p[q][u][0].x; ev[u][1] += p[q][u][0].y; ev[u][2] += p[q][u][0].z; ev[u][3] += p[q][u][0].w;
              ev[u][4] += p[q][u][1].x; ev[u][5] += p[q][u][1].y; ev[u][6] += p[q][u][1].z; ev[u][7] += p[q][u][1].w;
            }
        }
#pragma unroll
        for (int u = 0; u < PE; ++u) {
          const int en = lane + 32 * u, run = en % (DR / 8), n = en / (DR / 8);
          if (n < 8 * NT)
            F.Zf[(size_t)g * (L / 128) * FR + entry_index<NT>(rb * DR + run * 8, n)] = pack_frag8(ev[u]);
        }
    };
    #pragma unroll 1
    for (int li = warp; li < hi - lo; li += 2 * NCW) {
      const bool two = li + NCW < hi - lo;
      #pragma unroll 1
      for (int q = 0; q < (two ? 2 : 1); ++q) c_compute(li + q * NCW);  // one copy of the code
      fence_gpu();
      __syncwarp();
      // both tickets in flight at once; a block's last arriver reduces it
      int g0, rb0, a0, b0, g1 = 0, rb1 = 0, a1 = 0, b1 = 0;
      c_block(li, g0, rb0, a0, b0);
      if (two) c_block(li + NCW, g1, rb1, a1, b1);
      bool l0 = false, l1 = false;
      if (lane == 0) {
        const unsigned o0 = atomicAdd(ctr + cm.tk_down + (g0 * NRB + rb0) * CSTR, 1u);
        const unsigned o1 = two ? atomicAdd(ctr + cm.tk_down + (g1 * NRB + rb1) * CSTR, 1u) : 0u;
        l0 = o0 == (unsigned)(b0 - a0 - 1);
        l1 = two && o1 == (unsigned)(b1 - a1 - 1);
      }
      l0 = __shfl_sync(0xffffffffu, l0, 0);
      l1 = __shfl_sync(0xffffffffu, l1, 0);
      if (l0 || l1) {
        fence_gpu();
        #pragma unroll 1
        for (int q = 0; q < 2; ++q)
          if (q ? l1 : l0) c_reduce(q ? g1 : g0, q ? rb1 : rb0, q ? a1 : a0, q ? b1 : b0);
        fence_gpu();
        __syncwarp();
        if (lane == 0) {
          if (l0) atomicAdd(ctr + cm.done_down + g0 * CSTR, 1u);
          if (l1) atomicAdd(ctr + cm.done_down + g1 * CSTR, 1u);
        }
      }
    }
    jbase += hi - lo;
  }

  // ------------------------------------------------------------ D W_out
  {
    int lo, hi;
    split(n_actg * NRT_OUT, c, nC, lo, hi);
    cons_sync();
    if (ctid == 0) collect_keys(tb.key, lo, hi, [&](int i) { return i / NRT_OUT; }, err);
    cons_sync();
    if (warp == 0)
      wait_counts(lane < KEYS && tb.key[lane] >= 0 ? ctr + cm.done_down + tb.glist[tb.key[lane]] * CSTR : nullptr, (unsigned)NRB,
                  budget, err);
    cons_sync();
    #pragma unroll 1
    for (int s = 0; s < KEYS; ++s)
      if (tb.key[s] >= 0)
        copy_frags(kfr(s), F.Zf + (size_t)tb.glist[tb.key[s]] * (L / 128) * FR, (L / 128) * FR, ctid);
    cons_sync();
    #pragma unroll 1
    for (int li = warp; li < hi - lo; li += NCW) {
      const int i = lo + li, gi = i / NRT_OUT, rt = i % NRT_OUT, g = tb.glist[gi];
      const unsigned char* sl = cons_wait<NS>(tb, ring, jbase + li, budget, err);
      float acc[NT][4] = {};
      mma_ring_rows_swz<NT>(sl, L / 256, 0, reinterpret_cast<const uint16_t*>(sl + 16 * L / 2), L / 32, L / 128,
                            kfr(key_slot(tb.key, gi)), acc);
      cons_release<NS>(tb, jbase + li);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const int row = rt * 16 + gid + ((h & 2) ? 8 : 0), t = nt * 8 + 2 * tig + (h & 1);
          if (t < T) A.Yp[((size_t)g * 16 + t) * d + row] = acc[nt][h];
        }
      fence_gpu();
      __syncwarp();
      bool last = false;
      if (lane == 0) last = ticket_last(ctr + cm.tk_wout + rt * CSTR, (unsigned)n_actg);
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {  // combine in ascending group order: lane -> 4 rows x 1 token, one float4 per group
        fence_gpu();
#pragma unroll 1
        for (int q = lane; q < 4 * T; q += 32) {
          const int rq = q & 3, t = q >> 2, row = rt * 16 + rq * 4;
          float4 acc4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
          for (int g0 = 0; g0 < n_actg; g0 += 8) {
            float4 p4[8];
#pragma unroll
            for (int gg = 0; gg < 8; ++gg)
              p4[gg] = g0 + gg < n_actg
                           ? __ldcg(reinterpret_cast<const float4*>(A.Yp + ((size_t)tb.glist[g0 + gg] * 16 + t) * d + row))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int gg = 0; gg < 8; ++gg) {
              acc4.x += p4[gg].x; acc4.y += p4[gg].y; acc4.z += p4[gg].z; acc4.w += p4[gg].w;
            }
          }
          if (A.residual) {
            const uint2 rb = *reinterpret_cast<const uint2*>(A.residual + (size_t)t * d + row);
            acc4.x += __uint_as_float(rb.x << 16);
            acc4.y += __uint_as_float(rb.x & 0xffff0000u);
            acc4.z += __uint_as_float(rb.y << 16);
            acc4.w += __uint_as_float(rb.y & 0xffff0000u);
          }
          uint2 o;
          o.x = (uint32_t)f32_to_bf16_rne(acc4.x) | ((uint32_t)f32_to_bf16_rne(acc4.y) << 16);
          o.y = (uint32_t)f32_to_bf16_rne(acc4.z) | ((uint32_t)f32_to_bf16_rne(acc4.w) << 16);
          *reinterpret_cast<uint2*>(A.y + (size_t)t * d + row) = o;
        }
      }
    }
  }
  end_sync();
}

// ===================================================================== host
size_t fused_counter_words(int d, int E, int G, int L) { return 2 * (size_t)ctr_map(d, E, G, L).n; }

namespace {
// packed int4 [rows][K/2] as [rows][K/256][128 B], box {128, lines, box_rows}
bool map_q(CUtensorMap* m, const uint8_t* q, long long rows, int K, int lines, int box_rows) {
  const cuuint64_t dims[3] = {128, (cuuint64_t)(K / 256), (cuuint64_t)rows};
  const cuuint64_t strides[2] = {128, (cuuint64_t)(K / 2)};
  const cuuint32_t box[3] = {128, (cuuint32_t)lines, (cuuint32_t)box_rows};
  return tmap_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, q, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// bf16 scales [rows][K/32], box {box_cols, box_rows}
bool map_s(CUtensorMap* m, const uint16_t* s, long long rows, int K, int box_cols, int box_rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)(K / 32), (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)(K / 32 * 2)};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  return tmap_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, s, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}
}  // namespace

bool fused_make_maps(const DecodeArgs& A, DecodeMaps* mp) {
  if (!tmap_encode_fn() || !A.W_r) return false;
  const int d = A.d, E = A.E, G = A.G, L = A.L, f = A.f;
  if (d % KSEG != 0 || L % 256 != 0 || f % 256 != 0) return false;
  bool ok = true;
  {
    const cuuint64_t dims[3] = {256, (cuuint64_t)(d / 256), (cuuint64_t)E};
    const cuuint64_t strides[2] = {1024, (cuuint64_t)d * 4};
    const cuuint32_t box[3] = {256, KSEG / 256, 2};
    ok = ok && tmap_encode(&mp->wr, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, A.W_r, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  ok = ok && map_q(&mp->win_q, A.W_in_q, (long long)G * L, d, KSEG / 256, 16);
  ok = ok && map_s(&mp->win_s, A.W_in_s, (long long)G * L, d, KSEG / 32, 16);
  ok = ok && map_q(&mp->gate_q, A.gate_q, (long long)E * f, L, L / 256, 16);
  ok = ok && map_s(&mp->gate_s, A.gate_s, (long long)E * f, L, L / 32, 16);
  ok = ok && map_q(&mp->up_q, A.up_q, (long long)E * f, L, L / 256, 16);
  ok = ok && map_s(&mp->up_s, A.up_s, (long long)E * f, L, L / 32, 16);
  ok = ok && map_q(&mp->down_q, A.down_q, (long long)E * L, f, f / 256, DR);
  ok = ok && map_s(&mp->down_s, A.down_s, (long long)E * L, f, f / 32, DR);
  ok = ok && map_q(&mp->wout_q, A.W_out_q, (long long)G * d, L, L / 256, 16);
  ok = ok && map_s(&mp->wout_s, A.W_out_s, (long long)G * d, L, L / 32, 16);
  return ok;
}

bool fused_decode_supported(const DecodeArgs& A) {
  if (A.r != 0 || A.T < 1 || A.T > 16) return false;
  if (A.E > 512 || A.E % 2 != 0 || A.G > 64 || A.k > 16) return false;
  if (A.d % KSEG != 0 || A.d / KSEG > 8) return false;
  if (A.L != 256 && A.L != 512 && A.L != 1024) return false;  // gate/up/W_out chunks: 16 rows x L in one slot
  if (A.f != 256 && A.f != 512) return false;                  // down chunks: 32 rows x f in one slot
  if (A.f % 16 != 0 || (long long)A.T * A.k > MAX_ACT) return false;
  return true;
}

cudaError_t fused_set_attributes() {
  cudaFuncSetAttribute(decode_fused_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_smem<1>());
  cudaFuncSetAttribute(decode_fused_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_smem<2>());
  return cudaGetLastError();
}

int fused_grid(int num_sms) {
  int per1 = 0, per2 = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per1, decode_fused_kernel<1>, NTHR, dyn_smem<1>()) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per2, decode_fused_kernel<2>, NTHR, dyn_smem<2>()) !=
          cudaSuccess ||
      per1 < 1 || per2 < 1) {
    cudaGetLastError();
    return 0;
  }
  return num_sms;  // one CTA per SM
}

cudaError_t launch_decode_fused(const FusedArgs& F, int grid, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(NTHR);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (F.A.T <= 8) {
    cfg.dynamicSmemBytes = dyn_smem<1>();
    return cudaLaunchKernelEx(&cfg, decode_fused_kernel<1>, F);
  }
  cfg.dynamicSmemBytes = dyn_smem<2>();
  return cudaLaunchKernelEx(&cfg, decode_fused_kernel<2>, F);
}

}  // namespace lmoe
