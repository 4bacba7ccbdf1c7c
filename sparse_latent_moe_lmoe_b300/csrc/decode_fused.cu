// The decode-path layer (<= 16 tokens) as one persistent cooperative kernel
// built around a shared-memory weight ring (with the Recover-LoRA branch, the
// small kernels of lora.cu run before and after it).
//
// Per CTA (one per SM): 16 consumer warps and one producer warp. The
// producer's lane 0 walks the CTA's list of weight chunks for the whole layer
// and loads each into the next ring slot (18 KB) with TMA tensor copies, as
// far ahead as the ring allows; once the routing is known it also asks L2 to
// prefetch every expert and W_out chunk the CTA will need, so that HBM keeps
// streaming while the dependent phases run. The consumers contract the chunks
// on the tensor cores (int4 dequantised in registers, fp16 operands, fp32
// accumulation) against activation fragments in shared memory.
//
// Every unit of work is split into the same 16 warp tasks, so no warp idles
// within a phase; partial sums meet in shared memory, and after one barrier
// of the consumer warps every thread reduces one output element (a serial
// reducer warp would set the pace of the whole phase):
//   A1  router logits: whole expert rows (K = d) per CTA, each warp a K
//       slice; reduced in warp order -> logits
//   A2  H[g] = W_in[g] x: whole 16-row tiles (K = d) per CTA, each warp a K
//       slice; reduced in warp order -> H as fp16 fragments
//   R   every CTA routes all tokens (top-k, softmax, tables)
//   B   expert units (expert e, 32-wide slice of f): gate and up rows of the
//       slice (the 16 warp tasks are (matrix, 16-row tile, K quarter)), then
//       v = w silu(gate h) up h for the slice, then the slice's columns of
//       Down_e (each warp 1/16 of the rows of the latent output); the Down
//       results of a CTA's consecutive units of one group stay in registers
//       and are written once per group as a partial of Z[g]
//   C   Z[g] = the sum of its partials, in CTA order, by (group, 16-row) items
//   D   Y[g] = W_out[g] Z[g] by (group, 32-row) items; after its last item
//       a CTA takes one ticket per item, and the CTA that completes a row
//       block sums the groups in ascending order (+ residual) into y
// Between CTAs only five hand-offs remain: logits, H per group, Z partials
// per group, Z per group, and the final tickets per row block of y. Each is
// data, fence, counter atomic; counter seen by an acquire load, data. The
// counters come in two copies used by alternate launches; each launch clears
// the copy the next one uses.
//
// Every wait is bounded by the handle's cycle budget; the first wait of a CTA
// that runs out sets the timeout bit of the device error word and turns every
// later wait of that CTA into a no-op, so the kernel runs to its end (the
// output is then invalid and lmoe_check reports LMOE_ERR_TIMEOUT); the
// producer stops issuing copies and waits for the ones in flight.
#include "common.cuh"
#include "decode.cuh"
#include "ring.cuh"
#include "topk.cuh"

namespace lmoe {

// cold, once-per-phase code is kept out of line: the kernel's instruction
// footprint, not its arithmetic, bounds how fast every SM gets through it
#define LMOE_COLD __device__ __noinline__

namespace {

constexpr int NCW = 16, NCT = NCW * 32, PROD = NCW, NTHR = NCT + 32;
constexpr int RW = 8;             // routing warps while the others compute W_in
static_assert(NCW % (NCW - RW) == 0, "each W_in warp hands back W_in chunks for a whole number of warps");
constexpr int SLOT = 18432;      // 16 KB of packed int4 (or fp32 router rows) + 2 KB of scales
constexpr int FS = 32;           // f-slice of an expert unit
constexpr int MAX_RX = 4;        // router experts per CTA
constexpr int MAX_TILES = 4;     // W_in 16-row tiles per CTA
constexpr int MAX_MPW = 4;       // Down 16-row tiles per warp (L <= 1024)
constexpr int LMAX = 1024;

template <int NT>
__host__ __device__ constexpr int nslot() {
  return NT == 1 ? 8 : 4;
}
template <int NT>
__host__ __device__ constexpr int xbytes() {
  return 65536 * NT;
}
template <int NT>
__host__ __device__ constexpr int dyn_smem() {
  return 1024 + nslot<NT>() * SLOT + xbytes<NT>();
}
// byte offsets inside the activation region after phase A
template <int NT>
__host__ __device__ constexpr int off_pbuf() {
  return LMAX * NT * 16;  // after the H / Z fragments
}
template <int NT>
__host__ __device__ constexpr int off_vbuf() {
  return off_pbuf<NT>() + 2 * NCW * NT * 512;
}
template <int NT>
__host__ __device__ constexpr int off_zred() {
  return off_vbuf<NT>() + 2 * NT * 512;
}
static_assert(off_zred<1>() + 16384 <= xbytes<1>(), "activation region (one token tile)");
static_assert(off_zred<2>() + 16384 <= xbytes<2>(), "activation region (two token tiles)");

struct Tables {
  uint64_t full[8], empty[8], tbar;
  alignas(16) int32_t idx[16 * 16];
  float w[16 * 16];
  unsigned emask[16];        // bit e: expert e is routed by some token (E <= 512)
  int16_t elist[512];        // routed experts, ascending
  int16_t eslot[512];        // staged experts: the slot of each routed expert
  int16_t glist[64];         // routed groups, ascending
  int16_t gslot0[65];        // first expert slot of each routed group
  int16_t gplo[64], gpn[64], gpbase[64];  // Z partials of each routed group: first CTA, count, first slot
  int n_act, n_actg, par;
  int u_lo, u_hi, z_lo, z_hi, o_lo, o_hi;
  volatile int abort;        // a wait of this CTA ran out: later waits return at once
  volatile int x_issued;     // the consumers' loads of x are in flight: weight copies may start
  int tk_z[4];
  int16_t fin[64];           // per W_out item of this CTA: its row block when this CTA combines it, else -1
  union {
    float rred[NCW][MAX_RX][16];  // router partial logits per warp
    uint2 tkscr[NCW][32];         // top-k candidates, per routing warp
  } u;
};

LMOE_DEV void fence_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

LMOE_DEV unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Consumer warps only (the producer never joins).
LMOE_DEV void cons_sync() {
  __syncwarp();
  asm volatile("barrier.sync 1, %0;" ::"n"(NCT) : "memory");
}
// Every warp, once, at the end of the kernel.
LMOE_DEV void end_sync() { asm volatile("barrier.sync 2, %0;" ::"n"(NTHR) : "memory"); }
// The W_in warps and the routing warps, each among themselves.
constexpr int BAR_WIN = 3, BAR_ROUTE = 4;
LMOE_DEV void group_sync(int id, int n) {
  __syncwarp();
  asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Where a wait gave up, for diagnosis: the first timeout of a launch is
// recorded as bit 63 | site << 32 | CTA << 8 | warp in diag[0] (sites: the
// wait_site enum below).
enum WaitSite : unsigned {
  WS_ROUTER_SLOT = 1, WS_WIN_SLOT, WS_LOGITS, WS_H, WS_GU_SLOT, WS_V, WS_DOWN_SLOT, WS_ZPART, WS_Z, WS_PFREE,
  WS_WOUT_SLOT, WS_EMPTY, WS_TABLES, WS_DRAIN
};

LMOE_DEV void timeout_hit(Tables& tb, unsigned* err, unsigned site, unsigned long long* diag) {
  set_error(err, ERRBIT_TIMEOUT);
  tb.abort = 1;
  if (diag)
    atomicCAS(diag, 0ull,
              (1ull << 63) | ((unsigned long long)site << 32) | ((unsigned long long)blockIdx.x << 8) | (threadIdx.x >> 5));
}

// %globaltimer (ns), for the per-CTA phase record
LMOE_DEV unsigned long long gtime() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// One thread: until *p >= target (acquire loads), bounded.
LMOE_COLD void wait_ge(Tables& tb, const unsigned* p, unsigned target, long long budget, unsigned* err, unsigned site,
                       unsigned long long* diag) {
  if (tb.abort) return;
  const long long t0 = clock64();
#pragma unroll 1
  while (ld_acquire(p) < target) {
    if (clock64() - t0 > budget) {
      timeout_hit(tb, err, site, diag);
      return;
    }
    __nanosleep(40);
  }
}

// Whole warp: until *p >= target, every lane polling with acquire loads.
LMOE_COLD void warp_wait_ge(Tables& tb, const unsigned* p, unsigned target, long long budget, unsigned* err,
                            unsigned site, unsigned long long* diag) {
  if (tb.abort) return;
  const long long t0 = clock64();
#pragma unroll 1
  while (!__all_sync(0xffffffffu, ld_acquire(p) >= target)) {
    if (__any_sync(0xffffffffu, clock64() - t0 > budget)) {
      if ((threadIdx.x & 31) == 0) timeout_hit(tb, err, site, diag);
      __syncwarp();
      return;
    }
    __nanosleep(40);
  }
}

// try_wait with a suspend-time hint: a waiting warp sleeps in hardware until
// the phase completes or about `ns` nanoseconds pass, instead of spinning on
// issue slots the working warps need
LMOE_DEV bool mbar_sleep_wait(uint64_t* m, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(m)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// mbarrier phase wait, bounded; true once the phase completed, false when it
// gave up (a timeout of the CTA: every later wait returns false at once).
// The slow path is out of line: it is reached only when the phase is not
// complete at the first test.
LMOE_COLD bool mwait_slow(Tables& tb, uint64_t* m, uint32_t parity, long long budget, unsigned* err, unsigned site,
                          unsigned long long* diag) {
  if (tb.abort) return false;
  const long long t0 = clock64();
#pragma unroll 1
  while (!mbar_sleep_wait(m, parity, 4000u)) {
    if (tb.abort) return false;
    if (clock64() - t0 > budget) {
      timeout_hit(tb, err, site, diag);
      return false;
    }
  }
  return true;
}
LMOE_DEV bool mwait(Tables& tb, uint64_t* m, uint32_t parity, long long budget, unsigned* err, unsigned site,
                    unsigned long long* diag) {
  return mbar_test(m, parity) || mwait_slow(tb, m, parity, budget, err, site, diag);
}

// This warp is done with ring chunk j (acquire's `landed`). Every warp hands
// back every chunk, and only after the chunk's copy completed: an arrival
// made earlier could count toward the slot's previous use (a warp that does
// not read a chunk can run ahead) and complete that phase too early, and
// after a timeout, when waits give up, a slot whose copy is still in flight
// must never be re-armed and overwritten.
template <int NS>
LMOE_DEV void release_read(Tables& tb, int j, bool landed, uint32_t weight = 1) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0 && landed) {
    if (weight == 1)
      mbar_arrive(&tb.empty[j % NS]);
    else
      mbar_arrive_n(&tb.empty[j % NS], weight);
  }
}

template <int NS>
LMOE_DEV const unsigned char* acquire(Tables& tb, unsigned char* ring, int j, long long budget, unsigned* err,
                                      unsigned site, unsigned long long* diag, bool& landed) {
  landed = mwait(tb, &tb.full[j % NS], (uint32_t)(j / NS) & 1u, budget, err, site, diag);
  landed = __all_sync(0xffffffffu, landed);
  return ring + (j % NS) * SLOT;
}

// Counter layout (one copy; two copies alternate between launches). Every
// counter sits on a 128-byte line of its own (CSTR words apart).
constexpr int CSTR = 32;
struct CtrMap {
  int done_router, done_in, done_part, done_z, tk_wout, n;
};
__host__ __device__ inline CtrMap ctr_map(int d, int G) {
  CtrMap m;
  int o = 0;
  m.done_router = o; o += CSTR;
  m.done_in = o; o += G * CSTR;
  m.done_part = o; o += G * CSTR;
  m.done_z = o; o += G * CSTR;
  m.tk_wout = o; o += d / 32 * CSTR;
  m.n = o;
  return m;
}

// index range of CTA c of nC over n items (n nC < 2^32)
LMOE_DEV void split(int n, int c, int nC, int& lo, int& hi) {
  lo = (int)((unsigned)c * (unsigned)n / (unsigned)nC);
  hi = (int)((unsigned)(c + 1) * (unsigned)n / (unsigned)nC);
}
// the CTA whose range holds item u (of n split over nC)
LMOE_DEV int owner(int u, int n, int nC) { return (int)(((unsigned)(u + 1) * (unsigned)nC - 1u) / (unsigned)n); }
// how many of the CTAs a .. b-1 have a non-empty range of the n items: all of
// them when n >= nC, else one per item boundary crossed
LMOE_DEV int busy_ctas(int a, int b, int n, int nC) {
  const int d = (int)((unsigned)b * (unsigned)n / (unsigned)nC - (unsigned)a * (unsigned)n / (unsigned)nC);
  return d < b - a ? d : b - a;
}

// Index of the fragment entry holding elements k0 .. k0+7 (k0 a multiple of
// 8) of token n: frag_index(chunk of 128, token tile, m pair, lane), see
// common.cuh.
template <int NT>
LMOE_DEV int entry_index(int k0, int n) {
  return frag_index(k0 >> 7, n >> 3, (k0 & 31) >> 3, (n & 7) * 4 + ((k0 & 127) >> 5), NT);
}

// the routing weight of expert e for token t (0 when t does not pick e; the
// rows of tokens >= T and the entries past k hold no expert)
LMOE_DEV float route_weight(const Tables& tb, int t, int e) {
  const int4* ix = reinterpret_cast<const int4*>(tb.idx + t * 16);
  int j = -1;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int4 v = ix[q];
    j = v.x == e ? 4 * q : j;
    j = v.y == e ? 4 * q + 1 : j;
    j = v.z == e ? 4 * q + 2 : j;
    j = v.w == e ? 4 * q + 3 : j;
  }
  return j >= 0 ? tb.w[t * 16 + j] : 0.f;
}

// x (bf16 [T][d]) into shared memory chunk-major: [d/128][8 NT tokens][16
// units of 8 elements], tokens >= T zero
template <int NT>
LMOE_COLD void stage_x(Tables& tb, uint4* xs, const uint16_t* x, int T, int d, int ctid) {
  const int n = NT * d, du = d / 8;  // 16-byte units: all rows, one row
  const uint4* x4 = reinterpret_cast<const uint4*>(x);
#pragma unroll 1
  for (int i0 = ctid; i0 < n; i0 += 8 * NCT) {  // i: unit of the row-major [8 NT][d]
    uint4 v[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int i = i0 + r * NCT;
      v[r] = i < T * du ? __ldg(x4 + i) : make_uint4(0u, 0u, 0u, 0u);
    }
    if (i0 == ctid && ctid == 0) tb.x_issued = 1;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int i = i0 + r * NCT, tok = i / du, u = i % du;
      if (i < n) xs[((u >> 4) * 8 * NT + tok) * 16 + (u & 15)] = v[r];
    }
  }
}

// Chunk cc (128 elements of every token) of the staged x -> its fp16
// fragment entries, in place (one warp: the chunk's units and its entries
// occupy the same 128 NT slots).
template <int NT>
LMOE_DEV void chunk_to_frags(uint4* xs, int cc) {
  const int lane = threadIdx.x & 31;
  uint4* blk = xs + (size_t)cc * 128 * NT;
  uint4 v[4 * NT];
#pragma unroll
  for (int r = 0; r < 4 * NT; ++r) {  // entry r*32 + lane: token tile r/4, m pair r%4
    const int tok = (r >> 2) * 8 + (lane >> 2), u = (lane & 3) * 4 + (r & 3);
    v[r] = blk[tok * 16 + u];
  }
  __syncwarp();
#pragma unroll
  for (int r = 0; r < 4 * NT; ++r) {
    const uint32_t w4[4] = {v[r].x, v[r].y, v[r].z, v[r].w};
    float e[8];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      e[2 * h] = __uint_as_float(w4[h] << 16);
      e[2 * h + 1] = __uint_as_float(w4[h] & 0xffff0000u);
    }
    blk[r * 32 + lane] = pack_frag8(e);
  }
  __syncwarp();
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

// The work split that follows from the routing (one warp): this CTA's expert
// units, Z items and W_out items, and for every routed group the CTAs whose
// units write its Z partials (contiguous: units are ordered by expert, hence
// by group) and where its partials start.
LMOE_COLD void plan(Tables& tb, int c, int nC, int NSF, int L, int d) {
  const int lane = threadIdx.x & 31;
  const int n_act = tb.n_act, n_actg = tb.n_actg, NU = n_act * NSF;
  int run = 0;
#pragma unroll 1
  for (int g0 = 0; g0 < n_actg; g0 += 32) {
    const int gi = g0 + lane;
    int P = 0, lo = 0;
    if (gi < n_actg) {  // the CTAs that own units of the group (some CTAs own none when NU < nC)
      const int fu = tb.gslot0[gi] * NSF, lu = tb.gslot0[gi + 1] * NSF - 1;
      lo = owner(fu, NU, nC);
      P = busy_ctas(lo, owner(lu, NU, nC) + 1, NU, nC);
    }
    int pre = P;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, pre, o);
      if (lane >= o) pre += y;
    }
    if (gi < n_actg) {
      tb.gplo[gi] = (int16_t)lo;
      tb.gpn[gi] = (int16_t)P;
      tb.gpbase[gi] = (int16_t)(run + pre - P);
    }
    run += __shfl_sync(0xffffffffu, pre, 31);
  }
  if (lane == 0) {
    split(NU, c, nC, tb.u_lo, tb.u_hi);
    split(n_actg * (L / 16), c, nC, tb.z_lo, tb.z_hi);
    split(n_actg * (d / 32), c, nC, tb.o_lo, tb.o_hi);
  }
  __syncwarp();
}

// One out-of-line copy of the ring-slot contraction (ring.cuh), shared by the
// W_in, gate / up and W_out phases: the accumulators come back by value.
template <int NT>
struct Acc {
  float v[NT][4];
};
template <int NT, int WF>
__device__ __noinline__ Acc<NT> slot_mma(const unsigned char* w, int LPR, int row0, const uint16_t* s, int SS, int c0,
                                         int nc, const uint4* frag) {
  Acc<NT> r;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int h = 0; h < 4; ++h) r.v[nt][h] = 0.f;
  mma_slot<NT, WF>(w, LPR, row0, s, SS, c0, nc, frag, r.v);
  return r;
}

// the group slot (index in glist) of expert slot es
LMOE_DEV int group_slot(const Tables& tb, int es) {
  int gi = 0;
#pragma unroll 1
  while (gi + 1 < tb.n_actg && tb.gslot0[gi + 1] <= es) ++gi;
  return gi;
}

}  // namespace

// ==================================================================== kernel
template <int NT, int WF>
__global__ void __launch_bounds__(NTHR, 1) decode_fused_kernel(const __grid_constant__ FusedArgs F) {
  constexpr int NS = nslot<NT>();
  constexpr int FR = 128 * NT;  // fragment entries per 128 elements of an activation set
  extern __shared__ unsigned char dsm_raw[];
  __shared__ Tables tb;
  unsigned char* dsm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~(uintptr_t)1023);
  unsigned char* ring = dsm;
  unsigned char* xr = dsm + NS * SLOT;                      // activation region
  uint4* xf = reinterpret_cast<uint4*>(xr);                  // x / H / Z fragments
  float4* pbuf = reinterpret_cast<float4*>(xr + off_pbuf<NT>());  // [2][NCW][NT][32] partial tiles
  uint4* vbuf = reinterpret_cast<uint4*>(xr + off_vbuf<NT>());    // [2][NT][32] slice fragments
  float4* zred = reinterpret_cast<float4*>(xr + off_zred<NT>());  // [4 items][4 quarters][32][2]

  const DecodeArgs& A = F.A;
  const int T = A.T, d = A.d, E = A.E, G = A.G, k = A.k, L = A.L, f = A.f, epg = A.epg;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
  const int nC = gridDim.x, c = blockIdx.x;
  const int NSF = f / FS, CL = L / 128, PW = d < 2048 ? d : 2048, NPW = d / PW, MPW = L / 256;
  const long long budget = F.timeout;
  unsigned* err = A.err;
  const CtrMap cm = ctr_map(d, G);
  unsigned long long* diag = F.diag;  // [0] first timeout; [1 + 32 c + e] phase times of CTA c
  unsigned long long* trace = diag ? diag + 1 + (size_t)c * 32 : nullptr;

  // ---------------------------------------------------------------- set-up
  if (threadIdx.x == 0) {
    const unsigned long long old = atomicAdd(F.launches, 1ull);
    tb.par = (int)((old / (unsigned long long)nC) & 1ull);
    tb.abort = 0;
    tb.x_issued = 0;
#pragma unroll 1
    for (int s = 0; s < NS; ++s) {
      mbar_init(&tb.full[s], 1);
      mbar_init(&tb.empty[s], NCW);
    }
    mbar_init(&tb.tbar, 1);
    tb.tk_z[0] = tb.tk_z[1] = tb.tk_z[2] = tb.tk_z[3] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (threadIdx.x < 256) {
    tb.idx[threadIdx.x] = -1;
    tb.w[threadIdx.x] = 0.f;
  }
  if (threadIdx.x < 16) tb.emask[threadIdx.x] = 0u;
  __syncthreads();
  if (trace && threadIdx.x == 0) trace[0] = gtime();
  unsigned* ctr = F.ctr + (size_t)tb.par * cm.n;
  {  // clear the copy of the counters the next launch uses
    unsigned* nxt = F.ctr + (size_t)(tb.par ^ 1) * cm.n;
#pragma unroll 1
    for (int i = c * NTHR + threadIdx.x; i < cm.n; i += nC * NTHR) nxt[i] = 0u;
  }
  int e_lo, e_hi, t_lo, t_hi;
  split(E, c, nC, e_lo, e_hi);
  split(G * (L / 16), c, nC, t_lo, t_hi);
  const int ne = e_hi - e_lo, ntl = t_hi - t_lo;
  const int jA2 = ne, jB = jA2 + ntl * NPW;

  if (warp == PROD) {
    // ================================================== producer
    if (lane == 0) {
      const uint64_t pol = l2_evict_first();  // weights are read once per pass
      const uint32_t CH = 18u * L, WCH = 9u * PW;  // bytes of a unit / W_out chunk, of a W_in chunk
      {  // x first: its loads are small and every CTA waits on them, so they
         // must not queue behind this CTA's weight copies
        const long long t0 = clock64();
#pragma unroll 1
        while (!tb.x_issued && !tb.abort && clock64() - t0 < budget) __nanosleep(32);
      }
      // The CTA's chunks in ring order: router rows, W_in pieces, then (once
      // the routing tables exist) gate / up / Down of each unit, then W_out.
      // Prefetches into L2: the W_in pieces behind the router rows; the later
      // units once the ring holds the first ones (so that their own copies do
      // not queue behind the prefetches); W_out and the next layer's first
      // chunks only once every unit is issued (they are needed last, and HBM
      // time spent on them earlier is taken from the expert phase).
      const int npre = NS / 3;
      int u_lo = 0, nu = 0, o_lo = 0, no = 0, jD = jB, jEnd = jB, j = 0;
#pragma unroll 1
      for (;; ++j) {
        if (j == ne) {
#pragma unroll 1
          for (int i = 0; i < ntl * NPW; ++i) bulk_prefetch_l2(F.pk.win + ((size_t)t_lo * NPW + i) * WCH, WCH);
        }
        if (j == jB) {  // the routing tables, from the consumers
          mwait(tb, &tb.tbar, 0u, budget, err, WS_TABLES, diag);
          if (tb.abort) break;
          if (trace) trace[13] = gtime();
          u_lo = tb.u_lo;
          nu = tb.u_hi - tb.u_lo;
          o_lo = tb.o_lo;
          no = tb.o_hi - tb.o_lo;
          jD = jB + 3 * nu;
          jEnd = jD + no;
        }
        if (j == jB + 3 * npre && npre < nu) {
#pragma unroll 1
          for (int q = npre; q < nu; ++q) {
            const int u = u_lo + q, ue = F.slot_of ? tb.eslot[u / NSF] : tb.elist[u / NSF];
            bulk_prefetch_l2(F.pk.unit + ((size_t)ue * NSF + u % NSF) * 3 * CH, 3 * CH);
          }
        }
        if (j == jD && j >= jB) {
#pragma unroll 1
          for (int q = 0; q < no; ++q) {
            const int it = o_lo + q;
            bulk_prefetch_l2(F.pk.wout + ((size_t)tb.glist[it / (d / 32)] * (d / 32) + it % (d / 32)) * CH, CH);
          }
          if (F.has_next) {  // the next layer's first phase, behind this layer's requests
#pragma unroll 1
            for (int i = 0; i < ne; ++i)
              bulk_prefetch_l2(reinterpret_cast<const uint8_t*>(F.next_wr + (size_t)(e_lo + i) * d), 4u * d);
#pragma unroll 1
            for (int i = 0; i < ntl * NPW; ++i) bulk_prefetch_l2(F.next_win + ((size_t)t_lo * NPW + i) * WCH, WCH);
          }
        }
        if (j >= jB && j >= jEnd) break;
        const uint8_t* src;
        uint32_t bytes = CH;
        if (j < ne) {
          src = reinterpret_cast<const uint8_t*>(F.pk.wr + (size_t)(e_lo + j) * d);
          bytes = 4u * d;
        } else if (j < jB) {
          src = F.pk.win + ((size_t)t_lo * NPW + (j - ne)) * WCH;
          bytes = WCH;
        } else if (j < jD) {
          const int u = u_lo + (j - jB) / 3, ue = F.slot_of ? tb.eslot[u / NSF] : tb.elist[u / NSF];
          src = F.pk.unit + (((size_t)ue * NSF + u % NSF) * 3 + (j - jB) % 3) * CH;
        } else {
          const int it = o_lo + (j - jD);
          src = F.pk.wout + ((size_t)tb.glist[it / (d / 32)] * (d / 32) + it % (d / 32)) * CH;
        }
        // chunk j's slot, once every consumer warp handed back its previous use
        const int s = j % NS;
        if (j >= NS) mwait(tb, &tb.empty[s], (uint32_t)(j / NS - 1) & 1u, budget, err, WS_EMPTY, diag);
        if (tb.abort) break;
        mbar_expect_tx(&tb.full[s], bytes);
        bulk_load(ring + s * SLOT, src, bytes, &tb.full[s], pol);
        if (trace && (j == 0 || j == jB || j == jD)) trace[j == 0 ? 26 : j == jD ? 24 : 20] = gtime();
      }
      // Wait for the copies still in flight before the CTA may exit. They do
      // not depend on other CTAs, so this drain gets a budget of its own.
      if (trace) trace[10] = gtime();
      const long long drain = budget > (1ll << 28) ? budget : (1ll << 28);
#pragma unroll 1
      for (int jj = (j > NS ? j - NS : 0); jj < j; ++jj) mbar_wait(&tb.full[jj % NS], (jj / NS) & 1, drain, err);
    }
    // The whole producer warp stays resident until every consumer is done.
    __syncwarp();
    end_sync();
    return;
  }

  // ================================================================ consumers
  const int ctid = threadIdx.x;  // 0 .. NCT-1

  // ------------------------------------------------------------ A1 router
  // the router bias of this thread's logit, loaded now: its latency hides
  // behind the staging of x instead of the router phase's end
  const float bias = (A.b_r && ctid < ne * 16) ? __ldg(A.b_r + e_lo + (ctid >> 4)) : 0.f;
  if (F.pdl) asm volatile("griddepcontrol.wait;" ::: "memory");  // x is the previous layer's output
  stage_x<NT>(tb, xf, A.x, T, d, ctid);
  cons_sync();
  if (trace && ctid == 0) trace[1] = gtime();
  {
    const int OPW = d / 128;  // 8-element octets of K per warp
#pragma unroll 1
    for (int i = 0; i < ne; ++i) {
      bool landed;
      const float* wr = reinterpret_cast<const float*>(acquire<NS>(tb, ring, i, budget, err, WS_ROUTER_SLOT, diag, landed));
      if (trace && ctid == 0 && i == 0) trace[18] = gtime();
      float v[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) v[q] = 0.f;
#pragma unroll 1
      for (int o = warp * OPW + lane; o < (warp + 1) * OPW; o += 32) {
        const int k0 = o * 8;
        const float4 a = *reinterpret_cast<const float4*>(wr + k0), b = *reinterpret_cast<const float4*>(wr + k0 + 4);
#pragma unroll
        for (int n = 0; n < 8 * NT; ++n) {  // x as staged (bf16: exact in fp32)
          if (n >= T) break;
          const uint4 xv = xf[((o >> 4) * 8 * NT + n) * 16 + (o & 15)];
          float s = v[n];
          s = fmaf(a.x, __uint_as_float(xv.x << 16), s); s = fmaf(a.y, __uint_as_float(xv.x & 0xffff0000u), s);
          s = fmaf(a.z, __uint_as_float(xv.y << 16), s); s = fmaf(a.w, __uint_as_float(xv.y & 0xffff0000u), s);
          s = fmaf(b.x, __uint_as_float(xv.z << 16), s); s = fmaf(b.y, __uint_as_float(xv.z & 0xffff0000u), s);
          s = fmaf(b.z, __uint_as_float(xv.w << 16), s); s = fmaf(b.w, __uint_as_float(xv.w & 0xffff0000u), s);
          v[n] = s;
        }
      }
      release_read<NS>(tb, i, landed);
      // butterfly reduce-scatter over the warp: lanes 2q, 2q + 1 end with the
      // sum of v[q] over all lanes
#pragma unroll
      for (int h = 8; h >= 1; h >>= 1) {
        const bool hi = lane & (2 * h);
#pragma unroll
        for (int q = 0; q < h; ++q) {
          const float keep = hi ? v[q + h] : v[q], send = hi ? v[q] : v[q + h];
          v[q] = keep + __shfl_xor_sync(0xffffffffu, send, 2 * h);
        }
      }
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
      if ((lane & 1) == 0) tb.u.rred[warp][i][lane >> 1] = v[0];
    }
    cons_sync();
    if (ctid < ne * 16) {  // warps summed in order
      const int i = ctid >> 4, t = ctid & 15;
      if (t < T) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; ++w) s += tb.u.rred[w][i][t];
        if (A.b_r) s += bias;
        F.logits[(size_t)t * E + e_lo + i] = s;
      }
    }
    cons_sync();
    if (ctid == 0) {
      fence_gpu();
      atomicAdd(ctr + cm.done_router, 1u);
      if (trace) trace[2] = gtime();
    }
  }

  // ------------------------------------------------------------ A2 W_in || routing
  // Warps RW .. 15 compute H = W_in x while warps 0 .. RW-1 route: the routing
  // needs every CTA's logits, W_in needs nothing but its chunks, so the two
  // dependent fronts overlap instead of following each other.
  if (warp >= RW) {
    const int wt = ctid - RW * 32, wi = warp - RW;  // 0 .. 255, 0 .. 7
    // task of warp wi: 16-row tile wi / 2 of this CTA, and either piece wi % 2
    // of its K (two pieces) or half wi % 2 of its one piece
    const int ti = wi >> 1, sub = wi & 1, CPP = PW / 128;
    const int tp = NPW == 2 ? sub : 0, k0c = NPW == 2 ? 0 : sub * (CPP / 2), nkc = NPW == 2 ? CPP : CPP / 2;
    {  // x chunks -> fragments, d/1024 chunks per warp
      const int per = d / 128 / (NCW - RW);
#pragma unroll 1
      for (int cc = wi * per; cc < (wi + 1) * per; ++cc) chunk_to_frags<NT>(xf, cc);
    }
    group_sync(BAR_WIN, NCT - RW * 32);
    if (trace && wt == 0) trace[17] = gtime();
    Acc<NT> acc;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int h = 0; h < 4; ++h) acc.v[nt][h] = 0.f;
#pragma unroll 1
    for (int jj = 0; jj < ntl * NPW; ++jj) {
      bool landed;
      const unsigned char* sl = acquire<NS>(tb, ring, jA2 + jj, budget, err, WS_WIN_SLOT, diag, landed);
      if (jj == ti * NPW + tp) {
        if (trace && wt == 0) trace[19] = gtime();
        acc = slot_mma<NT, WF>(sl, PW / 256, 0, reinterpret_cast<const uint16_t*>(sl + 8 * PW), PW / 32, k0c, nkc,
                           xf + (size_t)(tp * CPP + k0c) * FR);
      }
      // a chunk this warp does not read is handed back once it landed; each
      // W_in warp arrives for itself and for one routing warp, which never
      // touches the W_in chunks (so that the slots recycle while it routes)
      release_read<NS>(tb, jA2 + jj, landed, NCW / (NCW - RW));
    }
    group_sync(BAR_WIN, NCT - RW * 32);  // every W_in warp is done with x: its region takes the partials
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      pbuf[(wi * NT + nt) * 32 + lane] = make_float4(acc.v[nt][0], acc.v[nt][1], acc.v[nt][2], acc.v[nt][3]);
    group_sync(BAR_WIN, NCT - RW * 32);
    // H rows: thread (tile, token n, row r), the tile's two partials summed in
    // order; eight consecutive rows of a token gathered into one fragment entry
    if (F.hl && F.pdl_hl) asm volatile("griddepcontrol.wait;" ::: "memory");  // Hl (lora_hl)
#pragma unroll 1
    for (int idx = wt; idx < MAX_TILES * FR; idx += NCT - RW * 32) {  // FR = 16 rows x 8 NT tokens per tile
      const int i = idx / FR, rem = idx % FR, n = rem >> 4, r = rem & 15;
      if (i >= ntl) break;  // warp-uniform: a warp's 32 threads share i
      const int ll = (r & 7) * 4 + ((n & 7) >> 1), h = 2 * (r >> 3) + (n & 1), nt = n >> 3;
      const float* pf = reinterpret_cast<const float*>(pbuf);
      const int tg = t_lo + i, g = tg / (L / 16), rt = tg % (L / 16);
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < 2; ++w) s += pf[((((2 * i + w) * NT + nt) * 32 + ll) << 2) + h];
      if (WF == 1) s *= __ldg(A.W_in_gs + g);  // the tensor scale of W_in[g]
      if (F.hl && n < T) s += __ldcg(F.hl + ((size_t)g * 16 + n) * L + rt * 16 + r);  // the LoRA branch
      float e[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) e[q] = __shfl_sync(0xffffffffu, s, (lane & ~7) + q);
      if ((r & 7) == 0) {
        F.Hf[(size_t)g * CL * FR + entry_index<NT>(rt * 16 + (r & 8), n)] = pack_frag8(e);
      }
    }
    group_sync(BAR_WIN, NCT - RW * 32);
    if (wt == 0) {
      fence_gpu();
#pragma unroll 1
      for (int i = 0; i < ntl; ++i) atomicAdd(ctr + cm.done_in + ((t_lo + i) / (L / 16)) * CSTR, 1u);
      if (trace) trace[3] = gtime();
    }
  } else {
    // Every CTA routes all tokens itself: a warp per token selects the top-k
    // (topk.cuh), then one warp builds the tables and the work split.
    if (ctid == 0) wait_ge(tb, ctr + cm.done_router, (unsigned)nC, budget, err, WS_LOGITS, diag);
    group_sync(BAR_ROUTE, RW * 32);
    if (trace && ctid == 0) trace[15] = gtime();
#pragma unroll 1
    for (int t = warp; t < T; t += RW) {
      const float2 sw = topk_warp_thr(F.logits + (size_t)t * E, E, k, tb.u.tkscr[warp]);
      if (lane < k) {
        const int e = __float_as_int(sw.x);
        tb.idx[t * 16 + lane] = e;
        tb.w[t * 16 + lane] = sw.y;
        atomicOr(&tb.emask[e >> 5], 1u << (e & 31));
        if (c == 0) {
          A.idx[t * k + lane] = e;
          A.w[t * k + lane] = sw.y;
        }
      }
      __syncwarp();
    }
    group_sync(BAR_ROUTE, RW * 32);
    if (trace && ctid == 0) trace[11] = gtime();
    if (warp == 0) {
      build_tables(tb, epg);
      if (F.slot_of) {  // staged experts: where each routed expert's chunks are
#pragma unroll 1
        for (int i = lane; i < tb.n_act; i += 32) tb.eslot[i] = (int16_t)__ldcg(F.slot_of + tb.elist[i]);
        __syncwarp();
      }
      if (trace && lane == 0) trace[16] = gtime();
      plan(tb, c, nC, NSF, L, d);
      if (lane == 0) mbar_arrive(&tb.tbar);  // the producer may stream the expert weights
    }
    // (the W_in chunks are handed back by the W_in warps alone, see above)
  }
  cons_sync();
  if (trace && ctid == 0) trace[4] = gtime();
  const int n_actg = tb.n_actg;

  // ------------------------------------------------------------ B expert units
  // Per unit q: the 16 gate / up tasks -> partials; one CTA barrier; then
  // every thread forms one element of the unit's slice v = w silu(gate h) up h
  // (the gate and up partials summed in K-quarter order), and the warps
  // contract the previous unit's slice with its Down columns. The partials and
  // slices are double-buffered, so the barrier of unit q + 1 also separates
  // the slice writes of unit q from their reads.
  {
    const int u_lo = tb.u_lo, nu = tb.u_hi - tb.u_lo;
    const int mat = warp >> 3, mt = (warp >> 2) & 1, cw = warp & 3;
    int gc0, gc1;
    split(CL, cw, 4, gc0, gc1);  // this warp's K chunks of its gate / up tile
    float zacc[MAX_MPW][NT][4];
#pragma unroll
    for (int m = 0; m < MAX_MPW; ++m)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int h = 0; h < 4; ++h) zacc[m][nt][h] = 0.f;
    int hg = -1;
#pragma unroll 1
    for (int q = 0; q <= nu; ++q) {
      const int par = q & 1;
      if (q < nu) {  // ---- gate / up of unit q
        const int u = u_lo + q, e = tb.elist[u / NSF], g = e / epg;
        if (g != hg) {  // this group's H into shared memory
          cons_sync();
          if (ctid == 0) wait_ge(tb, ctr + cm.done_in + g * CSTR, (unsigned)(L / 16), budget, err, WS_H, diag);
          cons_sync();
          copy_frags(xf, F.Hf + (size_t)g * CL * FR, CL * FR, ctid);
          cons_sync();
          if (trace && ctid == 0 && hg < 0) trace[5] = gtime();
          hg = g;
        }
        const int jg = jB + 3 * q;
        {  // the other matrix's chunk is not read by this warp: handed back once it landed
          bool landed;
          acquire<NS>(tb, ring, jg + 1 - mat, budget, err, WS_GU_SLOT, diag, landed);
          release_read<NS>(tb, jg + 1 - mat, landed);
        }
        float a[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int h = 0; h < 4; ++h) a[nt][h] = 0.f;
        {
          bool landed;
          const unsigned char* sl = acquire<NS>(tb, ring, jg + mat, budget, err, WS_GU_SLOT, diag, landed);
          if (trace && ctid == 0 && q == 0) trace[21] = gtime();
          mma_slot<NT, WF>(sl, L / 256, 16 * mt, reinterpret_cast<const uint16_t*>(sl + 16 * L), L / 32, gc0, gc1 - gc0,
                       xf + (size_t)gc0 * FR, a);  // inline: the Down accumulators stay live across it
          release_read<NS>(tb, jg + mat, landed);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          pbuf[((par * NCW + warp) * NT + nt) * 32 + lane] = make_float4(a[nt][0], a[nt][1], a[nt][2], a[nt][3]);
      }
      cons_sync();
      if (trace && ctid == 0 && q == 0) trace[12] = gtime();
      if (q < nu && ctid < 256 * NT) {  // ---- unit q's slice, one element per thread
        const int e = tb.elist[(u_lo + q) / NSF];
        const int h = ctid & 3, ln = (ctid >> 2) & 31, r2 = ctid >> 7, nt = r2 % NT, m2 = r2 / NT;
        const float* pf = reinterpret_cast<const float*>(pbuf);
        float gs = 0.f, us = 0.f;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          gs += pf[((((par * NCW + m2 * 4 + q4) * NT + nt) * 32 + ln) << 2) + h];
          us += pf[((((par * NCW + 8 + m2 * 4 + q4) * NT + nt) * 32 + ln) << 2) + h];
        }
        if (WF == 1) {  // the tensor scales of Gate_e and Up_e
          gs *= __ldg(A.gate_gs + e);
          us *= __ldg(A.up_gs + e);
        }
        const int r = 16 * m2 + (ln >> 2) + 8 * (h >> 1), n = nt * 8 + 2 * (ln & 3) + (h & 1);
        const float wv = route_weight(tb, n, e);
        const float v = wv != 0.f ? wv * gs * __frcp_rn(1.f + __expf(-gs)) * us : 0.f;
        const int el = r & 7, ent = (n >> 3) * 32 + (n & 7) * 4 + (r >> 3);
        reinterpret_cast<__half*>(vbuf + par * NT * 32)[ent * 8 + (el < 4 ? 2 * el : 2 * (el - 4) + 1)] =
            __float2half_rn(v);
      }
      if (q >= 1) {  // ---- Down of unit q - 1 (its slice was formed before this unit's barrier)
        const int qq = q - 1, pq = qq & 1, u = u_lo + qq, es = u / NSF;
        const int jd = jB + 3 * qq + 2;
        bool landed;
        const unsigned char* sl = acquire<NS>(tb, ring, jd, budget, err, WS_DOWN_SLOT, diag, landed);
        const uint32_t* wsl = reinterpret_cast<const uint32_t*>(sl);
        const uint16_t* sc = reinterpret_cast<const uint16_t*>(sl + 16 * L);
        if (WF == 0) {
#pragma unroll
          for (int m = 0; m < MAX_MPW; ++m)
            if (m < MPW) mma_slice32<NT, WF>(wsl, sc, warp * MPW + m, vbuf + pq * NT * 32, zacc[m]);
        } else {  // each expert's Down has its own tensor scale: applied before the group's sum
          const float sd = __ldg(A.down_gs + tb.elist[es]);
#pragma unroll
          for (int m = 0; m < MAX_MPW; ++m) {
            if (m >= MPW) break;
            float t[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int hh = 0; hh < 4; ++hh) t[nt][hh] = 0.f;
            mma_slice32<NT, WF>(wsl, sc, warp * MPW + m, vbuf + pq * NT * 32, t);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int hh = 0; hh < 4; ++hh) zacc[m][nt][hh] = fmaf(sd, t[nt][hh], zacc[m][nt][hh]);
          }
        }
        release_read<NS>(tb, jd, landed);
        if (trace && ctid == 0 && qq == 0) trace[14] = gtime();
        // the last unit of its group in this CTA: write the group's partial of Z
        const int g = tb.elist[es] / epg;
        const bool flush = qq + 1 == nu || tb.elist[(u + 1) / NSF] / epg != g;
        if (flush) {
          const int gi = group_slot(tb, es);
          const int slot = tb.gpbase[gi] + busy_ctas(tb.gplo[gi], c, tb.n_act * NSF, nC);
          float* zp = F.Zpart + (size_t)slot * 16 * L;
#pragma unroll
          for (int m = 0; m < MAX_MPW; ++m) {
            if (m >= MPW) break;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                const int row = 16 * (warp * MPW + m) + gid + 8 * (h >> 1), n = nt * 8 + 2 * tig + (h & 1);
                if (n < T) zp[(size_t)n * L + row] = zacc[m][nt][h];
                zacc[m][nt][h] = 0.f;
              }
          }
          fence_gpu();
          __syncwarp();
          if (lane == 0) atomicAdd(ctr + cm.done_part + g * CSTR, 1u);
        }
      }
    }
  }

  if (trace && ctid == 0) trace[6] = gtime();
  // ------------------------------------------------------------ C Z reduce
  {
    const int z_lo = tb.z_lo, nz = tb.z_hi - tb.z_lo;
    const int wg = warp >> 2, qt = warp & 3, run = lane & 1, n = lane >> 1;
#pragma unroll 1
    for (int r0 = 0; r0 < nz; r0 += 4) {
      const int zq = r0 + wg;
      if (zq < nz) {
        const int it = z_lo + zq, gi = it / (L / 16), rb = it % (L / 16), g = tb.glist[gi];
        const int P = tb.gpn[gi], base = tb.gpbase[gi];
        warp_wait_ge(tb, ctr + cm.done_part + g * CSTR, (unsigned)(NCW * P), budget, err, WS_ZPART, diag);
        int p0, p1;
        split(P, qt, 4, p0, p1);
        float4 s0 = make_float4(0.f, 0.f, 0.f, 0.f), s1 = s0;
        if (n < T) {
#pragma unroll 1
          for (int p = p0; p < p1; p += 4) {
            float4 v[4][2];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const float* src = F.Zpart + ((size_t)(base + p + q4) * 16 + n) * L + rb * 16 + run * 8;
              const bool ok = p + q4 < p1;
              v[q4][0] = ok ? __ldcg(reinterpret_cast<const float4*>(src)) : make_float4(0.f, 0.f, 0.f, 0.f);
              v[q4][1] = ok ? __ldcg(reinterpret_cast<const float4*>(src + 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              s0.x += v[q4][0].x; s0.y += v[q4][0].y; s0.z += v[q4][0].z; s0.w += v[q4][0].w;
              s1.x += v[q4][1].x; s1.y += v[q4][1].y; s1.z += v[q4][1].z; s1.w += v[q4][1].w;
            }
          }
        }
        zred[((wg * 4 + qt) * 32 + lane) * 2] = s0;
        zred[((wg * 4 + qt) * 32 + lane) * 2 + 1] = s1;
        __threadfence_block();
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atomicAdd(&tb.tk_z[wg], 1) == 3;
        if (__shfl_sync(0xffffffffu, last, 0)) {  // quarters summed in order
          __threadfence_block();
          float e[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const float4 a = zred[((wg * 4 + q4) * 32 + lane) * 2], b = zred[((wg * 4 + q4) * 32 + lane) * 2 + 1];
            e[0] += a.x; e[1] += a.y; e[2] += a.z; e[3] += a.w; e[4] += b.x; e[5] += b.y; e[6] += b.z; e[7] += b.w;
          }
          if (lane == 0) tb.tk_z[wg] = 0;
          if (n < 8 * NT) F.Zf[(size_t)g * CL * FR + entry_index<NT>(rb * 16 + run * 8, n)] = pack_frag8(e);
          if (F.zlin && n < T) {  // Z in fp32 for the LoRA branch
            float* zl = F.zlin + ((size_t)g * 16 + n) * L + rb * 16 + run * 8;
            *reinterpret_cast<float4*>(zl) = make_float4(e[0], e[1], e[2], e[3]);
            *reinterpret_cast<float4*>(zl + 4) = make_float4(e[4], e[5], e[6], e[7]);
          }
          fence_gpu();
          __syncwarp();
          if (lane == 0) atomicAdd(ctr + cm.done_z + g * CSTR, 1u);
        }
      }
      cons_sync();
    }
  }

  // ------------------------------------------------------------ D W_out
  // Per item (group g, 32 rows of Y[g]): the 16 warp tasks -> partials; one
  // CTA barrier; every thread sums one element over the 8 K-eighths in order
  // and writes it to Y[g]. After the CTA's last item, one ticket per item
  // (behind a release fence); the CTA that brings a row block's count to the
  // number of routed groups sums the groups in ascending order (+ residual)
  // into y.
  if (trace && ctid == 0) trace[7] = gtime();
  if (ctid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  {
    const int o_lo = tb.o_lo, no = tb.o_hi - tb.o_lo, jD = jB + 3 * (tb.u_hi - tb.u_lo);
    const int wm = warp >> 3;
    int oc0, oc1;
    split(CL, warp & 7, 8, oc0, oc1);
    int zg = -1;
#pragma unroll 1
    for (int q = 0; q <= no; ++q) {
      const int par = q & 1;
      if (q < no) {
        const int it = o_lo + q, g = tb.glist[it / (d / 32)];
        if (g != zg) {  // this group's Z into shared memory
          cons_sync();
          if (ctid == 0) wait_ge(tb, ctr + cm.done_z + g * CSTR, (unsigned)(L / 16), budget, err, WS_Z, diag);
          cons_sync();
          copy_frags(xf, F.Zf + (size_t)g * CL * FR, CL * FR, ctid);
          cons_sync();
          if (trace && ctid == 0 && zg < 0) trace[8] = gtime();
          zg = g;
        }
        float a[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int h = 0; h < 4; ++h) a[nt][h] = 0.f;
        bool landed;
        const unsigned char* sl = acquire<NS>(tb, ring, jD + q, budget, err, WS_WOUT_SLOT, diag, landed);
        if (trace && ctid == 0 && q == 0) trace[25] = gtime();
        const Acc<NT> t = slot_mma<NT, WF>(sl, L / 256, 16 * wm, reinterpret_cast<const uint16_t*>(sl + 16 * L), L / 32, oc0,
                                       oc1 - oc0, xf + (size_t)oc0 * FR);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int h = 0; h < 4; ++h) a[nt][h] = t.v[nt][h];
        release_read<NS>(tb, jD + q, landed);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          pbuf[((par * NCW + warp) * NT + nt) * 32 + lane] = make_float4(a[nt][0], a[nt][1], a[nt][2], a[nt][3]);
      }
      if (q > 0 && ctid < 256 * NT) {  // ---- item q - 1's rows of Y[g], one element per thread
        const int qq = q - 1, pq = qq & 1, it = o_lo + qq, g = tb.glist[it / (d / 32)], ot = it % (d / 32);
        const int h = ctid & 3, ln = (ctid >> 2) & 31, r2 = ctid >> 7, nt = r2 % NT, m2 = r2 / NT;
        const float* pf = reinterpret_cast<const float*>(pbuf);
        float s = 0.f;
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) s += pf[((((pq * NCW + m2 * 8 + q8) * NT + nt) * 32 + ln) << 2) + h];
        if (WF == 1) s *= __ldg(A.W_out_gs + g);  // the tensor scale of W_out[g]
        const int row = ot * 32 + 16 * m2 + (ln >> 2) + 8 * (h >> 1), n = nt * 8 + 2 * (ln & 3) + (h & 1);
        if (n < T) F.Yp[((size_t)g * 16 + n) * d + row] = s;
      }
      cons_sync();
    }
    if (!F.no_combine) {  // (with the LoRA branch, lora_out combines the groups)
      // the tickets: each behind a release fence, cumulative over the barrier above
      if (ctid < no) {
        const int ot = (o_lo + ctid) % (d / 32);
        fence_gpu();
        const unsigned old = atomicAdd(ctr + cm.tk_wout + ot * CSTR, 1u);
        tb.fin[ctid] = old == (unsigned)(n_actg - 1) ? (int16_t)ot : (int16_t)-1;
        if (old == (unsigned)(n_actg - 1)) fence_gpu();
      }
      cons_sync();
      // every group of a finished row block is in: combine in ascending group order
#pragma unroll 1
      for (int qd = ctid; qd < no * 8 * T; qd += NCT) {
        const int ot = tb.fin[qd / (8 * T)];
        if (ot < 0) continue;
        const int rem = qd % (8 * T), n = rem >> 3, row = ot * 32 + (rem & 7) * 4;
        float4 acc4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
        for (int g0 = 0; g0 < n_actg; g0 += 8) {
          float4 p4[8];
#pragma unroll
          for (int gg = 0; gg < 8; ++gg)
            p4[gg] = g0 + gg < n_actg
                         ? __ldcg(reinterpret_cast<const float4*>(F.Yp + ((size_t)tb.glist[g0 + gg] * 16 + n) * d + row))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int gg = 0; gg < 8; ++gg) {
            acc4.x += p4[gg].x; acc4.y += p4[gg].y; acc4.z += p4[gg].z; acc4.w += p4[gg].w;
          }
        }
        if (F.round_first) {  // the layer's output is rounded before the residual is added
          acc4.x = bf16_to_f32(f32_to_bf16_rne(acc4.x));
          acc4.y = bf16_to_f32(f32_to_bf16_rne(acc4.y));
          acc4.z = bf16_to_f32(f32_to_bf16_rne(acc4.z));
          acc4.w = bf16_to_f32(f32_to_bf16_rne(acc4.w));
        }
        if (A.residual) {
          const uint2 rb = *reinterpret_cast<const uint2*>(A.residual + (size_t)n * d + row);
          acc4.x += __uint_as_float(rb.x << 16);
          acc4.y += __uint_as_float(rb.x & 0xffff0000u);
          acc4.z += __uint_as_float(rb.y << 16);
          acc4.w += __uint_as_float(rb.y & 0xffff0000u);
        }
        uint2 o;
        o.x = (uint32_t)f32_to_bf16_rne(acc4.x) | ((uint32_t)f32_to_bf16_rne(acc4.y) << 16);
        o.y = (uint32_t)f32_to_bf16_rne(acc4.z) | ((uint32_t)f32_to_bf16_rne(acc4.w) << 16);
        *reinterpret_cast<uint2*>(A.y + (size_t)n * d + row) = o;
      }
    }
  }
  if (trace && ctid == 0) trace[9] = gtime();
  end_sync();
}

// ===================================================================== host
size_t fused_counter_words(int d, int E, int G, int L) {
  (void)E;
  (void)L;
  return 2 * (size_t)ctr_map(d, G).n;
}

size_t fused_zpart_bytes(int G, int L, int grid) { return (size_t)(grid + G) * 16 * L * 4; }
size_t fused_diag_bytes(int grid) { return (size_t)(1 + 32 * grid) * 8; }

// ------------------------------------------------------------ streaming pack
namespace {
// One chunk per CTA: `rows` rows of `wb` bytes of packed int4 (wb a multiple
// of 128) from q (row stride qs bytes), rows band*rows .. and bytes piece*wb ..
// of each row, written as 128-byte lines in the 128-byte swizzle (16-byte unit
// u of line i at unit u ^ (i & 7)); then the same rows' `wsc` bf16 scales
// from s (row stride ss), columns piece*wsc ... Chunk c (band c / npc, piece
// c % npc) goes to out + c * cstride + coff.
struct PackSpec {
  const uint8_t* q;
  size_t qs;
  const uint16_t* s;
  size_t ss;
  int rows, wb, wsc, npc;
  uint8_t* out;
  size_t cstride, coff;
  int fp4;  // NVFP4 codes: each 32-bit word re-ordered (fp4_word_order)
};

// An NVFP4 code word, natural order (element i in nibble i), re-ordered so
// that byte b holds elements b and b + 4.
__device__ __forceinline__ uint32_t fp4_word_order(uint32_t v) {
  uint32_t o = 0;
#pragma unroll
  for (int b = 0; b < 4; ++b) o |= (((v >> (4 * b)) & 15u) | (((v >> (4 * (b + 4))) & 15u) << 4)) << (8 * b);
  return o;
}
__device__ __forceinline__ uint4 fp4_order4(uint4 v) {
  return make_uint4(fp4_word_order(v.x), fp4_word_order(v.y), fp4_word_order(v.z), fp4_word_order(v.w));
}

__global__ void __launch_bounds__(256) pack_swz_kernel(PackSpec P) {
  const int c = blockIdx.x, band = c / P.npc, piece = c % P.npc;
  const size_t row0 = (size_t)band * P.rows;
  uint8_t* dst = P.out + (size_t)c * P.cstride + P.coff;
  const int lpr = P.wb / 128, nu = P.rows * lpr * 8;
  for (int i = threadIdx.x; i < nu; i += blockDim.x) {
    const int line = i >> 3, u = i & 7, r = line / lpr, li = line % lpr;
    uint4 v = *reinterpret_cast<const uint4*>(P.q + (row0 + r) * P.qs + (size_t)piece * P.wb + li * 128 + u * 16);
    if (P.fp4) v = fp4_order4(v);
    *reinterpret_cast<uint4*>(dst + line * 128 + ((u ^ (line & 7)) << 4)) = v;
  }
  uint16_t* sd = reinterpret_cast<uint16_t*>(dst + (size_t)P.rows * P.wb);
  for (int i = threadIdx.x; i < P.rows * P.wsc; i += blockDim.x) {
    const int r = i / P.wsc, cc = i % P.wsc;
    sd[i] = P.s[(row0 + r) * P.ss + (size_t)piece * P.wsc + cc];
  }
}

// The Down columns of unit c = (e, slice): for every latent row l, the 16
// bytes of Down_e[l] holding the slice's 32 int4 ([L][16 B], unswizzled),
// then the rows' scales of that slice ([L] bf16).
__global__ void __launch_bounds__(256) pack_down_kernel(const uint8_t* q, const uint16_t* s, int L, int f,
                                                        uint8_t* unit, int fp4) {
  const int nsf = f / FS, c = blockIdx.x, e = c / nsf, sl = c % nsf;
  uint8_t* dst = unit + ((size_t)c * 3 + 2) * 18 * L;
  for (int l = threadIdx.x; l < L; l += blockDim.x) {
    const size_t row = (size_t)e * L + l;
    const uint4 v = *reinterpret_cast<const uint4*>(q + row * (f / 2) + sl * 16);
    *reinterpret_cast<uint4*>(dst + (size_t)l * 16) = fp4 ? fp4_order4(v) : v;
    reinterpret_cast<uint16_t*>(dst + (size_t)16 * L)[l] = s[row * nsf + sl];
  }
}

size_t al256(size_t v) { return (v + 255) & ~(size_t)255; }
struct PackLayout {
  size_t win, unit, wout, end;
};
PackLayout pack_layout(int d, int E, int G, int L, int f, bool with_unit = true) {
  const int PW = d < 2048 ? d : 2048;
  PackLayout p;
  p.win = 0;
  p.unit = al256(p.win + (size_t)G * (L / 16) * (d / PW) * 9 * PW);
  p.wout = al256(p.unit + (with_unit ? (size_t)E * (f / FS) * 3 * 18 * L : 0));
  p.end = al256(p.wout + (size_t)G * (d / 32) * 18 * L);
  return p;
}
}  // namespace

size_t decode_pack_bytes(int d, int E, int G, int L, int f) { return pack_layout(d, E, G, L, f).end; }
size_t decode_pack_bytes_shared(int d, int E, int G, int L, int f) { return pack_layout(d, E, G, L, f, false).end; }
size_t decode_expert_bytes(int L, int f) { return (size_t)(f / FS) * 3 * 18 * L; }

cudaError_t launch_decode_pack(const DecodeArgs& A, uint8_t* buf, DecodePack* pk, cudaStream_t st,
                               uint8_t* unit_buf) {
  const int d = A.d, E = A.E, G = A.G, L = A.L, f = A.f, PW = d < 2048 ? d : 2048, nsf = f / FS;
  const PackLayout lay = pack_layout(d, E, G, L, f, unit_buf == nullptr);
  uint8_t* units = unit_buf ? unit_buf : buf + lay.unit;
  pk->wr = A.W_r;
  pk->win = buf + lay.win;
  pk->unit = units;
  pk->wout = buf + lay.wout;
  // W_in: 16-row tiles in pieces of PW columns
  const int fp4 = A.wfmt != 0;  // (the scales move as 16-bit words in both formats: one bf16 or two E4M3 per 32)
  PackSpec w{A.W_in_q, (size_t)d / 2, A.W_in_s, (size_t)d / 32, 16, PW / 2, PW / 32, d / PW, buf + lay.win,
             (size_t)9 * PW, 0, fp4};
  pack_swz_kernel<<<G * (L / 16) * (d / PW), 256, 0, st>>>(w);
  // gate and up: 32 rows (one f-slice of one expert) each, at parts 0 and 1 of the unit
  PackSpec g{A.gate_q, (size_t)L / 2, A.gate_s, (size_t)L / 32, FS, L / 2, L / 32, 1, units,
             (size_t)3 * 18 * L, 0, fp4};
  pack_swz_kernel<<<E * nsf, 256, 0, st>>>(g);
  PackSpec u = g;
  u.q = A.up_q;
  u.s = A.up_s;
  u.coff = (size_t)18 * L;
  pack_swz_kernel<<<E * nsf, 256, 0, st>>>(u);
  pack_down_kernel<<<E * nsf, 256, 0, st>>>(A.down_q, A.down_s, L, f, units, fp4);
  // W_out: 32-row blocks
  PackSpec o{A.W_out_q, (size_t)L / 2, A.W_out_s, (size_t)L / 32, 32, L / 2, L / 32, 1, buf + lay.wout,
             (size_t)18 * L, 0, fp4};
  pack_swz_kernel<<<G * (d / 32), 256, 0, st>>>(o);
  return cudaGetLastError();
}

bool fused_decode_supported(const DecodeArgs& A, int grid) {
  if ((A.r != 0 && !lora_fused_supported(A)) || A.T < 1 || A.T > 16 || grid < 1) return false;
  if (!A.W_r || (reinterpret_cast<uintptr_t>(A.W_r) & 15) != 0) return false;  // router rows by bulk copy
  if (A.E > 512 || A.G > 64 || A.k > 16 || A.E > MAX_RX * grid) return false;
  if (A.d > 4096 || !(A.d == 1024 || A.d % 2048 == 0)) return false;  // router rows and W_in pieces
  if (A.L != 256 && A.L != 512 && A.L != 1024) return false;
  if (A.f % FS != 0 || A.f < FS || (long long)A.T * A.k > 256) return false;
  if ((long long)A.G * (A.L / 16) > (long long)MAX_TILES * grid) return false;
  return true;
}

cudaError_t fused_set_attributes() {
  cudaFuncSetAttribute(decode_fused_kernel<1, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_smem<1>());
  cudaFuncSetAttribute(decode_fused_kernel<2, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_smem<2>());
  cudaFuncSetAttribute(decode_fused_kernel<1, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_smem<1>());
  cudaFuncSetAttribute(decode_fused_kernel<2, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_smem<2>());
  return cudaGetLastError();
}

int fused_grid(int num_sms) {
  int per1 = 0, per2 = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per1, decode_fused_kernel<1, 0>, NTHR, dyn_smem<1>()) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per2, decode_fused_kernel<2, 0>, NTHR, dyn_smem<2>()) !=
          cudaSuccess ||
      per1 < 1 || per2 < 1) {
    cudaGetLastError();
    return 0;
  }
  return num_sms;  // one CTA per SM
}

cudaError_t launch_decode_fused(const FusedArgs& F, int grid, cudaStream_t st, int pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(NTHR);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    // one CTA per SM: the CTAs become resident as the previous layer's exit,
    // and every wait across CTAs is bounded
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
  } else {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (F.A.T <= 8) {
    cfg.dynamicSmemBytes = dyn_smem<1>();
    return F.A.wfmt ? cudaLaunchKernelEx(&cfg, decode_fused_kernel<1, 1>, F)
                    : cudaLaunchKernelEx(&cfg, decode_fused_kernel<1, 0>, F);
  }
  cfg.dynamicSmemBytes = dyn_smem<2>();
  return F.A.wfmt ? cudaLaunchKernelEx(&cfg, decode_fused_kernel<2, 1>, F)
                  : cudaLaunchKernelEx(&cfg, decode_fused_kernel<2, 0>, F);
}

}  // namespace lmoe
