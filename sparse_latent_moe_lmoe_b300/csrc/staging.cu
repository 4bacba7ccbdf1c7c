// The staged expert cache of a layer (LMOE_FLAG_STAGED_EXPERTS).
//
// "Edge0-145B: Frontier AI Capabilities on Your Own Computer", "Under the
// Hood of Edge0", "Loading": frequently used experts stay in GPU memory, an
// expert library sits in system memory and experts are brought into GPU
// memory as needed. "Edge0-145B: Run a 145B Open-Source Model on Your
// Laptop", "The Three Pillars That Make It Fast": active experts load into a
// staged fixed-slot buffer, and a prerouter's prediction of the next layer's
// routing drives the prefetch so that the copies overlap the current layer.
//
// Here the library is the handle's page-locked host copy of every expert in
// the decode pass's chunk layout (one expert = its f/32 units of gate, up
// and Down chunks, contiguous), and GPU memory holds S fixed slots of that
// size. Two small kernels stage a set of experts:
//   plan  (one CTA): the experts of the set that hold no slot, and for each
//         a victim slot -- the next slots in clock order whose expert is not
//         in the set -- then the tables (expert -> slot, slot -> expert)
//   copy  (a grid): every planned expert from host memory into its slot
// Both use a few KB of shared memory and few registers, so on a second
// stream they run beside a decode pass (one CTA per SM) of another layer.
#include "common.cuh"
#include "decode.cuh"

namespace lmoe {

namespace {
constexpr int PLAN_THREADS = 256;
constexpr int MAX_WANT = 256;  // experts per staged set (16 tokens x k <= 16)

// ordered compaction over the CTA: returns this thread's position among the
// flagged threads (or -1) and adds the count to *total (all threads see it)
__device__ int ordered_pos(bool flag, int* warp_cnt, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned bal = __ballot_sync(0xffffffffu, flag);
  if (lane == 0) warp_cnt[warp] = __popc(bal);
  __syncthreads();
  int before = 0, all = 0;
#pragma unroll 1
  for (int w = 0; w < PLAN_THREADS / 32; ++w) {
    if (w < warp) before += warp_cnt[w];
    all += warp_cnt[w];
  }
  __syncthreads();
  *total = all;
  return flag ? before + __popc(bal & ((1u << lane) - 1u)) : -1;
}
}  // namespace

__global__ void __launch_bounds__(PLAN_THREADS) stage_plan_kernel(StagePlan P) {
  __shared__ unsigned want[32];  // E <= 1024
  __shared__ int miss[MAX_WANT], victim[MAX_WANT];
  __shared__ int warp_cnt[PLAN_THREADS / 32];
  const int t = threadIdx.x, E = P.E, S = P.S;
  if (t < 32) want[t] = 0u;
  __syncthreads();
  for (int a = t; a < P.n; a += PLAN_THREADS) {
    const int e = P.idx[a];
    if (e < 0 || e >= E) {
      set_error(P.err, ERRBIT_BAD_INDEX);
      continue;
    }
    atomicOr(&want[e >> 5], 1u << (e & 31));
  }
  __syncthreads();
  // the wanted experts without a slot, in ascending order
  int n_want = 0, n_miss = 0;
#pragma unroll 1
  for (int base = 0; base < E; base += PLAN_THREADS) {
    const int e = base + t;
    const bool w = e < E && ((want[e >> 5] >> (e & 31)) & 1u);
    const bool m = w && P.slot_of[e] < 0;
    int cw, cm;
    (void)ordered_pos(w, warp_cnt, &cw);
    const int pm = ordered_pos(m, warp_cnt, &cm);
    if (pm >= 0 && n_miss + pm < MAX_WANT) miss[n_miss + pm] = e;
    n_want += cw;
    n_miss += cm;
  }
  if (n_miss > MAX_WANT) n_miss = MAX_WANT;
  // victims: slots in clock order whose expert is not wanted
  const unsigned clock0 = P.st->clock;
  int n_vic = 0, last = -1;
#pragma unroll 1
  for (int base = 0; base < S && n_vic < n_miss; base += PLAN_THREADS) {
    const int r = base + t;
    const int s = (int)((clock0 + (unsigned)r) % (unsigned)S);
    bool free_slot = false;
    if (r < S) {
      const int old = P.expert_in[s];
      free_slot = old < 0 || !((want[old >> 5] >> (old & 31)) & 1u);
    }
    int cv;
    const int pv = ordered_pos(free_slot, warp_cnt, &cv);
    if (pv >= 0 && n_vic + pv < n_miss) {
      victim[n_vic + pv] = s;
      if (n_vic + pv == n_miss - 1) last = s;
    }
    n_vic += cv;
  }
  __syncthreads();
  const int n_copy = n_vic < n_miss ? n_vic : n_miss;
  if (n_copy < n_miss && P.must) set_error(P.err, ERRBIT_BAD_DATA);  // cannot happen when S >= the set's size
  // the tables: each victim's old expert loses its slot, each missing expert takes one
  for (int i = t; i < n_copy; i += PLAN_THREADS) {
    const int s = victim[i], e = miss[i], old = P.expert_in[s];
    if (old >= 0) P.slot_of[old] = -1;
    P.expert_in[s] = e;
    P.slot_of[e] = s;
    P.copies[i] = make_int2(e, s);
  }
  __shared__ int s_last;
  if (t == 0) s_last = -1;
  __syncthreads();
  if (last >= 0) s_last = last;
  __syncthreads();
  if (t == 0) {
    StageState* st = P.st;
    st->n_copy = (unsigned)n_copy;
    if (n_copy > 0 && s_last >= 0) st->clock = (unsigned)(s_last + 1) % (unsigned)S;
    st->bytes += (unsigned long long)n_copy * P.expert_bytes;
    if (P.must) {
      st->passes += 1;
      st->routed += (unsigned long long)n_want;
      st->hits += (unsigned long long)(n_want - n_miss);
      st->on_demand += (unsigned long long)n_copy;
    } else {
      st->prefetched += (unsigned long long)n_copy;
    }
  }
}

// every planned expert (n_copy of them, from the plan) from the host library
// into its slot: 16-byte words, several loads in flight per thread
__global__ void __launch_bounds__(256) stage_copy_kernel(const uint4* __restrict__ lib, uint4* __restrict__ slots,
                                                         const int2* __restrict__ copies, const StageState* st,
                                                         size_t words) {
  const size_t n = (size_t)st->n_copy * words;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
#pragma unroll 1
  for (size_t i0 = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i0 < n; i0 += 4 * stride) {
    uint4 v[4];
    size_t dst[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const size_t i = i0 + u * stride;
      dst[u] = (size_t)-1;
      if (i < n) {
        const size_t c = i / words, w = i % words;
        const int2 es = copies[c];
        v[u] = lib[(size_t)es.x * words + w];
        dst[u] = (size_t)es.y * words + w;
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (dst[u] != (size_t)-1) slots[dst[u]] = v[u];
  }
}

cudaError_t launch_stage_plan(const StagePlan& P, cudaStream_t st) {
  stage_plan_kernel<<<1, PLAN_THREADS, 0, st>>>(P);
  return cudaGetLastError();
}

cudaError_t launch_stage_copy(const StagePlan& P, const uint8_t* lib, uint8_t* slots, int num_sms, cudaStream_t st) {
  stage_copy_kernel<<<2 * num_sms, 256, 0, st>>>(reinterpret_cast<const uint4*>(lib), reinterpret_cast<uint4*>(slots),
                                                 P.copies, P.st, P.expert_bytes / 16);
  return cudaGetLastError();
}

}  // namespace lmoe
