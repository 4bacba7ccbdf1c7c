// The C ABI of the latent MoE layer (declared in include/lmoe.h): host-side
// validation, the handle, the workspace layout and the dispatch to the
// decode-path and prefill-path kernels.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>
#include <new>
#include <vector>

#include "../../include/lmoe.h"
#include "decode.cuh"
#include "prefill.cuh"

using namespace lmoe;

struct lmoe_handle {
  lmoe_config cfg;
  lmoe_weights w;
  int device;
  int num_sms;
  unsigned* d_err;       // device error word
  unsigned* d_tickets;   // ticket counters, zero between calls
  uint16_t* d_wr_split;  // [3][E][d] bf16 split of W_r (hi, mid, lo) for the tensor-core router
  long long timeout;
  int fused_grid;  // CTAs of the single-kernel decode pass (0: unavailable)
  DecodePack pk;                     // where the single-kernel decode pass streams its weights from
  bool pack_ok;                      // the decode pack exists (the single-kernel pass is possible)
  unsigned* d_ctr;                   // its arrival counters (two copies)
  unsigned long long* d_launches;    // its launch counter
  cudaStream_t aux;                  // second stream of the prefill path (fork / join by events)
  cudaEvent_t ev_fork, ev_join;
  uint8_t* d_pack;                   // the decode pass's chunk-major copy of the weights (decode_pack_bytes)
  std::vector<cudaEvent_t> events;
  // staged experts (LMOE_FLAG_STAGED_EXPERTS): the library in page-locked
  // host memory, the slots in GPU memory, their tables and the prerouter's
  // scratch
  bool staged;
  size_t expert_bytes;
  uint8_t* h_lib;                    // [E] experts in the decode pass's layout
  const uint8_t* d_lib;              // its device address
  uint8_t* d_slots;                  // [expert_slots] experts
  int32_t* d_slot_of;                // [E]
  int32_t* d_expert_in;              // [expert_slots]
  StageState* d_stage;
  int2* d_copies;                    // [256], the forward's plan
  int2* d_pre_copies;                // [256], the prerouter's plan
  float* d_pre_logits;               // [16][E]
  int32_t* d_pre_idx;                // [16][k]
  float* d_pre_w;                    // [16][k]
  unsigned* d_pre_tickets;           // the prerouter's router tickets
  cudaEvent_t ev_pf_in, ev_pf_done;  // stack: the prerouter's start and end on the second stream
  // lmoe_layer_forward_host: the last call's copies and layer as a CUDA
  // graph (captured on a stream of the handle's own, launched on the
  // caller's), replayed while the buffers and T stay the same
  struct HostGraph {
    const void* x;
    const void* r;
    void* y;
    void* ws;
    int T;
    cudaGraphExec_t exec;
  } hg;
  cudaStream_t cap;  // the capture stream (made on first use)
  // prefill-sized host calls: copy-in and copy-out streams and their events
  // (made on first use)
  cudaStream_t cin, cout;
  std::vector<cudaEvent_t> hev;
};

namespace {

constexpr int kMaxDecodeT = 16;
constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }
bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

lmoe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? LMOE_OK : LMOE_ERR_CUDA; }

lmoe_status validate_config(const lmoe_config* c) {
  if (!c) return LMOE_ERR_INVALID_ARG;
  if (c->d <= 0 || c->E <= 0 || c->G <= 0 || c->k <= 0 || c->L <= 0 || c->f <= 0) return LMOE_ERR_INVALID_ARG;
  if (c->weight_format != LMOE_WEIGHTS_INT4 && c->weight_format != LMOE_WEIGHTS_NVFP4) return LMOE_ERR_INVALID_ARG;
  if (c->qgroup != (c->weight_format == LMOE_WEIGHTS_NVFP4 ? 16 : 32)) return LMOE_ERR_UNSUPPORTED;
  if (c->E % c->G != 0) return LMOE_ERR_INVALID_ARG;
  if (c->k > c->E) return LMOE_ERR_INVALID_ARG;
  if (c->k > 16 || c->E > 1024 || c->G > 64) return LMOE_ERR_UNSUPPORTED;
  if (c->d % 128 != 0 || c->L % 32 != 0 || c->f % 32 != 0) return LMOE_ERR_UNSUPPORTED;
  if (c->L % 16 != 0 || c->f % 16 != 0) return LMOE_ERR_UNSUPPORTED;
  if (c->lora_rank < 0 || c->lora_rank > 128 || c->lora_rank % 16 != 0) return LMOE_ERR_UNSUPPORTED;
  if (c->flags & ~(unsigned)(LMOE_FLAG_MULTI_KERNEL_DECODE | LMOE_FLAG_STAGED_EXPERTS)) return LMOE_ERR_UNSUPPORTED;
  if ((c->flags & LMOE_FLAG_STAGED_EXPERTS) &&
      (c->expert_slots < (16 * c->k < c->E ? 16 * c->k : c->E) || c->expert_slots > c->E))
    return LMOE_ERR_INVALID_ARG;  // a pass's routed experts (at most min(E, 16 k)) must fit
  if (c->decode_max_T < 0 || c->decode_max_T > kMaxDecodeT) return LMOE_ERR_UNSUPPORTED;
  if (c->force_path < LMOE_PATH_AUTO || c->force_path > LMOE_PATH_PREFILL) return LMOE_ERR_INVALID_ARG;
  if (c->timeout_cycles < 0) return LMOE_ERR_INVALID_ARG;
  return LMOE_OK;
}

lmoe_status validate_weights(const lmoe_config* c, const lmoe_weights* w) {
  if (!w) return LMOE_ERR_INVALID_ARG;
  const void* req[] = {w->W_r, w->W_in_q, w->W_in_s, w->W_out_q, w->W_out_s, w->gate_q,
                       w->gate_s, w->up_q, w->up_s, w->down_q, w->down_s};
  for (const void* p : req) {
    if (!p) return LMOE_ERR_INVALID_ARG;
    if (!aligned16(p)) return LMOE_ERR_ALIGNMENT;
  }
  if (c->has_bias && !w->b_r) return LMOE_ERR_INVALID_ARG;
  if (c->weight_format == LMOE_WEIGHTS_NVFP4) {
    const void* gs[] = {w->W_in_gs, w->W_out_gs, w->gate_gs, w->up_gs, w->down_gs};
    for (const void* p : gs) {
      if (!p) return LMOE_ERR_INVALID_ARG;
      if (((uintptr_t)p & 3u) != 0) return LMOE_ERR_ALIGNMENT;
    }
  }
  if (c->lora_rank > 0) {
    const void* lr[] = {w->A_in, w->B_in, w->A_out, w->B_out};
    for (const void* p : lr) {
      if (!p) return LMOE_ERR_INVALID_ARG;
      if (!aligned16(p)) return LMOE_ERR_ALIGNMENT;
    }
  }
  return LMOE_OK;
}

lmoe_status check_handle(const lmoe_handle* h) { return h ? LMOE_OK : LMOE_ERR_INVALID_ARG; }

// K splits of the shared down-projection on the decode path: at most 8
// chunks of 128 per split (one activation slot), at least min(4, chunks).
int ks_in_for(const lmoe_config& c) {
  const int nch = (c.d + 127) / 128;
  const int a = nch < 4 ? nch : 4, b = (nch + 7) / 8;
  return a > b ? a : b;
}

// ticket layout in the handle: [0] route, [1 .. 1+d/64) multi-kernel wout
struct TicketMap {
  size_t total;
};
TicketMap ticket_map(const lmoe_config& c) {
  TicketMap t;
  t.total = 1 + (size_t)(c.d + 63) / 64 + lora_ticket_words(c.d, c.G);
  return t;
}

// ----------------------------------------------------------- workspace map
struct DecodeWs {
  size_t logits, idx, w, eo, sa, inv, go, gto, gt, ar, Hp, V, Z, Yp, Pin, Qout, Hf, Zf, Zpart, diag, perm_scratch, Lpart,
      end;
};

// grid: CTAs of the single-kernel decode pass (sizes its Z partials)
DecodeWs decode_ws(const lmoe_config& c, int T, int grid) {
  DecodeWs m;
  const int n = kMaxDecodeT;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_up(o + bytes);
    return at;
  };
  const int gk = c.G < c.k ? c.G : c.k;
  m.logits = take((size_t)n * c.E * 4);
  m.idx = take((size_t)n * c.k * 4);
  m.w = take((size_t)n * c.k * 4);
  m.eo = take((size_t)(c.E + 1) * 4);
  m.sa = take((size_t)n * c.k * 4);
  m.inv = take((size_t)n * c.k * 4);
  m.go = take((size_t)(c.G + 1) * 4);
  m.gto = take((size_t)(c.G + 1) * 4);
  m.gt = take((size_t)n * gk * 4);
  m.ar = take((size_t)n * c.k * 4);
  const int ks = ks_in_for(c) > c.d / 1024 ? ks_in_for(c) : c.d / 1024;
  m.Hp = take((size_t)ks * c.G * n * c.L * 4);
  m.V = take((size_t)256 * n * c.f * 4);  // [routed-expert slot <= 256][16][f]
  m.Z = take((size_t)c.G * n * c.L * 4);
  m.Yp = take((size_t)c.G * n * c.d * 4);
  m.Pin = take((size_t)c.G * n * (c.lora_rank > 0 ? c.lora_rank : 1) * 4);
  m.Qout = take((size_t)c.G * n * (c.lora_rank > 0 ? c.lora_rank : 1) * 4);
  m.Hf = take((size_t)c.G * c.L * 32);     // fp16 fragments, two token tiles: L/128 x 256 x 16 B
  m.Zf = take((size_t)c.G * c.L * 32);
  m.Zpart = take(fused_zpart_bytes(c.G, c.L, grid > 0 ? grid : 1));
  m.diag = take(fused_diag_bytes(grid > 0 ? grid : 1));
  m.perm_scratch = take(permute_scratch_bytes(T > n ? T : n, c.E, c.G));
  // the LoRA branch's partial sums around the single-kernel pass
  m.Lpart = take(c.lora_rank > 0 ? lora_ppart_bytes(c.d, c.G, c.lora_rank) + lora_qpart_bytes(c.L, c.G, c.lora_rank)
                                 : 0);
  m.end = o;
  return m;
}

PrefillArgs prefill_args(const lmoe_handle* h);

bool use_prefill(const lmoe_handle* h, int T) {
  const lmoe_config& c = h->cfg;
  if (!prefill_supported(prefill_args(h))) return false;
  if (c.force_path == LMOE_PATH_DECODE) return false;
  if (c.force_path == LMOE_PATH_PREFILL) return T > 0;
  const int mt = c.decode_max_T ? c.decode_max_T : kMaxDecodeT;
  return T > mt;
}

DecodeArgs base_args(const lmoe_handle* h, void* ws) {
  const lmoe_config& c = h->cfg;
  DecodeArgs A;
  memset(&A, 0, sizeof(A));
  A.d = c.d; A.E = c.E; A.G = c.G; A.k = c.k; A.L = c.L; A.f = c.f; A.r = c.lora_rank;
  A.epg = c.E / c.G;
  A.ks_in = ks_in_for(c);
  A.W_r = h->w.W_r; A.b_r = c.has_bias ? h->w.b_r : nullptr;
  A.W_in_q = h->w.W_in_q; A.W_in_s = h->w.W_in_s; A.W_out_q = h->w.W_out_q; A.W_out_s = h->w.W_out_s;
  A.gate_q = h->w.gate_q; A.gate_s = h->w.gate_s; A.up_q = h->w.up_q; A.up_s = h->w.up_s;
  A.down_q = h->w.down_q; A.down_s = h->w.down_s;
  A.A_in = h->w.A_in; A.B_in = h->w.B_in; A.A_out = h->w.A_out; A.B_out = h->w.B_out;
  A.wfmt = c.weight_format;
  A.W_in_gs = h->w.W_in_gs; A.W_out_gs = h->w.W_out_gs;
  A.gate_gs = h->w.gate_gs; A.up_gs = h->w.up_gs; A.down_gs = h->w.down_gs;
  const DecodeWs m = decode_ws(c, 0, h->num_sms);
  char* b = reinterpret_cast<char*>(ws);
  A.idx = reinterpret_cast<int32_t*>(b + m.idx);
  A.w = reinterpret_cast<float*>(b + m.w);
  A.pm.expert_offsets = reinterpret_cast<int32_t*>(b + m.eo);
  A.pm.sorted_assign = reinterpret_cast<int32_t*>(b + m.sa);
  A.pm.inv = reinterpret_cast<int32_t*>(b + m.inv);
  A.pm.group_offsets = reinterpret_cast<int32_t*>(b + m.go);
  A.pm.group_tok_offsets = reinterpret_cast<int32_t*>(b + m.gto);
  A.pm.group_tokens = reinterpret_cast<int32_t*>(b + m.gt);
  A.pm.assign_row = reinterpret_cast<int32_t*>(b + m.ar);
  A.Hp = reinterpret_cast<float*>(b + m.Hp);
  A.V = reinterpret_cast<float*>(b + m.V);
  A.Z = reinterpret_cast<float*>(b + m.Z);
  A.Yp = reinterpret_cast<float*>(b + m.Yp);
  A.Pin = reinterpret_cast<float*>(b + m.Pin);
  A.Qout = reinterpret_cast<float*>(b + m.Qout);
  A.tickets = h->d_tickets;
  A.err = h->d_err;
  return A;
}

float* ws_logits(const lmoe_handle* h, void* ws) {
  return reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + decode_ws(h->cfg, 0, h->num_sms).logits);
}

// Records an event; inside a stream capture the record becomes an external
// event node, which stays usable for timing after each graph launch.
void record_event(cudaEvent_t e, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
  else
    cudaEventRecord(e, s);
}

struct EventHook : StageHook {
  const std::vector<cudaEvent_t>* ev;
  int i = 0;
  void before(cudaStream_t s) override {
    if (ev && 2 * i < (int)ev->size()) record_event((*ev)[2 * i], s);
  }
  void after(cudaStream_t s) override {
    if (ev && 2 * i + 1 < (int)ev->size()) record_event((*ev)[2 * i + 1], s);
    ++i;
  }
};

lmoe_status pending_error() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? LMOE_OK : LMOE_ERR_CUDA;
}

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int cur;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

bool use_fused(const lmoe_handle* h, const DecodeArgs& A) {
  return !(h->cfg.flags & LMOE_FLAG_MULTI_KERNEL_DECODE) && h->fused_grid > 0 && h->pack_ok &&
         fused_decode_supported(A, h->fused_grid);
}

bool use_fused(const lmoe_handle* h, const DecodeArgs& A);

FusedArgs fused_args(const lmoe_handle* h, const DecodeArgs& A, void* ws) {
  FusedArgs F;
  memset(&F, 0, sizeof(F));
  F.A = A;
  F.pk = h->pk;
  const DecodeWs m = decode_ws(h->cfg, 0, h->num_sms);
  char* b = reinterpret_cast<char*>(ws);
  F.logits = reinterpret_cast<float*>(b + m.logits);
  F.Hf = reinterpret_cast<uint4*>(b + m.Hf);
  F.Zf = reinterpret_cast<uint4*>(b + m.Zf);
  F.Zpart = reinterpret_cast<float*>(b + m.Zpart);
  F.Yp = reinterpret_cast<float*>(b + m.Yp);
  F.diag = reinterpret_cast<unsigned long long*>(b + m.diag);
  F.ctr = h->d_ctr;
  F.launches = h->d_launches;
  F.timeout = h->timeout;
  return F;
}

// decode path for any T, in passes of <= 16 tokens
StagePlan stage_plan(const lmoe_handle* h, const int32_t* idx, int n, int must, int2* copies);

// the LoRA branch's tickets (after the multi-kernel path's) and partial sums
unsigned* lora_tickets(const lmoe_handle* h) { return h->d_tickets + 1 + (h->cfg.d + 63) / 64; }
float* lora_ppart(const lmoe_handle* h, void* ws) {
  return reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + decode_ws(h->cfg, 0, h->num_sms).Lpart);
}
float* lora_qpart(const lmoe_handle* h, void* ws) {
  return reinterpret_cast<float*>(reinterpret_cast<char*>(lora_ppart(h, ws)) +
                                  lora_ppart_bytes(h->cfg.d, h->cfg.G, h->cfg.lora_rank));
}

lmoe_status decode_layer(lmoe_handle* h, const uint16_t* x, int T, const uint16_t* residual, uint16_t* y, void* ws,
                         cudaStream_t st) {
  const lmoe_config& c = h->cfg;
  EventHook hook;
  hook.ev = h->events.empty() ? nullptr : &h->events;
  for (int t0 = 0; t0 < T; t0 += kMaxDecodeT) {
    DecodeArgs A = base_args(h, ws);
    A.T = T - t0 < kMaxDecodeT ? T - t0 : kMaxDecodeT;
    A.x = x + (size_t)t0 * c.d;
    A.residual = residual ? residual + (size_t)t0 * c.d : nullptr;
    A.y = y + (size_t)t0 * c.d;
    if (use_fused(h, A)) {
      FusedArgs F = fused_args(h, A, ws);
      cudaError_t e;
      if (h->staged) {  // route, then bring every routed expert without a slot into one
        hook.before(st);
        e = launch_route(A, 0, ws_logits(h, ws), st);
        hook.after(st);
        if (e != cudaSuccess) return LMOE_ERR_CUDA;
        const StagePlan P = stage_plan(h, A.idx, A.T * c.k, 1, h->d_copies);
        hook.before(st);
        e = launch_stage_plan(P, st);
        hook.after(st);
        if (e != cudaSuccess) return LMOE_ERR_CUDA;
        hook.before(st);
        e = launch_stage_copy(P, h->d_lib, h->d_slots, h->num_sms, st);
        hook.after(st);
        if (e != cudaSuccess) return LMOE_ERR_CUDA;
        F.slot_of = h->d_slot_of;
      }
      // the LoRA kernels and the single kernel chained by programmatic
      // dependent launch, unless stage events go between them
      const bool pdl = A.r > 0 && h->events.empty();
      if (A.r > 0) {  // the LoRA branch: lora_in before, lora_q and lora_out after
        // scratch of the multi-kernel sequence, unused by the single kernel:
        // P in Pin, Hl in V, Z in fp32 in Z, Q in Qout; the partials in Lpart
        F.hl = A.V;
        F.zlin = A.Z;
        F.no_combine = 1;
        F.pdl_hl = pdl ? 1 : 0;
        e = launch_lora_in(A, lora_ppart(h, ws), A.Pin, A.V, lora_tickets(h), st, &hook, pdl);
        if (e != cudaSuccess) return LMOE_ERR_CUDA;
      }
      hook.before(st);
      e = launch_decode_fused(F, h->fused_grid, st, pdl ? 1 : 0);
      hook.after(st);
      if (e != cudaSuccess) return LMOE_ERR_CUDA;
      if (A.r > 0) {
        hook.before(st);
        e = launch_lora_q(A, A.Z, lora_qpart(h, ws), A.Qout, lora_tickets(h), st, pdl);
        hook.after(st);
        if (e != cudaSuccess) return LMOE_ERR_CUDA;
        hook.before(st);
        e = launch_lora_out(A, F.Yp, A.Qout, lora_tickets(h), st, pdl);
        hook.after(st);
        if (e != cudaSuccess) return LMOE_ERR_CUDA;
      }
      continue;
    }
    if (A.wfmt != LMOE_WEIGHTS_INT4) return LMOE_ERR_UNSUPPORTED;  // the per-step kernels read int4 only
    hook.before(st);
    cudaError_t e = launch_route(A, 1, ws_logits(h, ws), st);
    hook.after(st);
    if (e != cudaSuccess) return LMOE_ERR_CUDA;
    if (A.r > 0) {
      hook.before(st);
      e = launch_lora_proj(A, 0, st);
      hook.after(st);
      if (e != cudaSuccess) return LMOE_ERR_CUDA;
    }
    e = launch_experts(A, 0, st, &hook);
    if (e != cudaSuccess) return LMOE_ERR_CUDA;
  }
  return LMOE_OK;
}

// The staged-expert state of a new handle: every expert's unit chunks are
// built once in GPU memory (from the caller's pointers, which may address
// host memory), moved into a page-locked host library, and the handle keeps
// expert_slots slots in GPU memory with empty tables.
lmoe_status create_stage(lmoe_handle* h, const DecodeArgs& probe) {
  const lmoe_config& c = h->cfg;
  h->staged = true;
  h->expert_bytes = decode_expert_bytes(c.L, c.f);
  const size_t lib_bytes = (size_t)c.E * h->expert_bytes;
  uint8_t* tmp = nullptr;
  if (cudaMalloc(&tmp, lib_bytes) != cudaSuccess) {
    cudaGetLastError();
    return LMOE_ERR_NO_MEMORY;
  }
  lmoe_status s = LMOE_OK;
  if (launch_decode_pack(probe, h->d_pack, &h->pk, 0, tmp) != cudaSuccess) s = LMOE_ERR_CUDA;
  if (s == LMOE_OK && cudaHostAlloc(&h->h_lib, lib_bytes, cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess) {
    h->h_lib = nullptr;
    s = LMOE_ERR_NO_MEMORY;
  }
  if (s == LMOE_OK && cudaMemcpy(h->h_lib, tmp, lib_bytes, cudaMemcpyDeviceToHost) != cudaSuccess) s = LMOE_ERR_CUDA;
  cudaFree(tmp);
  void* dl = nullptr;
  if (s == LMOE_OK && cudaHostGetDevicePointer(&dl, h->h_lib, 0) != cudaSuccess) s = LMOE_ERR_CUDA;
  if (s != LMOE_OK) {
    cudaGetLastError();
    return s;
  }
  h->d_lib = static_cast<const uint8_t*>(dl);
  const int S = c.expert_slots;
  if (cudaMalloc(&h->d_slots, (size_t)S * h->expert_bytes) != cudaSuccess ||
      cudaMalloc(&h->d_slot_of, (size_t)c.E * 4) != cudaSuccess ||
      cudaMalloc(&h->d_expert_in, (size_t)S * 4) != cudaSuccess ||
      cudaMalloc(&h->d_stage, sizeof(StageState)) != cudaSuccess ||
      cudaMalloc(&h->d_copies, 256 * sizeof(int2)) != cudaSuccess ||
      cudaMalloc(&h->d_pre_copies, 256 * sizeof(int2)) != cudaSuccess ||
      cudaMalloc(&h->d_pre_logits, (size_t)kMaxDecodeT * c.E * 4) != cudaSuccess ||
      cudaMalloc(&h->d_pre_idx, (size_t)kMaxDecodeT * c.k * 4) != cudaSuccess ||
      cudaMalloc(&h->d_pre_w, (size_t)kMaxDecodeT * c.k * 4) != cudaSuccess ||
      cudaMalloc(&h->d_pre_tickets, 64) != cudaSuccess) {
    cudaGetLastError();
    return LMOE_ERR_NO_MEMORY;
  }
  cudaMemset(h->d_slot_of, 0xff, (size_t)c.E * 4);
  cudaMemset(h->d_expert_in, 0xff, (size_t)S * 4);
  cudaMemset(h->d_stage, 0, sizeof(StageState));
  cudaMemset(h->d_pre_tickets, 0, 64);
  if (cudaEventCreateWithFlags(&h->ev_pf_in, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&h->ev_pf_done, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    return LMOE_ERR_CUDA;
  }
  h->pk.unit = h->d_slots;
  return LMOE_OK;
}

StagePlan stage_plan(const lmoe_handle* h, const int32_t* idx, int n, int must, int2* copies);
lmoe_status prefetch_on(lmoe_handle* h, const uint16_t* x, int T, cudaStream_t st);

StagePlan stage_plan(const lmoe_handle* h, const int32_t* idx, int n, int must, int2* copies) {
  StagePlan P;
  P.idx = idx;
  P.n = n;
  P.E = h->cfg.E;
  P.S = h->cfg.expert_slots;
  P.must = must;
  P.slot_of = h->d_slot_of;
  P.expert_in = h->d_expert_in;
  P.st = h->d_stage;
  P.copies = copies;
  P.expert_bytes = h->expert_bytes;
  P.err = h->d_err;
  return P;
}

// The prerouter of a staged handle: h's router on x (the tokens' input one
// layer early), top-k into the handle's own scratch, then the staging of
// those experts (as a prefetch).
lmoe_status prefetch_on(lmoe_handle* h, const uint16_t* x, int T, cudaStream_t st) {
  DecodeArgs A = base_args(h, nullptr);
  A.T = T;
  A.x = x;
  A.idx = h->d_pre_idx;
  A.w = h->d_pre_w;
  A.tickets = h->d_pre_tickets;
  if (launch_route(A, 0, h->d_pre_logits, st) != cudaSuccess) return LMOE_ERR_CUDA;
  const StagePlan P = stage_plan(h, h->d_pre_idx, T * h->cfg.k, 0, h->d_pre_copies);
  if (launch_stage_plan(P, st) != cudaSuccess) return LMOE_ERR_CUDA;
  if (launch_stage_copy(P, h->d_lib, h->d_slots, h->num_sms, st) != cudaSuccess) return LMOE_ERR_CUDA;
  return LMOE_OK;
}

PrefillArgs prefill_args(const lmoe_handle* h) {
  PrefillArgs P;
  memset(&P, 0, sizeof(P));
  const lmoe_config& c = h->cfg;
  P.d = c.d; P.E = c.E; P.G = c.G; P.k = c.k; P.L = c.L; P.f = c.f; P.r = c.lora_rank;
  P.epg = c.E / c.G;
  P.W_r = h->w.W_r; P.b_r = c.has_bias ? h->w.b_r : nullptr;
  P.W_r_split = h->d_wr_split;
  P.W_in_q = h->w.W_in_q; P.W_in_s = h->w.W_in_s; P.W_out_q = h->w.W_out_q; P.W_out_s = h->w.W_out_s;
  P.gate_q = h->w.gate_q; P.gate_s = h->w.gate_s; P.up_q = h->w.up_q; P.up_s = h->w.up_s;
  P.down_q = h->w.down_q; P.down_s = h->w.down_s;
  P.A_in = h->w.A_in; P.B_in = h->w.B_in; P.A_out = h->w.A_out; P.B_out = h->w.B_out;
  P.wfmt = c.weight_format;
  P.W_in_gs = h->w.W_in_gs; P.W_out_gs = h->w.W_out_gs;
  P.gate_gs = h->w.gate_gs; P.up_gs = h->w.up_gs; P.down_gs = h->w.down_gs;
  P.err = h->d_err;
  P.num_sms = h->num_sms;
  P.timeout = h->timeout;
  P.aux = h->aux;
  P.ev_fork = h->ev_fork;
  P.ev_join = h->ev_join;
  return P;
}

// Scratch of lmoe_layer_forward_noalloc, looked up once per device and
// primary context: the address is cached together with the context it
// belongs to, so a context made anew (after cudaDeviceReset) is looked up
// again instead of being handed a stale address.
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};
unsigned long long g_noalloc_ctx[kNoAllocMaxDevices] = {};

typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// Identifier of the current context (0 if the driver cannot say).
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_cur = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static bool looked = false;
  if (!looked) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
    cudaGetLastError();
    looked = true;
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_cur || get_cur(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (!get_id || get_id(ctx, &id) != CUDA_SUCCESS) return (unsigned long long)(uintptr_t)ctx;
  return id + 1;  // never 0
}

}  // namespace

// One fixed scratch array per device, in this library's device image: the
// workspace of lmoe_layer_forward_noalloc, which therefore allocates nothing.
static __device__ __align__(256) unsigned char lmoe_noalloc_scratch[LMOE_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of the scratch array on `device`, which must be current.
lmoe_status noalloc_scratch(int device, void** out) {
  if (device < 0 || device >= kNoAllocMaxDevices) return LMOE_ERR_UNSUPPORTED;
  // the runtime makes the primary context on first use; this call only looks
  // it up (cudaFree(0) would be the usual way to force it, but this entry
  // point calls no allocation routine at all)
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[device] || g_noalloc_ctx[device] != ctx || ctx == 0) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, lmoe_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return LMOE_ERR_CUDA;
    }
    g_noalloc_ptr[device] = p;
    g_noalloc_ctx[device] = current_context_id();
  }
  *out = g_noalloc_ptr[device];
  return LMOE_OK;
}

}  // namespace

extern "C" {

const char* lmoe_status_string(lmoe_status s) {
  switch (s) {
    case LMOE_OK: return "ok";
    case LMOE_ERR_INVALID_ARG: return "invalid argument";
    case LMOE_ERR_UNSUPPORTED: return "unsupported shape or option";
    case LMOE_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case LMOE_ERR_CUDA: return "CUDA error";
    case LMOE_ERR_TIMEOUT: return "device wait timed out";
    case LMOE_ERR_DEVICE_CHECK: return "device-side check failed (invalid data)";
    case LMOE_ERR_NO_MEMORY: return "out of device memory";
  }
  return "unknown status";
}

int lmoe_version(void) { return 101; }

lmoe_status lmoe_create(lmoe_handle** out, const lmoe_config* cfg, const lmoe_weights* w, int device) {
  if (!out) return LMOE_ERR_INVALID_ARG;
  *out = nullptr;
  lmoe_status s = validate_config(cfg);
  if (s != LMOE_OK) return s;
  s = validate_weights(cfg, w);
  if (s != LMOE_OK) return s;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) {
    cudaGetLastError();
    return device < 0 ? LMOE_ERR_INVALID_ARG : LMOE_ERR_CUDA;
  }
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return LMOE_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return LMOE_ERR_UNSUPPORTED;  // built for sm_103a only
  DeviceGuard guard(device);
  lmoe_handle* h = new (std::nothrow) lmoe_handle();
  if (!h) return LMOE_ERR_NO_MEMORY;
  h->cfg = *cfg;
  h->w = *w;
  h->device = device;
  h->num_sms = prop.multiProcessorCount;
  h->timeout = cfg->timeout_cycles ? cfg->timeout_cycles : (1ll << 31);
  const size_t nt = ticket_map(*cfg).total;
  if (cudaMalloc(&h->d_err, sizeof(unsigned)) != cudaSuccess ||
      cudaMalloc(&h->d_tickets, nt * sizeof(unsigned)) != cudaSuccess) {
    cudaGetLastError();
    lmoe_destroy(h);
    return LMOE_ERR_NO_MEMORY;
  }
  cudaMemset(h->d_err, 0, sizeof(unsigned));
  cudaMemset(h->d_tickets, 0, nt * sizeof(unsigned));
  if (cudaMalloc(&h->d_wr_split, (size_t)3 * cfg->E * cfg->d * 2) != cudaSuccess) {
    cudaGetLastError();
    lmoe_destroy(h);
    return LMOE_ERR_NO_MEMORY;
  }
  if (decode_set_attributes() != cudaSuccess || permute_set_attributes() != cudaSuccess ||
      lora_set_attributes() != cudaSuccess ||
      fused_set_attributes() != cudaSuccess || prefill_set_attributes() != cudaSuccess) {
    lmoe_destroy(h);
    return LMOE_ERR_CUDA;
  }
  h->fused_grid = fused_grid(h->num_sms);
  {
    const size_t nc = fused_counter_words(cfg->d, cfg->E, cfg->G, cfg->L);
    if (cudaMalloc(&h->d_ctr, nc * sizeof(unsigned)) != cudaSuccess ||
        cudaMalloc(&h->d_launches, sizeof(unsigned long long)) != cudaSuccess) {
      cudaGetLastError();
      lmoe_destroy(h);
      return LMOE_ERR_NO_MEMORY;
    }
    cudaMemset(h->d_ctr, 0, nc * sizeof(unsigned));
    cudaMemset(h->d_launches, 0, sizeof(unsigned long long));
    DecodeArgs probe = base_args(h, nullptr);
    probe.T = 1;
    h->pack_ok = false;
    if (h->fused_grid > 0 && fused_decode_supported(probe, h->fused_grid)) {
      const bool staged = (cfg->flags & LMOE_FLAG_STAGED_EXPERTS) != 0;
      const size_t pb = staged ? decode_pack_bytes_shared(cfg->d, cfg->E, cfg->G, cfg->L, cfg->f)
                               : decode_pack_bytes(cfg->d, cfg->E, cfg->G, cfg->L, cfg->f);
      if (cudaMalloc(&h->d_pack, pb) != cudaSuccess) {
        cudaGetLastError();
        lmoe_destroy(h);
        return LMOE_ERR_NO_MEMORY;
      }
      if (staged) {
        lmoe_status ss = create_stage(h, probe);
        if (ss != LMOE_OK) {
          lmoe_destroy(h);
          return ss;
        }
      } else if (launch_decode_pack(probe, h->d_pack, &h->pk, 0) != cudaSuccess) {
        lmoe_destroy(h);
        return LMOE_ERR_CUDA;
      }
      h->pack_ok = true;
    }
  }
  if (cudaStreamCreateWithFlags(&h->aux, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    lmoe_destroy(h);
    return LMOE_ERR_CUDA;
  }
  if (launch_split_router(h->w.W_r, cfg->E, cfg->d, h->d_wr_split, 0) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    lmoe_destroy(h);
    return LMOE_ERR_CUDA;
  }
  *out = h;
  return LMOE_OK;
}

lmoe_status lmoe_destroy(lmoe_handle* h) {
  if (!h) return LMOE_OK;
  DeviceGuard guard(h->device);
  cudaDeviceSynchronize();
  if (h->hg.exec) cudaGraphExecDestroy(h->hg.exec);
  if (h->cap) cudaStreamDestroy(h->cap);
  if (h->cin) cudaStreamDestroy(h->cin);
  if (h->cout) cudaStreamDestroy(h->cout);
  for (cudaEvent_t e : h->hev) cudaEventDestroy(e);
  if (h->d_err) cudaFree(h->d_err);
  if (h->d_tickets) cudaFree(h->d_tickets);
  if (h->d_wr_split) cudaFree(h->d_wr_split);
  if (h->d_ctr) cudaFree(h->d_ctr);
  if (h->d_launches) cudaFree(h->d_launches);
  if (h->d_pack) cudaFree(h->d_pack);
  if (h->h_lib) cudaFreeHost(h->h_lib);
  void* stage_bufs[] = {h->d_slots, h->d_slot_of, h->d_expert_in, h->d_stage, h->d_copies, h->d_pre_copies,
                        h->d_pre_logits, h->d_pre_idx, h->d_pre_w, h->d_pre_tickets};
  for (void* p : stage_bufs)
    if (p) cudaFree(p);
  if (h->ev_pf_in) cudaEventDestroy(h->ev_pf_in);
  if (h->ev_pf_done) cudaEventDestroy(h->ev_pf_done);
  if (h->ev_fork) cudaEventDestroy(h->ev_fork);
  if (h->ev_join) cudaEventDestroy(h->ev_join);
  if (h->aux) cudaStreamDestroy(h->aux);
  delete h;
  return pending_error();
}

size_t lmoe_workspace_size(const lmoe_handle* h, int T) {
  if (!h || T < 0) return 0;
  size_t a = decode_ws(h->cfg, T, h->num_sms).end;
  size_t b = prefill_workspace_bytes(prefill_args(h), T);
  return a > b ? a : b;
}

size_t lmoe_host_staging_size(const lmoe_handle* h, int T) {
  if (!h || T < 0) return 0;
  return 3 * align_up((size_t)T * h->cfg.d * 2);
}

lmoe_status lmoe_route(lmoe_handle* h, const uint16_t* x, int T, int32_t* idx, float* w, float* logits, void* ws,
                       lmoe_stream stream) {
  if (check_handle(h) != LMOE_OK || T < 0) return LMOE_ERR_INVALID_ARG;
  if (T == 0) return LMOE_OK;
  if (!x || !idx || !w || !ws) return LMOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(ws)) return LMOE_ERR_ALIGNMENT;
  lmoe_status s = pending_error();
  if (s != LMOE_OK) return s;
  DeviceGuard guard(h->device);
  cudaStream_t st = (cudaStream_t)stream;
  const lmoe_config& c = h->cfg;
  if (use_prefill(h, T)) {
    PrefillArgs P = prefill_args(h);
    return cuda_status(launch_prefill_route(P, x, T, idx, w, logits, ws, st));
  }
  for (int t0 = 0; t0 < T; t0 += kMaxDecodeT) {
    DecodeArgs A = base_args(h, ws);
    A.T = T - t0 < kMaxDecodeT ? T - t0 : kMaxDecodeT;
    A.x = x + (size_t)t0 * c.d;
    A.idx = idx + (size_t)t0 * c.k;
    A.w = w + (size_t)t0 * c.k;
    float* lg = logits ? logits + (size_t)t0 * c.E : ws_logits(h, ws);
    if (launch_route(A, 0, lg, st) != cudaSuccess) return LMOE_ERR_CUDA;
  }
  return LMOE_OK;
}

static lmoe_status check_perm(const lmoe_perm* p) {
  if (!p || !p->expert_offsets || !p->sorted_assign || !p->inv || !p->group_offsets || !p->group_tok_offsets ||
      !p->group_tokens || !p->assign_row)
    return LMOE_ERR_INVALID_ARG;
  return LMOE_OK;
}

static PermPtrs to_ptrs(const lmoe_perm* p) {
  PermPtrs q;
  q.expert_offsets = p->expert_offsets; q.sorted_assign = p->sorted_assign; q.inv = p->inv;
  q.group_offsets = p->group_offsets; q.group_tok_offsets = p->group_tok_offsets;
  q.group_tokens = p->group_tokens; q.assign_row = p->assign_row;
  return q;
}

lmoe_status lmoe_permute(lmoe_handle* h, const int32_t* idx, int T, const lmoe_perm* out, void* ws,
                         lmoe_stream stream) {
  if (check_handle(h) != LMOE_OK || T < 0) return LMOE_ERR_INVALID_ARG;
  if (check_perm(out) != LMOE_OK || !ws || (T > 0 && !idx)) return LMOE_ERR_INVALID_ARG;
  if (!aligned16(ws)) return LMOE_ERR_ALIGNMENT;
  lmoe_status s = pending_error();
  if (s != LMOE_OK) return s;
  DeviceGuard guard(h->device);
  const DecodeWs m = decode_ws(h->cfg, T, h->num_sms);
  void* scratch = reinterpret_cast<char*>(ws) + m.perm_scratch;
  return cuda_status(launch_permute(idx, T, h->cfg.E, h->cfg.G, h->cfg.k, to_ptrs(out), scratch, h->d_err,
                                    (cudaStream_t)stream));
}

lmoe_status lmoe_expert_forward(lmoe_handle* h, const uint16_t* x, int T, const int32_t* idx, const float* w,
                                const lmoe_perm* perm, float* Y, void* ws, lmoe_stream stream) {
  if (check_handle(h) != LMOE_OK || T < 0) return LMOE_ERR_INVALID_ARG;
  if (T == 0) return LMOE_OK;
  if (!x || !idx || !w || !Y || !ws || check_perm(perm) != LMOE_OK) return LMOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Y) || !aligned16(ws)) return LMOE_ERR_ALIGNMENT;
  lmoe_status s = pending_error();
  if (s != LMOE_OK) return s;
  DeviceGuard guard(h->device);
  cudaStream_t st = (cudaStream_t)stream;
  const lmoe_config& c = h->cfg;
  if (use_prefill(h, T) || (c.weight_format != LMOE_WEIGHTS_INT4 && prefill_supported(prefill_args(h)))) {
    // (NVFP4 weights: the per-step decode kernels read int4 only, so every T takes the grouped GEMMs)
    PrefillArgs P = prefill_args(h);
    return cuda_status(launch_prefill_experts(P, x, T, idx, w, to_ptrs(perm), Y, nullptr, nullptr, ws, st));
  }
  if (c.weight_format != LMOE_WEIGHTS_INT4) return LMOE_ERR_UNSUPPORTED;
  const DecodeWs m = decode_ws(c, T, h->num_sms);
  for (int t0 = 0; t0 < T; t0 += kMaxDecodeT) {
    DecodeArgs A = base_args(h, ws);
    A.T = T - t0 < kMaxDecodeT ? T - t0 : kMaxDecodeT;
    A.x = x + (size_t)t0 * c.d;
    // this pass's routing (caller's) and its own local permutation
    A.idx = const_cast<int32_t*>(idx) + (size_t)t0 * c.k;
    A.w = const_cast<float*>(w) + (size_t)t0 * c.k;
    void* scratch = reinterpret_cast<char*>(ws) + m.perm_scratch;
    if (launch_permute(A.idx, A.T, c.E, c.G, c.k, A.pm, scratch, h->d_err, st) != cudaSuccess) return LMOE_ERR_CUDA;
    if (A.r > 0 && launch_lora_proj(A, 0, st) != cudaSuccess) return LMOE_ERR_CUDA;
    A.tok0 = t0;
    A.idx_all = idx;
    A.assign_row_all = perm->assign_row;
    A.Yrows = Y;
    if (launch_experts(A, 1, st, nullptr) != cudaSuccess) return LMOE_ERR_CUDA;
  }
  return LMOE_OK;
}

lmoe_status lmoe_combine(lmoe_handle* h, const float* Y, const int32_t* idx, const lmoe_perm* perm, int T,
                         const uint16_t* residual, uint16_t* y, lmoe_stream stream) {
  if (check_handle(h) != LMOE_OK || T < 0) return LMOE_ERR_INVALID_ARG;
  if (T == 0) return LMOE_OK;
  if (!Y || !idx || !y || check_perm(perm) != LMOE_OK) return LMOE_ERR_INVALID_ARG;
  if (!aligned16(Y) || !aligned16(y) || (residual && !aligned16(residual))) return LMOE_ERR_ALIGNMENT;
  lmoe_status s = pending_error();
  if (s != LMOE_OK) return s;
  DeviceGuard guard(h->device);
  const lmoe_config& c = h->cfg;
  return cuda_status(launch_combine(Y, idx, perm->assign_row, T, c.d, c.k, c.E / c.G, residual, y,
                                    (cudaStream_t)stream));
}

lmoe_status lmoe_layer_forward(lmoe_handle* h, const uint16_t* x, int T, const uint16_t* residual, uint16_t* y,
                               void* ws, lmoe_stream stream) {
  if (check_handle(h) != LMOE_OK || T < 0) return LMOE_ERR_INVALID_ARG;
  if (T == 0) return LMOE_OK;
  if (!x || !y || !ws) return LMOE_ERR_INVALID_ARG;
  if (x == y) return LMOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || !aligned16(ws) || (residual && !aligned16(residual)))
    return LMOE_ERR_ALIGNMENT;
  lmoe_status s = pending_error();
  if (s != LMOE_OK) return s;
  DeviceGuard guard(h->device);
  cudaStream_t st = (cudaStream_t)stream;
  if (use_prefill(h, T)) {
    PrefillArgs P = prefill_args(h);
    return cuda_status(launch_prefill_layer(P, x, T, residual, y, ws, st, h->events.empty() ? nullptr : &h->events));
  }
  return decode_layer(h, x, T, residual, y, ws, st);
}

lmoe_status lmoe_layer_forward_noalloc(lmoe_handle* h, const uint16_t* x, int T, const uint16_t* residual,
                                       uint16_t* y, lmoe_stream stream) {
  if (check_handle(h) != LMOE_OK || T < 0 || T > LMOE_NOALLOC_MAX_T) return LMOE_ERR_INVALID_ARG;
  if (T == 0) return LMOE_OK;
  if (!x || !y || x == y) return LMOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || (residual && !aligned16(residual))) return LMOE_ERR_ALIGNMENT;
  if (decode_ws(h->cfg, T, h->num_sms).end > (size_t)LMOE_NOALLOC_SCRATCH_BYTES) return LMOE_ERR_UNSUPPORTED;
  lmoe_status s = pending_error();
  if (s != LMOE_OK) return s;
  DeviceGuard guard(h->device);
  void* ws = nullptr;
  s = noalloc_scratch(h->device, &ws);
  if (s != LMOE_OK) return s;
  return decode_layer(h, x, T, residual, y, ws, (cudaStream_t)stream);
}

lmoe_status lmoe_decode_routing(lmoe_handle* h, const void* ws, int T, int32_t* idx, float* w, float* logits,
                                lmoe_stream stream) {
  if (check_handle(h) != LMOE_OK || T < 0 || T > kMaxDecodeT) return LMOE_ERR_INVALID_ARG;
  if (T == 0) return LMOE_OK;
  if (!ws || !idx || !w) return LMOE_ERR_INVALID_ARG;
  if (!aligned16(ws)) return LMOE_ERR_ALIGNMENT;
  lmoe_status s = pending_error();
  if (s != LMOE_OK) return s;
  DeviceGuard guard(h->device);
  cudaStream_t st = (cudaStream_t)stream;
  const lmoe_config& c = h->cfg;
  const DecodeWs m = decode_ws(c, 0, h->num_sms);
  const char* b = reinterpret_cast<const char*>(ws);
  if (cudaMemcpyAsync(idx, b + m.idx, (size_t)T * c.k * 4, cudaMemcpyDeviceToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(w, b + m.w, (size_t)T * c.k * 4, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return LMOE_ERR_CUDA;
  if (logits && cudaMemcpyAsync(logits, b + m.logits, (size_t)T * c.E * 4, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return LMOE_ERR_CUDA;
  return LMOE_OK;
}

size_t lmoe_stack_workspace_size(const lmoe_handle* h, int T) {
  if (!h || T < 0) return 0;
  return align_up(lmoe_workspace_size(h, T)) + 2 * align_up((size_t)T * h->cfg.d * 2);
}

lmoe_status lmoe_stack_forward(lmoe_handle* const* layers, int n_layers, const uint16_t* x, int T, uint16_t* y,
                               void* ws, lmoe_stream stream) {
  if (!layers || n_layers < 1 || T < 0 || !x || !y || !ws) return LMOE_ERR_INVALID_ARG;
  const lmoe_handle* h0 = layers[0];
  if (!h0) return LMOE_ERR_INVALID_ARG;
  const lmoe_config& c0 = h0->cfg;
  for (int l = 1; l < n_layers; ++l) {
    const lmoe_handle* h = layers[l];
    if (!h || h->device != h0->device) return LMOE_ERR_INVALID_ARG;
    const lmoe_config& c = h->cfg;
    if (c.d != c0.d || c.E != c0.E || c.G != c0.G || c.k != c0.k || c.L != c0.L || c.f != c0.f ||
        c.lora_rank != c0.lora_rank)
      return LMOE_ERR_INVALID_ARG;
  }
  if (T == 0) return LMOE_OK;
  if (!aligned16(x) || !aligned16(y) || !aligned16(ws)) return LMOE_ERR_ALIGNMENT;
  if (c0.d % 8 != 0) return LMOE_ERR_UNSUPPORTED;
  size_t need = 0;
  for (int l = 0; l < n_layers; ++l) {
    const size_t n = lmoe_workspace_size(layers[l], T);
    need = n > need ? n : need;
  }
  const size_t act = align_up((size_t)T * c0.d * 2);
  char* b = reinterpret_cast<char*>(ws) + align_up(need);
  uint16_t* ybuf = reinterpret_cast<uint16_t*>(b);
  uint16_t* xbuf = reinterpret_cast<uint16_t*>(b + act);
  DeviceGuard guard(h0->device);
  cudaStream_t st = (cudaStream_t)stream;
  const size_t n = (size_t)T * c0.d;
  const uint16_t* xin = x;
  // Decode-sized batches on the single-kernel path: one launch per layer (the
  // residual rule is applied in the kernel's final combine), each layer a
  // programmatic dependent of the one before it (its weight stream starts
  // while the previous layer finishes), and each prefetching the next layer's
  // router rows and W_in tiles into L2 during its own tail.
  bool fused_all = T <= kMaxDecodeT && c0.lora_rank == 0;
  for (int l = 0; fused_all && l < n_layers; ++l) fused_all = !layers[l]->staged;
  for (int l = 0; fused_all && l < n_layers; ++l) {
    DecodeArgs A = base_args(layers[l], ws);
    A.T = T;
    fused_all = !use_prefill(layers[l], T) && use_fused(layers[l], A);
  }
  if (fused_all) {
    lmoe_status s = pending_error();
    if (s != LMOE_OK) return s;
    for (int l = 0; l < n_layers; ++l) {
      lmoe_handle* h = layers[l];
      uint16_t* xout = l == n_layers - 1 ? y : (l % 2 == 0 ? xbuf : ybuf);
      DecodeArgs A = base_args(h, ws);
      A.T = T;
      A.x = xin;
      A.residual = xin;
      A.y = xout;
      FusedArgs F = fused_args(h, A, ws);
      F.round_first = 1;
      F.pdl = l > 0 && layers[l - 1] != h;  // distinct handles: distinct counters
      if (l + 1 < n_layers && layers[l + 1] != h) {
        F.has_next = 1;
        F.next_wr = layers[l + 1]->pk.wr;
        F.next_win = layers[l + 1]->pk.win;
      }
      EventHook hook;
      hook.ev = h->events.empty() ? nullptr : &h->events;
      hook.before(st);
      const cudaError_t e = launch_decode_fused(F, h->fused_grid, st, F.pdl);
      hook.after(st);
      if (e != cudaSuccess) return LMOE_ERR_CUDA;
      xin = xout;
    }
    return LMOE_OK;
  }
  for (int l = 0; l < n_layers; ++l) {
    // staged experts: the next layer's prerouter on the second stream, given
    // this layer's input, while this layer runs
    lmoe_handle* nx = l + 1 < n_layers ? layers[l + 1] : nullptr;
    const bool pf = nx && nx->staged && T <= kMaxDecodeT && !use_prefill(nx, T);
    if (pf) {
      if (cudaEventRecord(nx->ev_pf_in, st) != cudaSuccess || cudaStreamWaitEvent(nx->aux, nx->ev_pf_in, 0) != cudaSuccess)
        return LMOE_ERR_CUDA;
      lmoe_status ps = prefetch_on(nx, xin, T, nx->aux);
      if (ps != LMOE_OK) return ps;
      if (cudaEventRecord(nx->ev_pf_done, nx->aux) != cudaSuccess) return LMOE_ERR_CUDA;
    }
    lmoe_status s = lmoe_layer_forward(layers[l], xin, T, nullptr, ybuf, ws, stream);
    if (s != LMOE_OK) return s;
    uint16_t* xout = l == n_layers - 1 ? y : xbuf;
    // (the prerouter reads xin, which the residual add may overwrite)
    if (pf && cudaStreamWaitEvent(st, nx->ev_pf_done, 0) != cudaSuccess) return LMOE_ERR_CUDA;
    if (launch_residual_add(xin, ybuf, n, xout, st) != cudaSuccess) return LMOE_ERR_CUDA;
    xin = xout;
  }
  return LMOE_OK;
}

namespace {
void drop_host_graph(lmoe_handle* h) {
  if (h->hg.exec) cudaGraphExecDestroy(h->hg.exec);
  h->hg = lmoe_handle::HostGraph{};
}

constexpr int kHostChunk = 4096;  // tokens per chunk of a prefill-sized host call
constexpr int kHostFirst = 1024;  // the first chunk: the compute starts after a short copy

// A prefill-sized host call as a pipeline of token chunks on three streams:
// the copy-in stream moves chunk i's x (and residual) while `st` computes
// chunk i - 1 and the copy-out stream returns chunk i - 2's y. The first
// chunk is short, so that the compute starts early; the rest are kHostChunk
// tokens (the last, what remains). The weights are dequantised once, into a
// workspace laid out for one full chunk; each chunk's tokens go through the
// layer exactly as in one call (every step of the layer is per token), and
// the chunks run one after another on `st`, so they share that workspace.
lmoe_status enqueue_host_chunked(lmoe_handle* h, const uint16_t* x_host, int T, const uint16_t* residual_host,
                                 uint16_t* y_host, void* ws, cudaStream_t st) {
  const int C = kHostChunk;
  // chunk i covers tokens [c0(i), c0(i) + cn(i))
  const int n = 1 + (T - kHostFirst + C - 1) / C;
  auto c0 = [&](int i) { return i == 0 ? 0 : kHostFirst + (i - 1) * C; };
  auto cn = [&](int i) { return (i == 0 ? kHostFirst : (T - c0(i) < C ? T - c0(i) : C)); };
  const size_t row = (size_t)h->cfg.d * 2, bytes = (size_t)T * row;
  char* stage = reinterpret_cast<char*>(ws) + align_up(lmoe_workspace_size(h, T));
  char* dx = stage;
  char* dr = stage + align_up(bytes);
  char* dy = stage + 2 * align_up(bytes);
  if (!h->cin && cudaStreamCreateWithFlags(&h->cin, cudaStreamNonBlocking) != cudaSuccess) return LMOE_ERR_CUDA;
  if (!h->cout && cudaStreamCreateWithFlags(&h->cout, cudaStreamNonBlocking) != cudaSuccess) return LMOE_ERR_CUDA;
  while ((int)h->hev.size() < 2 * n + 2) {
    cudaEvent_t e;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return LMOE_ERR_CUDA;
    h->hev.push_back(e);
  }
  cudaEvent_t* ev = h->hev.data();  // [0] start, [1] done, [2 + i] chunk i in, [2 + n + i] chunk i computed
  const PrefillArgs P = prefill_args(h);
  // the copies start after the caller's earlier work on st (which may still use the staging buffers)
  if (cudaEventRecord(ev[0], st) != cudaSuccess || cudaStreamWaitEvent(h->cin, ev[0], 0) != cudaSuccess ||
      cudaStreamWaitEvent(h->cout, ev[0], 0) != cudaSuccess)
    return LMOE_ERR_CUDA;
  for (int i = 0; i < n; ++i) {
    const size_t o = (size_t)c0(i) * row, nb = (size_t)cn(i) * row;
    if (cudaMemcpyAsync(dx + o, reinterpret_cast<const char*>(x_host) + o, nb, cudaMemcpyHostToDevice, h->cin) !=
            cudaSuccess ||
        (residual_host && cudaMemcpyAsync(dr + o, reinterpret_cast<const char*>(residual_host) + o, nb,
                                          cudaMemcpyHostToDevice, h->cin) != cudaSuccess) ||
        cudaEventRecord(ev[2 + i], h->cin) != cudaSuccess)
      return LMOE_ERR_CUDA;
  }
  if (launch_prefill_weights(P, C, ws, st) != cudaSuccess) return LMOE_ERR_CUDA;
  for (int i = 0; i < n; ++i) {
    const int Ti = cn(i);
    const size_t o = (size_t)c0(i) * row, nb = (size_t)Ti * row;
    if (cudaStreamWaitEvent(st, ev[2 + i], 0) != cudaSuccess) return LMOE_ERR_CUDA;
    if (launch_prefill_layer_chunk(P, reinterpret_cast<const uint16_t*>(dx + o), Ti, C,
                                   residual_host ? reinterpret_cast<const uint16_t*>(dr + o) : nullptr,
                                   reinterpret_cast<uint16_t*>(dy + o), ws, st) != cudaSuccess)
      return LMOE_ERR_CUDA;
    if (cudaEventRecord(ev[2 + n + i], st) != cudaSuccess || cudaStreamWaitEvent(h->cout, ev[2 + n + i], 0) != cudaSuccess ||
        cudaMemcpyAsync(reinterpret_cast<char*>(y_host) + o, dy + o, nb, cudaMemcpyDeviceToHost, h->cout) != cudaSuccess)
      return LMOE_ERR_CUDA;
  }
  if (cudaEventRecord(ev[1], h->cout) != cudaSuccess || cudaStreamWaitEvent(st, ev[1], 0) != cudaSuccess)
    return LMOE_ERR_CUDA;
  return LMOE_OK;
}

// the host-buffer call's work on `st`: copies in, the layer, the copy out
lmoe_status enqueue_host_call(lmoe_handle* h, const uint16_t* x_host, int T, const uint16_t* residual_host,
                              uint16_t* y_host, void* ws, cudaStream_t st) {
  if (use_prefill(h, T) && T >= 2 * kHostChunk && h->events.empty())
    return enqueue_host_chunked(h, x_host, T, residual_host, y_host, ws, st);
  const size_t bytes = (size_t)T * h->cfg.d * 2;
  char* stage = reinterpret_cast<char*>(ws) + align_up(lmoe_workspace_size(h, T));
  uint16_t* dx = reinterpret_cast<uint16_t*>(stage);
  uint16_t* dr = reinterpret_cast<uint16_t*>(stage + align_up(bytes));
  uint16_t* dy = reinterpret_cast<uint16_t*>(stage + 2 * align_up(bytes));
  if (cudaMemcpyAsync(dx, x_host, bytes, cudaMemcpyHostToDevice, st) != cudaSuccess) return LMOE_ERR_CUDA;
  if (residual_host && cudaMemcpyAsync(dr, residual_host, bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return LMOE_ERR_CUDA;
  const lmoe_status s = lmoe_layer_forward(h, dx, T, residual_host ? dr : nullptr, dy, ws, (lmoe_stream)st);
  if (s != LMOE_OK) return s;
  if (cudaMemcpyAsync(y_host, dy, bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess) return LMOE_ERR_CUDA;
  return LMOE_OK;
}
}  // namespace

lmoe_status lmoe_layer_forward_host(lmoe_handle* h, const uint16_t* x_host, int T, const uint16_t* residual_host,
                                    uint16_t* y_host, void* ws, lmoe_stream stream) {
  if (check_handle(h) != LMOE_OK || T < 0) return LMOE_ERR_INVALID_ARG;
  if (T == 0) return LMOE_OK;
  if (!x_host || !y_host || !ws) return LMOE_ERR_INVALID_ARG;
  if (!aligned16(ws)) return LMOE_ERR_ALIGNMENT;
  lmoe_status s = pending_error();
  if (s != LMOE_OK) return s;
  DeviceGuard guard(h->device);
  cudaStream_t st = (cudaStream_t)stream;
  // Repeated calls with the same buffers (a serving loop's staging buffers)
  // replay one CUDA graph of the copies and the layer instead of issuing
  // them one by one; every call still copies its inputs in and its output
  // out. Not for staged handles (their prefetch runs on its own stream), with
  // stage events set, or inside the caller's own stream capture.
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return LMOE_ERR_CUDA;
  const bool graph = !h->staged && h->events.empty() && cs == cudaStreamCaptureStatusNone;
  if (!graph) {
    s = enqueue_host_call(h, x_host, T, residual_host, y_host, ws, st);
    if (s != LMOE_OK) return s;
    return cuda_status(cudaStreamSynchronize(st));
  }
  lmoe_handle::HostGraph& g = h->hg;
  if (!(g.exec && g.x == x_host && g.r == residual_host && g.y == y_host && g.ws == ws && g.T == T)) {
    drop_host_graph(h);
    // capture on the handle's own stream (the caller's may be the legacy
    // default stream, which cannot be captured); it starts after the
    // caller's earlier work because the graph is launched on the caller's stream
    bool ok = h->cap || cudaStreamCreateWithFlags(&h->cap, cudaStreamNonBlocking) == cudaSuccess;
    ok = ok && cudaStreamBeginCapture(h->cap, cudaStreamCaptureModeThreadLocal) == cudaSuccess;
    if (ok) {
      s = enqueue_host_call(h, x_host, T, residual_host, y_host, ws, h->cap);
      cudaGraph_t cg = nullptr;
      const cudaError_t ec = cudaStreamEndCapture(h->cap, &cg);
      ok = s == LMOE_OK && ec == cudaSuccess && cg && cudaGraphInstantiate(&g.exec, cg, 0) == cudaSuccess;
      if (cg) cudaGraphDestroy(cg);
      if (s != LMOE_OK) {
        g.exec = nullptr;
        cudaGetLastError();
        return s;
      }
    }
    if (!ok) {  // not capturable here: issue the work directly
      g.exec = nullptr;
      cudaGetLastError();
      s = enqueue_host_call(h, x_host, T, residual_host, y_host, ws, st);
      if (s != LMOE_OK) return s;
      return cuda_status(cudaStreamSynchronize(st));
    }
    g.x = x_host; g.r = residual_host; g.y = y_host; g.ws = ws; g.T = T;
  }
  if (cudaGraphLaunch(g.exec, st) != cudaSuccess) {
    drop_host_graph(h);
    return LMOE_ERR_CUDA;
  }
  return cuda_status(cudaStreamSynchronize(st));
}

lmoe_status lmoe_check(lmoe_handle* h, lmoe_stream stream) {
  if (check_handle(h) != LMOE_OK) return LMOE_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return LMOE_ERR_CUDA;
  unsigned e = 0;
  if (cudaMemcpy(&e, h->d_err, sizeof(e), cudaMemcpyDeviceToHost) != cudaSuccess) return LMOE_ERR_CUDA;
  if (e && cudaMemset(h->d_err, 0, sizeof(unsigned)) != cudaSuccess) return LMOE_ERR_CUDA;
  if (e & ERRBIT_TIMEOUT) return LMOE_ERR_TIMEOUT;
  if (e) return LMOE_ERR_DEVICE_CHECK;
  return pending_error();
}

lmoe_status lmoe_set_timeout(lmoe_handle* h, long long cycles) {
  if (check_handle(h) != LMOE_OK || cycles < 0) return LMOE_ERR_INVALID_ARG;
  h->timeout = cycles ? cycles : (h->cfg.timeout_cycles ? h->cfg.timeout_cycles : (1ll << 31));
  drop_host_graph(h);  // the captured kernels carry the old budget
  return LMOE_OK;
}

lmoe_status lmoe_set_stage_events(lmoe_handle* h, void* const* events, int n) {
  if (check_handle(h) != LMOE_OK || n < 0 || (n > 0 && !events)) return LMOE_ERR_INVALID_ARG;
  h->events.clear();
  if (events)
    for (int i = 0; i < 2 * n; ++i) h->events.push_back((cudaEvent_t)events[i]);
  drop_host_graph(h);
  return LMOE_OK;
}

const char* lmoe_stage_name(const lmoe_handle* h, int T, int i, int* count) {
  static const char* dec[] = {"route", "win", "gateup", "down", "wout"};
  static const char* dec_lora[] = {"route", "lora_p", "win", "gateup", "down", "lora_q", "wout"};
  if (!h) {
    if (count) *count = 0;
    return "";
  }
  if (use_prefill(h, T)) return prefill_stage_name(prefill_args(h), T, i, count);
  const bool lora = h->cfg.lora_rank > 0;
  DecodeArgs probe = base_args(h, nullptr);
  probe.T = T < kMaxDecodeT ? T : kMaxDecodeT;
  if (T >= 1 && use_fused(h, probe)) {
    static const char* fl[] = {"lora_p", "lora_hl", "decode_fused", "lora_q", "lora_out"};
    static const char* stg[] = {"route", "stage_plan", "stage_copy"};
    const int ns = h->staged ? 3 : 0;
    const int passes = (T + kMaxDecodeT - 1) / kMaxDecodeT, per = ns + (lora ? 5 : 1);
    if (count) *count = per * passes;
    if (i < 0 || i >= per * passes) return "";
    const int j = i % per;
    if (j < ns) return stg[j];
    return lora ? fl[j - ns] : "decode_fused";
  }
  const int per = lora ? 7 : 5;
  const int passes = (T + kMaxDecodeT - 1) / kMaxDecodeT;
  if (count) *count = per * passes;
  if (i < 0 || i >= per * passes) return "";
  return lora ? dec_lora[i % per] : dec[i % per];
}

int lmoe_launch_count(const lmoe_handle* h, int T) {
  if (!h || T < 1) return 0;
  if (use_prefill(h, T)) return prefill_launch_count(prefill_args(h), T);
  int n = 0;
  lmoe_stage_name(h, T, 0, &n);  // decode: one kernel per stage
  return n;
}

lmoe_status lmoe_prefetch_experts(lmoe_handle* h, const uint16_t* x, int T, lmoe_stream stream) {
  if (check_handle(h) != LMOE_OK || !h->staged || T < 1 || T > kMaxDecodeT || !x) return LMOE_ERR_INVALID_ARG;
  if (!aligned16(x)) return LMOE_ERR_ALIGNMENT;
  lmoe_status s = pending_error();
  if (s != LMOE_OK) return s;
  DeviceGuard guard(h->device);
  return prefetch_on(h, x, T, (cudaStream_t)stream);
}

lmoe_status lmoe_get_stage_stats(lmoe_handle* h, lmoe_stage_stats* out) {
  if (check_handle(h) != LMOE_OK || !h->staged || !out) return LMOE_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  StageState st;
  if (cudaDeviceSynchronize() != cudaSuccess || cudaMemcpy(&st, h->d_stage, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess)
    return LMOE_ERR_CUDA;
  out->passes = st.passes;
  out->routed = st.routed;
  out->hits = st.hits;
  out->staged_on_demand = st.on_demand;
  out->prefetched = st.prefetched;
  out->bytes_copied = st.bytes;
  return LMOE_OK;
}

}  // extern "C"
