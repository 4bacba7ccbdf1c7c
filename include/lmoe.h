/*
 * lmoe -- the latent mixture-of-experts layer of Edge0-145B on NVIDIA B300
 * (sm_103a), behind a plain C ABI.
 *
 * The layer (sources, by page title and section):
 *  - "Edge0-145B: Frontier AI Capabilities on Your Own Computer", "Under the
 *    Hood of Edge0", paragraph "Architecture: share large matrices across
 *    sparse experts": groups of 64 experts share two large matrices, each
 *    expert keeps a small set of its own parameters.
 *  - "Edge0-145B: Run a 145B Open-Source Model on Your Laptop", "Not
 *    Compression -- Architecture": 512 experts, 10 active per token, 48
 *    layers; "The Three Pillars That Make It Fast": int4 expert tensors and a
 *    Recover-LoRA branch in parallel with the frozen 4-bit base.
 *
 * Concrete form (this library's stated assumption; the pages sketch it only):
 *   logits  l = x W_r^T (+ b)                               fp32 router
 *   top-k   the k largest l, descending, ties -> lower index; w = softmax over them
 *   group   g(e) = e / (E/G)
 *   h       = Win[g] x  (+ B_in[g]^T A_in[g]^T x)            Win: int4 [L][d]
 *   u_e     = Down_e( silu(Gate_e h) * Up_e h )               int4 [f][L], [f][L], [L][f]
 *   y       = sum_g Wout[g] sum_{j: g(e_j)=g} w_j u_{e_j}   (+ LoRA)  Wout: int4 [d][L]
 * int4: symmetric groups of 32 consecutive elements along the reduction
 * dimension, one bf16 scale per group; byte j of a row holds element 2j in
 * its low nibble and 2j+1 in its high nibble (two's complement, -7..7).
 *
 * Conventions for every entry point:
 *  - Pointers named x, y, idx, w, logits, Y, ws, residual and the weight
 *    pointers are DEVICE pointers on the handle's device, except in
 *    lmoe_layer_forward_host. bf16 tensors are passed as uint16_t bit
 *    patterns. All buffers are owned by the caller; the handle borrows the
 *    weight pointers for its lifetime (they must stay valid and unchanged).
 *  - Arrays read with 128-bit loads must be 16-byte aligned: x, y, residual,
 *    every weight pointer, Y and ws. Misalignment -> LMOE_ERR_ALIGNMENT.
 *  - Arguments are validated on the host before anything is launched; on an
 *    error nothing is enqueued. Work is enqueued on the given stream
 *    (NULL = legacy default stream) and the call returns without waiting.
 *    Errors raised by kernels are reported by the next call or by
 *    lmoe_check. No function throws across the ABI.
 *  - A handle is thread-compatible, not thread-safe: do not use one handle
 *    from two host threads at once. Calls enqueued on different streams with
 *    the same workspace race.
 */
#ifndef LMOE_H
#define LMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* lmoe_stream; /* == cudaStream_t */

typedef enum {
  LMOE_OK = 0,
  LMOE_ERR_INVALID_ARG = 1,   /* null pointer, bad size, bad handle */
  LMOE_ERR_UNSUPPORTED = 2,   /* a shape outside what the kernels support */
  LMOE_ERR_ALIGNMENT = 3,     /* a pointer not 16-byte aligned */
  LMOE_ERR_CUDA = 4,          /* a CUDA runtime error (launch or earlier async failure) */
  LMOE_ERR_TIMEOUT = 5,       /* a bounded device-side wait ran out */
  LMOE_ERR_DEVICE_CHECK = 6,  /* a kernel found invalid data (e.g. expert index out of range) */
  LMOE_ERR_NO_MEMORY = 7      /* lmoe_create could not allocate its private copies */
} lmoe_status;

/* config.flags: LMOE_FLAG_MULTI_KERNEL_DECODE runs the decode path as its
 * sequence of per-step kernels instead of the single persistent kernel.
 *
 * LMOE_FLAG_STAGED_EXPERTS keeps the per-expert weights (gate, up, Down) in
 * host memory and only `expert_slots` of them in GPU memory ("Edge0-145B:
 * Frontier AI Capabilities on Your Own Computer", "Under the Hood of Edge0",
 * "Loading": hot experts stay in GPU memory, an expert library sits in system
 * memory and experts are brought in as needed; "Edge0-145B: Run a 145B
 * Open-Source Model on Your Laptop", "The Three Pillars That Make It Fast":
 * active experts load into a staged fixed-slot buffer, and a prerouter's
 * prediction of the next layer's experts drives the prefetch). The caller's
 * gate / up / Down pointers may then be page-locked host memory that the
 * device can address (cudaHostAlloc, or cudaHostRegister with mapping).
 * lmoe_create copies them once into the handle's own page-locked library, in
 * the layout the decode pass streams. A decode-path pass (T <= 16, the
 * single-kernel pass) first routes its tokens, then copies every routed
 * expert that holds no slot into a slot (the slots are reused in clock order,
 * never one whose expert this pass routes), then runs the pass on the slots;
 * its output is bit for bit that of an unstaged handle. The prefill path and
 * the per-step decode kernels read the caller's expert pointers directly. */
enum { LMOE_FLAG_MULTI_KERNEL_DECODE = 1u, LMOE_FLAG_STAGED_EXPERTS = 2u };

/* config.weight_format: the five shared / expert weight families are int4
 * (symmetric per 32 elements, bf16 scales) or NVFP4 (NVIDIA's FP4 format, the
 * format of the NVFP4 checkpoint in "Edge0-145B: Run a 145B Open-Source Model
 * on Your Laptop", "What You Need to Run It"): FP4 E2M1 codes packed like the
 * int4 nibbles, an FP8 E4M3 scale per 16 elements along K, and an fp32 scale
 * per weight tensor. The router is fp32 in both. */
enum { LMOE_WEIGHTS_INT4 = 0, LMOE_WEIGHTS_NVFP4 = 1 };

/* Execution path for lmoe_layer_forward / lmoe_expert_forward. */
enum { LMOE_PATH_AUTO = 0, LMOE_PATH_DECODE = 1, LMOE_PATH_PREFILL = 2 };

typedef struct {
  int d;            /* model width; multiple of 128 */
  int E;            /* experts; multiple of G, <= 1024 */
  int G;            /* expert groups (shared-matrix groups); <= 64 */
  int k;            /* experts per token; 1 <= k <= min(16, E) */
  int L;            /* latent width; multiple of 32 (prefill path: of 64) */
  int f;            /* per-expert SwiGLU width; multiple of 32 (prefill path: of 64) */
  int qgroup;       /* scale group along the reduction dimension: 32 (int4) or 16 (NVFP4) */
  int lora_rank;    /* 0 = no LoRA branch; else a multiple of 16, <= 128 */
  int has_bias;     /* nonzero: router bias b_r is used */
  unsigned flags;   /* LMOE_FLAG_* bits */
  long long timeout_cycles; /* bound on any device-side wait (clock64 cycles); 0 = 2^31 */
  int decode_max_T; /* token count up to which AUTO takes the decode path; 0 = 16; <= 16 */
  int force_path;   /* LMOE_PATH_* */
  int weight_format; /* LMOE_WEIGHTS_*; NVFP4 layers run the single-kernel decode pass and the prefill
                        path (LMOE_ERR_UNSUPPORTED where only the multi-kernel decode path would fit) */
  int expert_slots;  /* LMOE_FLAG_STAGED_EXPERTS: experts held in GPU memory, min(E, 16 k) <= expert_slots <= E */
} lmoe_config;

/* Device pointers to the layer's weights (borrowed for the handle's life).
 * Shapes as in the layer description; packed int4 rows are [rows][K/2] bytes
 * and their scales [rows][K/32] bf16. With LMOE_WEIGHTS_NVFP4 the *_q rows
 * hold E2M1 codes ([rows][K/2] bytes, element 2j in the low nibble, bit 3 the
 * sign), each *_s points at E4M3 bytes [rows][K/16] (the same byte count as
 * the int4 scales; cast the pointer), and the *_gs arrays give each tensor's
 * fp32 scale: W_in_gs / W_out_gs [G] (one per group's matrix), gate_gs /
 * up_gs / down_gs [E] (one per expert's matrix). A weight is
 * e2m1(q) * e4m3(s) * gs. The *_gs pointers are NULL for int4. */
typedef struct {
  const float* W_r;           /* [E][d] fp32 */
  const float* b_r;           /* [E] fp32, or NULL when has_bias == 0 */
  const uint8_t* W_in_q;      /* [G][L][d/2] */
  const uint16_t* W_in_s;     /* [G][L][d/32] */
  const uint8_t* W_out_q;     /* [G][d][L/2] */
  const uint16_t* W_out_s;    /* [G][d][L/32] */
  const uint8_t* gate_q;      /* [E][f][L/2] */
  const uint16_t* gate_s;     /* [E][f][L/32] */
  const uint8_t* up_q;        /* [E][f][L/2] */
  const uint16_t* up_s;       /* [E][f][L/32] */
  const uint8_t* down_q;      /* [E][L][f/2] */
  const uint16_t* down_s;     /* [E][L][f/32] */
  const uint16_t* A_in;       /* [G][d][r] bf16, NULL when lora_rank == 0 */
  const uint16_t* B_in;       /* [G][r][L] */
  const uint16_t* A_out;      /* [G][L][r] */
  const uint16_t* B_out;      /* [G][r][d] */
  const float* W_in_gs;       /* NVFP4 only: [G] */
  const float* W_out_gs;      /* [G] */
  const float* gate_gs;       /* [E] */
  const float* up_gs;         /* [E] */
  const float* down_gs;       /* [E] */
} lmoe_weights;

/* The token permutation (device arrays, caller-allocated, capacities in
 * brackets). Assignment a = t*k + j is token t's j-th expert.
 *   expert_offsets [E+1]  exclusive prefix sum of tokens per expert
 *   sorted_assign  [T*k]  assignments sorted by (expert, a), stable
 *   inv            [T*k]  inv[sorted_assign[p]] = p
 *   group_offsets  [G+1]  = expert_offsets[g*E/G] (assignment level)
 *   group_tok_offsets [G+1], group_tokens [T*min(G,k)]: per group the
 *                         distinct tokens routed into it, ascending
 *   assign_row     [T*k]  row of (t, group of a) in group_tokens
 * Rows of Y in lmoe_expert_forward / lmoe_combine follow group_tokens. */
typedef struct {
  int32_t* expert_offsets;
  int32_t* sorted_assign;
  int32_t* inv;
  int32_t* group_offsets;
  int32_t* group_tok_offsets;
  int32_t* group_tokens;
  int32_t* assign_row;
} lmoe_perm;

typedef struct lmoe_handle lmoe_handle;

/* Human-readable name of a status (static string). */
const char* lmoe_status_string(lmoe_status s);

/* ABI version of this header (major*100 + minor). */
int lmoe_version(void);

/* Create a handle on `device` for the given shapes and weights. Validates the
 * config, checks the device is sm_103 with enough shared memory, and makes
 * the small private derived copies the kernels use (a 3-way bf16 split of
 * W_r for the tensor-core router; freed by lmoe_destroy). Does not read the
 * int4 weights. Synchronous. *out is NULL on error. */
lmoe_status lmoe_create(lmoe_handle** out, const lmoe_config* cfg, const lmoe_weights* w, int device);

/* Free the handle and its private copies (waits for the device first). NULL is a no-op. */
lmoe_status lmoe_destroy(lmoe_handle* h);

/* Bytes of workspace (device memory, 256-byte aligned) that a call with T
 * tokens needs; the same bound serves every entry point. 0 on a bad handle or T < 0. */
size_t lmoe_workspace_size(const lmoe_handle* h, int T);

/* Router and top-k. Source: "Edge0-145B: Run a 145B Open-Source Model on
 * Your Laptop", section "Not Compression -- Architecture" (512 experts, 10
 * active per token); the selection rule (descending logit, ties to the lower
 * index, softmax over the selected logits) is this library's reading.
 *  x [T][d] bf16 -> idx [T][k] int32 (descending logit, ties to the lower
 *  expert index), w [T][k] fp32 (softmax over the selected logits), and, if
 *  logits != NULL, the fp32 router logits [T][E] the selection was made on.
 *  T == 0 is a no-op. */
lmoe_status lmoe_route(lmoe_handle* h, const uint16_t* x, int T, int32_t* idx, float* w, float* logits, void* ws,
                       lmoe_stream stream);

/* Token permutation by group, then expert. Source: "Edge0-145B: Frontier AI
 * Capabilities on Your Own Computer", section "Under the Hood of Edge0",
 * paragraph "Architecture: share large matrices across sparse experts"
 * (groups of 64 experts share two large matrices, so tokens are gathered per
 * group first, then by expert). idx [T][k] ->
 * every array of *out (see lmoe_perm). Deterministic: bit-identical for
 * identical idx. Indices outside [0, E) set LMOE_ERR_DEVICE_CHECK. */
lmoe_status lmoe_permute(lmoe_handle* h, const int32_t* idx, int T, const lmoe_perm* out, void* ws,
                         lmoe_stream stream);

/* The latent expert FFN for routed tokens. Source: "Edge0-145B: Frontier AI
 * Capabilities on Your Own Computer", section "Under the Hood of Edge0",
 * paragraph "Architecture: share large matrices across sparse experts" (two
 * large matrices shared by a group of 64 experts, a small set of parameters
 * per expert), and "Edge0-145B: Run a 145B Open-Source Model on Your Laptop",
 * section "The Three Pillars That Make It Fast" (int4 expert tensors; the
 * Recover-LoRA branch beside the frozen 4-bit base). For every (group g,
 * token t) row r of the permutation,
 *   Y[r] = Wout[g] ( sum_{j: g(idx[t][j]) = g} w[t][j] * u_{idx[t][j]}( Win[g] x_t ) )  (+ LoRA)
 * x [T][d] bf16, idx/w [T][k], perm from lmoe_permute on the same idx,
 * Y [rows][d] fp32 with rows = group_tok_offsets[G] (capacity T*min(G,k)). */
lmoe_status lmoe_expert_forward(lmoe_handle* h, const uint16_t* x, int T, const int32_t* idx, const float* w,
                                const lmoe_perm* perm, float* Y, void* ws, lmoe_stream stream);

/* Weighted un-permute and combine. Source: the same "Architecture: share
 * large matrices across sparse experts" paragraph (the experts of a token
 * contribute through their groups' shared output matrices, so the weighted
 * expert outputs are summed per group before the shared up-projection and
 * the group results are summed per token). y_t = sum over the groups of t, in
 * ascending group order, of Y[row(g, t)] (+ residual_t), rounded once to
 * bf16. Y as produced by lmoe_expert_forward; residual [T][d] bf16 or NULL. */
lmoe_status lmoe_combine(lmoe_handle* h, const float* Y, const int32_t* idx, const lmoe_perm* perm, int T,
                         const uint16_t* residual, uint16_t* y, lmoe_stream stream);

/* The whole layer: y = bf16(layer(x) (+ residual)). Sources: every passage
 * cited above -- router and top-k ("Not Compression -- Architecture"), the
 * group-shared latent FFN and its combine ("Architecture: share large
 * matrices across sparse experts"), int4 tensors and Recover-LoRA ("The
 * Three Pillars That Make It Fast"). x, residual (nullable) and y are [T][d]
 * bf16; y may alias residual but not x. T <= decode_max_T (default 16) runs
 * the decode path in passes of at most 16 tokens, larger T the prefill path
 * (unless force_path says otherwise). */
lmoe_status lmoe_layer_forward(lmoe_handle* h, const uint16_t* x, int T, const uint16_t* residual, uint16_t* y,
                               void* ws, lmoe_stream stream);

/* Largest batch and scratch size of lmoe_layer_forward_noalloc. */
#define LMOE_NOALLOC_MAX_T 16
#define LMOE_NOALLOC_SCRATCH_BYTES (32u << 20)

/* The layer at decode batch sizes without a workspace argument, for callers
 * that cannot allocate device memory at call time: serving runtimes that
 * reserve nearly all of the device's memory for their own pools and caches
 * up front, and code that must not trigger the device-wide synchronisation
 * that cudaMalloc / cudaFree can cause. This entry point is an addition of
 * this library; the layer's description has no counterpart.
 *
 * It computes exactly what lmoe_layer_forward computes on the decode path
 * (one pass of at most LMOE_NOALLOC_MAX_T tokens, bit for bit the same
 * result), and it always takes the decode path: the handle's force_path and
 * decode_max_T are ignored here. Its scratch lives in one
 * fixed LMOE_NOALLOC_SCRATCH_BYTES array per device that is part of the
 * library's device image. Nothing is allocated by the call, by CUDA or by
 * anything else. x, residual (nullable) and y are [T][d] bf16 device
 * pointers as for lmoe_layer_forward, 16-byte aligned; y may alias residual
 * but not x.
 *
 * The first call on a device (and the first call after that device's
 * primary context was destroyed and made again, e.g. by cudaDeviceReset)
 * looks up that array's address, with the handle's device current; make that
 * first call outside any stream capture. All calls on a device share the one array and it keeps the last
 * call's contents; no word of it needs to start at zero, because every word a
 * call reads it has first written. Calls whose work overlaps on the GPU (two
 * streams, two handles on one device) race on the array and give undefined
 * results: order them on one stream, or use lmoe_layer_forward with separate
 * workspaces.
 *
 * Returns LMOE_ERR_INVALID_ARG for T < 0 or T > LMOE_NOALLOC_MAX_T (and for
 * the argument errors of lmoe_layer_forward), LMOE_ERR_UNSUPPORTED when the
 * layer's shape needs more than LMOE_NOALLOC_SCRATCH_BYTES of scratch at that
 * T, LMOE_ERR_ALIGNMENT and LMOE_ERR_CUDA as lmoe_layer_forward does. */
lmoe_status lmoe_layer_forward_noalloc(lmoe_handle* h, const uint16_t* x, int T, const uint16_t* residual,
                                       uint16_t* y, lmoe_stream stream);

/* The routing a decode-path pass used, read back from its workspace: after
 * lmoe_layer_forward with 1 <= T <= 16 tokens on the decode path (either
 * decode kernel sequence) with workspace ws, copies that call's expert
 * indices idx [T][k], weights w [T][k] and, if logits != NULL, router logits
 * [T][E] (fp32, the values the selection was made on) from ws into the
 * caller's device buffers, on `stream`. It exists so that the selection made
 * inside the single-kernel pass can be compared index for index with a
 * reference; it has no counterpart on the pages. Valid only until the next
 * call that uses ws. LMOE_ERR_INVALID_ARG for T outside [0, 16] or null
 * pointers. */
lmoe_status lmoe_decode_routing(lmoe_handle* h, const void* ws, int T, int32_t* idx, float* w, float* logits,
                                lmoe_stream stream);

/* The whole layer from and to HOST memory: copies x (and residual) from
 * host to the workspace, runs lmoe_layer_forward, copies y back and waits
 * for the stream. x_host, residual_host (nullable) and y_host are host
 * pointers ([T][d] bf16; page-locked memory gives asynchronous copies). The
 * workspace must hold lmoe_workspace_size(h, T) + lmoe_host_staging_size(h, T) bytes.
 * The handle keeps the last call's copies and layer as a CUDA graph and
 * replays it while x_host, residual_host, y_host, ws, T and the stream stay
 * the same (every call still copies its inputs in and its output out); a
 * call with other buffers captures anew. Staged handles, handles with stage
 * events set, and calls on a stream that is being captured issue the work
 * directly. A prefill-sized call (at least 8192 tokens on the prefill path)
 * runs as a pipeline of token chunks (1024 tokens, then 4096 each): each
 * chunk's copy in, its layer
 * and its copy out overlap those of its neighbours on three streams, the
 * weights are dequantised once, and the result is that of one
 * lmoe_layer_forward on all T tokens (every step of the layer is per token).
 * The handle is not safe to share between host threads. */
lmoe_status lmoe_layer_forward_host(lmoe_handle* h, const uint16_t* x_host, int T, const uint16_t* residual_host,
                                    uint16_t* y_host, void* ws, lmoe_stream stream);

/* Extra workspace bytes lmoe_layer_forward_host needs for its staging copies. */
size_t lmoe_host_staging_size(const lmoe_handle* h, int T);

/* A stack of layers without attention ("512 expert networks across 48
 * layers"): x_0 = x, x_{l+1} = bf16(x_l + bf16(layer_l(x_l))) for
 * l = 0 .. n_layers-1, y = x_{n_layers}. layers[l] are handles of the same
 * shape (d, E, G, k, L, f, lora_rank) on the same device, each with its own
 * weights; x and y are [T][d] bf16 device pointers (y may alias x). Each
 * layer computes exactly what lmoe_layer_forward computes. When every layer
 * takes the single-kernel decode pass (T <= 16), each layer is one launch:
 * the kernel rounds its output to bf16 and adds the residual in its final
 * combine, runs as a programmatic dependent of the previous layer's launch
 * (its weight stream starts while that layer finishes; x is read after it
 * completes), and prefetches the next layer's router rows and W_in tiles
 * into L2 during its own tail. Otherwise each layer runs as
 * lmoe_layer_forward without a residual, followed by a kernel that adds the
 * residual and rounds once. The two give the same bits. When the layers
 * are staged handles (LMOE_FLAG_STAGED_EXPERTS), layer l + 1's prerouter
 * runs on the handle's second stream while layer l runs (given x_l), and
 * layer l + 1 starts after it. ws must hold
 * lmoe_stack_workspace_size(layers[0], T) bytes. Returns LMOE_ERR_INVALID_ARG
 * for n_layers < 1, a null handle or mismatched shapes or devices, and the
 * errors of lmoe_layer_forward. */
lmoe_status lmoe_stack_forward(lmoe_handle* const* layers, int n_layers, const uint16_t* x, int T, uint16_t* y,
                               void* ws, lmoe_stream stream);

/* The prerouter of a staged handle h (LMOE_FLAG_STAGED_EXPERTS): selects
 * the top-k experts of h's router for the T <= 16 tokens x (device bf16
 * [T][d]) and copies those that hold no slot into h's slots, on `stream`,
 * as the forward does for a routed expert. It is meant for the next layer
 * of a stack, given the current layer's input one layer ahead; the
 * prediction here is h's own router applied to that earlier input (the
 * pages' prerouter is a trained head: a stated stand-in). It uses scratch
 * inside the handle, not a workspace, so it may run on a second stream while
 * another layer runs; it must not run concurrently with a forward or another
 * prefetch of the same handle. Returns LMOE_ERR_INVALID_ARG for a handle
 * without staging or T outside 1..16. */
lmoe_status lmoe_prefetch_experts(lmoe_handle* h, const uint16_t* x, int T, lmoe_stream stream);

/* Counters of a staged handle since its creation (host copy; waits for the
 * device): decode passes, experts those passes routed (distinct per pass),
 * routed experts already in a slot when their pass started (hits), experts
 * the passes had to copy themselves, experts the prerouter copied, and the
 * bytes copied from host memory. */
typedef struct {
  unsigned long long passes, routed, hits, staged_on_demand, prefetched, bytes_copied;
} lmoe_stage_stats;
lmoe_status lmoe_get_stage_stats(lmoe_handle* h, lmoe_stage_stats* out);

/* Workspace bytes of lmoe_stack_forward: one layer's workspace plus two
 * [T][d] bf16 activation buffers. 0 on a bad handle or T < 0. */
size_t lmoe_stack_workspace_size(const lmoe_handle* h, int T);

/* Wait for `stream`, then read and clear the handle's device error word.
 * Returns LMOE_OK, LMOE_ERR_TIMEOUT, LMOE_ERR_DEVICE_CHECK or LMOE_ERR_CUDA. */
lmoe_status lmoe_check(lmoe_handle* h, lmoe_stream stream);

/* Sets the handle's budget for bounded device-side waits (clock64 cycles;
 * 0 restores the config's value, or 2^31). The single-kernel decode pass
 * waits at grid barriers; when a wait runs out the kernel sets the device
 * error word and finishes without waiting further, so lmoe_check reports
 * LMOE_ERR_TIMEOUT and that call's output is invalid. A budget of 1 makes
 * every such wait run out at once (a test hook for the error path). */
lmoe_status lmoe_set_timeout(lmoe_handle* h, long long cycles);

/* Profiling hook: when events != NULL, lmoe_layer_forward records
 * events[2*i] / events[2*i+1] (cudaEvent_t) on its stream around launch i of
 * its kernel sequence, for i < n. The stage names are given by
 * lmoe_stage_name; in the prefill path, a stage (for instance "route": the
 * router GEMM and the top-k kernel) may span several kernels. Pass NULL to
 * turn it off. */
lmoe_status lmoe_set_stage_events(lmoe_handle* h, void* const* events, int n);

/* Name of kernel i of lmoe_layer_forward's sequence for T tokens ("" if none),
 * and the count of kernels launched per call through *count. */
const char* lmoe_stage_name(const lmoe_handle* h, int T, int i, int* count);

/* Number of kernels one lmoe_layer_forward call launches for T tokens (a
 * stage of the prefill path may launch several); 0 for a null handle or
 * T < 1. Host only; launches nothing. */
int lmoe_launch_count(const lmoe_handle* h, int T);

#ifdef __cplusplus
}
#endif
#endif /* LMOE_H */
