// Argument block and launchers of the decode-path kernels (<= 16 tokens).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lmoe {

// device error word bits
enum : unsigned { ERRBIT_TIMEOUT = 1u, ERRBIT_BAD_INDEX = 2u, ERRBIT_BAD_DATA = 4u };

struct PermPtrs {
  int32_t* expert_offsets;
  int32_t* sorted_assign;
  int32_t* inv;
  int32_t* group_offsets;
  int32_t* group_tok_offsets;
  int32_t* group_tokens;
  int32_t* assign_row;
};

// Everything one decode pass reads or writes (device pointers).
struct DecodeArgs {
  int T, d, E, G, k, L, f, r, epg, ks_in;
  // weights
  const float* W_r;
  const float* b_r;
  const uint8_t* W_in_q;
  const uint16_t* W_in_s;
  const uint8_t* W_out_q;
  const uint16_t* W_out_s;
  const uint8_t* gate_q;
  const uint16_t* gate_s;
  const uint8_t* up_q;
  const uint16_t* up_s;
  const uint8_t* down_q;
  const uint16_t* down_s;
  const uint16_t* A_in;
  const uint16_t* B_in;
  const uint16_t* A_out;
  const uint16_t* B_out;
  // weight format (LMOE_WEIGHTS_*) and, for NVFP4, the per-tensor fp32 scales
  // (the *_s pointers then hold E4M3 bytes)
  int wfmt;
  const float* W_in_gs;
  const float* W_out_gs;
  const float* gate_gs;
  const float* up_gs;
  const float* down_gs;
  // this pass's tokens
  const uint16_t* x;         // [T][d]
  const uint16_t* residual;  // [T][d] or null
  uint16_t* y;               // [T][d]
  int32_t* idx;              // [T][k]
  float* w;                  // [T][k]
  PermPtrs pm;               // permutation of this pass's tokens
  float* Hp;                 // [ks_in][G][16][L]
  float* V;                  // [16*k][f]
  float* Z;                  // [G][16][L]
  float* Yp;                 // [G][16][d]
  float* Pin;                // [G][16][r]
  float* Qout;               // [G][16][r]
  unsigned* tickets;         // [1 + d/64], zero between calls
  unsigned* err;             // device error word
  // expert_forward (rows mode): the caller's full routing and permutation
  int tok0;                  // index of this pass's first token
  const int32_t* idx_all;
  const int32_t* assign_row_all;
  float* Yrows;
};

// The single-kernel decode pass streams its weights from a copy made when the
// handle is created, laid out chunk by chunk in the order and form the
// consumers read them: every chunk is one contiguous run of packed 4-bit
// codes (its 128-byte lines already in the 128-byte swizzle of the
// shared-memory slot) followed by the chunk's scales, so one bulk copy moves
// it. NVFP4 code words are stored with byte b holding elements b and b + 4.
//   win   [G L/16 tiles of 16 rows][d/PW pieces][9 PW bytes], PW = min(d, 2048)
//   unit  [E][f/32 slices][gate rows, up rows, Down columns][18 L bytes]
//   wout  [G][d/32 blocks of 32 rows][18 L bytes]
// The router rows are read from W_r itself (fp32 rows, contiguous).
struct DecodePack {
  const float* wr;
  const uint8_t* win;
  const uint8_t* unit;
  const uint8_t* wout;
};
size_t decode_pack_bytes(int d, int E, int G, int L, int f);
// fills `pk` (win/unit/wout carved from `buf`, decode_pack_bytes long) from
// the layer's weights; wr is taken from A.W_r
cudaError_t launch_decode_pack(const DecodeArgs& A, uint8_t* buf, DecodePack* pk, cudaStream_t st,
                               uint8_t* unit_buf = nullptr);
// bytes of one expert's unit chunks (its f/32 units of gate, up and Down)
size_t decode_expert_bytes(int L, int f);
// decode_pack_bytes without the unit region (staged handles keep it elsewhere)
size_t decode_pack_bytes_shared(int d, int E, int G, int L, int f);

// The staged expert cache (staging.cu): device state of a handle's slots.
struct StageState {
  unsigned clock;   // the slot the next sweep for victims starts at
  unsigned n_copy;  // experts the last plan assigned to slots (read by the copy kernel)
  unsigned long long passes, routed, hits, on_demand, prefetched, bytes;
};
struct StagePlan {
  const int32_t* idx;  // the set to stage: n expert indices (repeats allowed)
  int n, E, S;
  int must;            // 1: a forward pass's routed set (counted as such); 0: a prefetch
  int32_t* slot_of;    // [E] slot of each expert or -1
  int32_t* expert_in;  // [S] expert in each slot or -1
  StageState* st;
  int2* copies;        // [256] (expert, slot) of the plan
  size_t expert_bytes; // one expert in the decode pass's layout (a multiple of 16)
  unsigned* err;
};
cudaError_t launch_stage_plan(const StagePlan& P, cudaStream_t st);
// lib: the device address of the host library
cudaError_t launch_stage_copy(const StagePlan& P, const uint8_t* lib, uint8_t* slots, int num_sms, cudaStream_t st);

// The single-kernel decode pass (decode_fused.cu).
struct FusedArgs {
  DecodeArgs A;
  DecodePack pk;
  float* logits;                 // [16][E]
  uint4* Hf;                     // [G][L/128][128 NT] H as fp16 fragments (NT = token tiles of the launch)
  float* Zpart;                  // [grid + G][16][L] partial sums of Z, one per (CTA, group) it worked on
  uint4* Zf;                     // [G][L/128][128 NT] Z as fragments
  float* Yp;                     // [G][16][d] per-group outputs of W_out
  unsigned* ctr;                 // arrival counters, two copies (fused_counter_words)
  unsigned long long* launches;  // launch counter (selects the counter copy)
  long long timeout;             // spin budget (clock64 cycles)
  // layer stacks: y = bf16(residual + bf16(layer(x))) instead of one rounding
  int round_first;
  // layer stacks: launched as a programmatic dependent of the previous layer
  // (the weight stream starts at once; x is read after griddepcontrol.wait)
  int pdl;
  // the LoRA branch: launched as a programmatic dependent of lora_hl; Hl is
  // read after griddepcontrol.wait (x and the weights are ready at launch)
  int pdl_hl;
  // layer stacks: the next layer's router rows and W_in chunks of this CTA
  // are prefetched into L2 once this layer's own weights are requested
  int has_next;
  const float* next_wr;
  const uint8_t* next_win;
  // the Recover-LoRA branch (lora.cu): Hl [G][16][L] is added to H; Z is also
  // written in fp32 to Zlin [G][16][L]; the per-group outputs are left in Yp
  // for lora_out to combine (no combine here)
  const float* hl;
  float* zlin;
  int no_combine;
  // staged experts: the unit chunks of expert e are read from slot
  // slot_of[e] of pk.unit (null: from expert e's own place)
  const int32_t* slot_of;
  // diagnosis: [0] where the first timed-out wait of a launch gave up, then
  // per CTA 32 %globaltimer stamps of its phases (a region of the workspace)
  unsigned long long* diag;
};
size_t fused_counter_words(int d, int E, int G, int L);
size_t fused_zpart_bytes(int G, int L, int grid);
size_t fused_diag_bytes(int grid);
bool fused_decode_supported(const DecodeArgs& A, int grid);
cudaError_t fused_set_attributes();
int fused_grid(int num_sms);
// pdl != 0: a plain launch with programmatic stream serialization (layer
// stacks, after another layer's pass); else a cooperative launch
cudaError_t launch_decode_fused(const FusedArgs& F, int grid, cudaStream_t st, int pdl = 0);

// Records timing events around each launch when attached.
struct StageHook {
  virtual void before(cudaStream_t) {}
  virtual void after(cudaStream_t) {}
  virtual ~StageHook() {}
};

cudaError_t decode_set_attributes();
cudaError_t permute_set_attributes();
cudaError_t launch_route(const DecodeArgs& A, int do_perm, float* logits_out, cudaStream_t st);
cudaError_t launch_lora_proj(const DecodeArgs& A, int which, cudaStream_t st);
cudaError_t launch_experts(const DecodeArgs& A, int mode, cudaStream_t st, StageHook* hook);
// out = bf16(x + y), n a multiple of 8 (the residual step of a layer stack)
// The Recover-LoRA branch around the single-kernel decode pass (lora.cu).
cudaError_t lora_set_attributes();
bool lora_fused_supported(const DecodeArgs& A);
// tickets: lora_ticket_words(d, G) words, zero between calls
size_t lora_ticket_words(int d, int G);
// scratch of the partial sums: Ppart [G][d/LORA_ROWS][16][r], Qpart [G][L/LORA_ROWS][16][r]
constexpr int LORA_ROWS = 128;
inline size_t lora_ppart_bytes(int d, int G, int r) { return (size_t)G * (d / LORA_ROWS) * 16 * r * 4; }
inline size_t lora_qpart_bytes(int L, int G, int r) { return (size_t)G * (L / LORA_ROWS) * 16 * r * 4; }
// lora_p then lora_hl (two kernels; the hook brackets each)
// pdl: lora_hl, lora_q and lora_out launch as programmatic dependents of
// their stream predecessors (lora_p, the single kernel, lora_q)
cudaError_t launch_lora_in(const DecodeArgs& A, float* Ppart, float* P, float* Hl, unsigned* tickets,
                           cudaStream_t st, StageHook* hook, bool pdl = false);
cudaError_t launch_lora_q(const DecodeArgs& A, const float* Zlin, float* Qpart, float* Q, unsigned* tickets,
                          cudaStream_t st, bool pdl = false);
cudaError_t launch_lora_out(const DecodeArgs& A, float* Yp, const float* Q, unsigned* tickets, cudaStream_t st,
                            bool pdl = false);
cudaError_t launch_residual_add(const uint16_t* x, const uint16_t* y, size_t n, uint16_t* out, cudaStream_t st);
cudaError_t launch_combine(const float* Y, const int32_t* idx, const int32_t* assign_row, int T, int d, int k,
                           int epg, const uint16_t* residual, uint16_t* y, cudaStream_t st);

// General permutation for any T (multi-CTA, deterministic).
size_t permute_scratch_bytes(int T, int E, int G);
cudaError_t launch_permute(const int32_t* idx, int T, int E, int G, int k, const PermPtrs& pm, void* scratch,
                           unsigned* err, cudaStream_t st);

}  // namespace lmoe
