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

// TMA descriptors of the weights for the single-kernel decode pass (made
// once per handle). Packed int4 matrices are viewed as [rows][K/256][128 B]
// (128-byte swizzle), their scales as [rows][K/32] bf16, W_r as
// [E][d/256][256] fp32, and the slice-major copy of Down as 128-byte lines
// ([E][f/32][L][16 B]) with scales [E][f/32][L].
struct DecodeMaps {
  CUtensorMap wr;
  CUtensorMap win_q, win_s;
  CUtensorMap gate_q, gate_s, up_q, up_s;
  CUtensorMap dsl_q, dsl_s;
  CUtensorMap wout_q, wout_s;
};

// The single-kernel decode pass (decode_fused.cu).
struct FusedArgs {
  DecodeArgs A;
  DecodeMaps maps;
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
  // layer stacks: the next layer's router rows and W_in tiles of this CTA are
  // prefetched into L2 once this layer's own weights are requested
  int has_next;
  CUtensorMap next_wr, next_win_q, next_win_s;
  // the Recover-LoRA branch (lora.cu): Hl [G][16][L] is added to H; Z is also
  // written in fp32 to Zlin [G][16][L]; the per-group outputs are left in Yp
  // for lora_out to combine (no combine here)
  const float* hl;
  float* zlin;
  int no_combine;
  // diagnosis: [0] where the first timed-out wait of a launch gave up, then
  // per CTA 16 %globaltimer stamps of its phases (a region of the workspace)
  unsigned long long* diag;
};
size_t fused_counter_words(int d, int E, int G, int L);
size_t fused_zpart_bytes(int G, int L, int grid);
size_t fused_diag_bytes(int grid);
// bytes of the slice-major copy of Down (packed int4 and scales)
size_t fused_down_copy_bytes(int E, int L, int f);
cudaError_t launch_repack_down(const uint8_t* q, const uint16_t* s, int E, int L, int f, uint8_t* qo, uint16_t* so,
                               cudaStream_t st);
// Encodes the tensor maps; false if the driver refuses one of them.
bool fused_make_maps(const DecodeArgs& A, const uint8_t* dsl_q, const uint16_t* dsl_s, DecodeMaps* maps);
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
cudaError_t launch_lora_in(const DecodeArgs& A, float* Ppart, float* P, float* Hl, unsigned* tickets, cudaStream_t st);
cudaError_t launch_lora_q(const DecodeArgs& A, const float* Zlin, float* Q, cudaStream_t st);
cudaError_t launch_lora_out(const DecodeArgs& A, const float* Yp, const float* Q, cudaStream_t st);
cudaError_t launch_residual_add(const uint16_t* x, const uint16_t* y, size_t n, uint16_t* out, cudaStream_t st);
cudaError_t launch_combine(const float* Y, const int32_t* idx, const int32_t* assign_row, int T, int d, int k,
                           int epg, const uint16_t* residual, uint16_t* y, cudaStream_t st);

// General permutation for any T (multi-CTA, deterministic).
size_t permute_scratch_bytes(int T, int E, int G);
cudaError_t launch_permute(const int32_t* idx, int T, int E, int G, int k, const PermPtrs& pm, void* scratch,
                           unsigned* err, cudaStream_t st);

}  // namespace lmoe
