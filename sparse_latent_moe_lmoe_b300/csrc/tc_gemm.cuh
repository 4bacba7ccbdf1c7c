// A persistent, warp-specialised tcgen05 GEMM for sm_103a:
//   D[128 x BN] (fp32, tensor memory) += A[128 x 64] . B[BN x 64]^T per K block,
// both operands 16-bit and K-major in 128-byte-swizzled shared memory (the
// layout tcgen05.mma reads through a shared-memory descriptor), brought in by
// the problem's own TMA boxes:
//   thread 0     issues each K block's copies (prob.load_a / load_b, or
//                prob.kprep before the stage wait and prob.kissue after it)
//   warp 8       one thread issues tcgen05.mma (kind::f16) and commits
//   warps 12..15 epilogue: tcgen05.ld from tensor memory, problem-specific
//                output (warp w reads TMEM lanes 32*(w%4) .. +31); warps
//                4..7 take the second half of each tile's columns beside
//                them when the problem asks for two epilogue sets
// Shared-memory stages are handed over with mbarriers (full: the copies'
// transaction bytes; empty: tcgen05.commit); two accumulators in tensor memory
// let the epilogue of one tile overlap the MMAs of the next. Every wait is
// bounded by a cycle budget; running out sets the timeout bit of the error
// word and the wait gives up (the output is then invalid).
#pragma once
#include "common.cuh"
#include "ring.cuh"

namespace lmoe {
namespace tc {

constexpr int BM = 128, BK = 64, MAX_STAGES = 4;
constexpr int NPROD_WARPS = 8, MMA_WARP = 8, EPI_WARP0 = 12, THREADS = 512;
constexpr int A_BYTES = BM * BK * 2;

LMOE_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
LMOE_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// K-major operand in 128-byte swizzle: rows of 128 B, 8-row groups 1024 B apart
LMOE_DEV uint64_t sdesc(const void* p) {
  uint64_t d = (uint64_t)((smem_u32(p) & 0x3FFFF) >> 4);
  d |= (uint64_t)1 << 16;            // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;            // descriptor version
  d |= (uint64_t)2 << 61;            // 128-byte swizzle
  return d;
}
// kind::f16 instruction descriptor: D fp32, A/B fp16 (ab_bf16 = 0) or bf16 (1), both K-major
LMOE_DEV uint32_t idesc(int M, int N, int ab_bf16) {
  return (1u << 4) | ((uint32_t)ab_bf16 << 7) | ((uint32_t)ab_bf16 << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
// byte offset of 16-byte chunk c (0..7) of row r in a [rows][128 B] swizzled tile
LMOE_DEV uint32_t swz(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

LMOE_DEV void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(id), "r"(accumulate));
}
LMOE_DEV void mma_commit(uint64_t* m) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(m))
               : "memory");
}
// 16 consecutive fp32 columns of this thread's TMEM lane
LMOE_DEV void tmem_ld16(uint32_t taddr, float v[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// int4 -> fp16 in natural order for one 32-bit word (elements 0..7 of the
// word, element i in bits 4i..4i+3), times the group scale s2:
// out[i] = (e_{2i}, e_{2i+1}). Exact: q*s needs at most 11 significant bits.
LMOE_DEV void dequant_word_natural(uint32_t v, __half2 s2, uint32_t out[4]) {
  const uint32_t hi = v >> 4;
  const __half2 k1032 = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t t;
    // bytes: [v.byte i, -, hi.byte i, -] -> nibbles e_{2i} (low half), e_{2i+1} (high half)
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(t) : "r"(v), "r"(hi), "r"(0x0400u | (i * 0x0101u)));
    asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(t) : "r"(t), "r"(0x000F000Fu), "r"(0x64086408u));  // (a&b)^c
    __half2 h = __hsub2(*reinterpret_cast<__half2*>(&t), k1032);
    h = __hmul2(h, s2);
    out[i] = *reinterpret_cast<uint32_t*>(&h);
  }
}

struct Tile {
  int prob;    // problem index (group / expert / 0)
  int m0;      // first row of the M tile within the problem
  int n0;      // first output column
  int rows;    // valid rows in this M tile (<= 128)
  int nkb;     // K blocks
  unsigned gm; // problem-specific (the groups a token tile reads, for W_out)
  int arow;    // problem-specific (the first A row of the tile, looked up once per tile)
  unsigned gl; // problem-specific (W_out: the tile's groups in order, 4 bits each, when G <= 16)
};

struct Shared {
  uint64_t full[MAX_STAGES], empty[MAX_STAGES], acc_full[2], acc_empty[2];
  uint32_t tmem_base;
  int scratch[1024 + 64];  // problem-specific (tile prefix sums)
};

// A problem P supplies BN (B rows per stage, <= 256), ACC_COLS (TMEM columns
// per accumulator), STAGES, EPI_SETS, KPREP, and init / num_tiles / tile /
// load_a / load_b (or kprep / kissue) / mma_stage / epilogue.
template <class P>
__global__ void __launch_bounds__(THREADS, 1) gemm_kernel(const __grid_constant__ P prob) {
  extern __shared__ __align__(1024) unsigned char dyn[];
  __shared__ Shared sh;
  constexpr int BN = P::BN;                      // B rows per stage (<= 256)
  constexpr int ACC_COLS = P::ACC_COLS;          // TMEM columns per accumulator
  constexpr int NACC = (2 * ACC_COLS <= 512) ? 2 : 1;
  constexpr int B_BYTES = BN * BK * 2;
  constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  constexpr int STAGES = P::STAGES;
  static_assert(STAGES <= MAX_STAGES, "stages");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dyn) + 1023) & ~(uintptr_t)1023);
  const long long budget = prob.budget;
  unsigned* err = prob.err;
  // one copy-issuing thread leaves warps 1..7 free: warps 4..7 become a
  // second epilogue set where the problem asks for it
  constexpr bool EPI2 = P::EPI_SETS == 2;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh.acc_full[a], 1);
      mbar_init(&sh.acc_empty[a], EPI2 ? 8 : 4);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sh.tmem_base)),
                 "r"(NACC * ACC_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  prob.init(sh.scratch);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
  const int ntiles = prob.num_tiles(sh.scratch);

  // epilogue over this CTA's tiles; half: -1 every column, 0 / 1 the first / second half
  auto epilogue_loop = [&](int half) {
    const int q = warp & 3;
    int tcount = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++tcount) {
      const Tile tl = prob.tile(sh.scratch, t);
      const int acc = tcount % NACC, ause = tcount / NACC;
      mbar_wait(&sh.acc_full[acc], ause & 1, budget, err);
      __syncwarp();
      tc_fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * ACC_COLS);
      prob.epilogue(sh.scratch, tl, q * 32 + lane, tbase, half);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.acc_empty[acc]);
    }
  };

  if (warp < NPROD_WARPS) {
    // ------------------------------------------------ producer: TMA only (one thread)
    if (tid == 0) {
      int kiter = 0;
      for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const Tile tl = prob.tile(sh.scratch, t);
        for (int kb = 0; kb < tl.nkb; ++kb, ++kiter) {
          const int s = kiter % STAGES, use = kiter / STAGES;
          unsigned char* sa = base + s * STAGE_BYTES;
          if constexpr (P::KPREP) {
            // the K block's copy coordinates are worked out before the wait
            // for its stage, so that only the copies follow the wait
            const auto kc = prob.kprep(tl, kb);
            if (use > 0) mbar_wait(&sh.empty[s], (use - 1) & 1, budget, err);
            mbar_expect_tx(&sh.full[s], (uint32_t)(A_BYTES + B_BYTES));
            prob.kissue(kc, sa, sa + A_BYTES, &sh.full[s]);
          } else {
            if (use > 0) mbar_wait(&sh.empty[s], (use - 1) & 1, budget, err);
            mbar_expect_tx(&sh.full[s], (uint32_t)(A_BYTES + B_BYTES));
            prob.load_a(tl, kb, sa, &sh.full[s]);
            prob.load_b(tl, kb, sa + A_BYTES, &sh.full[s]);
          }
        }
      }
    } else if (EPI2 && warp >= 4) {  // the second epilogue set (acc_empty counts 8 arrivals)
      epilogue_loop(1);
    }
  } else if (warp == MMA_WARP) {
    // -------------------------------------------------------------- MMA issue
    if (lane == 0) {
      int kiter = 0, tcount = 0;
      for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++tcount) {
        const Tile tl = prob.tile(sh.scratch, t);
        const int acc = tcount % NACC, ause = tcount / NACC;
        if (ause > 0) mbar_wait(&sh.acc_empty[acc], (ause - 1) & 1, budget, err);
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(acc * ACC_COLS);
        for (int kb = 0; kb < tl.nkb; ++kb, ++kiter) {
          const int s = kiter % STAGES, use = kiter / STAGES;
          mbar_wait(&sh.full[s], use & 1, budget, err);
          tc_fence_after();
          unsigned char* sa = base + s * STAGE_BYTES;
          unsigned char* sb = sa + A_BYTES;
          prob.mma_stage(tl, kb, d_tmem, sdesc(sa), sdesc(sb));
          mma_commit(&sh.empty[s]);
        }
        mma_commit(&sh.acc_full[acc]);
      }
    }
    __syncwarp();
  } else if (warp >= EPI_WARP0) {
    // --------------------------------------------------------------- epilogue
    epilogue_loop(EPI2 ? 0 : -1);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(NACC * ACC_COLS));
}

template <class P>
constexpr int smem_bytes() {
  return P::STAGES * (A_BYTES + P::BN * BK * 2) + 1024;
}

}  // namespace tc
}  // namespace lmoe
