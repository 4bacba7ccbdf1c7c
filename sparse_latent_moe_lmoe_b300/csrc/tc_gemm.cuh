// A persistent, warp-specialised tcgen05 GEMM for sm_103a:
//   D[128 x BN] (fp32, tensor memory) += A[128 x 64] . B[BN x 64]^T per K block,
// with operands staged by the CTA's own warps into 128-byte-swizzled shared
// memory (K-major, the layout tcgen05.mma reads through a shared-memory
// descriptor):
//   warps 0..7   producers: A rows (gathered through the problem's row map,
//                cp.async or bf16->fp16 conversion) and B rows (int4
//                dequantised to fp16 in registers, or bf16 copied)
//   warp 8       one thread issues tcgen05.mma (kind::f16) and commits
//   warps 12..15 epilogue: tcgen05.ld from tensor memory, problem-specific
//                output (warp w reads TMEM lanes 32*(w%4) .. +31); when both
//                operands come by TMA (one producer thread), warps 4..7 take
//                the second half of each tile's columns beside them
// Shared-memory stages are handed over with mbarriers (full: producer
// arrivals; empty: tcgen05.commit); two accumulators in tensor memory let
// the epilogue of one tile overlap the MMAs of the next. Every wait is
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

LMOE_DEV void cp16(void* s, const void* g, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(s)), "l"(g), "r"(valid ? 16 : 0)
               : "memory");
}
LMOE_DEV void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
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

// B_MODE 0: int4 + bf16 scales dequantised by the producers; 1: bf16 rows copied;
//         2: 16-bit rows loaded by the problem's own TMA boxes (prob.load_b,
//            128-byte swizzle, BN rows x 64 elements per stage)
// A_MODE 0: fp16 rows by cp.async; 1: bf16 rows converted to fp16; 2: bf16 rows by cp.async;
//        3: 16-bit rows by the problem's TMA boxes (prob.load_a; needs B_MODE 2)
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
  static_assert(P::B_MODE != 0 || BN <= NPROD_WARPS * 32, "int4 B rows: one per producer thread");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dyn) + 1023) & ~(uintptr_t)1023);
  const long long budget = prob.budget;
  unsigned* err = prob.err;
  // TMA operands leave warps 1..7 free: warps 4..7 become a second epilogue
  // set where the problem asks for it
  constexpr bool EPI2 = P::A_MODE == 3 && P::EPI_SETS == 2;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sh.full[s], P::A_MODE == 3 ? 1 : NPROD_WARPS * 32 + (P::B_MODE == 2 ? 1 : 0));
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

  constexpr bool ASYNC = P::A_MODE != 1 && P::B_MODE != 0;
  static_assert(P::A_MODE != 3 || P::B_MODE == 2, "A by TMA needs B by TMA");
  if (warp < NPROD_WARPS) {
   if constexpr (P::A_MODE == 3) {
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
   } else if constexpr (ASYNC) {
    // ------------------------------------------------ producers, all copies asynchronous
    // A rows by cp.async (gathered through the problem's row map), B by TMA
    // (B_MODE 2, thread 0) or cp.async (B_MODE 1); STAGES-1 K blocks ahead.
    const int pt = tid;  // 0..255
    const int ar = pt >> 1, ac0 = (pt & 1) * 4;
    constexpr int LA = STAGES - 1;
    int t_i = blockIdx.x, kb_i = 0;
    Tile tl_i = t_i < ntiles ? prob.tile(sh.scratch, t_i) : Tile{};
    int issued = 0, done = 0;
    auto issue_next = [&]() {
      const int kiter = issued, s = kiter % STAGES, use = kiter / STAGES;
      if (use > 0) mbar_wait(&sh.empty[s], (use - 1) & 1, budget, err);
      unsigned char* sa = base + s * STAGE_BYTES;
      unsigned char* sb = sa + A_BYTES;
      const void* src = ar < tl_i.rows ? prob.a_row(sh.scratch, tl_i, ar, kb_i) : nullptr;
      if (src) {
        const char* s1 = reinterpret_cast<const char*>(src);
#pragma unroll
        for (int c = 0; c < 4; ++c) cp16(sa + swz(ar, ac0 + c), s1 + (ac0 + c) * 16, true);
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4*>(sa + swz(ar, ac0 + c)) = make_uint4(0, 0, 0, 0);
      }
      if constexpr (P::B_MODE == 2) {
        if (pt == 0) {
          mbar_expect_tx(&sh.full[s], (uint32_t)B_BYTES);
          prob.load_b(tl_i, kb_i, sb, &sh.full[s]);
        }
      } else {
        for (int n = pt; n < BN; n += NPROD_WARPS * 32) {
          const uint16_t* bsrc = prob.b_row_bf16(sh.scratch, tl_i, n, kb_i);
          if (bsrc) {
#pragma unroll
            for (int c = 0; c < 8; ++c) cp16(sb + swz(n, c), bsrc + c * 8, true);
          } else {
#pragma unroll
            for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(sb + swz(n, c)) = make_uint4(0, 0, 0, 0);
          }
        }
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
      ++issued;
      if (++kb_i == tl_i.nkb) {
        kb_i = 0;
        t_i += gridDim.x;
        if (t_i < ntiles) tl_i = prob.tile(sh.scratch, t_i);
      }
    };
    while (issued < LA && t_i < ntiles) issue_next();
    while (done < issued) {
      if (t_i < ntiles) {
        issue_next();
        asm volatile("cp.async.wait_group %0;" ::"n"(LA) : "memory");
      } else {
        asm volatile("cp.async.wait_group 0;" ::: "memory");
      }
      fence_async_smem();
      mbar_arrive(&sh.full[done % STAGES]);
      ++done;
    }
   } else {
    // ---------------------------------------------------------------- producers
    // One K block ahead: while K block i is converted into its stage, the
    // global loads (cp.async for fp16 A rows, registers for int4 / bf16 data)
    // of block i+1 are already in flight.
    const int pt = tid;  // 0..255
    const int ar = pt >> 1, ac0 = (pt & 1) * 4;
    struct Regs {
      uint4 a[4];            // A_MODE 1: 4 chunks of bf16
      bool a_valid;
      uint4 w0, w1;          // B_MODE 0: 32 bytes of int4 for row pt (and pt + 256 for BN = 512: unused)
      uint16_t s0, s1;
      bool b_valid;
    };
    Regs cur, nxt;
    // the flat (tile, kb) sequence of this CTA
    int t_cur = blockIdx.x, kb_cur = 0;
    Tile tl_cur = t_cur < ntiles ? prob.tile(sh.scratch, t_cur) : Tile{};
    auto issue = [&](const Tile& tl, int kb, int kiter, Regs& R) {
      const int s = kiter % STAGES, use = kiter / STAGES;
      if (use > 0) mbar_wait(&sh.empty[s], (use - 1) & 1, budget, err);
      unsigned char* sa = base + s * STAGE_BYTES;
      unsigned char* sb = sa + A_BYTES;
      const bool valid = ar < tl.rows;
      const void* src = valid ? prob.a_row(sh.scratch, tl, ar, kb) : nullptr;
      R.a_valid = src != nullptr;
      if (P::A_MODE == 1) {
        const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
        for (int c = 0; c < 4; ++c) R.a[c] = src ? __ldg(s4 + ac0 + c) : make_uint4(0, 0, 0, 0);
      } else if (src) {
        const char* s1 = reinterpret_cast<const char*>(src);
#pragma unroll
        for (int c = 0; c < 4; ++c) cp16(sa + swz(ar, ac0 + c), s1 + (ac0 + c) * 16, true);
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4*>(sa + swz(ar, ac0 + c)) = make_uint4(0, 0, 0, 0);
      }
      if (P::B_MODE == 0) {
        const uint8_t* q;
        const uint16_t* sc;
        R.b_valid = pt < BN && prob.b_row(sh.scratch, tl, pt, kb, q, sc);
        if (R.b_valid) {
          R.w0 = ldg_stream(q);
          R.w1 = ldg_stream(q + 16);
          R.s0 = ldg_u16(sc);
          R.s1 = ldg_u16(sc + 1);
        }
      } else {
        for (int n = pt; n < BN; n += NPROD_WARPS * 32) {
          const uint16_t* bsrc = prob.b_row_bf16(sh.scratch, tl, n, kb);
          if (bsrc) {
#pragma unroll
            for (int c = 0; c < 8; ++c) cp16(sb + swz(n, c), bsrc + c * 8, true);
          } else {
#pragma unroll
            for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(sb + swz(n, c)) = make_uint4(0, 0, 0, 0);
          }
        }
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    };
    auto finish = [&](int kiter, const Regs& R) {
      const int s = kiter % STAGES;
      unsigned char* sa = base + s * STAGE_BYTES;
      unsigned char* sb = sa + A_BYTES;
      if (P::A_MODE == 1) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t u[4] = {R.a[c].x, R.a[c].y, R.a[c].z, R.a[c].w};
          uint32_t h[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) h[i] = pack_half2(__uint_as_float(u[i] << 16), __uint_as_float(u[i] & 0xffff0000u));
          *reinterpret_cast<uint4*>(sa + swz(ar, ac0 + c)) = make_uint4(h[0], h[1], h[2], h[3]);
        }
      }
      if (P::B_MODE == 0 && pt < BN) {
        uint4 w0 = make_uint4(0, 0, 0, 0), w1 = w0;
        uint16_t s0 = 0, s1 = 0;
        if (R.b_valid) {
          w0 = R.w0;
          w1 = R.w1;
          s0 = R.s0;
          s1 = R.s1;
        }
        const __half2 h0 = scale_h2(s0), h1 = scale_h2(s1);
        const uint32_t wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // chunk c = elements 8c .. 8c+7 = word c
          uint32_t o[4];
          dequant_word_natural(wv[c], c < 4 ? h0 : h1, o);
          *reinterpret_cast<uint4*>(sb + swz(pt, c)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    };
    int kiter = 0;
    if (t_cur < ntiles) issue(tl_cur, 0, 0, cur);
    while (t_cur < ntiles) {
      // position of the next K block
      int t_n = t_cur, kb_n = kb_cur + 1;
      Tile tl_n = tl_cur;
      if (kb_n == tl_cur.nkb) {
        t_n = t_cur + gridDim.x;
        kb_n = 0;
        if (t_n < ntiles) tl_n = prob.tile(sh.scratch, t_n);
      }
      if (t_n < ntiles) {
        issue(tl_n, kb_n, kiter + 1, nxt);
        asm volatile("cp.async.wait_group 1;" ::: "memory");
      } else {
        asm volatile("cp.async.wait_group 0;" ::: "memory");
      }
      finish(kiter, cur);
      fence_async_smem();
      mbar_arrive(&sh.full[kiter % STAGES]);
      cur = nxt;
      ++kiter;
      t_cur = t_n;
      kb_cur = kb_n;
      tl_cur = tl_n;
    }
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
