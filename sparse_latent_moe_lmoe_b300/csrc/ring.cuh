// A shared-memory weight ring for the decode path: one producer thread
// streams the CTA's weight chunks into fixed slots with TMA tensor copies
// (cp.async.bulk.tensor, completing on the slot's "full" mbarrier with a
// transaction count), far ahead of the warps that consume them; a consuming
// warp hands the slot back through its "empty" mbarrier.
//
// An int4 chunk in a slot is a TMA box in 128-byte swizzle: row r of the
// chunk is LPR 128-byte lines (line i = r*LPR + k/256 for element k), and
// 16-byte unit j of line i sits at unit j ^ (i & 7), so the 16-byte loads of
// the 8 rows a warp reads at once fall in different banks. The chunk's bf16
// scales, [rows][K/32], follow it in the slot as a second, unswizzled box.
#pragma once
#include "common.cuh"

namespace lmoe {

LMOE_DEV void mbar_expect_tx(uint64_t* m, uint32_t bytes) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(smem_u32(m)),
               "r"(bytes)
               : "memory");
}

// TMA tensor loads (tile mode) completing on mbarrier m; coordinates
// innermost first. The tensor map lives in kernel parameter space.
LMOE_DEV void tma_load_2d(void* dst, const void* tmap, int c0, int c1, uint64_t* m) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(smem_u32(dst)),
      "l"(tmap), "r"(c0), "r"(c1), "r"(smem_u32(m))
      : "memory");
}
LMOE_DEV void tma_load_3d(void* dst, const void* tmap, int c0, int c1, int c2, uint64_t* m) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(m))
      : "memory");
}

// An L2 policy under which the lines a copy brings in are evicted first
// (data read once per pass, such as weights streamed through a ring).
LMOE_DEV uint64_t l2_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
LMOE_DEV void tma_load_2d_hint(void* dst, const void* tmap, int c0, int c1, uint64_t* m, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(c0), "r"(c1), "r"(smem_u32(m)), "l"(pol)
      : "memory");
}
LMOE_DEV void tma_load_3d_hint(void* dst, const void* tmap, int c0, int c1, int c2, uint64_t* m, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(m)), "l"(pol)
      : "memory");
}

// Prefetch of one tensor-map box into L2 (no shared-memory destination).
LMOE_DEV void tma_prefetch_2d(const void* tmap, int c0, int c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(tmap), "r"(c0), "r"(c1)
               : "memory");
}
LMOE_DEV void tma_prefetch_3d(const void* tmap, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(tmap), "r"(c0), "r"(c1),
               "r"(c2)
               : "memory");
}

LMOE_DEV bool mbar_test(uint64_t* m, uint32_t parity) {
  uint32_t ok;
  asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
               : "=r"(ok)
               : "r"(smem_u32(m)), "r"(parity)
               : "memory");
  return ok != 0;
}

// acc[nt] += W[16 rows][128*nc elements] * fragments (see frag_index; chunk c
// of the slot uses fragment chunk c), with W in a ring slot as a TMA box with
// 128-byte swizzle: row r of the chunk is LPR 128-byte lines (line i = r*LPR
// + k/256 for element k), and 16-byte unit j of line i sits at unit
// j ^ (i & 7). `w` is the (1024-byte aligned) slot base, row0 the first row
// of the tile, `s` the chunk's scales [rows][SS].
template <int NT>
LMOE_DEV void mma_ring_rows_swz(const unsigned char* w, int LPR, int row0, const uint16_t* s, int SS, int nc,
                                const uint4* frag, float acc[NT][4]) {
  const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
  const int r0 = row0 + gid, r8 = r0 + 8;
  const uint16_t* s0 = s + r0 * SS + tig;
  const uint16_t* s8 = s + r8 * SS + tig;
  float acc2[NT][4];  // a second accumulator chain (odd m) halves the MMA dependency chain
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int h = 0; h < 4; ++h) acc2[nt][h] = 0.f;
  // the next chunk's weights and scales are loaded while this one is contracted
  auto ld = [&](int c, uint4& a, uint4& b, uint16_t& sa, uint16_t& sb) {
    const int i0 = r0 * LPR + (c >> 1), i8 = r8 * LPR + (c >> 1), j = ((c & 1) << 2) | tig;
    a = *reinterpret_cast<const uint4*>(w + i0 * 128 + ((j ^ (i0 & 7)) << 4));
    b = *reinterpret_cast<const uint4*>(w + i8 * 128 + ((j ^ (i8 & 7)) << 4));
    sa = s0[c * 4];
    sb = s8[c * 4];
  };
  uint4 a, b;
  uint16_t sa, sb;
  ld(0, a, b, sa, sb);
#pragma unroll 1
  for (int c = 0; c < nc; ++c) {
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w};
    const uint32_t wb[4] = {b.x, b.y, b.z, b.w};
    const __half2 h0 = scale_h2(sa), h8 = scale_h2(sb);
    if (c + 1 < nc) ld(c + 1, a, b, sa, sb);
    uint4 fv[4][NT];
#pragma unroll
    for (int mp = 0; mp < 4; ++mp)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) fv[mp][nt] = frag[frag_index(c, nt, mp, lane, NT)];
#pragma unroll
    for (int mp = 0; mp < 4; ++mp) {
      uint32_t A[4], B8[4];
      dequant_word(wa[mp], h0, A);
      dequant_word(wb[mp], h8, B8);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint4 f = fv[mp][nt];
        mma16816(acc[nt], A[0], B8[0], A[1], B8[1], f.x, f.y);
        mma16816(acc2[nt], A[2], B8[2], A[3], B8[3], f.z, f.w);
      }
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int h = 0; h < 4; ++h) acc[nt][h] += acc2[nt][h];
}

// Two matrices (same shape, same activations) in one pass: the fragment
// loads are shared and the two accumulator chains interleave.
template <int NT>
LMOE_DEV void mma_ring_rows_swz2(const unsigned char* w1, const uint16_t* s1, const unsigned char* w2,
                                 const uint16_t* s2, int LPR, int SS, int nc, const uint4* frag, float acc1[NT][4],
                                 float acc2[NT][4]) {
  const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
  const int r0 = gid, r8 = gid + 8;
  const uint16_t* s10 = s1 + r0 * SS + tig;
  const uint16_t* s18 = s1 + r8 * SS + tig;
  const uint16_t* s20 = s2 + r0 * SS + tig;
  const uint16_t* s28 = s2 + r8 * SS + tig;
  auto ld = [&](int c, uint4& a, uint4& b, uint4& a2, uint4& b2, uint16_t (&sc)[4]) {
    const int i0 = r0 * LPR + (c >> 1), i8 = r8 * LPR + (c >> 1), j = ((c & 1) << 2) | tig;
    const int o0 = i0 * 128 + ((j ^ (i0 & 7)) << 4), o8 = i8 * 128 + ((j ^ (i8 & 7)) << 4);
    a = *reinterpret_cast<const uint4*>(w1 + o0);
    b = *reinterpret_cast<const uint4*>(w1 + o8);
    a2 = *reinterpret_cast<const uint4*>(w2 + o0);
    b2 = *reinterpret_cast<const uint4*>(w2 + o8);
    sc[0] = s10[c * 4];
    sc[1] = s18[c * 4];
    sc[2] = s20[c * 4];
    sc[3] = s28[c * 4];
  };
  uint4 a, b, a2, b2;
  uint16_t sc[4];
  ld(0, a, b, a2, b2, sc);
#pragma unroll 1
  for (int c = 0; c < nc; ++c) {
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
    const uint32_t va[4] = {a2.x, a2.y, a2.z, a2.w}, vb[4] = {b2.x, b2.y, b2.z, b2.w};
    const __half2 h0 = scale_h2(sc[0]), h8 = scale_h2(sc[1]), g0 = scale_h2(sc[2]), g8 = scale_h2(sc[3]);
    if (c + 1 < nc) ld(c + 1, a, b, a2, b2, sc);
    uint4 fv[4][NT];
#pragma unroll
    for (int mp = 0; mp < 4; ++mp)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) fv[mp][nt] = frag[frag_index(c, nt, mp, lane, NT)];
#pragma unroll
    for (int mp = 0; mp < 4; ++mp) {
      uint32_t A[4], B8[4], C[4], D8[4];
      dequant_word(wa[mp], h0, A);
      dequant_word(wb[mp], h8, B8);
      dequant_word(va[mp], g0, C);
      dequant_word(vb[mp], g8, D8);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint4 f = fv[mp][nt];
        mma16816(acc1[nt], A[0], B8[0], A[1], B8[1], f.x, f.y);
        mma16816(acc2[nt], C[0], D8[0], C[1], D8[1], f.x, f.y);
        mma16816(acc1[nt], A[2], B8[2], A[3], B8[3], f.z, f.w);
        mma16816(acc2[nt], C[2], D8[2], C[3], D8[3], f.z, f.w);
      }
    }
  }
}

// Transpose a warp's m16n8 accumulators (rows r0..r0+15 of an activation
// that is the reduction dimension of the next contraction, tokens 8*nt + ..)
// into this lane's fragment entry: lane = 2*n + run holds rows r0 + 8*run ..
// + 7 of token n (n < 8*NT). Returns the 8 values in e[].
template <int NT>
LMOE_DEV void acc_to_entry(const float acc[NT][4], float e[8]) {
  const int lane = threadIdx.x & 31, run = lane & 1, n = lane >> 1;
  const int want = run * 2 + (n & 1), src_t = (n & 7) >> 1, want_nt = n >> 3;
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    float v = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float x = __shfl_sync(0xffffffffu, acc[nt][h], g * 4 + src_t);
        if (nt == want_nt && h == want) v = x;
      }
    e[g] = v;
  }
}

}  // namespace lmoe
