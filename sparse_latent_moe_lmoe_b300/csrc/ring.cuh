// A shared-memory weight ring for the decode path: one producer thread
// streams the CTA's weight chunks into fixed slots with TMA tensor copies
// (cp.async.bulk.tensor, completing on the slot's "full" mbarrier with a
// transaction count), far ahead of the warps that consume them; a consuming
// warp hands the slot back through its "empty" mbarrier.
//
// A chunk of packed 4-bit codes in a slot is in the 128-byte swizzle: row r
// of the chunk is LPR 128-byte lines (line i = r*LPR + k/256 for element k),
// and 16-byte unit j of line i sits at unit j ^ (i & 7), so the 16-byte loads
// of the 8 rows a warp reads at once fall in different banks. The chunk's
// scales ([rows][K/32] 16-bit words: one bf16 for int4, two E4M3 bytes for
// NVFP4) follow it in the slot, unswizzled.
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

// Bulk (untiled) copy of `bytes` from global into shared memory, completing
// on mbarrier m; both addresses 16-byte aligned, bytes a multiple of 16.
LMOE_DEV void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* m, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(m)), "l"(pol)
      : "memory");
}
// Prefetch of `bytes` of global memory into L2 (same alignment rules).
LMOE_DEV void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

LMOE_DEV bool mbar_test(uint64_t* m, uint32_t parity) {
  uint32_t ok;
  asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
               : "=r"(ok)
               : "r"(smem_u32(m)), "r"(parity)
               : "memory");
  return ok != 0;
}

// Weight formats of a chunk: 0 = int4 with one bf16 scale per 32 elements; 1
// = NVFP4 (E2M1 codes with one E4M3 scale per 16 elements). A lane's 16-bit
// scale word covers the same 32 elements in both: one bf16, or two E4M3
// bytes (the low byte for the first 16).
//
// NVFP4 words are stored with byte b holding elements b (low nibble) and
// b + 4 (high nibble), so one hardware conversion per byte yields the half2
// (e_b, e_{b+4}) that the fragments pair (the order dequant_word produces).
LMOE_DEV void dequant_fp4_word(uint32_t v, __half2 s2, uint32_t out[4]) {
  e2m1x8_to_h2x4(v, out);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 h = __hmul2(*reinterpret_cast<__half2*>(&out[i]), s2);  // code * scale: exact in fp16
    out[i] = *reinterpret_cast<uint32_t*>(&h);
  }
}

// a lane's scale word -> the half2 scales of its first and second 16 elements
template <int WF>
LMOE_DEV void lane_scales(uint16_t w, __half2& first, __half2& second) {
  if (WF == 0) {
    first = second = scale_h2(w);
  } else {
    const uint32_t h = e4m3x2_to_h2(w);
    const __half2 hh = *reinterpret_cast<const __half2*>(&h);
    first = __low2half2(hh);
    second = __high2half2(hh);
  }
}

template <int WF>
LMOE_DEV void dequant_any(uint32_t v, __half2 s2, uint32_t out[4]) {
  if (WF == 0)
    dequant_word(v, s2, out);
  else
    dequant_fp4_word(v, s2, out);
}

// acc[nt] += W[16 rows][chunks c0 .. c0+nc of 128 elements] * fragments,
// with W in a ring slot as a TMA box in 128-byte swizzle: row r of the box is
// LPR 128-byte lines (line i = r*LPR + k/256 for element k of the box), and
// 16-byte unit j of line i sits at unit j ^ (i & 7). `w` is the (1024-byte
// aligned) slot base, row0 the first row of the tile, `s` the box's scales
// [rows][SS]. Chunk c0 + c of the box meets fragment chunk c of `frag` (see
// frag_index; the caller offsets `frag` to the box's chunk c0).
template <int NT, int WF>
LMOE_DEV void mma_slot(const unsigned char* w, int LPR, int row0, const uint16_t* s, int SS, int c0, int nc,
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
    const int cc = c0 + c;
    const int i0 = r0 * LPR + (cc >> 1), i8 = r8 * LPR + (cc >> 1), j = ((cc & 1) << 2) | tig;
    a = *reinterpret_cast<const uint4*>(w + i0 * 128 + ((j ^ (i0 & 7)) << 4));
    b = *reinterpret_cast<const uint4*>(w + i8 * 128 + ((j ^ (i8 & 7)) << 4));
    sa = s0[cc * 4];
    sb = s8[cc * 4];
  };
  uint4 a = make_uint4(0u, 0u, 0u, 0u), b = a;
  uint16_t sa = 0, sb = 0;
  if (nc > 0) ld(0, a, b, sa, sb);
#pragma unroll 1
  for (int c = 0; c < nc; ++c) {
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w};
    const uint32_t wb[4] = {b.x, b.y, b.z, b.w};
    __half2 h0a, h0b, h8a, h8b;  // scales of rows r0 / r8, first and second 16 elements
    lane_scales<WF>(sa, h0a, h0b);
    lane_scales<WF>(sb, h8a, h8b);
    if (c + 1 < nc) ld(c + 1, a, b, sa, sb);
    uint4 fv[4][NT];
#pragma unroll
    for (int mp = 0; mp < 4; ++mp)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) fv[mp][nt] = frag[frag_index(c, nt, mp, lane, NT)];
#pragma unroll
    for (int mp = 0; mp < 4; ++mp) {
      uint32_t A[4], B8[4];
      dequant_any<WF>(wa[mp], mp < 2 ? h0a : h0b, A);
      dequant_any<WF>(wb[mp], mp < 2 ? h8a : h8b, B8);
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

// acc[nt] += W[16 rows m*16 ..][32 elements] * v, for a matrix slice of 32
// reduction elements per row held as [rows][16 bytes] (row r's 32 packed
// codes at byte 16 r) with one scale word per row, `sc`. Lane (gid, tig) reads word
// tig of rows gid and gid+8 -- elements 8 tig .. 8 tig + 7 -- so the matching
// activation entry vfr[nt*32 + lane] holds elements 8 tig .. 8 tig + 7 of
// token 8 nt + gid, packed as (e0,e4) (e1,e5) (e2,e6) (e3,e7).
template <int NT, int WF>
LMOE_DEV void mma_slice32(const uint32_t* wsl, const uint16_t* sc, int m, const uint4* vfr, float acc[NT][4]) {
  const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
  const int r0 = 16 * m + gid, r8 = r0 + 8;
  uint32_t A[4], B8[4];
  __half2 s0a, s0b, s8a, s8b;  // word tig holds elements 8 tig .. 8 tig + 7: the first 16 for tig < 2
  lane_scales<WF>(sc[r0], s0a, s0b);
  lane_scales<WF>(sc[r8], s8a, s8b);
  dequant_any<WF>(wsl[r0 * 4 + tig], tig < 2 ? s0a : s0b, A);
  dequant_any<WF>(wsl[r8 * 4 + tig], tig < 2 ? s8a : s8b, B8);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const uint4 f = vfr[nt * 32 + lane];
    mma16816(acc[nt], A[0], B8[0], A[1], B8[1], f.x, f.y);
    mma16816(acc[nt], A[2], B8[2], A[3], B8[3], f.z, f.w);
  }
}

}  // namespace lmoe
