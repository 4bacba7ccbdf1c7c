// Shared device helpers for the latent MoE kernels (sm_103a).
//
// Numerics (this library's reading of "int4 tensors" plus fp32 accumulation):
// every int4 weight is dequantised to q*s in fp16, which is exact because q
// has at most 3 significant bits and the bf16 scale s has 8 (q*s needs <= 11,
// fp16 has 11) as long as s lies in fp16's normal range; activations enter
// the tensor cores as fp16 and all accumulation is fp32.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "decode.cuh"

#define LMOE_DEV __device__ __forceinline__

namespace lmoe {

LMOE_DEV float bf16_to_f32(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

LMOE_DEV uint16_t f32_to_bf16_rne(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x7fffffu)) return (uint16_t)((u >> 16) | 0x40);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

LMOE_DEV uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

LMOE_DEV float silu(float a) { return a / (1.0f + __expf(-a)); }

// ---------------------------------------------------------------------------
// int4 -> fp16 dequantisation of one 32-bit word (8 nibbles, element i in
// bits 4i..4i+3). Produces four half2: (e0,e4), (e1,e5), (e2,e6), (e3,e7),
// each already multiplied by the group scale s2 = (s, s).
//   nibble n (two's complement q) -> n ^ 8 = q + 8 = u in [1, 15]
//   0x6400 | u         is the fp16 1024 + u       -> minus 1032 gives q
//   0x6400 | (u << 4)  is the fp16 1024 + 16 u    -> /16 - 72 gives q
// The xor with 8 is folded into the lop3 constant (the magic bits and the
// nibble bits do not overlap).
LMOE_DEV void dequant_word(uint32_t v, __half2 s2, uint32_t out[4]) {
  const uint32_t lo_mask = 0x000F000Fu, hi_mask = 0x00F000F0u;
  uint32_t t0, t1, t2, t3;
  const uint32_t magic_lo = 0x64086408u, magic_hi = 0x64806480u;
  asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(t0) : "r"(v), "r"(lo_mask), "r"(magic_lo));  // (a & b) ^ c
  asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(t1) : "r"(v), "r"(hi_mask), "r"(magic_hi));
  uint32_t w = v >> 8;
  asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(t2) : "r"(w), "r"(lo_mask), "r"(magic_lo));
  asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(t3) : "r"(w), "r"(hi_mask), "r"(magic_hi));
  const __half2 k1032 = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
  const __half2 inv16 = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));
  const __half2 m72 = __halves2half2(__ushort_as_half(0xD480), __ushort_as_half(0xD480));
  __half2 h0 = __hsub2(*reinterpret_cast<__half2*>(&t0), k1032);
  __half2 h1 = __hfma2(*reinterpret_cast<__half2*>(&t1), inv16, m72);
  __half2 h2 = __hsub2(*reinterpret_cast<__half2*>(&t2), k1032);
  __half2 h3 = __hfma2(*reinterpret_cast<__half2*>(&t3), inv16, m72);
  h0 = __hmul2(h0, s2);
  h1 = __hmul2(h1, s2);
  h2 = __hmul2(h2, s2);
  h3 = __hmul2(h3, s2);
  out[0] = *reinterpret_cast<uint32_t*>(&h0);
  out[1] = *reinterpret_cast<uint32_t*>(&h1);
  out[2] = *reinterpret_cast<uint32_t*>(&h2);
  out[3] = *reinterpret_cast<uint32_t*>(&h3);
}

// bf16 scale bits -> (s, s) in fp16
LMOE_DEV __half2 scale_h2(uint16_t sbits) {
  __half h = __float2half_rn(bf16_to_f32(sbits));
  return __halves2half2(h, h);
}

// Four bytes of FP4 E2M1 code pairs -> four half2, one per byte (the byte's
// low nibble in the low half); exact. Hardware conversions (sm_100 and later).
LMOE_DEV void e2m1x8_to_h2x4(uint32_t v, uint32_t out[4]) {
  asm("{ .reg .b8 a0, a1, a2, a3;\n"
      "  mov.b32 {a0, a1, a2, a3}, %4;\n"
      "  cvt.rn.f16x2.e2m1x2 %0, a0;\n"
      "  cvt.rn.f16x2.e2m1x2 %1, a1;\n"
      "  cvt.rn.f16x2.e2m1x2 %2, a2;\n"
      "  cvt.rn.f16x2.e2m1x2 %3, a3; }"
      : "=r"(out[0]), "=r"(out[1]), "=r"(out[2]), "=r"(out[3])
      : "r"(v));
}
// Two FP8 E4M3 bytes -> half2 (the low byte in the low half); exact.
LMOE_DEV uint32_t e4m3x2_to_h2(uint16_t w) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(w));
  return h;
}

// D += A * B, m16n8k16, fp16 inputs, fp32 accumulators
LMOE_DEV void mma16816(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

LMOE_DEV uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

LMOE_DEV uint16_t ldg_u16(const uint16_t* p) {
  uint16_t r;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(r) : "l"(p));
  return r;
}

// ---------------------------------------------------------------------------
// Activation fragments ("B operand" of m16n8k16 with weights as the A
// operand and tokens as N). The reduction dimension K is walked in chunks of
// 128; within a chunk, lane (gid = lane/4, tig = lane%4) of MMA m (0..7)
// holds the weight elements tig*32 + 8*(m/2) + {0,4 | 1,5} (m even) or
// {2,6 | 3,7} (m odd) of rows gid and gid+8 -- the order in which one 16-byte
// load of packed int4 (32 consecutive elements, exactly one scale group)
// dequantises. The matching activation fragment of token n = 8*nt + gid is
// built from the 8 consecutive elements K0 = 128*c + 32*tig + 8*mp, ..., +7
// (mp = m/2) packed as half2 (e0,e4), (e1,e5), (e2,e6), (e3,e7) = one uint4.
// Shared-memory layout: frag[((c*NT + nt)*4 + mp)*32 + lane] (uint4), which a
// warp reads conflict-free.
LMOE_DEV int frag_index(int c, int nt, int mp, int lane, int NT) { return ((c * NT + nt) * 4 + mp) * 32 + lane; }

LMOE_DEV uint4 pack_frag8(const float e[8]) {
  uint4 r;
  r.x = pack_half2(e[0], e[4]);
  r.y = pack_half2(e[1], e[5]);
  r.z = pack_half2(e[2], e[6]);
  r.w = pack_half2(e[3], e[7]);
  return r;
}

// acc[nt][*] += W[r0..r0+15][chunks c0..c1) * frags. W is packed int4 with
// row stride K/2 bytes and scales [rows][K/32]; K a multiple of 32 (lanes
// whose 32-element slice lies beyond K contribute zero). The fragment array
// base corresponds to chunk cf0 (frag chunk index = c - cf0). Weight loads
// run PF chunks ahead of the tensor-core work (a register ring).
template <int NT, int PF = 4>
LMOE_DEV void mma_rows(const uint8_t* __restrict__ q, const uint16_t* __restrict__ s, int K, int r0, int c0, int c1,
                       int cf0, const uint4* __restrict__ frag, float acc[NT][4]) {
  const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
  const size_t rs = (size_t)(K >> 1), ss = (size_t)(K >> 5);
  const uint8_t* q0 = q + (size_t)(r0 + gid) * rs + tig * 16;
  const uint8_t* q8 = q0 + 8 * rs;
  const uint16_t* s0 = s + (size_t)(r0 + gid) * ss + tig;
  const uint16_t* s8 = s0 + 8 * ss;
  uint4 w0[PF], w8[PF];
  uint16_t sc0[PF], sc8[PF];
  auto load = [&](int c, uint4& a, uint4& b, uint16_t& sa, uint16_t& sb) {
    if (c < c1 && c * 128 + tig * 32 < K) {
      a = ldg_stream(q0 + (size_t)c * 64);
      b = ldg_stream(q8 + (size_t)c * 64);
      sa = ldg_u16(s0 + c * 4);
      sb = ldg_u16(s8 + c * 4);
    } else {
      a = make_uint4(0, 0, 0, 0);
      b = a;
      sa = 0;
      sb = 0;
    }
  };
#pragma unroll
  for (int i = 0; i < PF; ++i) load(c0 + i, w0[i], w8[i], sc0[i], sc8[i]);
  for (int cb = c0; cb < c1; cb += PF) {
#pragma unroll
    for (int i = 0; i < PF; ++i) {
      const int c = cb + i;
      if (c < c1) {
        const uint32_t wa[4] = {w0[i].x, w0[i].y, w0[i].z, w0[i].w};
        const uint32_t wb[4] = {w8[i].x, w8[i].y, w8[i].z, w8[i].w};
        const __half2 h0 = scale_h2(sc0[i]), h8 = scale_h2(sc8[i]);
        load(c + PF, w0[i], w8[i], sc0[i], sc8[i]);
#pragma unroll
        for (int mp = 0; mp < 4; ++mp) {
          uint32_t A[4], B8[4];
          dequant_word(wa[mp], h0, A);
          dequant_word(wb[mp], h8, B8);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const uint4 b = frag[frag_index(c - cf0, nt, mp, lane, NT)];
            mma16816(acc[nt], A[0], B8[0], A[1], B8[1], b.x, b.y);  // m = 2mp
            mma16816(acc[nt], A[2], B8[2], A[3], B8[3], b.z, b.w);  // m = 2mp + 1
          }
        }
      }
    }
  }
}

LMOE_DEV void set_error(unsigned* err, unsigned bits) {
  if (err) atomicOr(err, bits);
}

// ------------------------------------------------------------- mbarriers
LMOE_DEV uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

LMOE_DEV void mbar_init(uint64_t* m, uint32_t cnt) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(m)), "r"(cnt));
}
LMOE_DEV void mbar_arrive(uint64_t* m) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(smem_u32(m)) : "memory");
}
// n arrivals at once
LMOE_DEV void mbar_arrive_n(uint64_t* m, uint32_t n) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0], %1; }" ::"r"(smem_u32(m)), "r"(n)
               : "memory");
}
// bounded wait for the phase with the given parity to complete
LMOE_DEV void mbar_wait(uint64_t* m, uint32_t parity, long long budget, unsigned* err) {
  const long long t0 = clock64();
  while (true) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_u32(m)), "r"(parity)
        : "memory");
    if (ok) return;
    if (clock64() - t0 > budget) {
      set_error(err, ERRBIT_TIMEOUT);
      return;
    }
  }
}

}  // namespace lmoe
