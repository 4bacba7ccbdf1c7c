// Top-k with softmax renormalisation of one token's router logits by one warp
// (E <= 512, k <= 16): the k largest logits in descending order, ties going to
// the lower expert index, and w_j = exp(l_j - l_max) / sum of those over the
// selected j.
//
// Each lane holds experts lane, lane + 32, ... as order-preserving integer
// keys. topk_warp_thr gathers the logits at or above a threshold and sorts
// them across the warp; topk_warp, its fallback, runs k rounds in which the
// warp takes the largest remaining key (a warp max reduction), then the
// lowest expert index holding it (a warp min reduction), and only the
// winning lane rescans its keys.
#pragma once
#include "common.cuh"

namespace lmoe {

// order-preserving key of a float (larger float <-> larger unsigned key)
static LMOE_DEV unsigned float_key(float x) {
  const unsigned b = __float_as_uint(x);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
static LMOE_DEV float key_float(unsigned k) { return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k); }

// Lane j < k returns (expert of the j-th pick as int bits, its weight); other
// lanes return (0, 0). `row` holds the token's E logits (read through L2).
// Used where more than 32 logits tie at the k-th place (see topk_warp_thr).
static __device__ __noinline__ float2 topk_warp(const float* row, int E, int k) {
  const int lane = threadIdx.x & 31;
  unsigned key[16];  // element i is expert lane + 32 i; 0 = none (below every finite key)
#pragma unroll
  for (int i = 0; i < 16; ++i) key[i] = lane + 32 * i < E ? float_key(__ldcg(row + lane + 32 * i)) : 0u;
  // this lane's best remaining element (ties to the lower i), recomputed by a
  // linear scan when the lane's head was taken: one copy of the scan keeps
  // the code small
  unsigned bk = 0;
  int bi = 0;
  bool stale = true;
  unsigned sel = 0, k0 = 0;
  int sel_e = 0;
#pragma unroll 1
  for (int j = 0; j < k; ++j) {
    if (stale) {
      bk = key[0];
      bi = 0;
#pragma unroll
      for (int i = 1; i < 16; ++i)
        if (key[i] > bk) {
          bk = key[i];
          bi = i;
        }
      stale = false;
    }
    const unsigned m = __reduce_max_sync(0xffffffffu, bk);
    const int mine = lane + 32 * bi;
    const unsigned wi = __reduce_min_sync(0xffffffffu, bk == m ? (unsigned)mine : 0xffffffffu);
    if ((unsigned)mine == wi) {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (i == bi) key[i] = 0u;
      stale = true;
    }
    if (j == 0) k0 = m;
    if (lane == j) {
      sel = m;
      sel_e = wi < (unsigned)E ? (int)wi : 0;
    }
  }
  const float ex = (lane < k) ? __expf(key_float(sel) - key_float(k0)) : 0.f;
  float z = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  return make_float2(__int_as_float(sel_e), lane < k ? ex / z : 0.f);
}

// The same selection by a threshold: the k-th largest of the 32 lane maxima
// bounds the k-th largest logit from below, so the logits at or above it
// (usually a few more than k) hold the whole answer; they are gathered in
// shared memory and sorted across the warp by (logit desc, expert asc).
// Falls back to topk_warp when more than 32 logits reach the threshold.
// `scratch` is 32 entries of shared memory owned by the calling warp.
static __device__ __noinline__ float2 topk_warp_thr(const float* row, int E, int k, uint2* scratch) {
  const int lane = threadIdx.x & 31;
  unsigned key[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) key[i] = lane + 32 * i < E ? float_key(__ldcg(row + lane + 32 * i)) : 0u;
  unsigned v = key[0];
#pragma unroll
  for (int i = 1; i < 16; ++i) v = max(v, key[i]);
  // bitonic sort of the lane maxima, descending (loops kept rolled: this code
  // runs once per token and its size, not its issue count, is what costs)
#pragma unroll 1
  for (int size = 2; size <= 32; size <<= 1)
#pragma unroll 1
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const unsigned o = __shfl_xor_sync(0xffffffffu, v, stride);
      const bool desc = (lane & size) == 0, lower = (lane & stride) == 0;
      v = (lower == desc) ? max(v, o) : min(v, o);
    }
  const unsigned tau = __shfl_sync(0xffffffffu, v, k - 1);
  int cnt = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) cnt += key[i] >= tau;
  int pre = cnt;  // inclusive prefix over lanes
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, pre, o);
    if (lane >= o) pre += y;
  }
  if (__shfl_sync(0xffffffffu, pre, 31) > 32) return topk_warp(row, E, k);
  int pos = pre - cnt;
#pragma unroll
  for (int i = 0; i < 16; ++i)
    if (key[i] >= tau) scratch[pos++] = make_uint2(key[i], (unsigned)(lane + 32 * i));
  __syncwarp();
  const int C = __shfl_sync(0xffffffffu, pre, 31);
  uint2 cd = lane < C ? scratch[lane] : make_uint2(0u, 0xffffffffu);
  __syncwarp();
  // bitonic sort of the candidates: larger logit first, then lower expert
#pragma unroll 1
  for (int size = 2; size <= 32; size <<= 1)
#pragma unroll 1
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const unsigned ox = __shfl_xor_sync(0xffffffffu, cd.x, stride), oy = __shfl_xor_sync(0xffffffffu, cd.y, stride);
      const bool desc = (lane & size) == 0, lower = (lane & stride) == 0;
      const bool mine_first = cd.x > ox || (cd.x == ox && cd.y < oy);
      if ((lower == desc) != mine_first) cd = make_uint2(ox, oy);
    }
  const unsigned k0 = __shfl_sync(0xffffffffu, cd.x, 0);
  const float ex = (lane < k) ? __expf(key_float(cd.x) - key_float(k0)) : 0.f;
  float z = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  return make_float2(__int_as_float(lane < k && cd.y < (unsigned)E ? (int)cd.y : 0), lane < k ? ex / z : 0.f);
}

}  // namespace lmoe
