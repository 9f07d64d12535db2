// Softmax and top-k of one token's logits by one warp: shared by the top-k kernel and the
// fused decode router, so both give the same bits.
#pragma once

#include "common.cuh"

namespace moe {

// (v, i) beats (w, j) when v > w, or v == w and i < j: descending logit, ties to lower index.
__device__ __forceinline__ bool beats(float v, int i, float w, int j) {
  return v > w || (v == w && i < j);
}

__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    int i2 = __shfl_xor_sync(0xffffffffu, i, o);
    if (beats(v2, i2, v, i)) { v = v2; i = i2; }
  }
}

struct TopK {
  int idx[2];
  float w[2];
};

// Warp-collective over the row l[0 .. E-1] (read through `ld`); every lane returns the same
// result.  Selection on the logits (ties to the lower index); k = 1: w = p[e1] = 1 / sum of
// exp(l - l_max); k = 2: w_j = p_j / (p_1 + p_2).  probs_row / copy_row (nullable) receive
// the softmax / a copy of the logits.
template <typename Load>
__device__ __forceinline__ TopK softmax_topk_warp(const float* l, int E, int k, int lane, Load ld,
                                                  float* probs_row, float* copy_row) {
  float v1 = -INFINITY;
  int i1 = 0x7fffffff;
  for (int e = lane; e < E; e += 32) {
    float v = ld(l + e);
    if (copy_row) copy_row[e] = v;
    if (beats(v, e, v1, i1)) { v1 = v; i1 = e; }
  }
  warp_argmax(v1, i1);
  float v2 = -INFINITY;
  int i2 = 0x7fffffff;
  if (k == 2) {
    for (int e = lane; e < E; e += 32) {
      float v = ld(l + e);
      if (e != i1 && beats(v, e, v2, i2)) { v2 = v; i2 = e; }
    }
    warp_argmax(v2, i2);
  }
  float s = 0.0f;
  for (int e = lane; e < E; e += 32) s += expf(ld(l + e) - v1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (probs_row) {
    float inv = 1.0f / s;
    for (int e = lane; e < E; e += 32) probs_row[e] = expf(ld(l + e) - v1) * inv;
  }
  TopK r;
  r.idx[0] = i1;
  r.idx[1] = i2;
  if (k == 1) {
    r.w[0] = 1.0f / s;                              // p[e1] = exp(0) / sum
    r.w[1] = 0.0f;
  } else {
    float q = expf(v2 - v1);                        // p2 / p1
    float z = 1.0f + q;
    r.w[0] = 1.0f / z;
    r.w[1] = q / z;
  }
  return r;
}

}  // namespace moe
