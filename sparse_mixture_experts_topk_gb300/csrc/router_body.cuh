// Router bodies shared by the decode-sized router kernel and the one-launch
// decode layer: the token finish (top-k, softmax, renormalised weights) and
// the (gate row, piece) dot products, so both compute every score, id and
// weight with the same operations in the same order.
//
// Qwen2-MoE code walkthrough (jsqmd.com), section 3.1: the gate is a
// bias-free nn.Linear(hidden, num_experts); its scores go through a softmax,
// torch.topk picks num_experts_per_tok experts, and the k probabilities are
// divided by their sum.
#pragma once

#include <float.h>

#include "bf16_dot.cuh"
#include "common.cuh"

namespace moe {
namespace route {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One warp per token: ls holds nt rows of E fp32 scores (row pitch E + 1).
// Lane l reads experts l, l + 32, ...  Pick j is a warp arg-max over the
// entries ranked after pick j - 1 in (score descending, index ascending)
// order, so no entry is taken twice; lane j keeps pick j.  The token's ids
// and weights are written, and its ls row is replaced by the full softmax
// (for the load-balancing sums).  Loops are kept rolled: the routers run
// once per layer with their code cold, and straight-line code costs more to
// fetch than the loop overhead it saves.
// s_hist (nullable, shared): counts of the chosen experts.
__device__ __forceinline__ void finish_tokens(float* ls, int nt, int64_t t0, int E, int K, float inv_tau,
                                              int32_t* __restrict__ ids, float* __restrict__ w, int warp0,
                                              int nwarps, int* s_hist = nullptr) {
  const int lane = threadIdx.x & 31;
#pragma unroll 1
  for (int tt = warp0; tt < nt; tt += nwarps) {
    float* row = ls + tt * (E + 1);
    float prev_v = INFINITY, my_v = -INFINITY;
    int prev_i = -1, my_id = 0x7fffffff;
#pragma unroll 1
    for (int j = 0; j < K; ++j) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll 1
      for (int e = lane; e < E; e += 32) {
        const float v = row[e];
        const bool after = v < prev_v || (v == prev_v && e > prev_i);
        if (after && (v > bv || (v == bv && e < bi))) {
          bv = v;
          bi = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) {
          bv = ov;
          bi = oi;
        }
      }
      if (lane == j) {
        my_v = bv;
        my_id = bi;
      }
      prev_v = bv;
      prev_i = bi;
    }
    const float m = __shfl_sync(0xffffffffu, my_v, 0);   // the first pick is the largest score
    float zs = 0.f;
#pragma unroll 1
    for (int e = lane; e < E; e += 32) {
      const float z = expf((row[e] - m) * inv_tau);
      row[e] = z;
      zs += z;
    }
    zs = warp_sum(zs);
    const float inv = 1.f / zs;
#pragma unroll 1
    for (int e = lane; e < E; e += 32) row[e] *= inv;
    const float z = lane < K ? expf((my_v - m) * inv_tau) : 0.f;
    float zsel = 0.f;
#pragma unroll 1
    for (int j = 0; j < K; ++j) zsel += __shfl_sync(0xffffffffu, z, j);
    if (lane < K) {
      const int64_t t = t0 + tt;
      ids[t * K + lane] = my_id;
      w[t * K + lane] = z / zsel;
      if (s_hist && (unsigned)my_id < (unsigned)E) atomicAdd(&s_hist[my_id], 1);   // NaN scores: none
    }
  }
}

constexpr int kSmallTok = 16;
constexpr int kSmallChunk = 8;
constexpr int kSmallMaxCta = 8;

// pieces of 32 * kSmallChunk 16-byte vectors per gate row of H bf16
__host__ __device__ inline int small_pieces(int H) { return (H / 8 + 32 * kSmallChunk - 1) / (32 * kSmallChunk); }

// One (gate row e, piece c) unit: the piece (gw, vectors c0 + lane + 32 u)
// dotted with each token row t < Tn <= MR of xs (shared or global memory),
// summed over the warp; lane 0 hands each token's score piece to
// store(t, v).  MR fixes the body's size, so a small batch runs (and
// fetches) a small body.
template <int MR, typename Store>
__device__ __forceinline__ void small_unit(const uint4 (&gw)[kSmallChunk], const uint4* xs, int kv, int c0,
                                           int Tn, Store store) {
  const int lane = threadIdx.x & 31;
  float acc[MR];
#pragma unroll
  for (int t = 0; t < MR; ++t) acc[t] = 0.f;
#pragma unroll
  for (int u = 0; u < kSmallChunk; ++u) {
    const int v = c0 + lane + 32 * u;
    if (v < kv) {
#pragma unroll
      for (int t = 0; t < MR; ++t)
        if (t < Tn) acc[t] = fma8_bf16(xs[t * kv + v], gw[u], acc[t]);
    }
  }
#pragma unroll
  for (int t = 0; t < MR; ++t) {
    if (t < Tn) {
      float v = acc[t];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) store(t, v);
    }
  }
}

// The unit for a batch of Tn tokens, with the smallest body that holds it.
template <typename Store>
__device__ __forceinline__ void small_unit_any(const uint4 (&gw)[kSmallChunk], const uint4* xs, int kv, int c0,
                                               int Tn, Store store) {
  if (Tn <= 1) small_unit<1>(gw, xs, kv, c0, Tn, store);
  else if (Tn <= 2) small_unit<2>(gw, xs, kv, c0, Tn, store);
  else if (Tn <= 4) small_unit<4>(gw, xs, kv, c0, Tn, store);
  else if (Tn <= 8) small_unit<8>(gw, xs, kv, c0, Tn, store);
  else small_unit<kSmallTok>(gw, xs, kv, c0, Tn, store);
}

}  // namespace route
}  // namespace moe
