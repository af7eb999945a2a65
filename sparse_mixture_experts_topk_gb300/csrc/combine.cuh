// Combine body of the combine kernel.
//
// out[t] = sum_j w[t, j] * y_perm[pos[t, j]] for the K slots of token t
// (a dropped slot, pos < 0, adds nothing), summed in fp32 in slot order j =
// 0..K-1 (Qwen2-MoE code walkthrough, jsqmd.com, section 3.1 item 2; MoE
// sparse-activation article, wmrh.cn, section 2.2, Dispatcher).
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kCombineUnroll = 4;
constexpr int kCombineChunk = 32 * kCombineUnroll;   // 16-byte vectors a warp covers per round

// Work items (token, column chunk of chunk_vec vectors; chunk_vec a multiple
// of kCombineChunk) taken by warps w0, w0 + nw, ... of the caller.  KP: K
// rounded up to 2, 4 or 8 so the slot arrays stay in registers.
template <typename T, int KP>
__device__ __forceinline__ void combine_items(const uint4* __restrict__ y_perm, const int32_t* __restrict__ pos,
                                              const float* __restrict__ w, int64_t Tn, int K, int vec_per_row,
                                              int chunk_vec, uint4* __restrict__ out, int64_t w0, int64_t nw) {
  constexpr int V = Vec<T>::N;
  const int lane = threadIdx.x & 31;
  const int nchunk = (vec_per_row + chunk_vec - 1) / chunk_vec;
  const int64_t items = Tn * nchunk;
  for (int64_t it = w0; it < items; it += nw) {
    const int64_t t = it / nchunk;
    const int c0 = (int)(it % nchunk) * chunk_vec;
    const int c1 = min(vec_per_row, c0 + chunk_vec);
    int p[KP];
    float wt[KP];
#pragma unroll
    for (int j = 0; j < KP; ++j) {
      if (j < K) {
        p[j] = pos[t * K + j];
        wt[j] = w[t * K + j];
      }
    }
    for (int v0 = c0 + lane; v0 < c1; v0 += kCombineChunk) {
      float acc[kCombineUnroll][V];
#pragma unroll
      for (int u = 0; u < kCombineUnroll; ++u)
#pragma unroll
        for (int i = 0; i < V; ++i) acc[u][i] = 0.f;
#pragma unroll
      for (int j = 0; j < KP; ++j) {
        if (j < K && p[j] >= 0) {
          uint4 raw[kCombineUnroll];
#pragma unroll
          for (int u = 0; u < kCombineUnroll; ++u) {
            const int v = v0 + 32 * u;
            if (v < c1) raw[u] = __ldcs(y_perm + (int64_t)p[j] * vec_per_row + v);
          }
#pragma unroll
          for (int u = 0; u < kCombineUnroll; ++u) {
            const int v = v0 + 32 * u;
            if (v < c1) {
              float f[V];
              Vec<T>::unpack(raw[u], f);
#pragma unroll
              for (int i = 0; i < V; ++i) acc[u][i] = fmaf(wt[j], f[i], acc[u][i]);
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kCombineUnroll; ++u) {
        const int v = v0 + 32 * u;
        if (v < c1) __stcs(out + t * vec_per_row + v, Vec<T>::pack(acc[u]));
      }
    }
  }
}

// Vectors per work item: a quarter of a 3584-wide bf16 row (kCombineChunk).
// Items this small keep every warp of a persistent grid busy to the end
// (8192 tokens make 32768 items for 3648 warps, nine rounds), where whole-row
// items left the last of 2.25 waves a quarter full; re-reading a token's pos
// and w per item costs 16 bytes.
__host__ __device__ inline int combine_chunk() { return kCombineChunk; }

}  // namespace moe
