// Combine (weighted unpermute) and the load-balancing loss.
//
// Combine: the k expert outputs of a token are summed with the renormalised
// routing weights (Qwen2-MoE code walkthrough, jsqmd.com, section 3.1 item 2;
// MoE sparse-activation article, wmrh.cn, section 2.2, Dispatcher).  A slot
// that the capacity dropped contributes nothing.  The sum runs in fp32 in the
// order j = 0..K-1, so the result is deterministic.
//
// Loss: jsqmd.com section 3.3, load_balancing_loss: E * sum_i f_i * P_i with
// P_i the mean router probability of expert i and f_i its share of the slots.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

// One warp per (token, column chunk) of chunk_vec 16-byte vectors (a multiple
// of kChunkVec; 4 vectors per lane per round): a large batch takes whole
// rows, so each warp reads its token's pos and w once; a small batch cuts
// rows into kChunkVec chunks so that it still spreads over many warps and
// each warp needs one round of loads.
constexpr int kUnroll = 4;
constexpr int kChunkVec = 32 * kUnroll;

// KP: K rounded up to 2, 4 or 8 (the slot arrays stay in registers).
template <typename T, int KP>
__global__ void __launch_bounds__(256, 3)   // 3 blocks (24 warps) an SM: the loads in flight set the speed
combine_kernel(const uint4* __restrict__ y_perm, const int32_t* __restrict__ pos,
               const float* __restrict__ w, int64_t Tn, int K, int vec_per_row, int chunk_vec,
               uint4* __restrict__ out) {
  constexpr int V = Vec<T>::N;
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int nchunk = (vec_per_row + chunk_vec - 1) / chunk_vec;
  const int64_t items = Tn * nchunk;
  const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t it = warp0; it < items; it += nwarps) {
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
    for (int v0 = c0 + lane; v0 < c1; v0 += kChunkVec) {
      float acc[kUnroll][V];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
#pragma unroll
        for (int i = 0; i < V; ++i) acc[u][i] = 0.f;
#pragma unroll
      for (int j = 0; j < KP; ++j) {
        if (j < K && p[j] >= 0) {
          uint4 raw[kUnroll];
#pragma unroll
          for (int u = 0; u < kUnroll; ++u) {
            const int v = v0 + 32 * u;
            if (v < c1) raw[u] = __ldcs(y_perm + (int64_t)p[j] * vec_per_row + v);
          }
#pragma unroll
          for (int u = 0; u < kUnroll; ++u) {
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
      for (int u = 0; u < kUnroll; ++u) {
        const int v = v0 + 32 * u;
        if (v < c1) __stcs(out + t * vec_per_row + v, Vec<T>::pack(acc[u]));
      }
    }
  }
}

__global__ void aux_kernel(const float* __restrict__ psum, const int32_t* __restrict__ count,
                           int E, int64_t Tn, int K, float* __restrict__ loss) {
  __shared__ float sa[256];
  pdl_enter();
  const int e = threadIdx.x;
  sa[e] = (e < E && Tn > 0) ? ((float)count[e] / (float)(Tn * K)) * (psum[e] / (float)Tn) : 0.f;
  __syncthreads();
  for (int o = 128; o > 0; o >>= 1) {
    if (e < o) sa[e] += sa[e + o];
    __syncthreads();
  }
  if (e == 0) *loss = (float)E * sa[0];
}

}  // namespace

cudaError_t launch_combine(const Shape& s, const void* y_perm, const int32_t* pos, const float* w,
                           void* out, cudaStream_t st) {
  if (s.T == 0) return cudaSuccess;
  const int vec = (int)((int64_t)s.H * s.esize() / 16);
  const int64_t cap = (int64_t)sm_count() * 8;    // blocks of 8 warps
  const int64_t small_items = s.T * ((vec + kChunkVec - 1) / kChunkVec);
  const int chunk = small_items <= cap * 8 ? kChunkVec : (vec + kChunkVec - 1) / kChunkVec * kChunkVec;
  const int64_t items = s.T * ((vec + chunk - 1) / chunk);
  int64_t grid = (items + 7) / 8;
  if (grid > cap) grid = cap;
  auto kern = s.dtype == MOE_BF16 ? (s.K <= 2 ? combine_kernel<bf16, 2>
                                               : s.K <= 4 ? combine_kernel<bf16, 4> : combine_kernel<bf16, 8>)
                                   : (s.K <= 2 ? combine_kernel<float, 2>
                                               : s.K <= 4 ? combine_kernel<float, 4> : combine_kernel<float, 8>);
  return launch_kernel(kern, dim3((unsigned)grid), dim3(256), 0, st, 1, (const uint4*)y_perm, pos, w, s.T, s.K,
                       vec, chunk, (uint4*)out);
}

cudaError_t launch_aux(const Shape& s, const float* psum, const int32_t* count, float* loss,
                       cudaStream_t st) {
  return launch_kernel(aux_kernel, dim3(1), dim3(256), 0, st, 1, psum, count, s.E, s.T, s.K, loss);
}

}  // namespace moe
