// Router: gate linear + softmax + top-k + renormalisation, one kernel.
//
// Qwen2-MoE code walkthrough (jsqmd.com), section 3.1: the gate is a bias-free
// nn.Linear(hidden, num_experts); its scores go through a softmax, torch.topk
// picks num_experts_per_tok experts, and the k probabilities are divided by
// their sum.  Here the k experts are chosen on the fp32 scores themselves
// (softmax is monotone), largest first, equal scores by ascending expert index,
// and w_j = exp((l_j - m)/tau) / sum_sel exp((l_i - m)/tau), which equals
// p_j / sum_sel p for p = softmax(l / tau) (tau = 1 unless the layer sets a
// router temperature, MoE sparse-activation article, wmrh.cn, section 5.2).
#include <float.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kRouterTok = 32;   // tokens per block (one per lane)
constexpr int kRouterKC = 32;    // hidden elements staged per step
constexpr int kRouterThreads = 256;
constexpr int kRouterWarps = kRouterThreads / 32;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Per block: kRouterTok tokens.  Thread (warp w, lane l) accumulates the
// scores of token l for experts w, w+8, w+16, ...  Then each warp finishes 4
// tokens: softmax statistics, top-k, weights.  p[t, e] of the block's tokens
// is summed per expert in token order into psum_part[block, e].
template <typename T>
__global__ void __launch_bounds__(kRouterThreads)
router_simt_kernel(const T* __restrict__ x, const T* __restrict__ Wg,
                   const float* __restrict__ gate_bias, int64_t Tn, int H, int E, int K, float inv_tau,
                   float* __restrict__ logits, int32_t* __restrict__ ids, float* __restrict__ w,
                   float* __restrict__ psum_part) {
  extern __shared__ float smem[];
  float* xs = smem;                                   // [TOK][KC+1]
  float* gs = xs + kRouterTok * (kRouterKC + 1);      // [E][KC+1]
  float* ls = gs + E * (kRouterKC + 1);               // [TOK][E+1]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t t0 = (int64_t)blockIdx.x * kRouterTok;
  const int nt = (int)min((int64_t)kRouterTok, Tn - t0);
  pdl_enter();

  float acc[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) acc[i] = 0.f;

  for (int k0 = 0; k0 < H; k0 += kRouterKC) {
    for (int i = tid; i < kRouterTok * kRouterKC; i += kRouterThreads) {
      const int r = i / kRouterKC, c = i % kRouterKC;
      float v = 0.f;
      if (r < nt && k0 + c < H) v = to_f32(x[(t0 + r) * (int64_t)H + k0 + c]);
      xs[r * (kRouterKC + 1) + c] = v;
    }
    for (int i = tid; i < E * kRouterKC; i += kRouterThreads) {
      const int r = i / kRouterKC, c = i % kRouterKC;
      float v = 0.f;
      if (k0 + c < H) v = to_f32(Wg[(int64_t)r * H + k0 + c]);
      gs[r * (kRouterKC + 1) + c] = v;
    }
    __syncthreads();
#pragma unroll 4
    for (int c = 0; c < kRouterKC; ++c) {
      const float xv = xs[lane * (kRouterKC + 1) + c];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int e = warp + kRouterWarps * i;
        if (e < E) acc[i] = fmaf(xv, gs[e * (kRouterKC + 1) + c], acc[i]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int e = warp + kRouterWarps * i;
    if (e < E) ls[lane * (E + 1) + e] = acc[i] + (gate_bias ? gate_bias[e] : 0.f);
  }
  __syncthreads();
  if (logits) {
    for (int i = tid; i < nt * E; i += kRouterThreads) {
      const int r = i / E, e = i % E;
      logits[(t0 + r) * (int64_t)E + e] = ls[r * (E + 1) + e];
    }
  }
  // softmax statistics and top-k; lane holds experts lane + 32 i
  for (int tt = warp; tt < nt; tt += kRouterWarps) {
    float v[8];
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      v[i] = (e < E) ? ls[tt * (E + 1) + e] : -INFINITY;
      m = fmaxf(m, v[i]);
    }
    m = warp_max(m);
    float zs = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      if (e < E) zs += expf((v[i] - m) * inv_tau);
    }
    zs = warp_sum(zs);
    unsigned taken = 0;
    int sel_id[8];
    float sel_z[8];
    float zsel = 0.f;
    for (int j = 0; j < K; ++j) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < bi))) {
          bv = v[i];
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
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      const float z = expf((bv - m) * inv_tau);
      sel_id[j] = bi;
      sel_z[j] = z;
      zsel += z;
    }
    if (lane == 0) {
      const int64_t t = t0 + tt;
      for (int j = 0; j < K; ++j) {
        ids[t * K + j] = sel_id[j];
        w[t * K + j] = sel_z[j] / zsel;
      }
    }
    // full-softmax probabilities for the load-balancing statistics
    const float inv = 1.f / zs;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      if (e < E) ls[tt * (E + 1) + e] = expf((v[i] - m) * inv_tau) * inv;
    }
  }
  __syncthreads();
  if (psum_part) {
    for (int e = tid; e < E; e += kRouterThreads) {
      float s = 0.f;
      for (int r = 0; r < nt; ++r) s += ls[r * (E + 1) + e];
      psum_part[(int64_t)blockIdx.x * E + e] = s;
    }
  }
}

__global__ void psum_reduce_kernel(const float* __restrict__ part, int64_t rows, int E,
                                   float* __restrict__ psum) {
  pdl_enter();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float s = 0.f;
    for (int64_t r = 0; r < rows; ++r) s += part[r * E + e];
    psum[e] = s;
  }
}

}  // namespace

int64_t router_partials(const Shape& s) { return (s.T + kRouterTok - 1) / kRouterTok; }

int64_t router_partial_rows(const Shape& s) {
  return router_on_tensor_cores(s) ? (s.T + 127) / 128 : router_partials(s);
}

cudaError_t launch_router(const Shape& s, const void* x, const void* Wg, const float* gate_bias,
                          float* logits, int32_t* ids, float* w, float* psum_part, int* err,
                          cudaStream_t st, int32_t* tile_hist) {
  if (s.T == 0) return cudaSuccess;
  if (router_on_tensor_cores(s))
    return launch_router_tc(s, x, Wg, gate_bias, logits, ids, w, psum_part, tile_hist, err, st);
  const size_t smem = sizeof(float) * (kRouterTok * (kRouterKC + 1) + s.E * (kRouterKC + 1) +
                                       kRouterTok * (s.E + 1));
  const int64_t grid = router_partials(s);
  if (s.dtype == MOE_BF16) {
    auto k = router_simt_kernel<bf16>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return launch_kernel(k, dim3((unsigned)grid), dim3(kRouterThreads), smem, st, 1, (const bf16*)x,
                         (const bf16*)Wg, gate_bias, s.T, s.H, s.E, s.K, s.inv_tau, logits, ids, w, psum_part);
  }
  auto k = router_simt_kernel<float>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  return launch_kernel(k, dim3((unsigned)grid), dim3(kRouterThreads), smem, st, 1, (const float*)x,
                       (const float*)Wg, gate_bias, s.T, s.H, s.E, s.K, s.inv_tau, logits, ids, w, psum_part);
}

cudaError_t launch_psum_reduce(const Shape& s, const float* psum_part, float* psum, cudaStream_t st) {
  if (s.T == 0) {
    return cudaMemsetAsync(psum, 0, sizeof(float) * s.E, st);
  }
  return launch_kernel(psum_reduce_kernel, dim3(1), dim3(256), 0, st, 1, (const float*)psum_part,
                       router_partial_rows(s), s.E, psum);
}

}  // namespace moe
