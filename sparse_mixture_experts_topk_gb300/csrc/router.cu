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
#include "router_body.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

using route::finish_tokens;
using route::kSmallChunk;
using route::kSmallMaxCta;
using route::kSmallTok;
using route::small_pieces;
using route::small_unit_any;

constexpr int kRouterTok = 32;   // tokens per block (one per lane)
constexpr int kRouterKC = 32;    // hidden elements staged per step
constexpr int kRouterThreads = 256;
constexpr int kRouterWarps = kRouterThreads / 32;

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
  finish_tokens(ls, nt, t0, E, K, inv_tau, ids, w, warp, kRouterWarps);
  __syncthreads();
  if (psum_part) {
    for (int e = tid; e < E; e += kRouterThreads) {
      float s = 0.f;
      for (int r = 0; r < nt; ++r) s += ls[r * (E + 1) + e];
      psum_part[(int64_t)blockIdx.x * E + e] = s;
    }
  }
}

// Decode-sized batches (T <= kSmallTok, bf16): the cost is reading Wg once
// and the latency of the few steps, so one cluster of up to 8 CTAs does it
// all.  A gate row is cut into pieces of 32 * kSmallChunk 16-byte vectors,
// and warp g of the cluster owns the (row, piece) units g, g + G, ... (G =
// its warps), so that with E * pieces <= G the whole of Wg is requested in
// one round; each lane loads its kSmallChunk vectors of a unit in one go
// (the first before the token rows are staged in shared memory) and dots
// them with every staged token (a body sized for the batch, so the hot loop
// stays small).  A unit's T partial scores go straight into the leader CTA's
// piece table over distributed shared memory; after one cluster barrier the
// leader adds each score's pieces in piece order, adds the bias, finishes
// each token (top-k, weights), counts the chosen experts as it picks them
// into tile_hist[0] (the layer's single 128-token tile) and sums the
// probabilities per expert in token order into psum_part[0].
// shared memory of the small router: token rows, score table, piece table
inline size_t small_smem(int64_t T, int H, int E) {
  return (size_t)T * H * sizeof(bf16) + (size_t)T * (E + 1) * sizeof(float) +
         (size_t)small_pieces(H) * T * E * sizeof(float);
}

__global__ void __launch_bounds__(kRouterThreads)
router_small_kernel(const bf16* __restrict__ x, const bf16* __restrict__ Wg,
                    const float* __restrict__ gate_bias, int Tn, int H, int E, int K, float inv_tau,
                    float* __restrict__ logits, int32_t* __restrict__ ids, float* __restrict__ w,
                    float* __restrict__ psum_part, int32_t* __restrict__ tile_hist) {
  // [Tn][H] token rows, then [Tn][E+1] scores, then [pieces][Tn][E] partial scores
  extern __shared__ uint4 s_x[];
  __shared__ int s_hist[256];
  constexpr int V = Vec<bf16>::N;
  const int kv = H / V;
  const int nch = small_pieces(H);                                     // pieces per gate row
  float* ls = reinterpret_cast<float*>(s_x + (size_t)Tn * kv);
  float* lp = ls + Tn * (E + 1);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t rank = tc::cluster_ctarank();
  const int g0 = (int)rank * kRouterWarps + warp;
  const int G = (int)gridDim.x * kRouterWarps;
  const int units = E * nch;
  const int mine = g0 < units ? (units - 1 - g0) / G + 1 : 0;
  for (int e = threadIdx.x; e < 256; e += kRouterThreads) s_hist[e] = 0;
  pdl_enter();
  uint4 gw[kSmallChunk];
  auto load_unit = [&](int p) {
    const int u = g0 + p * G;
    const int e = u / nch;
    const int c0 = (u % nch) * 32 * kSmallChunk;
    const uint4* row = reinterpret_cast<const uint4*>(Wg + (int64_t)e * H);
#pragma unroll
    for (int i = 0; i < kSmallChunk; ++i) {
      const int v = c0 + lane + 32 * i;
      if (v < kv) gw[i] = __ldg(row + v);
    }
  };
  if (mine > 0) load_unit(0);
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  for (int i = threadIdx.x; i < Tn * kv; i += kRouterThreads) s_x[i] = xv[i];
  __syncthreads();
  const uint32_t lp_leader = tc::map_peer(tc::smem_u32(lp), 0);
#pragma unroll 1
  for (int p = 0; p < mine; ++p) {
    const int u = g0 + p * G;
    const int e = u / nch, c = u % nch;
    const int c0 = c * 32 * kSmallChunk;
    const uint32_t dst = lp_leader + 4u * (uint32_t)(c * Tn * E + e);
    uint4 cur[kSmallChunk];
#pragma unroll
    for (int i = 0; i < kSmallChunk; ++i) cur[i] = gw[i];
    if (p + 1 < mine) load_unit(p + 1);   // the next unit's loads fly during this one
    small_unit_any(cur, s_x, kv, c0, Tn, [&](int t, float v) { tc::st_peer_f32(dst + 4u * (uint32_t)(t * E), v); });
  }
  tc::cluster_sync();              // every partial score is in the leader's piece table
  if (rank != 0) return;
#pragma unroll 1
  for (int i = threadIdx.x; i < Tn * E; i += kRouterThreads) {
    const int t = i / E, e = i % E;
    float v = 0.f;
#pragma unroll 1
    for (int c = 0; c < nch; ++c) v += lp[(c * Tn + t) * E + e];
    if (gate_bias) v += gate_bias[e];
    ls[t * (E + 1) + e] = v;
    if (logits) logits[(int64_t)t * E + e] = v;
  }
  __syncthreads();
  finish_tokens(ls, Tn, 0, E, K, inv_tau, ids, w, warp, kRouterWarps, s_hist);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kRouterThreads) {
    if (psum_part) {
      float sum = 0.f;
      for (int t = 0; t < Tn; ++t) sum += ls[t * (E + 1) + e];
      psum_part[e] = sum;
    }
    if (tile_hist) tile_hist[e] = s_hist[e];
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

bool router_small(const Shape& s) {
  // the token rows and the score table fit one CTA's shared memory
  return s.dtype == MOE_BF16 && s.T <= kSmallTok && s.E <= 256 && !(s.flags & MOE_FLAG_SIMT_ROUTER) &&
         small_smem(s.T, s.H, s.E) <= 200 * 1024;
}

int64_t router_partial_rows(const Shape& s) {
  if (router_small(s)) return 1;
  return router_on_tensor_cores(s) ? (s.T + 127) / 128 * router_tc_split(s) : router_partials(s);
}

cudaError_t launch_router(const Shape& s, const void* x, const void* Wg, const float* gate_bias,
                          float* logits, int32_t* ids, float* w, float* psum_part, int* err,
                          cudaStream_t st, int32_t* tile_hist) {
  if (s.T == 0) return cudaSuccess;
  if (router_small(s)) {
    const int need = (s.E * small_pieces(s.H) + kRouterWarps - 1) / kRouterWarps;
    const int cl = need < kSmallMaxCta ? need : kSmallMaxCta;
    const size_t smem = small_smem(s.T, s.H, s.E);
    cudaError_t e = cudaFuncSetAttribute(router_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(router_small_kernel, dim3((unsigned)cl), dim3(kRouterThreads), smem, st, (unsigned)cl,
                         (const bf16*)x, (const bf16*)Wg, gate_bias, (int)s.T, s.H, s.E, s.K, s.inv_tau, logits,
                         ids, w, psum_part, tile_hist);
  }
  if (router_on_tensor_cores(s))
    return launch_router_tc(s, x, Wg, gate_bias, logits, ids, w, psum_part, tile_hist, err, st);
  const size_t smem = sizeof(float) * (kRouterTok * (kRouterKC + 1) + s.E * (kRouterKC + 1) +
                                       kRouterTok * (s.E + 1));
  const int64_t grid = router_partials(s);
  if (s.dtype == MOE_BF16) {
    auto k = router_simt_kernel<bf16>;
    const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(k, dim3((unsigned)grid), dim3(kRouterThreads), smem, st, 1, (const bf16*)x,
                         (const bf16*)Wg, gate_bias, s.T, s.H, s.E, s.K, s.inv_tau, logits, ids, w, psum_part);
  }
  auto k = router_simt_kernel<float>;
  const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
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
