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
#include "combine.cuh"
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

// One warp per (token, column chunk) work item (combine_items).
template <typename T, int KP>
__global__ void __launch_bounds__(256, 3)   // 3 blocks (24 warps) an SM: the loads in flight set the speed
combine_kernel(const uint4* __restrict__ y_perm, const int32_t* __restrict__ pos,
               const float* __restrict__ w, int64_t Tn, int K, int vec_per_row, int chunk_vec,
               uint4* __restrict__ out) {
  pdl_enter();
  combine_items<T, KP>(y_perm, pos, w, Tn, K, vec_per_row, chunk_vec, out,
                       ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5, ((int64_t)gridDim.x * blockDim.x) >> 5);
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

__global__ void merge_stats_kernel(const int32_t* __restrict__ count_parts, const float* __restrict__ psum_parts,
                                   int n, int E, int64_t Tn, int K, int32_t* __restrict__ count,
                                   float* __restrict__ psum, int32_t* __restrict__ count_copy,
                                   float* __restrict__ aux, int32_t* __restrict__ dropped) {
  __shared__ float sa[256];
  pdl_enter();
  const int e = threadIdx.x;
  int c = 0;
  float p = 0.f;
  if (e < E) {
    for (int i = 0; i < n; ++i) {
      c += count_parts[(int64_t)i * E + e];
      p += psum_parts[(int64_t)i * E + e];
    }
    count[e] = c;
    psum[e] = p;
    if (count_copy) count_copy[e] = c;
  }
  sa[e] = (e < E && Tn > 0) ? ((float)c / (float)(Tn * K)) * (p / (float)Tn) : 0.f;
  __syncthreads();
  for (int o = 128; o > 0; o >>= 1) {
    if (e < o) sa[e] += sa[e + o];
    __syncthreads();
  }
  if (e == 0) {
    if (aux) *aux = (float)E * sa[0];
    if (dropped) *dropped = 0;
  }
}

__global__ void __launch_bounds__(256) zero_acc_kernel(float4* __restrict__ acc, int64_t n4) {
  pdl_enter();
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x)
    __stcg(acc + i, z);
}

// out = bf16(acc), 8 elements per thread step
__global__ void __launch_bounds__(256) acc_to_out_kernel(const float4* __restrict__ acc, uint4* __restrict__ out,
                                                         int64_t n8) {
  pdl_enter();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
    const float4 a = __ldcs(acc + 2 * i), b = __ldcs(acc + 2 * i + 1);
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    __stcs(out + i, Vec<bf16>::pack(v));
  }
}

}  // namespace

cudaError_t launch_zero_acc(const Shape& s, float* acc, cudaStream_t st) {
  const int64_t n4 = s.T * (int64_t)s.H / 4;
  const int64_t grid = (int64_t)sm_count() * 8;
  return launch_kernel(zero_acc_kernel, dim3((unsigned)grid), dim3(256), 0, st, 1, (float4*)acc, n4);
}

cudaError_t launch_acc_to_out(const Shape& s, const float* acc, void* out, cudaStream_t st) {
  const int64_t n8 = s.T * (int64_t)s.H / 8;
  const int64_t grid = (int64_t)sm_count() * 8;
  return launch_kernel(acc_to_out_kernel, dim3((unsigned)grid), dim3(256), 0, st, 1, (const float4*)acc, (uint4*)out,
                       n8);
}

cudaError_t launch_merge_stats(const Shape& s, const int32_t* count_parts, const float* psum_parts, int n,
                               int32_t* count, float* psum, int32_t* count_copy, float* aux, int32_t* dropped,
                               cudaStream_t st) {
  return launch_kernel(merge_stats_kernel, dim3(1), dim3(256), 0, st, 1, count_parts, psum_parts, n, s.E, s.T, s.K,
                       count, psum, count_copy, aux, dropped);
}

cudaError_t launch_combine(const Shape& s, const void* y_perm, const int32_t* pos, const float* w,
                           void* out, cudaStream_t st) {
  if (s.T == 0) return cudaSuccess;
  const int vec = (int)((int64_t)s.H * s.esize() / 16);
  // persistent: as many blocks of 8 warps as the SMs hold at once (3 each)
  const int64_t cap = (int64_t)sm_count() * 3;
  const int chunk = combine_chunk();
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
