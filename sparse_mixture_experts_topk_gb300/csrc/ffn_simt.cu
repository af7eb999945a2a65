// Expert FFN on CUDA cores: the fp32 layer, and the bf16 path used to
// cross-check the tensor-core kernels.
//
// Each expert is Linear -> GELU -> Linear (Qwen2-MoE module article, mlqm.cn,
// section 2.2; MoE sparse-activation article, wmrh.cn, section 2.2):
//   h[r] = GELU(W1[e] x_perm[r] + b1[e]),  y[r] = W2[e] h[r] + b2[e]
// for the rows r of expert e's segment [offs[e], offs[e+1]).  Both products
// are "A [rows, K] times B [N, K]^T" with K contiguous in both operands.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kBM = 64, kBN = 64, kBK = 16, kGemmThreads = 256;

// Map a linear m-tile index to (expert, row start, row end) from offs.
__device__ __forceinline__ bool find_tile(const int32_t* __restrict__ offs, int E, int tile, int bm,
                                          int* e_out, int* r0_out, int* r1_out) {
  int acc = 0;
  for (int e = 0; e < E; ++e) {
    const int a = offs[e], b = offs[e + 1];
    const int n = (b - a + bm - 1) / bm;
    if (tile < acc + n) {
      *e_out = e;
      *r0_out = a + (tile - acc) * bm;
      *r1_out = b;
      return true;
    }
    acc += n;
  }
  return false;
}

// C[r, n] = epi(sum_k A[r, k] B_e[n, k]) for one 64x64 tile.  With
// kEpi = kEpiSwiglu, B_e = [W1; W3] ([2N, K]) and C[r, n] =
// SiLU(sum_k A W1[n, k] + b1[n]) * (sum_k A W3[n, k] + b1[N + n]).
template <typename T, int kEpi>
__global__ void __launch_bounds__(kGemmThreads)
grouped_gemm_simt_kernel(const T* __restrict__ A, const int32_t* __restrict__ offs, int E,
                         const T* __restrict__ B, const float* __restrict__ bias, int N, int K,
                         T* __restrict__ C) {
  __shared__ int s_e, s_r0, s_r1;
  __shared__ float As[kBK][kBM + 4];
  constexpr bool kSwi = kEpi == kEpiSwiglu;
  __shared__ float Bs[kBK][kBN + 4];
  __shared__ float Us[kBK][kBN + 4];      // up-projection tile (SwiGLU only)
  pdl_enter();
  if (threadIdx.x == 0) {
    int e, r0, r1;
    if (!find_tile(offs, E, blockIdx.y, kBM, &e, &r0, &r1)) e = -1;
    s_e = e; s_r0 = r0; s_r1 = r1;
  }
  __syncthreads();
  const int e = s_e;
  if (e < 0) return;
  const int r0 = s_r0, r1 = s_r1;
  const int n0 = blockIdx.x * kBN;
  const T* Be = B + (int64_t)e * N * K * (kSwi ? 2 : 1);
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {};
  float accu[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += kBK) {
    {
      const int i = threadIdx.x;            // 256 threads x 4 elements
      const int row = i / 4, kq = (i % 4) * 4;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int k = k0 + kq + j;
        const int r = r0 + row;
        As[kq + j][row] = (r < r1 && k < K) ? to_f32(A[(int64_t)r * K + k]) : 0.f;
        const int n = n0 + row;
        Bs[kq + j][row] = (n < N && k < K) ? to_f32(Be[(int64_t)n * K + k]) : 0.f;
        if (kSwi) Us[kq + j][row] = (n < N && k < K) ? to_f32(Be[(int64_t)(N + n) * K + k]) : 0.f;
      }
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kBK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) { a[i] = As[kk][ty * 4 + i]; b[i] = Bs[kk][tx * 4 + i]; }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
      if (kSwi) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) accu[i][j] = fmaf(a[i], Us[kk][tx * 4 + j], accu[i][j]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = r0 + ty * 4 + i;
    if (r >= r1) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= N) continue;
      float v = acc[i][j] + (bias ? bias[(int64_t)e * N * (kSwi ? 2 : 1) + n] : 0.f);
      if (kEpi == kEpiGelu) v = gelu_erf(v);
      if (kSwi) {
        const float u = accu[i][j] + (bias ? bias[(int64_t)e * N * 2 + N + n] : 0.f);
        v = silu_f(v) * u;
      }
      C[(int64_t)r * N + n] = from_f32<T>(v);
    }
  }
}

template <typename T>
cudaError_t run_simt(const Shape& s, int64_t max_rows, const void* x_perm, const int32_t* offs,
                     const void* W1, const float* b1, const void* W2, const float* b2,
                     void* h_perm, void* y_perm, cudaStream_t st) {
  const int64_t mtiles = (max_rows + kBM - 1) / kBM + s.E;
  if (mtiles > 65535) return cudaErrorInvalidConfiguration;
  dim3 g1((s.F + kBN - 1) / kBN, (unsigned)mtiles);
  auto k1 = (s.flags & MOE_FLAG_SWIGLU) ? grouped_gemm_simt_kernel<T, kEpiSwiglu>
                                        : grouped_gemm_simt_kernel<T, kEpiGelu>;
  cudaError_t e = launch_kernel(k1, g1, dim3(kGemmThreads), 0, st, 1,
                                (const T*)x_perm, offs, s.E, (const T*)W1, b1, s.F, s.H, (T*)h_perm);
  if (e != cudaSuccess) return e;
  prof_mark(kMarkFirst, st);
  dim3 g2((s.H + kBN - 1) / kBN, (unsigned)mtiles);
  return launch_kernel(grouped_gemm_simt_kernel<T, kEpiPlain>, g2, dim3(kGemmThreads), 0, st, 1,
                       (const T*)h_perm, offs, s.E, (const T*)W2, b2, s.H, s.F, (T*)y_perm);
}

}  // namespace

cudaError_t launch_ffn_simt(const Shape& s, int64_t max_rows, const void* x_perm, const int32_t* offs,
                            const void* W1, const float* b1, const void* W2, const float* b2,
                            void* h_perm, void* y_perm, cudaStream_t st) {
  if (s.dtype == MOE_BF16)
    return run_simt<bf16>(s, max_rows, x_perm, offs, W1, b1, W2, b2, h_perm, y_perm, st);
  return run_simt<float>(s, max_rows, x_perm, offs, W1, b1, W2, b2, h_perm, y_perm, st);
}

}  // namespace moe
