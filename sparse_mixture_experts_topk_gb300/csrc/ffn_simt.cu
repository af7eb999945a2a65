// Expert FFN on CUDA cores: the fp32 layer, the bf16 fallback used to
// cross-check the tensor-core kernel, and the weight-streaming kernel for
// decode-sized batches.
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

// Weight streaming for segments of at most kMaxRows rows (decode-sized
// batches): the time is reading each used expert's weights once, so the
// kernel is built for bytes in flight.  Block (x, y) handles kStreamRows
// weight rows of the y-th expert that has rows (found from offs; blocks past
// the last such expert exit).  The segment's activation rows are staged in
// shared memory once per block; each warp takes rows of B in turn, and each
// lane issues kUnroll independent 16-byte weight loads before any arithmetic.
constexpr int kMaxRows = 16;
constexpr int kStreamWarps = 8, kStreamRowsPerWarp = 2;
constexpr int kStreamRows = kStreamWarps * kStreamRowsPerWarp;
constexpr int kUnroll = 8;

// With kEpi = kEpiSwiglu, B_e = [W1; W3] ([2N, K]) and output column n dots
// the activation rows with gate row n and up row N + n.
template <typename T, int kEpi>
__global__ void __launch_bounds__(kStreamWarps * 32)
stream_ffn_kernel(const T* __restrict__ A, const int32_t* __restrict__ offs, int E, int mcap,
                  const T* __restrict__ B, const float* __restrict__ bias, int N, int K,
                  T* __restrict__ C, int* err) {
  extern __shared__ uint4 s_act[];            // [m][K] activation rows, 16-byte vectors
  __shared__ int s_e;
  constexpr bool kSwi = kEpi == kEpiSwiglu;
  pdl_enter();
  if (threadIdx.x == 0) {
    // the blockIdx.y-th expert with a non-empty segment
    int found = -1, seen = 0;
    for (int e = 0; e < E && found < 0; ++e)
      if (offs[e + 1] > offs[e] && seen++ == (int)blockIdx.y) found = e;
    s_e = found;
  }
  __syncthreads();
  const int e = s_e;
  if (e < 0) return;
  const int r0 = offs[e], r1 = offs[e + 1];
  int m = r1 - r0;
  if (m > mcap) {                              // more rows than staged: report, compute the first mcap
    if (threadIdx.x == 0) set_error(err, kDevBadIndex);
    m = mcap;
  }
  constexpr int V = Vec<T>::N;
  const int kv = K / V;
  const uint4* Av = reinterpret_cast<const uint4*>(A + (int64_t)r0 * K);
  for (int i = threadIdx.x; i < m * kv; i += blockDim.x) s_act[i] = Av[i];
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const T* Be = B + (int64_t)e * N * K * (kSwi ? 2 : 1);
  for (int q = 0; q < kStreamRowsPerWarp; ++q) {
    const int n = blockIdx.x * kStreamRows + warp * kStreamRowsPerWarp + q;
    if (n >= N) break;
    const uint4* Bv = reinterpret_cast<const uint4*>(Be + (int64_t)n * K);
    const uint4* Uv = reinterpret_cast<const uint4*>(Be + (int64_t)(N + n) * K);   // SwiGLU up row
    float acc[kMaxRows], accu[kMaxRows];
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) acc[r] = accu[r] = 0.f;
    for (int v0 = lane; v0 < kv; v0 += 32 * kUnroll) {
      uint4 bw[kUnroll], uw[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int v = v0 + 32 * u;
        if (v < kv) {
          bw[u] = __ldcs(Bv + v);
          if (kSwi) uw[u] = __ldcs(Uv + v);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int v = v0 + 32 * u;
        if (v < kv) {
          float b[V], bu[V];
          Vec<T>::unpack(bw[u], b);
          if (kSwi) Vec<T>::unpack(uw[u], bu);
#pragma unroll
          for (int r = 0; r < kMaxRows; ++r) {
            if (r < m) {
              float a[V];
              Vec<T>::unpack(s_act[r * kv + v], a);
#pragma unroll
              for (int i = 0; i < V; ++i) {
                acc[r] = fmaf(a[i], b[i], acc[r]);
                if (kSwi) accu[r] = fmaf(a[i], bu[i], accu[r]);
              }
            }
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
      if (r < m) {
        float sg = acc[r], su = accu[r];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          sg += __shfl_xor_sync(0xffffffffu, sg, o);
          if (kSwi) su += __shfl_xor_sync(0xffffffffu, su, o);
        }
        if (lane == 0) {
          const int64_t bstride = (int64_t)N * (kSwi ? 2 : 1);
          float v = sg + (bias ? bias[e * bstride + n] : 0.f);
          if (kEpi == kEpiGelu) v = gelu_erf(v);
          if (kSwi) v = silu_f(v) * (su + (bias ? bias[e * bstride + N + n] : 0.f));
          C[(int64_t)(r0 + r) * N + n] = from_f32<T>(v);
        }
      }
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

template <typename T>
cudaError_t run_stream(const Shape& s, const void* x_perm, const int32_t* offs, const void* W1,
                       const float* b1, const void* W2, const float* b2, void* h_perm, void* y_perm,
                       int* err, cudaStream_t st) {
  // at most T*K experts have rows; each block stages <= min(T, 16) rows
  const int experts = (int)(s.S() < s.E ? s.S() : s.E);
  const int mcap = (int)(s.T < kMaxRows ? s.T : kMaxRows);
  const size_t smem1 = (size_t)mcap * s.H * s.esize();
  const size_t smem2 = (size_t)mcap * s.F * s.esize();
  auto k1 = (s.flags & MOE_FLAG_SWIGLU) ? stream_ffn_kernel<T, kEpiSwiglu> : stream_ffn_kernel<T, kEpiGelu>;
  auto k2 = stream_ffn_kernel<T, kEpiPlain>;
  cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2);
  if (e != cudaSuccess) return e;
  dim3 g1((s.F + kStreamRows - 1) / kStreamRows, experts);
  e = launch_kernel(k1, g1, dim3(kStreamWarps * 32), smem1, st, 1, (const T*)x_perm, offs, s.E, mcap,
                    (const T*)W1, b1, s.F, s.H, (T*)h_perm, err);
  if (e != cudaSuccess) return e;
  prof_mark(kMarkFirst, st);
  dim3 g2((s.H + kStreamRows - 1) / kStreamRows, experts);
  return launch_kernel(k2, g2, dim3(kStreamWarps * 32), smem2, st, 1, (const T*)h_perm, offs, s.E, mcap,
                       (const T*)W2, b2, s.H, s.F, (T*)y_perm, err);
}

}  // namespace

// decode-sized batches whose staged activation rows fit in shared memory
bool stream_ffn_eligible(const Shape& s) {
  if (s.T > kMaxRows || (s.flags & MOE_FLAG_NO_DECODE)) return false;
  const int64_t widest = s.H > s.F ? s.H : s.F;
  return s.T * widest * (int64_t)s.esize() <= 200 * 1024;
}

cudaError_t launch_ffn_simt(const Shape& s, int64_t max_rows, const void* x_perm, const int32_t* offs,
                            const void* W1, const float* b1, const void* W2, const float* b2,
                            void* h_perm, void* y_perm, cudaStream_t st) {
  if (s.dtype == MOE_BF16)
    return run_simt<bf16>(s, max_rows, x_perm, offs, W1, b1, W2, b2, h_perm, y_perm, st);
  return run_simt<float>(s, max_rows, x_perm, offs, W1, b1, W2, b2, h_perm, y_perm, st);
}

cudaError_t launch_ffn_stream(const Shape& s, const void* x_perm, const int32_t* offs, const void* W1,
                              const float* b1, const void* W2, const float* b2, void* h_perm,
                              void* y_perm, int* err, cudaStream_t st) {
  if (s.dtype == MOE_BF16)
    return run_stream<bf16>(s, x_perm, offs, W1, b1, W2, b2, h_perm, y_perm, err, st);
  return run_stream<float>(s, x_perm, offs, W1, b1, W2, b2, h_perm, y_perm, err, st);
}

}  // namespace moe
