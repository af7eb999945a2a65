// Bodies of the weight-streaming kernels: one staged weight row dotted with
// a few staged activation rows (bf16 operands into fp32 sums), and the
// bounded wait on a counter that another CTA raises.  Shared by the
// streaming expert kernel and the one-launch decode layer, so both compute
// every output value with the same operations in the same order.
#pragma once

#include <type_traits>

#include "bf16_dot.cuh"
#include "common.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace stream {

constexpr int kConsumers = 8;                    // consumer warps; a stage holds <= 8 rows
constexpr uint64_t kWaitNs = 2000000000ull;

// One weight row (SwiGLU: gate row w and up row u) against the m <= MR
// staged activation rows: lane l takes vectors l, l + 32, ...; fp32 sums,
// reduced across the warp; lane 0 adds the bias, applies the activation and
// writes out[r * N] for r < m.  bf16 rows are multiplied without widening
// (fma8_bf16); fp32 rows element by element.
template <typename T, int kEpi, int MR>
__device__ __forceinline__ void dot_rows(const uint4* w, const uint4* u, const uint4* act, int kv, int m,
                                         const float* be, int n, int N, T* out) {
  constexpr bool kSwi = kEpi == kEpiSwiglu;
  constexpr int V = Vec<T>::N;
  const int lane = threadIdx.x & 31;
  float acc[MR], accu[MR];
#pragma unroll
  for (int r = 0; r < MR; ++r) acc[r] = accu[r] = 0.f;
#pragma unroll 2
  for (int v = lane; v < kv; v += 32) {
    const uint4 wq = w[v];
    const uint4 uq = kSwi ? u[v] : wq;
#pragma unroll
    for (int r = 0; r < MR; ++r) {
      if (r < m) {
        const uint4 xq = act[r * kv + v];
        if constexpr (std::is_same<T, bf16>::value) {
          acc[r] = fma8_bf16(xq, wq, acc[r]);
          if (kSwi) accu[r] = fma8_bf16(xq, uq, accu[r]);
        } else {
          float x[V], b[V], bu[V];
          Vec<T>::unpack(xq, x);
          Vec<T>::unpack(wq, b);
          if (kSwi) Vec<T>::unpack(uq, bu);
#pragma unroll
          for (int i = 0; i < V; ++i) {
            acc[r] = fmaf(x[i], b[i], acc[r]);
            if (kSwi) accu[r] = fmaf(x[i], bu[i], accu[r]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < MR; ++r) {
    if (r < m) {
      float sg = acc[r], su = accu[r];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        sg += __shfl_xor_sync(0xffffffffu, sg, o);
        if (kSwi) su += __shfl_xor_sync(0xffffffffu, su, o);
      }
      if (lane == 0) {
        float v = sg + (be ? be[n] : 0.f);
        if (kEpi == kEpiGelu) v = gelu_erf(v);
        if (kSwi) v = silu_f(v) * (su + (be ? be[N + n] : 0.f));
        out[(int64_t)r * N] = from_f32<T>(v);
      }
    }
  }
}

// Dot weight row j of a staged ring stage with the staged activation rows
// (a body sized for the segment, so the hot loop stays small; kMR bounds the
// segment, and with it the registers the bodies take).
template <typename T, int kEpi, int kMR>
__device__ __forceinline__ void stage_row(const uint8_t* st, int j, int rps, uint32_t row_bytes, const uint4* act,
                                          int kv, int m, const float* be, int n, int N, T* out) {
  const uint4* wv = reinterpret_cast<const uint4*>(st + (size_t)j * row_bytes);
  const uint4* uv = reinterpret_cast<const uint4*>(st + (size_t)(rps + j) * row_bytes);
  if (m <= 1) dot_rows<T, kEpi, 1>(wv, uv, act, kv, m, be, n, N, out);
  else if (kMR <= 2 || m <= 2) dot_rows<T, kEpi, 2>(wv, uv, act, kv, m, be, n, N, out);
  else if (kMR <= 4 || m <= 4) dot_rows<T, kEpi, (kMR < 4 ? kMR : 4)>(wv, uv, act, kv, m, be, n, N, out);
  else if (kMR <= 8 || m <= 8) dot_rows<T, kEpi, (kMR < 8 ? kMR : 8)>(wv, uv, act, kv, m, be, n, N, out);
  else dot_rows<T, kEpi, kMR>(wv, uv, act, kv, m, be, n, N, out);
}

// Two weight rows (w0/u0 and w1/u1, output columns n and n + 1) against
// the same m <= MR staged activation rows: each activation vector is read
// once for both rows, and the two rows' sums are independent chains.  Every
// output is the same sum in the same order as dot_rows gives it.  bf16.
template <int kEpi, int MR>
__device__ __forceinline__ void dot_rows2(const uint4* w0, const uint4* u0, const uint4* w1, const uint4* u1,
                                          const uint4* act, int kv, int m, const float* be, int n, int N,
                                          bf16* out) {
  constexpr bool kSwi = kEpi == kEpiSwiglu;
  const int lane = threadIdx.x & 31;
  float a0[MR], a1[MR], b0[MR], b1[MR];
#pragma unroll
  for (int r = 0; r < MR; ++r) a0[r] = a1[r] = b0[r] = b1[r] = 0.f;
#pragma unroll 2
  for (int v = lane; v < kv; v += 32) {
    const uint4 p0 = w0[v], p1 = w1[v];
    const uint4 q0 = kSwi ? u0[v] : p0, q1 = kSwi ? u1[v] : p1;
#pragma unroll
    for (int r = 0; r < MR; ++r) {
      if (r < m) {
        const uint4 xq = act[r * kv + v];
        a0[r] = fma8_bf16(xq, p0, a0[r]);
        a1[r] = fma8_bf16(xq, p1, a1[r]);
        if (kSwi) {
          b0[r] = fma8_bf16(xq, q0, b0[r]);
          b1[r] = fma8_bf16(xq, q1, b1[r]);
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < MR; ++r) {
    if (r < m) {
      float g0 = a0[r], g1 = a1[r], s0 = b0[r], s1 = b1[r];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        g0 += __shfl_xor_sync(0xffffffffu, g0, o);
        g1 += __shfl_xor_sync(0xffffffffu, g1, o);
        if (kSwi) {
          s0 += __shfl_xor_sync(0xffffffffu, s0, o);
          s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        }
      }
      if (lane == 0) {
        float v0 = g0 + (be ? be[n] : 0.f), v1 = g1 + (be ? be[n + 1] : 0.f);
        if (kEpi == kEpiGelu) {
          v0 = gelu_erf(v0);
          v1 = gelu_erf(v1);
        }
        if (kSwi) {
          v0 = silu_f(v0) * (s0 + (be ? be[N + n] : 0.f));
          v1 = silu_f(v1) * (s1 + (be ? be[N + n + 1] : 0.f));
        }
        out[(int64_t)r * N] = from_f32<bf16>(v0);
        out[(int64_t)r * N + 1] = from_f32<bf16>(v1);
      }
    }
  }
}

// Weight rows j and j + 1 of a staged ring stage (output columns n, n + 1)
// for a segment of 2 <= m <= min(4, kMR) activation rows.
template <int kEpi, int kMR>
__device__ __forceinline__ void stage_pair(const uint8_t* st, int j, int rps, uint32_t row_bytes, const uint4* act,
                                           int kv, int m, const float* be, int n, int N, bf16* out) {
  const uint4* w0 = reinterpret_cast<const uint4*>(st + (size_t)j * row_bytes);
  const uint4* u0 = reinterpret_cast<const uint4*>(st + (size_t)(rps + j) * row_bytes);
  const uint4* w1 = reinterpret_cast<const uint4*>(st + (size_t)(j + 1) * row_bytes);
  const uint4* u1 = reinterpret_cast<const uint4*>(st + (size_t)(rps + j + 1) * row_bytes);
  if (m <= 1) dot_rows2<kEpi, 1>(w0, u0, w1, u1, act, kv, m, be, n, N, out);
  else if (kMR <= 2 || m <= 2) dot_rows2<kEpi, 2>(w0, u0, w1, u1, act, kv, m, be, n, N, out);
  else dot_rows2<kEpi, 4>(w0, u0, w1, u1, act, kv, m, be, n, N, out);
}

// Row j of stage g (rps rows a stage) is the CTA's row g rps + j of the
// product, and goes to consumer warp (g rps + j) mod kConsumers: with fewer
// rows than warps in a stage, the idle warps work on the next stage.
__device__ __forceinline__ int stage_row_of_warp(int g, int rps, int warp) {
  return ((warp - g * rps) % kConsumers + kConsumers) % kConsumers;
}

// Wait (bounded) until *p reaches `need`, acquire at GPU scope, then order
// the observed writes before this thread's later bulk copies (which read
// global memory through the async proxy).  False on timeout or abort.
__device__ __forceinline__ bool wait_count(const int* p, int need, const volatile int* abort) {
  uint64_t t0 = 0;
  for (int i = 0;; ++i) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    if (v >= need) {
      asm volatile("fence.proxy.async.global;" ::: "memory");
      return true;
    }
    if (*abort) return false;
    if ((i & 63) == 63) {
      const uint64_t now = tc::globaltimer();
      if (t0 == 0) t0 = now;
      else if (now - t0 > kWaitNs) return false;
    }
    __nanosleep(64);
  }
}

}  // namespace stream
}  // namespace moe
