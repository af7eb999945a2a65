// Expert FFN on the 5th-generation tensor cores: a persistent grouped GEMM
// with TMA-staged bf16 tiles, tcgen05.mma accumulating in TMEM, and a fused
// epilogue (bias, erf-GELU for the first product, bf16 rounding).
//
// Each expert is Linear -> GELU -> Linear (Qwen2-MoE module article,
// mlqm.cn, section 2.2).  For expert e with permuted rows [offs[e], offs[e+1]):
//   first product:  h = GELU(x_perm W1[e]^T + b1[e])   A = x_perm [rows, H], B = W1[e] [F, H]
//   second product: y = h W2[e]^T + b2[e]              A = h_perm [rows, F], B = W2[e] [H, F]
// Both operands are K-major (K contiguous), the nn.Linear [out, in] layout.
//
// Work unit: a 128 x BN output tile of one expert.  Tiles are numbered expert
// by expert, n-tile by n-tile, m-tile fastest, so CTAs running at the same
// time share each weight tile through L2; every CTA walks the tile list with
// a stride of the grid size.  Warp roles inside a CTA (192 threads):
//   warp 0     TMA producer: A and B k-blocks (64 elements = 128 bytes, 128B
//              swizzle) into a ring of shared-memory stages;
//   warp 1     MMA issuer (one thread): 4 x tcgen05.mma (K = 16 each) per
//              stage into one of two TMEM accumulators; owns TMEM alloc;
//   warps 2-5  epilogue: tcgen05.ld of the accumulator (one row per thread),
//              bias, GELU, bf16, 16-byte stores; frees the accumulator.
// Two accumulators let the epilogue of tile i overlap the MMAs of tile i+1.
// Every mbarrier wait is bounded: on expiry the kernel records a timeout in
// the workspace error word, the other roles see the abort flag, in-flight
// TMA loads and MMAs are drained (again with a bound), TMEM is freed and the
// kernel returns.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {

namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;              // bf16 elements per k-block = one 128-byte swizzle row
constexpr int kThreads = 192;
constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s: far beyond any healthy wait

template <int BN>
struct Cfg {
  static constexpr int kABytes = kBM * kBK * 2;
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = (196 * 1024) / kStageBytes > 8 ? 8 : (196 * 1024) / kStageBytes;
  static constexpr int kTmemCols = 2 * BN <= 256 ? 256 : 512;
  static constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes;
  static constexpr uint32_t kIdesc = tc::idesc_bf16_f32(kBM, BN);
};

// kEpi = kEpiSwiglu: B = [W1; W3] stacked per expert ([E, 2N, K]); a 256-wide
// accumulator tile holds 128 gate columns then the matching 128 up columns,
// and the tile writes SiLU(gate) * up for those 128 output columns.
template <int BN, int kEpi>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const int32_t* __restrict__ offs, int E, int N, int K,
                       const float* __restrict__ bias, bf16* __restrict__ C, int* err, int stall) {
  using Cf = Cfg<BN>;
  constexpr int S = Cf::kStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_offs[257];
  __shared__ int s_tstart[257];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ __align__(8) uint64_t s_bar[2 * S + 5];

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sA = tc::smem_u32(smem);
  const uint32_t sB = sA + S * Cf::kABytes;
  auto full = [&](int s) { return tc::smem_u32(&s_bar[s]); };
  auto empty = [&](int s) { return tc::smem_u32(&s_bar[S + s]); };
  auto tfull = [&](int a) { return tc::smem_u32(&s_bar[2 * S + a]); };
  auto tempty = [&](int a) { return tc::smem_u32(&s_bar[2 * S + 2 + a]); };
  const uint32_t done_bar = tc::smem_u32(&s_bar[2 * S + 4]);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr bool kSwi = kEpi == kEpiSwiglu;
  static_assert(!kSwi || BN == 256, "SwiGLU tiles pair 128 gate with 128 up columns");
  constexpr int kOut = kSwi ? BN / 2 : BN;     // output columns per tile
  const int nt = (N + kOut - 1) / kOut;
  const int nk = (K + kBK - 1) / kBK;

  if (warp == 0) {
    pdl_enter();   // the tile table reads offs, written by the previous kernel
    // per-expert tile counts and their exclusive prefix (E <= 256: 8 per lane)
    int loc[8];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      int v = 0;
      if (e < E) {
        const int o0 = offs[e], o1 = offs[e + 1];
        v = ((o1 - o0 + kBM - 1) / kBM) * nt;
        s_offs[e] = o0;
        if (e == E - 1) s_offs[E] = o1;
      }
      loc[i] = v;
      sum += v;
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    int run = incl - sum;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      if (e < E) s_tstart[e] = run;
      run += loc[i];
    }
    if (lane == 31) s_tstart[E] = incl;
    if (lane == 0) {
      for (int s = 0; s < S; ++s) {
        tc::mbar_init(full(s), 1);
        tc::mbar_init(empty(s), 1);
      }
      for (int a = 0; a < 2; ++a) {
        tc::mbar_init(tfull(a), 1);
        tc::mbar_init(tempty(a), 128);
      }
      tc::mbar_init(done_bar, 1);
      s_abort = 0;
      tc::fence_barrier_init();
      tc::fence_proxy_async_smem();
      tc::prefetch_tmap(&tmA);
      tc::prefetch_tmap(&tmB);
    }
  } else if (warp == 1) {
    tc::tmem_alloc(tc::smem_u32(&s_tmem), Cf::kTmemCols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp != 0) pdl_wait();
  const uint32_t tmem = s_tmem;
  const int total = s_tstart[E];

  auto decode = [&](int t, int& e, int& row0, int& row_end, int& n0) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_tstart[mid] <= t) lo = mid; else hi = mid - 1;
    }
    e = lo;
    const int mt = (s_offs[e + 1] - s_offs[e] + kBM - 1) / kBM;
    const int local = t - s_tstart[e];
    row0 = s_offs[e] + (local % mt) * kBM;
    row_end = s_offs[e + 1];
    n0 = (local / mt) * kOut;
  };

  uint32_t filled = 0, fill_par = 0;   // producer: per stage, ever filled / parity of its last fill
  bool producer = false;
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (tc::elect_one()) {
      producer = true;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      bool withhold = stall != 0;          // test hook: never arm or fill this CTA's first stage
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        int e, row0, row_end, n0;
        decode(t, e, row0, row_end, n0);
        for (int kb = 0; kb < nk; ++kb) {
          if (!tc::mbar_wait(empty(stage), phase ^ 1u, &s_abort, kWaitNs)) { ok = false; break; }
          if (withhold) {
            withhold = false;
            if (++stage == S) { stage = 0; phase ^= 1u; }
            continue;
          }
          tc::mbar_arrive_expect_tx(full(stage), Cf::kStageBytes);
          tc::tma_load_2d(sA + stage * Cf::kABytes, &tmA, full(stage), kb * kBK, row0);
          if (kSwi) {
            tc::tma_load_2d(sB + stage * Cf::kBBytes, &tmB, full(stage), kb * kBK, 2 * e * N + n0);
            tc::tma_load_2d(sB + stage * Cf::kBBytes + Cf::kBBytes / 2, &tmB, full(stage), kb * kBK,
                            2 * e * N + N + n0);
          } else {
            tc::tma_load_2d(sB + stage * Cf::kBBytes, &tmB, full(stage), kb * kBK, e * N + n0);
          }
          filled |= 1u << stage;
          fill_par = (fill_par & ~(1u << stage)) | (phase << stage);
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        set_error(err, kDevTimeout);
        s_abort = 1;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (tc::elect_one()) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        if (!tc::mbar_wait(tempty(acc), acc_phase ^ 1u, &s_abort, kWaitNs)) { ok = false; break; }
        tc::tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(acc * BN);
        for (int kb = 0; kb < nk; ++kb) {
          if (!tc::mbar_wait(full(stage), phase, &s_abort, kWaitNs)) { ok = false; break; }
          tc::tc_fence_after();
          const uint32_t a0 = sA + stage * Cf::kABytes, b0 = sB + stage * Cf::kBBytes;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            tc::mma_bf16(d, tc::sdesc_k128(a0 + k * 32), tc::sdesc_k128(b0 + k * 32), Cf::kIdesc,
                         (kb | k) != 0);
          tc::tc_commit(empty(stage));
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc::tc_commit(tfull(acc));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok) {
        set_error(err, kDevTimeout);
        s_abort = 1;
      }
      // every MMA this thread issued must finish before TMEM is released
      tc::tc_commit(done_bar);
      tc::mbar_wait(done_bar, 0, nullptr, kWaitNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;   // TMEM lanes 32q..32q+31 belong to this warp
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      int e, row0, row_end, n0;
      decode(t, e, row0, row_end, n0);
      if (!tc::mbar_wait(tfull(acc), acc_phase, &s_abort, kWaitNs)) {
        set_error(err, kDevTimeout);
        s_abort = 1;
        break;
      }
      tc::tc_fence_after();
      const int row = row0 + q * 32 + lane;
      const bool row_ok = row < row_end;
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      const float* be = bias ? bias + (int64_t)e * (kSwi ? 2 * N : N) : nullptr;
#pragma unroll 1
      for (int c = 0; c < kOut / 32; ++c) {
        const int col0 = n0 + c * 32;
        if (col0 >= N) break;
        uint32_t r[32], u[kSwi ? 32 : 1];
        tc::tmem_ld_32x32b_x32(tbase + c * 32, r);
        if (kSwi) tc::tmem_ld_32x32b_x32(tbase + kOut + c * 32, u);
        tc::tmem_wait_ld();
        if (row_ok) {
          bf16* dst = C + (int64_t)row * N + col0;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            if (col0 + g * 8 < N) {
              float v[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                float a = __uint_as_float(r[g * 8 + j]);
                if (be) a += be[col0 + g * 8 + j];
                if (kEpi == kEpiGelu) {
                  v[j] = gelu_erf(a);
                } else if (kSwi) {
                  float b = __uint_as_float(u[(g * 8 + j) % (kSwi ? 32 : 1)]);
                  if (be) b += be[N + col0 + g * 8 + j];
                  v[j] = silu_f(a) * b;
                } else {
                  v[j] = a;
                }
              }
              *reinterpret_cast<uint4*>(dst + g * 8) = Vec<bf16>::pack(v);
            }
          }
        }
      }
      tc::tc_fence_before();
      tc::mbar_arrive(tempty(acc));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  // after an abort, loads the producer issued but no MMA consumed must land before exit
  if (producer && s_abort)
    for (int s = 0; s < S; ++s)
      if ((filled >> s) & 1u) tc::mbar_wait(full(s), (fill_par >> s) & 1u, nullptr, kWaitNs);
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, Cf::kTmemCols);
  }
}

template <int BN, int kEpi>
cudaError_t run_gemm(const void* A, int64_t rows, const int32_t* offs, int E, const void* B, int N, int K,
                     const float* bias, void* C, int* err, cudaStream_t st, int stall) {
  using Cf = Cfg<BN>;
  CUtensorMap ma, mb;
  if (!tma_map_bf16(&ma, A, (uint64_t)rows, (uint64_t)K, kBM)) return cudaErrorNotSupported;
  constexpr bool kSwi = kEpi == kEpiSwiglu;
  if (!tma_map_bf16(&mb, B, (uint64_t)E * N * (kSwi ? 2 : 1), (uint64_t)K, kSwi ? BN / 2 : BN))
    return cudaErrorNotSupported;
  auto k = grouped_gemm_tc_kernel<BN, kEpi>;
  cudaError_t r = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cf::kSmem);
  if (r != cudaSuccess) return r;
  return launch_kernel(k, dim3(sm_count()), dim3(kThreads), Cf::kSmem, st, 1, ma, mb, offs, E, N, K, bias,
                       (bf16*)C, err, stall);
}

// 256-wide tiles unless 128-wide ones pad N less.
bool wide_tile(int N) {
  const int64_t p256 = (int64_t)((N + 255) / 256) * 256;
  const int64_t p128 = (int64_t)((N + 127) / 128) * 128;
  return p256 <= p128;
}

template <int kEpi>
cudaError_t run_product(const void* A, int64_t rows, const int32_t* offs, int E, const void* B, int N, int K,
                        const float* bias, void* C, int* err, cudaStream_t st, int stall = 0) {
  if (kEpi == kEpiSwiglu || wide_tile(N))
    return run_gemm<256, kEpi>(A, rows, offs, E, B, N, K, bias, C, err, st, stall);
  return run_gemm<128, kEpi == kEpiSwiglu ? kEpiPlain : kEpi>(A, rows, offs, E, B, N, K, bias, C, err, st, stall);
}

}  // namespace

cudaError_t launch_ffn_tc(const Shape& s, int64_t max_rows, const void* x_perm, const int32_t* offs,
                          const void* W1, const float* b1, const void* W2, const float* b2,
                          void* h_perm, void* y_perm, int* err, cudaStream_t st) {
  if (s.dtype != MOE_BF16 || max_rows <= 0 || max_rows >= ((int64_t)1 << 31)) return cudaErrorNotSupported;
  if ((int64_t)s.E * s.F >= ((int64_t)1 << 31) || (int64_t)s.E * s.H >= ((int64_t)1 << 31))
    return cudaErrorNotSupported;
  const int stall = (s.flags & MOE_FLAG_TEST_WAIT_TIMEOUT) ? 1 : 0;
  cudaError_t r = (s.flags & MOE_FLAG_SWIGLU)
                      ? run_product<kEpiSwiglu>(x_perm, max_rows, offs, s.E, W1, s.F, s.H, b1, h_perm, err, st, stall)
                      : run_product<kEpiGelu>(x_perm, max_rows, offs, s.E, W1, s.F, s.H, b1, h_perm, err, st, stall);
  if (r != cudaSuccess) return r;
  prof_mark(kMarkFirst, st);
  return run_product<kEpiPlain>(h_perm, max_rows, offs, s.E, W2, s.H, s.F, b2, y_perm, err, st);
}

}  // namespace moe
