// Expert FFN on CTA pairs: the grouped GEMM of ffn_tc.cu with 256 x 256
// output tiles computed by the two SMs of a 2-CTA cluster (tcgen05
// .cta_group::2).
//
// Same products (Qwen2-MoE module article, mlqm.cn, section 2.2: each expert
// is Linear -> GELU -> Linear):
//   first:  h = GELU(x_perm W1[e]^T + b1[e]);  second: y = h W2[e]^T + b2[e]
//
// Why pairs: with one SM per 128 x 256 tile, every k-block brings 48 KB into
// the SM (A 16 KB + B 32 KB) for 128 x 256 x 64 multiply-adds, and the
// measured kernel was bound by that load stream rather than by the tensor
// cores.  A pair computes 256 x 256 per k-block while each SM loads only its
// own 128 rows of A and its own 128 rows (N half) of B: 32 KB per SM for the
// same work per SM.  The price is that expert segments are padded to 256
// rows instead of 128.
//
// Roles, per CTA (192 threads), rank r = 0 (leader) or 1:
//   warp 0     TMA producer: A rows [row0 + 128 r, +128) and B rows
//              [n0 + 128 r, +128) of each k-block into this CTA's ring; both
//              CTAs' loads complete on the LEADER's `full` barrier, which the
//              leader arms for the 64 KB of the pair;
//   warp 1     leader only: one thread issues tcgen05.mma.cta_group::2
//              (M = 256, N = 256, K = 16) x 4 per stage; its commits arrive on
//              the `empty` / `tfull` barriers of both CTAs (multicast);
//   warps 2-5  epilogue in both CTAs: this CTA's 128 accumulator rows from its
//              own TMEM -> bias -> GELU -> bf16 -> global; then arrive on the
//              leader's `tempty` (256 arrivals = both CTAs).
// All waits are bounded (timeout -> error word + abort flag); the CTAs meet
// in cluster barriers after set-up and before exit so neither can touch the
// other's shared memory once it has left.
#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {

namespace {

constexpr int kBM = 128;             // rows per CTA (the pair covers 256)
constexpr int kBNh = 128;            // B rows per CTA (the pair covers N = 256)
constexpr int kBK = 64;
constexpr int kThreads = 192;
constexpr int kABytes = kBM * kBK * 2;
constexpr int kBBytes = kBNh * kBK * 2;
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kStages = 6;
constexpr int kTmemCols = 512;       // two 256-column accumulators
constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes;
constexpr uint64_t kWaitNs = 2000000000ull;

// kEpi = kEpiSwiglu: B = [W1; W3] stacked per expert ([E, 2N, K]); the
// leader loads 128 gate rows and the peer the matching 128 up rows, so each
// CTA's 256 accumulator columns are gate | up for 128 output columns.
template <int kEpi>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const int32_t* __restrict__ offs, int E, int N, int K,
                         const float* __restrict__ bias, bf16* __restrict__ C, int* err) {
  constexpr int S = kStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_offs[257];
  __shared__ int s_tstart[257];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ __align__(8) uint64_t s_bar[2 * S + 5];

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sA = tc::smem_u32(smem);
  const uint32_t sB = sA + S * kABytes;
  auto full = [&](int s) { return tc::smem_u32(&s_bar[s]); };
  auto empty = [&](int s) { return tc::smem_u32(&s_bar[S + s]); };
  auto tfull = [&](int a) { return tc::smem_u32(&s_bar[2 * S + a]); };
  auto tempty = [&](int a) { return tc::smem_u32(&s_bar[2 * S + 2 + a]); };
  const uint32_t done_bar = tc::smem_u32(&s_bar[2 * S + 4]);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = tc::cluster_ctarank();          // 0 = leader
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  constexpr bool kSwi = kEpi == kEpiSwiglu;
  constexpr int kOut = kSwi ? kBNh : 2 * kBNh;   // output columns per pair tile
  const int nt = (N + kOut - 1) / kOut;
  const int nk = (K + kBK - 1) / kBK;
  constexpr uint32_t kIdesc = tc::idesc_bf16_f32(2 * kBM, 2 * kBNh);

  if (warp == 0) {
    pdl_enter();   // the tile table reads offs, written by the previous kernel
    // per-expert pair-tile counts (256-row m-tiles x n-tiles) and their prefix
    int loc[8];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      int v = 0;
      if (e < E) {
        const int o0 = offs[e], o1 = offs[e + 1];
        v = ((o1 - o0 + 2 * kBM - 1) / (2 * kBM)) * nt;
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
        tc::mbar_init(full(s), 1);       // used in the leader: its arm + both CTAs' bytes
        tc::mbar_init(empty(s), 1);      // one multicast commit per use
      }
      for (int a = 0; a < 2; ++a) {
        tc::mbar_init(tfull(a), 1);
        tc::mbar_init(tempty(a), 2 * 128);   // used in the leader: both CTAs' epilogue threads
      }
      tc::mbar_init(done_bar, 1);
      s_abort = 0;
      tc::fence_barrier_init();
      tc::fence_proxy_async_smem();
      tc::prefetch_tmap(&tmA);
      tc::prefetch_tmap(&tmB);
    }
  } else if (warp == 1) {
    tc::tmem_alloc_pair(tc::smem_u32(&s_tmem), kTmemCols);
    tc::tmem_relinquish_pair();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::cluster_sync();             // both CTAs' barriers exist before either signals the other
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
    const int mt = (s_offs[e + 1] - s_offs[e] + 2 * kBM - 1) / (2 * kBM);
    const int local = t - s_tstart[e];
    row0 = s_offs[e] + (local % mt) * (2 * kBM) + (int)rank * kBM;   // this CTA's half
    row_end = s_offs[e + 1];
    n0 = (local / mt) * kOut;
  };

  uint32_t filled = 0, fill_par = 0;   // producer: per stage, ever filled / parity of its last fill
  bool producer = false;
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (tc::elect_one()) {
      producer = true;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = pair; t < total && ok; t += npairs) {
        int e, row0, row_end, n0;
        decode(t, e, row0, row_end, n0);
        for (int kb = 0; kb < nk; ++kb) {
          if (!tc::mbar_wait(empty(stage), phase ^ 1u, &s_abort, kWaitNs)) { ok = false; break; }
          const uint32_t fbar = tc::map_peer(full(stage), 0);
          if (rank == 0) tc::mbar_arrive_expect_tx(full(stage), 2 * kStageBytes);
          tc::tma_load_2d_pair(sA + stage * kABytes, &tmA, fbar, kb * kBK, row0);
          tc::tma_load_2d_pair(sB + stage * kBBytes, &tmB, fbar, kb * kBK,
                               kSwi ? 2 * e * N + (int)rank * N + n0 : e * N + n0 + (int)rank * kBNh);
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
    // ------------------------------------------------------------ MMA issuer (leader)
    if (rank == 0 && tc::elect_one()) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int t = pair; t < total && ok; t += npairs) {
        if (!tc::mbar_wait(tempty(acc), acc_phase ^ 1u, &s_abort, kWaitNs)) { ok = false; break; }
        tc::tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(acc * 2 * kBNh);
        for (int kb = 0; kb < nk; ++kb) {
          if (!tc::mbar_wait(full(stage), phase, &s_abort, kWaitNs)) { ok = false; break; }
          tc::tc_fence_after();
          const uint32_t a0 = sA + stage * kABytes, b0 = sB + stage * kBBytes;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            tc::mma_bf16_pair(d, tc::sdesc_k128(a0 + k * 32), tc::sdesc_k128(b0 + k * 32), kIdesc,
                              (kb | k) != 0);
          tc::tc_commit_pair_mc(empty(stage), 0x3);
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc::tc_commit_pair_mc(tfull(acc), 0x3);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok) {
        set_error(err, kDevTimeout);
        s_abort = 1;
      }
      // both CTAs learn when every MMA (which writes both TMEMs) has finished
      tc::tc_commit_pair_mc(done_bar, 0x3);
    }
    __syncwarp();
    if (lane == 0 && !tc::mbar_wait(done_bar, 0, nullptr, kWaitNs)) set_error(err, kDevTimeout);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = pair; t < total; t += npairs) {
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
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * 2 * kBNh);
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
      if (rank == 0) tc::mbar_arrive(tempty(acc));
      else tc::mbar_arrive_remote(tc::map_peer(tempty(acc), 0));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  // after an abort the leader drains its stage barriers, on which both CTAs'
  // loads complete, before either CTA may leave
  if (producer && rank == 0 && s_abort)
    for (int s = 0; s < S; ++s)
      if ((filled >> s) & 1u) tc::mbar_wait(full(s), (fill_par >> s) & 1u, nullptr, kWaitNs);
  tc::cluster_sync();             // neither CTA leaves while the other may still signal it
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc_pair(tmem, kTmemCols);
  }
}

template <int kEpi>
cudaError_t run_pair(const void* A, int64_t rows, const int32_t* offs, int E, const void* B, int N, int K,
                     const float* bias, void* C, int* err, cudaStream_t st) {
  CUtensorMap ma, mb;
  if (!tma_map_bf16(&ma, A, (uint64_t)rows, (uint64_t)K, kBM)) return cudaErrorNotSupported;
  if (!tma_map_bf16(&mb, B, (uint64_t)E * N * (kEpi == kEpiSwiglu ? 2 : 1), (uint64_t)K, kBNh))
    return cudaErrorNotSupported;
  auto kern = grouped_gemm_pair_kernel<kEpi>;
  cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
  if (r != cudaSuccess) return r;
  // one resident pair per two SMs (persistent); never more pairs than fit at once
  int pairs = sm_count() / 2;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
  int fit = 0;
  if (cudaOccupancyMaxActiveClusters(&fit, kern, &cfg) == cudaSuccess && fit > 0 && fit < pairs) pairs = fit;
  return launch_kernel(kern, dim3((unsigned)(2 * pairs)), dim3(kThreads), kSmem, st, 2, ma, mb, offs, E, N, K,
                       bias, (bf16*)C, err);
}

}  // namespace

cudaError_t launch_ffn_tc_pair(const Shape& s, int64_t max_rows, const void* x_perm, const int32_t* offs,
                               const void* W1, const float* b1, const void* W2, const float* b2,
                               void* h_perm, void* y_perm, int* err, cudaStream_t st) {
  if (s.dtype != MOE_BF16 || max_rows <= 0 || max_rows >= ((int64_t)1 << 31)) return cudaErrorNotSupported;
  if ((int64_t)s.E * s.F >= ((int64_t)1 << 31) || (int64_t)s.E * s.H >= ((int64_t)1 << 31))
    return cudaErrorNotSupported;
  cudaError_t r = (s.flags & MOE_FLAG_SWIGLU)
                      ? run_pair<kEpiSwiglu>(x_perm, max_rows, offs, s.E, W1, s.F, s.H, b1, h_perm, err, st)
                      : run_pair<kEpiGelu>(x_perm, max_rows, offs, s.E, W1, s.F, s.H, b1, h_perm, err, st);
  if (r != cudaSuccess) return r;
  prof_mark(kMarkFirst, st);
  return run_pair<kEpiPlain>(h_perm, max_rows, offs, s.E, W2, s.H, s.F, b2, y_perm, err, st);
}

}  // namespace moe
