// Router on the 5th-generation tensor cores (bf16 layers).
//
// Same operation as the CUDA-core router (Qwen2-MoE code walkthrough,
// jsqmd.com, section 3.1: bias-free gate linear, softmax, top-k, division of
// the k probabilities by their sum): scores l = x Wg^T (+ bias) accumulated in
// fp32; the k largest scores, largest first, equal scores by ascending expert
// index; w_j = exp((l_j - m)/tau) / sum_sel exp((l_i - m)/tau); p =
// softmax(l / tau) summed per expert for the load-balancing loss (tau = 1
// unless the layer sets a router temperature).
//
// The gate product is skinny (N = E <= 256) and its cost is reading x once,
// so the kernel is built to keep every SM streaming x at HBM speed until the
// end and to leave as little as possible after the last byte arrives:
//   * one CTA per SM; CTA c owns the tokens [c T / G, (c + 1) T / G) of the G
//     CTAs (at most one token more than any other CTA), split into sub-tiles
//     of at most 128 rows;
//   * a producer thread moves each k-block of a sub-tile (its token rows in
//     8-row boxes, 1 KB each, plus the k-block of Wg; 128-byte swizzle) into
//     a ring of stages; a stage holds the rows a 128-row MMA reads, so the
//     rows past the sub-tile read that stage's own Wg block or bytes no copy
//     writes, and the accumulator lanes they produce are never read;
//   * one thread issues tcgen05.mma M=128, N=E rounded up to 16, K=16 into
//     one of two TMEM accumulators, so a CTA with two sub-tiles streams the
//     second while the first one's epilogue runs;
//   * four epilogue warps (one per TMEM lane quarter) finish one token per
//     thread straight from TMEM: bias, top-k in k rounds (each round the best
//     entry ranked after the previous pick), softmax statistics, weights,
//     the per-expert probability sums (a 31-shuffle transpose-reduce per 32
//     experts, then the four warps in order) and the counts of the chosen
//     experts (the dispatch histogram of the CTA's slots, so the layer needs
//     no separate histogram pass);
//   * the epilogue warps run their code once on unused accumulator columns
//     while the first bytes stream (nothing is stored), so the real epilogue
//     does not wait on instruction fetches after the L2 has been flushed.
// Every mbarrier wait is bounded; on expiry the kernel records a timeout in
// the error word, skips the remaining work, waits for the copies it issued,
// frees TMEM and returns.
#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {

namespace {

constexpr int kBK = 64;                  // bf16 per k-block (128 bytes)
constexpr int kBoxRows = 8;              // token rows per TMA box
constexpr int kBoxBytes = kBoxRows * kBK * 2;
constexpr int kATile = 128 * kBK * 2;    // what one M = 128 MMA reads of A
constexpr int kMaxSub = 128;             // rows per sub-tile (TMEM lanes)
constexpr int kThreads = 256;
constexpr int kEpiWarp0 = 4;             // warps 4..7: the epilogue, lane quarter = warp % 4
constexpr int kEpiThreads = 128;
constexpr int kMaxStages = 16;
constexpr int kMinTokensPerCta = 16;
constexpr int kMaxCtas = 1024;
constexpr size_t kRingBudget = 216 * 1024;
constexpr uint64_t kWaitNs = 2000000000ull;

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// G: CTAs of the launch; every CTA owns at least kMinTokensPerCta tokens.
int64_t router_ctas(int64_t T, int sms) {
  int64_t g = (T + kMinTokensPerCta - 1) / kMinTokensPerCta;
  if (g > sms) g = sms;
  if (g > kMaxCtas) g = kMaxCtas;
  return g < 1 ? 1 : g;
}

// The 32 values v[0..31] of each lane summed over the warp's lanes: lane l
// ends with the sum for entry l in v[0] (each step hands half of the entries
// to the partner lane and adds the partner's half; a fixed order).
__device__ __forceinline__ float transpose_reduce(float (&v)[32], int lane) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool up = (lane & s) != 0;
#pragma unroll
    for (int i = 0; i < s; ++i) {
      const float send = up ? v[i] : v[i + s];
      const float keep = up ? v[i + s] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
    }
  }
  return v[0];
}

// Keep (v, e) if it ranks after the previous pick (score descending, index
// ascending) and before the best so far.
__device__ __forceinline__ void consider(float v, int e, float prev_v, int prev_i, float& bv, int& bi) {
  const bool after = v < prev_v || (v == prev_v && e > prev_i);
  const bool better = v > bv || (v == bv && e < bi);
  if (after && better) {
    bv = v;
    bi = e;
  }
}

struct EpiOut {
  const float* bias;   // shared [256]
  float* logits;
  int32_t* ids;
  float* w;
  int* hist;           // shared [256]
  float (*wsum)[256];  // shared [4][256]
};

// One sub-tile's epilogue on the 128 epilogue threads: the thread of lane
// quarter q and lane l finishes row 32 q + l of the accumulator at taddr
// (token t0 + row, if row < rows).  With `dry` nothing is stored and every
// row is treated as absent (an instruction warm-up).  Adds the sub-tile's
// probability sums of experts tid and tid + 128 (summed over the four warps
// in order) to ps[0] and ps[1] of epilogue thread tid.
template <bool kOneChunk>
__device__ __forceinline__ void epilogue_tile(uint32_t taddr, int64_t t0, int rows, bool dry, int E, int K,
                                              float inv_tau, const EpiOut& o, float (&ps)[2]) {
  const int lane = threadIdx.x & 31;
  const int q = (threadIdx.x >> 5) & 3;
  const int tid = (int)threadIdx.x - kEpiWarp0 * 32;
  const int row = q * 32 + lane;
  const bool live = !dry && row < rows;
  const int64_t t = t0 + row;
  const int nch = (E + 31) >> 5;
  float sel_v[8];
  int sel_i[8];
  float prev_v = INFINITY;
  int prev_i = -1;
  float zs = 0.f;
  float v1[32];                     // E <= 32: the scores, loaded once
  if constexpr (kOneChunk) {
    uint32_t r[32];
    tc::tmem_ld_32x32b_x32(taddr, r);
    tc::tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) v1[i] = i < E ? __uint_as_float(r[i]) + o.bias[i] : -INFINITY;
  }
  // k rounds, each the best entry ranked after the previous pick
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    sel_v[j] = -INFINITY;
    sel_i[j] = 0x7fffffff;
    if (j < K) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
      if constexpr (kOneChunk) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (i < E) consider(v1[i], i, prev_v, prev_i, bv, bi);
      } else {
#pragma unroll 1
        for (int c = 0; c < nch; ++c) {
          uint32_t r[32];
          tc::tmem_ld_32x32b_x32(taddr + (uint32_t)(32 * c), r);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int e = 32 * c + i;
            if (e < E) consider(__uint_as_float(r[i]) + o.bias[e], e, prev_v, prev_i, bv, bi);
          }
        }
      }
      sel_v[j] = bv;
      sel_i[j] = bi;
      prev_v = bv;
      prev_i = bi;
    }
  }
  const float m = sel_v[0];
  // softmax denominator, experts in ascending order
  if constexpr (kOneChunk) {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < E) zs += expf((v1[i] - m) * inv_tau);
  } else {
#pragma unroll 1
    for (int c = 0; c < nch; ++c) {
      uint32_t r[32];
      tc::tmem_ld_32x32b_x32(taddr + (uint32_t)(32 * c), r);
      tc::tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int e = 32 * c + i;
        if (e < E) zs += expf((__uint_as_float(r[i]) + o.bias[e] - m) * inv_tau);
      }
    }
  }
  const float inv = 1.f / zs;
  // routing weights of the chosen experts
  float z[8], zsel = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    z[j] = j < K ? expf((sel_v[j] - m) * inv_tau) : 0.f;
    zsel += z[j];
  }
  if (live) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < K) {
        o.ids[t * K + j] = sel_i[j];
        o.w[t * K + j] = z[j] / zsel;
        if ((unsigned)sel_i[j] < (unsigned)E) atomicAdd(&o.hist[sel_i[j]], 1);   // NaN scores: none
      }
    }
  }
  // probabilities summed over the warp's tokens, 32 experts at a time
#pragma unroll 1
  for (int c = 0; c < nch; ++c) {
    float p[32];
    if constexpr (kOneChunk) {
#pragma unroll
      for (int i = 0; i < 32; ++i) p[i] = v1[i];
    } else {
      uint32_t r[32];
      tc::tmem_ld_32x32b_x32(taddr + (uint32_t)(32 * c), r);
      tc::tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) p[i] = 32 * c + i < E ? __uint_as_float(r[i]) + o.bias[32 * c + i] : 0.f;
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int e = 32 * c + i;
      if (live && o.logits && e < E) o.logits[t * E + e] = p[i];
      p[i] = (live && e < E) ? expf((p[i] - m) * inv_tau) * inv : 0.f;
    }
    o.wsum[q][32 * c + lane] = transpose_reduce(p, lane);
  }
  epi_sync();
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int e = tid + h * kEpiThreads;
    if (e < E) ps[h] += ((o.wsum[0][e] + o.wsum[1][e]) + o.wsum[2][e]) + o.wsum[3][e];
  }
  epi_sync();   // wsum is free for the next sub-tile
}

__global__ void __launch_bounds__(kThreads, 1)
router_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmG, int64_t Tn,
                 int H, int E, int K, int npad, int acc_cols, int tmem_cols, int G, float inv_tau,
                 const float* __restrict__ gate_bias, float* __restrict__ logits, int32_t* __restrict__ ids,
                 float* __restrict__ w, float* __restrict__ psum_part, int32_t* __restrict__ tile_hist, int* err) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ float s_bias[256];
  __shared__ int s_hist[256];
  __shared__ float s_wsum[4][256];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ __align__(8) uint64_t s_bar[2 * kMaxStages + 5];

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t ring = tc::smem_u32(smem);
  const int warp = threadIdx.x >> 5;

  // this CTA's tokens and its stage layout
  const int c = blockIdx.x;
  const int64_t r0 = (int64_t)c * Tn / G, r1 = (int64_t)(c + 1) * Tn / G;
  const int n = (int)(r1 - r0);
  const int m = (n + kMaxSub - 1) / kMaxSub;          // sub-tiles
  const int qrows = (n + m - 1) / m;                  // rows per sub-tile (the last may have fewer)
  const int a_bytes = (qrows + kBoxRows - 1) / kBoxRows * kBoxBytes;
  const int b_bytes = npad * 128;
  const int stage_bytes = a_bytes + b_bytes > kATile ? a_bytes + b_bytes : kATile;
  int S = (int)(kRingBudget / (size_t)stage_bytes);
  if (S > kMaxStages) S = kMaxStages;
  const int nk = (H + kBK - 1) / kBK;
  const uint32_t idesc = tc::idesc_bf16_f32(128, npad);
  auto full = [&](int s) { return tc::smem_u32(&s_bar[s]); };
  auto empty = [&](int s) { return tc::smem_u32(&s_bar[kMaxStages + s]); };
  auto tfull = [&](int a) { return tc::smem_u32(&s_bar[2 * kMaxStages + a]); };
  auto tempty = [&](int a) { return tc::smem_u32(&s_bar[2 * kMaxStages + 2 + a]); };
  const uint32_t done_bar = tc::smem_u32(&s_bar[2 * kMaxStages + 4]);

  for (int e = threadIdx.x; e < 256; e += kThreads) s_hist[e] = 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(full(s), 1);
      tc::mbar_init(empty(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(tfull(a), 1);
      tc::mbar_init(tempty(a), kEpiThreads);
    }
    tc::mbar_init(done_bar, 1);
    s_abort = 0;
    tc::fence_barrier_init();
    tc::fence_proxy_async_smem();
    tc::prefetch_tmap(&tmX);
    tc::prefetch_tmap(&tmG);
  }
  if (warp == 1) {
    tc::tmem_alloc(tc::smem_u32(&s_tmem), tmem_cols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = s_tmem;

  uint32_t filled = 0, fill_par = 0;   // producer: per stage, ever filled / parity of its last fill
  bool producer = false;
  if (warp == 0) {
    pdl_enter();
    // ------------------------------------------------------------ TMA producer
    if (tc::elect_one()) {
      producer = true;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int i = 0; i < m && ok; ++i) {
        const int64_t row0 = r0 + (int64_t)i * qrows;
        const int rows = (int)min((int64_t)qrows, r1 - row0);
        const int nbox = (rows + kBoxRows - 1) / kBoxRows;
        for (int kb = 0; kb < nk; ++kb) {
          if (!tc::mbar_wait(empty(stage), phase ^ 1u, &s_abort, kWaitNs)) { ok = false; break; }
          const uint32_t base = ring + (uint32_t)(stage * stage_bytes);
          tc::mbar_arrive_expect_tx(full(stage), (uint32_t)(nbox * kBoxBytes + b_bytes));
          for (int bx = 0; bx < nbox; ++bx)
            tc::tma_load_2d(base + (uint32_t)(bx * kBoxBytes), &tmX, full(stage), kb * kBK,
                            (int)(row0 + bx * kBoxRows));
          tc::tma_load_2d(base + (uint32_t)a_bytes, &tmG, full(stage), kb * kBK, 0);
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
    pdl_wait();
    // ------------------------------------------------------------ MMA issuer
    if (tc::elect_one()) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t epar[2] = {1u, 0u};    // accumulator 1 is first freed by the warm-up pass
      bool ok = true;
      for (int i = 0; i < m && ok; ++i) {
        const int acc = i & 1;
        if (!tc::mbar_wait(tempty(acc), epar[acc], &s_abort, kWaitNs)) { ok = false; break; }
        epar[acc] ^= 1u;
        tc::tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(acc * acc_cols);
        for (int kb = 0; kb < nk; ++kb) {
          if (!tc::mbar_wait(full(stage), phase, &s_abort, kWaitNs)) { ok = false; break; }
          tc::tc_fence_after();
          const uint32_t a0 = ring + (uint32_t)(stage * stage_bytes), b0 = a0 + (uint32_t)a_bytes;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            tc::mma_bf16(d, tc::sdesc_k128(a0 + k * 32), tc::sdesc_k128(b0 + k * 32), idesc, (kb | k) ? 1u : 0u);
          tc::tc_commit(empty(stage));
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
        if (ok) tc::tc_commit(tfull(acc));   // arrives once the sub-tile's MMAs are done
      }
      if (!ok) {
        set_error(err, kDevTimeout);
        s_abort = 1;
      }
      tc::tc_commit(done_bar);   // arrives once every MMA above has finished
    }
    __syncwarp();
    if ((threadIdx.x & 31) == 0 && !tc::mbar_wait(done_bar, 0, nullptr, kWaitNs)) set_error(err, kDevTimeout);
    __syncwarp();
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------ epilogue
    const int tid = (int)threadIdx.x - kEpiWarp0 * 32;
    const uint32_t tq = tmem + ((uint32_t)(((warp & 3) * 32)) << 16);
    EpiOut o{s_bias, logits, ids, w, s_hist, s_wsum};
    const bool one = E <= 32;
    float psum[2] = {0.f, 0.f}, dummy[2] = {0.f, 0.f};
    // warm-up on accumulator 1 (no MMA writes it before this pass frees it)
    if (one) epilogue_tile<true>(tq + (uint32_t)acc_cols, 0, 0, true, E, K, inv_tau, o, dummy);
    else epilogue_tile<false>(tq + (uint32_t)acc_cols, 0, 0, true, E, K, inv_tau, o, dummy);
    tc::tc_fence_before();
    tc::mbar_arrive(tempty(1));
    pdl_wait();
    for (int e = tid; e < 256; e += kEpiThreads) s_bias[e] = (gate_bias && e < E) ? gate_bias[e] : 0.f;
    epi_sync();
    uint32_t fpar[2] = {0u, 0u};
    bool ok = true;
    for (int i = 0; i < m; ++i) {
      const int acc = i & 1;
      if (ok && !tc::mbar_wait(tfull(acc), fpar[acc], &s_abort, kWaitNs)) {
        set_error(err, kDevTimeout);
        s_abort = 1;
        ok = false;
      }
      fpar[acc] ^= 1u;
      tc::tc_fence_after();
      const int64_t row0 = r0 + (int64_t)i * qrows;
      const int rows = ok ? (int)min((int64_t)qrows, r1 - row0) : 0;
      // an aborted pass still runs (storing nothing) so the named barriers match
      if (one) epilogue_tile<true>(tq + (uint32_t)(acc * acc_cols), row0, rows, !ok, E, K, inv_tau, o, psum);
      else epilogue_tile<false>(tq + (uint32_t)(acc * acc_cols), row0, rows, !ok, E, K, inv_tau, o, psum);
      tc::tc_fence_before();
      tc::mbar_arrive(tempty(acc));
    }
    if (ok) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int e = tid + h * kEpiThreads;
        if (e < E) {
          if (psum_part) psum_part[(int64_t)c * E + e] = psum[h];
          if (tile_hist) tile_hist[(int64_t)c * E + e] = s_hist[e];
        }
      }
    }
  } else {
    pdl_wait();
  }

  tc::tc_fence_before();
  __syncthreads();
  // after an abort, copies issued but never consumed land before the CTA exits
  if (producer && s_abort)
    for (int s = 0; s < S; ++s)
      if ((filled >> s) & 1u) tc::mbar_wait(full(s), (fill_par >> s) & 1u, nullptr, kWaitNs);
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, tmem_cols);
  }
}

struct RouterCfg {
  int npad, acc_cols, tmem_cols;
  int64_t ctas;
  size_t smem;
};

RouterCfg router_cfg(const Shape& s) {
  RouterCfg c;
  c.npad = s.E < 16 ? 16 : (s.E + 15) / 16 * 16;
  c.acc_cols = (c.npad + 31) / 32 * 32;
  c.tmem_cols = 32;
  while (c.tmem_cols < 2 * c.acc_cols) c.tmem_cols *= 2;
  c.ctas = router_ctas(s.T, sm_count());
  c.smem = 1024 + kRingBudget;
  return c;
}

}  // namespace

int64_t router_tc_partials(const Shape& s) { return router_ctas(s.T, sm_count()); }

int64_t router_tc_partials_bound(const Shape& s) {
  int64_t g = (s.T + kMinTokensPerCta - 1) / kMinTokensPerCta;
  return g > kMaxCtas ? kMaxCtas : (g < 1 ? 1 : g);
}

bool router_on_tensor_cores(const Shape& s) {
  return s.dtype == MOE_BF16 && s.H >= kBK && s.E <= 256 && !(s.flags & MOE_FLAG_SIMT_ROUTER);
}

cudaError_t launch_router_tc(const Shape& s, const void* x, const void* Wg, const float* gate_bias,
                             float* logits, int32_t* ids, float* w, float* psum_part,
                             int32_t* tile_hist, int* err, cudaStream_t st) {
  const RouterCfg c = router_cfg(s);
  CUtensorMap mx, mg;
  if (!tma_map_bf16(&mx, x, (uint64_t)s.T, (uint64_t)s.H, kBoxRows)) return cudaErrorNotSupported;
  if (!tma_map_bf16(&mg, Wg, (uint64_t)s.E, (uint64_t)s.H, (uint32_t)c.npad)) return cudaErrorNotSupported;
  auto kern = router_tc_kernel;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)c.smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, dim3((unsigned)c.ctas), dim3(kThreads), c.smem, st, 1, mx, mg, s.T, s.H, s.E, s.K,
                       c.npad, c.acc_cols, c.tmem_cols, (int)c.ctas, s.inv_tau, gate_bias, logits, ids, w,
                       psum_part, tile_hist, err);
}

}  // namespace moe
