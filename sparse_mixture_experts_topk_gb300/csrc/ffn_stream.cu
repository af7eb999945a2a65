// Expert FFN for decode-sized batches (at most 16 tokens): weight streaming.
//
// Same products as the grouped GEMMs (Qwen2-MoE module article, mlqm.cn,
// section 2.2: each expert is Linear -> GELU -> Linear), for segments of at
// most 16 rows.  The time is reading every used expert's weights once, so
// the kernel is built around bytes in flight rather than arithmetic:
//   * one CTA per SM (two for batches of at most 2 tokens); CTA b serves
//     the (b mod A)-th of the A experts that have rows (found from offs with
//     a warp ballot), and the CTAs of one expert split its output columns
//     into contiguous ranges;
//   * a producer thread moves the expert's activation rows and then, stage
//     after stage, `rps` consecutive weight rows (one untiled bulk copy per
//     stage; SwiGLU: a second copy for the matching up rows) into a ring of
//     2-6 stages in shared memory (as many as fit beside the expert's
//     activation rows): 100-200 KB in flight per SM;
//   * consumer warps dot the staged weight rows with every activation row
//     (bf16 operands multiplied into fp32 sums over 16-byte vectors, a
//     shuffle reduction per row), add the bias, apply the activation and
//     store one output value per row; row r of the CTA's range goes to
//     warp r mod 8;
//   * both products run in one launch: the ring carries the first product's
//     weight rows and then the second's, so the second product's weights
//     stream right behind the first's, and its activation rows (the first
//     product's outputs for the expert) are loaded once every CTA of the
//     expert has stored and fenced its share (a per-expert counter).
// Every mbarrier wait and counter wait is bounded; on expiry the kernel
// records a timeout in the error word, lets the other warps leave, waits
// (bounded) for the copies it issued and returns.
#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "stream_body.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

using stream::kConsumers;
using stream::kWaitNs;
using stream::stage_row;
using stream::stage_row_of_warp;
using stream::wait_count;

constexpr int kMaxRows = 16;
constexpr int kThreads = (kConsumers + 1) * 32;  // + one producer warp
constexpr int kMaxStages = 6;
constexpr size_t kSmemBudget = 220 * 1024;

__host__ __device__ inline size_t act_bytes(int mcap, int K, int esize) { return ((size_t)mcap * K * esize + 127) / 128 * 128; }

// One product of a launch: activation rows A [rows, K], weights B
// [E, N, K] (SwiGLU: [E, 2N, K]), nullable bias, output rows C [rows, N],
// rps weight rows per ring stage.
template <typename T>
struct StreamProduct {
  const T* A;
  const T* B;
  const float* bias;
  T* C;
  int N, K, rps;
};

// The CTA's share of one product: its expert's output columns [n_begin,
// n_end) (the CTAs of an expert split them into contiguous ranges) in
// `groups` ring stages of rps rows.
struct StreamRange {
  int n_begin, n_end, groups;
};
__device__ __forceinline__ StreamRange stream_range(int N, int rps, int nblk, int slot) {
  StreamRange r;
  const int per = (N + nblk - 1) / nblk;
  r.n_begin = slot * per;
  r.n_end = min(N, r.n_begin + per);
  r.groups = r.n_begin < r.n_end ? (r.n_end - r.n_begin + rps - 1) / rps : 0;
  return r;
}

// nphase = 1: the product P0 (activation kEpi).  nphase = 2: P0, then the
// plain product P1 whose activation rows are P0's output rows of the same
// expert.  One weight ring runs through both, so the second product's
// weights stream right behind the first's; the second product's activation
// rows are loaded once every CTA of the expert has stored (and fenced) its
// share of them: each CTA adds 1 to done[e] after its first-product rows,
// and the CTA's first consumer waits (bounded) for done[e] to reach the
// expert's CTA count.  Every CTA finishes its first-product rows without
// waiting on another CTA, so every such wait ends.
template <typename T, int kEpi, int kMR>
__global__ void __launch_bounds__(kThreads, kMR <= 2 ? 2 : 1)
stream_ffn_kernel(StreamProduct<T> P0, StreamProduct<T> P1, int nphase, const int32_t* __restrict__ offs, int E,
                  int mcap, uint32_t dyn_bytes, int* __restrict__ done, int* err) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_e, s_na, s_abort, s_act1;
  __shared__ __align__(8) uint64_t s_bar[2 * kMaxStages + 1];
  constexpr bool kSwi = kEpi == kEpiSwiglu;
  constexpr int V = Vec<T>::N;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t s_act = tc::smem_u32(smem);
  auto full = [&](int s) { return tc::smem_u32(&s_bar[s]); };
  auto empty = [&](int s) { return tc::smem_u32(&s_bar[kMaxStages + s]); };
  const uint32_t act_bar = tc::smem_u32(&s_bar[2 * kMaxStages]);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      tc::mbar_init(full(s), 1);
      tc::mbar_init(empty(s), kConsumers);
    }
    tc::mbar_init(act_bar, 1);
    s_abort = 0;
    s_act1 = 0;
    tc::fence_barrier_init();
  }
  pdl_enter();
  if (warp == 0) {
    // the experts with rows: how many (na), and the (blockIdx.x mod na)-th;
    // all of offs is read in one round (E <= 256: 8 chunks of 32)
    unsigned bal[8];
    int na = 0;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int e = c * 32 + lane;
      bal[c] = __ballot_sync(0xffffffffu, e < E && offs[e + 1] > offs[e]);
      na += __popc(bal[c]);
    }
    int found = -1;
    if (na > 0) {
      int want = (int)(blockIdx.x % (unsigned)na);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int cnt = __popc(bal[c]);
        if (found < 0 && want < cnt) {
          const bool mine = ((bal[c] >> lane) & 1u) && __popc(bal[c] & lanemask_lt()) == want;
          found = c * 32 + __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
        }
        if (found < 0) want -= cnt;
      }
    }
    if (lane == 0) {
      s_e = found;
      s_na = na;
    }
  }
  __syncthreads();
  const int e = s_e, na = s_na;
  if (e < 0) return;
  const int r0 = offs[e];
  int m = offs[e + 1] - r0;
  if (m > mcap) {                               // more rows than staged: report, compute the first mcap
    if (threadIdx.x == 0) set_error(err, kDevBadIndex);
    m = mcap;
  }
  // the expert's activation rows first, then the ring in the rest of the
  // shared memory.  The launch's P0.rps rows per stage leave room for two
  // stages beside mcap rows; with fewer rows staged the CTA takes the most
  // rows per stage (up to kConsumers) that still leave three stages, and as
  // many stages as fit.  A second-product stage holds as many of its rows
  // as fit the same bytes.
  const uint32_t act_room = (uint32_t)max(act_bytes(m, P0.K, sizeof(T)),
                                          nphase > 1 ? act_bytes(m, P1.K, sizeof(T)) : (size_t)0);
  const uint32_t row0 = (uint32_t)P0.K * sizeof(T), row1 = (uint32_t)P1.K * sizeof(T);
  const uint32_t room = dyn_bytes - act_room, wrow0 = row0 * (kSwi ? 2u : 1u);
  int rps0 = P0.rps;
  for (int r = kConsumers; r > P0.rps; r >>= 1)
    if (room / ((uint32_t)r * wrow0) >= 3u) {
      rps0 = r;
      break;
    }
  const uint32_t stage_bytes = (uint32_t)rps0 * wrow0;
  const int rps1 = min(kConsumers, (int)(stage_bytes / row1));
  const int stages = min(kMaxStages, (int)(room / stage_bytes));
  const uint32_t s_ring = s_act + act_room;
  // this CTA's share of expert e in each product
  const int a = (int)(blockIdx.x % (unsigned)na);
  const int nblk = ((int)gridDim.x - 1 - a) / na + 1;
  const int slot = (int)(blockIdx.x / (unsigned)na);
  const StreamRange R0 = stream_range(P0.N, rps0, nblk, slot);
  const StreamRange R1 = nphase > 1 ? stream_range(P1.N, rps1, nblk, slot) : StreamRange{0, 0, 0};
  const int total = R0.groups + R1.groups;

  uint32_t filled = 0, fill_par = 0;   // producer: per stage, ever filled / parity of its last fill
  bool producer = false;
  if (warp == kConsumers) {
    // ------------------------------------------------------------ producer
    if (tc::elect_one()) {
      producer = true;
      tc::mbar_arrive_expect_tx(act_bar, (uint32_t)m * row0);
      tc::bulk_load(s_act, P0.A + (int64_t)r0 * P0.K, (uint32_t)m * row0, act_bar);
      bool ok = true;
      for (int g = 0; g < total; ++g) {
        const int s = g % stages;
        const uint32_t ph = (uint32_t)(g / stages) & 1u;
        if (!tc::mbar_wait(empty(s), ph ^ 1u, &s_abort, kWaitNs)) { ok = false; break; }
        const uint32_t dst = s_ring + (uint32_t)s * stage_bytes;
        if (g < R0.groups) {
          const int n0 = R0.n_begin + g * rps0;
          const uint32_t bytes = (uint32_t)min(rps0, R0.n_end - n0) * row0;
          const T* Be = P0.B + (int64_t)e * P0.N * P0.K * (kSwi ? 2 : 1);
          tc::mbar_arrive_expect_tx(full(s), kSwi ? 2 * bytes : bytes);
          tc::bulk_load(dst, Be + (int64_t)n0 * P0.K, bytes, full(s));
          if (kSwi) tc::bulk_load(dst + (uint32_t)rps0 * row0, Be + (int64_t)(P0.N + n0) * P0.K, bytes, full(s));
        } else {
          const int n0 = R1.n_begin + (g - R0.groups) * rps1;
          const uint32_t bytes = (uint32_t)min(rps1, R1.n_end - n0) * row1;
          tc::mbar_arrive_expect_tx(full(s), bytes);
          tc::bulk_load(dst, P1.B + ((int64_t)e * P1.N + n0) * P1.K, bytes, full(s));
        }
        filled |= 1u << s;
        fill_par = (fill_par & ~(1u << s)) | (ph << s);
      }
      if (!ok) {
        set_error(err, kDevTimeout);
        s_abort = 1;
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ consumers
    // After a failed wait a warp does no more work but still passes the
    // consumers' barrier below, so the other consumer warps never wait there
    // for it (and every later wait of theirs sees the abort flag).
    const uint4* act = reinterpret_cast<const uint4*>(smem);
    const uint8_t* ring = smem + act_room;
    bool ok = tc::mbar_wait(act_bar, 0, &s_abort, kWaitNs);
    for (int g = 0; g < R0.groups; ++g) {
      const int s = g % stages;
      const uint32_t ph = (uint32_t)(g / stages) & 1u;
      if (!ok || !tc::mbar_wait(full(s), ph, &s_abort, kWaitNs)) { ok = false; continue; }
      const int j = stage_row_of_warp(g, rps0, warp);
      const int n = R0.n_begin + g * rps0 + j;
      if (j < rps0 && n < R0.n_end)
        stage_row<T, kEpi, kMR>(ring + (size_t)s * stage_bytes, j, rps0, row0, act, P0.K / V, m,
                                P0.bias ? P0.bias + (int64_t)e * P0.N * (kSwi ? 2 : 1) : nullptr, n, P0.N,
                                P0.C + (int64_t)r0 * P0.N + n);
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(empty(s));   // this warp is done with the stage
    }
    if (nphase > 1) {
      // the first product is done here: its outputs fenced, the CTAs of the
      // expert counted, then the second product's activation rows loaded
      __threadfence();
      asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
      if (warp == 0 && lane == 0) {
        atomicAdd(done + e, 1);
        if (ok && wait_count(done + e, nblk, &s_abort)) {
          tc::mbar_arrive_expect_tx(act_bar, (uint32_t)m * row1);
          tc::bulk_load(s_act, P1.A + (int64_t)r0 * P1.K, (uint32_t)m * row1, act_bar);
          s_act1 = 1;
        } else {
          s_abort = 1;
        }
      }
      ok = ok && tc::mbar_wait(act_bar, 1, &s_abort, kWaitNs);
      for (int g = R0.groups; g < total; ++g) {
        const int s = g % stages;
        const uint32_t ph = (uint32_t)(g / stages) & 1u;
        if (!ok || !tc::mbar_wait(full(s), ph, &s_abort, kWaitNs)) { ok = false; continue; }
        const int j = stage_row_of_warp(g - R0.groups, rps1, warp);
        const int n = R1.n_begin + (g - R0.groups) * rps1 + j;
        if (j < rps1 && n < R1.n_end)
          stage_row<T, kEpiPlain, kMR>(ring + (size_t)s * stage_bytes, j, rps1, row1, act, P1.K / V, m,
                                       P1.bias ? P1.bias + (int64_t)e * P1.N : nullptr, n, P1.N,
                                       P1.C + (int64_t)r0 * P1.N + n);
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(empty(s));
      }
    }
    if (!ok) {
      if (lane == 0) set_error(err, kDevTimeout);
      s_abort = 1;
    }
  }
  __syncthreads();
  // after an abort, copies issued but never consumed land before the CTA leaves
  if (producer && s_abort) {
    tc::mbar_wait(act_bar, 0, nullptr, kWaitNs);
    if (s_act1) tc::mbar_wait(act_bar, 1, nullptr, kWaitNs);
    for (int s = 0; s < stages; ++s)
      if ((filled >> s) & 1u) tc::mbar_wait(full(s), (fill_par >> s) & 1u, nullptr, kWaitNs);
  }
}

// Rows per stage for one product, and the ring depth it guarantees: the
// most rows per stage (8, 4, 2 or 1) that leave room for two stages beside
// act_max bytes of activation rows (mcap rows).  The launch takes the whole
// budget of shared memory; in it an expert's activation rows come first and
// the ring takes what is left, so an expert with fewer rows gets a deeper
// ring (at one activation row of 7 KB, three 8-row stages instead of two).
struct StreamCfg {
  int rps, stages;   // stages: the depth with mcap rows staged
  size_t smem;
};

StreamCfg stream_cfg_room(size_t act_max, size_t row, size_t budget = kSmemBudget) {
  StreamCfg c{1, 0, budget};
  for (int rps = kConsumers; rps >= 1; rps /= 2) {
    const size_t lo = budget > act_max ? (budget - act_max) / ((size_t)rps * row) : 0;
    if (lo >= 2 || rps == 1) {
      c.rps = rps;
      c.stages = (int)std::min<size_t>(lo, kMaxStages);
      break;
    }
  }
  return c;
}

StreamCfg stream_cfg(int mcap, int K, int esize, bool swi) {
  return stream_cfg_room(act_bytes(mcap, K, esize), (size_t)K * esize * (swi ? 2 : 1));
}

// Both products in one launch: one ring whose stages hold rps0 rows of the
// first product's weights (gate and up rows for SwiGLU) and rps1 rows of
// the second's, beside activation rows of the wider of the two.
struct StreamFused {
  bool ok;
  StreamCfg c;
  int rps1;
  uint32_t stage_bytes;
};

// Batches of at most kPairRows tokens run two CTAs per SM (bodies for at
// most 2 rows, so both fit the register file), each with half the ring.
constexpr int kPairRows = 2;

StreamFused stream_fused_cfg(const Shape& s) {
  StreamFused f{};
  const int mcap = (int)(s.T < kMaxRows ? s.T : kMaxRows);
  const bool swi = (s.flags & MOE_FLAG_SWIGLU) != 0;
  const int es = s.esize();
  const size_t act = std::max(act_bytes(mcap, s.H, es), act_bytes(mcap, s.F, es));
  f.c = stream_cfg_room(act, (size_t)s.H * es * (swi ? 2 : 1), mcap <= kPairRows ? kSmemBudget / 2 : kSmemBudget);
  f.stage_bytes = (uint32_t)((size_t)f.c.rps * s.H * es * (swi ? 2 : 1));
  const size_t r1 = f.stage_bytes / ((size_t)s.F * es);
  f.rps1 = (int)(r1 < (size_t)kConsumers ? r1 : kConsumers);
  f.ok = f.c.stages >= 2 && f.rps1 >= 1;
  return f;
}

template <typename T>
cudaError_t run_stream(const Shape& s, const void* x_perm, const int32_t* offs, const void* W1,
                       const float* b1, const void* W2, const float* b2, void* h_perm, void* y_perm,
                       int* err, int32_t* sched, cudaStream_t st) {
  const bool swi = (s.flags & MOE_FLAG_SWIGLU) != 0;
  const int64_t experts = s.S() < s.E ? s.S() : s.E;   // at most T*K experts have rows
  const int mcap = (int)(s.T < kMaxRows ? s.T : kMaxRows);
  auto k1 = swi ? stream_ffn_kernel<T, kEpiSwiglu, kMaxRows> : stream_ffn_kernel<T, kEpiGelu, kMaxRows>;
  auto k2 = stream_ffn_kernel<T, kEpiPlain, kMaxRows>;
  auto k1p = swi ? stream_ffn_kernel<T, kEpiSwiglu, kPairRows> : stream_ffn_kernel<T, kEpiGelu, kPairRows>;
  const int per_sm = mcap <= kPairRows ? 2 : 1;
  // per_sm CTAs per SM, and no more CTAs than stages of rows to fill
  auto grid = [&](int64_t groups_per_expert, int ctas_per_sm) {
    int64_t g = (int64_t)sm_count() * ctas_per_sm;
    const int64_t most = experts * groups_per_expert;
    if (g > most) g = most;
    return dim3((unsigned)(g > 0 ? g : 1));
  };
  const StreamProduct<T> P1{(const T*)x_perm, (const T*)W1, b1, (T*)h_perm, s.F, s.H, 0};
  const StreamProduct<T> P2{(const T*)h_perm, (const T*)W2, b2, (T*)y_perm, s.H, s.F, 0};
  if (stream_fused(s) && sched) {
    // both products in one launch; the experts' counters sched[2 .. 2+E) are zero
    const StreamFused f = stream_fused_cfg(s);
    const size_t smem = f.c.smem;
    auto kf = per_sm > 1 ? k1p : k1;
    cudaError_t e = cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    StreamProduct<T> a = P1, b = P2;
    a.rps = f.c.rps;
    b.rps = f.rps1;
    const int64_t gpe = std::max<int64_t>((s.F + a.rps - 1) / a.rps, (s.H + b.rps - 1) / b.rps);
    e = launch_kernel(kf, grid(gpe, per_sm), dim3(kThreads), smem, st, 1, a, b, 2, offs, s.E, mcap,
                      (uint32_t)smem, (int*)(sched + 2), err);
    if (e != cudaSuccess) return e;
    prof_mark(kMarkFirst, st);
    return cudaSuccess;
  }
  const StreamCfg c1 = stream_cfg(mcap, s.H, (int)sizeof(T), swi);
  const StreamCfg c2 = stream_cfg(mcap, s.F, (int)sizeof(T), false);
  if (c1.stages < 1 || c2.stages < 1) return cudaErrorNotSupported;
  cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)c1.smem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)c2.smem);
  if (e != cudaSuccess) return e;
  StreamProduct<T> a = P1, b = P2;
  a.rps = c1.rps;
  b.rps = c2.rps;
  e = launch_kernel(k1, grid((s.F + a.rps - 1) / a.rps, 1), dim3(kThreads), c1.smem, st, 1, a, a, 1, offs, s.E, mcap,
                    (uint32_t)c1.smem, (int*)nullptr, err);
  if (e != cudaSuccess) return e;
  prof_mark(kMarkFirst, st);
  return launch_kernel(k2, grid((s.H + b.rps - 1) / b.rps, 1), dim3(kThreads), c2.smem, st, 1, b, b, 1, offs, s.E,
                       mcap, (uint32_t)c2.smem, (int*)nullptr, err);
}

}  // namespace

// Decode-sized batches whose activation rows and two stages of weight rows
// fit one CTA's shared memory; the rows are whole 16-byte vectors.
bool stream_ffn_eligible(const Shape& s) {
  if (s.T > kMaxRows || (s.flags & MOE_FLAG_NO_DECODE)) return false;
  const int v = 16 / s.esize();
  if (s.H % v != 0 || s.F % v != 0) return false;
  const int mcap = (int)(s.T < kMaxRows ? s.T : kMaxRows);
  const bool swi = (s.flags & MOE_FLAG_SWIGLU) != 0;
  return stream_cfg(mcap, s.H, s.esize(), swi).stages >= 2 && stream_cfg(mcap, s.F, s.esize(), false).stages >= 2;
}

// The eligible batches run both products in one launch unless the flags ask
// for one launch each or the two products' rows do not share a ring.
bool stream_fused(const Shape& s) {
  return stream_ffn_eligible(s) && !(s.flags & MOE_FLAG_FFN_SPLIT) && stream_fused_cfg(s).ok;
}

cudaError_t launch_ffn_stream(const Shape& s, const void* x_perm, const int32_t* offs, const void* W1,
                              const float* b1, const void* W2, const float* b2, void* h_perm,
                              void* y_perm, int* err, int32_t* sched, cudaStream_t st) {
  if (s.dtype == MOE_BF16)
    return run_stream<bf16>(s, x_perm, offs, W1, b1, W2, b2, h_perm, y_perm, err, sched, st);
  return run_stream<float>(s, x_perm, offs, W1, b1, W2, b2, h_perm, y_perm, err, sched, st);
}

}  // namespace moe
