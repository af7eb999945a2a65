// Expert FFN for decode-sized batches (at most 16 tokens): weight streaming.
//
// Same products as the grouped GEMMs (Qwen2-MoE module article, mlqm.cn,
// section 2.2: each expert is Linear -> GELU -> Linear), for segments of at
// most 16 rows.  The time is reading every used expert's weights once, so
// the kernel is built around bytes in flight rather than arithmetic:
//   * one CTA per SM; CTA b serves the (b mod A)-th of the A experts that
//     have rows (found from offs with a warp ballot), and the CTAs of one
//     expert split its output columns into contiguous ranges;
//   * a producer thread moves the expert's activation rows and then, stage
//     after stage, `rps` consecutive weight rows (one untiled bulk copy per
//     stage; SwiGLU: a second copy for the matching up rows) into a ring of
//     2-4 stages in shared memory: 100-200 KB in flight per SM;
//   * consumer warp w dots weight row w of each stage with every activation
//     row (fp32 sums over 16-byte vectors, a shuffle reduction per row), adds
//     the bias, applies the activation and stores one output value per row.
// Every mbarrier wait is bounded; on expiry the kernel records a timeout in
// the error word, lets the other warps leave, waits (bounded) for the copies
// it issued and returns.
#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {

namespace {

constexpr int kMaxRows = 16;
constexpr int kConsumers = 8;                    // consumer warps; a stage holds <= 8 rows
constexpr int kThreads = (kConsumers + 1) * 32;  // + one producer warp
constexpr int kMaxStages = 4;
constexpr size_t kSmemBudget = 220 * 1024;
constexpr uint64_t kWaitNs = 2000000000ull;

__host__ __device__ inline size_t act_bytes(int mcap, int K, int esize) { return ((size_t)mcap * K * esize + 127) / 128 * 128; }

// One weight row (SwiGLU: gate row w and up row u) against the m <= MR
// staged activation rows: lane l takes vectors l, l + 32, ...; fp32 sums,
// reduced across the warp; lane 0 adds the bias, applies the activation and
// writes out[r * N] for r < m.
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
    float b[V], bu[V];
    Vec<T>::unpack(w[v], b);
    if (kSwi) Vec<T>::unpack(u[v], bu);
#pragma unroll
    for (int r = 0; r < MR; ++r) {
      if (r < m) {
        float x[V];
        Vec<T>::unpack(act[r * kv + v], x);
#pragma unroll
        for (int i = 0; i < V; ++i) {
          acc[r] = fmaf(x[i], b[i], acc[r]);
          if (kSwi) accu[r] = fmaf(x[i], bu[i], accu[r]);
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

template <typename T, int kEpi>
__global__ void __launch_bounds__(kThreads, 1)
stream_ffn_kernel(const T* __restrict__ A, const int32_t* __restrict__ offs, int E, int mcap,
                  const T* __restrict__ B, const float* __restrict__ bias, int N, int K, int rps, int stages,
                  T* __restrict__ C, int* err) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_e, s_na, s_abort;
  __shared__ __align__(8) uint64_t s_bar[2 * kMaxStages + 1];
  constexpr bool kSwi = kEpi == kEpiSwiglu;
  constexpr int V = Vec<T>::N;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t row_bytes = (uint32_t)K * sizeof(T);
  const uint32_t stage_bytes = (uint32_t)rps * row_bytes * (kSwi ? 2u : 1u);
  const uint32_t s_act = tc::smem_u32(smem);
  const uint32_t s_ring = s_act + (uint32_t)act_bytes(mcap, K, sizeof(T));
  auto full = [&](int s) { return tc::smem_u32(&s_bar[s]); };
  auto empty = [&](int s) { return tc::smem_u32(&s_bar[kMaxStages + s]); };
  const uint32_t act_bar = tc::smem_u32(&s_bar[2 * kMaxStages]);

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      tc::mbar_init(full(s), 1);
      tc::mbar_init(empty(s), kConsumers);
    }
    tc::mbar_init(act_bar, 1);
    s_abort = 0;
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
  // this CTA's contiguous range of output columns of expert e
  const int a = (int)(blockIdx.x % (unsigned)na);
  const int nblk = ((int)gridDim.x - 1 - a) / na + 1;
  const int per = (N + nblk - 1) / nblk;
  const int n_begin = (int)(blockIdx.x / (unsigned)na) * per;
  const int n_end = min(N, n_begin + per);
  const int groups = n_begin < n_end ? (n_end - n_begin + rps - 1) / rps : 0;
  const T* Be = B + (int64_t)e * N * K * (kSwi ? 2 : 1);

  uint32_t filled = 0, fill_par = 0;   // producer: per stage, ever filled / parity of its last fill
  bool producer = false;
  if (warp == kConsumers) {
    // ------------------------------------------------------------ producer
    if (tc::elect_one()) {
      producer = true;
      tc::mbar_arrive_expect_tx(act_bar, (uint32_t)m * row_bytes);
      tc::bulk_load(s_act, A + (int64_t)r0 * K, (uint32_t)m * row_bytes, act_bar);
      bool ok = true;
      for (int g = 0; g < groups; ++g) {
        const int s = g % stages;
        const uint32_t ph = (uint32_t)(g / stages) & 1u;
        if (!tc::mbar_wait(empty(s), ph ^ 1u, &s_abort, kWaitNs)) { ok = false; break; }
        const int n0 = n_begin + g * rps;
        const uint32_t bytes = (uint32_t)min(rps, n_end - n0) * row_bytes;
        tc::mbar_arrive_expect_tx(full(s), kSwi ? 2 * bytes : bytes);
        const uint32_t dst = s_ring + (uint32_t)s * stage_bytes;
        tc::bulk_load(dst, Be + (int64_t)n0 * K, bytes, full(s));
        if (kSwi) tc::bulk_load(dst + (uint32_t)rps * row_bytes, Be + (int64_t)(N + n0) * K, bytes, full(s));
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
    const int kv = K / V;
    const uint4* act = reinterpret_cast<const uint4*>(smem);
    bool ok = tc::mbar_wait(act_bar, 0, &s_abort, kWaitNs);
    for (int g = 0; g < groups && ok; ++g) {
      const int s = g % stages;
      const uint32_t ph = (uint32_t)(g / stages) & 1u;
      if (!tc::mbar_wait(full(s), ph, &s_abort, kWaitNs)) { ok = false; break; }
      const int n = n_begin + g * rps + warp;
      if (warp < rps && n < n_end) {
        const uint8_t* st = smem + (s_ring - s_act) + (size_t)s * stage_bytes;
        const uint4* wv = reinterpret_cast<const uint4*>(st + (size_t)warp * row_bytes);
        const uint4* uv = reinterpret_cast<const uint4*>(st + (size_t)(rps + warp) * row_bytes);
        const float* be = bias ? bias + (int64_t)e * N * (kSwi ? 2 : 1) : nullptr;
        T* out = C + (int64_t)r0 * N + n;
        // a body sized for the segment, so the hot loop stays small
        if (m <= 1) dot_rows<T, kEpi, 1>(wv, uv, act, kv, m, be, n, N, out);
        else if (m <= 2) dot_rows<T, kEpi, 2>(wv, uv, act, kv, m, be, n, N, out);
        else if (m <= 4) dot_rows<T, kEpi, 4>(wv, uv, act, kv, m, be, n, N, out);
        else if (m <= 8) dot_rows<T, kEpi, 8>(wv, uv, act, kv, m, be, n, N, out);
        else dot_rows<T, kEpi, kMaxRows>(wv, uv, act, kv, m, be, n, N, out);
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(empty(s));   // this warp is done with the stage
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
    for (int s = 0; s < stages; ++s)
      if ((filled >> s) & 1u) tc::mbar_wait(full(s), (fill_par >> s) & 1u, nullptr, kWaitNs);
  }
}

// Rows per stage and ring depth for one product: the most rows per stage
// that still leave room for two stages beside the activation rows.
struct StreamCfg {
  int rps, stages;
  size_t smem;
};

StreamCfg stream_cfg(int mcap, int K, int esize, bool swi) {
  StreamCfg c{1, 0, 0};
  const size_t act = act_bytes(mcap, K, esize);
  const size_t row = (size_t)K * esize * (swi ? 2 : 1);
  for (int rps = kConsumers; rps >= 1; rps /= 2) {
    const size_t room = kSmemBudget > act ? kSmemBudget - act : 0;
    size_t st = room / ((size_t)rps * row);
    if (st > (size_t)kMaxStages) st = kMaxStages;
    if (st >= 2 || rps == 1) {
      c.rps = rps;
      c.stages = (int)st;
      break;
    }
  }
  c.smem = act + (size_t)c.stages * c.rps * row;
  return c;
}

template <typename T>
cudaError_t run_stream(const Shape& s, const void* x_perm, const int32_t* offs, const void* W1,
                       const float* b1, const void* W2, const float* b2, void* h_perm, void* y_perm,
                       int* err, cudaStream_t st) {
  const bool swi = (s.flags & MOE_FLAG_SWIGLU) != 0;
  const int64_t experts = s.S() < s.E ? s.S() : s.E;   // at most T*K experts have rows
  const int mcap = (int)(s.T < kMaxRows ? s.T : kMaxRows);
  auto k1 = swi ? stream_ffn_kernel<T, kEpiSwiglu> : stream_ffn_kernel<T, kEpiGelu>;
  auto k2 = stream_ffn_kernel<T, kEpiPlain>;
  const StreamCfg c1 = stream_cfg(mcap, s.H, (int)sizeof(T), swi);
  const StreamCfg c2 = stream_cfg(mcap, s.F, (int)sizeof(T), false);
  if (c1.stages < 1 || c2.stages < 1) return cudaErrorNotSupported;
  cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)c1.smem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)c2.smem);
  if (e != cudaSuccess) return e;
  // one CTA per SM, and no more CTAs than stages of rows to fill
  auto grid = [&](int N, int rps) {
    int64_t g = sm_count();
    const int64_t most = experts * ((N + rps - 1) / rps);
    if (g > most) g = most;
    return dim3((unsigned)(g > 0 ? g : 1));
  };
  e = launch_kernel(k1, grid(s.F, c1.rps), dim3(kThreads), c1.smem, st, 1, (const T*)x_perm, offs, s.E, mcap,
                    (const T*)W1, b1, s.F, s.H, c1.rps, c1.stages, (T*)h_perm, err);
  if (e != cudaSuccess) return e;
  prof_mark(kMarkFirst, st);
  return launch_kernel(k2, grid(s.H, c2.rps), dim3(kThreads), c2.smem, st, 1, (const T*)h_perm, offs, s.E, mcap,
                       (const T*)W2, b2, s.H, s.F, c2.rps, c2.stages, (T*)y_perm, err);
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

cudaError_t launch_ffn_stream(const Shape& s, const void* x_perm, const int32_t* offs, const void* W1,
                              const float* b1, const void* W2, const float* b2, void* h_perm,
                              void* y_perm, int* err, cudaStream_t st) {
  if (s.dtype == MOE_BF16)
    return run_stream<bf16>(s, x_perm, offs, W1, b1, W2, b2, h_perm, y_perm, err, st);
  return run_stream<float>(s, x_perm, offs, W1, b1, W2, b2, h_perm, y_perm, err, st);
}

}  // namespace moe
