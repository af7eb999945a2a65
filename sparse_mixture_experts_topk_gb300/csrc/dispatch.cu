// Dispatch: group the T*K routing slots by expert, stable in slot order, with
// the per-expert capacity, and gather the token rows into expert-contiguous
// order.
//
// Qwen2-MoE code walkthrough (jsqmd.com), section 3.1 item 3: tokens are
// regrouped by expert id with a scatter and an argsort; section 3.4: an
// expert takes at most expert_capacity tokens and the rest are dropped.  The
// Qwen2-MoE module article (mlqm.cn), section 2.2, gives the capacity
// ceil(total_tokens / num_experts) * num_experts_per_tok.
//
// No sort is run.  Slots are cut into blocks of consecutive slots:
//   1. hist:    per block, how many of its slots go to each expert;
//   2. scan:    per expert, exclusive prefix over blocks (rank base of each
//               block), totals, capacity cut, exclusive prefix over experts
//               (offs), dropped count; optionally the probability sums and
//               the load-balancing loss;
//   3. scatter: per block, the stable rank of each slot among the block's
//               slots of the same expert (warp match + per-warp counts), so
//               rank = block base + in-block rank; kept iff rank < capacity;
//   4. gather:  x_perm[pos[t K + j]] = x[t], one warp per token: each x row
//               is read once and written to its kept slots' rows.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kDispThreads = 256;
constexpr int kDispWarps = kDispThreads / 32;

__global__ void __launch_bounds__(kDispThreads)
dispatch_hist_kernel(const int32_t* __restrict__ ids, int64_t S, int E, int bslots,
                     int32_t* __restrict__ blk_hist, int* err) {
  __shared__ int hist[256];
  pdl_enter();
  for (int e = threadIdx.x; e < E; e += kDispThreads) hist[e] = 0;
  __syncthreads();
  const int64_t s0 = (int64_t)blockIdx.x * bslots;
  const int64_t s1 = min(S, s0 + bslots);
  for (int64_t s = s0 + threadIdx.x; s < s1; s += kDispThreads) {
    const int e = ids[s];
    if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
    else if (e != -1) set_error(err, kDevBadIndex);   // -1: the slot has no expert
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kDispThreads) blk_hist[(int64_t)blockIdx.x * E + e] = hist[e];
}

// Thread e of a 256-thread block holds run = the number of slots routed to
// expert e.  Cuts at the capacity and writes count, offs (exclusive prefix
// of the kept counts, offs[E] = kept rows) and the dropped total; with
// psum_part also the summed router probabilities and the load-balancing loss.
// Every output pointer may be null (that output is not written).
// s_offs (nullable): also receives offs[0..E] in shared memory.  p_pre >= 0
// (with psum_part set): this thread's probability sum, already added up in
// row order by the caller.
template <bool kRolled = false>
__device__ __forceinline__ void finish_counts(int run, int E, int C, int32_t* __restrict__ count,
                                              int32_t* __restrict__ offs, int32_t* __restrict__ dropped,
                                              const float* __restrict__ psum_part, int64_t prows,
                                              float* __restrict__ psum, float* __restrict__ aux, int64_t Tn,
                                              int K, int32_t* __restrict__ count_copy,
                                              int32_t* __restrict__ dropped_copy, int32_t* __restrict__ sched,
                                              int* s_offs = nullptr, float p_pre = -1.f) {
  __shared__ int sk[256];
  __shared__ int sd[256];
  __shared__ float sa[256];
  const int e = threadIdx.x;
  const int kept = (e < E) ? ((C > 0 && run > C) ? C : run) : 0;
  sk[e] = kept;
  sd[e] = (e < E) ? run - kept : 0;
  __syncthreads();
  // inclusive scan of kept (Hillis-Steele, 256 entries)
#pragma unroll(kRolled ? 1 : 8)
  for (int o = 1; o < 256; o <<= 1) {
    const int v = (e >= o) ? sk[e - o] : 0;
    const int d = (e >= o) ? sd[e - o] : 0;
    __syncthreads();
    sk[e] += v;
    sd[e] += d;
    __syncthreads();
  }
  if (e < E) {
    if (count) count[e] = run;
    if (count_copy) count_copy[e] = run;
    if (offs) {
      offs[e] = sk[e] - kept;
      if (e == E - 1) offs[E] = sk[e];
    }
    if (s_offs) {
      s_offs[e] = sk[e] - kept;
      if (e == E - 1) s_offs[E] = sk[e];
    }
  }
  if (e == 255) {
    if (dropped) *dropped = sd[255];
    if (dropped_copy) *dropped_copy = sd[255];
  }
  if (sched) {
    // the expert GEMMs that follow take tiles from sched[0..1] and count the
    // finished hidden columns of each 256-row block of the kept rows in the rest
    const int words = 2 + (sk[255] >> 8) + E + 1;
    for (int i = e; i < words; i += 256) sched[i] = 0;
  }
  if (psum_part) {
    float p = p_pre;
    if (e < E && p_pre < 0.f) {
      p = 0.f;
      // rows added in order; eight loads in flight
      int64_t r = 0;
      for (; r + 8 <= prows; r += 8) {
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = psum_part[(r + i) * E + e];
#pragma unroll
        for (int i = 0; i < 8; ++i) p += v[i];
      }
      for (; r < prows; ++r) p += psum_part[r * E + e];
    }
    if (e < E && psum) psum[e] = p;
    if (aux) {
      // E * sum_i (count_i / (T K)) * (psum_i / T), reduced in a fixed order
      sa[e] = (e < E && Tn > 0) ? ((float)run / (float)(Tn * K)) * (p / (float)Tn) : 0.f;
      __syncthreads();
#pragma unroll(kRolled ? 1 : 8)
      for (int o = 128; o > 0; o >>= 1) {
        if (e < o) sa[e] += sa[e + o];
        __syncthreads();
      }
      if (e == 0) *aux = (float)E * sa[0];
    }
  }
}

// One block; thread e owns expert e (E <= 256).  With `staged`, the
// [nblk, E] histogram is first copied to shared memory with coalesced loads
// and scanned there; with `staged_p`, the [prows, E] probability partials
// are copied in the same pass (so their loads overlap) and summed there.
__global__ void __launch_bounds__(256)
dispatch_scan_kernel(const int32_t* __restrict__ blk_hist, int64_t nblk, int E, int C, int staged,
                     int staged_p, int32_t* __restrict__ blk_base, int32_t* __restrict__ count,
                     int32_t* __restrict__ offs, int32_t* __restrict__ dropped,
                     const float* __restrict__ psum_part, int64_t prows, float* __restrict__ psum,
                     float* __restrict__ aux, int64_t Tn, int K, int32_t* __restrict__ count_copy,
                     int32_t* __restrict__ dropped_copy, int32_t* __restrict__ sched) {
  extern __shared__ int sh[];          // [nblk, E] when staged, then [prows, E] floats when staged_p
  pdl_enter();
  const int e = threadIdx.x;
  const int64_t n = nblk * E;
  const int64_t np = staged_p ? prows * E : 0;
  float* sp = reinterpret_cast<float*>(sh + (staged ? n : 0));
  if (staged || staged_p) {
    // eight loads of each kind in flight per thread before any store
    const int64_t nh = staged ? n : 0;
    const int64_t m = nh > np ? nh : np;
    for (int64_t i0 = threadIdx.x; i0 < m; i0 += 256 * 8) {
      int h[8];
      float q[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t i = i0 + 256 * u;
        h[u] = i < nh ? blk_hist[i] : 0;
        q[u] = i < np ? psum_part[i] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t i = i0 + 256 * u;
        if (i < nh) sh[i] = h[u];
        if (i < np) sp[i] = q[u];
      }
    }
    __syncthreads();
  }
  // probability sums: G = 256 / E thread groups each add every G-th row (in
  // row order), then thread e adds the G group sums in group order
  __shared__ float s_pg[256];
  float p_pre = -1.f;
  if (staged_p) {
    const int G = 256 / E;
    const int g = threadIdx.x / E, ee = threadIdx.x % E;
    if (g < G) {
      float a = 0.f;
      for (int64_t r = g; r < prows; r += G) a += sp[r * E + ee];
      s_pg[g * E + ee] = a;
    }
    __syncthreads();
    if (e < E) {
      p_pre = 0.f;
      for (int gg = 0; gg < G; ++gg) p_pre += s_pg[gg * E + e];
    }
  }
  int run = 0;
  if (staged) {
    if (e < E) {
      for (int64_t b = 0; b < nblk; ++b) {
        const int h = sh[b * E + e];
        sh[b * E + e] = run;
        run += h;
      }
    }
    __syncthreads();
    for (int64_t i = threadIdx.x; i < n; i += 256) blk_base[i] = sh[i];
  } else if (e < E) {
    int64_t b = 0;
    // batches of independent loads, then the dependent running sum
    for (; b + 8 <= nblk; b += 8) {
      int h[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) h[i] = blk_hist[(b + i) * E + e];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        blk_base[(b + i) * E + e] = run;
        run += h[i];
      }
    }
    for (; b < nblk; ++b) {
      const int h = blk_hist[b * E + e];
      blk_base[b * E + e] = run;
      run += h;
    }
  }
  finish_counts(run, E, C, count, offs, dropped, psum_part, prows, psum, aux, Tn, K, count_copy,
                dropped_copy, sched, nullptr, p_pre);
}

// One 256-slot chunk of the stable placement: this thread holds slot s
// (valid or not) routed to expert e (-1: none or out of range).
// running[e] (shared) is the rank the chunk's first slot of expert e takes
// and is advanced past the chunk; ranks within the chunk come from a warp
// match plus per-warp counts.  s_src (nullable) gets a shared copy of src.
template <bool kRolled = false>
__device__ __forceinline__ void scatter_chunk(int e, int64_t s, bool valid, int E, int C, int (*wcnt)[256],
                                              int* running, const int32_t* offs, int32_t* __restrict__ pos,
                                              int32_t* __restrict__ src, int* s_src) {
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int i = tid; i < kDispWarps * 256; i += kDispThreads) (&wcnt[0][0])[i] = 0;
  __syncthreads();
  const unsigned peers = __match_any_sync(0xffffffffu, e);
  const unsigned below = peers & lanemask_lt();
  if (e >= 0 && below == 0) wcnt[warp][e] = __popc(peers);
  __syncthreads();
  if (valid) {
    int p = -1;
    if (e >= 0) {
      int r = running[e] + __popc(below);
#pragma unroll(kRolled ? 1 : 4)
      for (int w2 = 0; w2 < warp; ++w2) r += wcnt[w2][e];
      if (C <= 0 || r < C) {
        p = offs[e] + r;
        src[p] = (int32_t)s;
        if (s_src) s_src[p] = (int)s;
      }
    }
    pos[s] = p;
  }
  __syncthreads();
  for (int e2 = tid; e2 < E; e2 += kDispThreads) {
    int add = 0;
#pragma unroll(kRolled ? 1 : kDispWarps)
    for (int w2 = 0; w2 < kDispWarps; ++w2) add += wcnt[w2][e2];
    running[e2] += add;
  }
  __syncthreads();
}

// Stable placement of slots [s0, s1), their expert ids read from ids.
__device__ __forceinline__ void scatter_slots(const int32_t* __restrict__ ids, int64_t s0, int64_t s1, int E,
                                              int C, int* running, const int32_t* offs,
                                              int32_t* __restrict__ pos, int32_t* __restrict__ src) {
  __shared__ int wcnt[kDispWarps][256];
  for (int64_t c0 = s0; c0 < s1; c0 += kDispThreads) {
    const int64_t s = c0 + threadIdx.x;
    int e = -1;
    if (s < s1) {
      e = ids[s];
      if (e < 0 || e >= E) e = -1;   // reported by the histogram pass
    }
    scatter_chunk(e, s, s < s1, E, C, wcnt, running, offs, pos, src, nullptr);
  }
}

__global__ void __launch_bounds__(kDispThreads)
dispatch_scatter_kernel(const int32_t* __restrict__ ids, int64_t S, int E, int C, int bslots,
                        const int32_t* __restrict__ blk_base, const int32_t* __restrict__ offs,
                        int32_t* __restrict__ pos, int32_t* __restrict__ src) {
  __shared__ int running[256];
  pdl_enter();
  const int64_t s0 = (int64_t)blockIdx.x * bslots;
  const int64_t s1 = min(S, s0 + bslots);
  for (int e = threadIdx.x; e < E; e += kDispThreads) running[e] = blk_base[(int64_t)blockIdx.x * E + e];
  scatter_slots(ids, s0, s1, E, C, running, offs, pos, src);
}

// x_perm[pos[t K + j]] = x[t] for every kept slot j of token t: each x row
// is read once and written to its (at most K) rows, one warp per token, 4
// vectors a lane in flight.  (Every kept row of x_perm is the image of
// exactly one slot, so each is written once.)  x_perm is stored evict-first:
// the first expert product streams it from DRAM either way.  KP: K rounded
// up to 2, 4 or 8.
template <int KP>
__global__ void __launch_bounds__(256)
dispatch_gather_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ pos, int64_t Tn, int K,
                       int vec_per_row, uint4* __restrict__ x_perm) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t t = warp0; t < Tn; t += nwarps) {
    int64_t dst[KP];
#pragma unroll
    for (int j = 0; j < KP; ++j) {
      const int p = j < K ? pos[t * K + j] : -1;
      dst[j] = p >= 0 ? (int64_t)p * vec_per_row : -1;
    }
    const uint4* a = x + t * vec_per_row;
    int v = lane;
    for (; v + 96 < vec_per_row; v += 128) {
      const uint4 u0 = a[v], u1 = a[v + 32], u2 = a[v + 64], u3 = a[v + 96];
#pragma unroll
      for (int j = 0; j < KP; ++j) {
        if (dst[j] >= 0) {
          uint4* b = x_perm + dst[j];
          __stcs(b + v, u0); __stcs(b + v + 32, u1); __stcs(b + v + 64, u2); __stcs(b + v + 96, u3);
        }
      }
    }
    for (; v < vec_per_row; v += 32) {
      const uint4 u = a[v];
#pragma unroll
      for (int j = 0; j < KP; ++j)
        if (dst[j] >= 0) __stcs(x_perm + dst[j] + v, u);
    }
  }
}

// Scan and scatter in one kernel, when the router has counted its 128-token
// tiles: every block reads the whole [nblk, E] table of tile counts (eight
// loads in flight per thread), takes its rank base (the counts of the tiles
// before it) and the experts' totals and offsets, and places its tile's
// slots.  One more block, the last, places nothing: it writes the counts,
// offsets, dropped slots, probability sums (added up exactly as the scan
// kernel does) and the loss, beside the others instead of after one of
// them (measured: block 0 doing it as well took twice as long as the rest).
__global__ void __launch_bounds__(kDispThreads)
dispatch_scan_scatter_kernel(const int32_t* __restrict__ ids, int64_t S, int E, int C, int bslots,
                             const int32_t* __restrict__ blk_hist, int64_t nblk, int32_t* __restrict__ count,
                             int32_t* __restrict__ offs, int32_t* __restrict__ dropped,
                             const float* __restrict__ psum_part, int64_t prows, float* __restrict__ psum,
                             float* __restrict__ aux, int64_t Tn, int K, int32_t* __restrict__ count_copy,
                             int32_t* __restrict__ dropped_copy, int32_t* __restrict__ sched,
                             int32_t* __restrict__ pos, int32_t* __restrict__ src) {
  extern __shared__ int sh[];          // [nblk, E] tile counts
  __shared__ int running[256];
  __shared__ int s_offs[257];
  __shared__ int wcnt[kDispWarps][256];
  __shared__ float s_pg[256];
  pdl_enter();
  const int e = threadIdx.x;
  const bool leader = blockIdx.x == nblk;   // the statistics block
  const int64_t n = nblk * E;
  for (int64_t i0 = threadIdx.x; i0 < n; i0 += 256 * 8) {
    int h[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) h[u] = i0 + 256 * u < n ? blk_hist[i0 + 256 * u] : 0;
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (i0 + 256 * u < n) sh[i0 + 256 * u] = h[u];
  }
  float p_pre = -1.f;
  if (leader && psum_part) {
    // G = 256 / E thread groups each add every G-th row in row order, then
    // thread e adds the G group sums in group order
    const int G = 256 / E;
    const int g = threadIdx.x / E, ee = threadIdx.x % E;
    if (g < G) {
      float a = 0.f;
      for (int64_t r = g; r < prows; r += G) a += psum_part[r * E + ee];
      s_pg[g * E + ee] = a;
    }
    __syncthreads();
    if (e < E) {
      p_pre = 0.f;
      for (int gg = 0; gg < G; ++gg) p_pre += s_pg[gg * E + e];
    }
  }
  __syncthreads();
  int base = 0, total = 0;
  if (e < E) {
    for (int64_t b = 0; b < nblk; ++b) {
      const int h = sh[b * E + e];
      if (b < (int64_t)blockIdx.x) base += h;
      total += h;
    }
  }
  running[e] = base;
  finish_counts(total, E, C, leader ? count : nullptr, leader ? offs : nullptr, leader ? dropped : nullptr,
                leader ? psum_part : nullptr, prows, leader ? psum : nullptr, leader ? aux : nullptr, Tn, K,
                leader ? count_copy : nullptr, leader ? dropped_copy : nullptr, leader ? sched : nullptr, s_offs,
                p_pre);
  if (leader) return;   // it owns no slots
  __syncthreads();
  const int64_t s0 = (int64_t)blockIdx.x * bslots;
  const int64_t s1 = min(S, s0 + bslots);
  for (int64_t c0 = s0; c0 < s1; c0 += kDispThreads) {
    const int64_t sl = c0 + threadIdx.x;
    int ex = -1;
    if (sl < s1) {
      ex = ids[sl];
      if (ex < 0 || ex >= E) ex = -1;   // the router writes only ids in range (NaN scores: none taken)
    }
    scatter_chunk(ex, sl, sl < s1, E, C, wcnt, running, s_offs, pos, src, nullptr);
  }
}

// A small batch in one block: histogram, counts, stable placement and the
// row gather, with the same arithmetic and results as the four-kernel path.
// Each thread reads its (at most 4) slots' expert ids and its expert's
// probability partials once, up front; offsets and src stay in shared
// memory, so the only dependent global reads are those and the x rows.
constexpr int kSmallChunks = 4;
constexpr int kSmallSlots = kSmallChunks * kDispThreads;

__global__ void __launch_bounds__(kDispThreads)
dispatch_small_kernel(const int32_t* __restrict__ ids, int64_t S, int E, int C, int32_t* __restrict__ count,
                      int32_t* __restrict__ offs, int32_t* __restrict__ dropped,
                      const float* __restrict__ psum_part, int64_t prows, float* __restrict__ psum,
                      float* __restrict__ aux, int64_t Tn, int K, int32_t* __restrict__ count_copy,
                      int32_t* __restrict__ dropped_copy, int32_t* __restrict__ pos, int32_t* __restrict__ src,
                      const uint4* __restrict__ x, int vec_per_row, uint4* __restrict__ x_perm, int* err,
                      int32_t* __restrict__ sched) {
  __shared__ int hist[256];
  __shared__ int s_offs[257];
  __shared__ int s_src[kSmallSlots];
  __shared__ int wcnt[kDispWarps][256];
  pdl_enter();
  const int e = threadIdx.x;
  hist[e] = 0;
  int my[kSmallChunks];
#pragma unroll
  for (int c = 0; c < kSmallChunks; ++c) {
    const int64_t s = (int64_t)c * kDispThreads + threadIdx.x;
    my[c] = s < S ? ids[s] : -1;
  }
  float p = -1.f;
  if (psum_part && e < E) {
    p = 0.f;
    for (int64_t r = 0; r < prows; ++r) p += psum_part[r * E + e];
  }
  __syncthreads();
#pragma unroll
  for (int c = 0; c < kSmallChunks; ++c) {
    const int64_t s = (int64_t)c * kDispThreads + threadIdx.x;
    if (s < S) {
      if (my[c] >= 0 && my[c] < E) atomicAdd(&hist[my[c]], 1);
      else if (my[c] != -1) set_error(err, kDevBadIndex);   // -1: the slot has no expert
    }
    if (my[c] < 0 || my[c] >= E) my[c] = -1;
  }
  __syncthreads();
  const int run = (e < E) ? hist[e] : 0;
  finish_counts<true>(run, E, C, count, offs, dropped, psum_part, prows, psum, aux, Tn, K, count_copy,
                      dropped_copy, sched, s_offs, p);
  hist[e] = 0;       // reused as the running rank
  __syncthreads();
#pragma unroll
  for (int c = 0; c < kSmallChunks; ++c) {
    const int64_t s0 = (int64_t)c * kDispThreads;
    if (s0 < S) scatter_chunk<true>(my[c], s0 + threadIdx.x, s0 + threadIdx.x < S, E, C, wcnt, hist, s_offs, pos, src,
                              s_src);
  }
  if (x) {
    const int rows = s_offs[E];
    const int lane = threadIdx.x & 31;
    for (int r = threadIdx.x >> 5; r < rows; r += kDispWarps) {
      const uint4* a = x + (int64_t)(s_src[r] / K) * vec_per_row;
      uint4* b = x_perm + (int64_t)r * vec_per_row;
      int v = lane;
      for (; v + 96 < vec_per_row; v += 128) {
        const uint4 u0 = a[v], u1 = a[v + 32], u2 = a[v + 64], u3 = a[v + 96];
        b[v] = u0; b[v + 32] = u1; b[v + 64] = u2; b[v + 96] = u3;
      }
      for (; v < vec_per_row; v += 32) b[v] = a[v];
    }
  }
}

}  // namespace

int dispatch_block_slots(const Shape& s) {
  // at most 64 blocks so the per-expert scan over blocks stays short
  int64_t b = (s.S() + 63) / 64;
  if (b < 2048) b = 2048;
  b = (b + kDispThreads - 1) / kDispThreads * kDispThreads;
  return (int)b;
}

int64_t dispatch_blocks(const Shape& s) {
  const int64_t b = dispatch_block_slots(s);
  return (s.S() + b - 1) / b;
}

namespace {
// the fused scan + scatter keeps the whole table of tile counts in shared memory
constexpr size_t kFusedScanTable = 96 * 1024;

cudaError_t launch_gather(const Shape& s, const void* x, const int32_t* pos, void* x_perm, cudaStream_t st) {
  const int vec = (int)((int64_t)s.H * s.esize() / 16);
  auto kern = s.K <= 2 ? dispatch_gather_kernel<2> : s.K <= 4 ? dispatch_gather_kernel<4> : dispatch_gather_kernel<8>;
  int64_t grid = (s.T + 7) / 8;                      // 8 warps (tokens) a block
  if (grid > (int64_t)sm_count() * 8) grid = (int64_t)sm_count() * 8;
  return launch_kernel(kern, dim3((unsigned)grid), dim3(256), 0, st, 1, (const uint4*)x, pos, s.T, s.K, vec,
                       (uint4*)x_perm);
}
}  // namespace

int dispatch_launches(const Shape& s, bool hist_ready) {
  if (dispatch_small(s)) return 1;
  const int64_t nblk = hist_ready ? (s.T + kRouterTileTokens - 1) / kRouterTileTokens : dispatch_blocks(s);
  if (hist_ready && (size_t)nblk * s.E * sizeof(int) <= kFusedScanTable) return 2;   // scan+scatter, gather
  return (hist_ready ? 0 : 1) + 3;                                                   // (hist,) scan, scatter, gather
}

bool dispatch_small(const Shape& s) {
  // one block wins while its serial passes stay a few microseconds: up to
  // four 256-slot chunks and 256 KB of rows for its eight warps to copy
  return s.S() <= kSmallSlots && s.S() * s.H * s.esize() <= 256 * 1024;
}

cudaError_t launch_dispatch(const Shape& s, const int32_t* ids, const void* x, void* x_perm,
                            const DispatchOut& o, int* err, cudaStream_t st) {
  const int64_t S = s.S();
  if (dispatch_small(s)) {
    const int vec = (int)((int64_t)s.H * s.esize() / 16);
    const cudaError_t e =
        launch_kernel(dispatch_small_kernel, dim3(1), dim3(kDispThreads), 0, st, 1, ids, S, s.E, s.C, o.count,
                      o.offs, o.dropped, (const float*)o.psum_part,
                      o.psum_part ? router_partial_rows(s) : (int64_t)0, o.psum, o.aux, s.T, s.K, o.count_copy,
                      o.dropped_copy, o.pos, o.src, (const uint4*)(x && x_perm ? x : nullptr), vec,
                      (uint4*)x_perm, err, o.sched);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  // blocks of slots: the router's 128-token tiles when it already counted
  // them, else blocks sized for a short scan
  const int bslots = o.hist_ready ? kRouterTileTokens * s.K : dispatch_block_slots(s);
  const int64_t nblk = o.hist_ready ? (s.T + kRouterTileTokens - 1) / kRouterTileTokens
                                    : dispatch_blocks(s);
  cudaError_t e = cudaSuccess;
  const size_t table = (size_t)nblk * s.E * sizeof(int);
  if (o.hist_ready && nblk > 0 && table <= kFusedScanTable) {
    // the opt-in covers dynamic plus static shared memory above 48 KB
    e = cudaFuncSetAttribute(dispatch_scan_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)table);
    const int64_t prows = o.psum_part ? router_partial_rows(s) : (int64_t)0;
    if (e == cudaSuccess)
      e = launch_kernel(dispatch_scan_scatter_kernel, dim3((unsigned)nblk + 1), dim3(kDispThreads), table, st, 1,
                        ids, S, s.E, s.C, bslots, (const int32_t*)o.blk_hist, nblk, o.count, o.offs, o.dropped,
                        o.psum_part, prows, o.psum, o.aux, s.T, s.K, o.count_copy, o.dropped_copy, o.sched,
                        o.pos, o.src);
    if (e == cudaSuccess && x && x_perm && S > 0) e = launch_gather(s, x, o.pos, x_perm, st);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  if (nblk > 0 && !o.hist_ready)
    e = launch_kernel(dispatch_hist_kernel, dim3((unsigned)nblk), dim3(kDispThreads), 0, st, 1, ids, S, s.E,
                      bslots, o.blk_hist, err);
  const size_t sm = (size_t)nblk * s.E * sizeof(int);
  const int64_t prows = o.psum_part ? router_partial_rows(s) : (int64_t)0;
  const size_t smp = (size_t)prows * s.E * sizeof(float);
  const int staged = sm <= 96 * 1024 ? 1 : 0;
  const int staged_p = (o.psum_part && (staged ? sm : 0) + smp <= 192 * 1024) ? 1 : 0;
  const size_t smem = (staged ? sm : 0) + (staged_p ? smp : 0);
  if (e == cudaSuccess && smem > 0)
    e = cudaFuncSetAttribute(dispatch_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess)
    e = launch_kernel(dispatch_scan_kernel, dim3(1), dim3(256), smem, st, 1, (const int32_t*)o.blk_hist, nblk,
                      s.E, s.C, staged, staged_p, o.blk_base, o.count, o.offs, o.dropped, o.psum_part, prows,
                      o.psum, o.aux, s.T, s.K, o.count_copy, o.dropped_copy, o.sched);
  if (e == cudaSuccess && nblk > 0)
    e = launch_kernel(dispatch_scatter_kernel, dim3((unsigned)nblk), dim3(kDispThreads), 0, st, 1, ids, S, s.E,
                      s.C, bslots, (const int32_t*)o.blk_base, (const int32_t*)o.offs, o.pos, o.src);
  if (e == cudaSuccess && x && x_perm && S > 0) e = launch_gather(s, x, o.pos, x_perm, st);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace moe
