// drop_tokens=False: the slots an expert's capacity would drop move to their
// token's next-best expert with room (Qwen2-MoE code walkthrough, jsqmd.com,
// section 3.4: with drop_tokens False, tokens over capacity are routed to the
// next-best expert instead of being dropped).
//
// The rule, in slot order s = t K + j: the slots the capacity keeps stay; each
// other slot goes to the best-scored expert (score descending, index
// ascending) that its token does not already use -- neither among its K
// choices nor as the target of an earlier move -- and that still has room
// (capacity minus the slots it already holds); with none, the slot is
// dropped.  Taken literally this is a walk over the slots, one at a time.
//
// First, for every token with a slot over capacity, its unchosen experts are
// ranked by score (all SMs, a warp per token).  Then one block reproduces the
// walk exactly, in epochs.  In an epoch every
// pending slot computes its move against the room left at the start of the
// epoch: the token's (r + 1)-th best eligible expert, r = the token's pending
// slots before it in this epoch (they take the 1st .. r-th best).  Walking
// the pending slots in order, each expert accepts requests until its room is
// used; the first request an expert cannot take ends the epoch.  Every move
// before that one is what the one-at-a-time walk would do (the experts it
// picked still had room at its turn, and an expert only ever loses room), so
// those moves are committed; the expert that overflowed is now full, and the
// next epoch starts at the request it refused.  Every epoch but the last
// fills an expert, so there are at most E + 1 epochs.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kGroup = kThreads / kWarps;   // chunks per pass of the pending-list build (32)

// Per token with a slot over capacity: the experts it did not choose,
// ranked by score descending, index ascending (alts[t E + i], i < E - K).
// One warp per token; lane l ranks the experts l, l + 32, ... by counting
// the unchosen experts that rank above each.
constexpr int kRankWarps = 8;
__global__ void __launch_bounds__(32 * kRankWarps)
reroute_rank_kernel(const float* __restrict__ scores, const int32_t* __restrict__ ids,
                    const int32_t* __restrict__ pos, int64_t Tn, int E, int K, uint8_t* __restrict__ alts) {
  __shared__ float s_sc[kRankWarps][256];
  __shared__ int s_ch[kRankWarps][256];
  pdl_enter();
  const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
  const int64_t nw = (int64_t)gridDim.x * kRankWarps;
  for (int64_t t = (int64_t)blockIdx.x * kRankWarps + wi; t < Tn; t += nw) {
    const bool over = __any_sync(0xffffffffu, lane < K && pos[t * K + lane] < 0);
    if (!over) continue;
    for (int e = lane; e < E; e += 32) {
      s_sc[wi][e] = scores[t * E + e];
      s_ch[wi][e] = 0;
    }
    __syncwarp();
    if (lane < K) {
      const int c = ids[t * K + lane];
      if (c >= 0 && c < E) s_ch[wi][c] = 1;
    }
    __syncwarp();
    for (int e = lane; e < E; e += 32) {
      if (s_ch[wi][e]) continue;
      const float v = s_sc[wi][e];
      int rank = 0;
      for (int e2 = 0; e2 < E; ++e2) {
        const float v2 = s_sc[wi][e2];
        rank += (!s_ch[wi][e2] && (v2 > v || (v2 == v && e2 < e))) ? 1 : 0;
      }
      alts[t * E + rank] = (uint8_t)e;
    }
    __syncwarp();
  }
}

// The (r + 1)-th expert of token t's ranked alternatives that has room left
// (bit e of `full` clear) and is not the target of one of the token's earlier
// moves; -1 if there are fewer than r + 1.
__device__ __forceinline__ int choose(const uint8_t* __restrict__ alts, const int32_t* __restrict__ ids,
                                      const int32_t* __restrict__ fin, int64_t t, int E, int K, int r,
                                      const uint32_t* full) {
  // the token's moves so far (a moved slot's expert differs from its choice)
  int moved[8];
  bool any_moved = false;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int f = j < K ? fin[t * K + j] : -1;
    moved[j] = (j < K && f != ids[t * K + j]) ? f : -1;
    any_moved |= moved[j] >= 0;
  }
  const uint8_t* lst = alts + t * E;
  const int na = E - K;
  int seen = 0;
#pragma unroll 1
  for (int i0 = 0; i0 < na; i0 += 8) {
    int e8[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) e8[u] = i0 + u < na ? (int)lst[i0 + u] : -1;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = e8[u];
      if (e < 0 || ((full[e >> 5] >> (e & 31)) & 1u)) continue;
      if (any_moved) {
        bool skip = false;
#pragma unroll
        for (int j = 0; j < 8; ++j) skip |= moved[j] == e;
        if (skip) continue;
      }
      if (seen == r) return e;
      ++seen;
    }
  }
  return -1;
}

__global__ void __launch_bounds__(kThreads, 1)
reroute_kernel(const uint8_t* __restrict__ alts, const int32_t* __restrict__ ids, const int32_t* __restrict__ pos,
               const int32_t* __restrict__ offs, int64_t Tn, int E, int K, int C, int32_t* __restrict__ fin,
               int32_t* __restrict__ pend, int32_t* __restrict__ choice, int32_t* __restrict__ dropped,
               int32_t* __restrict__ dropped_copy) {
  __shared__ int room[256];
  __shared__ uint32_t s_full[8];         // bit e: expert e has no room left
  __shared__ int running[256];
  __shared__ int wcnt[kWarps][256];
  __shared__ int s_scan[kThreads];
  __shared__ int s_pend[8 + kThreads];   // the chunk's pending slots, after the (up to) 8 before it
  __shared__ int s_istar;
  __shared__ int s_drop;
  pdl_enter();
  const int tid = threadIdx.x, warp = tid >> 5;
  const int64_t S = Tn * K;
  for (int e = tid; e < E; e += kThreads) room[e] = C - (offs[e + 1] - offs[e]);
  if (tid == 0) s_drop = 0;
  // the pending slots (over capacity, valid expert id), in slot order.
  // Groups of kGroup chunks of kThreads slots: thread tid loads slot
  // chunk * kThreads + tid of each chunk (coalesced, 8 loads in flight),
  // the warps' ballots are counted per (chunk, warp), one block scan over
  // those counts places every pending slot.
  int n = 0;
  for (int64_t g0 = 0; g0 < S; g0 += (int64_t)kGroup * kThreads) {
    uint32_t mine = 0;
#pragma unroll 1
    for (int c0 = 0; c0 < kGroup; c0 += 8) {
      int e8[8], p8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t sl = g0 + (int64_t)(c0 + u) * kThreads + tid;
        e8[u] = sl < S ? ids[sl] : -1;
        p8[u] = sl < S ? pos[sl] : 0;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t sl = g0 + (int64_t)(c0 + u) * kThreads + tid;
        const bool valid = e8[u] >= 0 && e8[u] < E;
        if (sl < S) fin[sl] = valid ? e8[u] : -1;
        if (valid && p8[u] < 0) mine |= 1u << (c0 + u);
      }
    }
#pragma unroll 1
    for (int c = 0; c < kGroup; ++c) {
      const unsigned bal = __ballot_sync(0xffffffffu, (mine >> c) & 1u);
      if ((tid & 31) == 0) s_scan[c * kWarps + warp] = __popc(bal);
    }
    __syncthreads();
    // exclusive scan of the kGroup x kWarps counts, (chunk, warp) order
    const int mycnt = s_scan[tid];
    for (int o = 1; o < kThreads; o <<= 1) {
      const int v = tid >= o ? s_scan[tid - o] : 0;
      __syncthreads();
      s_scan[tid] += v;
      __syncthreads();
    }
    const int total = s_scan[kThreads - 1];
    const int excl_mine = s_scan[tid] - mycnt;
    __syncthreads();
    s_scan[tid] = excl_mine;
    __syncthreads();
#pragma unroll 1
    for (int c = 0; c < kGroup; ++c) {
      const unsigned bal = __ballot_sync(0xffffffffu, (mine >> c) & 1u);
      if ((mine >> c) & 1u)
        pend[n + s_scan[c * kWarps + warp] + __popc(bal & lanemask_lt())] =
            (int32_t)(g0 + (int64_t)c * kThreads + tid);
    }
    __syncthreads();
    n += total;
  }
  __syncthreads();

  int base = 0;
  while (base < n) {
    for (int e = tid; e < E; e += kThreads) running[e] = 0;
    if (tid < 8) {
      uint32_t m = 0;
      for (int b = 0; b < 32; ++b) {
        const int e = tid * 32 + b;
        if (e < E && room[e] <= 0) m |= 1u << b;
      }
      s_full[tid] = m;
    }
    if (tid == 0) s_istar = n;
    __syncthreads();
    // requests in order from `base`, one chunk of kThreads at a time, until
    // an expert overflows
    for (int c0 = base; c0 < n; c0 += kThreads) {
      const int i = c0 + tid;
      const bool live = i < n;
      // the chunk's pending slots (one coalesced load), and the K - 1 before
      // it that a token's first slots in the chunk may follow
      s_pend[8 + tid] = live ? pend[i] : -1;
      if (tid < 8) s_pend[tid] = (c0 - 8 + tid >= base) ? pend[c0 - 8 + tid] : -1;
      __syncthreads();
      int c = -1;
      if (live) {
        const int s = s_pend[8 + tid];
        const int64_t t = s / K;
        int r = 0;
        while (r < K - 1 && s_pend[8 + tid - 1 - r] >= 0 && s_pend[8 + tid - 1 - r] / K == t) ++r;
        c = choose(alts, ids, fin, t, E, K, r, s_full);
        choice[i] = c;
      }
      // rank of the request among this epoch's requests for its expert
      for (int x = tid; x < kWarps * 256; x += kThreads) (&wcnt[0][0])[x] = 0;
      __syncthreads();
      const int key = (live && c >= 0) ? c : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, key);
      const unsigned below = peers & lanemask_lt();
      if (key >= 0 && below == 0) wcnt[warp][key] = __popc(peers);
      __syncthreads();
      if (key >= 0) {
        int rank = running[key] + __popc(below);
        for (int w2 = 0; w2 < warp; ++w2) rank += wcnt[w2][key];
        if (rank >= room[key]) atomicMin(&s_istar, i);
      }
      __syncthreads();
      for (int e = tid; e < E; e += kThreads) {
        int add = 0;
        for (int w2 = 0; w2 < kWarps; ++w2) add += wcnt[w2][e];
        running[e] += add;
      }
      __syncthreads();
      if (s_istar < n) break;
    }
    // commit every move before the first refused request
    const int istar = s_istar;
    for (int i = base + tid; i < istar; i += kThreads) {
      const int c = choice[i];
      fin[pend[i]] = c;
      if (c >= 0) atomicSub(&room[c], 1);
      else atomicAdd(&s_drop, 1);
    }
    __syncthreads();
    base = istar;
  }
  if (tid == 0) {
    if (dropped) *dropped = s_drop;
    if (dropped_copy) *dropped_copy = s_drop;
  }
}

}  // namespace

cudaError_t launch_reroute(const Shape& s, const float* scores, const int32_t* ids, const int32_t* pos,
                           const int32_t* offs, int32_t* fin, int32_t* pend, int32_t* choice, uint8_t* alts,
                           int32_t* dropped, int32_t* dropped_copy, cudaStream_t st) {
  if (s.T == 0) {
    if (dropped) return cudaMemsetAsync(dropped, 0, sizeof(int32_t), st);
    return cudaSuccess;
  }
  int64_t grid = (s.T + kRankWarps - 1) / kRankWarps;
  if (grid > (int64_t)sm_count() * 8) grid = (int64_t)sm_count() * 8;
  cudaError_t e = launch_kernel(reroute_rank_kernel, dim3((unsigned)grid), dim3(32 * kRankWarps), 0, st, 1, scores,
                                ids, pos, s.T, s.E, s.K, alts);
  if (e != cudaSuccess) return e;
  return launch_kernel(reroute_kernel, dim3(1), dim3(kThreads), 0, st, 1, (const uint8_t*)alts, ids, pos, offs, s.T,
                       s.E, s.K, s.C, fin, pend, choice, dropped, dropped_copy);
}

}  // namespace moe
