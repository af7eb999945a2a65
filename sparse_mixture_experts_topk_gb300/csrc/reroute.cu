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
// One block reproduces the walk exactly, in epochs.  In an epoch every
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

// The (r + 1)-th best expert of token t that is eligible (room left and not
// used by the token), ranked by score descending, index ascending; -1 if
// fewer than r + 1 are eligible.
__device__ __forceinline__ int choose(const float* __restrict__ scores, const int32_t* __restrict__ ids,
                                      const int32_t* __restrict__ fin, int64_t t, int E, int K, int r,
                                      const int* room) {
  // the experts the token uses: its K choices and its moves so far
  int used[16];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    used[2 * j] = j < K ? ids[t * K + j] : -1;
    used[2 * j + 1] = j < K ? fin[t * K + j] : -1;
  }
  const float* sc = scores + t * E;
  float prev_v = INFINITY;
  int prev_i = -1;
  int pick = -1;
#pragma unroll 1
  for (int round = 0; round <= r; ++round) {
    float bv = -INFINITY;
    int bi = -1;
#pragma unroll 1
    for (int e = 0; e < E; ++e) {
      bool skip = room[e] <= 0;
#pragma unroll
      for (int j = 0; j < 16; ++j) skip |= used[j] == e;
      if (skip) continue;
      const float v = sc[e];
      const bool after = v < prev_v || (v == prev_v && e > prev_i);
      const bool better = bi < 0 || v > bv || (v == bv && e < bi);
      if (after && better) {
        bv = v;
        bi = e;
      }
    }
    if (bi < 0) return -1;
    pick = bi;
    prev_v = bv;
    prev_i = bi;
  }
  return pick;
}

__global__ void __launch_bounds__(kThreads, 1)
reroute_kernel(const float* __restrict__ scores, const int32_t* __restrict__ ids, const int32_t* __restrict__ pos,
               const int32_t* __restrict__ offs, int64_t Tn, int E, int K, int C, int32_t* __restrict__ fin,
               int32_t* __restrict__ pend, int32_t* __restrict__ choice, int32_t* __restrict__ dropped,
               int32_t* __restrict__ dropped_copy) {
  __shared__ int room[256];
  __shared__ int running[256];
  __shared__ int wcnt[kWarps][256];
  __shared__ int s_scan[kThreads];
  __shared__ int s_istar;
  __shared__ int s_drop;
  pdl_enter();
  const int tid = threadIdx.x, warp = tid >> 5;
  const int64_t S = Tn * K;
  for (int e = tid; e < E; e += kThreads) room[e] = C - (offs[e + 1] - offs[e]);
  if (tid == 0) s_drop = 0;
  // the pending slots (over capacity, valid expert id), in slot order: each
  // thread counts a contiguous range, then a block scan places them
  const int64_t per = (S + kThreads - 1) / kThreads;
  const int64_t a = (int64_t)tid * per, b = min(S, a + per);
  int mine = 0;
  for (int64_t s = a; s < b; ++s) {
    const int e = ids[s];
    const bool valid = e >= 0 && e < E;
    fin[s] = valid ? e : -1;
    mine += (valid && pos[s] < 0) ? 1 : 0;
  }
  s_scan[tid] = mine;
  __syncthreads();
  for (int o = 1; o < kThreads; o <<= 1) {
    const int v = tid >= o ? s_scan[tid - o] : 0;
    __syncthreads();
    s_scan[tid] += v;
    __syncthreads();
  }
  const int n = s_scan[kThreads - 1];
  int w_at = s_scan[tid] - mine;
  for (int64_t s = a; s < b; ++s) {
    const int e = ids[s];
    if (e >= 0 && e < E && pos[s] < 0) pend[w_at++] = (int32_t)s;
  }
  __syncthreads();

  int base = 0;
  while (base < n) {
    for (int e = tid; e < E; e += kThreads) running[e] = 0;
    if (tid == 0) s_istar = n;
    __syncthreads();
    // requests in order from `base`, one chunk of kThreads at a time, until
    // an expert overflows
    for (int c0 = base; c0 < n; c0 += kThreads) {
      const int i = c0 + tid;
      const bool live = i < n;
      int c = -1;
      if (live) {
        const int s = pend[i];
        const int64_t t = s / K;
        int r = 0;
        while (i - 1 - r >= base && pend[i - 1 - r] / K == t) ++r;
        c = choose(scores, ids, fin, t, E, K, r, room);
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
                           const int32_t* offs, int32_t* fin, int32_t* pend, int32_t* choice, int32_t* dropped,
                           int32_t* dropped_copy, cudaStream_t st) {
  if (s.T == 0) {
    if (dropped) return cudaMemsetAsync(dropped, 0, sizeof(int32_t), st);
    return cudaSuccess;
  }
  return launch_kernel(reroute_kernel, dim3(1), dim3(kThreads), 0, st, 1, scores, ids, pos, offs, s.T, s.E, s.K,
                       s.C, fin, pend, choice, dropped, dropped_copy);
}

}  // namespace moe
