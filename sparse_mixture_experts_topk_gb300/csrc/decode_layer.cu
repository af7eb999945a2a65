// The whole layer for decode-sized bf16 batches (at most 16 tokens) in one
// launch: gate scores, top-k routing, the placement of the slots by expert,
// both expert products and the weighted combine.
//
// The layer is the one the other kernels compute step by step (Qwen2-MoE
// code walkthrough, jsqmd.com, section 3.1: gate linear, softmax, top-k,
// renormalised weights, expert FFNs, weighted sum; Qwen2-MoE module article,
// mlqm.cn, section 2.2: capacity), and every value is computed with the same
// operations in the same order as there, so the outputs are the same bits.
// At these sizes the time is reading the used experts' weights once plus
// the latency of the steps between, so the steps run inside one grid that
// holds every CTA at once (one or two per SM):
//   1. gate scores: (gate row, piece, group of up to four tokens) units, with
//      the pieces of the decode router, spread over the grid's consumer
//      warps; each unit's partial scores go to a global table and raise a
//      counter;
//   2. every CTA waits for the counter, sums the pieces and finishes every
//      token itself (top-k, weights, probabilities) in shared memory, then
//      places the slots: per expert in slot order, the first C kept;
//   3. the used experts' weight rows, first product then second, in expert
//      order: CTA b takes the b-th share of each product's rows, the shares
//      cut at equal sums of a per-row cost that grows with the expert's
//      token rows (the dots of experts with many rows are compute-bound), a
//      share possibly spanning several experts, and streams it in ring
//      stages of at most rps rows of one expert.  A producer warp moves the
//      stages through a ring of bulk copies; an activation warp moves each
//      expert's rows (x rows for the first product, h rows for the second,
//      the latter once all F columns of the expert's first product are
//      counted) into one of two buffers; eight consumer warps dot them, two
//      weight rows a warp for experts of one to four rows;
//   4. once every CTA has counted itself done with the second product, the
//      CTAs that own output items combine them.
// Counter waits need every CTA resident: the grid is one or two CTAs per SM
// and the host checks that many fit.  Every wait is bounded; on expiry the
// kernel records a timeout in the error word, skips the remaining work,
// waits (bounded) for the copies it issued and returns.  The counters are
// zeroed by a one-block kernel launched just before.
#include <algorithm>

#include "combine.cuh"
#include "common.cuh"
#include "internal.h"
#include "router_body.cuh"
#include "stream_body.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

using stream::kConsumers;
using stream::kWaitNs;
using stream::stage_pair;
using stream::stage_row;
using stream::stage_row_of_warp;
using stream::wait_count;

constexpr int kMaxTok = 16;
constexpr int kMaxSlots = kMaxTok * 8;
constexpr int kProducer = kConsumers;        // warp 8: weight ring
constexpr int kActWarp = kConsumers + 1;     // warp 9: activation rows
constexpr int kThreads = (kConsumers + 2) * 32;
constexpr int kMaxStages = 6;
// dynamic shared memory per CTA: one CTA per SM, or two (each with 1 KB
// reserved and its static arrays beside the dynamic part)
constexpr uint32_t kDynSingle = 220 * 1024;
constexpr uint32_t kDynPair = 104 * 1024;
// counters: [0] gate-score units done, [1] CTAs done with the second
// product, [2 + e] first-product units of expert e done
constexpr int kCtrFixed = 2;

struct DecodeArgs {
  const bf16* x;
  const bf16* Wg;
  const float* gate_bias;
  const bf16* W1;
  const float* b1;
  const bf16* W2;
  const float* b2;
  bf16* out;
  int T, H, E, K, F, C;
  float inv_tau;
  float* part;           // [pieces][T][E] partial gate scores
  int* ctr;              // [kCtrFixed + E], zero at launch
  bf16* h;               // [kept rows][F]
  bf16* y;               // [kept rows][H]
  int32_t* count;
  int32_t* count_copy;
  int32_t* dropped;
  int32_t* dropped_copy;
  float* psum;
  float* aux;
  int* err;
  uint32_t dyn_bytes;
};

// The streaming plan for a largest expert of mmax rows: nab activation
// buffers of `slot` bytes, then a ring of `stages` stages of rps0 weight
// rows of the first product (rps1 of the second in the same bytes).  Prefers
// two buffers and the most rows per stage that leave three stages, then two.
struct DecodePlan {
  int nab, rps0, rps1, stages;
  uint32_t slot, stage_bytes;
};

__host__ __device__ inline uint32_t round128(uint64_t b) { return (uint32_t)((b + 127) / 128 * 128); }

__host__ __device__ inline bool decode_plan(uint32_t dyn, int mmax, int H, int F, bool swi, DecodePlan* p) {
  const uint32_t row0 = (uint32_t)H * 2u, row1 = (uint32_t)F * 2u, wrow0 = row0 * (swi ? 2u : 1u);
  p->slot = round128((uint64_t)mmax * (uint32_t)(H > F ? H : F) * 2u);
  for (int nab = 2; nab >= 1; --nab) {
    if ((uint64_t)nab * p->slot >= dyn) continue;
    const uint32_t room = dyn - (uint32_t)nab * p->slot;
    for (int need = 3; need >= 2; --need)
      for (int r = kConsumers; r >= 1; r >>= 1) {
        const uint32_t sb = (uint32_t)r * wrow0;
        if (sb >= row1 && room / sb >= (uint32_t)need) {
          p->nab = nab;
          p->rps0 = r;
          p->stage_bytes = sb;
          p->rps1 = (int)(sb / row1) < kConsumers ? (int)(sb / row1) : kConsumers;
          p->stages = (int)(room / sb) < kMaxStages ? (int)(room / sb) : kMaxStages;
          return true;
        }
      }
  }
  return false;
}

// The stages of one CTA: its rows [r, rb) of the first product's A * F
// weight rows (expert ai = row / F, column n0 = row % F), then its rows
// [r2a, r2b) of the second product's A * H; each stage at most rps rows of
// one expert.  gl counts the stages within each product.
struct Stage {
  bool second;
  int ai, n0, rows, gl;
};
struct StageWalk {
  int r, rb, r2a, r2b, F, H, rps0, rps1;
  bool second = false;
  int gl = 0;
  __device__ __forceinline__ bool next(Stage& sg) {
    if (!second && r >= rb) {
      second = true;
      r = r2a;
      rb = r2b;
      gl = 0;
    }
    if (r >= rb) return false;
    const int N = second ? H : F, rps = second ? rps1 : rps0;
    sg.second = second;
    sg.ai = r / N;
    sg.n0 = r % N;
    sg.rows = min(rps, min(rb - r, N - sg.n0));
    sg.gl = gl++;
    r += sg.rows;
    return true;
  }
};

// Relative time per weight row of an expert with m rows, as measured on
// the layer: the dots of one and two rows keep up with HBM, more rows make
// a CTA's stages compute-bound.  The shares of the weight rows follow it.
__device__ __forceinline__ int row_cost(int m) { return m <= 1 ? 8 : m == 2 ? 9 : m == 3 ? 12 : m == 4 ? 14 : 3 * m; }

// The first row of the b-th of nb shares of the A experts' N-row weight
// matrices (rows of expert a are a N .. a N + N - 1), the shares cut at
// equal sums of row_cost over their rows.
__device__ __forceinline__ int share_start(int b, int nb, int A, int N, const int* ue, const int* offs) {
  int64_t total = 0;
  for (int a = 0; a < A; ++a) total += (int64_t)N * row_cost(offs[ue[a] + 1] - offs[ue[a]]);
  const int64_t x = total * b / nb;
  int64_t c = 0;
  for (int a = 0; a < A; ++a) {
    const int w = row_cost(offs[ue[a] + 1] - offs[ue[a]]);
    const int64_t span = (int64_t)N * w;
    if (x < c + span) return a * N + (int)((x - c) / w);
    c += span;
  }
  return A * N;
}

__device__ __forceinline__ void bar_consumers() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory"); }

// Tokens per gate-score unit: a unit is (gate row, piece, group of up to
// kTokGroup tokens).  Each token's score piece is the same sum in the same
// order whichever unit computes it.
constexpr int kTokGroup = 4;

// One unit: the piece's kSmallChunk x 32 vectors of the gate row, staged in
// gws ([chunk][lane]), dotted with tokens t0 .. t0 + nt - 1 of xs; lane l
// takes vectors c0 + l + 32 u in order u = 0, 1, ... (as the decode router
// does), sums over the warp, and lane 0 hands each token's piece to
// store(t, v).  The loop over u stays rolled: this code runs once per layer
// with its instructions cold.
template <typename Store>
__device__ __forceinline__ void score_group(const uint4* gws, const uint4* xs, int kv, int c0, int t0, int nt,
                                            Store store) {
  const int lane = threadIdx.x & 31;
  float acc[kTokGroup];
#pragma unroll
  for (int t = 0; t < kTokGroup; ++t) acc[t] = 0.f;
#pragma unroll 1
  for (int u = 0; u < route::kSmallChunk; ++u) {
    const int v = c0 + lane + 32 * u;
    if (v < kv) {
      const uint4 g = gws[u * 32 + lane];
#pragma unroll
      for (int t = 0; t < kTokGroup; ++t)
        if (t < nt) acc[t] = fma8_bf16(xs[(t0 + t) * kv + v], g, acc[t]);
    }
  }
#pragma unroll
  for (int t = 0; t < kTokGroup; ++t) {
    if (t < nt) {
      float v = acc[t];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) store(t0 + t, v);
    }
  }
}

template <int kEpi, int kMR>
__global__ void __launch_bounds__(kThreads, kMR <= 2 ? 2 : 1) decode_layer_kernel(const DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_ids[kMaxSlots];
  __shared__ float s_w[kMaxSlots];
  __shared__ int s_pos[kMaxSlots];
  __shared__ int s_src[kMaxSlots];
  __shared__ int s_run[256];
  __shared__ int s_offs[257];
  __shared__ int s_ue[256];
  __shared__ float s_sa[256];
  __shared__ int s_A, s_mmax, s_drop, s_abort;
  __shared__ int s_rows[4];   // this CTA's rows [r1a, r1b) and [r2a, r2b)
  __shared__ __align__(8) uint64_t s_bar[2 * kMaxStages + 5];
  constexpr bool kSwi = kEpi == kEpiSwiglu;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nb = (int)gridDim.x, b = (int)blockIdx.x;
  const int T = a.T, H = a.H, E = a.E, K = a.K, F = a.F, S = T * K;
  const int kvH = H / 8, kvF = F / 8;
  auto full = [&](int s) { return tc::smem_u32(&s_bar[s]); };
  auto empty = [&](int s) { return tc::smem_u32(&s_bar[kMaxStages + s]); };
  auto act_full = [&](int i) { return tc::smem_u32(&s_bar[2 * kMaxStages + i]); };
  auto act_empty = [&](int i) { return tc::smem_u32(&s_bar[2 * kMaxStages + 2 + i]); };
  const uint32_t xbar = tc::smem_u32(&s_bar[2 * kMaxStages + 4]);

  if (tid == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      tc::mbar_init(full(s), 1);
      tc::mbar_init(empty(s), kConsumers);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(act_full(i), 1);
      tc::mbar_init(act_empty(i), kConsumers);
    }
    tc::mbar_init(xbar, 1);
    s_abort = 0;
    tc::fence_barrier_init();
  }
  __syncthreads();
  pdl_enter();

  // ---------------------------------------------------------- 1. gate scores
  // unit u = (gate row, piece, token group) -> CTA u mod nb, consumer warp
  // (u / nb) mod 8; CTAs with units stage the token rows, and each of their
  // warps stages its unit's gate piece after them
  const int pieces = route::small_pieces(H);
  const int groups = (T + kTokGroup - 1) / kTokGroup;
  const int units = E * pieces * groups;
  const int unit_warps = nb * kConsumers;
  const bool x_staged = b < units;
  if (x_staged) {
    if (tid == 0) {
      tc::mbar_arrive_expect_tx(xbar, (uint32_t)(T * H * 2));
      tc::bulk_load(tc::smem_u32(smem), a.x, (uint32_t)(T * H * 2), xbar);
    }
    const int first = b + nb * warp;
    if (warp < kConsumers && first < units) {
      uint4* gws = reinterpret_cast<uint4*>(smem + round128((uint64_t)T * H * 2)) + warp * route::kSmallChunk * 32;
      uint4 gw[route::kSmallChunk];
      auto load_unit = [&](int u) {
        const int e = u / (pieces * groups);
        const int c0 = (u / groups % pieces) * 32 * route::kSmallChunk;
        const uint4* row = reinterpret_cast<const uint4*>(a.Wg + (int64_t)e * H);
#pragma unroll
        for (int i = 0; i < route::kSmallChunk; ++i) {
          const int v = c0 + lane + 32 * i;
          if (v < kvH) gw[i] = __ldg(row + v);
        }
      };
      load_unit(first);
      int done = 0;
      if (tc::mbar_wait(xbar, 0, &s_abort, kWaitNs)) {
#pragma unroll 1
        for (int u = first; u < units; u += unit_warps) {
          const int e = u / (pieces * groups), c = u / groups % pieces, t0 = (u % groups) * kTokGroup;
          __syncwarp();
#pragma unroll
          for (int i = 0; i < route::kSmallChunk; ++i) gws[i * 32 + lane] = gw[i];
          __syncwarp();
          if (u + unit_warps < units) load_unit(u + unit_warps);   // the next unit's loads fly meanwhile
          score_group(gws, reinterpret_cast<const uint4*>(smem), kvH, c * 32 * route::kSmallChunk, t0,
                      min(kTokGroup, T - t0), [&](int t, float v) { a.part[((int64_t)c * T + t) * E + e] = v; });
          ++done;
        }
      } else if (lane == 0) {
        set_error(a.err, kDevTimeout);
        s_abort = 1;
      }
      __syncwarp();
      if (lane == 0 && done > 0) {
        __threadfence();
        atomicAdd(a.ctr, done);
      }
    }
  }
  if (tid == 0 && !wait_count(a.ctr, units, &s_abort)) {
    set_error(a.err, kDevTimeout);
    s_abort = 1;
  }
  __syncthreads();
  const bool routed = !s_abort;

  // ---------------------------------------------------------- 2. routing, placement
  float* ls = reinterpret_cast<float*>(smem);   // [T][E + 1], over the staged token rows
  if (routed) {
#pragma unroll 1
    for (int i = tid; i < T * E; i += kThreads) {
      const int t = i / E, e = i % E;
      float v = 0.f;
#pragma unroll 1
      for (int c = 0; c < pieces; ++c) v += __ldcg(a.part + ((int64_t)c * T + t) * E + e);
      if (a.gate_bias) v += a.gate_bias[e];
      ls[t * (E + 1) + e] = v;
    }
  }
  __syncthreads();
  if (routed) route::finish_tokens(ls, T, 0, E, K, a.inv_tau, s_ids, s_w, warp, kThreads / 32);
  __syncthreads();
  if (routed && warp == 0) {
    // stable ranks per expert in slot order (warp match per 32 slots)
    for (int e = lane; e < 256; e += 32) s_run[e] = 0;
    __syncwarp();
#pragma unroll 1
    for (int c0 = 0; c0 < S; c0 += 32) {
      const int s = c0 + lane;
      int e = s < S ? s_ids[s] : -1;
      if (s < S && (e < 0 || e >= E)) {   // NaN scores: no expert
        if (b == 0) set_error(a.err, kDevBadIndex);
        e = -1;
      }
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const unsigned below = peers & lanemask_lt();
      const int rank = e >= 0 ? s_run[e] + __popc(below) : -1;
      __syncwarp();
      if (e >= 0 && below == 0) s_run[e] += __popc(peers);
      __syncwarp();
      if (s < S) {
        s_ids[s] = e;
        s_pos[s] = rank;
      }
    }
    __syncwarp();
    // kept rows per expert (the first C), their offsets, the experts with rows
    int kept[8], sum = 0, drop = 0, mx = 0, used = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      const int r = e < E ? s_run[e] : 0;
      kept[i] = (a.C > 0 && r > a.C) ? a.C : r;
      sum += kept[i];
      drop += r - kept[i];
      mx = max(mx, kept[i]);
      used += kept[i] > 0;
    }
    int incl = sum, uincl = used;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o), u = __shfl_up_sync(0xffffffffu, uincl, o);
      if (lane >= o) {
        incl += v;
        uincl += u;
      }
    }
    int off = incl - sum, uoff = uincl - used;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      s_offs[e] = off;
      off += kept[i];
      if (kept[i] > 0) s_ue[uoff++] = e;
    }
    if (lane == 31) {
      s_offs[256] = incl;
      s_A = uincl;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      drop += __shfl_xor_sync(0xffffffffu, drop, o);
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (lane == 0) {
      s_drop = drop;
      s_mmax = mx;
    }
    __syncwarp();
    // this CTA's shares of the two products' weight rows
    if (lane < 4) {
      const int N = lane < 2 ? F : H;
      s_rows[lane] = share_start(b + (lane & 1), nb, s_A, N, s_ue, s_offs);
    }
#pragma unroll 1
    for (int c0 = 0; c0 < S; c0 += 32) {
      const int s = c0 + lane;
      if (s < S) {
        const int e = s_ids[s], r = s_pos[s];
        const int p = (e >= 0 && (a.C <= 0 || r < a.C)) ? s_offs[e] + r : -1;
        s_pos[s] = p;
        if (p >= 0) s_src[p] = s;
      }
    }
  }
  __syncthreads();
  if (routed && b == 0 && tid < 256) {
    // the layer's statistics: counts, probability sums (the loss is
    // reduced after the expert products, off the critical path)
    const int e = tid;
    float p = 0.f;
    if (e < E) {
      float sum = 0.f;
#pragma unroll 1
      for (int t = 0; t < T; ++t) sum += ls[t * (E + 1) + e];
      p += sum;
      if (a.psum) a.psum[e] = p;
      if (a.count) a.count[e] = s_run[e];
      if (a.count_copy) a.count_copy[e] = s_run[e];
    }
    s_sa[e] = p;
    if (e == 0) {
      if (a.dropped) *a.dropped = s_drop;
      if (a.dropped_copy) *a.dropped_copy = s_drop;
    }
  }
  tc::fence_proxy_async_smem();   // the generic writes above before the bulk copies into the same bytes
  __syncthreads();                // ls is dead from here: the ring takes its place

  // ---------------------------------------------------------- 3. expert products
  DecodePlan pl{};
  const bool planned = routed && decode_plan(a.dyn_bytes, s_mmax, H, F, kSwi, &pl);
  if (routed && !planned && tid == 0) set_error(a.err, kDevBadIndex);
  const uint32_t row0 = (uint32_t)H * 2u, row1 = (uint32_t)F * 2u;
  // this CTA's weight rows: the b-th of nb shares of the A * F rows of the
  // first product and of the A * H rows of the second, cut at equal cost
  const int r1a = planned ? s_rows[0] : 0, r1b = planned ? s_rows[1] : 0;
  const int r2a = planned ? s_rows[2] : 0, r2b = planned ? s_rows[3] : 0;
  const StageWalk walk0{r1a, r1b, r2a, r2b, F, H, pl.rps0, pl.rps1};
  const uint32_t s_act = tc::smem_u32(smem), s_ring = s_act + (uint32_t)pl.nab * pl.slot;
  const uint8_t* ring = smem + (size_t)pl.nab * pl.slot;

  uint32_t filled = 0, fill_par = 0;   // producer: per stage, ever filled / parity of its last fill
  uint32_t afilled = 0, afill_par = 0;  // activation warp: the same per buffer
  bool producer = false, loader = false;
  if (warp == kProducer) {
    // ------------------------------------------------------------ producer
    if (tc::elect_one()) {
      producer = true;
      bool ok = true;
      StageWalk walk = walk0;
      Stage sg;
#pragma unroll 1
      for (int g = 0; planned && walk.next(sg); ++g) {
        const int s = g % pl.stages;
        const uint32_t ph = (uint32_t)(g / pl.stages) & 1u;
        if (!tc::mbar_wait(empty(s), ph ^ 1u, &s_abort, kWaitNs)) {
          ok = false;
          break;
        }
        const uint32_t dst = s_ring + (uint32_t)s * pl.stage_bytes;
        const int e = s_ue[sg.ai];
        if (!sg.second) {
          const uint32_t bytes = (uint32_t)sg.rows * row0;
          const bf16* Be = a.W1 + (int64_t)e * F * H * (kSwi ? 2 : 1);
          tc::mbar_arrive_expect_tx(full(s), kSwi ? 2 * bytes : bytes);
          tc::bulk_load(dst, Be + (int64_t)sg.n0 * H, bytes, full(s));
          if (kSwi) tc::bulk_load(dst + (uint32_t)pl.rps0 * row0, Be + (int64_t)(F + sg.n0) * H, bytes, full(s));
        } else {
          const uint32_t bytes = (uint32_t)sg.rows * row1;
          tc::mbar_arrive_expect_tx(full(s), bytes);
          tc::bulk_load(dst, a.W2 + ((int64_t)e * H + sg.n0) * F, bytes, full(s));
        }
        filled |= 1u << s;
        fill_par = (fill_par & ~(1u << s)) | (ph << s);
      }
      if (!ok) {
        set_error(a.err, kDevTimeout);
        s_abort = 1;
      }
    }
    __syncwarp();
  } else if (warp == kActWarp) {
    // ------------------------------------------------------------ activation rows
    if (tc::elect_one() && planned && (r1b > r1a || r2b > r2a)) {
      loader = true;
      int seg = 0;
      bool ok = true;
      auto load_seg = [&](bool second, int ai) {
        const int i = seg % pl.nab;
        if (seg >= pl.nab && !tc::mbar_wait(act_empty(i), (uint32_t)(seg / pl.nab - 1) & 1u, &s_abort, kWaitNs))
          return false;
        const int e = s_ue[ai], r0 = s_offs[e], m = s_offs[e + 1] - r0;
        const uint32_t dst = s_act + (uint32_t)i * pl.slot;
        if (second) {
          // the expert's h rows, once all F of its first-product columns are counted
          if (!wait_count(a.ctr + kCtrFixed + e, F, &s_abort)) return false;
          tc::mbar_arrive_expect_tx(act_full(i), (uint32_t)m * row1);
          tc::bulk_load(dst, a.h + (int64_t)r0 * F, (uint32_t)m * row1, act_full(i));
        } else {
          tc::mbar_arrive_expect_tx(act_full(i), (uint32_t)m * row0);
          for (int r = 0; r < m; ++r)
            tc::bulk_load(dst + (uint32_t)r * row0, a.x + (int64_t)(s_src[r0 + r] / K) * H, row0, act_full(i));
        }
        afilled |= 1u << i;
        afill_par = (afill_par & ~(1u << i)) | (((uint32_t)(seg / pl.nab) & 1u) << i);
        ++seg;
        return true;
      };
      if (r1b > r1a)
        for (int ai = r1a / F; ok && ai <= (r1b - 1) / F; ++ai) ok = load_seg(false, ai);
      if (r2b > r2a)
        for (int ai = r2a / H; ok && ai <= (r2b - 1) / H; ++ai) ok = load_seg(true, ai);
      if (!ok) {
        set_error(a.err, kDevTimeout);
        s_abort = 1;
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ consumers
    // A warp whose wait failed does no more work but still passes every
    // consumers' barrier, so the other consumer warps never wait there for it.
    bool ok = planned;
    int seg = -1, cur_ai = -1, seg_rows = 0, e = 0, r0 = 0, m = 0;
    bool cur_second = false;
    const uint4* act = nullptr;
    auto fail = [&]() {
      ok = false;
      if (lane == 0) set_error(a.err, kDevTimeout);
      s_abort = 1;
    };
    auto end_seg = [&]() {
      __syncwarp();
      if (ok && lane == 0) tc::mbar_arrive(act_empty(seg % pl.nab));   // done with the rows
      if (!cur_second) {
        // the expert's first-product columns of this CTA: fenced, then counted
        __threadfence();
        bar_consumers();
        if (tid == 0 && ok) atomicAdd(a.ctr + kCtrFixed + e, seg_rows);
      }
    };
    StageWalk walk = walk0;
    Stage sg;
#pragma unroll 1
    for (int g = 0; planned && walk.next(sg); ++g) {
      if (seg < 0 || sg.second != cur_second || sg.ai != cur_ai) {
        if (seg >= 0) end_seg();
        ++seg;
        cur_second = sg.second;
        cur_ai = sg.ai;
        seg_rows = 0;
        e = s_ue[sg.ai];
        r0 = s_offs[e];
        m = s_offs[e + 1] - r0;
        act = reinterpret_cast<const uint4*>(smem + (size_t)(seg % pl.nab) * pl.slot);
        if (ok && !tc::mbar_wait(act_full(seg % pl.nab), (uint32_t)(seg / pl.nab) & 1u, &s_abort, kWaitNs))
          fail();
      }
      seg_rows += sg.rows;
      const int s = g % pl.stages;
      const uint32_t ph = (uint32_t)(g / pl.stages) & 1u;
      if (!ok) continue;
      if (!tc::mbar_wait(full(s), ph, &s_abort, kWaitNs)) {
        fail();
        continue;
      }
      const uint8_t* st = ring + (size_t)s * pl.stage_bytes;
      // a segment of 2-4 rows dots two weight rows per warp (twice the
      // independent sums, half the activation reads); else one
      const bool pairs = m >= 1 && m <= (kMR < 4 ? kMR : 4);
      const int rps = sg.second ? pl.rps1 : pl.rps0;
      const int j = stage_row_of_warp(sg.gl, pairs ? (rps + 1) / 2 : rps, warp) * (pairs ? 2 : 1);
      if (j < sg.rows) {
        const bool two = pairs && j + 1 < sg.rows;
        const int c = sg.n0 + j;
        if (!sg.second) {
          const float* be = a.b1 ? a.b1 + (int64_t)e * F * (kSwi ? 2 : 1) : nullptr;
          bf16* o = a.h + (int64_t)r0 * F + c;
          if (two) stage_pair<kEpi, kMR>(st, j, rps, row0, act, kvH, m, be, c, F, o);
          else stage_row<bf16, kEpi, kMR>(st, j, rps, row0, act, kvH, m, be, c, F, o);
        } else {
          const float* be = a.b2 ? a.b2 + (int64_t)e * H : nullptr;
          bf16* o = a.y + (int64_t)r0 * H + c;
          if (two) stage_pair<kEpiPlain, kMR>(st, j, rps, row1, act, kvF, m, be, c, H, o);
          else stage_row<bf16, kEpiPlain, kMR>(st, j, rps, row1, act, kvF, m, be, c, H, o);
        }
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(empty(s));   // this warp is done with the stage
    }
    if (seg >= 0) end_seg();

    if (routed && b == 0) {
      // the loss: E * sum_i (count_i / (T K)) * (psum_i / T), reduced over 256
      // entries in a fixed order
      const int e = tid;
      s_sa[e] = (e < E && T > 0) ? ((float)s_run[e] / (float)(T * K)) * (s_sa[e] / (float)T) : 0.f;
      bar_consumers();
#pragma unroll 1
      for (int o = 128; o > 0; o >>= 1) {
        if (e < o) s_sa[e] += s_sa[e + o];
        bar_consumers();
      }
      if (e == 0 && a.aux) *a.aux = (float)E * s_sa[0];
    }

    // ---------------------------------------------------------- 4. combine
    // this CTA's second-product rows are fenced and counted; the CTAs with
    // output items wait for every CTA's count, then combine (item it ->
    // CTA it mod nb, consumer warp it / nb mod 8)
    __threadfence();
    bar_consumers();
    if (tid == 0 && planned) atomicAdd(a.ctr + 1, 1);
    const int chunk = combine_chunk();
    const int64_t items = (int64_t)T * ((kvH + chunk - 1) / chunk);
    if (planned && b < items) {
      if (tid == 0 && !wait_count(a.ctr + 1, nb, &s_abort)) {
        set_error(a.err, kDevTimeout);
        s_abort = 1;
      }
      bar_consumers();
      if (!s_abort) {
        const uint4* yv = reinterpret_cast<const uint4*>(a.y);
        uint4* ov = reinterpret_cast<uint4*>(a.out);
        const int64_t w0 = b + (int64_t)nb * warp, nw = (int64_t)nb * kConsumers;
        if (K <= 2) combine_items<bf16, 2>(yv, s_pos, s_w, T, K, kvH, chunk, ov, w0, nw);
        else if (K <= 4) combine_items<bf16, 4>(yv, s_pos, s_w, T, K, kvH, chunk, ov, w0, nw);
        else combine_items<bf16, 8>(yv, s_pos, s_w, T, K, kvH, chunk, ov, w0, nw);
      }
    }
  }
  __syncthreads();
  // after an abort, copies issued but never consumed land before the CTA leaves
  if (s_abort) {
    if (tid == 0 && x_staged) tc::mbar_wait(xbar, 0, nullptr, kWaitNs);
    if (producer)
      for (int s = 0; s < pl.stages; ++s)
        if ((filled >> s) & 1u) tc::mbar_wait(full(s), (fill_par >> s) & 1u, nullptr, kWaitNs);
    if (loader)
      for (int i = 0; i < pl.nab; ++i)
        if ((afilled >> i) & 1u) tc::mbar_wait(act_full(i), (afill_par >> i) & 1u, nullptr, kWaitNs);
  }
}

// The counters the layer kernel waits on, zeroed once the kernel before it
// on the stream (which may still use them) has finished.
__global__ void decode_ctr_zero_kernel(int* ctr, int n) {
  pdl_trigger();
  pdl_wait();
  for (int i = threadIdx.x; i < n; i += blockDim.x) ctr[i] = 0;
}

// CTAs per SM: two for batches of at most two tokens (bodies for two rows,
// so both fit the register file), else one.
int decode_per_sm(const Shape& s) { return s.T <= 2 ? 2 : 1; }

using KernelFn = void (*)(const DecodeArgs);

KernelFn decode_kernel_for(const Shape& s) {
  const bool swi = (s.flags & MOE_FLAG_SWIGLU) != 0;
  if (decode_per_sm(s) == 2) return swi ? decode_layer_kernel<kEpiSwiglu, 2> : decode_layer_kernel<kEpiGelu, 2>;
  return swi ? decode_layer_kernel<kEpiSwiglu, kMaxTok> : decode_layer_kernel<kEpiGelu, kMaxTok>;
}

uint32_t decode_dyn(const Shape& s) { return decode_per_sm(s) == 2 ? kDynPair : kDynSingle; }

// Shared memory needs at the batch's worst case (one expert with all T
// rows): the staged token rows, the score table, and a plan.
bool decode_fits(const Shape& s, uint32_t dyn) {
  const uint64_t xrows = (uint64_t)s.T * s.H * 2;
  if (xrows >= (1u << 20)) return false;
  if (round128(xrows) + (uint64_t)kConsumers * route::kSmallChunk * 32 * 16 > dyn) return false;
  if ((uint64_t)s.T * (s.E + 1) * 4 > dyn) return false;
  DecodePlan p;
  return decode_plan(dyn, (int)s.T, s.H, s.F, (s.flags & MOE_FLAG_SWIGLU) != 0, &p);
}

}  // namespace

bool decode_layer_eligible(const Shape& s) {
  if (s.dtype != MOE_BF16 || s.T < 1 || s.T > kMaxTok || s.E > 256 || s.K > 8) return false;
  if (s.flags & (MOE_FLAG_DECODE_SPLIT | MOE_FLAG_NO_DECODE | MOE_FLAG_FFN_SPLIT | MOE_FLAG_SIMT_ROUTER))
    return false;
  if ((s.flags & MOE_FLAG_REROUTE) && s.C > 0) return false;
  if (!router_small(s) || !stream_fused(s)) return false;
  return decode_fits(s, decode_dyn(s));
}

size_t decode_part_floats(const Shape& s) { return (size_t)route::small_pieces(s.H) * (size_t)s.T * s.E; }
int decode_ctr_words(const Shape& s) { return kCtrFixed + s.E; }

cudaError_t launch_decode_layer(const Shape& s, const DecodeIO& io, cudaStream_t st) {
  const uint32_t dyn = decode_dyn(s);
  const int per_sm = decode_per_sm(s);
  if (!decode_fits(s, dyn)) return cudaErrorNotSupported;
  KernelFn k = decode_kernel_for(s);
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
  if (e != cudaSuccess) return e;
  // every CTA must be resident at once (the counter waits)
  int fit = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, k, kThreads, dyn);
  if (e != cudaSuccess) return e;
  if (fit < per_sm) return cudaErrorNotSupported;
  e = launch_kernel(decode_ctr_zero_kernel, dim3(1), dim3(256), 0, st, 1, io.ctr, decode_ctr_words(s));
  if (e != cudaSuccess) return e;
  DecodeArgs a;
  a.x = (const bf16*)io.x;
  a.Wg = (const bf16*)io.Wg;
  a.gate_bias = io.gate_bias;
  a.W1 = (const bf16*)io.W1;
  a.b1 = io.b1;
  a.W2 = (const bf16*)io.W2;
  a.b2 = io.b2;
  a.out = (bf16*)io.out;
  a.T = (int)s.T;
  a.H = s.H;
  a.E = s.E;
  a.K = s.K;
  a.F = s.F;
  a.C = s.C;
  a.inv_tau = s.inv_tau;
  a.part = io.part;
  a.ctr = io.ctr;
  a.h = (bf16*)io.h;
  a.y = (bf16*)io.y;
  a.count = io.count;
  a.count_copy = io.count_copy;
  a.dropped = io.dropped;
  a.dropped_copy = io.dropped_copy;
  a.psum = io.psum;
  a.aux = io.aux;
  a.err = io.err;
  a.dyn_bytes = dyn;
  return launch_kernel(k, dim3((unsigned)(sm_count() * per_sm)), dim3(kThreads), dyn, st, 1, a);
}

}  // namespace moe
