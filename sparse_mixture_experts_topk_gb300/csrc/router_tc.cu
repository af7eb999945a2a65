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
// so the kernel is built to stream x at HBM speed:
//   * one 128-token tile per CTA group; x and Wg k-blocks (64 bf16 = 128
//     bytes, 128B swizzle) arrive by TMA into a ring of up to 8 stages (as
//     deep as shared memory allows with the grid in one wave);
//   * one thread issues tcgen05.mma M=128, N=E rounded up to 16, K=16 into
//     TMEM (fp32);
//   * when the tiles fill less than half the GPU, the hidden dimension is
//     split over a CTA pair (a 2-CTA cluster); each CTA copies its partial
//     scores TMEM -> shared memory (a sum of two partials does not depend on
//     their order, so either CTA may add them);
//   * each CTA of the pair then finishes half of the tile's tokens with all
//     of its 256 threads: the peer's partial scores added by coalesced
//     distributed-shared-memory loads, then the bias; G = 2 ks lanes per
//     token take the k best experts in k rounds of a group arg-max (each
//     round restricted to the entries ranked after the previous pick), then
//     the softmax statistics and weights; the tokens' probabilities are
//     summed per expert into psum_part[tile * ks + rank], and the tile's
//     chosen experts are counted into tile_hist[tile] (the dispatch
//     histogram of the tile's 128*k slots, so the layer needs no separate
//     histogram pass; the peer's counts reach the leader by a distributed
//     shared-memory reduction).
// Every mbarrier wait is bounded; on expiry the kernel records a timeout in
// the error word, skips the remaining work, still meets both cluster
// barriers, frees TMEM and returns.
#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {

namespace {

constexpr int kTok = 128;        // tokens per tile = TMEM lanes
constexpr int kBK = 64;          // bf16 per k-block
constexpr int kThreads = 256;
constexpr int kMaxStages = 8;
constexpr int kABytes = kTok * kBK * 2;
constexpr uint64_t kWaitNs = 2000000000ull;

struct RouterCfg {
  int stages;      // ring depth
  int npad;        // MMA N: E rounded up to a multiple of 16 (>= 16)
  int tmem_cols;   // power of two >= max(32, npad)
  int b_bytes;     // one Wg k-block: npad rows x 128 bytes
  size_t smem;     // dynamic shared memory
};

// 16 bytes from a cluster peer's shared memory (ordered after the preceding
// cluster barrier, which clobbers memory; no clobber here, so several can be
// in flight together).
__device__ __forceinline__ float4 ld_peer_v4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

// Row pitch (fp32 words) of the score table: E padded to whole 32-word rows,
// plus the G = 2 ks lanes that finish one token, so that G-wide vector stores
// from TMEM and the G-lane token groups both meet 32 distinct banks.
__host__ __device__ inline int part_pitch(int npad, int ks) { return (npad + 31) / 32 * 32 + 2 * ks; }

// ctas_per_sm: how many CTAs each SM must hold for the grid to run in one wave
RouterCfg router_cfg(int E, int ks, int ctas_per_sm) {
  RouterCfg c;
  c.npad = E < 16 ? 16 : (E + 15) / 16 * 16;
  c.tmem_cols = 32;
  while (c.tmem_cols < c.npad) c.tmem_cols *= 2;
  c.b_bytes = c.npad * 128;
  const size_t budget = (size_t)(200 * 1024) / (size_t)(ctas_per_sm < 1 ? 1 : ctas_per_sm);
  c.stages = (int)(budget / (size_t)(kABytes + c.b_bytes));
  if (c.stages > kMaxStages) c.stages = kMaxStages;
  if (c.stages < 2) c.stages = 2;
  const size_t ring = (size_t)c.stages * (kABytes + c.b_bytes);
  const size_t part = (size_t)kTok * part_pitch(c.npad, ks) * sizeof(float);
  c.smem = 1024 + (ring > part ? ring : part);
  return c;
}

__global__ void __launch_bounds__(kThreads)
router_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmG,
                 int64_t Tn, int H, int E, int K, int npad, int tmem_cols, int ks, int kStages, float inv_tau,
                 const float* __restrict__ gate_bias, float* __restrict__ logits,
                 int32_t* __restrict__ ids, float* __restrict__ w, float* __restrict__ psum_part,
                 int32_t* __restrict__ tile_hist, int* err) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_hist[256];
  __shared__ float s_red[kThreads];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ __align__(8) uint64_t s_bar[2 * kMaxStages + 1];

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sA = tc::smem_u32(smem);
  const int b_bytes = npad * 128;
  const uint32_t sB = sA + kStages * kABytes;
  float* part = reinterpret_cast<float*>(smem);   // reuses the ring once the MMAs are done
  const int G = 2 * ks;                           // lanes per token in the epilogue
  const int ld = part_pitch(npad, ks);
  auto full = [&](int s) { return tc::smem_u32(&s_bar[s]); };
  auto empty = [&](int s) { return tc::smem_u32(&s_bar[kStages + s]); };
  const uint32_t done_bar = tc::smem_u32(&s_bar[2 * kStages]);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ks > 1 ? tc::cluster_ctarank() : 0;
  const int64_t tile = blockIdx.x / ks;
  const int64_t t0 = tile * kTok;
  const int nk = (H + kBK - 1) / kBK;
  const int kb0 = (int)((int64_t)nk * rank / ks);
  const int kb1 = (int)((int64_t)nk * (rank + 1) / ks);
  const uint32_t idesc = tc::idesc_bf16_f32(kTok, npad);

  for (int e = threadIdx.x; e < 256; e += kThreads) s_hist[e] = 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(full(s), 1);
      tc::mbar_init(empty(s), 1);
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
  pdl_enter();                     // first global access below
  const uint32_t tmem = s_tmem;

  uint32_t filled = 0, fill_par = 0;   // producer: per stage, ever filled / parity of its last fill
  bool producer = false;
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (tc::elect_one()) {
      producer = true;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!tc::mbar_wait(empty(stage), phase ^ 1u, &s_abort, kWaitNs)) { ok = false; break; }
        tc::mbar_arrive_expect_tx(full(stage), kABytes + b_bytes);
        tc::tma_load_2d(sA + stage * kABytes, &tmX, full(stage), kb * kBK, (int)t0);
        tc::tma_load_2d(sB + stage * b_bytes, &tmG, full(stage), kb * kBK, 0);
        filled |= 1u << stage;
        fill_par = (fill_par & ~(1u << stage)) | (phase << stage);
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
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
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!tc::mbar_wait(full(stage), phase, &s_abort, kWaitNs)) { ok = false; break; }
        tc::tc_fence_after();
        const uint32_t a0 = sA + stage * kABytes, b0 = sB + stage * b_bytes;
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)
          tc::mma_bf16(tmem, tc::sdesc_k128(a0 + k * 32), tc::sdesc_k128(b0 + k * 32), idesc,
                       (kb > kb0 || k > 0) ? 1u : 0u);
        tc::tc_commit(empty(stage));
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
      if (!ok) {
        set_error(err, kDevTimeout);
        s_abort = 1;
      }
      tc::tc_commit(done_bar);   // arrives once every MMA above has finished
    }
    __syncwarp();
  }

  bool ok = tc::mbar_wait(done_bar, 0, nullptr, kWaitNs);
  if (!ok) set_error(err, kDevTimeout);
  // after an abort, loads issued but never consumed land before the ring is reused
  if (producer && (s_abort || !ok))
    for (int s = 0; s < kStages; ++s)
      if ((filled >> s) & 1u) tc::mbar_wait(full(s), (fill_par >> s) & 1u, nullptr, kWaitNs);
  ok = ok && !s_abort && kb1 > kb0;
  tc::tc_fence_after();
  __syncthreads();                 // the ring is free: every load landed and was consumed

  // partial scores TMEM -> shared memory, all 128 rows: warps w and w + 4
  // both read TMEM lanes 32 (w % 4) .. + 31 and take alternate 32-column
  // chunks; each thread stores its row's values G at a time (the row pitch is
  // G mod 32 words, so these stores and the token groups' reads below are
  // free of bank conflicts)
  {
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    for (int c = (warp >> 2) * 32; c < npad; c += 64) {
      uint32_t r[32];
      tc::tmem_ld_32x32b_x32(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)c, r);
      tc::tmem_wait_ld();
      float* dst = part + row * ld + c;
      if (G == 4) {
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          if (c + j < npad)
            *reinterpret_cast<float4*>(dst + j) =
                ok ? make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]), __uint_as_float(r[j + 2]),
                                 __uint_as_float(r[j + 3]))
                   : make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
#pragma unroll
        for (int j = 0; j < 32; j += 2)
          if (c + j < npad)
            *reinterpret_cast<float2*>(dst + j) =
                ok ? make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])) : make_float2(0.f, 0.f);
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, tmem_cols);
  }

  // this CTA finishes the tile's rows [h0, h0 + nrow); with a pair it first
  // adds the other CTA's partial scores of those rows (ks <= 2: the sum of
  // two partials is the same in either order), then the gate bias.  Each
  // thread keeps one column slice (4 columns with a pair, 1 without) and
  // walks rows, so its bias is loaded once.
  const int nrow = kTok / ks;
  const int h0 = (int)rank * nrow;
  if (ks > 1) {
    tc::cluster_sync();            // both partials are in shared memory
    const int q = npad / 4;        // 16-byte slices per row
    const int rpp = kThreads / q;  // rows per pass
    const int r_off = (int)threadIdx.x / q, c4 = (int)threadIdx.x % q;
    float4 bv = make_float4(0.f, 0.f, 0.f, 0.f);
    if (gate_bias) {
      const int e = 4 * c4;
      bv = make_float4(e < E ? gate_bias[e] : 0.f, e + 1 < E ? gate_bias[e + 1] : 0.f,
                       e + 2 < E ? gate_bias[e + 2] : 0.f, e + 3 < E ? gate_bias[e + 3] : 0.f);
    }
    const uint32_t peer = tc::map_peer(tc::smem_u32(part), rank ^ 1u);
    if (r_off < rpp) {
      for (int r0 = r_off; r0 < nrow; r0 += 4 * rpp) {
        float4 pv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int rr = r0 + u * rpp;
          if (rr < nrow) pv[u] = ld_peer_v4(peer + 4u * (uint32_t)((h0 + rr) * ld + 4 * c4));
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int rr = r0 + u * rpp;
          if (rr < nrow) {
            float4* a = reinterpret_cast<float4*>(part + (h0 + rr) * ld + 4 * c4);
            float4 v = *a;
            v.x = (v.x + pv[u].x) + bv.x;
            v.y = (v.y + pv[u].y) + bv.y;
            v.z = (v.z + pv[u].z) + bv.z;
            v.w = (v.w + pv[u].w) + bv.w;
            *a = v;
          }
        }
      }
    }
  } else if (gate_bias) {
    const int rpp = kThreads / npad;
    const int r_off = (int)threadIdx.x / npad, e = (int)threadIdx.x % npad;
    const float b = e < E ? gate_bias[e] : 0.f;
    if (r_off < rpp)
#pragma unroll 1
      for (int rr = r_off; rr < nrow; rr += rpp) part[(h0 + rr) * ld + e] += b;
  }
  __syncthreads();
  const int64_t nt = (Tn - t0) < kTok ? (Tn - t0) : kTok;
  if (logits) {
    for (int i = threadIdx.x; i < nrow * E; i += kThreads) {
      const int rr = h0 + i / E, e = i % E;
      if (rr < nt) logits[(t0 + rr) * E + e] = part[rr * ld + e];
    }
  }

  // ------------------------------------------------------------ per token
  // G consecutive lanes finish one token; lane `sub` of the group holds the
  // experts sub, sub + G, ...  Selection j takes the best entry (score
  // descending, index ascending) among those ranked after selection j - 1,
  // so no entry is taken twice and no mask is kept.
  {
    const int sub = threadIdx.x & (G - 1);
    const int row = h0 + (int)threadIdx.x / G;
    const int64_t t = t0 + row;
    const bool live = row < nt;
    float* lr = part + row * ld;
    const int nv = E > sub ? (E - sub + G - 1) / G : 0;
    float sel_v[8];
    int sel_i[8];
    float prev_v = INFINITY;
    int prev_i = -1;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      sel_v[j] = -INFINITY;
      sel_i[j] = 0x7fffffff;
      if (j < K) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll 4
        for (int i = 0; i < nv; ++i) {
          const int e = sub + G * i;
          const float v = lr[e];
          const bool after = v < prev_v || (v == prev_v && e > prev_i);
          const bool better = v > bv || (v == bv && e < bi);
          if (after && better) {
            bv = v;
            bi = e;
          }
        }
        for (int o = 1; o < G; o <<= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
          if (ov > bv || (ov == bv && oi < bi)) {
            bv = ov;
            bi = oi;
          }
        }
        sel_v[j] = bv;
        sel_i[j] = bi;
        prev_v = bv;
        prev_i = bi;
      }
    }
    // full softmax for the load-balancing sums; the butterfly leaves the same
    // total in every lane of the group
    const float m = sel_v[0];
    float zs = 0.f;
#pragma unroll 4
    for (int i = 0; i < nv; ++i) {
      const int e = sub + G * i;
      const float z = expf((lr[e] - m) * inv_tau);
      lr[e] = z;
      zs += z;
    }
    for (int o = 1; o < G; o <<= 1) zs += __shfl_xor_sync(0xffffffffu, zs, o);
    const float inv = 1.f / zs;
#pragma unroll 4
    for (int i = 0; i < nv; ++i) {
      const int e = sub + G * i;
      lr[e] = live ? lr[e] * inv : 0.f;
    }
    float zsel = 0.f, z[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      z[j] = j < K ? expf((sel_v[j] - m) * inv_tau) : 0.f;
      zsel += z[j];
    }
    if (live) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j < K && (j & (G - 1)) == sub) {
          ids[t * K + j] = sel_i[j];
          w[t * K + j] = z[j] / zsel;
          if ((unsigned)sel_i[j] < (unsigned)E) atomicAdd(&s_hist[sel_i[j]], 1);   // NaN scores: none
        }
      }
    }
  }
  __syncthreads();
  // the tile's probabilities summed per expert: S interleaved row chunks per
  // expert, then the chunks' sums in order
  if (psum_part) {
    const int S = E >= kThreads ? 1 : kThreads / E;
    if ((int)threadIdx.x < S * E) {
      const int e = (int)threadIdx.x % E, c = (int)threadIdx.x / E;
      float sum = 0.f;
      for (int rr = h0 + c; rr < h0 + nrow; rr += S) sum += part[rr * ld + e];
      s_red[threadIdx.x] = sum;
    }
    __syncthreads();
    if ((int)threadIdx.x < E) {
      float sum = 0.f;
      for (int c = 0; c < S; ++c) sum += s_red[c * E + threadIdx.x];
      psum_part[(tile * ks + rank) * E + threadIdx.x] = sum;
    }
  }
  if (tile_hist && rank != 0)
    for (int e = threadIdx.x; e < E; e += kThreads)
      tc::red_peer_add_u32(tc::map_peer(tc::smem_u32(&s_hist[e]), 0), (uint32_t)s_hist[e]);
  if (ks > 1) tc::cluster_sync();  // the peer's counts have reached the leader; neither leaves early
  if (tile_hist && rank == 0)
    for (int e = threadIdx.x; e < E; e += kThreads) tile_hist[tile * E + e] = s_hist[e];
}

}  // namespace

// The hidden dimension is split over a CTA pair when that still fits one
// wave (wider splits measured slower: cluster scheduling and the reduction;
// the pair epilogue also relies on at most two partials).
int router_tc_split(const Shape& s) {
  const int64_t tiles = (s.T + kTok - 1) / kTok;
  const int nk = (s.H + kBK - 1) / kBK;
  return (tiles * 2 <= sm_count() && nk >= 2) ? 2 : 1;
}

bool router_on_tensor_cores(const Shape& s) {
  return s.dtype == MOE_BF16 && s.H >= kBK && s.E <= 256 && !(s.flags & MOE_FLAG_SIMT_ROUTER);
}

cudaError_t launch_router_tc(const Shape& s, const void* x, const void* Wg, const float* gate_bias,
                             float* logits, int32_t* ids, float* w, float* psum_part,
                             int32_t* tile_hist, int* err, cudaStream_t st) {
  const int64_t tiles = (s.T + kTok - 1) / kTok;
  const int sms = sm_count();
  const int ks = router_tc_split(s);
  const int per_sm = (int)((tiles * ks + sms - 1) / sms);
  const RouterCfg c = router_cfg(s.E, ks, per_sm);
  CUtensorMap mx, mg;
  if (!tma_map_bf16(&mx, x, (uint64_t)s.T, (uint64_t)s.H, kTok)) return cudaErrorNotSupported;
  if (!tma_map_bf16(&mg, Wg, (uint64_t)s.E, (uint64_t)s.H, (uint32_t)c.npad)) return cudaErrorNotSupported;
  auto kern = router_tc_kernel;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)c.smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, dim3((unsigned)(tiles * ks)), dim3(kThreads), c.smem, st, (unsigned)ks, mx, mg, s.T,
                       s.H, s.E, s.K, c.npad, c.tmem_cols, ks, c.stages, s.inv_tau, gate_bias, logits, ids, w, psum_part,
                       tile_hist, err);
}

}  // namespace moe
