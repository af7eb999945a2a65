// Expert FFN on CTA pairs: the grouped GEMM of ffn_tc.cu computed by the two
// SMs of a 2-CTA cluster (tcgen05 .cta_group::2, MMA M = 256).
//
// Same products (Qwen2-MoE module article, mlqm.cn, section 2.2: each expert
// is Linear -> GELU -> Linear):
//   first:  h = GELU(x_perm W1[e]^T + b1[e]);  second: y = h W2[e]^T + b2[e]
//
// Why pairs: with one SM per 128 x 256 tile, every k-block brings 48 KB into
// the SM (A 16 KB + B 32 KB) for 128 x 256 x 64 multiply-adds, and the
// measured kernel was bound by that load stream rather than by the tensor
// cores.  A pair computes 256 x 256 per k-block while each SM loads 32 KB.
//
// Orientation, per tile.  A full 256-row block of an expert's token rows
// runs in row orientation: MMA M = the 256 token rows (128 per CTA), N = 256
// weight rows (output columns, 128 per CTA), and each epilogue thread owns
// one token row of its CTA's accumulator.  An expert's last block, when it
// holds at most 128 rows, runs swapped in the GELU and plain products (a
// longer one keeps the row orientation: measured, its swapped tile took
// 20.2 us against 17.9 us for a full row-orientation tile):
// M = 256 weight rows, N = the block's token rows rounded up to 16 and split
// across the pair, so the block is padded to a multiple of 16 instead of to
// 256 (20% of the MMA work at the 8192-token layer).  Each CTA then loads
// only the 32-row boxes of token rows its half needs; the accumulator holds
// the transposed tile (TMEM lane = output column, column = token row), and
// each epilogue warp transposes its 32 x 32 blocks through 2 KB of shared
// memory so that global stores stay 16-byte vectors along the row.  A
// swapped block of at most 48 rows runs wide: each stage brings the weight
// rows of two n-tiles (in the stage's A and B slots) and the block's token
// rows (a third, 3 KB slot), and the MMA issuer writes two accumulators,
// 128 columns apart.  Such a block's tiles are bound by how fast the ring
// turns over, not by the MMAs, so twice the weight bytes per stage halves
// their count (measured: a 32-row tail tile took as long as a full one).  Full
// blocks stay in row orientation because that transpose costs shared-memory
// bandwidth the tensor cores need (measured: 15% slower for full tiles).
// The SwiGLU first product keeps the row orientation for every block (N =
// 128 gate rows in the leader and the matching 128 up rows in the peer), so
// each CTA's accumulator holds gate | up for the same output columns.
//
// One launch, both products.  The persistent pairs take the first
// product's tiles and then the second's from one queue.  A second-product
// tile needs every hidden column of its 256-row block, so its producers wait
// on that block's counter, which each epilogue warp of the block's
// first-product tiles advances once its stores are visible GPU-wide.  The
// pairs that finish the first product early thus start on the second instead
// of idling until the last first-product tile is done (with one launch per
// product they idled 10 us on average at the 8192-token layer).
//
// Roles, per CTA (192 threads), rank r = 0 (leader) or 1:
//   warp 0     TMA producer: this CTA's share of A and B for each k-block into
//              its ring; both CTAs' loads complete on the LEADER's `full`
//              barrier, which the leader arms for the pair's bytes;
//   warp 1     leader only: one thread issues tcgen05.mma.cta_group::2
//              (M = 256, K = 16) x 4 per stage; its commits arrive on the
//              `empty` / `tfull` barriers of both CTAs (multicast);
//   warps 2-5  epilogue in both CTAs: this CTA's 128 accumulator lanes from its
//              own TMEM -> bias -> activation -> bf16 -> global; then arrive on
//              the leader's `tempty` (256 arrivals = both CTAs).
// All waits are bounded (timeout -> error word + abort flag); the CTAs meet
// in cluster barriers after set-up and before exit so neither can touch the
// other's shared memory once it has left.
//
// Gathering instantiation (kGather): the first product's token rows are read
// from x by the slot list instead of from x_perm, so the layer runs no
// gather kernel (Qwen2-MoE walkthrough, jsqmd.com, section 3.1 item 3).  The
// whole of warp 0 copies them with 16-byte cp.async copies into the stage,
// in the 128-byte swizzle; a stage counts as full once both CTAs' warps have
// waited for their copies, fenced them for the async proxy and arrived.  It
// gives the same bits as x_perm and is measured about 4x slower (the small
// copies do not keep up with the MMAs), so it is not the default.
#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {

namespace {

constexpr int kBM = 128;             // A rows per CTA (the pair covers M = 256)
constexpr int kBNh = 128;            // B rows per CTA at most (the pair covers N <= 256)
constexpr int kBK = 64;
constexpr int kBoxB = 32;            // swapped: token rows per B box
constexpr int kBoxT = 24;            // wide swapped tiles: token rows per box (a stage's T region)
constexpr int kWideRows = 48;        // a tail block of at most this many rows runs wide
constexpr int kSwapRows = 128;       // a tail block of more rows runs in row orientation
constexpr int kThreads = 192;
constexpr int kEpiWarps = 8;         // epilogue warps per pair (4 per CTA)
constexpr int kABytes = kBM * kBK * 2;
constexpr int kBBytes = kBNh * kBK * 2;
constexpr int kBoxBytes = kBoxB * kBK * 2;
constexpr int kTBytes = kBoxT * kBK * 2;
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kStages = 6;
constexpr int kTmemCols = 512;       // two 256-column accumulators
constexpr int kXposeBytes = 4 * 32 * 32 * 2;   // epilogue transpose blocks, one per warp
constexpr size_t kSmem = 1024 + (size_t)kStages * (kStageBytes + kTBytes) + kXposeBytes;
constexpr uint64_t kWaitNs = 2000000000ull;
// Tile queue: the leader's producer takes tiles from a global counter and
// publishes them here, in both CTAs, for every other role.  No role can be
// more than kStages + 2 tiles behind the producer (its ring and the two
// accumulators hold it back), so 16 entries never overwrite one still unread.
constexpr int kTQ = 16;
// gathered token rows: each lane copies one 16-byte chunk of rows
// lane / 8 + 4 i of the CTA's (at most 128) rows
constexpr int kGatherPer = kBM / 4;
// a gathered stage is signalled once at most this many newer ones are still copying
constexpr int kGatherLag = 4;
static_assert(kGatherLag < kStages, "gathered stages signalled too late");
static_assert(kTQ > kStages + 3, "tile queue shorter than the pipeline");
constexpr int kTqAbort = -2;

// One product of a launch: output columns N, reduction length K, the
// nullable per-expert bias and the output rows C [rows, N].  With acc set
// (the second product only) the rows are not stored: row r, the slot
// s = src[r] of token t = s / topk, adds wts[s] * bf16(y) to acc[t, :] (fp32,
// zeroed beforehand) -- the weighted combine done in the epilogue.
// With gx set (the first product only) the token rows are not read from the
// tensor maps: kept row r is row gsrc[r] / topk of gx [gtok, K], copied by
// the producer warp.
struct PairProduct {
  int N, K;
  const float* bias;
  bf16* C;
  const int32_t* src;
  const float* wts;
  float* acc;
  int topk;
  const bf16* gx;
  const int32_t* gsrc;
  int gtok;
};

// acc[0..7] += w * v[0..7] with two 16-byte vector reductions (addr 32-byte aligned)
__device__ __forceinline__ void red_add8(float* addr, float w, const float* v) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(w * v[0]), "f"(w * v[1]),
               "f"(w * v[2]), "f"(w * v[3])
               : "memory");
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr + 4), "f"(w * v[4]), "f"(w * v[5]),
               "f"(w * v[6]), "f"(w * v[7])
               : "memory");
}

// Wait (bounded) until the counter reaches `need`, with acquire semantics at
// GPU scope; then order those observed writes before this thread's later
// tensor copies (a proxy fence: the copies read global memory through the
// async proxy).  False on timeout or abort.
__device__ __forceinline__ bool wait_count(const int* p, int need, const volatile int* abort) {
  uint64_t t0 = 0;
  for (int i = 0;; ++i) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    if (v >= need) {
      asm volatile("fence.proxy.async.global;" ::: "memory");
      return true;
    }
    if (*abort) return false;
    if ((i & 63) == 63) {
      const uint64_t now = tc::globaltimer();
      if (t0 == 0) t0 = now;
      else if (now - t0 > kWaitNs) return false;
    }
    __nanosleep(64);
  }
}

// An expert of `rows` token rows has a wide tail when its last 256-row block
// holds at most kWideRows rows and runs swapped (ok): that block's tiles then
// cover two n-tiles each, the weight rows of both in one stage (the A and B
// slots) with its few token rows in the stage's T slot, so a stage carries
// 35 KB per CTA instead of 19-22 KB.
__device__ __forceinline__ bool wide_tail(int rows, bool ok) {
  if (!ok || rows <= 0) return false;
  const int mt = (rows + 2 * kBM - 1) / (2 * kBM);
  return rows - (mt - 1) * 2 * kBM <= kWideRows;
}
// The expert's pair tiles in one product of nt n-tiles.
__device__ __forceinline__ int expert_tiles(int rows, int nt, bool ok) {
  const int mt = (rows + 2 * kBM - 1) / (2 * kBM);
  if (!(wide_tail(rows, ok) && nt >= 2)) return mt * nt;
  return (nt / 2) * (2 * (mt - 1) + 1) + (nt % 2) * mt;
}

// One tile's epilogue: this warp's 32 accumulator lanes (TMEM lane quarter
// q) -> bias -> activation -> bf16 -> global.  Swapped tiles hold the
// transposed block (lane = output column, column = token row) and go through
// the warp's 2 KB transpose buffer so stores stay 16-byte vectors along rows.
template <int kEpi>
__device__ __forceinline__ void tile_epilogue(uint32_t tbase, bool swap, int e, int row_base, int nrows, int row_end,
                                              int n0, uint32_t rank, int q, int lane, bf16* xb,
                                              const PairProduct& P) {
  constexpr bool kSwi = kEpi == kEpiSwiglu;
  constexpr int kOut = kSwi ? kBNh : 2 * kBNh;
  const int N = P.N;
  bf16* C = P.C;
  const float* be = P.bias ? P.bias + (int64_t)e * (kSwi ? 2 * N : N) : nullptr;
  if (swap) {
    // lane = output column f, accumulator column j = token row row_base + j
    const int f = n0 + (int)rank * kBM + q * 32 + lane;
    const float bf = (be && f < N) ? be[f] : 0.f;
    const int fv = n0 + (int)rank * kBM + q * 32 + 8 * (lane & 3);   // this lane's 8 stored columns
#pragma unroll 1
    for (int c = 0; c * 32 < nrows; ++c) {
      uint32_t r[32];
      tc::tmem_ld_32x32b_x32(tbase + c * 32, r);
      tc::tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float a = __uint_as_float(r[j]) + bf;
        xb[j * 32 + lane] = __float2bfloat16_rn(kEpi == kEpiGelu ? gelu_erf(a) : a);
      }
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int jj = (lane >> 2) + 8 * i;
        const int row = row_base + c * 32 + jj;
        if (row < row_end && fv < N) {
          const uint4 u = *reinterpret_cast<const uint4*>(xb + jj * 32 + 8 * (lane & 3));
          if (kEpi == kEpiPlain && P.acc) {
            const int sl = P.src[row];
            float v[8];
            Vec<bf16>::unpack(u, v);
            red_add8(P.acc + (int64_t)(sl / P.topk) * N + fv, P.wts[sl], v);
          } else {
            *reinterpret_cast<uint4*>(C + (int64_t)row * N + fv) = u;
          }
        }
      }
      __syncwarp();
    }
  } else {
    const int row = row_base + (int)rank * kBM + q * 32 + lane;
    const bool row_ok = row < row_end;
    // fused combine: this row's token and routing weight
    const bool comb = kEpi == kEpiPlain && P.acc != nullptr;
    const int sl = (comb && row_ok) ? P.src[row] : 0;
    const float wt = (comb && row_ok) ? P.wts[sl] : 0.f;
    float* acc_row = comb ? P.acc + (int64_t)(sl / P.topk) * N : nullptr;
#pragma unroll 1
    for (int c = 0; c < kOut / 32; ++c) {
      const int col0 = n0 + c * 32;
      if (col0 >= N) break;
      uint32_t r[32], u[kSwi ? 32 : 1];
      tc::tmem_ld_32x32b_x32(tbase + c * 32, r);
      if (kSwi) tc::tmem_ld_32x32b_x32(tbase + kOut + c * 32, u);
      tc::tmem_wait_ld();
      if (row_ok) {
        bf16* dst = comb ? nullptr : C + (int64_t)row * N + col0;
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
            const uint4 pk = Vec<bf16>::pack(v);
            if (comb) {
              float y[8];
              Vec<bf16>::unpack(pk, y);                  // y rounded to bf16, as stored
              red_add8(acc_row + col0 + g * 8, wt, y);
            } else {
              *reinterpret_cast<uint4*>(dst + g * 8) = pk;
            }
          }
        }
      }
    }
  }
}

// One launch runs one product, or both (nphase = 2): the tiles of the first
// product (activation kEpiA), then those of the second (plain), from one
// tile queue.  A second-product tile reads the hidden rows of one 256-row
// block, which all first-product tiles of that block write; each epilogue
// warp of such a tile adds 1 to ready[block] once its stores are visible, and
// both producers of a second-product tile wait until ready[block] = 8 x
// (first-product tiles per block).  First-product tiles never wait and every
// one of them is handed out before any second-product tile, so every wait
// ends.  The block index is (offs[e] >> 8) + e + (row block within e), which
// is unique and below rows / 256 + E + 1.
//
// Tensor maps, per product p: tmX = token rows [rows, K] in 128-row boxes
// (row-orientation A), tmXs = the same rows in 32-row boxes (swapped B), tmW
// = weight rows [E N, K] in 128-row boxes (row-orientation B, swapped A),
// tmXt = the token rows in 16-row boxes (wide swapped tiles).
// kEpiA = kEpiSwiglu: tmW0 covers [W1; W3] stacked per expert ([E, 2N, K]);
// the leader loads 128 gate rows and the peer the matching 128 up rows.
// swap_tail = 0 keeps every block in row orientation.
// kGather: the first product's token rows come from P0.gx by P0.gsrc (the
// producer warp copies them), not from tmX0 / tmXs0 / tmXt0.
template <int kEpiA, bool kGather>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmX0, const __grid_constant__ CUtensorMap tmXs0,
                         const __grid_constant__ CUtensorMap tmW0, const __grid_constant__ CUtensorMap tmXt0,
                         const __grid_constant__ CUtensorMap tmX1, const __grid_constant__ CUtensorMap tmXs1,
                         const __grid_constant__ CUtensorMap tmW1, const __grid_constant__ CUtensorMap tmXt1,
                         const int32_t* __restrict__ offs, int E, PairProduct P0, PairProduct P1, int nphase,
                         int swap_tail, int* __restrict__ next_tile, int* __restrict__ ready, int* err) {
  constexpr int S = kStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_offs[257];
  __shared__ int s_tstart[2][257];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ __align__(8) uint64_t s_bar[2 * S + 5];
  __shared__ __align__(8) unsigned long long s_tq[kTQ];   // (sequence + 1) << 32 | tile, tile -1 = end

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sA = tc::smem_u32(smem);
  const uint32_t sB = sA + S * kABytes;
  const uint32_t sT = sB + S * kBBytes;   // wide swapped tiles' token rows, kTBytes a stage
  bf16* xpose = reinterpret_cast<bf16*>(smem + (size_t)S * (kStageBytes + kTBytes));   // [4][32][32]
  auto full = [&](int s) { return tc::smem_u32(&s_bar[s]); };
  auto empty = [&](int s) { return tc::smem_u32(&s_bar[S + s]); };
  auto tfull = [&](int a) { return tc::smem_u32(&s_bar[2 * S + a]); };
  auto tempty = [&](int a) { return tc::smem_u32(&s_bar[2 * S + 2 + a]); };
  const uint32_t done_bar = tc::smem_u32(&s_bar[2 * S + 4]);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = tc::cluster_ctarank();          // 0 = leader
  constexpr bool kSwiA = kEpiA == kEpiSwiglu;
  constexpr int kOutA = kSwiA ? kBNh : 2 * kBNh;   // output columns per pair tile, first product
  constexpr int kOutB = 2 * kBNh;                  // second product
  const int nt0 = (P0.N + kOutA - 1) / kOutA;
  const int nt1 = (P1.N + kOutB - 1) / kOutB;
  const int nk0 = (P0.K + kBK - 1) / kBK;
  const int nk1 = (P1.K + kBK - 1) / kBK;
  // wide tails: swapped blocks only (the SwiGLU first product never swaps)
  auto wide_ok = [&](int p, int st) { return st != 0 && !(p == 0 && kSwiA); };

  if (warp == 0) {
    pdl_enter();   // the tile table reads offs, written by the previous kernel
    // per-expert pair-tile counts (256-row blocks x n-tiles, a wide tail
    // covering two n-tiles) of both products and their prefixes
    int loc0[8], loc1[8];
    int sum0 = 0, sum1 = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      int rows = 0;
      if (e < E) {
        const int o0 = offs[e], o1 = offs[e + 1];
        rows = o1 - o0;
        s_offs[e] = o0;
        if (e == E - 1) s_offs[E] = o1;
      }
      loc0[i] = expert_tiles(rows, nt0, wide_ok(0, swap_tail));
      loc1[i] = nphase > 1 ? expert_tiles(rows, nt1, wide_ok(1, swap_tail)) : 0;
      sum0 += loc0[i];
      sum1 += loc1[i];
    }
    int incl0 = sum0, incl1 = sum1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t0 = __shfl_up_sync(0xffffffffu, incl0, o);
      const int t1 = __shfl_up_sync(0xffffffffu, incl1, o);
      if (lane >= o) {
        incl0 += t0;
        incl1 += t1;
      }
    }
    int run0 = incl0 - sum0, run1 = incl1 - sum1;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      if (e < E) {
        s_tstart[0][e] = run0;
        s_tstart[1][e] = run1;
      }
      run0 += loc0[i];
      run1 += loc1[i];
    }
    if (lane == 31) {
      s_tstart[0][E] = incl0;
      s_tstart[1][E] = incl1;
    }
    if (lane == 0) {
      for (int s = 0; s < S; ++s) {
        // used in the leader: its arm + both CTAs' bytes (+ both producers'
        // arrivals when the first product's token rows are gathered)
        tc::mbar_init(full(s), kGather ? 3 : 1);
        tc::mbar_init(empty(s), 1);      // one multicast commit per use
      }
      for (int a = 0; a < 2; ++a) {
        tc::mbar_init(tfull(a), 1);
        tc::mbar_init(tempty(a), 2 * 128);   // used in the leader: both CTAs' epilogue threads
      }
      tc::mbar_init(done_bar, 1);
      s_abort = 0;
      for (int i = 0; i < kTQ; ++i) s_tq[i] = 0ull;
      tc::fence_barrier_init();
      tc::fence_proxy_async_smem();
      tc::prefetch_tmap(&tmX0);
      tc::prefetch_tmap(&tmXs0);
      tc::prefetch_tmap(&tmW0);
      tc::prefetch_tmap(&tmXt0);
      if (nphase > 1) {
        tc::prefetch_tmap(&tmX1);
        tc::prefetch_tmap(&tmXs1);
        tc::prefetch_tmap(&tmW1);
        tc::prefetch_tmap(&tmXt1);
      }
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
  const int total0 = s_tstart[0][E];
  const int total = total0 + s_tstart[1][E];

  // the leader's producer publishes tile `t` (or -1, the end) as entry `seq`
  auto tq_publish = [&](int seq, int t) {
    const unsigned long long v = ((unsigned long long)(unsigned)(seq + 1) << 32) | (unsigned)t;
    volatile unsigned long long* slot = &s_tq[seq & (kTQ - 1)];
    *slot = v;
    tc::st_peer_u64(tc::map_peer(tc::smem_u32(&s_tq[seq & (kTQ - 1)]), 1), v);
  };
  // entry `seq` of this CTA's queue: a tile, -1 at the end, kTqAbort if the
  // kernel is aborting or the entry did not arrive in time
  auto tq_read = [&](int seq) -> int {
    volatile unsigned long long* slot = &s_tq[seq & (kTQ - 1)];
    const unsigned long long want = (unsigned long long)(unsigned)(seq + 1);
    uint64_t t0 = 0;
    for (int i = 0;; ++i) {
      const unsigned long long v = *slot;
      if ((v >> 32) == want) return (int)(unsigned)(v & 0xffffffffull);
      if (s_abort) return kTqAbort;
      if ((i & 255) == 255) {
        const uint64_t now = tc::globaltimer();
        if (t0 == 0) t0 = now;
        else if (now - t0 > kWaitNs) return kTqAbort;
      }
    }
  };

  // tile t -> product p, expert e, its first token row (the pair's), the
  // rows of that block (<= 256), the MMA N (swapped: rows rounded up to 16;
  // else 256), the first output column and the block's ready counter.  Tiles
  // run product by product, expert by expert, row blocks inner.
  // With a wide tail (at most kWideRows rows) an expert's n-tiles go in
  // pairs: the full blocks of n-tile 2c, those of n-tile 2c + 1, then the
  // one tail tile of both (so both weight slabs are still in L2); an odd
  // last n-tile keeps its own tail.  Otherwise n-tiles outer, row blocks inner.
  struct Tile {
    int p, e, row_base, nrows, row_end, mma_n, n0, block;
    bool swap, wide;
  };
  auto decode = [&](int t) {
    Tile d;
    d.p = t >= total0 ? 1 : 0;
    const int tl = t - (d.p ? total0 : 0);
    const int* ts = s_tstart[d.p];
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (ts[mid] <= tl) lo = mid; else hi = mid - 1;
    }
    d.e = lo;
    const int rows = s_offs[d.e + 1] - s_offs[d.e];
    const int mt = (rows + 2 * kBM - 1) / (2 * kBM);
    const int nt = d.p ? nt1 : nt0;
    const int local = tl - ts[d.e];
    int rb, col;
    d.wide = false;
    if (wide_tail(rows, wide_ok(d.p, swap_tail)) && nt >= 2) {
      const int per = 2 * (mt - 1) + 1;   // tiles of an n-tile pair
      if (local < (nt / 2) * per) {
        const int c2 = local / per, w = local % per;
        if (w < mt - 1) {
          col = 2 * c2;
          rb = w;
        } else if (w < 2 * (mt - 1)) {
          col = 2 * c2 + 1;
          rb = w - (mt - 1);
        } else {
          col = 2 * c2;
          rb = mt - 1;
          d.wide = true;
        }
      } else {
        col = nt - 1;
        rb = local - (nt / 2) * per;
      }
    } else {
      rb = local % mt;
      col = local / mt;
    }
    d.row_base = s_offs[d.e] + rb * (2 * kBM);
    d.row_end = s_offs[d.e + 1];
    d.nrows = min(2 * kBM, d.row_end - d.row_base);
    d.swap = !(d.p == 0 && kSwiA) && swap_tail && d.nrows <= kSwapRows;
    d.mma_n = d.swap ? (d.nrows + 15) / 16 * 16 : 2 * kBNh;
    d.n0 = col * (d.p ? kOutB : kOutA);
    d.block = (s_offs[d.e] >> 8) + d.e + rb;
    return d;
  };

  uint32_t filled = 0, fill_par = 0;   // producer: per stage, ever filled / parity of its last fill
  bool producer = false;
  if (warp == 0) {
    if constexpr (!kGather) {
      // ------------------------------------------------------------ TMA producer (both CTAs)
      if (tc::elect_one()) {
        producer = true;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        int t_next = rank == 0 ? atomicAdd(next_tile, 1) : 0;
        for (int seq = 0; ok; ++seq) {
          int t;
          if (rank == 0) {
            t = t_next < total ? t_next : -1;
            tq_publish(seq, t);
            if (t >= 0) t_next = atomicAdd(next_tile, 1);   // the following tile, fetched while this one loads
          } else {
            t = tq_read(seq);
            if (t == kTqAbort) { ok = false; break; }
          }
          if (t < 0) break;
          const Tile d = decode(t);
          // a second-product tile reads hidden rows that other SMs write
          if (d.p == 1 && !wait_count(ready + d.block, kEpiWarps * nt0, &s_abort)) { ok = false; break; }
          const CUtensorMap* mX = d.p ? &tmX1 : &tmX0;
          const CUtensorMap* mXs = d.p ? &tmXs1 : &tmXs0;
          const CUtensorMap* mW = d.p ? &tmW1 : &tmW0;
          const int N = d.p ? P1.N : P0.N;
          const int nk = d.p ? nk1 : nk0;
          // swapped: this CTA's token rows start half the MMA N into the block
          const int half = d.mma_n / 2;
          const int nbox = (half + kBoxB - 1) / kBoxB;
          const uint32_t tx = d.wide ? 2u * (uint32_t)(kABytes + kBBytes + kTBytes)
                                     : d.swap ? 2u * (uint32_t)(kABytes + nbox * kBoxBytes) : 2u * kStageBytes;
          const CUtensorMap* mXt = d.p ? &tmXt1 : &tmXt0;
          for (int kb = 0; kb < nk; ++kb) {
            if (!tc::mbar_wait(empty(stage), phase ^ 1u, &s_abort, kWaitNs)) { ok = false; break; }
            const uint32_t fbar = tc::map_peer(full(stage), 0);
            if (rank == 0) tc::mbar_arrive_expect_tx(full(stage), tx);
            if (d.wide) {   // A, B = the weight rows of n-tiles n0 and n0 + 256, T = this CTA's token rows
              tc::tma_load_2d_pair(sA + stage * kABytes, mW, fbar, kb * kBK, d.e * N + d.n0 + (int)rank * kBM);
              tc::tma_load_2d_pair(sB + stage * kBBytes, mW, fbar, kb * kBK,
                                   d.e * N + d.n0 + 2 * kBM + (int)rank * kBM);
              tc::tma_load_2d_pair(sT + stage * kTBytes, mXt, fbar, kb * kBK, d.row_base + (int)rank * half);
            } else if (d.swap) {   // A = weight rows, B = this CTA's half of the token rows
              tc::tma_load_2d_pair(sA + stage * kABytes, mW, fbar, kb * kBK, d.e * N + d.n0 + (int)rank * kBM);
              for (int i = 0; i < nbox; ++i)
                tc::tma_load_2d_pair(sB + stage * kBBytes + i * kBoxBytes, mXs, fbar, kb * kBK,
                                     d.row_base + (int)rank * half + i * kBoxB);
            } else {        // A = this CTA's 128 token rows, B = its 128 weight rows
              tc::tma_load_2d_pair(sA + stage * kABytes, mX, fbar, kb * kBK, d.row_base + (int)rank * kBM);
              tc::tma_load_2d_pair(sB + stage * kBBytes, mW, fbar, kb * kBK,
                                   (d.p == 0 && kSwiA) ? 2 * d.e * N + (int)rank * N + d.n0
                                                       : d.e * N + d.n0 + (int)rank * kBNh);
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
    } else {
      // ------------------------------------------------------------ gathering producer (both CTAs)
      // Lane 0 takes the tiles, waits on the ring and issues the TMA copies.
      // The first product's token rows are copied by the whole warp,
      // 16 bytes a lane (8 lanes to a row's 128-byte segment, placed in the
      // 128-byte swizzle the MMA descriptors read); such a stage is signalled
      // on the leader's `full` barrier only once this warp's copies into it
      // have landed and been fenced for the tensor cores.
      producer = lane == 0;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int npend = 0;                              // gathered stages before `stage` not yet signalled
      const int rg = lane >> 3, ch = lane & 7;   // this lane's rows rg + 4 i, 16-byte chunk ch
      auto signal = [&](int st) {                // this CTA's part of stage st is in place
        if (lane == 0) {
          if (rank == 0) tc::mbar_arrive(full(st));
          else tc::mbar_arrive_remote(tc::map_peer(full(st), 0));
        }
      };
      auto settle = [&](int keep) {              // signal all but the `keep` newest gathered stages
        if (npend <= keep) return;
        tc::cp_async_wait_max(keep);
        tc::fence_proxy_async_smem();
        __syncwarp();
        for (; npend > keep; --npend) signal((stage - npend + S) % S);
      };
      int t_next = (rank == 0 && lane == 0) ? atomicAdd(next_tile, 1) : 0;
      for (int seq = 0; ok; ++seq) {
        int t = 0;
        if (lane == 0) {
          if (rank == 0) {
            t = t_next < total ? t_next : -1;
            tq_publish(seq, t);
            if (t >= 0) t_next = atomicAdd(next_tile, 1);   // the following tile, fetched while this one loads
          } else {
            t = tq_read(seq);
          }
        }
        t = __shfl_sync(0xffffffffu, t, 0);
        if (t == kTqAbort) { ok = false; break; }
        if (t < 0) break;
        const Tile d = decode(t);
        const bool gat = d.p == 0;
        // a second-product tile reads hidden rows that other SMs write (and
        // those may wait on stages this warp has not signalled yet)
        if (d.p == 1) {
          settle(0);
          int w = 1;
          if (lane == 0) w = wait_count(ready + d.block, kEpiWarps * nt0, &s_abort) ? 1 : 0;
          if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
        }
        const CUtensorMap* mX = d.p ? &tmX1 : &tmX0;
        const CUtensorMap* mXs = d.p ? &tmXs1 : &tmXs0;
        const CUtensorMap* mW = d.p ? &tmW1 : &tmW0;
        const int N = d.p ? P1.N : P0.N;
        const int nk = d.p ? nk1 : nk0;
        // swapped: this CTA's token rows start half the MMA N into the block
        const int half = d.mma_n / 2;
        const int nbox = (half + kBoxB - 1) / kBoxB;
        uint32_t tx = d.wide ? 2u * (uint32_t)(kABytes + kBBytes + kTBytes)
                             : d.swap ? 2u * (uint32_t)(kABytes + nbox * kBoxBytes) : 2u * kStageBytes;
        const CUtensorMap* mXt = d.p ? &tmXt1 : &tmXt0;
        // gathered: where this lane's rows start in gx (16-byte units), ~0u for
        // a row past the block's end (its accumulator row is never stored)
        uint32_t rv[kGatherPer];
        int nper = 0;
        if (gat) {
          tx = d.wide ? 2u * (uint32_t)(kABytes + kBBytes) : d.swap ? 2u * (uint32_t)kABytes : 2u * (uint32_t)kBBytes;
          const int nload = d.swap ? half : kBM;
          const int first = d.row_base + (int)rank * nload;
          nper = (nload + 3) / 4;
  #pragma unroll
          for (int i = 0; i < kGatherPer; ++i) {
            rv[i] = ~0u;
            const int j = rg + 4 * i, r = first + j;
            if (i < nper && j < nload && r < d.row_end) {
              const int sl = P0.gsrc[r];
              if (sl >= 0 && sl / P0.topk < P0.gtok) rv[i] = (uint32_t)(sl / P0.topk) * (uint32_t)(P0.K / 8);
              else set_error(err, kDevBadIndex);
            }
          }
        }
        for (int kb = 0; kb < nk; ++kb) {
          // the slot's previous contents are consumed: while it is not, the
          // gathered stages still pending are signalled as they land, oldest
          // first; with none pending lane 0 alone waits (the other lanes
          // parked, so the warp takes no issue slots from the epilogue warp
          // beside it)
          {
            int r = 0;
            while (npend > 0) {
              if (lane == 0) r = tc::mbar_test_wait(empty(stage), phase ^ 1u) ? 1 : 0;
              r = __shfl_sync(0xffffffffu, r, 0);
              if (r) break;
              settle(npend - 1);
            }
            if (!r) {
              if (lane == 0) r = tc::mbar_wait(empty(stage), phase ^ 1u, &s_abort, kWaitNs) ? 1 : 2;
              r = __shfl_sync(0xffffffffu, r, 0);
            }
            if (r != 1) { ok = false; break; }
          }
          if (lane == 0) {
            const uint32_t fbar = tc::map_peer(full(stage), 0);
            if (rank == 0) tc::mbar_arrive_expect_tx(full(stage), tx);
            if (d.wide) {   // A, B = the weight rows of n-tiles n0 and n0 + 256, T = this CTA's token rows
              tc::tma_load_2d_pair(sA + stage * kABytes, mW, fbar, kb * kBK, d.e * N + d.n0 + (int)rank * kBM);
              tc::tma_load_2d_pair(sB + stage * kBBytes, mW, fbar, kb * kBK,
                                   d.e * N + d.n0 + 2 * kBM + (int)rank * kBM);
              if (!gat)
                tc::tma_load_2d_pair(sT + stage * kTBytes, mXt, fbar, kb * kBK, d.row_base + (int)rank * half);
            } else if (d.swap) {   // A = weight rows, B = this CTA's half of the token rows
              tc::tma_load_2d_pair(sA + stage * kABytes, mW, fbar, kb * kBK, d.e * N + d.n0 + (int)rank * kBM);
              if (!gat)
                for (int i = 0; i < nbox; ++i)
                  tc::tma_load_2d_pair(sB + stage * kBBytes + i * kBoxBytes, mXs, fbar, kb * kBK,
                                       d.row_base + (int)rank * half + i * kBoxB);
            } else {        // A = this CTA's 128 token rows, B = its 128 weight rows
              if (!gat)
                tc::tma_load_2d_pair(sA + stage * kABytes, mX, fbar, kb * kBK, d.row_base + (int)rank * kBM);
              tc::tma_load_2d_pair(sB + stage * kBBytes, mW, fbar, kb * kBK,
                                   (d.p == 0 && kSwiA) ? 2 * d.e * N + (int)rank * N + d.n0
                                                       : d.e * N + d.n0 + (int)rank * kBNh);
            }
            filled |= 1u << stage;
            fill_par = (fill_par & ~(1u << stage)) | (phase << stage);
          }
          if (gat) {
            // token row j of the stage's token slot: 128 bytes at j * 128, its
            // 16-byte chunk c stored at chunk c ^ (j & 7) (the slots are
            // 1024-byte aligned); columns past K are zero-filled
            const uint32_t dst0 = d.wide ? sT + stage * kTBytes : d.swap ? sB + stage * kBBytes : sA + stage * kABytes;
            const bool in_k = kb * kBK + ch * 8 < P0.K;
            const uint4* xs = reinterpret_cast<const uint4*>(P0.gx);
  #pragma unroll
            for (int i = 0; i < kGatherPer; ++i) {
              if (i < nper && rv[i] != ~0u) {
                const int j = rg + 4 * i;
                tc::cp_async16(dst0 + j * 128 + ((ch ^ (j & 7)) << 4), xs + rv[i] + (in_k ? kb * (kBK / 8) + ch : 0),
                               in_k ? 16u : 0u);
              }
            }
            tc::cp_async_commit();
            ++npend;
          } else {
            signal(stage);
          }
          if (++stage == S) { stage = 0; phase ^= 1u; }
          if (gat) settle(kGatherLag);
        }
      }
      // every copy of this warp has landed, and its stages are signalled, before the CTA goes on
      settle(0);
      if (!ok && lane == 0) {
        set_error(err, kDevTimeout);
        s_abort = 1;
      }
      __syncwarp();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader)
    if (rank == 0 && tc::elect_one()) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int seq = 0; ok; ++seq) {
        const int t = tq_read(seq);
        if (t == kTqAbort) { ok = false; break; }
        if (t < 0) break;
        const Tile dt = decode(t);
        const uint32_t idesc = tc::idesc_bf16_f32(2 * kBM, dt.mma_n);
        const int nk = dt.p ? nk1 : nk0;
        if (!tc::mbar_wait(tempty(acc), acc_phase ^ 1u, &s_abort, kWaitNs)) { ok = false; break; }
        tc::tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(acc * 2 * kBNh);
        for (int kb = 0; kb < nk; ++kb) {
          // gathered stages are completed by both producers' arrivals (cluster acquire)
          if (!(kGather ? tc::mbar_wait<true>(full(stage), phase, &s_abort, kWaitNs)
                        : tc::mbar_wait(full(stage), phase, &s_abort, kWaitNs))) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t a0 = sA + stage * kABytes, b0 = sB + stage * kBBytes;
          if (dt.wide) {
            // two weight groups against the same token rows, into columns 0 and 128
            const uint32_t t0 = sT + stage * kTBytes;
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k) {
              tc::mma_bf16_pair(d, tc::sdesc_k128(a0 + k * 32), tc::sdesc_k128(t0 + k * 32), idesc, (kb | k) != 0);
              tc::mma_bf16_pair(d + kBM, tc::sdesc_k128(b0 + k * 32), tc::sdesc_k128(t0 + k * 32), idesc,
                                (kb | k) != 0);
            }
          } else {
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
              tc::mma_bf16_pair(d, tc::sdesc_k128(a0 + k * 32), tc::sdesc_k128(b0 + k * 32), idesc,
                                (kb | k) != 0);
          }
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
    bf16* xb = xpose + q * 32 * 32;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int seq = 0;; ++seq) {
      const int t = tq_read(seq);
      if (t == kTqAbort) {
        set_error(err, kDevTimeout);
        s_abort = 1;
        break;
      }
      if (t < 0) break;
      const Tile d = decode(t);
      if (!tc::mbar_wait(tfull(acc), acc_phase, &s_abort, kWaitNs)) {
        set_error(err, kDevTimeout);
        s_abort = 1;
        break;
      }
      tc::tc_fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * 2 * kBNh);
      // a wide tile holds n-tile n0 in columns 0.. and n-tile n0 + 256 in columns 128..
      const int groups = d.wide ? 2 : 1;
      if (d.p == 0) {
        for (int g = 0; g < groups; ++g)
          tile_epilogue<kEpiA>(tbase + g * kBM, d.swap, d.e, d.row_base, d.nrows, d.row_end, d.n0 + g * 2 * kBM,
                               rank, q, lane, xb, P0);
        if (nphase > 1) {
          // this warp's stores are visible GPU-wide before the block's counter
          // moves (by one per n-tile written)
          __threadfence();
          __syncwarp();
          if (lane == 0) atomicAdd(ready + d.block, groups);
        }
      } else {
        for (int g = 0; g < groups; ++g)
          tile_epilogue<kEpiPlain>(tbase + g * kBM, d.swap, d.e, d.row_base, d.nrows, d.row_end, d.n0 + g * 2 * kBM,
                                   rank, q, lane, xb, P1);
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

// The four tensor maps of one product: token rows A [rows, K] in 128-, 32-
// and 16-row boxes, weight rows [wrows, K] in 128-row boxes.
bool pair_maps(CUtensorMap* mx, CUtensorMap* mxs, CUtensorMap* mw, CUtensorMap* mxt, const void* A, int64_t rows,
               const void* B, int64_t wrows, int K) {
  return tma_map_bf16(mx, A, (uint64_t)rows, (uint64_t)K, kBM) &&
         tma_map_bf16(mxs, A, (uint64_t)rows, (uint64_t)K, kBoxB) &&
         tma_map_bf16(mw, B, (uint64_t)wrows, (uint64_t)K, kBNh) &&
         tma_map_bf16(mxt, A, (uint64_t)rows, (uint64_t)K, kBoxT);
}

// One persistent launch: one resident pair per two SMs, never more pairs
// than fit at once.
template <int kEpiA, bool kGather = false>
cudaError_t launch_pair(const CUtensorMap (&m)[8], const int32_t* offs, int E, const PairProduct& P0,
                        const PairProduct& P1, int nphase, int swap_tail, int* next_tile, int* ready, int* err,
                        cudaStream_t st) {
  auto kern = grouped_gemm_pair_kernel<kEpiA, kGather>;
  cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
  if (r != cudaSuccess) return r;
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
  return launch_kernel(kern, dim3((unsigned)(2 * pairs)), dim3(kThreads), kSmem, st, 2, m[0], m[1], m[2], m[3], m[4],
                       m[5], m[6], m[7], offs, E, P0, P1, nphase, swap_tail, next_tile, ready, err);
}

}  // namespace

// sched[0], sched[1]: tile counters; sched[2 ..]: the row blocks' ready
// counters (rows / 256 + E + 1 of them), all zero on entry.
cudaError_t launch_ffn_tc_pair(const Shape& s, int64_t max_rows, const void* x_perm, const int32_t* offs,
                               const void* W1, const float* b1, const void* W2, const float* b2,
                               void* h_perm, void* y_perm, int* err, int32_t* sched, cudaStream_t st,
                               const CombineInto* comb, const GatherRows* gather) {
  if (!sched) return cudaErrorInvalidValue;
  if (s.dtype != MOE_BF16 || max_rows <= 0 || max_rows >= ((int64_t)1 << 31)) return cudaErrorNotSupported;
  if ((int64_t)s.E * s.F >= ((int64_t)1 << 31) || (int64_t)s.E * s.H >= ((int64_t)1 << 31))
    return cudaErrorNotSupported;
  const bool swi = (s.flags & MOE_FLAG_SWIGLU) != 0;
  // each expert's last, short row block runs swapped unless all are forced to rows
  const int swap_tail = (s.flags & MOE_FLAG_GEMM_ROWS) ? 0 : 1;
  CUtensorMap m1[4], m2[4];
  if (!pair_maps(&m1[0], &m1[1], &m1[2], &m1[3], x_perm, max_rows, W1, (int64_t)s.E * s.F * (swi ? 2 : 1), s.H) ||
      !pair_maps(&m2[0], &m2[1], &m2[2], &m2[3], h_perm, max_rows, W2, (int64_t)s.E * s.H, s.F))
    return cudaErrorNotSupported;
  if (gather && (!gather->x || !gather->src || s.H % 8 != 0 || s.T >= ((int64_t)1 << 31) ||
                 s.T * (s.H / 8) >= ((int64_t)1 << 32)))
    return cudaErrorNotSupported;
  const PairProduct P1{s.F, s.H, b1, (bf16*)h_perm, nullptr, nullptr, nullptr, s.K,
                       gather ? (const bf16*)gather->x : nullptr, gather ? gather->src : nullptr, (int)s.T};
  const PairProduct P2{s.H, s.F, b2, (bf16*)y_perm, comb ? comb->src : nullptr, comb ? comb->w : nullptr,
                       comb ? comb->acc : nullptr, s.K};
  if (!(s.flags & MOE_FLAG_FFN_SPLIT)) {
    // both products in one launch: the second's tiles start on row blocks the first has finished
    const CUtensorMap m[8] = {m1[0], m1[1], m1[2], m1[3], m2[0], m2[1], m2[2], m2[3]};
    cudaError_t r =
        gather ? (swi ? launch_pair<kEpiSwiglu, true>(m, offs, s.E, P1, P2, 2, swap_tail, sched, sched + 2, err, st)
                      : launch_pair<kEpiGelu, true>(m, offs, s.E, P1, P2, 2, swap_tail, sched, sched + 2, err, st))
               : (swi ? launch_pair<kEpiSwiglu>(m, offs, s.E, P1, P2, 2, swap_tail, sched, sched + 2, err, st)
                      : launch_pair<kEpiGelu>(m, offs, s.E, P1, P2, 2, swap_tail, sched, sched + 2, err, st));
    if (r != cudaSuccess) return r;
    prof_mark(kMarkFirst, st);
    return cudaSuccess;
  }
  const CUtensorMap ma[8] = {m1[0], m1[1], m1[2], m1[3], m1[0], m1[1], m1[2], m1[3]};
  cudaError_t r =
      gather ? (swi ? launch_pair<kEpiSwiglu, true>(ma, offs, s.E, P1, P1, 1, swap_tail, sched, nullptr, err, st)
                    : launch_pair<kEpiGelu, true>(ma, offs, s.E, P1, P1, 1, swap_tail, sched, nullptr, err, st))
             : (swi ? launch_pair<kEpiSwiglu>(ma, offs, s.E, P1, P1, 1, swap_tail, sched, nullptr, err, st)
                    : launch_pair<kEpiGelu>(ma, offs, s.E, P1, P1, 1, swap_tail, sched, nullptr, err, st));
  if (r != cudaSuccess) return r;
  prof_mark(kMarkFirst, st);
  const CUtensorMap mb[8] = {m2[0], m2[1], m2[2], m2[3], m2[0], m2[1], m2[2], m2[3]};
  return launch_pair<kEpiPlain>(mb, offs, s.E, P2, P2, 1, swap_tail, sched + 1, nullptr, err, st);
}

}  // namespace moe
