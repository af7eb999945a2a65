// Host-side launchers shared between the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Device error word (first error wins); lives at offset 0 of the workspace.
enum DevErr : int { kDevOk = 0, kDevTimeout = 1, kDevBadIndex = 2 };

struct Shape {
  int64_t T;
  int H, E, K, F, C;   // C <= 0: no capacity limit
  int dtype;           // MOE_F32 | MOE_BF16
  uint32_t flags;
  float inv_tau;       // 1 / router softmax temperature
  int64_t S() const { return T * (int64_t)K; }
  size_t esize() const { return dtype == MOE_BF16 ? 2 : 4; }
};

// The kernels' view of a validated layer description (temperature -> 1/tau).
Shape shape_of(const moe_desc& d);

// Number of SMs of the current device (cached per device).
int sm_count();

// Launch with programmatic dependent launch allowed (the kernel waits for its
// predecessor itself, see pdl_enter) and an optional cluster size.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                 unsigned cluster, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Stage-boundary events of moe_layer_forward (set by moe_profile_events; no-op
// when unset).  Marks: 0 start, 1 router, 2 dispatch, 3 first product,
// 4 second product, 5 combine.
enum ProfMark { kMarkStart = 0, kMarkRouter, kMarkDispatch, kMarkFirst, kMarkSecond, kMarkCombine, kMarks };
void prof_mark(int mark, cudaStream_t st);

// Row-major bf16 matrix [rows, cols] as a 2D TMA tensor map with a box of
// 64 columns (128 bytes, 128-byte swizzle) x box_rows rows; false on failure.
bool tma_map_bf16(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows);

// ---------------------------------------------------------------- router
// Upper bound of the rows of per-block probability partial sums the router
// writes (workspace sizing), and the rows the chosen router writes.
int64_t router_partials(const Shape& s);
bool router_small(const Shape& s);   // one-cluster router for decode-sized bf16 batches
int64_t router_partial_rows(const Shape& s);
bool router_on_tensor_cores(const Shape& s);
int router_tc_split(const Shape& s);   // CTAs the tensor-core router splits the hidden dimension over (1 or 2)
// tile_hist (nullable): [ceil(T/128), E] count of each 128-token tile's
// chosen experts, in slot order blocks of 128*K slots.
cudaError_t launch_router_tc(const Shape& s, const void* x, const void* Wg, const float* gate_bias,
                             float* logits, int32_t* ids, float* w, float* psum_part,
                             int32_t* tile_hist, int* err, cudaStream_t st);
constexpr int kRouterTileTokens = 128;
cudaError_t launch_router(const Shape& s, const void* x, const void* Wg, const float* gate_bias,
                          float* logits, int32_t* ids, float* w, float* psum_part, int* err,
                          cudaStream_t st, int32_t* tile_hist = nullptr);
// psum[e] = sum over partial rows in order.
cudaError_t launch_psum_reduce(const Shape& s, const float* psum_part, float* psum, cudaStream_t st);

// ---------------------------------------------------------------- dispatch
int64_t dispatch_blocks(const Shape& s);
int dispatch_block_slots(const Shape& s);
bool dispatch_small(const Shape& s);
int dispatch_launches(const Shape& s, bool hist_ready);   // kernels launch_dispatch issues (S > 0)   // one-block dispatch (launch_dispatch picks it itself)
struct DispatchOut {
  int32_t* count;      // [E]
  int32_t* offs;       // [E+1]
  int32_t* src;        // [rows]
  int32_t* pos;        // [S]
  int32_t* dropped;    // [1] or null
  int32_t* blk_hist;   // [nblk * E] scratch
  int32_t* blk_base;   // [nblk * E] scratch
  // optional extras folded into the scan kernel
  const float* psum_part;  // partial rows or null
  bool hist_ready;         // blk_hist already holds the router's per-tile counts
  float* psum;             // [E] or null
  float* aux;              // [1] or null (needs psum_part)
  int32_t* count_copy;     // [E] or null
  int32_t* dropped_copy;   // [1] or null
  int32_t* sched;          // [sched_words] the expert GEMMs' counters, zeroed here, or null
};
cudaError_t launch_dispatch(const Shape& s, const int32_t* ids, const void* x, void* x_perm,
                            const DispatchOut& o, int* err, cudaStream_t st);

// drop_tokens=False: fin [S] = each slot's expert after the over-capacity
// slots (pos < 0 in the capacity-limited dispatch with row offsets offs) have
// moved to their token's next-best expert with room, or -1; scores [T, E] are
// the router's; pend, choice: [S] and alts: [T, E] scratch.  dropped
// (nullable): slots left without an expert.  Two launches.
cudaError_t launch_reroute(const Shape& s, const float* scores, const int32_t* ids, const int32_t* pos,
                           const int32_t* offs, int32_t* fin, int32_t* pend, int32_t* choice, uint8_t* alts,
                           int32_t* dropped, int32_t* dropped_copy, cudaStream_t st);

// ---------------------------------------------------------------- expert FFN
// The SM-pair expert GEMMs' counters: two tile counters, then one ready
// counter per 256-row block of the kept rows (at most rows / 256 + E + 1).
inline int64_t sched_words(int64_t rows, int E) { return 2 + rows / 256 + E + 1; }
// Decode-sized batches that run the weight-streaming kernels, and those of
// them that run both products in one launch (its per-expert counters are
// sched[2 .. 2 + E)).
bool stream_ffn_eligible(const Shape& s);
bool stream_fused(const Shape& s);
// The weighted combine folded into the second product's epilogue (K <= 2,
// SM-pair kernels): row r adds w[src[r]] * y to acc[src[r] / K] (fp32,
// zeroed beforehand) instead of storing y.
struct CombineInto {
  const int32_t* src;
  const float* w;
  float* acc;
};
bool combine_fusable(const Shape& s, int64_t max_rows);
// The first product's token rows read from x by the slot list (kept row r:
// x row src[r] / K) instead of from x_perm (SM-pair kernels only).
struct GatherRows {
  const void* x;
  const int32_t* src;
};
// sched: sched_words(max_rows, E) zeroed ints (the SM-pair kernel's counters)
cudaError_t launch_ffn(const Shape& s, int64_t max_rows, const void* x_perm, const int32_t* offs,
                       const void* W1, const float* b1, const void* W2, const float* b2,
                       void* h_perm, void* y_perm, int* err, int32_t* sched, cudaStream_t st,
                       const CombineInto* comb = nullptr, const GatherRows* gather = nullptr);

// ---------------------------------------------------------------- one-launch decode layer
// bf16 batches of at most 16 tokens whose rows, score table and weight ring
// fit one CTA's shared memory, unless the flags ask for the separate steps.
bool decode_layer_eligible(const Shape& s);
// workspace: [pieces][T][E] fp32 partial gate scores, and the counters
size_t decode_part_floats(const Shape& s);
int decode_ctr_words(const Shape& s);
struct DecodeIO {
  const void* x;
  const void* Wg;
  const float* gate_bias;
  const void* W1;
  const float* b1;
  const void* W2;
  const float* b2;
  void* out;
  float* part;
  int* ctr;
  void* h;      // [kept rows, F]
  void* y;      // [kept rows, H]
  int32_t* count;
  int32_t* count_copy;
  int32_t* dropped;
  int32_t* dropped_copy;
  float* psum;
  float* aux;
  int* err;
};
// Two launches: the counters zeroed, then the layer.
cudaError_t launch_decode_layer(const Shape& s, const DecodeIO& io, cudaStream_t st);

// ---------------------------------------------------------------- combine / aux
cudaError_t launch_combine(const Shape& s, const void* y_perm, const int32_t* pos, const float* w,
                           void* out, cudaStream_t st);
cudaError_t launch_aux(const Shape& s, const float* psum, const int32_t* count, float* loss,
                       cudaStream_t st);
// acc [T, H] fp32 = 0, and out [T, H] = bf16(acc) (the fused combine's two ends)
cudaError_t launch_zero_acc(const Shape& s, float* acc, cudaStream_t st);
cudaError_t launch_acc_to_out(const Shape& s, const float* acc, void* out, cudaStream_t st);
// The statistics of a layer run in pieces of tokens: count[e] and psum[e]
// summed over the n pieces in order, then the loss of the whole batch (s.T
// tokens); count_copy, aux and dropped (0: no capacity) are nullable.
cudaError_t launch_merge_stats(const Shape& s, const int32_t* count_parts, const float* psum_parts, int n,
                               int32_t* count, float* psum, int32_t* count_copy, float* aux, int32_t* dropped,
                               cudaStream_t st);

}  // namespace moe
