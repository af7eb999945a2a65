// C ABI of the MoE layer library: argument checks, workspace layout and the
// order of launches.  All device work is in the other translation units.
#include <stdint.h>
#include <string.h>

#include <cudaTypedefs.h>

#include "../../include/moe.h"
#include "internal.h"

namespace moe {

bool stream_ffn_eligible(const Shape& s);
cudaError_t launch_ffn_simt(const Shape& s, int64_t max_rows, const void* x_perm, const int32_t* offs,
                            const void* W1, const float* b1, const void* W2, const float* b2,
                            void* h_perm, void* y_perm, cudaStream_t st);
cudaError_t launch_ffn_stream(const Shape& s, const void* x_perm, const int32_t* offs, const void* W1,
                              const float* b1, const void* W2, const float* b2, void* h_perm,
                              void* y_perm, int* err, int32_t* sched, cudaStream_t st);
bool stream_fused(const Shape& s);
// Tensor-core paths; return cudaErrorNotSupported when they do not apply.
cudaError_t launch_ffn_tc(const Shape& s, int64_t max_rows, const void* x_perm, const int32_t* offs,
                          const void* W1, const float* b1, const void* W2, const float* b2,
                          void* h_perm, void* y_perm, int* err, cudaStream_t st);
cudaError_t launch_ffn_tc_pair(const Shape& s, int64_t max_rows, const void* x_perm, const int32_t* offs,
                               const void* W1, const float* b1, const void* W2, const float* b2,
                               void* h_perm, void* y_perm, int* err, int32_t* sched, cudaStream_t st,
                               const CombineInto* comb, const GatherRows* gather);

// SM-pair tiles move a third less data per SM for the same MMA work.  The
// single-SM kernel pads each expert's rows to 128; the pair kernel runs its
// GELU and plain products with the token rows on the MMA's N side, padded to
// 16 (8 rows per expert on average), and the SwiGLU first product with rows
// padded to 256.  Both pad the output columns to their tile width.
// Estimated cost of each: padded tile area over its relative load
// efficiency.
bool use_pair_gemm(const Shape& s, int64_t rows) {
  if (s.flags & MOE_FLAG_GEMM_PAIR) return true;
  if (s.flags & MOE_FLAG_GEMM_SINGLE) return false;
  const double r = (double)rows;
  auto pad = [](int n, int t) { return (double)((n + t - 1) / t * t); };
  const double single = (r + 64.0 * s.E) * (pad(s.F, 128) + pad(s.H, 128));
  const bool m_rows = (s.flags & MOE_FLAG_GEMM_ROWS) != 0;   // token rows on the MMA's M side
  const double first = (r + ((s.flags & MOE_FLAG_SWIGLU) || m_rows ? 128.0 : 8.0) * s.E) * pad(s.F, 256);
  const double paired = (first + (r + (m_rows ? 128.0 : 8.0) * s.E) * pad(s.H, 256)) / 1.5;
  return paired < single;
}

namespace {
thread_local cudaEvent_t g_prof[kMarks];
thread_local bool g_prof_on = false;
}  // namespace

void prof_mark(int mark, cudaStream_t st) {
  if (g_prof_on && mark >= 0 && mark < kMarks) cudaEventRecord(g_prof[mark], st);
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}
}  // namespace

bool tma_map_bf16(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

// The kernel launch_ffn runs (MOE_FFN_*); the same tests in the same order.
int ffn_kernel(const Shape& s, int64_t max_rows) {
  if (stream_ffn_eligible(s)) return stream_fused(s) ? MOE_FFN_STREAM : MOE_FFN_STREAM_SPLIT;
  if (s.dtype == MOE_BF16 && !(s.flags & MOE_FLAG_SIMT_FFN)) {
    if (use_pair_gemm(s, max_rows)) return (s.flags & MOE_FLAG_FFN_SPLIT) ? MOE_FFN_TC_PAIRS : MOE_FFN_TC_FUSED;
    return MOE_FFN_TC_SINGLE;
  }
  return MOE_FFN_SIMT;
}

// The combine runs in the second product's epilogue when asked for, with
// at most two slots per token (two fp32 additions onto zero give the same
// sum in either order, so the result does not depend on which tile comes
// first) and on the SM-pair kernels.
bool combine_fusable(const Shape& s, int64_t max_rows) {
  if (!(s.flags & MOE_FLAG_FUSED_COMBINE) || s.K > 2 || s.T == 0) return false;
  const int k = ffn_kernel(s, max_rows);
  return k == MOE_FFN_TC_FUSED || k == MOE_FFN_TC_PAIRS;
}

cudaError_t launch_ffn(const Shape& s, int64_t max_rows, const void* x_perm, const int32_t* offs,
                       const void* W1, const float* b1, const void* W2, const float* b2,
                       void* h_perm, void* y_perm, int* err, int32_t* sched, cudaStream_t st,
                       const CombineInto* comb, const GatherRows* gather) {
  if (s.T == 0 || max_rows == 0) return cudaSuccess;
  if (gather && !(s.dtype == MOE_BF16 && !(s.flags & MOE_FLAG_SIMT_FFN) && !stream_ffn_eligible(s) &&
                  use_pair_gemm(s, max_rows)))
    return cudaErrorNotSupported;
  if (stream_ffn_eligible(s))
    return launch_ffn_stream(s, x_perm, offs, W1, b1, W2, b2, h_perm, y_perm, err, sched, st);
  // bf16 runs on the tensor cores; there is no silent fallback (an
  // unsupported shape or a missing tensor-map entry point is an error)
  if (s.dtype == MOE_BF16 && !(s.flags & MOE_FLAG_SIMT_FFN)) {
    if (use_pair_gemm(s, max_rows))
      return launch_ffn_tc_pair(s, max_rows, x_perm, offs, W1, b1, W2, b2, h_perm, y_perm, err, sched, st, comb,
                                gather);
    return launch_ffn_tc(s, max_rows, x_perm, offs, W1, b1, W2, b2, h_perm, y_perm, err, st);
  }
  return launch_ffn_simt(s, max_rows, x_perm, offs, W1, b1, W2, b2, h_perm, y_perm, st);
}

Shape shape_of(const moe_desc& d) {
  Shape s;
  s.T = d.T; s.H = d.H; s.E = d.E; s.K = d.K; s.F = d.F;
  s.C = d.capacity > 0 ? d.capacity : 0;
  s.dtype = d.dtype; s.flags = d.flags;
  s.inv_tau = d.temperature > 0.f ? 1.f / d.temperature : 1.f;
  return s;
}

namespace {

struct Layout {
  size_t err, sched, ids, w, psum_part, psum, blk_hist, blk_base, count, offs, dropped, aux, src, pos;
  size_t pend, choice, alts, scores, fin, count_chunks, psum_chunks, acc, dec_part, dec_ctr;
  size_t x_perm, h_perm, x_stage, out_stage, total;
  int64_t rows;
};

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int64_t rows_for(const moe_desc& d) {
  const int64_t S = d.T * (int64_t)d.K;
  if (d.capacity > 0) {
    const int64_t c = (int64_t)d.E * d.capacity;
    return c < S ? c : S;
  }
  return S;
}

int check_desc(const moe_desc* d) {
  if (!d) return MOE_ERR_INVALID;
  if (d->T < 0 || d->K < 1 || d->K > 8 || d->E < d->K || d->E > 256) return MOE_ERR_INVALID;
  if (d->H < 8 || d->H % 8 || d->F < 8 || d->F % 8) return MOE_ERR_INVALID;
  if (d->dtype != MOE_F32 && d->dtype != MOE_BF16) return MOE_ERR_INVALID;
  if (d->T * (int64_t)d->K >= ((int64_t)1 << 31)) return MOE_ERR_INVALID;
  if (d->T > 0 && (int64_t)d->H * d->T >= ((int64_t)1 << 40)) return MOE_ERR_INVALID;
  if (!(d->temperature == d->temperature) || d->temperature > 3.0e38f || d->temperature < -3.0e38f)
    return MOE_ERR_INVALID;   // NaN or infinite
  return MOE_OK;
}

Layout layout_of(const moe_desc& d) {
  const Shape s = shape_of(d);
  Layout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) / 256 * 256;
    return o;
  };
  const size_t S = (size_t)s.S(), E = (size_t)s.E, es = s.esize();
  L.rows = rows_for(d);
  L.err = take(256);            // error word
  L.sched = take((size_t)sched_words(L.rows, s.E) * 4);   // the GEMMs' tile and row-block counters
  L.ids = take(S * 4);
  L.w = take(S * 4);
  L.psum_part = take((size_t)router_partials(s) * E * 4);
  L.psum = take(E * 4);
  // per-block dispatch tables: the standalone blocking or the router's 128-token tiles
  const int64_t tiles = (s.T + kRouterTileTokens - 1) / kRouterTileTokens;
  const int64_t nblk = dispatch_blocks(s) > tiles ? dispatch_blocks(s) : tiles;
  L.blk_hist = take((size_t)nblk * E * 4);
  L.blk_base = take((size_t)nblk * E * 4);
  L.count = take(E * 4);
  L.offs = take((E + 1) * 4);
  L.dropped = take(4);
  L.aux = take(4);
  L.src = take((size_t)L.rows * 4);
  L.pos = take(S * 4);
  L.pend = take(S * 4);          // moving over-capacity slots (drop_tokens=False)
  L.choice = take(S * 4);
  L.alts = take((size_t)s.T * E);
  L.scores = L.fin = 0;
  if (d.flags & MOE_FLAG_REROUTE) {
    L.scores = take((size_t)s.T * E * 4);
    L.fin = take(S * 4);
  }
  L.x_perm = take((size_t)L.rows * s.H * es);   // also holds y_perm in the layer call
  L.h_perm = take((size_t)L.rows * s.F * es);
  L.acc = 0;
  if (d.flags & MOE_FLAG_FUSED_COMBINE) L.acc = take((size_t)s.T * s.H * 4);   // fp32 combine target
  L.dec_part = L.dec_ctr = 0;
  if (s.T >= 1 && s.T <= 16) {           // the one-launch decode layer's score pieces and counters
    L.dec_part = take(decode_part_floats(s) * 4);
    L.dec_ctr = take((size_t)decode_ctr_words(s) * 4);
  }
  L.count_chunks = take(2 * E * 4);   // per-piece counts and sums of the chunked host-I/O path
  L.psum_chunks = take(2 * E * 4);
  L.x_stage = L.out_stage = 0;
  if (d.flags & MOE_FLAG_HOST_IO) {
    L.x_stage = take((size_t)s.T * s.H * es);
    L.out_stage = take((size_t)s.T * s.H * es);
  }
  L.total = off;
  return L;
}

int check_ws(const moe_desc& d, const void* ws, size_t ws_bytes) {
  if (!ws || ((uintptr_t)ws & 255u)) return MOE_ERR_WORKSPACE;
  if (ws_bytes < layout_of(d).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

template <typename P> P* at(void* ws, size_t off) { return reinterpret_cast<P*>((char*)ws + off); }

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  return e == cudaErrorNotSupported ? MOE_ERR_UNSUPPORTED : MOE_ERR_CUDA;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID: return "MOE_ERR_INVALID: bad argument (null pointer, shape or alignment)";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: layer not implemented by this library";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call failed";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT: a kernel gave up a bounded wait";
    case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE: a kernel index check fired";
    default: return "unknown moe status";
  }
}

int64_t moe_capacity_default(int64_t T, int32_t E, int32_t K) {
  if (E <= 0 || K <= 0 || T < 0) return -1;
  return (T + E - 1) / E * K;
}

int64_t moe_max_rows(const moe_desc* desc) {
  if (check_desc(desc) != MOE_OK) return -1;
  return rows_for(*desc);
}

int moe_workspace_size(const moe_desc* desc, size_t* bytes) {
  if (check_desc(desc) != MOE_OK || !bytes) return MOE_ERR_INVALID;
  *bytes = layout_of(*desc).total;
  return MOE_OK;
}

int moe_router_topk(const moe_desc* desc, const void* x, const void* Wg, const float* gate_bias,
                    float* logits, int32_t* ids, float* w, float* psum, void* ws, size_t ws_bytes,
                    void* stream) {
  int rc = check_desc(desc);
  if (rc) return rc;
  const moe_desc& d = *desc;
  if ((rc = check_ws(d, ws, ws_bytes))) return rc;
  if (d.T > 0 && (!x || !Wg || !ids || !w)) return MOE_ERR_INVALID;
  if ((x && !aligned16(x)) || (Wg && !aligned16(Wg))) return MOE_ERR_INVALID;
  const Layout L = layout_of(d);
  const Shape s = shape_of(d);
  cudaStream_t st = (cudaStream_t)stream;
  float* part = psum ? at<float>(ws, L.psum_part) : nullptr;
  cudaError_t e = launch_router(s, x, Wg, gate_bias, logits, ids, w, part, at<int>(ws, L.err), st);
  if (e == cudaSuccess && psum) e = launch_psum_reduce(s, part, psum, st);
  return cuda_status(e);
}

int moe_dispatch(const moe_desc* desc, const int32_t* ids, const void* x, int32_t* count, int32_t* offs,
                 int32_t* src, int32_t* pos, void* x_perm, int32_t* dropped, void* ws, size_t ws_bytes,
                 void* stream) {
  int rc = check_desc(desc);
  if (rc) return rc;
  const moe_desc& d = *desc;
  if ((rc = check_ws(d, ws, ws_bytes))) return rc;
  if (!count || !offs || (d.T > 0 && (!ids || !src || !pos))) return MOE_ERR_INVALID;
  if (x && (!x_perm || !aligned16(x) || !aligned16(x_perm))) return MOE_ERR_INVALID;
  const Layout L = layout_of(d);
  const Shape s = shape_of(d);
  DispatchOut o;
  memset(&o, 0, sizeof(o));
  o.count = count; o.offs = offs; o.src = src; o.pos = pos; o.dropped = dropped;
  o.blk_hist = at<int32_t>(ws, L.blk_hist);
  o.blk_base = at<int32_t>(ws, L.blk_base);
  return cuda_status(launch_dispatch(s, ids, x, x_perm, o, at<int>(ws, L.err), (cudaStream_t)stream));
}

int moe_reroute(const moe_desc* desc, const float* logits, const int32_t* ids, const int32_t* pos,
                const int32_t* offs, int32_t* ids_out, int32_t* dropped, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_desc(desc);
  if (rc) return rc;
  const moe_desc& d = *desc;
  if ((rc = check_ws(d, ws, ws_bytes))) return rc;
  if (d.T > 0 && (!logits || !ids || !pos || !offs || !ids_out)) return MOE_ERR_INVALID;
  const Layout L = layout_of(d);
  return cuda_status(launch_reroute(shape_of(d), logits, ids, pos, offs, ids_out, at<int32_t>(ws, L.pend),
                                    at<int32_t>(ws, L.choice), at<uint8_t>(ws, L.alts), dropped, nullptr,
                                    (cudaStream_t)stream));
}

int moe_expert_ffn(const moe_desc* desc, const void* x_perm, const int32_t* offs, const void* W1,
                   const float* b1, const void* W2, const float* b2, void* h_perm, void* y_perm,
                   void* ws, size_t ws_bytes, void* stream) {
  int rc = check_desc(desc);
  if (rc) return rc;
  const moe_desc& d = *desc;
  if ((rc = check_ws(d, ws, ws_bytes))) return rc;
  if (!x_perm || !offs || !W1 || !W2 || !h_perm || !y_perm) return MOE_ERR_INVALID;
  if (!aligned16(x_perm) || !aligned16(W1) || !aligned16(W2) || !aligned16(h_perm) || !aligned16(y_perm))
    return MOE_ERR_INVALID;
  const Layout L = layout_of(d);
  const Shape s = shape_of(d);
  cudaStream_t st = (cudaStream_t)stream;
  int32_t* sched = at<int32_t>(ws, L.sched);
  // no dispatch kernel zeroed them
  cudaError_t e = cudaMemsetAsync(sched, 0, (size_t)sched_words(L.rows, s.E) * sizeof(int32_t), st);
  if (e == cudaSuccess)
    e = launch_ffn(s, L.rows, x_perm, offs, W1, b1, W2, b2, h_perm, y_perm, at<int>(ws, L.err), sched, st);
  return cuda_status(e);
}

int moe_combine(const moe_desc* desc, const void* y_perm, const int32_t* pos, const float* w, void* out,
                void* stream) {
  int rc = check_desc(desc);
  if (rc) return rc;
  const moe_desc& d = *desc;
  if (d.T > 0 && (!y_perm || !pos || !w || !out)) return MOE_ERR_INVALID;
  if (d.T > 0 && (!aligned16(y_perm) || !aligned16(out))) return MOE_ERR_INVALID;
  return cuda_status(launch_combine(shape_of(d), y_perm, pos, w, out, (cudaStream_t)stream));
}

int moe_aux_loss(const moe_desc* desc, const float* psum, const int32_t* count, float* loss,
                 void* stream) {
  int rc = check_desc(desc);
  if (rc) return rc;
  if (!psum || !count || !loss) return MOE_ERR_INVALID;
  return cuda_status(launch_aux(shape_of(*desc), psum, count, loss, (cudaStream_t)stream));
}

namespace moe {
// In the layer call the router counts its 128-token tiles' chosen experts
// (the dispatch histogram) when the multi-block dispatch will read them.
bool layer_fused_hist(const Shape& s) { return router_on_tensor_cores(s) && !dispatch_small(s); }
// drop_tokens=False in the layer call: a capacity-limited dispatch without
// the gather, the move of the over-capacity slots, then a dispatch of the
// moved routing (no capacity cut: no expert is over any more).
bool layer_reroutes(const Shape& s) { return (s.flags & MOE_FLAG_REROUTE) && s.C > 0 && s.T > 0; }
// The first product gathers its token rows from x when asked for, on the
// SM-pair kernels, except where the over-capacity slots are moved (that
// path dispatches twice).
bool layer_gathers(const Shape& s, int64_t max_rows) {
  if (!(s.flags & MOE_FLAG_GATHER_GEMM) || s.T == 0 || layer_reroutes(s)) return false;
  const int k = ffn_kernel(s, max_rows);
  return k == MOE_FFN_TC_FUSED || k == MOE_FFN_TC_PAIRS;
}
Shape final_shape(const Shape& s) {
  Shape f = s;
  f.C = 0;
  return f;
}
// Host-I/O layers without a capacity are split into kIoChunks pieces of
// tokens: a token's output depends only on its own row then, so the pieces
// give the same outputs, and the copy of one piece overlaps the layer on
// another.  Every piece reads all the expert weights again, so the pieces
// stay few.
constexpr int kIoChunks = 2;
// The last piece's combine runs as this many launches, so that the copy of
// each part of its output overlaps the combine of the next.
constexpr int kLastParts = 2;
constexpr int64_t kIoMinChunkTokens = 1024;

bool io_chunked(const Shape& s) {
  return (s.flags & MOE_FLAG_HOST_IO) && s.C <= 0 && s.T >= kIoChunks * kIoMinChunkTokens;
}
int64_t io_chunk_begin(const Shape& s, int c) { return s.T * c / kIoChunks; }
}  // namespace moe

int moe_layer_launches(const moe_desc* desc) {
  int rc = check_desc(desc);
  if (rc) return rc;
  const Shape s = shape_of(*desc);
  if (s.T > 0 && decode_layer_eligible(s)) return 2;   // counters zeroed, the one-launch layer
  int n = 0;
  if (s.T > 0) n += 1;                                  // router
  n += dispatch_launches(s, layer_fused_hist(s));       // one block, or (histogram,) scan, scatter, gather
  if (s.T > 0 && combine_fusable(s, rows_for(*desc))) n += 1;   // zeroing the fp32 combine target
  if (layer_gathers(s, rows_for(*desc)) && !dispatch_small(s)) n -= 1;   // the first product gathers
  if (layer_reroutes(s)) {
    if (!dispatch_small(s)) n -= 1;                     // the first dispatch gathers nothing
    n += 2 + dispatch_launches(final_shape(s), false);  // the move (2), then the dispatch of the moved routing
  }
  if (s.T > 0 && io_chunked(s)) {                       // two pieces of tokens, then the statistics
    n = 1;
    for (int c = 0; c < kIoChunks; ++c) {
      moe_desc dc = *desc;
      dc.T = io_chunk_begin(s, c + 1) - io_chunk_begin(s, c);
      dc.flags &= ~MOE_FLAG_HOST_IO;
      n += moe_layer_launches(&dc);
      // the last piece's combine as kLastParts launches
      if (c == kIoChunks - 1 && !combine_fusable(shape_of(dc), rows_for(dc))) n += kLastParts - 1;
    }
    return n;
  }
  if (s.T > 0) {                                        // expert FFN, combine
    const int k = ffn_kernel(s, rows_for(*desc));
    n += (k == MOE_FFN_TC_FUSED || k == MOE_FFN_STREAM ? 1 : 2) + 1;
  }
  return n;
}

int moe_layer_decode_fused(const moe_desc* desc) {
  int rc = check_desc(desc);
  if (rc) return rc;
  const Shape s = shape_of(*desc);
  return s.T > 0 && decode_layer_eligible(s) ? 1 : 0;
}

int moe_ffn_kernel(const moe_desc* desc) {
  int rc = check_desc(desc);
  if (rc) return rc;
  return ffn_kernel(shape_of(*desc), rows_for(*desc));
}

namespace moe {
namespace {

// Where one pass of the layer puts its statistics.
struct LayerStats {
  int32_t* count;         // [E] routing counts (workspace)
  float* psum;            // [E] probability sums (workspace)
  float* aux;             // [1] loss, or null
  int32_t* count_copy;    // [E] caller's count, or null
  int32_t* dropped_copy;  // [1] caller's dropped, or null
};

// The combine of a layer pass run as `parts` launches over consecutive
// ranges of its tokens, each followed by its event (so a copy of that range
// of out can start while the rest is combined).  Same outputs: a token's
// output depends on its own slots only.
struct CombineParts {
  int parts;
  cudaEvent_t* done;
};

// The layer on device buffers xd -> outd (T = s.T tokens), on stream st.
cudaError_t run_layer(const Shape& s, int64_t rows, const Layout& L, void* ws, const void* xd, const void* Wg,
                      const float* gate_bias, const void* W1, const float* b1, const void* W2, const float* b2,
                      void* outd, const LayerStats& ls, bool marks, cudaStream_t st,
                      const CombineParts* cparts = nullptr) {
  int* err = at<int>(ws, L.err);
  if (decode_layer_eligible(s)) {
    DecodeIO io;
    io.x = xd;
    io.Wg = Wg;
    io.gate_bias = gate_bias;
    io.W1 = W1;
    io.b1 = b1;
    io.W2 = W2;
    io.b2 = b2;
    io.out = outd;
    io.part = at<float>(ws, L.dec_part);
    io.ctr = at<int>(ws, L.dec_ctr);
    io.h = at<void>(ws, L.h_perm);
    io.y = at<void>(ws, L.x_perm);
    io.count = ls.count;
    io.count_copy = ls.count_copy;
    io.dropped = at<int32_t>(ws, L.dropped);
    io.dropped_copy = ls.dropped_copy;
    io.psum = ls.psum;
    io.aux = ls.aux;
    io.err = err;
    const cudaError_t e = launch_decode_layer(s, io, st);
    if (marks)   // one launch: every stage ends with it
      for (int m = kMarkRouter; m <= kMarkCombine; ++m) prof_mark(m, st);
    return e;
  }
  cudaError_t e = cudaSuccess;
  int32_t* ids = at<int32_t>(ws, L.ids);
  float* w = at<float>(ws, L.w);
  float* part = at<float>(ws, L.psum_part);
  const bool fused_hist = layer_fused_hist(s);
  const bool rr = layer_reroutes(s);
  const bool gat = layer_gathers(s, rows);   // no gather kernel: the first product reads x itself
  float* scores = rr ? at<float>(ws, L.scores) : nullptr;
  e = launch_router(s, xd, Wg, gate_bias, scores, ids, w, part, err, st,
                    fused_hist ? at<int32_t>(ws, L.blk_hist) : nullptr);
  if (marks) prof_mark(kMarkRouter, st);
  if (e == cudaSuccess) {
    DispatchOut o;
    memset(&o, 0, sizeof(o));
    o.hist_ready = fused_hist;
    o.count = ls.count;
    o.offs = at<int32_t>(ws, L.offs);
    o.src = at<int32_t>(ws, L.src);
    o.pos = at<int32_t>(ws, L.pos);
    o.blk_hist = at<int32_t>(ws, L.blk_hist);
    o.blk_base = at<int32_t>(ws, L.blk_base);
    o.psum_part = part;
    o.psum = ls.psum;
    o.aux = ls.aux;
    o.count_copy = ls.count_copy;
    if (!rr) {
      o.dropped = at<int32_t>(ws, L.dropped);
      o.dropped_copy = ls.dropped_copy;
      o.sched = at<int32_t>(ws, L.sched);
    }
    e = launch_dispatch(s, ids, rr || gat ? nullptr : xd, rr || gat ? nullptr : at<void>(ws, L.x_perm), o, err,
                        st);
  }
  if (e == cudaSuccess && rr) {
    // the routing's own counts (the loss) are in; now move the slots the
    // capacity dropped, and group the moved routing
    int32_t* fin = at<int32_t>(ws, L.fin);
    e = launch_reroute(s, scores, ids, at<int32_t>(ws, L.pos), at<int32_t>(ws, L.offs), fin,
                       at<int32_t>(ws, L.pend), at<int32_t>(ws, L.choice), at<uint8_t>(ws, L.alts),
                       at<int32_t>(ws, L.dropped), ls.dropped_copy, st);
    if (e == cudaSuccess) {
      DispatchOut o;
      memset(&o, 0, sizeof(o));
      o.offs = at<int32_t>(ws, L.offs);
      o.src = at<int32_t>(ws, L.src);
      o.pos = at<int32_t>(ws, L.pos);
      o.blk_hist = at<int32_t>(ws, L.blk_hist);
      o.blk_base = at<int32_t>(ws, L.blk_base);
      o.sched = at<int32_t>(ws, L.sched);
      e = launch_dispatch(final_shape(s), fin, xd, at<void>(ws, L.x_perm), o, err, st);
    }
  }
  const bool fuse = combine_fusable(s, rows);
  float* acc = fuse ? at<float>(ws, L.acc) : nullptr;
  if (e == cudaSuccess && fuse) e = launch_zero_acc(s, acc, st);
  if (marks) prof_mark(kMarkDispatch, st);
  void* x_perm = at<void>(ws, L.x_perm);
  void* h_perm = at<void>(ws, L.h_perm);
  void* y_perm = x_perm;   // x_perm is dead once the first product has run
  const CombineInto ci{at<int32_t>(ws, L.src), w, acc};
  const GatherRows gr{xd, at<int32_t>(ws, L.src)};
  if (e == cudaSuccess)
    e = launch_ffn(s, rows, x_perm, at<int32_t>(ws, L.offs), W1, b1, W2, b2, h_perm, y_perm, err,
                   at<int32_t>(ws, L.sched), st, fuse ? &ci : nullptr, gat ? &gr : nullptr);
  if (marks) prof_mark(kMarkSecond, st);
  if (e == cudaSuccess) {
    if (fuse) {
      e = launch_acc_to_out(s, acc, outd, st);
    } else if (cparts && cparts->parts > 1) {
      const size_t row_bytes = (size_t)s.H * s.esize();
      for (int p = 0; p < cparts->parts && e == cudaSuccess; ++p) {
        const int64_t t0 = s.T * p / cparts->parts, t1 = s.T * (p + 1) / cparts->parts;
        Shape sp = s;
        sp.T = t1 - t0;
        e = launch_combine(sp, y_perm, at<int32_t>(ws, L.pos) + t0 * s.K, w + t0 * s.K,
                           (char*)outd + t0 * row_bytes, st);
        if (e == cudaSuccess) e = cudaEventRecord(cparts->done[p], st);
      }
    } else {
      e = launch_combine(s, y_perm, at<int32_t>(ws, L.pos), w, outd, st);
    }
  }
  if (marks) prof_mark(kMarkCombine, st);
  return e;
}

// The copy streams and events of the chunked host-I/O path, created once per
// host thread and device.
struct IoRes {
  bool ok = false;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, in[kIoChunks] = {}, done[kIoChunks] = {}, end = nullptr;
  cudaEvent_t part[kLastParts] = {};   // the last piece's combine, by parts
};
constexpr int kMaxIoDevices = 64;
thread_local IoRes g_io[kMaxIoDevices];

cudaError_t io_resources(IoRes** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxIoDevices) return cudaErrorInvalidDevice;
  IoRes& r = g_io[dev];
  if (!r.ok) {
    const unsigned ef = cudaEventDisableTiming;
    if ((e = cudaStreamCreateWithFlags(&r.h2d, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&r.d2h, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&r.start, ef)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&r.end, ef)) != cudaSuccess) return e;
    for (int c = 0; c < kIoChunks; ++c) {
      if ((e = cudaEventCreateWithFlags(&r.in[c], ef)) != cudaSuccess) return e;
      if ((e = cudaEventCreateWithFlags(&r.done[c], ef)) != cudaSuccess) return e;
    }
    for (int p = 0; p < kLastParts; ++p)
      if ((e = cudaEventCreateWithFlags(&r.part[p], ef)) != cudaSuccess) return e;
    r.ok = true;
  }
  *out = &r;
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

int moe_layer_forward(const moe_desc* desc, const void* x, const void* Wg, const float* gate_bias,
                      const void* W1, const float* b1, const void* W2, const float* b2, void* out,
                      float* aux, int32_t* count, int32_t* dropped, void* ws, size_t ws_bytes,
                      void* stream) {
  int rc = check_desc(desc);
  if (rc) return rc;
  const moe_desc& d = *desc;
  if ((rc = check_ws(d, ws, ws_bytes))) return rc;
  if (!Wg || !W1 || !W2) return MOE_ERR_INVALID;
  if (d.T > 0 && (!x || !out)) return MOE_ERR_INVALID;
  if (!aligned16(Wg) || !aligned16(W1) || !aligned16(W2)) return MOE_ERR_INVALID;
  const bool host_io = (d.flags & MOE_FLAG_HOST_IO) != 0;
  if (!host_io && d.T > 0 && (!aligned16(x) || !aligned16(out))) return MOE_ERR_INVALID;
  const Layout L = layout_of(d);
  const Shape s = shape_of(d);
  cudaStream_t st = (cudaStream_t)stream;
  const size_t row_bytes = (size_t)s.H * s.esize();
  cudaError_t e = cudaSuccess;
  if (host_io && io_chunked(s)) {
    // two pieces of tokens: the H2D of the second overlaps the layer on the
    // first, the D2H of the first the layer on the second
    IoRes* io = nullptr;
    if ((e = io_resources(&io)) != cudaSuccess) return cuda_status(e);
    char* xs = at<char>(ws, L.x_stage);
    char* os = at<char>(ws, L.out_stage);
    e = cudaEventRecord(io->start, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(io->h2d, io->start, 0);
    for (int c = 0; c < kIoChunks && e == cudaSuccess; ++c) {
      const int64_t t0 = io_chunk_begin(s, c), t1 = io_chunk_begin(s, c + 1);
      e = cudaMemcpyAsync(xs + t0 * row_bytes, (const char*)x + t0 * row_bytes, (size_t)(t1 - t0) * row_bytes,
                          cudaMemcpyHostToDevice, io->h2d);
      if (e == cudaSuccess) e = cudaEventRecord(io->in[c], io->h2d);
    }
    for (int c = 0; c < kIoChunks && e == cudaSuccess; ++c) {
      const int64_t t0 = io_chunk_begin(s, c), t1 = io_chunk_begin(s, c + 1);
      Shape sc = s;
      sc.T = t1 - t0;
      moe_desc dc = d;
      dc.T = sc.T;
      const LayerStats ls{at<int32_t>(ws, L.count_chunks) + (size_t)c * s.E,
                          at<float>(ws, L.psum_chunks) + (size_t)c * s.E, nullptr, nullptr, nullptr};
      const bool last = c == kIoChunks - 1;
      const CombineParts cp{kLastParts, io->part};
      e = cudaStreamWaitEvent(st, io->in[c], 0);
      if (e == cudaSuccess)
        e = run_layer(sc, rows_for(dc), L, ws, xs + t0 * row_bytes, Wg, gate_bias, W1, b1, W2, b2,
                      os + t0 * row_bytes, ls, false, st, last && !combine_fusable(sc, rows_for(dc)) ? &cp : nullptr);
      if (e == cudaSuccess) e = cudaEventRecord(io->done[c], st);
    }
    for (int c = 0; c < kIoChunks && e == cudaSuccess; ++c) {
      const int64_t t0 = io_chunk_begin(s, c), t1 = io_chunk_begin(s, c + 1);
      Shape sc = s;
      sc.T = t1 - t0;
      moe_desc dc = d;
      dc.T = sc.T;
      if (c == kIoChunks - 1 && !combine_fusable(sc, rows_for(dc))) {
        // the last piece's output in parts, each as soon as its combine is done
        for (int p = 0; p < kLastParts && e == cudaSuccess; ++p) {
          const int64_t a = t0 + sc.T * p / kLastParts, b = t0 + sc.T * (p + 1) / kLastParts;
          e = cudaStreamWaitEvent(io->d2h, io->part[p], 0);
          if (e == cudaSuccess)
            e = cudaMemcpyAsync((char*)out + a * row_bytes, os + a * row_bytes, (size_t)(b - a) * row_bytes,
                                cudaMemcpyDeviceToHost, io->d2h);
        }
        continue;
      }
      e = cudaStreamWaitEvent(io->d2h, io->done[c], 0);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync((char*)out + t0 * row_bytes, os + t0 * row_bytes, (size_t)(t1 - t0) * row_bytes,
                            cudaMemcpyDeviceToHost, io->d2h);
    }
    // the whole batch's counts and loss from the pieces' sums
    if (e == cudaSuccess)
      e = launch_merge_stats(s, at<int32_t>(ws, L.count_chunks), at<float>(ws, L.psum_chunks), kIoChunks,
                             at<int32_t>(ws, L.count), at<float>(ws, L.psum), count, aux, dropped, st);
    if (e == cudaSuccess) e = cudaEventRecord(io->end, io->d2h);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, io->end, 0);   // the caller's stream covers it all
    return cuda_status(e);
  }
  const size_t xbytes = (size_t)s.T * row_bytes;
  const void* xd = x;
  void* outd = out;
  prof_mark(kMarkStart, st);
  if (host_io && s.T > 0) {
    xd = at<void>(ws, L.x_stage);
    outd = at<void>(ws, L.out_stage);
    e = cudaMemcpyAsync((void*)xd, x, xbytes, cudaMemcpyHostToDevice, st);
  }
  const LayerStats ls{at<int32_t>(ws, L.count), at<float>(ws, L.psum), aux, count, dropped};
  if (e == cudaSuccess)
    e = run_layer(s, L.rows, L, ws, xd, Wg, gate_bias, W1, b1, W2, b2, outd, ls, true, st);
  if (e == cudaSuccess && host_io && s.T > 0)
    e = cudaMemcpyAsync(out, outd, xbytes, cudaMemcpyDeviceToHost, st);
  return cuda_status(e);
}

int moe_profile_events(void* const* events, int n) {
  if (!events || n <= 0) {
    g_prof_on = false;
    return MOE_OK;
  }
  if (n < kMarks) return MOE_ERR_INVALID;
  for (int i = 0; i < kMarks; ++i) {
    if (!events[i]) return MOE_ERR_INVALID;
    g_prof[i] = (cudaEvent_t)events[i];
  }
  g_prof_on = true;
  return MOE_OK;
}

int moe_get_device_error(void* ws, int32_t* code, void* stream) {
  if (!ws || !code) return MOE_ERR_INVALID;
  cudaStream_t st = (cudaStream_t)stream;
  int h = 0;
  if (cudaMemcpyAsync(&h, ws, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemsetAsync(ws, 0, sizeof(int), st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  *code = h == kDevOk ? MOE_OK : (h == kDevTimeout ? MOE_ERR_TIMEOUT : MOE_ERR_DEVICE);
  return MOE_OK;
}

}  // extern "C"
