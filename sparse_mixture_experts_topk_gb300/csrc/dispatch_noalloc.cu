// moe_dispatch_noalloc: the dispatch step for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc at the point where they route tokens:
// code running inside an allocator or memory-pool callback, runtimes that own
// every device byte up front and hand none out, or plugin hosts that forbid
// allocation on their execution path.  moe_dispatch needs a caller-sized
// workspace for its per-block expert histograms; this variant keeps that
// scratch in a fixed array in device memory that belongs to the library
// instead.  The caller still passes every input and output buffer.
//
// The array is a file-scope __device__ variable of kScratchBytes (64 KiB).
// Every GPU that loads the library holds it until the process exits.  Host
// code cannot use the array's name as a device address: each call looks the
// address up with cudaGetSymbolAddress, with the call's device current, and
// keeps it per device.  A call made while its stream is being captured uses
// the kept address instead, so the first call on each device must come before
// any stream capture; a device reset (cudaDeviceReset) or an unload of the
// library makes the kept address stale until the next call outside capture.
// All calls on a device share the one array, so calls that overlap on the
// GPU (different streams, or different host threads) race on it and must be
// serialised by the caller.  The histogram and prefix kernels write every
// scratch word they later read, so stale contents from an earlier call are
// never used and nothing needs clearing; the optional error word the caller
// passes is cleared by each call.
#include <mutex>

#include "internal.h"

namespace moe {
namespace {

// Two int32 tables of [dispatch blocks][E] (per-block histograms and their
// prefix over blocks).
constexpr size_t kScratchBytes = 64 * 1024;

static __device__ __align__(256) unsigned char g_dispatch_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device: looked up
// afresh outside stream capture (cheap), the address kept from the last such
// lookup while `st` is being captured.
cudaError_t scratch_address(cudaStream_t st, void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  const bool capturing = cudaStreamIsCapturing(st, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!capturing || !g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_dispatch_noalloc(const moe_desc* desc, const int32_t* ids, const void* x,
                                    int32_t* count, int32_t* offs, int32_t* src, int32_t* pos,
                                    void* x_perm, int32_t* dropped, int32_t* device_error,
                                    void* stream) {
  const int64_t rows = moe_max_rows(desc);     // also validates desc
  if (rows < 0) return MOE_ERR_INVALID;
  const moe_desc& d = *desc;
  if (!count || !offs || (d.T > 0 && (!ids || !src || !pos))) return MOE_ERR_INVALID;
  if (x && (!x_perm || ((uintptr_t)x & 15u) || ((uintptr_t)x_perm & 15u))) return MOE_ERR_INVALID;
  const Shape s = shape_of(d);
  const size_t table = (size_t)dispatch_blocks(s) * s.E * sizeof(int32_t);
  if (2 * table > kScratchBytes) return MOE_ERR_UNSUPPORTED;   // beyond the fixed scratch
  cudaStream_t st = (cudaStream_t)stream;
  void* base = nullptr;
  if (scratch_address(st, &base) != cudaSuccess) return MOE_ERR_CUDA;
  if (device_error && cudaMemsetAsync(device_error, 0, sizeof(int32_t), st) != cudaSuccess)
    return MOE_ERR_CUDA;
  DispatchOut o = {};
  o.count = count; o.offs = offs; o.src = src; o.pos = pos; o.dropped = dropped;
  o.blk_hist = reinterpret_cast<int32_t*>(base);
  o.blk_base = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(base) + table);
  cudaError_t e = launch_dispatch(s, ids, x, x_perm, o, reinterpret_cast<int*>(device_error), st);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
