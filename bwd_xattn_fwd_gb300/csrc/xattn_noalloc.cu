// xattn_bwd_noalloc: the bf16 backward with its scratch memory in a fixed device array
// owned by the library, for callers that must not allocate device memory.
//
// Who needs it: code that runs under a no-allocation rule once it is up (for example a
// latency-critical training or serving loop, where cudaFree's implicit device-wide
// synchronisation is not acceptable), and hosts whose device memory is already fully
// reserved by another allocator, so a cudaMalloc/cudaMallocAsync issued by this
// library would fail. xattn_bwd takes its scratch with cudaMallocAsync; this entry
// point takes none.
//
// The scratch is a file-scope device array of XATTN_NOALLOC_SCRATCH_BYTES (64 MiB).
// CUDA loads a library's device code lazily, so the array is placed on a GPU by the
// first call of this entry point on that GPU, and stays there until the process exits.
// Host code cannot use the array's name as a device address (on the host it names a
// stand-in object), so that first call looks the address up with cudaGetSymbolAddress
// while the device is current (which is what loads the module and places the array),
// and every later call reuses it. A failed lookup (say the device had no 64 MiB left)
// is not remembered: the next call tries again.
#include <cmath>
#include <mutex>

#include "xattn.h"
#include "xattn_internal.h"

namespace xattn {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[XATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxNoAllocDevices = 64;

std::mutex g_slots_mutex;
void *g_slots[kMaxNoAllocDevices];   // scratch address per device; null until found

// Device address of the scratch array on the current device. Only a successful lookup is
// kept, so a device where it failed once is tried again on the next call.
xattn_status scratch_address(int dev, void **out) {
  if (dev < 0 || dev >= kMaxNoAllocDevices) return XATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_slots_mutex);
  if (g_slots[dev] == nullptr) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();   // do not leave the failure for the caller's next error check
      return XATTN_ERR_CUDA;
    }
    g_slots[dev] = ptr;
  }
  *out = g_slots[dev];
  return XATTN_OK;
}

}  // namespace
}  // namespace xattn

extern "C" xattn_status xattn_bwd_noalloc(const void *q, const void *k, const void *v,
                                          const void *o, const void *dO, const float *lse,
                                          int B, int S, int nh, int nkv, int hd, float scale,
                                          void *dq, void *dk, void *dv, void *stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return XATTN_ERR_NULL_PTR;
  // Every check that a step below would make runs first, so a rejected call launches
  // nothing.
  if (B <= 0 || S <= 0 || nh <= 0 || nkv <= 0 || hd <= 0) return XATTN_ERR_BAD_SHAPE;
  if (nh % nkv != 0) return XATTN_ERR_GROUP;
  if (hd != 32 && hd != 64) return XATTN_ERR_UNSUPPORTED_HD;
  if (!std::isfinite(scale)) return XATTN_ERR_BAD_SCALE;
  if (scale != 0.f && std::fabs(scale) < 0x1p-64f) return XATTN_ERR_BAD_SCALE;
  for (const void *p : {q, k, v, o, dO, static_cast<const void *>(dq), static_cast<const void *>(dk),
                        static_cast<const void *>(dv)})
    if (reinterpret_cast<uintptr_t>(p) & 15u) return XATTN_ERR_MISALIGNED;
  const size_t need = xattn_bwd_workspace_bytes(B, S, nh, hd);
  if (need == 0) return XATTN_ERR_BAD_SHAPE;
  if (need > static_cast<size_t>(XATTN_NOALLOC_SCRATCH_BYTES)) return XATTN_ERR_SCRATCH_LIMIT;
  // The scratch address is the current device's, so the stream must belong to it.
  int dev = 0, stream_dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return XATTN_ERR_CUDA;
  if (cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &stream_dev) != cudaSuccess ||
      stream_dev != dev)
    return XATTN_ERR_CUDA;
  void *scratch = nullptr;
  const xattn_status st = xattn::scratch_address(dev, &scratch);
  if (st != XATTN_OK) return st;
  // The three steps rewrite every scratch byte they read (the preprocess writes every
  // auxiliary row, pad rows included, and every D_i, and zeroes the dQ accumulator), so
  // contents left by an earlier call never leak into this one.
  xattn_status r = xattn_bwd_preprocess(o, dO, lse, B, S, nh, hd, scale, scratch, need, stream);
  if (r == XATTN_OK)
    r = xattn_bwd_main(q, k, v, dO, B, S, nh, nkv, hd, scale, dk, dv, scratch, need, stream);
  if (r == XATTN_OK) r = xattn_bwd_dq_convert(B, S, nh, hd, scale, dq, scratch, need, stream);
  return r;
}
