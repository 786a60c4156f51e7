// C ABI of libxattn (declared in include/xattn.h): argument checks, TMA tensor maps,
// scratch handling and kernel launches. No call synchronises the device except
// xattn_check_device_status.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "xattn.h"
#include "sm103_ptx.cuh"
#include "xattn_internal.h"

namespace xattn {
namespace {

// Device status word, written by kernels whose bounded waits expire.
__device__ int g_device_status;

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  bool sm103 = false;
  int *status = nullptr;
};
DeviceInfo g_dev[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

uint64_t wait_limit_ns() {
  static const uint64_t v = [] {
    const char *s = std::getenv("XATTN_WAIT_LIMIT_NS");
    const unsigned long long x = s ? std::strtoull(s, nullptr, 10) : 0ull;
    return x > 0 ? static_cast<uint64_t>(x) : static_cast<uint64_t>(2000000000ull);
  }();
  return v;
}

}  // namespace

bool pdl_enabled() {
  static const bool v = std::getenv("XATTN_NO_PDL") == nullptr;
  return v;
}

namespace {

// Self-test of the bounded waits: one CTA waits on an mbarrier that nothing ever arrives
// on (phase 0 of a barrier expecting one arrival), with the same wait the kernels use.
// The wait runs out after limit_ns and records XATTN_ERR_DEVICE_TIMEOUT in the status
// word; nothing else happens on the device.
__global__ void wait_selftest_kernel(int *status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtl ctl{&abort_flag, status, limit_ns};
  (void)mbar_wait(smem_u32(&bar), 0, ctl);
}

// A bounds check that fails by construction (index n of a range of n elements, never
// used for an access): in a debug build it records XATTN_ERR_DEVICE_BOUNDS.
__global__ void bounds_selftest_kernel(int *status, int n) {
  const int i = n;
  XATTN_DCHECK(i < n, status);
  (void)i;
  (void)status;
}

xattn_status device_info(DeviceInfo **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return XATTN_ERR_CUDA;
  DeviceInfo &d = g_dev[dev];
  std::call_once(d.once, [&d, dev] {
    int major = 0, minor = 0;
    d.err = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (d.err == cudaSuccess) d.err = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    d.sm103 = (major == 10 && minor == 3);
    if (d.err == cudaSuccess) d.err = cudaGetSymbolAddress(reinterpret_cast<void **>(&d.status), g_device_status);
  });
  if (d.err != cudaSuccess) return XATTN_ERR_CUDA;
  *out = &d;
  return XATTN_OK;
}

xattn_status get_encode() {
  std::call_once(g_encode_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode ? XATTN_OK : XATTN_ERR_CUDA;
}

// 4-D map over a contiguous [B, S, H, hd] bf16 tensor; box = one head's 128-row tile, or
// at hd = 128 one 64-column half of it (a swizzled box row is at most 128 bytes; the
// kernels load the two halves as two sub-tiles). The 128-byte (hd = 64, 128) or 64-byte
// (hd = 32) swizzle matches the UMMA operand layout. Rows past S read as zeros.
xattn_status make_map(CUtensorMap *map, const void *ptr, int B, int S, int H, int hd) {
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(hd), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(B)};
  const cuuint64_t row = static_cast<cuuint64_t>(hd) * 2;
  const cuuint64_t strides[3] = {row, row * H, row * H * S};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(hd > 64 ? 64 : hd), 1, static_cast<cuuint32_t>(kTileRows), 1};
  const cuuint32_t elem[4] = {1, 1, 1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims,
                              strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              hd == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? XATTN_OK : XATTN_ERR_CUDA;
}

// 4-D fp32 map over the [B, S, nh, hd] dQ accumulator. The box is half a head row
// (hd/2 floats: 128 bytes at hd = 64, 64 bytes at hd = 32, with the matching swizzle)
// by 128 rows; the backward adds shared-memory tiles into it with TMA reduce-adds.
// Rows past S are skipped by the TMA unit.
xattn_status make_map_dq(CUtensorMap *map, float *ptr, int B, int S, int nh, int hd) {
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(hd), static_cast<cuuint64_t>(nh),
                              static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(B)};
  const cuuint64_t row = static_cast<cuuint64_t>(hd) * 4;
  const cuuint64_t strides[3] = {row, row * nh, row * nh * S};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(hd / 2), 1, static_cast<cuuint32_t>(kTileRows), 1};
  const cuuint32_t elem[4] = {1, 1, 1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ptr, dims, strides, box, elem,
                              CU_TENSOR_MAP_INTERLEAVE_NONE,
                              hd == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? XATTN_OK : XATTN_ERR_CUDA;
}

// 4-D map over the backward's [B, nh, S_pad, 16] bf16 auxiliary rows; box = 16 columns
// (32 bytes, 32-byte swizzle) by 128 rows.
xattn_status make_map_aux(CUtensorMap *map, void *ptr, int B, int S, int nh) {
  const cuuint64_t S_pad = static_cast<cuuint64_t>(padded_rows(S));
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kAuxCols), S_pad, static_cast<cuuint64_t>(nh),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t row = kAuxCols * 2;
  const cuuint64_t strides[3] = {row, row * S_pad, row * S_pad * nh};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(kAuxCols), static_cast<cuuint32_t>(kTileRows), 1, 1};
  const cuuint32_t elem[4] = {1, 1, 1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, ptr, dims, strides, box, elem,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? XATTN_OK : XATTN_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

xattn_status check_shape(int B, int S, int nh, int nkv, int hd, float scale) {
  if (B <= 0 || S <= 0 || nh <= 0 || nkv <= 0 || hd <= 0) return XATTN_ERR_BAD_SHAPE;
  // Keep every element index and grid size well inside their integer types.
  const long long elems = static_cast<long long>(B) * S * nh * hd;
  if (elems > (1ll << 40) || static_cast<long long>(B) * nh * ((S + 127) / 128) > (1ll << 31) - 1)
    return XATTN_ERR_BAD_SHAPE;
  if (nh % nkv != 0) return XATTN_ERR_GROUP;
  if (!std::isfinite(scale)) return XATTN_ERR_BAD_SCALE;
  return XATTN_OK;
}

// The bf16 backward folds -LSE/scale into a tensor-core operand; it takes scale == 0
// exactly, and any |scale| >= 2^-64 (so that LSE/scale stays far from overflow).
xattn_status check_bwd_scale(float scale) {
  if (!std::isfinite(scale)) return XATTN_ERR_BAD_SCALE;
  if (scale != 0.f && std::fabs(scale) < 0x1p-64f) return XATTN_ERR_BAD_SCALE;
  return XATTN_OK;
}

xattn_status check_bf16(int hd) { return (hd == 32 || hd == 64) ? XATTN_OK : XATTN_ERR_UNSUPPORTED_HD; }
xattn_status check_bf16_fwd(int hd) {
  return (hd == 32 || hd == 64 || hd == 128) ? XATTN_OK : XATTN_ERR_UNSUPPORTED_HD;
}

// With XATTN_VERBOSE set in the environment, CUDA failures are also reported on stderr.
xattn_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return XATTN_OK;
  static const bool verbose = std::getenv("XATTN_VERBOSE") != nullptr;
  if (verbose) std::fprintf(stderr, "libxattn: CUDA error %d: %s\n", static_cast<int>(e), cudaGetErrorString(e));
  return XATTN_ERR_CUDA;
}

#define XATTN_TRY(expr)                          \
  do {                                           \
    const xattn_status st_ = (expr);             \
    if (st_ != XATTN_OK) return st_;             \
  } while (0)

xattn_status bf16_device(DeviceInfo **dev) {
  XATTN_TRY(device_info(dev));
  if (!(*dev)->sm103) return XATTN_ERR_NO_DEVICE_SUPPORT;
  return get_encode();
}

xattn_status check_workspace(void *ws, size_t bytes, int B, int S, int nh, int hd) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return XATTN_ERR_WORKSPACE;
  if (bytes < bwd_workspace_bytes(B, S, nh, hd, true)) return XATTN_ERR_WORKSPACE;
  return XATTN_OK;
}

}  // namespace
}  // namespace xattn

using namespace xattn;

extern "C" {

xattn_status xattn_fwd(const void *q, const void *k, const void *v, int B, int S, int nh, int nkv,
                       int hd, float scale, void *o, float *lse, void *stream) {
  if (!q || !k || !v || !o || !lse) return XATTN_ERR_NULL_PTR;
  XATTN_TRY(check_shape(B, S, nh, nkv, hd, scale));
  XATTN_TRY(check_bf16_fwd(hd));
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return XATTN_ERR_MISALIGNED;
  DeviceInfo *dev = nullptr;
  XATTN_TRY(bf16_device(&dev));
  CUtensorMap mq, mk, mv;
  XATTN_TRY(make_map(&mq, q, B, S, nh, hd));
  XATTN_TRY(make_map(&mk, k, B, S, nkv, hd));
  XATTN_TRY(make_map(&mv, v, B, S, nkv, hd));
  return cuda_status(launch_fwd_bf16(mq, mk, mv, static_cast<__nv_bfloat16 *>(o), lse, B, S, nh, nkv,
                                     hd, scale, dev->status, wait_limit_ns(),
                                     static_cast<cudaStream_t>(stream)));
}

int xattn_bwd_dq_mode(int S, int nh, int nkv, int hd, int deterministic) {
  if (S <= 0 || nh <= 0 || nkv <= 0 || nh % nkv != 0) return -1;
  if (hd != 32 && hd != 64 && hd != 128) return -1;
  if (!deterministic && hd != 128) return XATTN_BWD_FUSED_DQ;
  return bwd_resident_dq_ok(S, nh, nkv, hd) ? XATTN_BWD_RESIDENT_DQ : XATTN_BWD_QUERY_DQ;
}

int xattn_decode_runs(int B, int T, int nh, int nkv, int hd, int num_sms) {
  if (B <= 0 || T <= 0 || nh <= 0 || nkv <= 0 || nh % nkv != 0 || num_sms <= 0) return -1;
  if (nh / nkv > kMaxDecodeGroup || (hd != 32 && hd != 64 && hd != 128)) return -1;
  const long long chunks = (static_cast<long long>(T) + decode_chunk_keys(hd) - 1) / decode_chunk_keys(hd);
  if (static_cast<long long>(B) * nkv * chunks > 0x7fffffffLL) return -1;
  return decode_runs(B, T, nh, nkv, hd, num_sms);
}

size_t xattn_bwd_workspace_bytes(int B, int S, int nh, int hd) {
  if (B <= 0 || S <= 0 || nh <= 0 || hd <= 0) return 0;
  return bwd_workspace_bytes(B, S, nh, hd, true);
}

xattn_status xattn_bwd_preprocess(const void *o, const void *dO, const float *lse, int B, int S,
                                  int nh, int hd, float scale, void *workspace,
                                  size_t workspace_bytes, void *stream) {
  if (!o || !dO || !lse) return XATTN_ERR_NULL_PTR;
  XATTN_TRY(check_shape(B, S, nh, nh, hd, scale));
  XATTN_TRY(check_bwd_scale(scale));
  XATTN_TRY(check_bf16(hd));
  if (!aligned16(o) || !aligned16(dO)) return XATTN_ERR_MISALIGNED;
  XATTN_TRY(check_workspace(workspace, workspace_bytes, B, S, nh, hd));
  DeviceInfo *dev = nullptr;
  XATTN_TRY(bf16_device(&dev));
  const BwdWorkspace ws = bwd_workspace_carve(workspace, B, S, nh, hd);
  return cuda_status(launch_bwd_preprocess(static_cast<const __nv_bfloat16 *>(o),
                                           static_cast<const __nv_bfloat16 *>(dO), lse, B, S, nh, hd,
                                           scale, ws, true, static_cast<cudaStream_t>(stream)));
}

xattn_status xattn_bwd_main(const void *q, const void *k, const void *v, const void *dO, int B,
                            int S, int nh, int nkv, int hd, float scale, void *dk, void *dv,
                            void *workspace, size_t workspace_bytes, void *stream) {
  if (!q || !k || !v || !dO || !dk || !dv) return XATTN_ERR_NULL_PTR;
  XATTN_TRY(check_shape(B, S, nh, nkv, hd, scale));
  XATTN_TRY(check_bwd_scale(scale));
  XATTN_TRY(check_bf16(hd));
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(dk) ||
      !aligned16(dv))
    return XATTN_ERR_MISALIGNED;
  XATTN_TRY(check_workspace(workspace, workspace_bytes, B, S, nh, hd));
  DeviceInfo *dev = nullptr;
  XATTN_TRY(bf16_device(&dev));
  CUtensorMap mq, mk, mv, mdo;
  XATTN_TRY(make_map(&mq, q, B, S, nh, hd));
  XATTN_TRY(make_map(&mk, k, B, S, nkv, hd));
  XATTN_TRY(make_map(&mv, v, B, S, nkv, hd));
  XATTN_TRY(make_map(&mdo, dO, B, S, nh, hd));
  const BwdWorkspace ws = bwd_workspace_carve(workspace, B, S, nh, hd);
  CUtensorMap maux, mdq;
  XATTN_TRY(make_map_aux(&maux, ws.aux, B, S, nh));
  XATTN_TRY(make_map_dq(&mdq, ws.dqacc, B, S, nh, hd));
  return cuda_status(launch_bwd_main_bf16(mq, mk, mv, mdo, maux, &mdq, static_cast<__nv_bfloat16 *>(dk),
                                          static_cast<__nv_bfloat16 *>(dv), B, S, nh, nkv, hd, scale,
                                          dev->status, wait_limit_ns(),
                                          static_cast<cudaStream_t>(stream)));
}

xattn_status xattn_bwd_dq_convert(int B, int S, int nh, int hd, float scale, void *dq,
                                  void *workspace, size_t workspace_bytes, void *stream) {
  if (!dq) return XATTN_ERR_NULL_PTR;
  XATTN_TRY(check_shape(B, S, nh, nh, hd, scale));
  XATTN_TRY(check_bf16(hd));
  if (!aligned16(dq)) return XATTN_ERR_MISALIGNED;
  XATTN_TRY(check_workspace(workspace, workspace_bytes, B, S, nh, hd));
  DeviceInfo *dev = nullptr;
  XATTN_TRY(bf16_device(&dev));
  const BwdWorkspace ws = bwd_workspace_carve(workspace, B, S, nh, hd);
  return cuda_status(launch_dq_convert(ws.dqacc, static_cast<__nv_bfloat16 *>(dq),
                                       static_cast<size_t>(B) * S * nh * hd, scale,
                                       static_cast<cudaStream_t>(stream)));
}

xattn_status xattn_bwd(const void *q, const void *k, const void *v, const void *o, const void *dO,
                       const float *lse, int B, int S, int nh, int nkv, int hd, float scale, void *dq,
                       void *dk, void *dv, void *stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return XATTN_ERR_NULL_PTR;
  XATTN_TRY(check_shape(B, S, nh, nkv, hd, scale));
  XATTN_TRY(check_bwd_scale(scale));
  XATTN_TRY(check_bf16_fwd(hd));
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return XATTN_ERR_MISALIGNED;
  // hd = 128: dV, dK and a dQ accumulator do not fit in TMEM together, so dQ comes from
  // the query-stationary kernel (the deterministic backward).
  if (hd == 128) return xattn_bwd_deterministic(q, k, v, o, dO, lse, B, S, nh, nkv, hd, scale, dq, dk, dv, stream);
  DeviceInfo *dev = nullptr;
  XATTN_TRY(bf16_device(&dev));
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t bytes = bwd_workspace_bytes(B, S, nh, hd, true);
  void *ws = nullptr;
  if (cudaMallocAsync(&ws, bytes, st) != cudaSuccess) return XATTN_ERR_CUDA;
  xattn_status r = xattn_bwd_preprocess(o, dO, lse, B, S, nh, hd, scale, ws, bytes, stream);
  if (r == XATTN_OK) r = xattn_bwd_main(q, k, v, dO, B, S, nh, nkv, hd, scale, dk, dv, ws, bytes, stream);
  if (r == XATTN_OK) r = xattn_bwd_dq_convert(B, S, nh, hd, scale, dq, ws, bytes, stream);
  const cudaError_t fe = cudaFreeAsync(ws, st);
  if (r == XATTN_OK && fe != cudaSuccess) r = XATTN_ERR_CUDA;
  return r;
}

xattn_status xattn_decode(const void *q, const void *k_cache, const void *v_cache, int B, int T,
                          int nh, int nkv, int hd, float scale, void *o, float *lse, void *stream) {
  if (!q || !k_cache || !v_cache || !o || !lse) return XATTN_ERR_NULL_PTR;
  XATTN_TRY(check_shape(B, T, nh, nkv, hd, scale));
  if (nh / nkv > kMaxDecodeGroup) return XATTN_ERR_GROUP;
  if (hd != 32 && hd != 64 && hd != 128) return XATTN_ERR_UNSUPPORTED_HD;
  // One CTA per (batch, kv head, chunk): the grid is one-dimensional.
  const long long chunks = (static_cast<long long>(T) + decode_chunk_keys(hd) - 1) / decode_chunk_keys(hd);
  if (static_cast<long long>(B) * nkv * chunks > 0x7fffffffLL) return XATTN_ERR_BAD_SHAPE;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return XATTN_ERR_MISALIGNED;
  DeviceInfo *dev = nullptr;
  XATTN_TRY(bf16_device(&dev));
  CUtensorMap mk, mv;
  XATTN_TRY(make_map(&mk, k_cache, B, T, nkv, hd));
  XATTN_TRY(make_map(&mv, v_cache, B, T, nkv, hd));
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  void *ws = nullptr;
  if (cudaMallocAsync(&ws, decode_workspace_bytes(B, T, nh, hd), st) != cudaSuccess) return XATTN_ERR_CUDA;
  xattn_status r = cuda_status(launch_decode_bf16(mk, mv, static_cast<const __nv_bfloat16 *>(q),
                                                  static_cast<__nv_bfloat16 *>(o), lse, B, T, nh, nkv, hd, scale, ws,
                                                  dev->status, wait_limit_ns(), st));
  const cudaError_t fe = cudaFreeAsync(ws, st);
  if (r == XATTN_OK && fe != cudaSuccess) r = XATTN_ERR_CUDA;
  return r;
}

xattn_status xattn_bwd_deterministic(const void *q, const void *k, const void *v, const void *o,
                                     const void *dO, const float *lse, int B, int S, int nh,
                                     int nkv, int hd, float scale, void *dq, void *dk, void *dv,
                                     void *stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return XATTN_ERR_NULL_PTR;
  XATTN_TRY(check_shape(B, S, nh, nkv, hd, scale));
  XATTN_TRY(check_bwd_scale(scale));
  XATTN_TRY(check_bf16_fwd(hd));
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return XATTN_ERR_MISALIGNED;
  DeviceInfo *dev = nullptr;
  XATTN_TRY(bf16_device(&dev));
  CUtensorMap mq, mk, mv, mdo;
  XATTN_TRY(make_map(&mq, q, B, S, nh, hd));
  XATTN_TRY(make_map(&mk, k, B, S, nkv, hd));
  XATTN_TRY(make_map(&mv, v, B, S, nkv, hd));
  XATTN_TRY(make_map(&mdo, dO, B, S, nh, hd));
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t bytes = bwd_workspace_bytes(B, S, nh, hd, false);
  void *base = nullptr;
  if (cudaMallocAsync(&base, bytes, st) != cudaSuccess) return XATTN_ERR_CUDA;
  const BwdWorkspace ws = bwd_workspace_carve(base, B, S, nh, hd);
  CUtensorMap maux;
  xattn_status r = make_map_aux(&maux, ws.aux, B, S, nh);
  if (r == XATTN_OK)
    r = cuda_status(launch_bwd_preprocess(static_cast<const __nv_bfloat16 *>(o),
                                          static_cast<const __nv_bfloat16 *>(dO), lse, B, S, nh, hd,
                                          scale, ws, false, st));
  if (r == XATTN_OK && bwd_resident_dq_ok(S, nh, nkv, hd)) {
    // Small problems: one kernel, dQ resident in TMEM over each head's key tiles.
    r = cuda_status(launch_bwd_main_resident_bf16(mq, mk, mv, mdo, maux, static_cast<__nv_bfloat16 *>(dk),
                                                  static_cast<__nv_bfloat16 *>(dv), static_cast<__nv_bfloat16 *>(dq),
                                                  B, S, nh, nkv, hd, scale, dev->status, wait_limit_ns(), st));
  } else {
    if (r == XATTN_OK)
      r = cuda_status(launch_bwd_main_bf16(mq, mk, mv, mdo, maux, nullptr, static_cast<__nv_bfloat16 *>(dk),
                                           static_cast<__nv_bfloat16 *>(dv), B, S, nh, nkv, hd, scale,
                                           dev->status, wait_limit_ns(), st));
    if (r == XATTN_OK)
      r = cuda_status(launch_bwd_dq_bf16(mq, mk, mv, mdo, lse, ws, static_cast<__nv_bfloat16 *>(dq), B, S,
                                         nh, nkv, hd, scale, dev->status, wait_limit_ns(), st));
  }
  const cudaError_t fe = cudaFreeAsync(base, st);
  if (r == XATTN_OK && fe != cudaSuccess) r = XATTN_ERR_CUDA;
  return r;
}

xattn_status xattn_fwd_f32(const float *q, const float *k, const float *v, int B, int S, int nh,
                           int nkv, int hd, float scale, float *o, float *lse, void *stream) {
  if (!q || !k || !v || !o || !lse) return XATTN_ERR_NULL_PTR;
  XATTN_TRY(check_shape(B, S, nh, nkv, hd, scale));
  if (hd > 128) return XATTN_ERR_UNSUPPORTED_HD;
  DeviceInfo *dev = nullptr;
  XATTN_TRY(device_info(&dev));
  return cuda_status(launch_fwd_f32(q, k, v, o, lse, B, S, nh, nkv, hd, scale,
                                    static_cast<cudaStream_t>(stream)));
}

xattn_status xattn_bwd_f32(const float *q, const float *k, const float *v, const float *o,
                           const float *dO, const float *lse, int B, int S, int nh, int nkv, int hd,
                           float scale, float *dq, float *dk, float *dv, void *stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return XATTN_ERR_NULL_PTR;
  XATTN_TRY(check_shape(B, S, nh, nkv, hd, scale));
  if (hd > 128) return XATTN_ERR_UNSUPPORTED_HD;
  DeviceInfo *dev = nullptr;
  XATTN_TRY(device_info(&dev));
  return cuda_status(launch_bwd_f32(q, k, v, o, dO, lse, dq, dk, dv, B, S, nh, nkv, hd, scale,
                                    static_cast<cudaStream_t>(stream)));
}

const char *xattn_status_string(xattn_status s) {
  switch (s) {
    case XATTN_OK: return "ok";
    case XATTN_ERR_NULL_PTR: return "a required pointer is NULL";
    case XATTN_ERR_BAD_SHAPE: return "B, S, nh, nkv and hd must be positive and within size limits";
    case XATTN_ERR_GROUP: return "nh must be a multiple of nkv";
    case XATTN_ERR_UNSUPPORTED_HD: return "unsupported head dimension (bf16: 32, 64 or 128; the backward's stage calls and xattn_bwd_noalloc: 32 or 64; fp32: <= 128)";
    case XATTN_ERR_MISALIGNED: return "a bf16 tensor pointer is not 16-byte aligned";
    case XATTN_ERR_CUDA: return "a CUDA runtime or driver call failed";
    case XATTN_ERR_NO_DEVICE_SUPPORT: return "the current device is not compute capability 10.3 (sm_103)";
    case XATTN_ERR_DEVICE_TIMEOUT: return "a bounded on-device wait expired";
    case XATTN_ERR_BAD_SCALE: return "scale must be finite";
    case XATTN_ERR_WORKSPACE: return "workspace is NULL, not 256-byte aligned, or too small";
    case XATTN_ERR_SCRATCH_LIMIT:
      return "these sizes need more scratch than xattn_bwd_noalloc's fixed array holds";
    case XATTN_ERR_DEVICE_BOUNDS:
      return "an on-device bounds check failed (debug build)";
  }
  return "unknown xattn status";
}

xattn_status xattn_selftest_wait_timeout(unsigned long long limit_ns, void *stream) {
  if (limit_ns < 1000ull || limit_ns > 10000000000ull) return XATTN_ERR_BAD_SHAPE;
  DeviceInfo *dev = nullptr;
  XATTN_TRY(device_info(&dev));
  wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev->status, limit_ns);
  return cuda_status(cudaGetLastError());
}

int xattn_build_flags(void) {
#ifdef XATTN_DEBUG
  return XATTN_BUILD_DEVICE_CHECKS;
#else
  return 0;
#endif
}

xattn_status xattn_selftest_bounds_check(void *stream) {
  DeviceInfo *dev = nullptr;
  XATTN_TRY(device_info(&dev));
  bounds_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev->status, 1);
  return cuda_status(cudaGetLastError());
}

xattn_status xattn_check_device_status(void *stream) {
  DeviceInfo *dev = nullptr;
  XATTN_TRY(device_info(&dev));
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return XATTN_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, dev->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return XATTN_ERR_CUDA;
  if (word != 0) {
    const int zero = 0;
    if (cudaMemcpy(dev->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return XATTN_ERR_CUDA;
    return static_cast<xattn_status>(word);
  }
  return XATTN_OK;
}

}  // extern "C"
