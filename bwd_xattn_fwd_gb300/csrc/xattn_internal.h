// Internal launch interface between the C-ABI layer (xattn_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace xattn {

constexpr int kTileRows = 128;                  // rows of Q / K / V per tile
constexpr float kLog2e = 1.4426950408889634f;   // 1 / ln 2
constexpr float kLn2 = 0.6931471805599453f;

// Launches kernel<<<grid, threads, smem, stream>>>(args...) with programmatic stream
// serialization, so that its set-up overlaps the tail of the previous kernel in the
// stream (each kernel waits for its predecessor with griddepcontrol.wait before touching
// global memory). XATTN_NO_PDL in the environment turns this off (ordinary launches).
bool pdl_enabled();

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, unsigned threads, size_t smem,
                       cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// Rows of the per-(batch, head) workspace vectors, padded to whole tiles.
__host__ __device__ inline int padded_rows(int S) { return (S + kTileRows - 1) / kTileRows * kTileRows; }

// Row i of the backward's per-(batch, head) auxiliary operand: 16 bf16 values (one
// tensor-core K step). Columns 0-2 hold -LSE_i / scale and columns 3-5 hold -D_i, each
// as a sum of three bf16 terms (hi + mid + lo, about 24 significant bits); the rest are
// zero, and pad rows (S <= i < S_pad) are all zero. With scale == 0 columns 0-2 hold
// -LSE_i log2(e) instead (the products then skip Q K^T).
constexpr int kAuxCols = 16;

struct BwdWorkspace {
  __nv_bfloat16 *aux;  // [B, nh, S_pad, kAuxCols]
  float *D;            // [B, S, nh]  D_i = dO_i . O_i in fp32
  float *dqacc;        // [B, S, nh, hd]  fused dQ only: fp32 accumulator of dS K (no scale)
};

// fused_dq: the workspace also holds the fp32 dQ accumulator (default backward).
size_t bwd_workspace_bytes(int B, int S, int nh, int hd, bool fused_dq);
BwdWorkspace bwd_workspace_carve(void *base, int B, int S, int nh, int hd);

// bf16 tcgen05 path (hd in {32, 64}).
cudaError_t launch_fwd_bf16(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                            __nv_bfloat16 *o, float *lse, int B, int S, int nh, int nkv, int hd,
                            float scale, int *status, uint64_t timeout_ns, cudaStream_t stream);

cudaError_t launch_bwd_preprocess(const __nv_bfloat16 *o, const __nv_bfloat16 *dO,
                                  const float *lse, int B, int S, int nh, int hd, float scale,
                                  const BwdWorkspace &ws, bool fused_dq, cudaStream_t stream);

// dK and dV (key-stationary), and with mdq non-null also dQ added into the fp32
// accumulator. maux: bf16 map over the auxiliary rows (box = 16 columns x 128 rows,
// 32-byte swizzle); mdq: fp32 map over the dQ accumulator (box = half a head row x 128
// rows), used for TMA reduce-adds.
cudaError_t launch_bwd_main_bf16(const CUtensorMap &mq, const CUtensorMap &mk,
                                 const CUtensorMap &mv, const CUtensorMap &mdo,
                                 const CUtensorMap &maux, const CUtensorMap *mdq,
                                 __nv_bfloat16 *dk, __nv_bfloat16 *dv,
                                 int B, int S, int nh, int nkv, int hd, float scale, int *status,
                                 uint64_t timeout_ns, cudaStream_t stream);

// Small problems: the backward with dQ resident in tensor memory (one CTA per (batch, kv
// head), all its key tiles; dQ accumulated over them in a fixed order and written once in
// bf16). Needs the workspace of the preprocess without the dQ accumulator. Usable when
// bwd_resident_dq_ok(S, nh, nkv, hd): hd in {32, 64} and group * ceil(S / 128) * hd <= 64.
bool bwd_resident_dq_ok(int S, int nh, int nkv, int hd);
cudaError_t launch_bwd_main_resident_bf16(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                                          const CUtensorMap &mdo, const CUtensorMap &maux, __nv_bfloat16 *dk,
                                          __nv_bfloat16 *dv, __nv_bfloat16 *dq, int B, int S, int nh, int nkv,
                                          int hd, float scale, int *status, uint64_t timeout_ns,
                                          cudaStream_t stream);

cudaError_t launch_dq_convert(const float *dqacc, __nv_bfloat16 *dq, size_t n_elems,
                              float scale, cudaStream_t stream);

// dQ of the deterministic backward (query-stationary), written in bf16; lse is the
// forward's [B, S, nh] output.
cudaError_t launch_bwd_dq_bf16(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                               const CUtensorMap &mdo, const float *lse, const BwdWorkspace &ws,
                               __nv_bfloat16 *dq, int B, int S, int nh, int nkv, int hd, float scale,
                               int *status, uint64_t timeout_ns, cudaStream_t stream);

// Decode (one query per sequence against its T cached keys/values), bf16, hd in
// {32, 64, 128}, group = nh / nkv <= kMaxDecodeGroup. mk, mv: maps over the caches as
// make_map builds them for [B, T, nkv, hd]. A chunk is decode_chunk_keys(hd) keys (32 KB
// of K); the workspace holds each chunk's (max, sum, partial O) per query head:
// decode_workspace_bytes() bytes.
constexpr int kMaxDecodeGroup = 16;
int decode_chunk_keys(int hd);
size_t decode_workspace_bytes(int B, int T, int nh, int hd);
// Key runs per (batch, kv head) that launch_decode_bf16 uses on a GPU with `sms` SMs
// (1: one CTA streams a whole cache and writes O; more: per-run records and a combine).
int decode_runs(int B, int T, int nh, int nkv, int hd, int sms);
cudaError_t launch_decode_bf16(const CUtensorMap &mk, const CUtensorMap &mv, const __nv_bfloat16 *q,
                               __nv_bfloat16 *o, float *lse, int B, int T, int nh, int nkv, int hd, float scale,
                               void *workspace, int *status, uint64_t timeout_ns, cudaStream_t stream);

// fp32 CUDA-core path (hd <= 128).
cudaError_t launch_fwd_f32(const float *q, const float *k, const float *v, float *o, float *lse,
                           int B, int S, int nh, int nkv, int hd, float scale,
                           cudaStream_t stream);
cudaError_t launch_bwd_f32(const float *q, const float *k, const float *v, const float *o,
                           const float *dO, const float *lse, float *dq, float *dk, float *dv,
                           int B, int S, int nh, int nkv, int hd, float scale,
                           cudaStream_t stream);

}  // namespace xattn
