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

// Rows of the per-(batch, head) workspace vectors, padded to whole tiles.
__host__ __device__ inline int padded_rows(int S) { return (S + kTileRows - 1) / kTileRows * kTileRows; }

struct BwdWorkspace {
  float *D;      // [B, nh, S_pad]  -D_i = -(dO_i . O_i) ; zero in pad rows
  float *lse2;   // [B, nh, S_pad]  -LSE_i * log2(e) ; -inf in pad rows
  float *dqacc;  // [B, S, nh, hd]  fp32 dQ accumulator
};

size_t bwd_workspace_bytes(int B, int S, int nh, int hd);
BwdWorkspace bwd_workspace_carve(void *base, int B, int S, int nh, int hd);

// bf16 tcgen05 path (hd in {32, 64}).
cudaError_t launch_fwd_bf16(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                            __nv_bfloat16 *o, float *lse, int B, int S, int nh, int nkv, int hd,
                            float scale, int *status, uint64_t timeout_ns, cudaStream_t stream);

cudaError_t launch_bwd_preprocess(const __nv_bfloat16 *o, const __nv_bfloat16 *dO,
                                  const float *lse, int B, int S, int nh, int hd,
                                  const BwdWorkspace &ws, cudaStream_t stream);

// mdq: fp32 map over the dQ accumulator (box = half a head row x 128 rows), used for
// TMA reduce-adds.
cudaError_t launch_bwd_main_bf16(const CUtensorMap &mq, const CUtensorMap &mk,
                                 const CUtensorMap &mv, const CUtensorMap &mdo,
                                 const CUtensorMap &mdq,
                                 const BwdWorkspace &ws, __nv_bfloat16 *dk, __nv_bfloat16 *dv,
                                 int B, int S, int nh, int nkv, int hd, float scale, int *status,
                                 uint64_t timeout_ns, cudaStream_t stream);

cudaError_t launch_dq_convert(const float *dqacc, __nv_bfloat16 *dq, size_t n_elems,
                              cudaStream_t stream);

// fp32 CUDA-core path (hd <= 128).
cudaError_t launch_fwd_f32(const float *q, const float *k, const float *v, float *o, float *lse,
                           int B, int S, int nh, int nkv, int hd, float scale,
                           cudaStream_t stream);
cudaError_t launch_bwd_f32(const float *q, const float *k, const float *v, const float *o,
                           const float *dO, const float *lse, float *dq, float *dk, float *dv,
                           int B, int S, int nh, int nkv, int hd, float scale,
                           cudaStream_t stream);

}  // namespace xattn
