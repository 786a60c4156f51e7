// fp32 mode of fused causal attention with grouped KV heads, on the CUDA cores in IEEE
// fp32 (no TF32 rounding of operands).
//
// Same method as the bf16 path (xtrain "演进总览" / docs/evolution.md, rows T14 and
// T15): an online softmax over the keys (the scores are never stored), per-row LSE,
// and a backward that recomputes the scores and uses D_i = dO_i . O_i. The gradient of
// a kv head is accumulated over its query group in a fixed order with no atomics.
//
// One warp per output row: lane l holds head dimensions l, l+32, l+64, l+96 (hd <= 128),
// dot products are warp shuffle reductions. Key/query rows are streamed through the warp
// in blocks of 32 so that each lane computes one score of the block at a time.
#include "xattn_internal.h"

namespace xattn {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kMaxSlots = 4;  // hd <= 32 * kMaxSlots

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// Row-dot of a lane-distributed vector with a row in global memory.
__device__ __forceinline__ float row_dot(const float (&x)[kMaxSlots], const float *row, int hd, int lane) {
  float acc = 0.f;
#pragma unroll
  for (int s = 0; s < kMaxSlots; ++s) {
    const int d = lane + 32 * s;
    if (d < hd) acc = fmaf(x[s], row[d], acc);
  }
  return warp_sum(acc);
}

__device__ __forceinline__ void load_row(float (&x)[kMaxSlots], const float *row, int hd, int lane) {
#pragma unroll
  for (int s = 0; s < kMaxSlots; ++s) {
    const int d = lane + 32 * s;
    x[s] = d < hd ? row[d] : 0.f;
  }
}

// Forward: warp per (b, i, h). Online softmax over keys j <= i.
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    fwd_f32_kernel(const float *__restrict__ q, const float *__restrict__ k,
                   const float *__restrict__ v, float *__restrict__ o, float *__restrict__ lse,
                   int B, int S, int nh, int nkv, int hd, float scale) {
  const long long w = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (w >= static_cast<long long>(B) * S * nh) return;
  const int h = static_cast<int>(w % nh);
  const int i = static_cast<int>((w / nh) % S);
  const int b = static_cast<int>(w / (static_cast<long long>(nh) * S));
  const int kvh = h / (nh / nkv);
  float qi[kMaxSlots], acc[kMaxSlots] = {0.f, 0.f, 0.f, 0.f};
  load_row(qi, q + w * hd, hd, lane);
  float mrow = -INFINITY, lrow = 0.f;
  for (int j = 0; j <= i; ++j) {
    const size_t kv_row = ((static_cast<size_t>(b) * S + j) * nkv + kvh) * hd;
    const float s = scale * row_dot(qi, k + kv_row, hd, lane);
    const float mnew = fmaxf(mrow, s);
    const float alpha = expf(mrow - mnew);  // 0 on the first key
    const float p = expf(s - mnew);
    lrow = lrow * alpha + p;
#pragma unroll
    for (int sl = 0; sl < kMaxSlots; ++sl) {
      const int d = lane + 32 * sl;
      acc[sl] = acc[sl] * alpha + (d < hd ? p * v[kv_row + d] : 0.f);
    }
    mrow = mnew;
  }
  const float inv = 1.f / lrow;
#pragma unroll
  for (int sl = 0; sl < kMaxSlots; ++sl) {
    const int d = lane + 32 * sl;
    if (d < hd) o[w * hd + d] = acc[sl] * inv;
  }
  if (lane == 0) lse[w] = mrow + logf(lrow);
}

// dQ: warp per query row (b, i, h). dQ_i = scale sum_{j<=i} P_ij (dO_i.v_j - D_i) k_j.
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    bwd_dq_f32_kernel(const float *__restrict__ q, const float *__restrict__ k,
                      const float *__restrict__ v, const float *__restrict__ o,
                      const float *__restrict__ dO, const float *__restrict__ lse,
                      float *__restrict__ dq, int B, int S, int nh, int nkv, int hd, float scale) {
  const long long w = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (w >= static_cast<long long>(B) * S * nh) return;
  const int h = static_cast<int>(w % nh);
  const int i = static_cast<int>((w / nh) % S);
  const int b = static_cast<int>(w / (static_cast<long long>(nh) * S));
  const int kvh = h / (nh / nkv);
  float qi[kMaxSlots], doi[kMaxSlots], oi[kMaxSlots], acc[kMaxSlots] = {0.f, 0.f, 0.f, 0.f};
  load_row(qi, q + w * hd, hd, lane);
  load_row(doi, dO + w * hd, hd, lane);
  load_row(oi, o + w * hd, hd, lane);
  float Di = 0.f;
#pragma unroll
  for (int s = 0; s < kMaxSlots; ++s) Di = fmaf(doi[s], oi[s], Di);
  Di = warp_sum(Di);
  const float L = lse[w];
  for (int j = 0; j <= i; ++j) {
    const size_t kv_row = ((static_cast<size_t>(b) * S + j) * nkv + kvh) * hd;
    const float p = expf(scale * row_dot(qi, k + kv_row, hd, lane) - L);
    const float dp = row_dot(doi, v + kv_row, hd, lane);
    const float ds = p * (dp - Di);
#pragma unroll
    for (int sl = 0; sl < kMaxSlots; ++sl) {
      const int d = lane + 32 * sl;
      if (d < hd) acc[sl] = fmaf(ds, k[kv_row + d], acc[sl]);
    }
  }
#pragma unroll
  for (int sl = 0; sl < kMaxSlots; ++sl) {
    const int d = lane + 32 * sl;
    if (d < hd) dq[w * hd + d] = scale * acc[sl];
  }
}

// dK, dV: warp per key row (b, j, kvh); loops over the query group r = 0.. in order
// and over queries i >= j.
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    bwd_dkdv_f32_kernel(const float *__restrict__ q, const float *__restrict__ k,
                        const float *__restrict__ v, const float *__restrict__ o,
                        const float *__restrict__ dO, const float *__restrict__ lse,
                        float *__restrict__ dk, float *__restrict__ dv, int B, int S, int nh,
                        int nkv, int hd, float scale) {
  const long long w = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (w >= static_cast<long long>(B) * S * nkv) return;
  const int kvh = static_cast<int>(w % nkv);
  const int j = static_cast<int>((w / nkv) % S);
  const int b = static_cast<int>(w / (static_cast<long long>(nkv) * S));
  const int group = nh / nkv;
  float kj[kMaxSlots], vj[kMaxSlots];
  float ak[kMaxSlots] = {0.f, 0.f, 0.f, 0.f}, av[kMaxSlots] = {0.f, 0.f, 0.f, 0.f};
  load_row(kj, k + w * hd, hd, lane);
  load_row(vj, v + w * hd, hd, lane);
  for (int r = 0; r < group; ++r) {
    const int h = kvh * group + r;
    for (int i = j; i < S; ++i) {
      const size_t qrow = ((static_cast<size_t>(b) * S + i) * nh + h);
      const float *dOi = dO + qrow * hd;
      const float *oi = o + qrow * hd;
      const float *qi = q + qrow * hd;
      const float p = expf(scale * row_dot(kj, qi, hd, lane) - lse[qrow]);
      const float dp = row_dot(vj, dOi, hd, lane);
      float part = 0.f;
#pragma unroll
      for (int s = 0; s < kMaxSlots; ++s) {
        const int d = lane + 32 * s;
        if (d < hd) part = fmaf(dOi[d], oi[d], part);
      }
      const float Di = warp_sum(part);
      const float ds = p * (dp - Di);
#pragma unroll
      for (int sl = 0; sl < kMaxSlots; ++sl) {
        const int d = lane + 32 * sl;
        if (d < hd) {
          ak[sl] = fmaf(ds, qi[d], ak[sl]);
          av[sl] = fmaf(p, dOi[d], av[sl]);
        }
      }
    }
  }
#pragma unroll
  for (int sl = 0; sl < kMaxSlots; ++sl) {
    const int d = lane + 32 * sl;
    if (d < hd) {
      dk[w * hd + d] = scale * ak[sl];
      dv[w * hd + d] = av[sl];
    }
  }
}

unsigned warps_grid(long long warps) {
  return static_cast<unsigned>((warps + kWarpsPerBlock - 1) / kWarpsPerBlock);
}

}  // namespace

cudaError_t launch_fwd_f32(const float *q, const float *k, const float *v, float *o, float *lse,
                           int B, int S, int nh, int nkv, int hd, float scale,
                           cudaStream_t stream) {
  const long long rows = static_cast<long long>(B) * S * nh;
  fwd_f32_kernel<<<warps_grid(rows), kWarpsPerBlock * 32, 0, stream>>>(q, k, v, o, lse, B, S, nh,
                                                                        nkv, hd, scale);
  return cudaGetLastError();
}

cudaError_t launch_bwd_f32(const float *q, const float *k, const float *v, const float *o,
                           const float *dO, const float *lse, float *dq, float *dk, float *dv,
                           int B, int S, int nh, int nkv, int hd, float scale,
                           cudaStream_t stream) {
  const long long qrows = static_cast<long long>(B) * S * nh;
  const long long krows = static_cast<long long>(B) * S * nkv;
  bwd_dq_f32_kernel<<<warps_grid(qrows), kWarpsPerBlock * 32, 0, stream>>>(q, k, v, o, dO, lse, dq,
                                                                           B, S, nh, nkv, hd, scale);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  bwd_dkdv_f32_kernel<<<warps_grid(krows), kWarpsPerBlock * 32, 0, stream>>>(
      q, k, v, o, dO, lse, dk, dv, B, S, nh, nkv, hd, scale);
  return cudaGetLastError();
}

}  // namespace xattn
