// Forward of fused causal attention with grouped KV heads on sm_103a tensor cores.
//
// Method (xtrain "演进总览" / docs/evolution.md, phase table row T14): one kernel, an
// online softmax tiled over KV, the S x S scores never leave the chip, and each row's
// log-sum-exp is kept for the backward. Grouped KV heads (row T15): query head h reads
// kv head h / group.
//
// GB300 mapping (one CTA per 128-row query tile, 12 warps):
//   warp 0     : TMA producer. Q tile once; K/V tiles into a 3-stage shared-memory ring.
//   warp 1     : allocates TMEM; one lane issues tcgen05.mma:
//                  S_n  = Q K_n^T  (A, B from shared memory)      -> TMEM, double-buffered
//                  O   += P_n V_n  (A = P from TMEM, B from smem) -> TMEM accumulator
//   warps 4-11 : softmax, one thread per query row (TMEM lane) and key-column half.
//                Loads S_n, applies the causal mask on the diagonal tile, keeps the
//                running max and sum in fp32 (log2 domain), writes P_n (bf16) to TMEM,
//                and rescales O only when the running max grows by more than 2^8 (the
//                stale max is exact because the final normalisation uses the same max).
//                Epilogue: O / l in bf16 and LSE = (m + log2 l) ln 2.
// Causal tile skipping: query tile m visits key tiles 0..m only. Tiles are issued
// longest first (m descending) so the last wave holds short tiles.
#include "sm103_ptx.cuh"
#include "xattn_internal.h"

namespace xattn {
namespace {

constexpr int kFwdThreads = 384;  // 12 warps, see the role map in the kernel
constexpr int kFwdStages = 3;

template <int HD>
struct FwdLayout {
  static constexpr uint32_t kRowBytes = HD * 2;
  static constexpr uint32_t kTileBytes = kTileRows * kRowBytes;
  static constexpr uint32_t kSwizzle = (HD == 64) ? kSwizzle128 : kSwizzle64;
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = kQ + kTileBytes;
  static constexpr uint32_t kV = kK + kFwdStages * kTileBytes;
  static constexpr uint32_t kRed = kV + kFwdStages * kTileBytes;  // max [2][2][128], l [2][128]
  static constexpr uint32_t kBars = kRed + 3 * 1024;
  // barriers: q_full, full[S], empty[S], s_full[2], p_full[2], o_done, mma_final, pair[4]
  static constexpr int kNumBars = 1 + 2 * kFwdStages + 2 + 2 + 2 + 4;
  static constexpr uint32_t kMisc = kBars + 8 * kNumBars;
  static constexpr uint32_t kUsed = kMisc + 32;
  // Ask for enough shared memory that one CTA occupies an SM: each CTA holds all 512
  // TMEM columns, so a second resident CTA would only spin in tcgen05.alloc.
  static constexpr uint32_t kDynBytes = (kUsed + 1024 > 120 * 1024) ? kUsed + 1024 : 120 * 1024;
};

// Warp-uniform bounded wait: every lane waits, then all agree.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtl &ctl) {
  const bool ok = mbar_wait(bar, parity, ctl);
  return __all_sync(0xffffffffu, ok);
}

// TMEM <-> registers for half an O row (HD/2 columns).
template <int N>
__device__ __forceinline__ void tmem_ld_half(uint32_t taddr, uint32_t *r) {
  if constexpr (N == 32) tmem_ld_x32(taddr, r);
  else tmem_ld_x16(taddr, r);
}
template <int N>
__device__ __forceinline__ void tmem_st_half(uint32_t taddr, const uint32_t *r) {
  if constexpr (N == 32) tmem_st_x32(taddr, r);
  else tmem_st_x16(taddr, r);
}

// Role map (12 warps):
//   warp 0    : TMA producer (Q once, K/V through a 3-stage ring)
//   warp 1    : TMEM owner and MMA issuer
//   warps 2-3 : idle
//   warps 4-11: softmax, one thread per query row; warps 4-7 take key columns 0-63 of
//               each 128-column tile and warps 8-11 columns 64-127, so each SM
//               sub-partition interleaves two softmax warps. The two halves of a row
//               exchange their partial maxima through shared memory each tile.
// TMEM columns: S double buffer [0,128) [128,256) fp32 | O [256,256+HD) fp32 |
//               P double buffer [320,384) [384,448) bf16
template <int HD>
__global__ void __maxnreg__(168)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                    const __grid_constant__ CUtensorMap mv, __nv_bfloat16 *__restrict__ o,
                    float *__restrict__ lse, int B, int S, int nh, int nkv, float scale_log2,
                    int *status, unsigned long long timeout_ns) {
  using L = FwdLayout<HD>;
  constexpr int kHalf = HD / 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Tile of this CTA, longest first.
  const int num_m = (S + kTileRows - 1) / kTileRows;
  const int BH = B * nh;
  const int m = num_m - 1 - static_cast<int>(blockIdx.x) / BH;
  const int bh = static_cast<int>(blockIdx.x) % BH;
  const int b = bh / nh, h = bh % nh;
  const int kvh = h / (nh / nkv);
  const int n_kv = m + 1;

  const uint32_t sQ = smem_u32(smem + L::kQ);
  const uint32_t sK = smem_u32(smem + L::kK);
  const uint32_t sV = smem_u32(smem + L::kV);
  float *red_max = reinterpret_cast<float *>(smem + L::kRed);          // [2 tiles][2 halves][128]
  float *red_l = reinterpret_cast<float *>(smem + L::kRed + 2048);     // [2 halves][128]
  const uint32_t bar0 = smem_u32(smem + L::kBars);
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  const uint32_t q_full = bar(0);
  auto full = [&](int s) { return bar(1 + s); };
  auto empty = [&](int s) { return bar(1 + kFwdStages + s); };
  auto s_full = [&](int x) { return bar(1 + 2 * kFwdStages + x); };
  auto p_full = [&](int x) { return bar(3 + 2 * kFwdStages + x); };
  const uint32_t o_done = bar(5 + 2 * kFwdStages);
  const uint32_t mma_final = bar(6 + 2 * kFwdStages);
  auto pair_bar = [&](int q) { return bar(7 + 2 * kFwdStages + q); };
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMisc + 16);
  const WaitCtl ctl{abort_flag, status, timeout_ns};

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(q_full, 1);
    for (int s = 0; s < kFwdStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(s_full(x), 1);
      mbar_init(p_full(x), 256);
    }
    mbar_init(o_done, 1);
    mbar_init(mma_final, 1);
    for (int q = 0; q < 4; ++q) mbar_init(pair_bar(q), 64);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mq);
    tma_prefetch_desc(&mk);
    tma_prefetch_desc(&mv);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t tS[2] = {tmem, tmem + 128};
  const uint32_t tO = tmem + 256;
  const uint32_t tP[2] = {tmem + 320, tmem + 384};

  if (warp == 0) {
    // ---------------- TMA producer (converged warp, one elected lane issues) ----------------
    mbar_expect_tx_elect(q_full, L::kTileBytes);
    tma_load_4d_elect(sQ, &mq, q_full, 0, h, m * kTileRows, b);
    int issued = 0;
    for (int n = 0, s = 0, ph = 0; n < n_kv; ++n) {
      if (!warp_wait(empty(s), ph ^ 1, ctl)) break;
      mbar_expect_tx_elect(full(s), 2 * L::kTileBytes);
      tma_load_4d_elect(sK + s * L::kTileBytes, &mk, full(s), 0, kvh, n * kTileRows, b);
      tma_load_4d_elect(sV + s * L::kTileBytes, &mv, full(s), 0, kvh, n * kTileRows, b);
      issued = n + 1;
      if (++s == kFwdStages) { s = 0; ph ^= 1; }
    }
    // Let every copy in flight land before the CTA can exit.
    mbar_drain(q_full, 0, ctl);
    for (int n = (issued > kFwdStages ? issued - kFwdStages : 0); n < issued; ++n)
      mbar_drain(full(n % kFwdStages), (n / kFwdStages) & 1, ctl);
  } else if (warp == 1) {
    // ---------------- MMA issuer (converged warp, one elected lane issues) ----------------
    constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t idesc_pv = idesc_bf16_f32(128, HD, false, true);
    constexpr uint32_t kStageDesc = L::kTileBytes >> 4;        // stage stride, descriptor units
    constexpr uint32_t kVStep = (16 * L::kRowBytes) >> 4;      // 16 key rows of V
    // Descriptors are built once; a K step of 16 elements is +32 bytes (+2) within the
    // swizzled K-major rows of Q and K, and +16 rows of the MN-major V tile.
    const uint64_t dQ = smem_desc(sQ, 16, 8 * L::kRowBytes, L::kSwizzle);
    const uint64_t dK = smem_desc(sK, 16, 8 * L::kRowBytes, L::kSwizzle);
    const uint64_t dV = smem_desc(sV, 8192, 8 * L::kRowBytes, L::kSwizzle);
    auto issue_qk = [&](uint32_t d, int s) {
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk)
        mma_ss_elect(d, dQ + 2 * kk, dK + s * kStageDesc + 2 * kk, idesc_qk, kk > 0);
    };
    bool ok = warp_wait(q_full, 0, ctl) && warp_wait(full(0), 0, ctl);
    if (ok) {
      tc_fence_after();
      issue_qk(tS[0], 0);
      mma_commit_elect(s_full(0));
    }
    for (int n = 0, s = 0, s1 = 1 % kFwdStages, ph1 = (1 / kFwdStages) & 1; ok && n < n_kv; ++n) {
      if (n + 1 < n_kv) {
        // S(n+1) goes into the buffer of S(n-1), which the softmax finished reading
        // before it signalled P(n-1) (waited for in the previous iteration).
        if (!warp_wait(full(s1), ph1, ctl)) break;
        tc_fence_after();
        issue_qk(tS[(n + 1) & 1], s1);
        mma_commit_elect(s_full((n + 1) & 1));
      }
      if (!warp_wait(p_full(n & 1), (n >> 1) & 1, ctl)) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kTileRows / 16; ++kk)
        mma_ts_elect(tO, tP[n & 1] + kk * 8, dV + s * kStageDesc + kk * kVStep, idesc_pv,
                     (n > 0 || kk > 0) ? 1u : 0u);
      mma_commit_elect(empty(s));
      mma_commit_elect(o_done);
      if (++s == kFwdStages) s = 0;
      if (++s1 == kFwdStages) { s1 = 0; ph1 ^= 1; }
    }
    mma_commit_elect(mma_final);
    mbar_drain(mma_final, 0, ctl);
  } else if (warp >= 4) {
    // ---------------- softmax + epilogue ----------------
    const int g = (warp - 4) >> 2;           // key-column half of every tile
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t pbar = pair_bar(quarter);
    uint32_t pair_phase = 0;
    float mrow = -INFINITY, lpart = 0.f;
    bool ok = true;
    for (int n = 0; n < n_kv; ++n) {
      if (!warp_wait(s_full(n & 1), (n >> 1) & 1, ctl)) { ok = false; break; }
      tc_fence_after();
      uint32_t r[64];
      tmem_ld_x32(tS[n & 1] + lane_off + 64 * g, r);
      tmem_ld_x32(tS[n & 1] + lane_off + 64 * g + 32, r + 32);
      tmem_wait_ld();
      reg_fence<64>(r);
      // Causal mask (diagonal tile only; the branch is uniform across the CTA).
      if (n == m) {
        const int col0 = 64 * g;
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (col0 + c > row) r[c] = __float_as_uint(-INFINITY);
      }
      // Row maximum of the raw scores (scale > 0, so the scaled maximum is its image).
      float mx4[4];
#pragma unroll
      for (int a = 0; a < 4; ++a)
        mx4[a] = fmax3(__uint_as_float(r[2 * a]), __uint_as_float(r[2 * a + 1]), -INFINITY);
#pragma unroll
      for (int c = 8; c < 64; c += 2)
        mx4[(c >> 1) & 3] = fmax3(mx4[(c >> 1) & 3], __uint_as_float(r[c]), __uint_as_float(r[c + 1]));
      const float pmax = fmax3(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3]));
      // Row maximum across the two column halves (double-buffered by tile parity).
      red_max[((n & 1) * 2 + g) * 128 + row] = pmax;
      mbar_arrive(pbar);
      if (!warp_wait(pbar, pair_phase & 1, ctl)) { ok = false; break; }
      ++pair_phase;
      const float mx = fmaxf(pmax, red_max[((n & 1) * 2 + (g ^ 1)) * 128 + row]) * scale_log2;
      // Conditional rescaling: keep the stale max unless some row of the warp grew by
      // more than 2^8; the decision is per warp because TMEM loads/stores are collective,
      // and both halves of a row reach the same decision from the same maxima.
      const float mnew = fmaxf(mrow, mx);
      const bool rescale = __any_sync(0xffffffffu, mnew > mrow + 8.0f);
      const float m_use = rescale ? mnew : mrow;
      const float alpha = rescale ? ex2_approx(mrow - mnew) : 1.f;
      const float neg_m = -m_use;
      float ps[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        float x0, x1;
        ffma2(x0, x1, __uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]), scale_log2,
              scale_log2, neg_m, neg_m);
        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
        const int a = (e & 1) * 2;
        fadd2(ps[a], ps[a + 1], ps[a], ps[a + 1], p0, p1);
        pk[e] = pack_bf16x2(p0, p1);
      }
      // P(n) goes into the buffer PV(n-2) read; that PV was waited for last iteration.
      tmem_st_x16(tP[n & 1] + lane_off + 32 * g, pk);
      tmem_st_x16(tP[n & 1] + lane_off + 32 * g + 16, pk + 16);
      // PV(n-1) is waited for on every tile, not only when rescaling: a parity wait is
      // only unambiguous if the waiter has seen every earlier phase of the barrier.
      if (n > 0) {
        if (!warp_wait(o_done, (n - 1) & 1, ctl)) { ok = false; break; }
        tc_fence_after();
        if (rescale) {
          uint32_t ov[kHalf];
          tmem_ld_half<kHalf>(tO + lane_off + kHalf * g, ov);
          tmem_wait_ld();
          reg_fence<kHalf>(ov);
#pragma unroll
          for (int e = 0; e < kHalf; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
          tmem_st_half<kHalf>(tO + lane_off + kHalf * g, ov);
        }
      }
      lpart = lpart * alpha + ((ps[0] + ps[1]) + (ps[2] + ps[3]));
      mrow = m_use;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_full(n & 1));
    }
    if (ok && warp_wait(o_done, (n_kv - 1) & 1, ctl)) {
      tc_fence_after();
      red_l[g * 128 + row] = lpart;
      mbar_arrive(pbar);
      if (warp_wait(pbar, pair_phase & 1, ctl)) {
        const float l = lpart + red_l[(g ^ 1) * 128 + row];
        const int i = m * kTileRows + row;
        const float inv = 1.f / l;
        uint32_t ov[kHalf];
        tmem_ld_half<kHalf>(tO + lane_off + kHalf * g, ov);
        tmem_wait_ld();
        reg_fence<kHalf>(ov);
        if (i < S) {
          __nv_bfloat16 *orow = o + (static_cast<size_t>(b) * S + i) * nh * HD +
                                static_cast<size_t>(h) * HD + kHalf * g;
          uint4 *dst = reinterpret_cast<uint4 *>(orow);
#pragma unroll
          for (int e = 0; e < kHalf / 8; ++e)
            dst[e] = make_uint4(
                pack_bf16x2(__uint_as_float(ov[8 * e + 0]) * inv, __uint_as_float(ov[8 * e + 1]) * inv),
                pack_bf16x2(__uint_as_float(ov[8 * e + 2]) * inv, __uint_as_float(ov[8 * e + 3]) * inv),
                pack_bf16x2(__uint_as_float(ov[8 * e + 4]) * inv, __uint_as_float(ov[8 * e + 5]) * inv),
                pack_bf16x2(__uint_as_float(ov[8 * e + 6]) * inv, __uint_as_float(ov[8 * e + 7]) * inv));
          if (g == 0) lse[(static_cast<size_t>(b) * S + i) * nh + h] = (mrow + __log2f(l)) * kLn2;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int HD>
cudaError_t launch_fwd_hd(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                          __nv_bfloat16 *o, float *lse, int B, int S, int nh, int nkv, float scale,
                          int *status, uint64_t timeout_ns, cudaStream_t stream) {
  using L = FwdLayout<HD>;
  cudaError_t err = cudaFuncSetAttribute(attn_fwd_kernel<HD>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kDynBytes);
  if (err != cudaSuccess) return err;
  const int num_m = (S + kTileRows - 1) / kTileRows;
  const unsigned grid = static_cast<unsigned>(B) * nh * num_m;
  attn_fwd_kernel<HD><<<grid, kFwdThreads, L::kDynBytes, stream>>>(
      mq, mk, mv, o, lse, B, S, nh, nkv, scale * kLog2e, status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_bf16(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                            __nv_bfloat16 *o, float *lse, int B, int S, int nh, int nkv, int hd,
                            float scale, int *status, uint64_t timeout_ns, cudaStream_t stream) {
  if (hd == 64)
    return launch_fwd_hd<64>(mq, mk, mv, o, lse, B, S, nh, nkv, scale, status, timeout_ns, stream);
  if (hd == 32)
    return launch_fwd_hd<32>(mq, mk, mv, o, lse, B, S, nh, nkv, scale, status, timeout_ns, stream);
  return cudaErrorInvalidValue;
}

}  // namespace xattn
