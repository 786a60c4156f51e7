// dQ of the backward of fused causal attention with grouped KV heads on sm_103a.
//
// Method (xtrain "演进总览" / docs/evolution.md, phase table row T14): recompute the
// scores from Q, K and the saved log-sum-exp, use D_i = dO_i . O_i in place of the
// softmax Jacobian. This kernel produces dQ only; dK and dV come from the key-stationary
// kernel in attn_bwd_sm103.cu.
//
// One CTA per (batch, query head h, 128-row query tile m), longest first. Q_m and dO_m
// stay in shared memory, dQ_m accumulates in TMEM over the key tiles n = 0 .. m (causal
// tile skipping) and is written once, in bf16, at the end: no atomics, no fp32
// accumulator in global memory, and a fixed summation order, so dQ is reproducible.
// Per key tile n (K_n, V_n of kv head h / group):
//   S  = Q_m K_n^T            (TMEM, 128 x 128 fp32; A and B from shared memory)
//   dP = dO_m V_n^T           (TMEM, 128 x 128 fp32)
//   P  = exp2(S scale log2e - LSE_i log2e)   (LSE_i and D_i of the thread's query row
//   dS = P (dP - D_i)                          are registers) -> bf16 into TMEM
//   dQ_m += dS K_n            (A = dS from TMEM, B = K_n from shared memory)
// dQ = scale * accumulator (the softmax scale is applied once, at the end).
#include "sm103_ptx.cuh"
#include "xattn_internal.h"

namespace xattn {
namespace {

// 12 warps: 0 TMA producer, 1 TMEM owner + MMA issuer, 2-3 idle, 4-11 two groups of 4
// warps (one per TMEM lane quarter); group g owns key columns [64 g, 64 g + 64) of
// every tile, one query row per thread.
constexpr int kDqThreads = 384;

// hd = 128: two K / V stages (32 KB tiles), and every tile is two 64-column sub-tiles laid
// out like hd = 64 tiles (a 256-byte row does not fit one 128-byte swizzle atom).
template <int HD>
struct DqLayout {
  static constexpr int kStages = HD == 128 ? 2 : 3;                 // K / V stages
  static constexpr uint32_t kRowBytes = HD * 2;
  static constexpr uint32_t kTileBytes = kTileRows * kRowBytes;
  static constexpr uint32_t kAtomBytes = kRowBytes < 128 ? kRowBytes : 128;  // sub-tile row
  static constexpr int kSubTiles = static_cast<int>(kRowBytes / kAtomBytes);
  static constexpr uint32_t kSubBytes = kTileRows * kAtomBytes;
  static constexpr uint32_t kSwizzle = (HD == 32) ? kSwizzle64 : kSwizzle128;
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kdO = kQ + kTileBytes;
  static constexpr uint32_t kK = kdO + kTileBytes;                   // kStages stages
  static constexpr uint32_t kV = kK + kStages * kTileBytes;          // kStages stages
  // barriers: q_full, full[S], empty[S], s_full, s_free, dp_full, dp_free, ds_full,
  //           dq_done, acc_done
  static constexpr int kNumBars = 1 + 2 * kStages + 7;
  static constexpr uint32_t kBars = kV + kStages * kTileBytes;
  static constexpr uint32_t kMisc = kBars + 8 * kNumBars;
  static constexpr uint32_t kUsed = kMisc + 32;
  static constexpr uint32_t kDynBytes = kUsed + 1024;
  static_assert(kDynBytes <= 227 * 1024, "exceeds the opt-in shared memory of one CTA");
};

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtl &ctl) {
  const bool ok = mbar_wait(bar, parity, ctl);
  return __all_sync(0xffffffffu, ok);
}

// TMEM columns: S [0,128) fp32 | dP [128,256) fp32 | dS bf16 [256,320) | dQ [320,320+HD)
// (at most 448 columns, hd = 128 included).
// S and dP are each released (s_free, dp_free) as soon as both groups have loaded their
// columns, so the next tile's products overlap this tile's arithmetic; the dS slot is
// rewritten only after dQ(n-1) has read it (dq_done).
template <int HD>
__global__ void __maxnreg__(168)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                       const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
                       const float *__restrict__ lse, const float *__restrict__ Dvec,
                       __nv_bfloat16 *__restrict__ dq, int B, int S, int nh, int nkv, float scale,
                       int *status, unsigned long long timeout_ns) {
  using L = DqLayout<HD>;
  constexpr int kDqStages = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Unit of this CTA: query tile m (most key tiles first), batch b, query head h.
  const int num_m = (S + kTileRows - 1) / kTileRows;
  const int BH = B * nh;
  const int m = num_m - 1 - static_cast<int>(blockIdx.x) / BH;
  const int bh = static_cast<int>(blockIdx.x) % BH;
  const int b = bh / nh, h = bh % nh;
  const int kvh = h / (nh / nkv);
  const int T = m + 1;                      // key tiles n = 0 .. m

  const uint32_t sQ = smem_u32(smem + L::kQ);
  const uint32_t sdO = smem_u32(smem + L::kdO);
  const uint32_t sK = smem_u32(smem + L::kK);
  const uint32_t sV = smem_u32(smem + L::kV);
  const uint32_t bar0 = smem_u32(smem + L::kBars);
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  const uint32_t q_full = bar(0);
  auto full = [&](int s) { return bar(1 + s); };
  auto empty = [&](int s) { return bar(1 + kDqStages + s); };
  constexpr int kB = 1 + 2 * kDqStages;
  const uint32_t s_full = bar(kB + 0), s_free = bar(kB + 1), dp_full = bar(kB + 2);
  const uint32_t dp_free = bar(kB + 3), ds_full = bar(kB + 4), dq_done = bar(kB + 5);
  const uint32_t acc_done = bar(kB + 6);
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMisc + 16);
  const WaitCtl ctl{abort_flag, status, timeout_ns};

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(q_full, 1);
    for (int s = 0; s < kDqStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, 256);
    mbar_init(dp_full, 1);
    mbar_init(dp_free, 256);
    mbar_init(ds_full, 256);
    mbar_init(dq_done, 1);
    mbar_init(acc_done, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mq);
    tma_prefetch_desc(&mk);
    tma_prefetch_desc(&mv);
    tma_prefetch_desc(&mdo);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_dep_launch();
  grid_dep_wait();
  const uint32_t tmem = *tmem_holder;
  const uint32_t tS = tmem, tdP = tmem + 128, tdS = tmem + 256, tdQ = tmem + 320;
  // One 128-row tile of a [B, S, heads, hd] tensor: one TMA box per 64-column sub-tile.
  // Debug builds check the tile's coordinates and that it lands inside the tile region.
  auto load_tile = [&](uint32_t dst, const CUtensorMap *map, uint32_t bar, int head, int row0, int bb) {
    XATTN_DCHECK(head >= 0 && head < nh && row0 >= 0 && row0 < (S + kTileRows - 1) / kTileRows * kTileRows &&
                     row0 % kTileRows == 0 && bb >= 0 && bb < B && dst >= smem_u32(smem) &&
                     dst + L::kTileBytes <= smem_u32(smem + L::kBars),
                 status);
#pragma unroll
    for (int c = 0; c < L::kSubTiles; ++c) {
      XATTN_DCHECK((c * static_cast<int>(L::kAtomBytes / 2)) % 8 == 0 && c * static_cast<int>(L::kAtomBytes / 2) < HD,
                   status);
      tma_load_4d_elect(dst + c * L::kSubBytes, map, bar, c * static_cast<int>(L::kAtomBytes / 2), head, row0, bb);
    }
  };

  if (warp == 0) {
    // ---------------- TMA producer (converged warp, one elected lane issues) ----------------
    mbar_expect_tx_elect(q_full, 2 * L::kTileBytes);
    load_tile(sQ, &mq, q_full, h, m * kTileRows, b);
    load_tile(sdO, &mdo, q_full, h, m * kTileRows, b);
    int issued = 0;
    for (int n = 0, s = 0, use = 0; n < T; ++n) {
      if (!warp_wait(empty(s), (use & 1) ^ 1, ctl)) break;
      mbar_expect_tx_elect(full(s), 2 * L::kTileBytes);
      XATTN_DCHECK(kvh < nkv && s < kDqStages, status);
      load_tile(sK + s * L::kTileBytes, &mk, full(s), kvh, n * kTileRows, b);
      load_tile(sV + s * L::kTileBytes, &mv, full(s), kvh, n * kTileRows, b);
      issued = n + 1;
      if (++s == kDqStages) { s = 0; ++use; }
    }
    // Every load has landed before the CTA can exit (the consumers may have given up).
    mbar_drain(q_full, 0, ctl);
    for (int n = (issued > kDqStages ? issued - kDqStages : 0); n < issued; ++n)
      mbar_drain(full(n % kDqStages), (n / kDqStages) & 1, ctl);
  } else if (warp == 1) {
    // ---------------- MMA issuer (converged warp, one elected lane issues) ----------------
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);  // S, dP
    // dQ (B = K, MN-major): one N = 64 product per 64-column sub-tile at hd = 128.
    constexpr uint32_t idesc_dq = idesc_bf16_f32(128, HD / L::kSubTiles, false, true);
    constexpr uint32_t kStageDesc = L::kTileBytes >> 4;
    constexpr uint32_t kSubDesc = L::kSubBytes >> 4;                     // sub-tile stride
    constexpr uint32_t kRowStep = (16 * L::kAtomBytes) >> 4;             // 16 key rows of K
    // K-major operands advance +32 bytes (+2) per 16-element K step (the fifth step
    // starts the second sub-tile); the MN-major K tile (dQ's B: K dimension = keys)
    // advances 16 rows.
    const uint64_t kQ_k = smem_desc(sQ, 16, 8 * L::kAtomBytes, L::kSwizzle);
    const uint64_t kdO_k = smem_desc(sdO, 16, 8 * L::kAtomBytes, L::kSwizzle);
    const uint64_t kK_k = smem_desc(sK, 16, 8 * L::kAtomBytes, L::kSwizzle);
    const uint64_t kV_k = smem_desc(sV, 16, 8 * L::kAtomBytes, L::kSwizzle);
    const uint64_t kK_mn = smem_desc(sK, 8192, 8 * L::kAtomBytes, L::kSwizzle);
    auto issue_s = [&](uint32_t d, uint64_t a, uint64_t bdesc) {
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const uint32_t koff = (kk / 4) * kSubDesc + (kk % 4) * 2;
        mma_ss_elect(d, a + koff, bdesc + koff, idesc_s, kk > 0);
      }
    };
    bool ok = warp_wait(q_full, 0, ctl) && warp_wait(full(0), 0, ctl);
    if (ok) {
      tc_fence_after();
      issue_s(tS, kQ_k, kK_k);                                     // S(0)
      mma_commit_elect(s_full);
      issue_s(tdP, kdO_k, kV_k);                                   // dP(0)
      mma_commit_elect(dp_full);
    }
    for (int n = 0, s = 0; ok && n < T; ++n) {
      const int s1 = (s + 1 == kDqStages) ? 0 : s + 1;
      const bool more = n + 1 < T;
      const uint32_t ph = n & 1;
      if (more) {
        // The next tile's products as soon as the compute warps have read this tile's.
        if (!warp_wait(full(s1), ((n + 1) / kDqStages) & 1, ctl) || !warp_wait(s_free, ph, ctl)) break;
        tc_fence_after();
        issue_s(tS, kQ_k, kK_k + s1 * kStageDesc);                 // S(n+1)
        mma_commit_elect(s_full);
        if (!warp_wait(dp_free, ph, ctl)) break;
        tc_fence_after();
        issue_s(tdP, kdO_k, kV_k + s1 * kStageDesc);               // dP(n+1)
        mma_commit_elect(dp_full);
      }
      if (!warp_wait(ds_full, ph, ctl)) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kTileRows / 16; ++kk)                  // dQ += dS K_n
#pragma unroll
        for (int c = 0; c < L::kSubTiles; ++c)
          mma_ts_elect(tdQ + c * (HD / L::kSubTiles), tdS + kk * 8, kK_mn + s * kStageDesc + c * kSubDesc + kk * kRowStep,
                       idesc_dq, (n > 0 || kk > 0) ? 1u : 0u);
      mma_commit_elect(dq_done);
      mma_commit_elect(empty(s));                                  // K_n, V_n fully consumed
      s = s1;
    }
    mma_commit_elect(acc_done);
    mbar_drain(acc_done, 0, ctl);
  } else if (warp >= 4) {
    // ---------------- P and dS: one query row per thread, 64 key columns per group ----------------
    const int g = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int i = quarter * 32 + lane;                // query row within the tile
    const int ig = m * kTileRows + i;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int c0 = 64 * g;                            // first key column of this group
    // Per-row constants: the exponent is S scale log2e - LSE_i log2e (valid for any
    // scale, 0 included); pad rows (ig >= S) have zero Q and dO rows and use 0.
    const size_t row = (static_cast<size_t>(b) * S + ig) * nh + h;
    const float scale_log2 = scale * kLog2e;
    const float nlse2 = ig < S ? -lse[row] * kLog2e : 0.f;
    const float nD = ig < S ? -Dvec[row] : 0.f;
    bool ok = true;
    for (int n = 0; n < T; ++n) {
      const bool diag = (n == m);
      // P = exp2(S scale log2e - LSE log2e) for this group's 64 columns, in fp32.
      if (!warp_wait(s_full, n & 1, ctl)) { ok = false; break; }
      tc_fence_after();
      uint32_t p[64];
      tmem_ld_x32(tS + lane_off + c0, p);
      tmem_ld_x32(tS + lane_off + c0 + 32, p + 32);
      tmem_wait_ld();
      reg_fence<64>(p);
      tc_fence_before();
      mbar_arrive(s_free);
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        float x0, x1;
        ffma2(x0, x1, __uint_as_float(p[2 * e]), __uint_as_float(p[2 * e + 1]), scale_log2, scale_log2,
              nlse2, nlse2);
        float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
        if (diag) {                                   // key c0 + c > query i is masked
          if (c0 + 2 * e > i) p0 = 0.f;
          if (c0 + 2 * e + 1 > i) p1 = 0.f;
        }
        p[2 * e] = __float_as_uint(p0);
        p[2 * e + 1] = __float_as_uint(p1);
      }
      // dS = P (dP - D) in two 32-column halves, bf16 into the dS slot.
      if (!warp_wait(dp_full, n & 1, ctl)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t d[32];
        tmem_ld_x32(tdP + lane_off + c0 + 32 * half, d);
        tmem_wait_ld();
        reg_fence<32>(d);
        if (half == 1) {                              // dP(n) fully read
          tc_fence_before();
          mbar_arrive(dp_free);
        }
        uint32_t ds[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float t0, t1;
          fadd2(t0, t1, __uint_as_float(d[2 * e]), __uint_as_float(d[2 * e + 1]), nD, nD);
          fmul2(t0, t1, t0, t1, __uint_as_float(p[32 * half + 2 * e]), __uint_as_float(p[32 * half + 2 * e + 1]));
          ds[e] = pack_bf16x2(t0, t1);
        }
        if (half == 0 && n > 0) {
          // dQ(n-1) has finished reading the dS slot.
          if (!warp_wait(dq_done, (n - 1) & 1, ctl)) { ok = false; break; }
          tc_fence_after();
        }
        tmem_st_x16(tdS + lane_off + c0 / 2 + 16 * half, ds);
      }
      if (!ok) break;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(ds_full);
    }
    // Epilogue: dq = bf16(scale * accumulator); group g writes head-dim columns
    // [g HD/2, (g+1) HD/2) of the thread's row.
    if (ok && warp_wait(acc_done, 0, ctl)) {
      tc_fence_after();
      constexpr int kHalf = HD / 2;
#pragma unroll
      for (int c = 0; c < kHalf; c += 16) {
        uint32_t v[16];
        tmem_ld_x16(tdQ + lane_off + g * kHalf + c, v);
        tmem_wait_ld();
        reg_fence<16>(v);
        if (ig < S) {
          XATTN_DCHECK(static_cast<size_t>(row) * HD + g * kHalf + c + 16 <= static_cast<size_t>(B) * S * nh * HD,
                       status);
          uint4 *dst = reinterpret_cast<uint4 *>(dq + row * HD + g * kHalf + c);
#pragma unroll
          for (int e = 0; e < 2; ++e)
            dst[e] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * e]) * scale, __uint_as_float(v[8 * e + 1]) * scale),
                                pack_bf16x2(__uint_as_float(v[8 * e + 2]) * scale, __uint_as_float(v[8 * e + 3]) * scale),
                                pack_bf16x2(__uint_as_float(v[8 * e + 4]) * scale, __uint_as_float(v[8 * e + 5]) * scale),
                                pack_bf16x2(__uint_as_float(v[8 * e + 6]) * scale, __uint_as_float(v[8 * e + 7]) * scale));
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
cudaError_t launch_dq_hd(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                         const CUtensorMap &mdo, const float *lse, const float *D, __nv_bfloat16 *dq,
                         int B, int S, int nh, int nkv, float scale, int *status, uint64_t timeout_ns,
                         cudaStream_t stream) {
  using L = DqLayout<HD>;
  cudaError_t err = cudaFuncSetAttribute(attn_bwd_dq_kernel<HD>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kDynBytes);
  if (err != cudaSuccess) return err;
  const int num_m = (S + kTileRows - 1) / kTileRows;
  const unsigned grid = static_cast<unsigned>(B) * nh * num_m;
  return launch_pdl(attn_bwd_dq_kernel<HD>, grid, kDqThreads, L::kDynBytes, stream, mq, mk, mv, mdo, lse, D, dq,
                    B, S, nh, nkv, scale, status, timeout_ns);
}

}  // namespace

cudaError_t launch_bwd_dq_bf16(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                               const CUtensorMap &mdo, const float *lse, const BwdWorkspace &ws,
                               __nv_bfloat16 *dq, int B, int S, int nh, int nkv, int hd, float scale,
                               int *status, uint64_t timeout_ns, cudaStream_t stream) {
  if (hd == 64)
    return launch_dq_hd<64>(mq, mk, mv, mdo, lse, ws.D, dq, B, S, nh, nkv, scale, status, timeout_ns, stream);
  if (hd == 32)
    return launch_dq_hd<32>(mq, mk, mv, mdo, lse, ws.D, dq, B, S, nh, nkv, scale, status, timeout_ns, stream);
  if (hd == 128)
    return launch_dq_hd<128>(mq, mk, mv, mdo, lse, ws.D, dq, B, S, nh, nkv, scale, status, timeout_ns, stream);
  return cudaErrorInvalidValue;
}

}  // namespace xattn
