// Backward of fused causal attention with grouped KV heads on sm_103a tensor cores.
//
// Method (xtrain "演进总览" / docs/evolution.md, phase table row T14): recompute the
// scores from Q, K and the saved log-sum-exp, use D_i = dO_i . O_i in place of the
// softmax Jacobian, and produce dQ, dK, dV. Row T15: the gradient of a kv head is the
// sum over its query group, taken deterministically without atomics.
//
// Three kernels, in stream order:
//   1. preprocess (HBM-bound): D_i = sum_d dO_id O_id in fp32, the log2-domain LSE
//      rows laid out [B, nh, S_pad] (both stored negated), and a zeroed fp32 dQ
//      accumulator.
//   2. main (tensor cores). One CTA per (batch, kv head, 128-row key tile n). The K_n
//      and V_n tiles stay in shared memory; the dK_n / dV_n accumulators stay in TMEM
//      while the CTA walks every query head r of the group and every query tile m >= n
//      (causal tile skipping). That walk *is* the group sum of row T15: no atomics on
//      dK/dV, and a fixed order, so they are reproducible. Per (r, m):
//        S^T  = K_n Q_m^T               (TMEM, 128 x 128 fp32)
//        dP^T = V_n dO_m^T              (TMEM, 128 x 128 fp32)
//        P^T  = exp2(S^T scale log2e - LSE2_m)      -> bf16 into a TMEM slot
//        dS^T = scale * P^T (dP^T - D_m)            -> bf16 into the same slot, and
//                                                      into shared memory (MN-major)
//        dV_n += P^T dO_m ,  dK_n += dS^T Q_m       (A operand from TMEM)
//        dQ_m  = dS K_n                 (TMEM) -> shared memory -> TMA reduce-add into
//                                                      the fp32 accumulator
//      Warps: 0 = TMA producer, 1 = TMEM owner + MMA issuer, 4-11 = P/dS (one thread
//      per key row, two warps per row splitting the 128 query columns), which also
//      drain each dQ tile from TMEM.
//   3. dq convert: dq = bf16(accumulator).
#include "sm103_ptx.cuh"
#include "xattn_internal.h"

namespace xattn {

size_t bwd_workspace_bytes(int B, int S, int nh, int hd) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t rows = static_cast<size_t>(B) * nh * padded_rows(S);
  return up(rows * 4) * 2 + up(static_cast<size_t>(B) * S * nh * hd * 4);
}

BwdWorkspace bwd_workspace_carve(void *base, int B, int S, int nh, int hd) {
  (void)hd;
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t rows = static_cast<size_t>(B) * nh * padded_rows(S);
  uint8_t *p = static_cast<uint8_t *>(base);
  BwdWorkspace ws;
  ws.D = reinterpret_cast<float *>(p);
  ws.lse2 = reinterpret_cast<float *>(p + up(rows * 4));
  ws.dqacc = reinterpret_cast<float *>(p + 2 * up(rows * 4));
  return ws;
}

namespace {

// ------------------------------------------------------------------------------------
// 1. preprocess
// ------------------------------------------------------------------------------------
// One group of (hd / 8) lanes per row (b, i, h): each lane reads 8 bf16 of O and dO
// (16 B each), the group reduces with shuffles. Rows are enumerated in memory order of
// O/dO, so the loads are fully coalesced. The same lanes zero the row of the dQ
// accumulator. Both vectors are stored negated (-D and -LSE log2 e), which is the form
// the main kernel adds. Pad rows (S <= i < S_pad) get 0 and -inf, so that the main
// kernel's partial query tiles contribute exactly zero.
template <int HD>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(
    const __nv_bfloat16 *__restrict__ o, const __nv_bfloat16 *__restrict__ dO,
    const float *__restrict__ lse, float *__restrict__ D, float *__restrict__ lse2,
    float *__restrict__ dqacc, int B, int S, int nh) {
  constexpr int kLanesPerRow = HD / 8;
  const int S_pad = padded_rows(S);
  const long long n_rows = static_cast<long long>(B) * S * nh;
  const long long n_pad = static_cast<long long>(B) * nh * (S_pad - S);
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long row = tid / kLanesPerRow;
  const int sub = static_cast<int>(tid % kLanesPerRow);
  const bool is_row = row < n_rows;
  float acc = 0.f;
  if (is_row) {
    const uint4 ov = *reinterpret_cast<const uint4 *>(o + row * HD + sub * 8);
    const uint4 dv = *reinterpret_cast<const uint4 *>(dO + row * HD + sub * 8);
    const uint32_t a[4] = {ov.x, ov.y, ov.z, ov.w};
    const uint32_t c[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc = fmaf(bf16lo_to_f32(a[e]), bf16lo_to_f32(c[e]), acc);
      acc = fmaf(bf16hi_to_f32(a[e]), bf16hi_to_f32(c[e]), acc);
    }
  }
  // Every lane of the warp takes part in the reduction (a warp may straddle the end of
  // the real rows); the lane groups are aligned, so no group mixes real and pad rows.
#pragma unroll
  for (int off = kLanesPerRow / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (is_row) {
    float4 *z = reinterpret_cast<float4 *>(dqacc + row * HD + sub * 8);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (sub == 0) {
      const int h = static_cast<int>(row % nh);
      const long long bi = row / nh;
      const int i = static_cast<int>(bi % S);
      const int b = static_cast<int>(bi / S);
      const size_t dst = (static_cast<size_t>(b) * nh + h) * S_pad + i;
      D[dst] = -acc;
      lse2[dst] = -lse[row] * kLog2e;
    }
  } else if (row - n_rows < n_pad && sub == 0) {
    const long long p = row - n_rows;
    const int pad = S_pad - S;
    const long long bh = p / pad;
    const int i = S + static_cast<int>(p % pad);
    D[bh * S_pad + i] = 0.f;
    lse2[bh * S_pad + i] = -INFINITY;
  }
}

// ------------------------------------------------------------------------------------
// 3. dq convert: 8 elements per thread (two 16-byte loads, one 16-byte store).
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) dq_convert_kernel(const float *__restrict__ acc,
                                                         __nv_bfloat16 *__restrict__ dq,
                                                         size_t n8) {
  const size_t t = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= n8) return;
  const float4 a = reinterpret_cast<const float4 *>(acc)[2 * t];
  const float4 c = reinterpret_cast<const float4 *>(acc)[2 * t + 1];
  reinterpret_cast<uint4 *>(dq)[t] = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w),
                                                pack_bf16x2(c.x, c.y), pack_bf16x2(c.z, c.w));
}

// ------------------------------------------------------------------------------------
// 2. main kernel
// ------------------------------------------------------------------------------------
// Column groups of the P/dS work: each group of 4 warps owns 128 / kBwdGroups query
// columns of every tile. Registers are split evenly over the 4 SM sub-partitions, so the
// per-thread limit follows from the warp count (4 + 4 * groups warps).
#ifndef XATTN_BWD_GROUPS
#define XATTN_BWD_GROUPS 2
#endif
#if XATTN_BWD_GROUPS == 4
#define XATTN_BWD_MAXNREG 96    // 20 warps: 5 per sub-partition
#elif XATTN_BWD_GROUPS == 2
#define XATTN_BWD_MAXNREG 168   // 12 warps: 3 per sub-partition
#else
#error "XATTN_BWD_GROUPS must be 2 or 4"
#endif
constexpr int kBwdGroups = XATTN_BWD_GROUPS;
constexpr int kBwdThreads = 128 + 128 * kBwdGroups;

template <int HD>
struct BwdLayout {
  static constexpr uint32_t kRowBytes = HD * 2;
  static constexpr uint32_t kTileBytes = kTileRows * kRowBytes;
  static constexpr uint32_t kSwizzle = (HD == 64) ? kSwizzle128 : kSwizzle64;
  static constexpr uint32_t kK = 0;
  static constexpr uint32_t kV = kK + kTileBytes;
  static constexpr uint32_t kQ = kV + kTileBytes;          // 2 stages
  static constexpr uint32_t kdO = kQ + 2 * kTileBytes;     // 2 stages
  static constexpr uint32_t kdS = kdO + 2 * kTileBytes;    // 128 x 128 bf16, MN-major, 32 KB
  // dQ staging for the TMA reduce-add: 2 buffers x 2 head-dim halves x 128 rows of
  // HD/2 floats, swizzled like the tensor map's box.
  static constexpr uint32_t kDqRowBytes = HD / 2 * 4;
  static constexpr uint32_t kDqHalfBytes = kTileRows * kDqRowBytes;
  static constexpr uint32_t kdQs = kdS + 32768;
  static constexpr uint32_t kVec = kdQs + 4 * kDqHalfBytes;  // -LSE2[2][128], -D[2][128] fp32
  // barriers: kv_full, full[2], empty[2], s_full, dp_full, p_full, ds_full, dq_full,
  //           dq_empty, acc_done, dv_done, dk_done, dqs_full[2], dqs_empty[2]
  static constexpr int kNumBars = 18;
  static constexpr uint32_t kBars = kVec + 4 * 512;
  static constexpr uint32_t kMisc = kBars + 8 * kNumBars;
  static constexpr uint32_t kUsed = kMisc + 32;
  static constexpr uint32_t kDynBytes = (kUsed + 1024 > 120 * 1024) ? kUsed + 1024 : 120 * 1024;
};

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtl &ctl) {
  const bool ok = mbar_wait(bar, parity, ctl);
  return __all_sync(0xffffffffu, ok);
}

// Offset of element (key row j, query column i) of the 128 x 128 dS^T tile, stored as
// the A operand of dQ = dS K: M = query (contiguous), K = key rows; two 64-column
// atoms of 128-byte rows with the 128-byte swizzle (16-byte chunk ^= row % 8).
__device__ __forceinline__ uint32_t ds_offset(int j, int i) {
  return static_cast<uint32_t>((i >> 6) * 16384 + j * 128 + ((((i & 63) >> 3) ^ (j & 7)) << 4));
}

// Role map (4 + 4 * kBwdGroups warps):
//   warp 0     : TMA producer
//   warp 1     : TMEM owner and MMA issuer
//   warp 2     : dQ reducer: TMA reduce-adds each staged dQ tile into the fp32
//                accumulator (2 bulk operations per tile instead of scattered atomics)
//   warp 3     : idle
//   warps 4.. : P^T / dS^T, one thread per key row; warp group g (4 warps, one per TMEM
//               lane quarter) owns query columns [g*C, (g+1)*C), C = 128 / kBwdGroups, so
//               each SM sub-partition interleaves kBwdGroups of them. They also move
//               dQ(t-1) from TMEM to a double-buffered shared-memory tile (one query row
//               per thread, group g taking head-dim columns [g*HD/G, (g+1)*HD/G)).
// TMEM columns: S^T [0,128) fp32 | dP^T [128,256) fp32 | P^T, then dS^T, bf16 [256,320)
//               | dV [320,384) | dK [384,448) | dQ [448,512)
// P^T and dS^T share one slot that no other result overlaps, so the two column halves
// never write over values the other half still has to read; the MMA readers of that
// slot (dV reads P^T, dK reads dS^T) are waited for before it is overwritten.
template <int HD>
__global__ void __maxnreg__(XATTN_BWD_MAXNREG)
    attn_bwd_main_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                         const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
                         const __grid_constant__ CUtensorMap mdq,
                         const float *__restrict__ Dvec, const float *__restrict__ lse2,
                         __nv_bfloat16 *__restrict__ dk,
                         __nv_bfloat16 *__restrict__ dv, int B, int S, int nh, int nkv,
                         float scale, float scale_log2, int *status, unsigned long long timeout_ns) {
  using L = BwdLayout<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Unit of this CTA: key tile n (most work first), batch b, kv head kvh.
  const int num_m = (S + kTileRows - 1) / kTileRows;
  const int S_pad = num_m * kTileRows;
  const int BK = B * nkv;
  const int n = static_cast<int>(blockIdx.x) / BK;
  const int bk = static_cast<int>(blockIdx.x) % BK;
  const int b = bk / nkv, kvh = bk % nkv;
  const int group = nh / nkv;
  const int per_head = num_m - n;         // query tiles m = n .. num_m-1
  const int T = group * per_head;         // iterations (r, m)

  const uint32_t sK = smem_u32(smem + L::kK);
  const uint32_t sV = smem_u32(smem + L::kV);
  const uint32_t sQ = smem_u32(smem + L::kQ);
  const uint32_t sdO = smem_u32(smem + L::kdO);
  uint8_t *sdS_ptr = smem + L::kdS;
  const uint32_t sdS = smem_u32(sdS_ptr);
  uint8_t *sdQs_ptr = smem + L::kdQs;
  float *sLSE = reinterpret_cast<float *>(smem + L::kVec);         // [2][128]  -LSE log2 e
  float *sD = reinterpret_cast<float *>(smem + L::kVec + 1024);    // [2][128]  -D
  const uint32_t bar0 = smem_u32(smem + L::kBars);
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  const uint32_t kv_full = bar(0);
  auto full = [&](int s) { return bar(1 + s); };
  auto empty = [&](int s) { return bar(3 + s); };
  const uint32_t s_full = bar(5), dp_full = bar(6), p_full = bar(7), ds_full = bar(8);
  const uint32_t dq_full = bar(9), dq_empty = bar(10), acc_done = bar(11);
  const uint32_t dv_done = bar(12), dk_done = bar(13);
  auto dqs_full = [&](int x) { return bar(14 + x); };
  auto dqs_empty = [&](int x) { return bar(16 + x); };
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMisc + 16);
  const WaitCtl ctl{abort_flag, status, timeout_ns};

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(kv_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(p_full, 128 * kBwdGroups);
    mbar_init(ds_full, 128 * kBwdGroups);
    mbar_init(dq_full, 1);
    mbar_init(dq_empty, 128 * kBwdGroups);
    mbar_init(acc_done, 1);
    mbar_init(dv_done, 1);
    mbar_init(dk_done, 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(dqs_full(x), 128 * kBwdGroups);
      mbar_init(dqs_empty(x), 1);
    }
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mq);
    tma_prefetch_desc(&mk);
    tma_prefetch_desc(&mv);
    tma_prefetch_desc(&mdo);
    tma_prefetch_desc(&mdq);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t tS = tmem, tdP = tmem + 128, tP = tmem + 256;
  const uint32_t tdV = tmem + 320, tdK = tmem + 384, tdQ = tmem + 448;

  if (warp == 0) {
    // ---------------- TMA producer (converged warp, one elected lane issues) ----------------
    mbar_expect_tx_elect(kv_full, 2 * L::kTileBytes);
    tma_load_4d_elect(sK, &mk, kv_full, 0, kvh, n * kTileRows, b);
    tma_load_4d_elect(sV, &mv, kv_full, 0, kvh, n * kTileRows, b);
    int issued = 0;
    for (int t = 0, r = 0, m = n; t < T; ++t) {
      const int h = kvh * group + r;
      const int s = t & 1;
      if (!warp_wait(empty(s), ((t >> 1) & 1) ^ 1, ctl)) break;
      mbar_expect_tx_elect(full(s), 2 * L::kTileBytes + 2 * 512);
      tma_load_4d_elect(sQ + s * L::kTileBytes, &mq, full(s), 0, h, m * kTileRows, b);
      tma_load_4d_elect(sdO + s * L::kTileBytes, &mdo, full(s), 0, h, m * kTileRows, b);
      const size_t vec = (static_cast<size_t>(b) * nh + h) * S_pad + static_cast<size_t>(m) * kTileRows;
      bulk_load_elect(smem_u32(sLSE + s * 128), lse2 + vec, 512, full(s));
      bulk_load_elect(smem_u32(sD + s * 128), Dvec + vec, 512, full(s));
      issued = t + 1;
      if (++m == num_m) { m = n; ++r; }
    }
    mbar_drain(kv_full, 0, ctl);
    for (int t = (issued > 2 ? issued - 2 : 0); t < issued; ++t)
      mbar_drain(full(t & 1), (t >> 1) & 1, ctl);
  } else if (warp == 1) {
    // ---------------- MMA issuer (converged warp, one elected lane issues) ----------------
    constexpr uint32_t idesc_t = idesc_bf16_f32(128, 128, false, false);  // S^T, dP^T
    constexpr uint32_t idesc_acc = idesc_bf16_f32(128, HD, false, true);  // dV, dK (A in TMEM)
    constexpr uint32_t idesc_dq = idesc_bf16_f32(128, HD, true, true);    // dQ (A = dS, MN-major)
    constexpr uint32_t kStageDesc = L::kTileBytes >> 4;   // stage stride, descriptor units
    constexpr uint32_t kRowStep = (16 * L::kRowBytes) >> 4;  // 16 rows of an MN-major tile
    // Descriptors are built once. K-major operands (Q, K, V, dO as K-major) advance
    // +32 bytes (+2) per 16-element K step; MN-major ones advance 16 rows.
    const uint64_t kK_k = smem_desc(sK, 16, 8 * L::kRowBytes, L::kSwizzle);
    const uint64_t kV_k = smem_desc(sV, 16, 8 * L::kRowBytes, L::kSwizzle);
    const uint64_t kQ_k = smem_desc(sQ, 16, 8 * L::kRowBytes, L::kSwizzle);
    const uint64_t kdO_k = smem_desc(sdO, 16, 8 * L::kRowBytes, L::kSwizzle);
    const uint64_t kQ_mn = smem_desc(sQ, 8192, 8 * L::kRowBytes, L::kSwizzle);
    const uint64_t kdO_mn = smem_desc(sdO, 8192, 8 * L::kRowBytes, L::kSwizzle);
    const uint64_t kK_mn = smem_desc(sK, 8192, 8 * L::kRowBytes, L::kSwizzle);
    const uint64_t kdS_mn = smem_desc(sdS, 16384, 1024, kSwizzle128);
    auto issue_kmajor = [&](uint32_t d, uint64_t a, uint64_t bdesc) {
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) mma_ss_elect(d, a + 2 * kk, bdesc + 2 * kk, idesc_t, kk > 0);
    };
    auto issue_acc = [&](uint32_t d, uint64_t bdesc, bool first) {
#pragma unroll
      for (int kk = 0; kk < kTileRows / 16; ++kk)
        mma_ts_elect(d, tP + kk * 8, bdesc + kk * kRowStep, idesc_acc, (!first || kk > 0) ? 1u : 0u);
    };
    bool ok = warp_wait(kv_full, 0, ctl) && warp_wait(full(0), 0, ctl);
    if (ok) {
      tc_fence_after();
      issue_kmajor(tS, kK_k, kQ_k);
      mma_commit_elect(s_full);
      issue_kmajor(tdP, kV_k, kdO_k);
      mma_commit_elect(dp_full);
    }
    for (int t = 0; ok && t < T; ++t) {
      const int s = t & 1;
      const bool more = t + 1 < T;
      if (!warp_wait(p_full, t & 1, ctl)) break;
      tc_fence_after();
      issue_acc(tdV, kdO_mn + s * kStageDesc, t == 0);                       // dV += P^T dO
      mma_commit_elect(dv_done);
      if (more) {
        if (!warp_wait(full(s ^ 1), ((t + 1) >> 1) & 1, ctl)) break;
        tc_fence_after();
        issue_kmajor(tS, kK_k, kQ_k + (s ^ 1) * kStageDesc);                 // S^T(t+1)
        mma_commit_elect(s_full);
      }
      if (!warp_wait(ds_full, t & 1, ctl)) break;
      tc_fence_after();
      issue_acc(tdK, kQ_mn + s * kStageDesc, t == 0);                        // dK += dS^T Q
      mma_commit_elect(empty(s));
      mma_commit_elect(dk_done);
      if (!warp_wait(dq_empty, (t & 1) ^ 1, ctl)) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kTileRows / 16; ++kk)                            // dQ = dS K
        mma_ss_elect(tdQ, kdS_mn + kk * 128, kK_mn + kk * kRowStep, idesc_dq, kk > 0);
      mma_commit_elect(dq_full);
      if (more) {
        issue_kmajor(tdP, kV_k, kdO_k + (s ^ 1) * kStageDesc);               // dP^T(t+1)
        mma_commit_elect(dp_full);
      }
    }
    mma_commit_elect(acc_done);
    mbar_drain(acc_done, 0, ctl);
  } else if (warp == 2) {
    // ---------------- dQ reducer ----------------
    for (int k = 0; k < T; ++k) {
      const int buf = k & 1;
      if (!warp_wait(dqs_full(buf), (k >> 1) & 1, ctl)) break;
      if (lane == 0) {
        const int h = kvh * group + k / per_head, m = n + k % per_head;
        const uint32_t src = smem_u32(sdQs_ptr + buf * 2 * L::kDqHalfBytes);
        tma_reduce_add_4d(&mdq, src, 0, h, m * kTileRows, b);
        tma_reduce_add_4d(&mdq, src + L::kDqHalfBytes, HD / 2, h, m * kTileRows, b);
        bulk_commit_group();
        bulk_wait_read_all();          // the staging buffer may be rewritten
        mbar_arrive(dqs_empty(buf));
      }
      __syncwarp();
    }
    if (lane == 0) bulk_wait_all();    // every reduce-add has landed before the CTA exits
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------- P^T and dS^T: one thread per key row, C query columns ----------------
    constexpr int C = 128 / kBwdGroups;        // query columns per thread
    constexpr int kDq = HD / kBwdGroups;       // dQ head-dim columns drained per thread
    const int g = (warp - 4) >> 2;             // column group
    const int quarter = warp & 3;
    const int j = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int col_f32 = C * g;
    const uint32_t col_bf16 = static_cast<uint32_t>(C / 2 * g);
    // dQ(k) from TMEM (query row j of its tile, head-dim columns [g*kDq, (g+1)*kDq)) into
    // staging buffer k & 1, swizzled like the reduce's tensor-map box (two halves of HD/2
    // floats per row); warp 2 then adds it to global memory.
    auto drain_dq = [&](int k) -> bool {
      const int buf = k & 1;
      uint32_t v[kDq];
      if constexpr (kDq == 32) tmem_ld_x32(tdQ + lane_off + kDq * g, v);
      else if constexpr (kDq == 16) tmem_ld_x16(tdQ + lane_off + kDq * g, v);
      else tmem_ld_x8(tdQ + lane_off + kDq * g, v);
      tmem_wait_ld();
      reg_fence<kDq>(v);
      tc_fence_before();
      mbar_arrive(dq_empty);
      if (!warp_wait(dqs_empty(buf), ((k >> 1) & 1) ^ 1, ctl)) return false;
      const int first = kDq * g;                      // first head-dim column
      const int half = first / (HD / 2);
      const int chunk0 = (first % (HD / 2)) / 4;      // 16-byte chunk within the row
      uint8_t *row = sdQs_ptr + (buf * 2 + half) * L::kDqHalfBytes + j * L::kDqRowBytes;
#pragma unroll
      for (int c = 0; c < kDq / 4; ++c) {
        const int ch = chunk0 + c;
        const int sw = (HD == 64) ? (ch ^ (j & 7)) : (ch ^ ((j >> 1) & 3));
        *reinterpret_cast<uint4 *>(row + (sw << 4)) =
            make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(dqs_full(buf));
      return true;
    };
    auto ld_cols = [&](uint32_t taddr, uint32_t *r) {
#pragma unroll
      for (int c = 0; c < C; c += 32) tmem_ld_x32(taddr + c, r + c);
      tmem_wait_ld();
      reg_fence<C>(r);
    };
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      const int m = n + t % per_head;
      const int s = t & 1;
      const bool diag = (m == n);
      // Phase 1: P^T = exp2(S^T scale log2e - LSE2), masked above the diagonal.
      if (!warp_wait(s_full, t & 1, ctl)) { ok = false; break; }
      tc_fence_after();
      uint32_t r[C];
      ld_cols(tS + lane_off + col_f32, r);
      const float4 *nlse4 = reinterpret_cast<const float4 *>(sLSE + s * 128 + col_f32);
      uint32_t pk[C / 2];
#pragma unroll
      for (int q4 = 0; q4 < C / 4; ++q4) {
        const float4 nl = nlse4[q4];
        float x0, x1, x2, x3;
        ffma2(x0, x1, __uint_as_float(r[4 * q4]), __uint_as_float(r[4 * q4 + 1]), scale_log2,
              scale_log2, nl.x, nl.y);
        ffma2(x2, x3, __uint_as_float(r[4 * q4 + 2]), __uint_as_float(r[4 * q4 + 3]), scale_log2,
              scale_log2, nl.z, nl.w);
        float p0 = ex2_approx(x0), p1 = ex2_approx(x1), p2 = ex2_approx(x2), p3 = ex2_approx(x3);
        if (diag) {
          const int i = col_f32 + 4 * q4;
          if (i + 0 < j) p0 = 0.f;
          if (i + 1 < j) p1 = 0.f;
          if (i + 2 < j) p2 = 0.f;
          if (i + 3 < j) p3 = 0.f;
        }
        pk[2 * q4] = pack_bf16x2(p0, p1);
        pk[2 * q4 + 1] = pack_bf16x2(p2, p3);
      }
      // The P^T slot still holds dS^T(t-1) until dK(t-1) has read it.
      if (t > 0 && !warp_wait(dk_done, (t - 1) & 1, ctl)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < C / 2; c += 16) tmem_st_x16(tP + lane_off + col_bf16 + c, pk + c);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_full);

      // Phase 2: dS^T = scale P^T (dP^T - D).
      if (!warp_wait(dp_full, t & 1, ctl)) { ok = false; break; }
      tc_fence_after();
      ld_cols(tdP + lane_off + col_f32, r);
      // dQ(t-1) must be done reading the shared-memory copy of dS (its result is drained
      // here), and dV(t) must be done reading P^T before dS^T replaces it in TMEM.
      if (t > 0) {
        if (!warp_wait(dq_full, (t - 1) & 1, ctl)) { ok = false; break; }
        tc_fence_after();
        if (!drain_dq(t - 1)) { ok = false; break; }
      }
      if (!warp_wait(dv_done, t & 1, ctl)) { ok = false; break; }
      tc_fence_after();
      const float4 *nd4 = reinterpret_cast<const float4 *>(sD + s * 128 + col_f32);
#pragma unroll
      for (int c32 = 0; c32 < C; c32 += 32) {
        uint32_t dsk[16];
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const int c = c32 + 4 * q4;
          const float4 nd = nd4[c / 4];
          const uint32_t pa = pk[c / 2], pb = pk[c / 2 + 1];
          float t0, t1, t2, t3;
          fadd2(t0, t1, __uint_as_float(r[c]), __uint_as_float(r[c + 1]), nd.x, nd.y);
          fadd2(t2, t3, __uint_as_float(r[c + 2]), __uint_as_float(r[c + 3]), nd.z, nd.w);
          fmul2(t0, t1, t0, t1, bf16lo_to_f32(pa), bf16hi_to_f32(pa));
          fmul2(t2, t3, t2, t3, bf16lo_to_f32(pb), bf16hi_to_f32(pb));
          fmul2(t0, t1, t0, t1, scale, scale);
          fmul2(t2, t3, t2, t3, scale, scale);
          dsk[2 * q4] = pack_bf16x2(t0, t1);
          dsk[2 * q4 + 1] = pack_bf16x2(t2, t3);
        }
        tmem_st_x16(tP + lane_off + col_bf16 + c32 / 2, dsk);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          *reinterpret_cast<uint4 *>(sdS_ptr + ds_offset(j, col_f32 + c32 + 8 * e)) =
              make_uint4(dsk[4 * e], dsk[4 * e + 1], dsk[4 * e + 2], dsk[4 * e + 3]);
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(ds_full);
    }
    // Epilogue: drain the last dQ; then the groups store the dV and dK rows, each group a
    // contiguous slice of [dV | dK] (dK already carries the scale).
    if (ok && warp_wait(dq_full, (T - 1) & 1, ctl)) {
      tc_fence_after();
      ok = drain_dq(T - 1);
    } else {
      ok = false;
    }
    if (ok && warp_wait(acc_done, 0, ctl)) {
      tc_fence_after();
      constexpr int kPer = 2 * HD / kBwdGroups;   // output columns per group
      const int first = kPer * g;                 // in the concatenation [dV | dK]
      const bool is_dk = first >= HD;
      const int c0 = first % HD;
      const int jg = n * kTileRows + j;
      const size_t row_off = (static_cast<size_t>(b) * S + jg) * nkv * HD + static_cast<size_t>(kvh) * HD;
      const uint32_t tsrc = (is_dk ? tdK : tdV) + c0;
      __nv_bfloat16 *dst_row = (is_dk ? dk : dv) + row_off + c0;
#pragma unroll
      for (int c = 0; c < kPer; c += 16) {
        uint32_t v[16];
        tmem_ld_x16(tsrc + lane_off + c, v);
        tmem_wait_ld();
        reg_fence<16>(v);
        if (jg < S) {
          uint4 *dst = reinterpret_cast<uint4 *>(dst_row + c);
#pragma unroll
          for (int e = 0; e < 2; ++e)
            dst[e] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * e]), __uint_as_float(v[8 * e + 1])),
                                pack_bf16x2(__uint_as_float(v[8 * e + 2]), __uint_as_float(v[8 * e + 3])),
                                pack_bf16x2(__uint_as_float(v[8 * e + 4]), __uint_as_float(v[8 * e + 5])),
                                pack_bf16x2(__uint_as_float(v[8 * e + 6]), __uint_as_float(v[8 * e + 7])));
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
cudaError_t launch_main_hd(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                           const CUtensorMap &mdo, const CUtensorMap &mdq, const BwdWorkspace &ws, __nv_bfloat16 *dk,
                           __nv_bfloat16 *dv, int B, int S, int nh, int nkv, float scale,
                           int *status, uint64_t timeout_ns, cudaStream_t stream) {
  using L = BwdLayout<HD>;
  cudaError_t err = cudaFuncSetAttribute(attn_bwd_main_kernel<HD>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kDynBytes);
  if (err != cudaSuccess) return err;
  const int num_n = (S + kTileRows - 1) / kTileRows;
  const unsigned grid = static_cast<unsigned>(B) * nkv * num_n;
  attn_bwd_main_kernel<HD><<<grid, kBwdThreads, L::kDynBytes, stream>>>(
      mq, mk, mv, mdo, mdq, ws.D, ws.lse2, dk, dv, B, S, nh, nkv, scale, scale * kLog2e,
      status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_preprocess(const __nv_bfloat16 *o, const __nv_bfloat16 *dO,
                                  const float *lse, int B, int S, int nh, int hd,
                                  const BwdWorkspace &ws, cudaStream_t stream) {
  const long long n_rows = static_cast<long long>(B) * S * nh;
  const long long n_pad = static_cast<long long>(B) * nh * (padded_rows(S) - S);
  const int lanes = hd / 8;
  const long long threads = (n_rows + n_pad) * lanes;
  const unsigned grid = static_cast<unsigned>((threads + 255) / 256);
  if (hd == 64)
    bwd_preprocess_kernel<64><<<grid, 256, 0, stream>>>(o, dO, lse, ws.D, ws.lse2, ws.dqacc, B, S, nh);
  else if (hd == 32)
    bwd_preprocess_kernel<32><<<grid, 256, 0, stream>>>(o, dO, lse, ws.D, ws.lse2, ws.dqacc, B, S, nh);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_bwd_main_bf16(const CUtensorMap &mq, const CUtensorMap &mk,
                                 const CUtensorMap &mv, const CUtensorMap &mdo,
                                 const CUtensorMap &mdq, const BwdWorkspace &ws, __nv_bfloat16 *dk, __nv_bfloat16 *dv,
                                 int B, int S, int nh, int nkv, int hd, float scale, int *status,
                                 uint64_t timeout_ns, cudaStream_t stream) {
  if (hd == 64)
    return launch_main_hd<64>(mq, mk, mv, mdo, mdq, ws, dk, dv, B, S, nh, nkv, scale, status, timeout_ns, stream);
  if (hd == 32)
    return launch_main_hd<32>(mq, mk, mv, mdo, mdq, ws, dk, dv, B, S, nh, nkv, scale, status, timeout_ns, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_dq_convert(const float *dqacc, __nv_bfloat16 *dq, size_t n_elems,
                              cudaStream_t stream) {
  const size_t n8 = n_elems / 8;
  const unsigned grid = static_cast<unsigned>((n8 + 255) / 256);
  if (grid == 0) return cudaSuccess;
  dq_convert_kernel<<<grid, 256, 0, stream>>>(dqacc, dq, n8);
  return cudaGetLastError();
}

}  // namespace xattn
