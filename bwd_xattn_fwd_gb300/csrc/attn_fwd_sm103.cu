// Forward of fused causal attention with grouped KV heads on sm_103a tensor cores.
//
// Method (xtrain "演进总览" / docs/evolution.md, phase table row T14): one kernel, an
// online softmax tiled over KV, the S x S scores never leave the chip, and each row's
// log-sum-exp is kept for the backward. Grouped KV heads (row T15): query head h reads
// kv head h / group.
//
// GB300 mapping: a unit of work is one pair of 128-row query tiles A = 2j and B = 2j+1
// of one (batch, head) -- 256 query rows that share every K/V tile they read. Persistent
// CTAs, one per SM, take the units in turn (longest first). 12 warps:
//   warp 0     : TMA producer. Q_A and Q_B once per unit, into one of two buffers, so a
//                unit's query tiles land while the previous unit still runs; K/V tiles
//                through a ring that runs on across units (3 stages with query groups,
//                4 with one query head per kv head, 2 at hd = 128).
//   warps 1, 3 : MMA issuers, warp 1 for tile A (and TMEM owner), warp 3 for tile B
//                (converged warps, one elected lane issues):
//                  S_X(n) = Q_X K_n^T  (A, B from shared memory) -> TMEM
//                  O_X   += P_X(n) V_n (A = P from TMEM)          -> TMEM accumulator
//                so the tensor core works on one tile while the other tile's softmax
//                runs; S_X(n+1) is issued as soon as the softmax has read S_X(n), before
//                it finishes P_X(n). Each K/V stage is released by a commit from both.
//   warps 4-7  : softmax of tile A, one thread per query row (TMEM lane), all 128 key
//                columns of a tile; warps 8-11 the same for tile B.
//   warp 2     : idle.
// Softmax per key tile: causal mask on the diagonal tile, running max and sum in fp32
// (log2 domain), P in bf16 to TMEM, O rescaled only when the running max grows by more
// than 2^8 (the stale max is exact because the final normalisation uses the same max).
// Epilogue: O / l in bf16, LSE = (m + log2 l) ln 2.
// Causal tile skipping: tile m visits key tiles 0..m.
// TMEM columns: S_A [0,128) S_B [128,256) fp32 | O_A [256,256+HD) O_B [320,320+HD) fp32 |
//               P_A [384,448) P_B [448,512) bf16 pairs; at hd = 128: O_A [256,384),
//               O_B [384,512), and P_X in the first 64 columns of S_X.
#include <type_traits>

#include "sm103_ptx.cuh"
#include "xattn_internal.h"

namespace xattn {
namespace {

constexpr int kFwdThreads = 384;  // 12 warps

// hd = 128 differs from hd = 32 / 64 in three ways, all fixed here at compile time:
//  * a 256-byte row does not fit one 128-byte swizzle atom, so every tile is stored (and
//    loaded by TMA) as two 64-column sub-tiles, each laid out like an hd = 64 tile;
//  * shared memory holds one Q buffer and two K/V stages (three Q+K/V stages of 32 KB
//    tiles would not fit);
//  * O_A and O_B take 128 TMEM columns each, so P_X is written over the columns of S_X
//    (kAliasP) and S_X(n+1) is issued after PV_X(n), whose read of P_X(n) the tensor
//    pipe completes first (one thread's MMAs execute in issue order).
// kRing: K/V stages. Three with query groups (the group's query heads read each K/V tile
// within one pass, mostly from L2); four with one query head per kv head, whose tiles come
// from DRAM more often (measured faster there: dim768 forward 83.9 -> 81.3 us, and 2 %
// slower with query groups).
template <int HD, int kRing = (HD == 128 ? 2 : 3)>
struct FwdLayout {
  static constexpr int kStages = kRing;                              // K/V ring
  static constexpr int kQBufs = HD == 128 ? 1 : 2;                  // Q buffers (Q_A, Q_B each)
  static constexpr bool kAliasP = HD == 128;
  static constexpr uint32_t kRowBytes = HD * 2;
  static constexpr uint32_t kTileBytes = kTileRows * kRowBytes;
  static constexpr uint32_t kAtomBytes = kRowBytes < 128 ? kRowBytes : 128;  // sub-tile row
  static constexpr int kSubTiles = static_cast<int>(kRowBytes / kAtomBytes);
  static constexpr uint32_t kSubBytes = kTileRows * kAtomBytes;
  static constexpr uint32_t kSwizzle = (HD == 32) ? kSwizzle64 : kSwizzle128;
  static constexpr uint32_t kQ = 0;                                  // kQBufs x (Q_A, Q_B)
  static constexpr uint32_t kK = kQ + 2 * kQBufs * kTileBytes;
  static constexpr uint32_t kV = kK + kStages * kTileBytes;
  static constexpr uint32_t kBars = kV + kStages * kTileBytes;
  // barriers: full[S], empty[S], s_full[2], p_full[2], o_done[2], s_free[2], o_free[2],
  //           q_full[2], mma_final[2] (one each per Q buffer)
  static constexpr int kNumBars = 2 * kStages + 2 + 2 + 2 + 2 + 2 + 2 + 2;
  static constexpr uint32_t kMisc = kBars + 8 * kNumBars;
  static constexpr uint32_t kUsed = kMisc + 32;
  // Ask for enough shared memory that one CTA occupies an SM: each CTA holds all 512
  // TMEM columns, so a second resident CTA would only spin in tcgen05.alloc.
  static constexpr uint32_t kDynBytes = (kUsed + 1024 > 120 * 1024) ? kUsed + 1024 : 120 * 1024;
  static_assert(kDynBytes <= 227 * 1024, "exceeds the opt-in shared memory of one CTA");
  static_assert(kSubBytes % 1024 == 0 && kTileBytes % 1024 == 0, "swizzled tiles need 1024-byte alignment");
};


// 2^x for a pair on the FMA pipe: x = j + f with j = rint(x) and |f| <= 1/2 (x clamped
// at -126), 2^f from a cubic fitted to it on [-1/2, 1/2] by least squares on Chebyshev
// nodes (relative error below 8e-5), and j added into the exponent field.
__device__ __forceinline__ void exp2_fma2(float x0, float x1, float &y0, float &y1) {
  constexpr float kRound = 12582912.f;   // 1.5 * 2^23: x + kRound is rint(x) in the low bits
  constexpr float c0 = 0.9999279975891113f, c1 = 0.6932597756385803f;
  constexpr float c2 = 0.24261167645454407f, c3 = 0.05517822131514549f;
  x0 = fmaxf(x0, -126.f);
  x1 = fmaxf(x1, -126.f);
  float j0, j1, t0, t1, f0, f1, p0, p1;
  fadd2(j0, j1, x0, x1, kRound, kRound);
  fadd2(t0, t1, j0, j1, -kRound, -kRound);
  ffma2(f0, f1, t0, t1, -1.f, -1.f, x0, x1);
  ffma2(p0, p1, f0, f1, c3, c3, c2, c2);
  ffma2(p0, p1, p0, p1, f0, f1, c1, c1);
  ffma2(p0, p1, p0, p1, f0, f1, c0, c0);
  y0 = __int_as_float(__float_as_int(p0) + (__float_as_int(j0) << 23));
  y1 = __int_as_float(__float_as_int(p1) + (__float_as_int(j1) << 23));
}

// Warp-uniform bounded wait: every lane waits, then all agree.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtl &ctl) {
  const bool ok = mbar_wait(bar, parity, ctl);
  return __all_sync(0xffffffffu, ok);
}

// kNegScale: scale < 0, so the row maximum of the scaled scores is the scaled minimum of
// the raw ones.
template <int HD, bool kNegScale, int kRing>
__global__ void __maxnreg__(168)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                    const __grid_constant__ CUtensorMap mv, __nv_bfloat16 *__restrict__ o,
                    float *__restrict__ lse, int B, int S, int nh, int nkv, float scale_log2,
                    int *status, unsigned long long timeout_ns) {
  using L = FwdLayout<HD, kRing>;
  constexpr int kFwdStages = L::kStages;
  constexpr int kQBufs = L::kQBufs;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  // Warp-uniform by construction; the broadcast lets the compiler see it.
  const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0), lane = threadIdx.x & 31;

  // Work units (tile pair jp of one (batch, head)) are numbered longest first. The CTAs
  // are persistent: CTA c of G takes unit k G + c in even rounds k and k G + G - 1 - c in
  // odd ones. Every role walks the same units; the barriers' phases count over all of
  // them (waits for the phase before the first -- parity 1 of a fresh barrier -- return
  // at once, so the first unit needs no special case).
  const int num_m = (S + kTileRows - 1) / kTileRows;
  const int num_pairs = (num_m + 1) / 2;
  const int BH = B * nh;
  const int num_units = num_pairs * BH;
  const int G = static_cast<int>(gridDim.x), cta = static_cast<int>(blockIdx.x);
  auto unit_at = [G, cta](int k) { return k * G + ((k & 1) ? G - 1 - cta : cta); };
// Fields of unit u, as constants of the role loop that processes it.
#define XATTN_FWD_UNIT(u)                                       \
  const int jp = num_pairs - 1 - (u) / BH;                      \
  const int b = ((u) % BH) / nh, h = (u) % nh;                  \
  const int kvh = h / (nh / nkv);                               \
  const int mA = 2 * jp, mB = 2 * jp + 1;                       \
  const bool hasB = mB < num_m;                                 \
  const int n_last = hasB ? mB : mA; /* last key tile */        \
  (void)b;                                                      \
  (void)kvh;                                                    \
  (void)n_last

  const uint32_t sQ = smem_u32(smem + L::kQ);
  const uint32_t sK = smem_u32(smem + L::kK);
  const uint32_t sV = smem_u32(smem + L::kV);
  const uint32_t bar0 = smem_u32(smem + L::kBars);
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  auto full = [&](int s) { return bar(s); };
  auto empty = [&](int s) { return bar(kFwdStages + s); };
  auto s_full = [&](int x) { return bar(2 * kFwdStages + x); };
  auto p_full = [&](int x) { return bar(2 + 2 * kFwdStages + x); };
  auto o_done = [&](int x) { return bar(4 + 2 * kFwdStages + x); };
  auto s_free = [&](int x) { return bar(6 + 2 * kFwdStages + x); };
  auto o_free = [&](int x) { return bar(8 + 2 * kFwdStages + x); };   // O_X read by the epilogue
  // Q buffer qb (units alternate between the two): its tiles landed / the unit's products
  // that read them are done. Each completes once per use of its buffer, every two units.
  auto q_full = [&](int qb) { return bar(10 + 2 * kFwdStages + qb); };
  auto mma_final = [&](int qb) { return bar(12 + 2 * kFwdStages + qb); };
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMisc + 16);
  const WaitCtl ctl{abort_flag, status, timeout_ns};

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    // Each K/V stage is released by both MMA issuers (warp 1 for tile A, warp 3 for B).
    for (int s = 0; s < kFwdStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 2);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(s_full(x), 1);
      mbar_init(p_full(x), 128);
      mbar_init(o_done(x), 1);
      mbar_init(s_free(x), 128);
      mbar_init(o_free(x), 128);
    }
    for (int qb = 0; qb < 2; ++qb) {
      mbar_init(q_full(qb), 1);
      mbar_init(mma_final(qb), 2);
    }
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
  grid_dep_launch();
  grid_dep_wait();
  const uint32_t tmem = __shfl_sync(0xffffffffu, *tmem_holder, 0);
  auto tS = [&](int x) { return tmem + 128u * x; };
  auto tO = [&](int x) { return tmem + 256u + (L::kAliasP ? 128u : 64u) * x; };
  auto tP = [&](int x) { return L::kAliasP ? tS(x) : tmem + 384u + 64u * x; };
  // One 128-row tile of a [B, S, heads, hd] tensor: one TMA box per 64-column sub-tile.
  // Debug builds check the tile's coordinates (heads < nh covers both Q and K/V) and that
  // it lands inside the tile region of shared memory.
  const int S_pad = (S + kTileRows - 1) / kTileRows * kTileRows;
  (void)S_pad;
  auto load_tile = [&](uint32_t dst, const CUtensorMap *map, uint32_t bar, int head, int row0, int bb) {
    XATTN_DCHECK(head >= 0 && head < nh && row0 >= 0 && row0 < S_pad && row0 % kTileRows == 0 && bb >= 0 &&
                     bb < B && dst >= smem_u32(smem) && dst + L::kTileBytes <= smem_u32(smem) + L::kBars,
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
    // The K/V ring runs on across units (ring index R counts tiles over all of them). A
    // unit's Q tiles go to buffer units % 2 once the products of the unit two before it
    // (the buffer's previous user) are done -- normally long before -- so they land while
    // the previous unit still runs; then the unit's K/V tiles as stages come free.
    int units = 0, R = 0, issued = 0;
    auto load_kv = [&](int n, int kvh, int b) -> bool {
      const int s = R % kFwdStages;
      if (!warp_wait(empty(s), ((R / kFwdStages) & 1) ^ 1, ctl)) return false;
      mbar_expect_tx_elect(full(s), 2 * L::kTileBytes);
      XATTN_DCHECK(kvh < nkv && n <= (S - 1) / kTileRows, status);
      load_tile(sK + s * L::kTileBytes, &mk, full(s), kvh, n * kTileRows, b);
      load_tile(sV + s * L::kTileBytes, &mv, full(s), kvh, n * kTileRows, b);
      issued = ++R;
      return true;
    };
    bool ok = true;
#pragma unroll 1
    for (int k = 0; ok; ++k) {
      const int u = unit_at(k);
      if (u >= num_units) break;
      XATTN_FWD_UNIT(u);
      const int qb = units % kQBufs;
      const uint32_t sQb = sQ + qb * 2 * L::kTileBytes;
      // Phase units/kQBufs - 1 of mma_final[qb]: the products of unit units - kQBufs.
      if (!warp_wait(mma_final(qb), ((units / kQBufs) & 1) ^ 1, ctl)) break;
      mbar_expect_tx_elect(q_full(qb), (hasB ? 2 : 1) * L::kTileBytes);
      load_tile(sQb, &mq, q_full(qb), h, mA * kTileRows, b);
      if (hasB) load_tile(sQb + L::kTileBytes, &mq, q_full(qb), h, mB * kTileRows, b);
      ++units;
#pragma unroll 1
      for (int n = 0; ok && n <= n_last; ++n) ok = load_kv(n, kvh, b);
    }
    // Let every copy in flight land before the CTA can exit.
    for (int j = (units > kQBufs ? units - kQBufs : 0); j < units; ++j)
      mbar_drain(q_full(j % kQBufs), (j / kQBufs) & 1, ctl);
    for (int n = (issued > kFwdStages ? issued - kFwdStages : 0); n < issued; ++n)
      mbar_drain(full(n % kFwdStages), (n / kFwdStages) & 1, ctl);
  } else if (warp == 1 || warp == 3) {
    // ---------------- MMA issuers: warp 1 for query tile A, warp 3 for tile B ----------------
    // Two issuers let the two softmax warpgroups run independently of each other's pace
    // (a single issuer would impose its own A/B order), and split the issue cost over two
    // SM sub-partitions. The tensor pipe takes their MMAs in arrival order; the K/V
    // stages are released by a commit from each (empty counts 2).
    const int x = warp == 1 ? 0 : 1;
    constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false, false);
    // PV is one N = 64 product per 64-column sub-tile of V (and of O) at hd = 128.
    constexpr uint32_t idesc_pv = idesc_bf16_f32(128, HD / L::kSubTiles, false, true);
    constexpr uint32_t kStageDesc = L::kTileBytes >> 4;        // tile stride, descriptor units
    constexpr uint32_t kSubDesc = L::kSubBytes >> 4;           // sub-tile stride
    constexpr uint32_t kVStep = (16 * L::kAtomBytes) >> 4;     // 16 key rows of V
    // Descriptors are built once; a K step of 16 elements is +32 bytes (+2) within the
    // swizzled K-major rows of Q and K (the fifth step starts the second sub-tile), and
    // +16 rows of the MN-major V tile.
    const uint64_t dQ = smem_desc(sQ, 16, 8 * L::kAtomBytes, L::kSwizzle) + x * kStageDesc;
    const uint64_t dK = smem_desc(sK, 16, 8 * L::kAtomBytes, L::kSwizzle);
    const uint64_t dV = smem_desc(sV, 8192, 8 * L::kAtomBytes, L::kSwizzle);
    const uint32_t tSx = tS(x), tOx = tO(x), tPx = tP(x);
    // Each product's MMAs and commits are issued by one elected lane; the warp then
    // reconverges.
    auto issue_qk = [&](int s, int qb) {
      const uint64_t dQb = dQ + qb * 2 * kStageDesc;
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t koff = (kk / 4) * kSubDesc + (kk % 4) * 2;
          mma_ss(tSx, dQb + koff, dK + s * kStageDesc + koff, idesc_qk, kk > 0);
        }
        mma_commit(s_full(x));
      }
      __syncwarp();
    };
    // Release of stage s: each issuer that uses key tile n commits once, or twice when it
    // is the tile's only user.
    auto issue_pv = [&](int s, bool first, bool sole_user) {
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < kTileRows / 16; ++kk)
#pragma unroll
          for (int c = 0; c < L::kSubTiles; ++c)
            mma_ts(tOx + c * (HD / L::kSubTiles), tPx + kk * 8, dV + s * kStageDesc + c * kSubDesc + kk * kVStep,
                   idesc_pv, (!first || kk > 0) ? 1u : 0u);
        mma_commit(o_done(x));
        mma_commit(empty(s));                      // this issuer is done with K_n and V_n
        if (sole_user) mma_commit(empty(s));
      }
      __syncwarp();
    };
    // Per key tile n: S_X(n+1) as soon as the softmax has loaded S_X(n) (s_free), then
    // PV_X(n) once P_X(n) is in TMEM (p_full). The next scores are thus computed while the
    // softmax is still producing P_X(n).
    // Release of stage s: each issuer that uses key tile n commits once, or twice when it
    // is the tile's only user (tile mB when there is a tile B; every tile when there is
    // not). An issuer never arrives for a tile it does not use, so its arrivals cannot
    // land in an earlier phase of the stage that the other issuer has not released yet.
    // R: ring index of the unit's key tile 0; gx: this tile's key steps over all units.
    bool ok = true;
    int units = 0, unitsx = 0;
    auto ring_stage = [](int r) { return r % kFwdStages; };
    auto ring_phase = [](int r) { return static_cast<uint32_t>((r / kFwdStages) & 1); };
#pragma unroll 1
    for (int k = 0, R = 0, gx = 0; ok; ++k) {
      const int u = unit_at(k);
      if (u >= num_units) break;
      XATTN_FWD_UNIT(u);
      const int mX = x == 0 ? mA : mB;
      const int qb = units % kQBufs;
      // This unit's Q tiles have landed (phase units/kQBufs of q_full[qb]). Waited for by both
      // issuers in every unit, even without tile B, so each sees every phase in order and
      // its mma_final arrival below can never count towards an earlier use of the buffer.
      if (!warp_wait(q_full(qb), (units / kQBufs) & 1, ctl)) break;
      if (x == 0 || hasB) {
        // The unit's first scores: key tile 0 landed, and S_X of the previous unit read;
        // its first PV overwrites O_X, which the previous epilogue has read.
        ok = warp_wait(full(ring_stage(R)), ring_phase(R), ctl) && warp_wait(s_free(x), (gx - 1) & 1, ctl);
        if (!ok) break;
        tc_fence_after();
        issue_qk(ring_stage(R), qb);
        if (!warp_wait(o_free(x), (unitsx - 1) & 1, ctl)) { ok = false; break; }
#pragma unroll 1
        for (int n = 0; n <= mX; ++n, ++gx) {
          const bool shared_tile = x == 0 ? hasB : n <= mA;
          if constexpr (!L::kAliasP) {
            if (n + 1 <= mX) {
              if (!warp_wait(s_free(x), gx & 1, ctl) ||
                  !warp_wait(full(ring_stage(R + n + 1)), ring_phase(R + n + 1), ctl)) { ok = false; break; }
              tc_fence_after();
              issue_qk(ring_stage(R + n + 1), qb);
            }
            if (!warp_wait(p_full(x), gx & 1, ctl)) { ok = false; break; }
            tc_fence_after();
            issue_pv(ring_stage(R + n), n == 0, !shared_tile);
          } else {
            // P_X(n) sits in S_X's columns: PV_X(n) first, then S_X(n+1) over them.
            if (!warp_wait(p_full(x), gx & 1, ctl)) { ok = false; break; }
            tc_fence_after();
            issue_pv(ring_stage(R + n), n == 0, !shared_tile);
            if (n + 1 <= mX) {
              if (!warp_wait(full(ring_stage(R + n + 1)), ring_phase(R + n + 1), ctl)) { ok = false; break; }
              tc_fence_after();
              issue_qk(ring_stage(R + n + 1), qb);
            }
          }
        }
        if (!ok) break;
        ++unitsx;
      }
      if (elect_one()) mma_commit(mma_final(qb));  // covers every MMA of this unit
      __syncwarp();
      R += n_last + 1;
      ++units;
    }
    if (units > 0) mbar_drain(mma_final((units - 1) % kQBufs), ((units - 1) / kQBufs) & 1, ctl);
  } else if (warp >= 4) {
    // ---------------- softmax + epilogue: one thread per query row of tile X ----------------
    const int x = (warp - 4) >> 2;          // 0 = tile A, 1 = tile B
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tSx = tS(x) + lane_off, tOx = tO(x) + lane_off, tPx = tP(x) + lane_off;
    bool ok = true;
#pragma unroll 1
    for (int k = 0, gx = 0; ok; ++k) {
      const int u = unit_at(k);
      if (u >= num_units) break;
      XATTN_FWD_UNIT(u);
      const int mX = x == 0 ? mA : mB;
      if (x == 1 && !hasB) continue;
      float mrow = -INFINITY, lrow = 0.f;
      // One key step; `masked` selects the diagonal tile's copy, compiled apart from the
      // loop over the other tiles so that their code carries no mask. On the diagonal
      // tile the warp's rows are 32 q .. 32 q + 31 (q = quarter): 32-column chunks below q
      // are wholly visible, chunk q is masked per lane (key column > row), chunks above q
      // are wholly masked (P = 0 without exponentials); q is warp-uniform, so each chunk
      // takes one branch-free path.
      auto step = [&](auto masked, int n) -> bool {
        constexpr bool kDiag = decltype(masked)::value;
        if (!warp_wait(s_full(x), gx & 1, ctl)) return false;
        tc_fence_after();
        // The whole row of S_X(n) comes into registers with one TMEM read, and the buffer
        // is released at once: S_X(n+1) is computed while this softmax runs.
        uint32_t r[128];
#pragma unroll
        for (int c = 0; c < 128; c += 32) tmem_ld_x32(tSx + c, r + c);
        tmem_wait_ld();
        reg_fence<128>(r);
        tc_fence_before();
        mbar_arrive(s_free(x));
        // The row maximum of the scaled scores: the scaled maximum of the raw scores
        // (scale >= 0) or their scaled minimum (scale < 0); masked columns do not count.
        constexpr float kFill = kNegScale ? INFINITY : -INFINITY;
        float mx4[4] = {kFill, kFill, kFill, kFill};
        auto max_chunk = [&](auto mask_chunk, int c32) {
#pragma unroll
          for (int c = c32; c < c32 + 32; c += 2) {
            float v0 = __uint_as_float(r[c]), v1 = __uint_as_float(r[c + 1]);
            if (decltype(mask_chunk)::value) {
              if (c > row) v0 = kFill;
              if (c + 1 > row) v1 = kFill;
            }
            float &a = mx4[(c >> 1) & 3];
            a = kNegScale ? fmin3(a, v0, v1) : fmax3(a, v0, v1);
          }
        };
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          if (!kDiag || cc < quarter) max_chunk(std::false_type{}, 32 * cc);
          else if (cc == quarter) max_chunk(std::true_type{}, 32 * cc);
        }
        const float mx = (kNegScale ? fmin3(mx4[0], mx4[1], fminf(mx4[2], mx4[3]))
                                    : fmax3(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3]))) * scale_log2;
        // Conditional rescaling: keep the stale max unless some row of the warp grew by
        // more than 2^8; the decision is per warp because TMEM loads/stores are collective.
        const float mnew = fmaxf(mrow, mx);
        const bool rescale = __any_sync(0xffffffffu, mnew > mrow + 8.0f);
        const float m_use = rescale ? mnew : mrow;
        // rescale is warp-uniform, so this is a uniform branch: the common path issues no
        // special-function op here (one would queue behind the other warpgroup's
        // exponentials on the shared unit).
        float alpha = 1.f;
        if (rescale) alpha = ex2_approx(mrow - mnew);
        const float neg_m = -m_use;
        // Exponents, the causal mask on them (-inf -> exact zeros for any scale, 0
        // included), the exponentials, row sums and bf16 P, packed in place into r[0, 64).
        // One pair in eight of the other tiles' chunks is exponentiated on the FMA pipe
        // (exp2_fma2) instead of MUFU, which both tiles' softmax warps share (the diagonal
        // copy keeps MUFU: measured slightly faster there).
        // The first three quarters of P are computed before waiting for the previous PV_X
        // (which still reads P_X), so that product's latency overlaps the exponentials;
        // storing them before the last quarter keeps the register peak at one S row.
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
        auto exp_chunk = [&](auto mask_chunk, int c32) {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int c = c32 + 2 * e;
            float x0, x1;
            ffma2(x0, x1, __uint_as_float(r[c]), __uint_as_float(r[c + 1]), scale_log2, scale_log2,
                  neg_m, neg_m);
            if (decltype(mask_chunk)::value) {
              if (c > row) x0 = -INFINITY;
              if (c + 1 > row) x1 = -INFINITY;
            }
            float p0, p1;
            if (!kDiag && !decltype(mask_chunk)::value && (e & 7) == 7) {
              exp2_fma2(x0, x1, p0, p1);
            } else {
              p0 = ex2_approx(x0);
              p1 = ex2_approx(x1);
            }
            const int a = (e & 1) * 2;
            fadd2(ps[a], ps[a + 1], ps[a], ps[a + 1], p0, p1);
            r[c32 / 2 + e] = pack_bf16x2(p0, p1);
          }
        };
        auto chunk = [&](int cc) {
          if (!kDiag || cc < quarter) {
            exp_chunk(std::false_type{}, 32 * cc);
          } else if (cc == quarter) {
            exp_chunk(std::true_type{}, 32 * cc);
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) r[16 * cc + e] = 0u;
          }
        };
        chunk(0);
        chunk(1);
        chunk(2);
        if (!warp_wait(o_done(x), (gx - 1) & 1, ctl)) return false;
        tc_fence_after();
        tmem_st_x32(tPx, r);
        tmem_st_x16(tPx + 32, r + 32);
        chunk(3);
        tmem_st_x16(tPx + 48, r + 48);
        if (rescale && n > 0) {
#pragma unroll
          for (int c = 0; c < HD; c += 32) {
            uint32_t ov[32];
            tmem_ld_x32(tOx + c, ov);
            tmem_wait_ld();
            reg_fence<32>(ov);
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st_x32(tOx + c, ov);
          }
        }
        lrow = lrow * alpha + ((ps[0] + ps[1]) + (ps[2] + ps[3]));
        mrow = m_use;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(p_full(x));
        return true;
      };
#pragma unroll 1
      for (int n = 0; n < mX; ++n, ++gx) {
        if (!step(std::false_type{}, n)) { ok = false; break; }
      }
      if (ok) {
        if (!step(std::true_type{}, mX)) ok = false;
        ++gx;
      }
      if (!ok) break;
      // Epilogue: O / l in bf16 and the LSE; then O_X is free for the next unit.
      if (!warp_wait(o_done(x), (gx - 1) & 1, ctl)) break;
      tc_fence_after();
      const int i = mX * kTileRows + row;
      const float inv = 1.f / lrow;
      __nv_bfloat16 *orow = o + (static_cast<size_t>(b) * S + i) * nh * HD + static_cast<size_t>(h) * HD;
      XATTN_DCHECK(i >= S || (static_cast<size_t>(b) * S + i) * nh * HD + static_cast<size_t>(h + 1) * HD <=
                                 static_cast<size_t>(B) * S * nh * HD,
                   status);
#pragma unroll
      for (int c = 0; c < HD; c += 32) {
        uint32_t ov[32];
        tmem_ld_x32(tOx + c, ov);
        tmem_wait_ld();
        reg_fence<32>(ov);
        if (i < S) {
          uint4 *dst = reinterpret_cast<uint4 *>(orow + c);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_uint4(
                pack_bf16x2(__uint_as_float(ov[8 * e + 0]) * inv, __uint_as_float(ov[8 * e + 1]) * inv),
                pack_bf16x2(__uint_as_float(ov[8 * e + 2]) * inv, __uint_as_float(ov[8 * e + 3]) * inv),
                pack_bf16x2(__uint_as_float(ov[8 * e + 4]) * inv, __uint_as_float(ov[8 * e + 5]) * inv),
                pack_bf16x2(__uint_as_float(ov[8 * e + 6]) * inv, __uint_as_float(ov[8 * e + 7]) * inv));
        }
      }
      if (i < S) lse[(static_cast<size_t>(b) * S + i) * nh + h] = (mrow + __log2f(lrow)) * kLn2;
      tc_fence_before();
      mbar_arrive(o_free(x));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}
#undef XATTN_FWD_UNIT

template <int HD, bool kNegScale, int kRing>
cudaError_t launch_fwd_sign(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                            __nv_bfloat16 *o, float *lse, int B, int S, int nh, int nkv, float scale,
                            int *status, uint64_t timeout_ns, cudaStream_t stream) {
  using L = FwdLayout<HD, kRing>;
  cudaError_t err = cudaFuncSetAttribute(attn_fwd_kernel<HD, kNegScale, kRing>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kDynBytes);
  if (err != cudaSuccess) return err;
  // Persistent CTAs: one per SM, or one per unit when there are fewer units.
  int dev = 0, sms = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
  const int num_m = (S + kTileRows - 1) / kTileRows;
  const long long units = static_cast<long long>(B) * nh * ((num_m + 1) / 2);
  const unsigned grid = static_cast<unsigned>(units < sms ? units : sms);
  return launch_pdl(attn_fwd_kernel<HD, kNegScale, kRing>, grid, kFwdThreads, L::kDynBytes, stream, mq, mk, mv, o,
                    lse, B, S, nh, nkv, scale * kLog2e, status, timeout_ns);
}

template <int HD>
cudaError_t launch_fwd_hd(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                          __nv_bfloat16 *o, float *lse, int B, int S, int nh, int nkv, float scale,
                          int *status, uint64_t timeout_ns, cudaStream_t stream) {
  constexpr int kRingGroups = FwdLayout<HD>::kStages;
  constexpr int kRingMha = HD == 128 ? kRingGroups : 4;
  if (nh == nkv) {
    if (scale < 0.f)
      return launch_fwd_sign<HD, true, kRingMha>(mq, mk, mv, o, lse, B, S, nh, nkv, scale, status, timeout_ns, stream);
    return launch_fwd_sign<HD, false, kRingMha>(mq, mk, mv, o, lse, B, S, nh, nkv, scale, status, timeout_ns, stream);
  }
  if (scale < 0.f)
    return launch_fwd_sign<HD, true, kRingGroups>(mq, mk, mv, o, lse, B, S, nh, nkv, scale, status, timeout_ns, stream);
  return launch_fwd_sign<HD, false, kRingGroups>(mq, mk, mv, o, lse, B, S, nh, nkv, scale, status, timeout_ns, stream);
}

}  // namespace

cudaError_t launch_fwd_bf16(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                            __nv_bfloat16 *o, float *lse, int B, int S, int nh, int nkv, int hd,
                            float scale, int *status, uint64_t timeout_ns, cudaStream_t stream) {
  if (hd == 64)
    return launch_fwd_hd<64>(mq, mk, mv, o, lse, B, S, nh, nkv, scale, status, timeout_ns, stream);
  if (hd == 32)
    return launch_fwd_hd<32>(mq, mk, mv, o, lse, B, S, nh, nkv, scale, status, timeout_ns, stream);
  if (hd == 128)
    return launch_fwd_hd<128>(mq, mk, mv, o, lse, B, S, nh, nkv, scale, status, timeout_ns, stream);
  return cudaErrorInvalidValue;
}

}  // namespace xattn
