// Backward of fused causal attention with grouped KV heads on sm_103a tensor cores.
//
// Method (xtrain "演进总览" / docs/evolution.md, phase table row T14): recompute the
// scores from Q, K and the saved log-sum-exp, use D_i = dO_i . O_i in place of the
// softmax Jacobian, and produce dQ, dK, dV. Row T15: the gradient of a kv head is the
// sum over its query group, taken deterministically without atomics.
//
// Three kernels, in stream order:
//   1. preprocess (HBM-bound): D_i = sum_d dO_id O_id in fp32, and per query row the
//      bf16 auxiliary operand row holding -LSE_i/scale and -D_i.
//   2. main, this file (tensor cores): dK and dV. A unit of work is one (batch, kv head,
//      128-row key tile n); persistent CTAs, one per SM, take the units in turn. The K_n
//      and V_n tiles stay in shared memory; the dK_n / dV_n accumulators stay in TMEM
//      while the CTA walks every query head r of the group and every query tile m >= n
//      (causal tile skipping). That walk *is* the group sum of row T15: no atomics on
//      dK/dV, and a fixed order, so they are reproducible. Per (r, m):
//        S^T  = K_n Q_m^T - LSE/scale   (TMEM, 128 x 128 fp32; the per-query term is one
//        dP^T = V_n dO_m^T - D          extra tensor-core K step over the auxiliary rows)
//        P^T  = exp2(S^T scale log2e)               -> bf16 into TMEM
//        dS^T = P^T dP^T                            -> bf16 into TMEM (for dK) and, with
//                                                      fused dQ, shared memory (for dQ)
//        dV_n += P^T dO_m ,  dK_n += dS^T Q_m       (A operands from TMEM; with fused dQ
//                                                      and one query head per kv head,
//                                                      dK reads dS^T from shared memory)
//      The softmax scale of dS is applied once, to dK_n in the epilogue.
//      Warps: 0 = TMA producer, 1 = TMEM owner + MMA issuer of S^T and dV,
//      3 = MMA issuer of dP^T and dK, 4-7 = P, 8-11 = dS (one thread per key row).
//   3. dQ: by default the main kernel also computes dQ_m = dS K_n per iteration and
//      adds it into an fp32 accumulator with TMA reduce-adds, and a convert kernel
//      writes dq = bf16(scale * accumulator); the deterministic backward instead runs
//      the query-stationary dQ kernel of attn_bwd_dq_sm103.cu (dQ accumulated in TMEM
//      over the key tiles, written once).
#include <type_traits>

#include "sm103_ptx.cuh"
#include "xattn_internal.h"

namespace xattn {

// Workspace: auxiliary rows | D | (fused dQ only) the fp32 dQ accumulator.
size_t bwd_workspace_bytes(int B, int S, int nh, int hd, bool fused_dq) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t rows = static_cast<size_t>(B) * nh * padded_rows(S);
  const size_t base = up(rows * kAuxCols * 2) + up(static_cast<size_t>(B) * S * nh * 4);
  return fused_dq ? base + up(static_cast<size_t>(B) * S * nh * hd * 4) : base;
}

BwdWorkspace bwd_workspace_carve(void *base, int B, int S, int nh, int hd) {
  (void)hd;
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t rows = static_cast<size_t>(B) * nh * padded_rows(S);
  uint8_t *p = static_cast<uint8_t *>(base);
  BwdWorkspace ws;
  ws.aux = reinterpret_cast<__nv_bfloat16 *>(p);
  ws.D = reinterpret_cast<float *>(p + up(rows * kAuxCols * 2));
  ws.dqacc = reinterpret_cast<float *>(p + up(rows * kAuxCols * 2) + up(static_cast<size_t>(B) * S * nh * 4));
  return ws;
}

namespace {

// ------------------------------------------------------------------------------------
// 1. preprocess
// ------------------------------------------------------------------------------------
// v ~= hi + mid + lo with three bf16 terms (each rounded to nearest); the residual is
// below 2^-26 |v|.
__device__ __forceinline__ void split3_bf16(float v, uint16_t out[3]) {
  const __nv_bfloat16 hi = __float2bfloat16_rn(v);
  const float r1 = v - __bfloat162float(hi);
  const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
  const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
  out[0] = __bfloat16_as_ushort(hi);
  out[1] = __bfloat16_as_ushort(mid);
  out[2] = __bfloat16_as_ushort(lo);
}

// One group of (hd / 8) lanes per row (b, i, h): each lane reads 8 bf16 of O and dO
// (16 B each), the group reduces with shuffles. Rows are enumerated in memory order of
// O/dO, so the loads are fully coalesced. The same lanes zero the row of the fused dQ
// accumulator when there is one (dqacc non-null). The group's first lane writes D_i in
// fp32 (read by the dQ kernel, [B, S, nh] like lse) and the row's auxiliary operand:
// -LSE/scale and -D, the two per-query terms that the dK/dV kernel's tensor-core
// products add to S^T and dP^T. Pad rows (S <= i < S_pad) are all zero: their Q and dO
// rows are zero too, so they contribute nothing whatever P is there.
template <int HD>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(
    const __nv_bfloat16 *__restrict__ o, const __nv_bfloat16 *__restrict__ dO,
    const float *__restrict__ lse, uint4 *__restrict__ aux, float *__restrict__ D,
    float *__restrict__ dqacc, int B, int S, int nh, float lse_mult) {
  constexpr int kLanesPerRow = HD / 8;
  grid_dep_launch();
  grid_dep_wait();
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
    if (dqacc != nullptr) {
      float4 *z = reinterpret_cast<float4 *>(dqacc + row * HD + sub * 8);
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (sub == 0) {
      D[row] = acc;
      const int h = static_cast<int>(row % nh);
      const long long bi = row / nh;
      const int i = static_cast<int>(bi % S);
      const int b = static_cast<int>(bi / S);
      const size_t dst = (static_cast<size_t>(b) * nh + h) * S_pad + i;
      uint16_t l[3], d[3];
      split3_bf16(-lse[row] * lse_mult, l);
      split3_bf16(-acc, d);
      aux[2 * dst] = make_uint4(l[0] | (static_cast<uint32_t>(l[1]) << 16), l[2] | (static_cast<uint32_t>(d[0]) << 16),
                                d[1] | (static_cast<uint32_t>(d[2]) << 16), 0u);
      aux[2 * dst + 1] = make_uint4(0u, 0u, 0u, 0u);
    }
  } else if (row - n_rows < n_pad && sub == 0) {
    const long long p = row - n_rows;
    const int pad = S_pad - S;
    const long long bh = p / pad;
    const int i = S + static_cast<int>(p % pad);
    aux[2 * (bh * S_pad + i)] = make_uint4(0u, 0u, 0u, 0u);
    aux[2 * (bh * S_pad + i) + 1] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// ------------------------------------------------------------------------------------
// 2. main kernel
// ------------------------------------------------------------------------------------
// 12 warps. Registers are split evenly over the 4 SM sub-partitions (3 warps each), so
// the per-thread limit is 65536 / 4 / 96 rounded down to the allocation granule.
constexpr int kBwdThreads = 384;

// kFusedDq: the kernel also computes dQ = dS K per iteration and adds it into the fp32
// accumulator with TMA reduce-adds (the default backward). Without it the kernel writes
// dK and dV only and the query-stationary dQ kernel produces dQ (the deterministic
// backward); dS^T then stays in TMEM, so dK reads it there and the shared memory of the
// dS tile and the dQ staging goes to a fourth Q / dO stage.
template <int HD, bool kFusedDq>
struct BwdLayout {
  // Two rings of query-tile operands, each sized by how long a stage is held: Q and the
  // auxiliary rows are read until dK(t), at the very end of an iteration; dO only until
  // dP^T(t) and dV(t).
  // hd = 128 (dK / dV only): 32 KB tiles leave room for two stages of each, every tile
  // is two 64-column sub-tiles laid out like hd = 64 tiles (a 256-byte row does not fit
  // one 128-byte swizzle atom), and dV, dK take 128 TMEM columns each, so P^T is written
  // over S^T and dS^T over dP^T (kAlias).
  static_assert(!(kFusedDq && HD == 128), "hd = 128 runs with the query-stationary dQ kernel");
  static constexpr bool kAlias = HD == 128;
  static constexpr int kQStages = HD == 128 ? 2 : kFusedDq ? 3 : 4;  // Q + auxiliary rows
  static constexpr int kOStages = HD == 128 ? 2 : kFusedDq ? 2 : 4;  // dO
  static constexpr uint32_t kRowBytes = HD * 2;
  static constexpr uint32_t kTileBytes = kTileRows * kRowBytes;
  static constexpr uint32_t kAtomBytes = kRowBytes < 128 ? kRowBytes : 128;  // sub-tile row
  static constexpr int kSubTiles = static_cast<int>(kRowBytes / kAtomBytes);
  static constexpr uint32_t kSubBytes = kTileRows * kAtomBytes;
  static constexpr uint32_t kSwizzle = (HD == 32) ? kSwizzle64 : kSwizzle128;
  static constexpr uint32_t kK = 0;
  static constexpr uint32_t kV = kK + kTileBytes;
  static constexpr uint32_t kQ = kV + kTileBytes;                    // kQStages stages
  static constexpr uint32_t kdO = kQ + kQStages * kTileBytes;        // kOStages stages
  // Fused dQ only: three 128 x 128 bf16 dS tiles (32 KB each; iteration t uses tile
  // t % 3, so dS(t+1) is written while dK(t) and dQ(t) still read dS(t)). Once dK(t) and
  // dQ(t) are done the tile stages dQ(t) for the TMA reduce-add (fp32, 2 head-dim halves x
  // 128 rows of HD/2 floats, swizzled like the tensor map's box): the dQ drain never waits
  // for an earlier reduce-add, and dS(t+3) waits for the reduce-add of dQ(t) to have read
  // the tile, two iterations later. The resident dQ uses tiles t % 2 only.
  static constexpr uint32_t kdS = kdO + kOStages * kTileBytes;
  static constexpr uint32_t kdSBytes = 32768;
  static constexpr int kdSTiles = 3;
  static constexpr uint32_t kDqRowBytes = HD / 2 * 4;
  static constexpr uint32_t kDqHalfBytes = kTileRows * kDqRowBytes;
  static_assert(!kFusedDq || 2 * kDqHalfBytes <= kdSBytes, "a dQ tile is staged in a dS tile");
  // Auxiliary K step of S^T and dP^T: the key-side operand is constant (ones under the
  // LSE columns, or under the D columns, of every row), so it is three 8-row x 16-byte
  // core matrices read without swizzle and with a zero row-group stride: [1 1 1 0 ...],
  // [0 0 0 1 1 1 0 0] and zeros. The query-side rows (128 x 16 bf16, 32-byte swizzle,
  // 4 KB) come with each stage.
  static constexpr uint32_t kAuxTileBytes = kTileRows * kAuxCols * 2;
  static constexpr uint32_t kAuxA = kFusedDq ? kdS + kdSTiles * kdSBytes : kdS;
  static constexpr uint32_t kAuxB = kAuxA + 1024;                    // kQStages stages
  static constexpr int kNumBars = 1 + 2 * (kQStages + kOStages) + (kFusedDq ? 21 : 11);
  static constexpr uint32_t kBars = kAuxB + kQStages * kAuxTileBytes;
  static constexpr uint32_t kMisc = kBars + 8 * kNumBars;
  static constexpr uint32_t kUsed = kMisc + 32;
  static constexpr uint32_t kDynBytes = kUsed + 1024;
  static_assert(kDynBytes <= 227 * 1024, "exceeds the opt-in shared memory of one CTA");
  static_assert(kAuxB % 1024 == 0 && kdS % 1024 == 0, "tile alignment");
};

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtl &ctl) {
  const bool ok = mbar_wait(bar, parity, ctl);
  return __all_sync(0xffffffffu, ok);
}

// Offset of element (key row j, query column i) of the 128 x 128 dS^T tile in shared
// memory (fused dQ): two 64-column halves of 128-byte rows (one row per key) with the
// 128-byte swizzle (16-byte chunk ^= row % 8). Read as the A operand of dQ = dS K it is
// MN-major (M = query, contiguous); read as the A operand of dK = dS^T Q it is K-major
// (M = key rows, K = query), so one copy serves both products.
__device__ __forceinline__ uint32_t ds_offset(int j, int i) {
  return static_cast<uint32_t>((i >> 6) * 16384 + j * 128 + ((((i & 63) >> 3) ^ (j & 7)) << 4));
}

// Role map (12 warps):
//   warp 0     : TMA producer
//   warp 1     : TMEM owner; MMA issuer of S^T and dV
//   warp 2     : fused dQ: the dQ reducer, TMA reduce-adds of each staged dQ tile into
//                the fp32 accumulator (2 bulk operations per tile instead of scattered
//                atomics); otherwise idle
//   warp 3     : MMA issuer of dP^T, dK (and dQ)
//   warps 4-7  : P^T = exp2(S^T scale log2e), S^T already holding -LSE/scale, one
//                thread per key row, all 128 query columns (the special-function work)
//   warps 8-11 : dS^T = P^T (dP^T - D), dP^T already holding -D, one thread per key
//                row (the FMA work); fused dQ: also the dQ drain (TMEM -> the shared-
//                memory dS tile the dQ was computed from, one query row per thread)
// The two compute warpgroups work on consecutive (r, m) iterations at the same time, so
// each SM sub-partition runs one warp of each and the exponentials of iteration t+1
// overlap the dS arithmetic of iteration t.
// TMEM columns: S^T [0,128) fp32 | dP^T [128,256) fp32 | P^T bf16 [256,320) |
//               dV [320,384) | dK [384,448) | dQ fp32 (fused) or dS^T bf16 [448,512)
//               (kDsTmem: dS^T bf16 over dP^T's first 64 columns)
// Each region has one producer and its readers release it with an mbarrier before it is
// rewritten: S^T (s_free), dP^T (dp_free; kDsTmem: ds_full and the issue order of dK),
// P^T (p_free by the dS warps, dv_done by the dV product), dQ (dq_empty) or dS^T
// (dk_done).
// mdq (fused dQ only): fp32 map over the dQ accumulator.
//
// kResident (with kFusedDq, small problems): a CTA takes every key tile of one (batch, kv
// head) in turn, and the dQ tiles of the head's query rows stay in TMEM (columns
// [448, 512): the head's group x num_m dQ tiles must fit, group * num_m * HD <= 64),
// accumulated over the key tiles in a fixed order and written once, in bf16, after the
// head's last key tile: no fp32 accumulator in global memory, no reduce-adds, no convert
// pass, and dQ is reproducible. dq: the bf16 output (resident mode only).
//
// kDsTmem (fused dQ, not resident): dK reads dS^T from TMEM (see below).
template <int HD, bool kFusedDq, bool kResident = false, bool kDsTmem = false>
__global__ void __maxnreg__(168)
    attn_bwd_main_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                         const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
                         const __grid_constant__ CUtensorMap maux, const __grid_constant__ CUtensorMap mdq,
                         __nv_bfloat16 *__restrict__ dk,
                         __nv_bfloat16 *__restrict__ dv, __nv_bfloat16 *__restrict__ dq, int B, int S, int nh,
                         int nkv, float scale, int *status, unsigned long long timeout_ns) {
  static_assert(kFusedDq || !kResident, "the resident dQ is a fused-dQ mode");
  using L = BwdLayout<HD, kFusedDq>;
  constexpr int kQS = L::kQStages, kOS = L::kOStages;
  // kDsTmem (fused dQ, not resident): the dS warps also write dS^T in bf16 over the
  // first 64 columns of dP^T (which they have read by then), and dK reads its A operand
  // there instead of from the shared-memory dS tile (32 KB less shared-memory traffic per
  // iteration; only dQ reads the tile). The next dP^T overwrites those columns, so the
  // dS side issues it after dK (its MMAs execute in issue order) instead of as soon as
  // the dS warps have read dP^T: worth it on long units (query groups; measured on gqa
  // 92.4 -> 89.9 us, long 314 -> 307 us), not on the short units of one query head per
  // kv head (32 x 1024 x 12 heads: 193.8 -> 196.6 us).
  static_assert(!kDsTmem || (kFusedDq && !kResident), "dS^T in TMEM is a fused-dQ mode");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  // Warp-uniform by construction; the broadcast lets the compiler see it.
  const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0), lane = threadIdx.x & 31;

  // Work units (key tile n, batch b, kv head kvh). The CTAs are persistent: CTA c of G
  // takes unit k G + c in even rounds k and k G + G - 1 - c in odd ones, which evens out
  // the CTAs' total work. Every role walks the same units; the barriers' phases count
  // iterations over all of them.
  // With query groups (group > 1) the units are numbered most work first (n ascending):
  // they are long, and the order balances the CTAs. With one query head per kv head the
  // units are short (at most num_m iterations) and are numbered head by head instead
  // (n fastest), so the CTAs running at the same time work on the same heads and share
  // their Q, dO and auxiliary tiles in L2 (measured on 32 x 1024 x 12 heads: 248 -> 202
  // us; on the grouped workloads the same order is 10 % slower).
  const int num_m = (S + kTileRows - 1) / kTileRows;
  const int BK = B * nkv;
  const int group = nh / nkv;
  const int num_units = num_m * BK;
  const bool head_major = kResident || group == 1;
  const int G = static_cast<int>(gridDim.x), cta = static_cast<int>(blockIdx.x);
  // Resident dQ: CTA c takes heads c, c + G, ... and each head's key tiles in order.
  auto unit_at = [&](int k) {
    if constexpr (kResident) return (cta + G * (k / num_m)) * num_m + k % num_m;
    return k * G + ((k & 1) ? G - 1 - cta : cta);
  };
  int n = 0, b = 0, kvh = 0, per_head = 0, T = 0;
  auto set_unit = [&](int u) {
    const int bk = head_major ? u / num_m : u % BK;
    n = head_major ? u % num_m : u / BK;
    b = bk / nkv;
    kvh = bk % nkv;
    per_head = num_m - n;                 // query tiles m = n .. num_m-1
    T = group * per_head;                 // iterations (r, m)
  };

  const uint32_t sK = smem_u32(smem + L::kK);
  const uint32_t sV = smem_u32(smem + L::kV);
  const uint32_t sQ = smem_u32(smem + L::kQ);
  const uint32_t sdO = smem_u32(smem + L::kdO);
  uint8_t *sdS_ptr = smem + L::kdS;          // fused dQ only
  const uint32_t sdS = smem_u32(sdS_ptr);
  const uint32_t sAuxA = smem_u32(smem + L::kAuxA);
  const uint32_t sAuxB = smem_u32(smem + L::kAuxB);
  // scale == 0: S^T is the auxiliary term alone (-LSE log2 e) and is not scaled.
  const bool qk = (scale != 0.f);
  const float scale_log2 = qk ? scale * kLog2e : 1.f;
  const uint32_t bar0 = smem_u32(smem + L::kBars);
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  const uint32_t kv_full = bar(0);
  auto q_full = [&](int s) { return bar(1 + s); };
  auto q_empty = [&](int s) { return bar(1 + kQS + s); };
  auto o_full = [&](int s) { return bar(1 + 2 * kQS + s); };
  auto o_empty = [&](int s) { return bar(1 + 2 * kQS + kOS + s); };
  constexpr int kB = 1 + 2 * (kQS + kOS);
  const uint32_t s_full = bar(kB + 0), s_free = bar(kB + 1), dp_full = bar(kB + 2), dp_free = bar(kB + 3);
  const uint32_t p_full = bar(kB + 4), p_free = bar(kB + 5), dv_done = bar(kB + 6), ds_full = bar(kB + 7);
  const uint32_t acc_done = bar(kB + 8);     // a unit's products are done
  const uint32_t acc_free = bar(kB + 9);     // its epilogue has read dV and dK
  const uint32_t dk_done = bar(kB + 10);                              // dK(t) read dS^T(t)
  const uint32_t dq_full = bar(kB + 10), dq_empty = bar(kB + 11);     // fused dQ
  // dQ staged in dS tile t % 3 / that tile read by its reduce-add: one phase of each per
  // use of the tile. (One dqs_full for all tiles would be ambiguous: the drain no longer
  // waits for the previous reduce-add, so it can run two phases ahead of the reducer.)
  auto dqs_full = [&](int tile) { return bar(tile == 0 ? kB + 12 : kB + 18 + tile); };
  auto dqs_empty = [&](int tile) { return bar(tile == 0 ? kB + 13 : kB + 16 + tile); };
  // Resident dQ: dS tile b's readers (dK and dQ of its iteration) are done (one phase per
  // use of the tile), and the head's dQ tiles have been read out of TMEM.
  auto ds_done = [&](int buf) { return bar(kB + 14 + buf); };
  const uint32_t dqt_free = bar(kB + 16);
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMisc + 16);
  const WaitCtl ctl{abort_flag, status, timeout_ns};

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(kv_full, 1);
    for (int s = 0; s < kQS; ++s) {
      mbar_init(q_full(s), 1);
      mbar_init(q_empty(s), 2);                      // one commit from each MMA issuer
    }
    for (int s = 0; s < kOS; ++s) {
      mbar_init(o_full(s), 1);
      mbar_init(o_empty(s), 2);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, 128);
    mbar_init(dp_full, 1);
    mbar_init(dp_free, 128);
    mbar_init(p_full, 128);
    mbar_init(p_free, 128);
    mbar_init(dv_done, 1);
    mbar_init(ds_full, 128);
    mbar_init(acc_done, 2);
    mbar_init(acc_free, 256);
    if constexpr (kFusedDq) {
      mbar_init(dq_full, 1);
      mbar_init(dq_empty, 128);
      for (int i = 0; i < L::kdSTiles; ++i) {
        mbar_init(dqs_full(i), 128);
        mbar_init(dqs_empty(i), 1);
      }
      mbar_init(ds_done(0), 1);
      mbar_init(ds_done(1), 1);
      mbar_init(dqt_free, 128);
    } else {
      mbar_init(dk_done, 1);
    }
    fence_mbar_init();
  }
  // Constant key-side auxiliary core matrices (8 rows of 16 bytes each): [1 1 1 0 0 0 0 0]
  // (S^T), [0 0 0 1 1 1 0 0] (dP^T), zeros (the second 8 columns of the K step).
  if (threadIdx.x < 24) {
    const int cm = threadIdx.x / 8, r = threadIdx.x % 8;
    const uint32_t one = 0x3F80u;   // bf16 1.0
    const uint4 val = (cm == 0) ? make_uint4(one | (one << 16), one, 0u, 0u)
                    : (cm == 1) ? make_uint4(0u, one << 16, one | (one << 16), 0u)
                                : make_uint4(0u, 0u, 0u, 0u);
    *reinterpret_cast<uint4 *>(smem + L::kAuxA + cm * 128 + r * 16) = val;
  }
  fence_proxy_async_smem();
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mq);
    tma_prefetch_desc(&mk);
    tma_prefetch_desc(&mv);
    tma_prefetch_desc(&mdo);
    tma_prefetch_desc(&maux);
    if constexpr (kFusedDq) tma_prefetch_desc(&mdq);
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
  // hd = 128: S^T [0,128) with P^T in its first 64 columns | dP^T [128,256) with dS^T
  // in its first 64 | dV [256,384) | dK [384,512).
  const uint32_t tS = tmem, tdP = tmem + 128, tP = L::kAlias ? tS : tmem + 256;
  const uint32_t tdV = tmem + (L::kAlias ? 256 : 320), tdK = tmem + 384;
  const uint32_t tdQ = tmem + 448;                                       // fused dQ: dQ
  const uint32_t tdS = (L::kAlias || kDsTmem) ? tdP : tmem + 448;        // dS^T (bf16)
  // One 128-row tile of a [B, S, heads, hd] tensor: one TMA box per 64-column sub-tile.
  // Debug builds check the tile's coordinates (heads < nh covers both Q/dO and K/V) and
  // that it lands inside the K / V / Q / dO region of shared memory.
  const int S_pad = num_m * kTileRows;
  (void)S_pad;
  auto load_tile = [&](uint32_t dst, const CUtensorMap *map, uint32_t bar, int head, int row0, int bb) {
    XATTN_DCHECK(head >= 0 && head < nh && row0 >= 0 && row0 < S_pad && row0 % kTileRows == 0 && bb >= 0 &&
                     bb < B && dst >= sK && dst + L::kTileBytes <= smem_u32(smem + L::kdO) + kOS * L::kTileBytes,
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
    // The Q / dO rings run on across units. A unit's first kOStages ring loads only need
    // stages released by earlier iterations, so they are issued before waiting for the
    // previous unit's products (acc_done): only then are K and V overwritten. (Waits for
    // the phase before the first -- parity 1 of a fresh barrier -- return at once, so
    // the first unit and iteration need no special case in any role.)
    int issued_q = 0, issued_o = 0, units = 0;
    int g = 0, sq = 0, uq = 0, so = 0, uo = 0;
    auto load_ring = [&](int t) -> bool {
      const int h = kvh * group + t / per_head, m = n + t % per_head;
      if (!warp_wait(q_empty(sq), (uq & 1) ^ 1, ctl)) return false;
      mbar_expect_tx_elect(q_full(sq), L::kTileBytes + L::kAuxTileBytes);
      load_tile(sQ + sq * L::kTileBytes, &mq, q_full(sq), h, m * kTileRows, b);
      XATTN_DCHECK(sq < kQS && m < num_m && h < nh, status);
      tma_load_4d_elect(sAuxB + sq * L::kAuxTileBytes, &maux, q_full(sq), 0, m * kTileRows, h, b);
      issued_q = g + 1;
      if (!warp_wait(o_empty(so), (uo & 1) ^ 1, ctl)) return false;
      mbar_expect_tx_elect(o_full(so), L::kTileBytes);
      load_tile(sdO + so * L::kTileBytes, &mdo, o_full(so), h, m * kTileRows, b);
      issued_o = g + 1;
      ++g;
      if (++sq == kQS) { sq = 0; ++uq; }
      if (++so == kOS) { so = 0; ++uo; }
      return true;
    };
    bool ok = true;
#pragma unroll 1
    for (int k = 0; ok; ++k) {
      const int u = unit_at(k);
      if (u >= num_units) break;
      set_unit(u);
      const int pre = T < kOS ? T : kOS;
      for (int t = 0; ok && t < pre; ++t) ok = load_ring(t);
      if (!ok || !warp_wait(acc_done, (units - 1) & 1, ctl)) break;
      mbar_expect_tx_elect(kv_full, 2 * L::kTileBytes);
      XATTN_DCHECK(kvh < nkv && n < num_m, status);
      load_tile(sK, &mk, kv_full, kvh, n * kTileRows, b);
      load_tile(sV, &mv, kv_full, kvh, n * kTileRows, b);
      ++units;
      for (int t = pre; ok && t < T; ++t) ok = load_ring(t);
    }
    // Every load has landed before the CTA can exit (the consumers may have given up).
    if (units > 0) mbar_drain(kv_full, (units - 1) & 1, ctl);
    for (int t = (issued_q > kQS ? issued_q - kQS : 0); t < issued_q; ++t)
      mbar_drain(q_full(t % kQS), (t / kQS) & 1, ctl);
    for (int t = (issued_o > kOS ? issued_o - kOS : 0); t < issued_o; ++t)
      mbar_drain(o_full(t % kOS), (t / kOS) & 1, ctl);
  } else if (warp == 1 || warp == 3) {
    // ---------------- MMA issuers (converged warps, one elected lane issues) ----------------
    // Warp 1 issues the products the P warps depend on (S^T, dV); warp 3 those of the dS
    // warps (dP^T, dK, and dQ when fused). Each stream is in order, but neither waits
    // behind the other, so S^T(t+1) never queues behind a dQ that is waiting for the dQ
    // drain. The tensor
    // pipe takes the two streams' MMAs in arrival order; each stage is released by one
    // commit from each issuer (empty counts 2), and acc_done gets one from each.
    const bool p_side = warp == 1;
    constexpr uint32_t idesc_t = idesc_bf16_f32(128, 128, false, false);  // S^T, dP^T
    // dV, dK (A K-major): one N = 64 product per 64-column sub-tile at hd = 128.
    constexpr uint32_t idesc_acc = idesc_bf16_f32(128, HD / L::kSubTiles, false, true);
    constexpr uint32_t kStageDesc = L::kTileBytes >> 4;   // stage stride, descriptor units
    constexpr uint32_t kSubDesc = L::kSubBytes >> 4;      // sub-tile stride
    constexpr uint32_t kRowStep = (16 * L::kAtomBytes) >> 4;  // 16 rows of an MN-major tile
    // Descriptors are built once. K-major operands advance +32 bytes (+2) per
    // 16-element K step (the fifth step starts the second sub-tile); MN-major ones
    // advance 16 rows.
    const uint64_t kA_k = smem_desc(p_side ? sK : sV, 16, 8 * L::kAtomBytes, L::kSwizzle);
    const uint64_t kB_k = smem_desc(p_side ? sQ : sdO, 16, 8 * L::kAtomBytes, L::kSwizzle);
    const uint64_t kQ_mn = smem_desc(sQ, 8192, 8 * L::kAtomBytes, L::kSwizzle);
    const uint64_t kdO_mn = smem_desc(sdO, 8192, 8 * L::kAtomBytes, L::kSwizzle);
    const uint64_t kK_mn = smem_desc(sK, 8192, 8 * L::kAtomBytes, L::kSwizzle);       // fused dQ
    const uint64_t kdS_mn = smem_desc(sdS, 16384, 1024, kSwizzle128);
    const uint64_t kdS_k = smem_desc(sdS, 16, 1024, kSwizzle128);
    constexpr uint32_t idesc_dq = idesc_bf16_f32(128, HD, true, true);  // dQ (A = dS, MN-major)
    // No swizzle: LBO = the distance to the zero core matrix (second K chunk), SBO = 0.
    const uint64_t kAuxA = p_side ? smem_desc(sAuxA, 256, 0, 0) : smem_desc(sAuxA + 128, 128, 0, 0);
    const uint64_t kAuxQ = smem_desc(sAuxB, 16, 256, kSwizzle32);
    constexpr uint32_t kAuxStageDesc = L::kAuxTileBytes >> 4;
    // S^T = K Q^T - LSE/scale (P side) or dP^T = V dO^T - D (dS side): the head-dim K
    // steps, then one auxiliary K step that adds the per-query term (key-side ones x
    // query-side terms). With scale == 0 S^T is the auxiliary term alone.
    const uint32_t tD = p_side ? tS : tdP;
    const bool with_qk = p_side ? qk : true;
    // The score product of iteration u reads Q ring stage sq (Q, or only the auxiliary
    // rows on the dS side) and, on the dS side, dO ring stage so.
    const uint32_t t_full = p_side ? s_full : dp_full;    // this side's score product
    const uint32_t t_free = p_side ? s_free : dp_free;
    // Each product's MMAs and commits are issued by one elected lane; the warp then
    // reconverges.
    auto issue_t = [&](int sq, int so) {
      if (elect_one()) {
        if (with_qk) {
          const uint64_t b_k = kB_k + (p_side ? sq : so) * kStageDesc;
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t koff = (kk / 4) * kSubDesc + (kk % 4) * 2;
            mma_ss(tD, kA_k + koff, b_k + koff, idesc_t, kk > 0);
          }
        }
        mma_ss(tD, kAuxA, kAuxQ + sq * kAuxStageDesc, idesc_t, with_qk ? 1u : 0u);
        mma_commit(t_full);
        if (!p_side) mma_commit(o_empty(so));        // dP^T is the dS side's last dO read
      }
      __syncwarp();
    };
    // Each issuer waits for the stages it reads, phase by phase: the P side for Q before
    // S^T and for dO before dV, the dS side for both before dP^T.
    auto wait_operands = [&](int u, int sq, int so) {
      return warp_wait(q_full(sq), (u / kQS) & 1, ctl) &&
             (p_side || warp_wait(o_full(so), (u / kOS) & 1, ctl));
    };
    bool ok = true;
    int units = 0, heads = 0;
#pragma unroll 1
    for (int k = 0, g = 0, sq = 0, so = 0; ok; ++k) {
      const int u = unit_at(k);
      if (u >= num_units) break;
      set_unit(u);
      // The unit's first score product: K and V have landed, and this side's warps have
      // read the previous score tile (the last one of the previous unit).
      // kDsTmem, dS side: the previous dP^T columns hold the last dS^T, which this warp's
      // own dK (issued before) reads first; the dS warps had read that dP^T before ds_full.
      ok = warp_wait(kv_full, units & 1, ctl) && wait_operands(g, sq, so) &&
           ((kDsTmem && !p_side) || warp_wait(t_free, (g - 1) & 1, ctl));
      // With P^T over S^T, S^T overwrites the previous P^T: the dS warps have read it.
      if (L::kAlias && p_side) ok = ok && warp_wait(p_free, (g - 1) & 1, ctl);
      if (!ok) break;
      tc_fence_after();
      issue_t(sq, so);
      // The unit's first accumulation overwrites dV / dK: the previous unit's epilogue
      // has read them.
      if (!warp_wait(acc_free, (units - 1) & 1, ctl)) break;
#pragma unroll 1
      for (int t = 0; t < T; ++t, ++g) {
        const int sq1 = (sq + 1 == kQS) ? 0 : sq + 1;
        const int so1 = (so + 1 == kOS) ? 0 : so + 1;
        const bool more = t + 1 < T;
        const uint32_t ph = g & 1;
        // The next score product as soon as this side's warps have read the current one
        // -- or, with P^T / dS^T in the score columns (kAlias), after this iteration's dV
        // / dK product (the tensor pipe runs one thread's MMAs in issue order, so that
        // product reads P^T / dS^T before the next scores overwrite them) and, on the P
        // side, once the dS warps have read P^T.
        auto issue_next = [&]() -> bool {
          if (!more) return true;
          if (!wait_operands(g + 1, sq1, so1) || (!(kDsTmem && !p_side) && !warp_wait(t_free, ph, ctl)))
            return false;
          if (L::kAlias && p_side && !warp_wait(p_free, ph, ctl)) return false;
          tc_fence_after();
          issue_t(sq1, so1);
          return true;
        };
        if (!L::kAlias && !(kDsTmem && !p_side) && !issue_next()) { ok = false; break; }
        if (p_side) {
          if (!warp_wait(o_full(so), (g / kOS) & 1, ctl) || !warp_wait(p_full, ph, ctl)) { ok = false; break; }
          tc_fence_after();
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < kTileRows / 16; ++kk)                      // dV += P^T dO
#pragma unroll
              for (int c = 0; c < L::kSubTiles; ++c)
                mma_ts(tdV + c * (HD / L::kSubTiles), tP + kk * 8,
                       kdO_mn + so * kStageDesc + c * kSubDesc + kk * kRowStep, idesc_acc,
                       (t > 0 || kk > 0) ? 1u : 0u);
            mma_commit(dv_done);
            mma_commit(q_empty(sq));                 // S^T and dV are done with both stages
            mma_commit(o_empty(so));
          }
          __syncwarp();
        } else {
          if (!warp_wait(ds_full, ph, ctl)) { ok = false; break; }
          tc_fence_after();
          if constexpr (kFusedDq) {
            const uint32_t dsb = (kResident ? (g & 1) : (g % L::kdSTiles)) * (L::kdSBytes >> 4);  // dS tile
            if (elect_one()) {
#pragma unroll
              for (int kk = 0; kk < kTileRows / 16; ++kk) {                  // dK += dS^T Q
                if constexpr (kDsTmem)
                  mma_ts(tdK, tdS + kk * 8, kQ_mn + sq * kStageDesc + kk * kRowStep, idesc_acc,
                         (t > 0 || kk > 0) ? 1u : 0u);
                else
                  mma_ss(tdK, kdS_k + dsb + (kk >> 2) * 1024 + (kk & 3) * 2,
                         kQ_mn + sq * kStageDesc + kk * kRowStep, idesc_acc, (t > 0 || kk > 0) ? 1u : 0u);
              }
              mma_commit(q_empty(sq));               // dP^T and dK are done with the Q stage
            }
            __syncwarp();
            // kDsTmem: the next dP^T, over this dS^T, after dK in issue order.
            if (kDsTmem && !issue_next()) { ok = false; break; }
            if constexpr (kResident) {
              // dQ of query tile (r, m) += dS K_n, in its own TMEM columns; the head's first
              // key tile (n = 0, which every query tile sees) overwrites. The head's first
              // product waits for the previous head's dQ read-out.
              if (n == 0 && t == 0 && !warp_wait(dqt_free, (heads - 1) & 1, ctl)) { ok = false; break; }
              tc_fence_after();
              const uint32_t col = static_cast<uint32_t>(((t / per_head) * num_m + n + t % per_head) * HD);
              XATTN_DCHECK(col + HD <= 64u, status);     // the resident dQ tiles fit columns [448, 512)
              if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < kTileRows / 16; ++kk)
                  mma_ss(tdQ + col, kdS_mn + dsb + kk * 128, kK_mn + kk * kRowStep, idesc_dq, (n > 0 || kk > 0) ? 1u : 0u);
                mma_commit(ds_done(g & 1));            // dK and dQ are done with dS tile g % 2
              }
              __syncwarp();
            } else {
              if (!warp_wait(dq_empty, ph ^ 1, ctl)) { ok = false; break; }
              tc_fence_after();
              if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < kTileRows / 16; ++kk)                  // dQ = dS K
                  mma_ss(tdQ, kdS_mn + dsb + kk * 128, kK_mn + kk * kRowStep, idesc_dq, kk > 0);
                mma_commit(dq_full);
              }
              __syncwarp();
            }
          } else {
            if (elect_one()) {
#pragma unroll
              for (int kk = 0; kk < kTileRows / 16; ++kk)                    // dK += dS^T Q
#pragma unroll
                for (int c = 0; c < L::kSubTiles; ++c)
                  mma_ts(tdK + c * (HD / L::kSubTiles), tdS + kk * 8,
                         kQ_mn + sq * kStageDesc + c * kSubDesc + kk * kRowStep, idesc_acc,
                         (t > 0 || kk > 0) ? 1u : 0u);
              mma_commit(q_empty(sq));               // dP^T and dK are done with the Q stage
              mma_commit(dk_done);
            }
            __syncwarp();
          }
        }
        if (L::kAlias && !issue_next()) { ok = false; break; }
        sq = sq1;
        so = so1;
      }
      if (!ok) break;
      if (elect_one()) mma_commit(acc_done);
      __syncwarp();
      ++units;
      if (n == num_m - 1) ++heads;            // resident dQ: the head's last key tile
    }
    if (units > 0) mbar_drain(acc_done, (units - 1) & 1, ctl);
  } else if (kFusedDq && !kResident && warp == 2) {
    // ---------------- dQ reducer ----------------
    // Both head-dim halves of a staged tile are issued before one wait for their reads.
    bool ok = true;
#pragma unroll 1
    for (int k = 0, g = 0; ok; ++k) {
      const int u = unit_at(k);
      if (u >= num_units) break;
      set_unit(u);
#pragma unroll 1
      for (int t = 0; t < T; ++t, ++g) {
        if (!warp_wait(dqs_full(g % L::kdSTiles), (g / L::kdSTiles) & 1, ctl)) { ok = false; break; }
        if (lane == 0) {
          const int h = kvh * group + t / per_head, m = n + t % per_head;
          const uint32_t src = smem_u32(sdS_ptr + (g % L::kdSTiles) * L::kdSBytes);
          // fp32 box: the innermost coordinates 0 and HD/2 are 16-byte multiples.
          XATTN_DCHECK(h < nh && m < num_m && (HD / 2) % 4 == 0 && src >= sdS &&
                           src + 2 * L::kDqHalfBytes <= sdS + L::kdSTiles * L::kdSBytes,
                       status);
          tma_reduce_add_4d(&mdq, src, 0, h, m * kTileRows, b);
          tma_reduce_add_4d(&mdq, src + L::kDqHalfBytes, HD / 2, h, m * kTileRows, b);
          bulk_commit_group();
          bulk_wait_read_all();        // the tile may take the next dS
          mbar_arrive(dqs_empty(g % L::kdSTiles));
        }
        __syncwarp();
      }
    }
    if (lane == 0) bulk_wait_all();    // every reduce-add has landed before the CTA exits
    __syncwarp();
  } else if (warp >= 4 && warp < 8) {
    // ---------------- P^T: one thread per key row j, 4 chunks of 32 query columns ----------------
    const int quarter = warp & 3;
    const int j = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    bool ok = true;
#pragma unroll 1
    for (int k = 0, g = 0, units = 0; ok; ++k) {
      const int u = unit_at(k);
      if (u >= num_units) break;
      set_unit(u);
#pragma unroll 1
      for (int t = 0; t < T; ++t, ++g) {
        const int m = n + t % per_head;
        const bool diag = (m == n);
        if (!warp_wait(s_full, g & 1, ctl)) { ok = false; break; }
        tc_fence_after();
        // The whole row of S^T(t) comes into registers with one TMEM read and the buffer is
        // released at once, so S^T(t+1) is computed while these exponentials run.
        uint32_t r[128];
#pragma unroll
        for (int c = 0; c < 128; c += 32) tmem_ld_x32(tS + lane_off + c, r + c);
        tmem_wait_ld();
        reg_fence<128>(r);
        tc_fence_before();
        mbar_arrive(s_free);
        // 4 chunks of 32 query columns. Within a chunk the 32 exponents are computed
        // first, then the 32 exponentials, then the bf16 pairs: independent
        // special-function operations back to back, which one warp per SM sub-partition
        // needs to keep that unit busy (measured: the exponential chunks take half the
        // time of a per-pair interleaved order). On the diagonal tile, query column
        // i < key row j is masked (P = 0); the common body has no mask.
        auto chunk = [&](auto masked, auto chunk_index, uint32_t *pk) {
          constexpr int c = decltype(chunk_index)::value;
          float xs[32];
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            fmul2(xs[e], xs[e + 1], __uint_as_float(r[32 * c + e]), __uint_as_float(r[32 * c + e + 1]),
                  scale_log2, scale_log2);
#pragma unroll
          for (int e = 0; e < 32; ++e) xs[e] = ex2_approx(xs[e]);
          if constexpr (decltype(masked)::value) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (32 * c + e < j) xs[e] = 0.f;
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(xs[2 * e], xs[2 * e + 1]);
        };
        auto body = [&](auto masked) -> bool {
          uint32_t pk[16];
          chunk(masked, std::integral_constant<int, 0>{}, pk);
          // P^T of the previous iteration must have been read by the dS warps and by dV.
          if (!warp_wait(p_free, (g - 1) & 1, ctl) || !warp_wait(dv_done, (g - 1) & 1, ctl)) return false;
          tc_fence_after();
          tmem_st_x16(tP + lane_off, pk);
          chunk(masked, std::integral_constant<int, 1>{}, pk);
          tmem_st_x16(tP + lane_off + 16, pk);
          chunk(masked, std::integral_constant<int, 2>{}, pk);
          tmem_st_x16(tP + lane_off + 32, pk);
          chunk(masked, std::integral_constant<int, 3>{}, pk);
          tmem_st_x16(tP + lane_off + 48, pk);
          return true;
        };
        if (!(diag ? body(std::true_type{}) : body(std::false_type{}))) ok = false;
        if (!ok) break;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(p_full);
      }
      if (!ok) break;
      // Epilogue: dV rows (bf16), then the dV columns are free for the next unit.
      if (!warp_wait(acc_done, units & 1, ctl)) break;
      tc_fence_after();
      const int jg = n * kTileRows + j;
      const size_t row_off = (static_cast<size_t>(b) * S + jg) * nkv * HD + static_cast<size_t>(kvh) * HD;
      XATTN_DCHECK(jg >= S || row_off + HD <= static_cast<size_t>(B) * S * nkv * HD, status);
#pragma unroll
      for (int c = 0; c < HD; c += 16) {
        uint32_t v[16];
        tmem_ld_x16(tdV + lane_off + c, v);
        tmem_wait_ld();
        reg_fence<16>(v);
        if (jg < S) {
          uint4 *dst = reinterpret_cast<uint4 *>(dv + row_off + c);
#pragma unroll
          for (int e = 0; e < 2; ++e)
            dst[e] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * e]), __uint_as_float(v[8 * e + 1])),
                                pack_bf16x2(__uint_as_float(v[8 * e + 2]), __uint_as_float(v[8 * e + 3])),
                                pack_bf16x2(__uint_as_float(v[8 * e + 4]), __uint_as_float(v[8 * e + 5])),
                                pack_bf16x2(__uint_as_float(v[8 * e + 6]), __uint_as_float(v[8 * e + 7])));
        }
      }
      tc_fence_before();
      mbar_arrive(acc_free);
      ++units;
    }
  } else if (warp >= 8) {
    // ---------------- dS^T (and the fused dQ drain): one thread per key row j ----------------
    const int quarter = warp & 3;
    const int j = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    // Fused dQ: dQ(k) from TMEM (query row j of its tile) into dS tile k % 3 (dK(k) and
    // dQ(k), its last readers, are done once dq_full shows dQ(k)), swizzled like the
    // reduce's tensor-map box (two halves of HD/2 floats per row); warp 2 then adds it to
    // global memory. The phases of dq_full are waited in order, one per call: dQ(k+1) is
    // only issued after this call has read dQ(k) (dq_empty).
    auto drain_dq = [&](int k) -> bool {
      if (!warp_wait(dq_full, k & 1, ctl)) return false;
      tc_fence_after();
      uint32_t v[HD];
#pragma unroll
      for (int c = 0; c < HD; c += 32) tmem_ld_x32(tdQ + lane_off + c, v + c);
      tmem_wait_ld();
      reg_fence<HD>(v);
      tc_fence_before();
      mbar_arrive(dq_empty);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint8_t *row = sdS_ptr + (k % L::kdSTiles) * L::kdSBytes + half * L::kDqHalfBytes + j * L::kDqRowBytes;
        XATTN_DCHECK(half * L::kDqHalfBytes + (j + 1) * L::kDqRowBytes <= L::kdSBytes, status);
#pragma unroll
        for (int ch = 0; ch < HD / 8; ++ch) {
          const int sw = (HD == 64) ? (ch ^ (j & 7)) : (ch ^ ((j >> 1) & 3));
          const uint32_t *x = v + half * (HD / 2) + 4 * ch;
          *reinterpret_cast<uint4 *>(row + (sw << 4)) = make_uint4(x[0], x[1], x[2], x[3]);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(dqs_full(k % L::kdSTiles));
      return true;
    };
    bool ok = true;
#pragma unroll 1
    for (int k = 0, g = 0, units = 0; ok; ++k) {
      const int u = unit_at(k);
      if (u >= num_units) break;
      set_unit(u);
#pragma unroll 1
      for (int t = 0; t < T; ++t, ++g) {
        if (!warp_wait(p_full, g & 1, ctl) || !warp_wait(dp_full, g & 1, ctl)) { ok = false; break; }
        tc_fence_after();
        // 4 chunks of 32 query columns: P^T bf16 (16 TMEM columns) and dP^T (32 columns).
        uint32_t pa[16], da[32], pb[16], db[32];
        tmem_ld_x16(tP + lane_off, pa);
        tmem_ld_x32(tdP + lane_off, da);
        tmem_wait_ld();
        reg_fence<16>(pa);
        reg_fence<32>(da);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t *pc = (c & 1) ? pb : pa, *dc = (c & 1) ? db : da;
          uint32_t *pn = (c & 1) ? pa : pb, *dn = (c & 1) ? da : db;
          if (c < 3) {
            tmem_ld_x16(tP + lane_off + 16 * (c + 1), pn);
            tmem_ld_x32(tdP + lane_off + 32 * (c + 1), dn);
          }
          // The dS^T buffer about to be written has been read. Without fused dQ the previous
          // dK read dS^T from TMEM (dk_done); the fused cases follow below.
          if (!kFusedDq && c == 0) {
            if (!warp_wait(dk_done, (g - 1) & 1, ctl)) {
              tmem_wait_ld();    // the loads of chunk 1 are still in flight
              ok = false;
              break;
            }
            tc_fence_after();
          }
          // Resident dQ (no per-iteration dQ drain): wait for dK and dQ of iteration g-2,
          // the last readers of dS tile g % 2 (one phase of ds_done per use of the tile).
          if (kResident && c == 0) {
            if (!warp_wait(ds_done(g & 1), ((g >> 1) & 1) ^ 1, ctl)) {
              tmem_wait_ld();
              ok = false;
              break;
            }
          }
          // Fused dQ: tile g % 3 last staged dQ(g-3); its reduce-add has read it (one phase
          // of dqs_empty per use of the tile). dK(g-3) and dQ(g-3) were done before that
          // dQ was drained.
          if (kFusedDq && !kResident && c == 0) {
            if (!warp_wait(dqs_empty(g % L::kdSTiles), ((g / L::kdSTiles) & 1) ^ 1, ctl)) {
              tmem_wait_ld();
              ok = false;
              break;
            }
          }
          uint32_t dsk[16];
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            const uint32_t p01 = pc[2 * q4], p23 = pc[2 * q4 + 1];
            float t0, t1, t2, t3;
            fmul2(t0, t1, __uint_as_float(dc[4 * q4]), __uint_as_float(dc[4 * q4 + 1]), bf16lo_to_f32(p01),
                  bf16hi_to_f32(p01));
            fmul2(t2, t3, __uint_as_float(dc[4 * q4 + 2]), __uint_as_float(dc[4 * q4 + 3]), bf16lo_to_f32(p23),
                  bf16hi_to_f32(p23));
            dsk[2 * q4] = pack_bf16x2(t0, t1);
            dsk[2 * q4 + 1] = pack_bf16x2(t2, t3);
          }
          if constexpr (kFusedDq) {
            XATTN_DCHECK(ds_offset(j, 32 * c + 24) + 16 <= L::kdSBytes && ds_offset(j, 32 * c) + 16 <= L::kdSBytes,
                         status);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              *reinterpret_cast<uint4 *>(sdS_ptr + (kResident ? (g & 1) : (g % L::kdSTiles)) * L::kdSBytes +
                                         ds_offset(j, 32 * c + 8 * e)) =
                  make_uint4(dsk[4 * e], dsk[4 * e + 1], dsk[4 * e + 2], dsk[4 * e + 3]);
            // dS^T columns [16c, 16c + 16) lie in dP^T columns already read (chunks <= c/2).
            if constexpr (kDsTmem) tmem_st_x16(tdS + lane_off + 16 * c, dsk);
          } else {
            tmem_st_x16(tdS + lane_off + 16 * c, dsk);
          }
          if (c < 3) {
            tmem_wait_ld();
            reg_fence<16>(pn);
            reg_fence<32>(dn);
          }
          if (c == 2) {          // P^T(t) and dP^T(t) are all in registers
            tc_fence_before();
            mbar_arrive(p_free);
            if constexpr (!kDsTmem) mbar_arrive(dp_free);   // kDsTmem: ds_full covers it
          }
        }
        if (!ok) break;
        if constexpr (kFusedDq) {
          if constexpr (kDsTmem) {
            tmem_wait_st();
            tc_fence_before();
          }
          fence_proxy_async_smem();
          mbar_arrive(ds_full);
          if (!kResident && t > 0 && !drain_dq(g - 1)) { ok = false; break; }
        } else {
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(ds_full);
        }
      }
      if (!ok) break;
      // Epilogue: the unit's last dQ (fused), then the dK rows (bf16, times the softmax
      // scale); the dK columns are then free for the next unit.
      if constexpr (kFusedDq && !kResident) {
        if (!drain_dq(g - 1)) break;
      }
      if (!warp_wait(acc_done, units & 1, ctl)) break;
      tc_fence_after();
      const int jg = n * kTileRows + j;
      const size_t row_off = (static_cast<size_t>(b) * S + jg) * nkv * HD + static_cast<size_t>(kvh) * HD;
      XATTN_DCHECK(jg >= S || row_off + HD <= static_cast<size_t>(B) * S * nkv * HD, status);
#pragma unroll
      for (int c = 0; c < HD; c += 16) {
        uint32_t v[16];
        tmem_ld_x16(tdK + lane_off + c, v);
        tmem_wait_ld();
        reg_fence<16>(v);
        if (jg < S) {
          float f[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) f[e] = __uint_as_float(v[e]) * scale;
          uint4 *dst = reinterpret_cast<uint4 *>(dk + row_off + c);
#pragma unroll
          for (int e = 0; e < 2; ++e)
            dst[e] = make_uint4(pack_bf16x2(f[8 * e], f[8 * e + 1]), pack_bf16x2(f[8 * e + 2], f[8 * e + 3]),
                                pack_bf16x2(f[8 * e + 4], f[8 * e + 5]), pack_bf16x2(f[8 * e + 6], f[8 * e + 7]));
        }
      }
      tc_fence_before();
      mbar_arrive(acc_free);
      ++units;
      if constexpr (kResident) {
        if (n == num_m - 1) {
          // The head's dQ tiles are complete after its last key tile (acc_done covers
          // every dQ product): dq = bf16(scale * accumulator), query row j of each tile.
#pragma unroll 1
          for (int r = 0; r < group; ++r) {
#pragma unroll 1
            for (int m = 0; m < num_m; ++m) {
              const uint32_t col = static_cast<uint32_t>((r * num_m + m) * HD);
              const int i = m * kTileRows + j;
              __nv_bfloat16 *qrow =
                  dq + ((static_cast<size_t>(b) * S + i) * nh + static_cast<size_t>(kvh) * group + r) * HD;
              XATTN_DCHECK(i >= S || ((static_cast<size_t>(b) * S + i) * nh + static_cast<size_t>(kvh) * group + r + 1) *
                                             HD <= static_cast<size_t>(B) * S * nh * HD,
                           status);
#pragma unroll
              for (int c = 0; c < HD; c += 16) {
                uint32_t v[16];
                tmem_ld_x16(tdQ + lane_off + col + c, v);
                tmem_wait_ld();
                reg_fence<16>(v);
                if (i < S) {
                  float f[16];
#pragma unroll
                  for (int e = 0; e < 16; ++e) f[e] = __uint_as_float(v[e]) * scale;
                  uint4 *dst = reinterpret_cast<uint4 *>(qrow + c);
#pragma unroll
                  for (int e = 0; e < 2; ++e)
                    dst[e] = make_uint4(pack_bf16x2(f[8 * e], f[8 * e + 1]), pack_bf16x2(f[8 * e + 2], f[8 * e + 3]),
                                        pack_bf16x2(f[8 * e + 4], f[8 * e + 5]),
                                        pack_bf16x2(f[8 * e + 6], f[8 * e + 7]));
                }
              }
            }
          }
          tc_fence_before();
          mbar_arrive(dqt_free);
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

template <int HD, bool kFusedDq, bool kResident = false, bool kDsTmem = false>
cudaError_t launch_main_hd(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                           const CUtensorMap &mdo, const CUtensorMap &maux, const CUtensorMap &mdq,
                           __nv_bfloat16 *dk, __nv_bfloat16 *dv, __nv_bfloat16 *dq, int B, int S, int nh,
                           int nkv, float scale, int *status, uint64_t timeout_ns, cudaStream_t stream) {
  using L = BwdLayout<HD, kFusedDq>;
  auto kernel = attn_bwd_main_kernel<HD, kFusedDq, kResident, kDsTmem>;
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kDynBytes);
  if (err != cudaSuccess) return err;
  // Persistent CTAs: one per SM, or one per unit (resident dQ: per head) when there are
  // fewer.
  int dev = 0, sms = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
  const long long units = static_cast<long long>(B) * nkv * (kResident ? 1 : (S + kTileRows - 1) / kTileRows);
  const unsigned grid = static_cast<unsigned>(units < sms ? units : sms);
  return launch_pdl(kernel, grid, kBwdThreads, L::kDynBytes, stream, mq, mk, mv, mdo, maux, mdq, dk, dv, dq, B, S,
                    nh, nkv, scale, status, timeout_ns);
}

// 3. dq convert (fused dQ): 8 elements per thread (two 16-byte loads, one 16-byte
// store). The accumulator holds dS K without the softmax scale.
__global__ void __launch_bounds__(256) dq_convert_kernel(const float *__restrict__ acc,
                                                         __nv_bfloat16 *__restrict__ dq,
                                                         size_t n8, float scale) {
  grid_dep_launch();
  grid_dep_wait();
  const size_t t = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= n8) return;
  const float4 a = reinterpret_cast<const float4 *>(acc)[2 * t];
  const float4 c = reinterpret_cast<const float4 *>(acc)[2 * t + 1];
  reinterpret_cast<uint4 *>(dq)[t] =
      make_uint4(pack_bf16x2(a.x * scale, a.y * scale), pack_bf16x2(a.z * scale, a.w * scale),
                 pack_bf16x2(c.x * scale, c.y * scale), pack_bf16x2(c.z * scale, c.w * scale));
}

}  // namespace

cudaError_t launch_bwd_preprocess(const __nv_bfloat16 *o, const __nv_bfloat16 *dO,
                                  const float *lse, int B, int S, int nh, int hd, float scale,
                                  const BwdWorkspace &ws, bool fused_dq, cudaStream_t stream) {
  float *dqacc = fused_dq ? ws.dqacc : nullptr;
  // -LSE/scale, or -LSE log2 e when scale == 0 (then the main kernel's S^T is the
  // auxiliary term alone and is used unscaled).
  const float lse_mult = (scale == 0.f) ? kLog2e : 1.0f / scale;
  uint4 *aux = reinterpret_cast<uint4 *>(ws.aux);
  const long long n_rows = static_cast<long long>(B) * S * nh;
  const long long n_pad = static_cast<long long>(B) * nh * (padded_rows(S) - S);
  const int lanes = hd / 8;
  const long long threads = (n_rows + n_pad) * lanes;
  const unsigned grid = static_cast<unsigned>((threads + 255) / 256);
  if (hd == 64)
    return launch_pdl(bwd_preprocess_kernel<64>, grid, 256, 0, stream, o, dO, lse, aux, ws.D, dqacc, B, S, nh,
                      lse_mult);
  if (hd == 32)
    return launch_pdl(bwd_preprocess_kernel<32>, grid, 256, 0, stream, o, dO, lse, aux, ws.D, dqacc, B, S, nh,
                      lse_mult);
  if (hd == 128)
    return launch_pdl(bwd_preprocess_kernel<128>, grid, 256, 0, stream, o, dO, lse, aux, ws.D, dqacc, B, S, nh,
                      lse_mult);
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_main_bf16(const CUtensorMap &mq, const CUtensorMap &mk,
                                 const CUtensorMap &mv, const CUtensorMap &mdo,
                                 const CUtensorMap &maux, const CUtensorMap *mdq,
                                 __nv_bfloat16 *dk, __nv_bfloat16 *dv,
                                 int B, int S, int nh, int nkv, int hd, float scale, int *status,
                                 uint64_t timeout_ns, cudaStream_t stream) {
  // Without a dQ accumulator map the kernel computes dK and dV only; its mdq parameter
  // is then unused (maux stands in for it).
  const CUtensorMap &md = mdq ? *mdq : maux;
  if (mdq && nh != nkv) {     // query groups: dK reads dS^T from TMEM
    if (hd == 64)
      return launch_main_hd<64, true, false, true>(mq, mk, mv, mdo, maux, md, dk, dv, nullptr, B, S, nh, nkv, scale,
                                                   status, timeout_ns, stream);
    if (hd == 32)
      return launch_main_hd<32, true, false, true>(mq, mk, mv, mdo, maux, md, dk, dv, nullptr, B, S, nh, nkv, scale,
                                                   status, timeout_ns, stream);
  }
  if (hd == 64)
    return mdq ? launch_main_hd<64, true>(mq, mk, mv, mdo, maux, md, dk, dv, nullptr, B, S, nh, nkv, scale, status, timeout_ns, stream)
               : launch_main_hd<64, false>(mq, mk, mv, mdo, maux, md, dk, dv, nullptr, B, S, nh, nkv, scale, status, timeout_ns, stream);
  if (hd == 32)
    return mdq ? launch_main_hd<32, true>(mq, mk, mv, mdo, maux, md, dk, dv, nullptr, B, S, nh, nkv, scale, status, timeout_ns, stream)
               : launch_main_hd<32, false>(mq, mk, mv, mdo, maux, md, dk, dv, nullptr, B, S, nh, nkv, scale, status, timeout_ns, stream);
  if (hd == 128 && !mdq)
    return launch_main_hd<128, false>(mq, mk, mv, mdo, maux, md, dk, dv, nullptr, B, S, nh, nkv, scale, status, timeout_ns, stream);
  return cudaErrorInvalidValue;
}

bool bwd_resident_dq_ok(int S, int nh, int nkv, int hd) {
  const int num_m = (S + kTileRows - 1) / kTileRows;
  return (hd == 32 || hd == 64) && static_cast<long long>(nh / nkv) * num_m * hd <= 64;
}

cudaError_t launch_bwd_main_resident_bf16(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                                          const CUtensorMap &mdo, const CUtensorMap &maux, __nv_bfloat16 *dk,
                                          __nv_bfloat16 *dv, __nv_bfloat16 *dq, int B, int S, int nh, int nkv,
                                          int hd, float scale, int *status, uint64_t timeout_ns,
                                          cudaStream_t stream) {
  if (!bwd_resident_dq_ok(S, nh, nkv, hd)) return cudaErrorInvalidValue;
  // The resident kernel reads no dQ accumulator map; maux stands in for it.
  if (hd == 64)
    return launch_main_hd<64, true, true>(mq, mk, mv, mdo, maux, maux, dk, dv, dq, B, S, nh, nkv, scale, status,
                                          timeout_ns, stream);
  return launch_main_hd<32, true, true>(mq, mk, mv, mdo, maux, maux, dk, dv, dq, B, S, nh, nkv, scale, status,
                                        timeout_ns, stream);
}

cudaError_t launch_dq_convert(const float *dqacc, __nv_bfloat16 *dq, size_t n_elems,
                              float scale, cudaStream_t stream) {
  const size_t n8 = n_elems / 8;
  const unsigned grid = static_cast<unsigned>((n8 + 255) / 256);
  if (grid == 0) return cudaSuccess;
  return launch_pdl(dq_convert_kernel, grid, 256, 0, stream, dqacc, dq, n8, scale);
}

}  // namespace xattn
