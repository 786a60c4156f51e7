// Decode attention: one new query per sequence against that sequence's cached keys and
// values, for every query head, with grouped KV heads.
//
// Method (xtrain "演进总览" / docs/evolution.md, post-training milestones M2a-M2c): the
// decode step's attention is a single query against the cached K/V and equals the last
// row of full causal attention over the T cached positions; it is batch-agnostic over the
// sequences (M2b decodes a prompt's G samples together, bh = G * nh), and the cache stays
// on the device (M2c). Grouped KV heads as in the training path (row T15): query head h
// reads kv head h / group.
//
// GB300 mapping. Per (sequence, kv head) the work is two thin products against the
// cache -- S^T = K q^T (keys x the group's query heads) and O^T = V^T P^T -- so it is bound
// by HBM reading the cache once. Both products run on the tensor cores (tcgen05, fp32
// accumulators in TMEM), which leaves the CUDA cores only the softmax of a chunk.
//   1. decode_partial_kernel: one CTA of 4 warps per (sequence, kv head, run of chunks),
//      a chunk being C = 16384 / hd keys (512, 256, 128 at hd = 32, 64, 128), so its K and
//      its V are 32 KB each (three CTAs share an SM). A (sequence, kv head) is one run
//      when the B x nkv pairs fill the SMs in one wave of resident CTAs; shorter batches
//      split it into more runs (decode_nsplit).
//      * Loads: one K and one V buffer. Thread 0 issues the run's first TMA loads before
//        anything else (128-key boxes of one kv head, swizzled like the training
//        kernels' tiles; keys past T read as zeros); the next chunk's K loads as soon as
//        this chunk's scores are done, its V as soon as this chunk's P V is done. The
//        threads write the group's query rows, padded to 16 rows, as a K-major tile.
//      * Scores: per 128-key tile, S^T = K q^T (M = 128 keys, N = 16, K = hd) into TMEM.
//      * Softmax: thread i owns key i of every tile (its TMEM lane). The chunk maximum
//        and sum of each head (fp32, log2 domain) are reduced over the CTA; P^T goes to
//        shared memory in bf16 as a K-major operand whose row (tile j, head r) holds the
//        128 keys of tile j; the sum adds the rounded values that P V uses.
//      * P V: one product per chunk. A = the chunk's V tiles read as one MN-major operand
//        of M = 128 rows, row (tile j, head-dim element d) (hd = 64: two tiles, each one
//        64-element swizzle atom; hd = 32: four; hd = 128: one tile of two atoms);
//        B = P^T with N = (C/128) x G columns (tile j', head r). The blocks j = j' are the
//        tiles' partial outputs; the others are discarded (the products are tiny next to
//        the loads).
//      * Merge: thread (tile j, d) reads its block's head columns and folds the chunk into
//        its running output, rescaled by 2^(M_old - M_new) as the run's maximum grows.
//      * End of the run: the tiles' partials are summed through shared memory; a whole
//        sequence writes O (bf16) and LSE = (M + log2 L) ln 2, a part of one writes
//        (M, L, partial O) per head to the scratch.
//   2. decode_combine_kernel (runs > 1 only): one warp per (sequence, query head) merges
//      the runs (rescaling each by 2^(m_r - M)), writes O in bf16 and the LSE.
#include "sm103_ptx.cuh"
#include "xattn_internal.h"

namespace xattn {

int decode_chunk_keys(int hd) { return 16384 / hd; }

size_t decode_workspace_bytes(int B, int T, int nh, int hd) {
  const int ck = decode_chunk_keys(hd);
  const size_t chunks = static_cast<size_t>((T + ck - 1) / ck);
  return static_cast<size_t>(B) * nh * chunks * (static_cast<size_t>(hd) + 2) * sizeof(float);
}

namespace {

constexpr int kDecThreads = 128;   // one thread per key of a 128-key tile (TMEM lane)

// Key runs per (batch, kv head) for bk pairs of `chunks` chunks and `slots` resident CTAs
// on `sms` SMs:
//  * bk >= sms and bk <= slots: one run each (every CTA resident at once, streaming its
//    whole cache; no combine);
//  * bk < sms: as many runs as fill one wave of CTAs (the parallelism a short batch lacks);
//  * bk > slots: the count that minimises (waves of CTAs) x (chunks per CTA, the length of
//    a CTA's chain), a split costing about one chunk more for its combine.
// Every run is non-empty.
int decode_nsplit(int bk, int chunks, int slots, int sms) {
  auto fit = [chunks](int s) {   // largest count <= s whose runs are all non-empty
    s = s < 1 ? 1 : (s > chunks ? chunks : s);
    while (s > 1 && (s - 1) * ((chunks + s - 1) / s) >= chunks) --s;
    return s;
  };
  if (bk <= slots) return bk >= sms ? 1 : fit(slots / bk);
  int best = 1;
  long long best_cost = -1;
  const int top = chunks < 4096 ? chunks : 4096;
  for (int s = 1; s <= top; ++s) {
    if (fit(s) != s) continue;
    const int per = (chunks + s - 1) / s;
    const long long waves = (static_cast<long long>(bk) * s + slots - 1) / slots;
    const long long cost = waves * per + (s > 1 ? 1 : 0);
    if (best_cost < 0 || cost < best_cost) best = s, best_cost = cost;
  }
  return best;
}

// Shared memory and TMEM of one CTA; G = the group padded to 4, 8 or 16 (at least
// 16 / kSub, so that P V has N a multiple of 16).
//   [kK, +32 KB)  the chunk's K tiles (tile j at j * kTileBytes; at hd = 128 two 64-column
//                 sub-tiles each); after the scores, the epilogue's per-tile partials
//                 [kSub][G][HD] fp32
//   [kV, +32 KB)  the chunk's V tiles, same layout
//   [kQP, ...)    the query tile [16 rows x hd] (K-major, the tiles' swizzle), then P^T
//                 [kNpv rows x 128 keys] bf16 (K-major, 128-byte swizzle, two 64-key columns)
//   [kRed, ...)   per-warp maxima and sums [2][4 warps][16 heads]
//   barriers: full_k, full_v, s_done, o_done; TMEM address; abort flag
// TMEM columns: S^T of tile j at [16 j, 16 j + 16); O^T at [kTmemO, kTmemO + kNpv).
template <int HD, int G>
struct DecLayout {
  static constexpr int kSub = 128 / HD;                       // 128-key tiles per chunk
  static constexpr int kChunk = 128 * kSub;                   // keys per chunk
  static constexpr uint32_t kAtomBytes = HD * 2 < 128 ? HD * 2 : 128;   // swizzle-atom row
  static constexpr int kSubTiles = HD * 2 / static_cast<int>(kAtomBytes);
  static constexpr uint32_t kSubBytes = kTileRows * kAtomBytes;
  static constexpr uint32_t kTileBytes = kTileRows * HD * 2;
  static constexpr uint32_t kKVBytes = kSub * kTileBytes;
  static constexpr uint32_t kSwizzle = HD == 32 ? kSwizzle64 : kSwizzle128;
  static constexpr int kNpv = kSub * G;
  static constexpr uint32_t kPColBytes = kNpv * 128;          // 64 keys of every P^T row
  static constexpr uint32_t kPBytes = 2 * kPColBytes;
  static constexpr uint32_t kQColBytes = 16 * kAtomBytes;     // one atom column of the query tile
  static constexpr uint32_t kQBytes = kSubTiles * kQColBytes;
  static constexpr uint32_t kK = 0;
  static constexpr uint32_t kV = kKVBytes;
  static constexpr uint32_t kQP = 2 * kKVBytes;
  static constexpr uint32_t kRed = kQP + (kQBytes + 1023) / 1024 * 1024 + kPBytes;
  static constexpr uint32_t kBars = kRed + 2 * 4 * 16 * 4;
  static constexpr uint32_t kMisc = kBars + 4 * 8;
  static constexpr uint32_t kUsed = kMisc + 32;
  static constexpr uint32_t kDynBytes = kUsed + 1024;        // + alignment of the base to 1 KB
  static constexpr uint32_t kTmemO = 16 * kSub;
  static constexpr uint32_t kTmemCols = kTmemO + kNpv <= 32 ? 32 : (kTmemO + kNpv <= 64 ? 64 : 128);
  static_assert(kNpv % 16 == 0 && kTmemO + kNpv <= 128, "P V: N a multiple of 16, TMEM within 128 columns");
  static_assert(kSub * G * HD * 4 <= kKVBytes, "the epilogue's partials fit the K region");
  static_assert(kPColBytes % 1024 == 0 && kSubBytes % 1024 == 0 && kQP % 1024 == 0,
                "swizzled operands need 1024-byte alignment");
  static_assert(3 * (kDynBytes + 1024) <= 228 * 1024 || G == 16, "three CTAs per SM");
};

// Resident CTAs per SM: shared memory (228 KB, 1 KB reserved per CTA), at most three
// (the launch bounds' register budget).
template <int HD, int G>
constexpr int decode_ctas_per_sm() {
  constexpr int n = static_cast<int>((228u * 1024u) / (DecLayout<HD, G>::kDynBytes + 1024u));
  return n < 3 ? n : 3;
}

// Warp-uniform bounded wait: every lane waits, then all agree.
__device__ __forceinline__ bool dec_warp_wait(uint32_t bar, uint32_t parity, const WaitCtl &ctl) {
  const bool ok = mbar_wait(bar, parity, ctl);
  return __all_sync(0xffffffffu, ok);
}

// A CTA takes one (batch, kv head) and a contiguous run of its chunks [c0, c1): the run's
// chunks stream through one K and one V buffer (the next chunk's K loads as soon as this
// chunk's scores are done, its V as soon as this chunk's P V is done), and the chunks are
// merged online: per head a running maximum M and sum L, and per thread (tile j, element
// d) the partial outputs of its O^T row, rescaled by 2^(M_old - M_new) as M grows.
// Whole sequences in one run (nsplit == 1) end with O (bf16) and the LSE; otherwise each
// run writes a record (M, L, partial O) per head, merged by decode_combine_kernel.
// GV: heads computed (the group rounded up to 4, 8 or 16; GV <= G). Heads GV..G-1 only pad
// the operand tiles: their scores are not reduced and their P^T rows are not written (they
// reach O^T columns that nothing reads).
template <int HD, int G, int GV>
__global__ void __launch_bounds__(kDecThreads, 3) decode_partial_kernel(
    const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
    const __nv_bfloat16 *__restrict__ q, float *__restrict__ ws_o, float *__restrict__ ws_ml,
    __nv_bfloat16 *__restrict__ o, float *__restrict__ lse, int B, int T, int nh, int nkv, int nsplit,
    float scale_log2, int *status, unsigned long long timeout_ns) {
  using L = DecLayout<HD, G>;
  static_assert(GV <= G, "computed heads within the padded tile");
  extern __shared__ uint8_t dsm_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0), lane = threadIdx.x & 31;
  const int t = threadIdx.x;
  const int group = nh / nkv;
  const int BK = B * nkv;
  const int bk = static_cast<int>(blockIdx.x % static_cast<unsigned>(BK));
  const int split = static_cast<int>(blockIdx.x / static_cast<unsigned>(BK));
  const int b = bk / nkv, kvh = bk % nkv;
  const int chunks = (T + L::kChunk - 1) / L::kChunk;
  const int per = (chunks + nsplit - 1) / nsplit;
  const int c0 = split * per, c1 = min(chunks, c0 + per);    // c0 < c1 (the host picks nsplit)

  const uint32_t sK = smem_u32(smem + L::kK), sV = smem_u32(smem + L::kV), sQP = smem_u32(smem + L::kQP);
  float *red_max = reinterpret_cast<float *>(smem + L::kRed);   // [4][16]
  float *red_sum = red_max + 64;                                  // [4][16]
  const uint32_t bar0 = smem_u32(smem + L::kBars);
  const uint32_t full_k = bar0, full_v = bar0 + 8, s_done = bar0 + 16, o_done = bar0 + 24;
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMisc + 16);
  const WaitCtl ctl{abort_flag, status, timeout_ns};

  // Loads of chunk c's K tiles (or V tiles) into the K (V) buffer, by thread 0.
  auto load_kv = [&](const CUtensorMap *map, uint32_t dst, uint32_t bar, int c) {
    XATTN_DCHECK(b < B && kvh < nkv && c < chunks, status);
    mbar_expect_tx(bar, L::kKVBytes);
#pragma unroll
    for (int j = 0; j < L::kSub; ++j)
#pragma unroll
      for (int sub = 0; sub < L::kSubTiles; ++sub)
        tma_load_4d(dst + j * L::kTileBytes + sub * L::kSubBytes, map, bar, sub * 64, kvh,
                    c * L::kChunk + j * kTileRows, b);
  };
  // Thread 0 starts the first chunk's loads first; the TMEM allocation and the query tile
  // follow while they are in flight.
  if (t == 0) {
    *abort_flag = 0;
    for (int i = 0; i < 4; ++i) mbar_init(bar0 + 8u * i, 1);
    fence_mbar_init();
    grid_dep_wait();
    load_kv(&mk, sK, full_k, c0);
    load_kv(&mv, sV, full_v, c0);
  }
  if (warp == 0) {
    __syncwarp();
    tmem_alloc(smem_u32(tmem_holder), L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_dep_launch();
  grid_dep_wait();
  const uint32_t tmem = __shfl_sync(0xffffffffu, *tmem_holder, 0);

  // ---- the query tile: rows r < group are query heads kvh * group + r, the rest zero ----
  {
    constexpr int kPieces = HD / 8;                              // 16-byte pieces per row
    constexpr int kAtomPieces = static_cast<int>(L::kAtomBytes / 16);
    const __nv_bfloat16 *qg = q + (static_cast<size_t>(b) * nh + static_cast<size_t>(kvh) * group) * HD;
    for (int e = t; e < 16 * kPieces; e += kDecThreads) {
      const int n = e / kPieces, pc = e % kPieces;
      uint4 val = make_uint4(0u, 0u, 0u, 0u);
      if (n < group) val = *reinterpret_cast<const uint4 *>(qg + n * HD + 8 * pc);
      const int col = pc / kAtomPieces, ch = pc % kAtomPieces;
      const int sw = L::kAtomBytes == 128 ? (ch ^ (n & 7)) : (ch ^ ((n >> 1) & 3));
      const uint32_t qoff = col * L::kQColBytes + n * L::kAtomBytes + (sw << 4);
      XATTN_DCHECK(qoff + 16 <= L::kQBytes, status);
      *reinterpret_cast<uint4 *>(smem + L::kQP + qoff) = val;
    }
    fence_proxy_async_smem();
  }
  __syncthreads();

  // The query tile stays in [kQP, kQP + kQBytes); P^T goes after it.
  constexpr uint32_t kPOff = (L::kQBytes + 1023) / 1024 * 1024;
  static_assert(L::kQP + kPOff + L::kPBytes <= L::kRed, "query tile and P^T both fit");
  const uint32_t sP = sQP + kPOff;
  constexpr uint32_t idesc_s = idesc_bf16_f32(128, 16, false, false);
  constexpr uint32_t idesc_pv = idesc_bf16_f32(128, L::kNpv, true, false);
  // thread t's O^T row: (tile j, element d)
  const int m = warp * 32 + lane, jrow = m / HD, drow = m % HD;
  float Mh[GV], Lh[GV], acc[GV];   // running max / sum per head (every thread), partial outputs
#pragma unroll
  for (int r = 0; r < GV; ++r) Mh[r] = -INFINITY, Lh[r] = 0.f, acc[r] = 0.f;

  bool ok = true;
  int last_s = -1, last_o = -1, k_loaded = c0 + 1, v_loaded = c0 + 1;   // chunks whose loads were issued
#pragma unroll 1
  for (int c = c0; c < c1; ++c) {
    const uint32_t par = static_cast<uint32_t>((c - c0) & 1);
    const int key0 = c * L::kChunk;
    // ---- scores S^T = K q^T, one M = 128, N = 16 product per tile ----
    if (warp == 0) {
      ok = ok && dec_warp_wait(full_k, par, ctl);
      if (ok) {
        tc_fence_after();
        const uint64_t dK = smem_desc(sK, 16, 8 * L::kAtomBytes, L::kSwizzle);
        const uint64_t dQ = smem_desc(sQP, 16, 8 * L::kAtomBytes, L::kSwizzle);
        if (elect_one()) {
#pragma unroll
          for (int j = 0; j < L::kSub; ++j)
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) {
              // a K step of 16 elements is +32 bytes within a swizzled row; the fifth step
              // starts the second 64-column atom (hd = 128)
              const uint32_t kstep = (kk % 4) * 2;
              mma_ss(tmem + 16u * j, dK + j * (L::kTileBytes >> 4) + (kk / 4) * (L::kSubBytes >> 4) + kstep,
                     dQ + (kk / 4) * (L::kQColBytes >> 4) + kstep, idesc_s, kk > 0 ? 1u : 0u);
            }
          mma_commit(s_done);
        }
        __syncwarp();
        last_s = c - c0;
      }
    }
    ok = ok && mbar_wait(s_done, par, ctl);
    // The scores are done with the K buffer: the next chunk's K tiles load meanwhile.
    if (t == 0 && ok && c + 1 < c1) {
      load_kv(&mk, sK, full_k, c + 1);
      k_loaded = c + 2;
    }

    // ---- chunk softmax: thread t owns key key0 + 128 j + t of tile j ----
    float x[L::kSub][GV];
    {
      uint32_t sr[16 * L::kSub];
      tc_fence_after();
      const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
      if constexpr (L::kSub == 1) {
        tmem_ld_x16(tl, sr);
      } else {
#pragma unroll
        for (int i = 0; i < 16 * L::kSub; i += 32) tmem_ld_x32(tl + i, sr + i);
      }
      tmem_wait_ld();
      reg_fence<16 * L::kSub>(sr);
#pragma unroll
      for (int j = 0; j < L::kSub; ++j)
#pragma unroll
        for (int r = 0; r < GV; ++r) x[j][r] = __uint_as_float(sr[16 * j + r]) * scale_log2;
    }
    bool valid[L::kSub];
#pragma unroll
    for (int j = 0; j < L::kSub; ++j) valid[j] = key0 + j * kTileRows + t < T;
#pragma unroll
    for (int r = 0; r < GV; ++r) {
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < L::kSub; ++j)
        if (valid[j]) mx = fmaxf(mx, x[j][r]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      if (lane == 0) red_max[warp * 16 + r] = mx;
    }
    __syncthreads();
    float mc[GV];   // the chunk's maximum per head
#pragma unroll
    for (int r = 0; r < GV; ++r) {
      // finite for r < group: every chunk holds at least one key below T
      mc[r] = fmaxf(fmaxf(red_max[r], red_max[16 + r]), fmaxf(red_max[32 + r], red_max[48 + r]));
      float l = 0.f;
#pragma unroll
      for (int j = 0; j < L::kSub; ++j) {
        const float p = (valid[j] && r < group) ? ex2_approx(x[j][r] - mc[r]) : 0.f;
        const __nv_bfloat16 pb = __float2bfloat16_rn(p);
        l += __bfloat162float(pb);
        // P^T row (j, r), key t: 64-key column t / 64, 16-byte chunk (t % 64) / 8 swizzled
        const int n = j * G + r;
        const uint32_t off = kPOff + (t >> 6) * L::kPColBytes + n * 128 + ((((t & 63) >> 3) ^ (n & 7)) << 4) +
                             (t & 7) * 2;
        XATTN_DCHECK(off + 2 <= kPOff + L::kPBytes, status);
        *reinterpret_cast<__nv_bfloat16 *>(smem + L::kQP + off) = pb;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
      if (lane == 0) red_sum[warp * 16 + r] = l;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- P V: O^T = [V tiles as M = 128 rows (j, d)] x [P^T, N = kSub x G] ----
    if (warp == 0 && ok) {
      ok = dec_warp_wait(full_v, par, ctl);
      if (ok) {
        tc_fence_after();
        // MN-major A: LBO = distance between 64-element atoms along M (the next tile, or
        // the second sub-tile at hd = 128), SBO = 8 key rows; a K step is 16 key rows.
        const uint64_t dV = smem_desc(sV, L::kSubBytes, 8 * L::kAtomBytes, L::kSwizzle);
        const uint64_t dP = smem_desc(sP, 16, 1024, kSwizzle128);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kTileRows / 16; ++kk)
            mma_ss(tmem + L::kTmemO, dV + kk * ((16 * L::kAtomBytes) >> 4),
                   dP + (kk / 4) * (L::kPColBytes >> 4) + (kk % 4) * 2, idesc_pv, kk > 0 ? 1u : 0u);
          mma_commit(o_done);
        }
        __syncwarp();
        last_o = c - c0;
      }
    }
    ok = ok && mbar_wait(o_done, par, ctl);
    // P V is done with the V buffer: the next chunk's V tiles load meanwhile.
    if (t == 0 && ok && c + 1 < c1) {
      load_kv(&mv, sV, full_v, c + 1);
      v_loaded = c + 2;
    }

    // ---- merge the chunk: rescale to the new running maximum and add ----
    {
      tc_fence_after();
      uint32_t orow[GV < 8 ? 8 : GV];
      const uint32_t ta = tmem + (static_cast<uint32_t>(warp * 32) << 16) + L::kTmemO + jrow * G;
      if constexpr (GV == 16) {
        tmem_ld_x16(ta, orow);
      } else {
        tmem_ld_x8(ta, orow);
      }
      tmem_wait_ld();
      reg_fence<(GV < 8 ? 8 : GV)>(orow);
#pragma unroll
      for (int r = 0; r < GV; ++r) {
        const float lc = (red_sum[r] + red_sum[16 + r]) + (red_sum[32 + r] + red_sum[48 + r]);
        const float mn = fmaxf(Mh[r], mc[r]);
        const float a_old = ex2_approx(Mh[r] - mn), a_new = ex2_approx(mc[r] - mn);   // 2^-inf = 0
        acc[r] = acc[r] * a_old + __uint_as_float(orow[r]) * a_new;
        Lh[r] = Lh[r] * a_old + lc * a_new;
        Mh[r] = mn;
      }
    }
    // Every thread has read red_max / red_sum and the O^T rows before the next chunk
    // overwrites them; on a failed wait anywhere all threads leave the loop together.
    tc_fence_before();
    if (__syncthreads_or(!ok)) {
      ok = false;
      break;
    }
  }

  // ---- the run's result: the tiles' partials summed through shared memory ----
  float *part = reinterpret_cast<float *>(smem + L::kK);   // [kSub][G][HD]; K is no longer read
  float *stat = red_max;                                   // [0, 16): M, [16, 32): L per head
  if (ok) {
    XATTN_DCHECK(((jrow + 1) * G) * HD <= L::kSub * G * HD && drow < HD, status);
#pragma unroll
    for (int r = 0; r < GV; ++r) part[(jrow * G + r) * HD + drow] = acc[r];
    if (t == 0) {
#pragma unroll
      for (int r = 0; r < GV; ++r) stat[r] = Mh[r], stat[16 + r] = Lh[r];
    }
  }
  __syncthreads();
  if (ok) {
    const size_t h0 = static_cast<size_t>(b) * nh + static_cast<size_t>(kvh) * group;
    const size_t rec0 = (static_cast<size_t>(bk) * nsplit + split) * group;   // records [B, nkv, nsplit, group]
    for (int e = t; e < group * HD; e += kDecThreads) {
      const int r = e / HD, d = e % HD;
      float a = 0.f;
#pragma unroll
      for (int j = 0; j < L::kSub; ++j) a += part[(j * G + r) * HD + d];
      if (nsplit == 1) {
        o[(h0 + r) * HD + d] = __float2bfloat16_rn(a / stat[16 + r]);
      } else {
        XATTN_DCHECK((rec0 + r + 1) * HD <= static_cast<size_t>(B) * nh * nsplit * HD, status);
        ws_o[(rec0 + r) * HD + d] = a;
      }
    }
    if (t < group) {
      if (nsplit == 1) {
        lse[h0 + t] = (stat[t] + __log2f(stat[16 + t])) * kLn2;
      } else {
        ws_ml[2 * (rec0 + t)] = stat[t];
        ws_ml[2 * (rec0 + t) + 1] = stat[16 + t];
      }
    }
  }

  // ---- teardown: let copies and products in flight land, then free TMEM ----
  if (t == 0) {
    mbar_drain(full_k, static_cast<uint32_t>((k_loaded - 1 - c0) & 1), ctl);
    mbar_drain(full_v, static_cast<uint32_t>((v_loaded - 1 - c0) & 1), ctl);
    if (last_s >= 0) mbar_drain(s_done, static_cast<uint32_t>(last_s & 1), ctl);
    if (last_o >= 0) mbar_drain(o_done, static_cast<uint32_t>(last_o & 1), ctl);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, L::kTmemCols);
}

// One warp per (batch, query head): merge the chunks, write O (bf16) and the LSE. The
// chunk weights 2^(m_c - M) are computed once, one chunk per lane, and passed along by
// shuffles; the loads of the partial outputs are independent across chunks.
template <int HD>
__global__ void __launch_bounds__(128) decode_combine_kernel(const float *__restrict__ ws_o,
                                                             const float *__restrict__ ws_ml,
                                                             __nv_bfloat16 *__restrict__ o,
                                                             float *__restrict__ lse, int B, int nh,
                                                             int nkv, int chunks) {
  constexpr int kPerLane = HD / 32;          // head-dim elements per lane (1, 2 or 4)
  grid_dep_launch();
  grid_dep_wait();
  const int warp = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (warp >= B * nh) return;
  const int b = warp / nh, h = warp % nh;
  const int group = nh / nkv, kvh = h / group, r = h % group;
  const size_t rec0 = (static_cast<size_t>(b) * nkv + kvh) * chunks * group + r;   // chunk 0
  float M = -INFINITY;
  for (int c = lane; c < chunks; c += 32) M = fmaxf(M, ws_ml[2 * (rec0 + static_cast<size_t>(c) * group)]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float L = 0.f, a[kPerLane];
#pragma unroll
  for (int e = 0; e < kPerLane; ++e) a[e] = 0.f;
  for (int c0 = 0; c0 < chunks; c0 += 32) {
    // lane i holds the weight of chunk c0 + i
    const int cl = c0 + lane;
    const size_t recl = rec0 + static_cast<size_t>(cl) * group;
    const float wl = cl < chunks ? ex2_approx(ws_ml[2 * recl] - M) : 0.f;
    L += cl < chunks ? ws_ml[2 * recl + 1] * wl : 0.f;
    const int n = min(32, chunks - c0);
#pragma unroll 8
    for (int i = 0; i < n; ++i) {
      const float w = __shfl_sync(0xffffffffu, wl, i);
      const float *src = ws_o + (rec0 + static_cast<size_t>(c0 + i) * group) * HD + lane * kPerLane;
#pragma unroll
      for (int e = 0; e < kPerLane; ++e) a[e] = fmaf(src[e], w, a[e]);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
  const float inv = 1.f / L;
  __nv_bfloat16 *orow = o + (static_cast<size_t>(b) * nh + h) * HD + lane * kPerLane;
#pragma unroll
  for (int e = 0; e < kPerLane; ++e) orow[e] = __float2bfloat16_rn(a[e] * inv);
  if (lane == 0) lse[static_cast<size_t>(b) * nh + h] = (M + __log2f(L)) * kLn2;
}

template <int HD, int G, int GV>
cudaError_t launch_decode_hd(const CUtensorMap &mk, const CUtensorMap &mv, const __nv_bfloat16 *q,
                             __nv_bfloat16 *o, float *lse, int B, int T, int nh, int nkv, float scale,
                             void *workspace, int *status, uint64_t timeout_ns, cudaStream_t stream) {
  using L = DecLayout<HD, G>;
  const int chunks = (T + L::kChunk - 1) / L::kChunk;
  int dev = 0, sms = 0;
  cudaError_t err;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
  const int nsplit = decode_nsplit(B * nkv, chunks, decode_ctas_per_sm<HD, G>() * sms, sms);
  float *ws_o = static_cast<float *>(workspace);
  float *ws_ml = ws_o + static_cast<size_t>(B) * nh * nsplit * HD;
  if ((err = cudaFuncSetAttribute(decode_partial_kernel<HD, G, GV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(L::kDynBytes))) != cudaSuccess)
    return err;
  const unsigned grid1 = static_cast<unsigned>(static_cast<long long>(B) * nkv * nsplit);
  err = launch_pdl(decode_partial_kernel<HD, G, GV>, dim3(grid1), kDecThreads, L::kDynBytes, stream, mk, mv, q,
                   ws_o, ws_ml, o, lse, B, T, nh, nkv, nsplit, scale * kLog2e, status,
                   static_cast<unsigned long long>(timeout_ns));
  if (err != cudaSuccess || nsplit == 1) return err;
  const unsigned blocks = static_cast<unsigned>((static_cast<long long>(B) * nh * 32 + 127) / 128);
  return launch_pdl(decode_combine_kernel<HD>, blocks, 128, 0, stream, static_cast<const float *>(ws_o),
                    static_cast<const float *>(ws_ml), o, lse, B, nh, nkv, nsplit);
}

template <int HD, int G>
int decode_runs_hd(int B, int T, int nkv, int sms) {
  using L = DecLayout<HD, G>;
  const int chunks = (T + L::kChunk - 1) / L::kChunk;
  return decode_nsplit(B * nkv, chunks, decode_ctas_per_sm<HD, G>() * sms, sms);
}

}  // namespace

int decode_runs(int B, int T, int nh, int nkv, int hd, int sms) {
  const int group = nh / nkv;
  if (hd == 32) return group <= 4 ? decode_runs_hd<32, 4>(B, T, nkv, sms)
                                  : (group <= 8 ? decode_runs_hd<32, 8>(B, T, nkv, sms) : decode_runs_hd<32, 16>(B, T, nkv, sms));
  if (hd == 64) return group <= 8 ? decode_runs_hd<64, 8>(B, T, nkv, sms) : decode_runs_hd<64, 16>(B, T, nkv, sms);
  return decode_runs_hd<128, 16>(B, T, nkv, sms);
}

cudaError_t launch_decode_bf16(const CUtensorMap &mk, const CUtensorMap &mv, const __nv_bfloat16 *q,
                               __nv_bfloat16 *o, float *lse, int B, int T, int nh, int nkv, int hd, float scale,
                               void *workspace, int *status, uint64_t timeout_ns, cudaStream_t stream) {
  const int group = nh / nkv;
  if (group > kMaxDecodeGroup) return cudaErrorInvalidValue;
  // G: the padded width of the query and P^T tiles (at least 16 / (128 / hd) so that P V
  // has N a multiple of 16); GV: the heads computed.
#define XATTN_DECODE(HD, G, GV) \
  return launch_decode_hd<HD, G, GV>(mk, mv, q, o, lse, B, T, nh, nkv, scale, workspace, status, timeout_ns, stream)
  if (hd == 32) {
    if (group <= 4) XATTN_DECODE(32, 4, 4);
    if (group <= 8) XATTN_DECODE(32, 8, 8);
    XATTN_DECODE(32, 16, 16);
  }
  if (hd == 64) {
    if (group <= 4) XATTN_DECODE(64, 8, 4);
    if (group <= 8) XATTN_DECODE(64, 8, 8);
    XATTN_DECODE(64, 16, 16);
  }
  if (hd == 128) {
    if (group <= 4) XATTN_DECODE(128, 16, 4);
    if (group <= 8) XATTN_DECODE(128, 16, 8);
    XATTN_DECODE(128, 16, 16);
  }
#undef XATTN_DECODE
  return cudaErrorInvalidValue;
}

}  // namespace xattn
