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
// GB300 mapping. The work is a matrix-vector product per (sequence, query head): two
// multiply-adds per cached K or V element and group, so it is bound by HBM reading the
// cache, not by arithmetic -- it runs on the CUDA cores, with every cached byte read once.
//   1. decode_partial_kernel: one CTA per (batch, kv head, 256-key chunk), 256 threads.
//      The chunk's K and V rows are copied once into shared memory (coalesced 16-byte
//      cp.async pieces, all in flight at once; V lands during the score pass) and serve
//      all `group` query heads of the kv head: one key per thread for the scores, a
//      chunk-local softmax (max and sum in fp32, log2 domain), then two head-dim elements
//      per thread over a contiguous run of keys for the unnormalised partial outputs.
//      Each chunk writes (max, sum, partial O) per query head to the scratch buffer.
//      The arithmetic, not HBM, is what the CTAs spend most issue slots on, so both
//      passes use the packed two-lane fp32 FMA (__ffma2_rn): the scores pair adjacent
//      head-dim elements, P V pairs adjacent keys (two partial sums per output, added at
//      the end); each lane is an ordinary fp32 fma.
//   2. decode_combine_kernel: one warp per (batch, query head) merges the chunks
//      (rescaling each by 2^(m_c - M)), writes O in bf16 and LSE = (M + log2 L) ln 2.
#include "sm103_ptx.cuh"
#include "xattn_internal.h"

namespace xattn {

size_t decode_workspace_bytes(int B, int T, int nh, int hd) {
  const size_t chunks = static_cast<size_t>((T + kDecodeChunk - 1) / kDecodeChunk);
  return static_cast<size_t>(B) * nh * chunks * (static_cast<size_t>(hd) + 2) * sizeof(float);
}

namespace {

constexpr int kDecodeThreads = kDecodeChunk;   // one key per thread in the score pass
constexpr int kDecodeWarps = kDecodeThreads / 32;

// Dynamic shared memory of decode_partial_kernel:
//   region A: first the chunk's K rows [kChunk][HD + 8] bf16 (padded by 16 bytes so that
//             one-row-per-thread reads spread over all banks); after the score pass, which
//             is their last reader, the exponentials p [group][kChunk] and the per
//             key-subset partial outputs acc [nks][group][HD] (nks = kDecodeThreads / (HD/2))
//   vs  [kChunk][HD + 8] bf16  the chunk's V rows (K and V are copied with cp.async at the
//                              start in two groups: the score pass waits for K only)
//   q   [group][HD] float      the query rows, pre-scaled by scale * log2(e)
//   red [kDecodeWarps][group]  warp partials of the max / sum
template <int HD>
__host__ __device__ constexpr int decode_row_elems() { return HD + 8; }

template <int HD>
__host__ __device__ constexpr size_t decode_region_a_bytes(int group) {
  const size_t k_rows = static_cast<size_t>(kDecodeChunk) * decode_row_elems<HD>() * 2;
  const size_t p_acc = sizeof(float) * static_cast<size_t>(group) * (kDecodeChunk + (kDecodeThreads / (HD / 2)) * HD);
  return k_rows > p_acc ? k_rows : p_acc;
}

template <int HD>
__host__ __device__ constexpr size_t decode_smem_bytes(int group) {
  return decode_region_a_bytes<HD>(group) + static_cast<size_t>(kDecodeChunk) * decode_row_elems<HD>() * 2 +
         sizeof(float) * static_cast<size_t>(group) * (HD + kDecodeWarps);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// MAXG: a compile-time bound on the group (4, 8 or 16), so the per-head register arrays
// are no larger than needed.
template <int HD, int MAXG>
__global__ void __launch_bounds__(kDecodeThreads) decode_partial_kernel(
    const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
    const __nv_bfloat16 *__restrict__ v, float *__restrict__ ws_o, float *__restrict__ ws_ml, int T,
    int nh, int nkv, float scale_log2) {
  constexpr int kPairs = HD / 2;                       // head-dim pairs
  constexpr int kSubsets = kDecodeThreads / kPairs;    // key subsets of the PV pass
  extern __shared__ __align__(16) uint8_t dsm_raw[];
  grid_dep_launch();
  grid_dep_wait();
  const int group = nh / nkv;
  const int chunk = blockIdx.y, chunks = gridDim.y;
  const int bk = blockIdx.x, b = bk / nkv, kvh = bk % nkv;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  constexpr int kRow = decode_row_elems<HD>();          // padded smem row, elements
  const size_t region_a = decode_region_a_bytes<HD>(group);
  __nv_bfloat16 *kt = reinterpret_cast<__nv_bfloat16 *>(dsm_raw);                   // [kChunk][kRow]
  float *ps = reinterpret_cast<float *>(dsm_raw);       // [group][kDecodeChunk], after the scores
  float *acc = ps + group * kDecodeChunk;               // [kSubsets][group][HD], after the scores
  __nv_bfloat16 *vs = reinterpret_cast<__nv_bfloat16 *>(dsm_raw + region_a);         // [kChunk][kRow]
  float *qs = reinterpret_cast<float *>(vs + kDecodeChunk * kRow);                  // [group][HD]
  float *red = qs + group * HD;                         // [kDecodeWarps][group]

  const int j = chunk * kDecodeChunk + t;
  const bool valid = j < T;
  const size_t row_stride = static_cast<size_t>(nkv) * HD;           // elements between keys
  const size_t kv_base = (static_cast<size_t>(b) * T * nkv + kvh) * HD;
  // The chunk's K rows, then its V rows, stream into shared memory: consecutive threads
  // copy consecutive 16-byte pieces of a row, so every request is a whole row segment.
  // Rows past T are not copied and never read. V lands while the scores are computed.
  const int n_valid = min(kDecodeChunk, T - chunk * kDecodeChunk);
  constexpr int kPieces = HD / 8;                       // 16-byte pieces per row
  {
    const __nv_bfloat16 *kc = k + kv_base + static_cast<size_t>(chunk) * kDecodeChunk * row_stride;
    const __nv_bfloat16 *vc = v + kv_base + static_cast<size_t>(chunk) * kDecodeChunk * row_stride;
    for (int e = t; e < n_valid * kPieces; e += kDecodeThreads) {
      const int row = e / kPieces, pc = e % kPieces;
      cp_async16(smem_u32(kt + row * kRow + 8 * pc), kc + static_cast<size_t>(row) * row_stride + 8 * pc);
    }
    cp_async_commit();
    for (int e = t; e < n_valid * kPieces; e += kDecodeThreads) {
      const int row = e / kPieces, pc = e % kPieces;
      cp_async16(smem_u32(vs + row * kRow + 8 * pc), vc + static_cast<size_t>(row) * row_stride + 8 * pc);
    }
    cp_async_commit();
  }

  // Query rows of the group's heads (kvh * group + r), scaled into the log2 domain.
  const __nv_bfloat16 *qg = q + (static_cast<size_t>(b) * nh + static_cast<size_t>(kvh) * group) * HD;
  for (int e = t; e < group * HD; e += kDecodeThreads) qs[e] = __bfloat162float(qg[e]) * scale_log2;
  cp_async_wait<1>();                                   // this thread's K pieces have landed
  __syncthreads();                                      // ... and every thread's

  // ---- scores: thread t takes key j = chunk * kDecodeChunk + t, all heads of the group ----
  float s[MAXG];
  {
    float2 s2[MAXG];
#pragma unroll
    for (int r = 0; r < MAXG; ++r) s2[r] = make_float2(0.f, 0.f);
    if (valid) {
      const uint4 *krow = reinterpret_cast<const uint4 *>(kt + t * kRow);
#pragma unroll
      for (int c = 0; c < HD / 8; ++c) {
        const uint4 kv8 = krow[c];
        const float2 k01 = make_float2(bf16lo_to_f32(kv8.x), bf16hi_to_f32(kv8.x));
        const float2 k23 = make_float2(bf16lo_to_f32(kv8.y), bf16hi_to_f32(kv8.y));
        const float2 k45 = make_float2(bf16lo_to_f32(kv8.z), bf16hi_to_f32(kv8.z));
        const float2 k67 = make_float2(bf16lo_to_f32(kv8.w), bf16hi_to_f32(kv8.w));
#pragma unroll
        for (int r = 0; r < MAXG; ++r) {
          if (r < group) {
            const float4 qa = *reinterpret_cast<const float4 *>(qs + r * HD + 8 * c);
            const float4 qb = *reinterpret_cast<const float4 *>(qs + r * HD + 8 * c + 4);
            s2[r] = __ffma2_rn(make_float2(qa.x, qa.y), k01, s2[r]);
            s2[r] = __ffma2_rn(make_float2(qa.z, qa.w), k23, s2[r]);
            s2[r] = __ffma2_rn(make_float2(qb.x, qb.y), k45, s2[r]);
            s2[r] = __ffma2_rn(make_float2(qb.z, qb.w), k67, s2[r]);
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < MAXG; ++r) s[r] = s2[r].x + s2[r].y;
  }

  // ---- chunk softmax per head: max, exponentials, sum (log2 domain) ----
  float mx[MAXG] = {};
#pragma unroll
  for (int r = 0; r < MAXG; ++r) {
    if (r < group) {
      float m = valid ? s[r] : -INFINITY;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      if (lane == 0) red[warp * group + r] = m;
    }
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < MAXG; ++r) {
    if (r < group) {
      float m = red[r];
#pragma unroll
      for (int w = 1; w < kDecodeWarps; ++w) m = fmaxf(m, red[w * group + r]);
      mx[r] = m;                                       // finite: the chunk has a valid key
    }
  }
  __syncthreads();                                     // red is reused for the sums
#pragma unroll
  for (int r = 0; r < MAXG; ++r) {
    if (r < group) {
      const float p = valid ? ex2_approx(s[r] - mx[r]) : 0.f;
      ps[r * kDecodeChunk + t] = p;
      float l = p;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
      if (lane == 0) red[warp * group + r] = l;
    }
  }
  __syncthreads();

  // ---- P V: thread (subset ks, pair dp) sums the keys [ks * kPer, (ks + 1) * kPer) of
  // the chunk for head-dim elements 2 dp and 2 dp + 1; the exponentials of four keys
  // come in one 16-byte broadcast read ----
  const int dp = t % kPairs, ks = t / kPairs;
  float o0[MAXG], o1[MAXG];
#pragma unroll
  for (int r = 0; r < MAXG; ++r) o0[r] = o1[r] = 0.f;
  cp_async_wait<0>();
  __syncthreads();                                     // every thread's V pieces have landed
  const uint32_t *vcol = reinterpret_cast<const uint32_t *>(vs) + dp;
  constexpr int kPer = kDecodeChunk / kSubsets;        // contiguous keys per subset
  const int k0 = ks * kPer;
  const int kn = max(0, min(kPer, n_valid - k0));
  const float *pk = ps + k0;
  int jj = 0;
  {
    float2 ae[MAXG], ao[MAXG];                         // even / odd head-dim element, key pairs
#pragma unroll
    for (int r = 0; r < MAXG; ++r) ae[r] = ao[r] = make_float2(0.f, 0.f);
#pragma unroll(MAXG > 8 ? 1 : 2)
    for (; jj + 4 <= kn; jj += 4) {
      uint32_t vv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) vv[u] = vcol[(k0 + jj + u) * (kRow / 2)];
      const float2 e01 = make_float2(bf16lo_to_f32(vv[0]), bf16lo_to_f32(vv[1]));
      const float2 e23 = make_float2(bf16lo_to_f32(vv[2]), bf16lo_to_f32(vv[3]));
      const float2 o01 = make_float2(bf16hi_to_f32(vv[0]), bf16hi_to_f32(vv[1]));
      const float2 o23 = make_float2(bf16hi_to_f32(vv[2]), bf16hi_to_f32(vv[3]));
#pragma unroll
      for (int r = 0; r < MAXG; ++r) {
        if (r < group) {
          const float4 p4 = *reinterpret_cast<const float4 *>(pk + r * kDecodeChunk + jj);
          const float2 p01 = make_float2(p4.x, p4.y), p23 = make_float2(p4.z, p4.w);
          ae[r] = __ffma2_rn(p01, e01, ae[r]);
          ae[r] = __ffma2_rn(p23, e23, ae[r]);
          ao[r] = __ffma2_rn(p01, o01, ao[r]);
          ao[r] = __ffma2_rn(p23, o23, ao[r]);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < MAXG; ++r) {
      o0[r] = ae[r].x + ae[r].y;
      o1[r] = ao[r].x + ao[r].y;
    }
  }
  for (; jj < kn; ++jj) {
    const uint32_t vv = vcol[(k0 + jj) * (kRow / 2)];
    const float v0 = bf16lo_to_f32(vv), v1 = bf16hi_to_f32(vv);
#pragma unroll
    for (int r = 0; r < MAXG; ++r) {
      if (r < group) {
        const float p = pk[r * kDecodeChunk + jj];
        o0[r] = fmaf(p, v0, o0[r]);
        o1[r] = fmaf(p, v1, o1[r]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < MAXG; ++r) {
    if (r < group) {
      acc[(ks * group + r) * HD + 2 * dp] = o0[r];
      acc[(ks * group + r) * HD + 2 * dp + 1] = o1[r];
    }
  }
  __syncthreads();

  // ---- chunk result: (max, sum, partial O) per head of the group ----
  const size_t rec = (static_cast<size_t>(bk) * chunks + chunk) * group;   // [B, nkv, chunks, group]
  for (int e = t; e < group * HD; e += kDecodeThreads) {
    const int r = e / HD, d = e % HD;
    float a = 0.f;
#pragma unroll 4
    for (int q4 = 0; q4 < kSubsets; ++q4) a += acc[(q4 * group + r) * HD + d];
    ws_o[(rec + r) * HD + d] = a;
  }
  if (t < group) {
    float l = 0.f;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) l += red[w * group + t];
    // mx[] lives in registers (compile-time indexed): pick this thread's head.
    float m = 0.f;
#pragma unroll
    for (int r = 0; r < MAXG; ++r)
      if (r == t) m = mx[r];
    ws_ml[2 * (rec + t)] = m;
    ws_ml[2 * (rec + t) + 1] = l;
  }
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

template <int HD, int MAXG>
cudaError_t launch_decode_hd(const __nv_bfloat16 *q, const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                             __nv_bfloat16 *o, float *lse, int B, int T, int nh, int nkv, float scale,
                             void *workspace, cudaStream_t stream) {
  const int group = nh / nkv;
  const int chunks = (T + kDecodeChunk - 1) / kDecodeChunk;
  float *ws_o = static_cast<float *>(workspace);
  float *ws_ml = ws_o + static_cast<size_t>(B) * nh * chunks * HD;
  const size_t smem = decode_smem_bytes<HD>(group);
  cudaError_t err = cudaFuncSetAttribute(decode_partial_kernel<HD, MAXG>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  const dim3 grid1(static_cast<unsigned>(B * nkv), static_cast<unsigned>(chunks));
  err = launch_pdl(decode_partial_kernel<HD, MAXG>, grid1, kDecodeThreads, smem, stream, q, k, v, ws_o, ws_ml, T,
                   nh, nkv, scale * kLog2e);
  if (err != cudaSuccess) return err;
  const unsigned blocks = static_cast<unsigned>((static_cast<long long>(B) * nh * 32 + 127) / 128);
  return launch_pdl(decode_combine_kernel<HD>, blocks, 128, 0, stream, static_cast<const float *>(ws_o),
                    static_cast<const float *>(ws_ml), o, lse, B, nh, nkv, chunks);
}

}  // namespace

cudaError_t launch_decode_bf16(const __nv_bfloat16 *q, const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                               __nv_bfloat16 *o, float *lse, int B, int T, int nh, int nkv, int hd,
                               float scale, void *workspace, cudaStream_t stream) {
  const int group = nh / nkv;
  if (group > kMaxDecodeGroup) return cudaErrorInvalidValue;
#define XATTN_DECODE_G(HD)                                                                              \
  if (group <= 4) return launch_decode_hd<HD, 4>(q, k, v, o, lse, B, T, nh, nkv, scale, workspace, stream); \
  if (group <= 8) return launch_decode_hd<HD, 8>(q, k, v, o, lse, B, T, nh, nkv, scale, workspace, stream); \
  return launch_decode_hd<HD, 16>(q, k, v, o, lse, B, T, nh, nkv, scale, workspace, stream)
  if (hd == 64) { XATTN_DECODE_G(64); }
  if (hd == 32) { XATTN_DECODE_G(32); }
  if (hd == 128) { XATTN_DECODE_G(128); }
#undef XATTN_DECODE_G
  return cudaErrorInvalidValue;
}

}  // namespace xattn
