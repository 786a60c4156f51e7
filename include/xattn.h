/*
 * libxattn: fused causal scaled-dot-product attention with grouped KV heads (GQA),
 * forward and backward, for NVIDIA GB300 (sm_103a).
 *
 * The operation (xtrain "演进总览" / docs/evolution.md, phase table):
 *   - row T14: one fused attention op. The forward runs an online softmax tiled over
 *     KV and never materialises the S x S scores; it keeps each row's log-sum-exp.
 *     The backward recomputes the scores and replaces the softmax Jacobian by
 *     D_i = sum_d dO_id O_id, giving dQ, dK and dV.
 *   - row T15: grouped KV heads. Query head h reads kv head h / (nh / nkv); the
 *     gradient of a kv head is the deterministic sum over its query group.
 *   - causal masking as in the composed path of xtrain "Known Issues & Perf Backlog"
 *     (docs/known-issues.md), KI-1 fix: query i sees keys j <= i (diagonal included);
 *     queries and keys have the same length S.
 *
 * Definition (natural log; scale multiplies the scores before the softmax):
 *   s_ij = scale * q_i . k_j (j <= i),  LSE_i = log sum_{j<=i} exp(s_ij),
 *   P_ij = exp(s_ij - LSE_i),  O_i = sum_j P_ij v_j,
 *   dS_ij = P_ij (dO_i . v_j - dO_i . O_i),
 *   dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_{group} sum_i dS_ij q_i,
 *   dV_j = sum_{group} sum_i P_ij dO_i.
 *
 * Layout: every tensor is contiguous and row-major.
 *   q, o, dO, dq : [B, S, nh,  hd]
 *   k, v, dk, dv : [B, S, nkv, hd]
 *   lse          : [B, S, nh] float (natural log of the scaled scores' sum of exps)
 *
 * Conventions shared by every entry point:
 *   - Pointers are DEVICE pointers owned by the caller, unless a comment says
 *     otherwise. Inputs are read only. Outputs are overwritten, never accumulated into.
 *   - stream is a cudaStream_t (NULL = the legacy default stream) of the current
 *     device. Calls enqueue work and return; none synchronises the device (xtrain
 *     docs/06-performance.md, "Phase T7", design decision 3: no per-op synchronisation).
 *   - Argument checks run before any launch. On a check failure nothing is enqueued
 *     and the outputs are untouched. Launch failures return XATTN_ERR_CUDA.
 *   - A kernel that waits on an on-chip barrier longer than a bounded time (about
 *     two seconds) gives up, records XATTN_ERR_DEVICE_TIMEOUT in a device status word
 *     and finishes; xattn_check_device_status reports it.
 *   - CUDA graphs: the calls may be captured on a stream and replayed, once the device
 *     has seen one ordinary call (the first call on a device looks up its device
 *     status word; make that call outside the capture). Entry points that take
 *     scratch with cudaMallocAsync record it in the graph as stream-ordered
 *     allocation nodes.
 */
#ifndef XATTN_H
#define XATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    XATTN_OK = 0,
    XATTN_ERR_NULL_PTR = 1,           /* a required pointer is NULL */
    XATTN_ERR_BAD_SHAPE = 2,          /* B, S, nh, nkv or hd <= 0, or a size overflows int32 */
    XATTN_ERR_GROUP = 3,              /* nh is not a multiple of nkv */
    XATTN_ERR_UNSUPPORTED_HD = 4,     /* bf16: hd not in {32, 64, 128} (the backward's
                                         stage calls and xattn_bwd_noalloc: {32, 64});
                                         fp32: hd > 128 */
    XATTN_ERR_MISALIGNED = 5,         /* a bf16 tensor pointer is not 16-byte aligned */
    XATTN_ERR_CUDA = 6,               /* a CUDA runtime or driver call failed */
    XATTN_ERR_NO_DEVICE_SUPPORT = 7,  /* the current device is not compute capability 10.3 */
    XATTN_ERR_DEVICE_TIMEOUT = 8,     /* a bounded on-device wait expired (reported later) */
    XATTN_ERR_BAD_SCALE = 9,          /* scale is not finite (bf16 backward: or
                                         0 < |scale| < 2^-64) */
    XATTN_ERR_WORKSPACE = 10,         /* workspace pointer NULL/misaligned or too small */
    XATTN_ERR_SCRATCH_LIMIT = 11,     /* xattn_bwd_noalloc: sizes need more than its fixed scratch */
    XATTN_ERR_DEVICE_BOUNDS = 12      /* debug builds only: an on-device bounds check failed
                                         (reported later, like a timeout) */
} xattn_status;

/*
 * Forward, bf16 (xtrain docs/evolution.md, row T14: online softmax tiled over KV,
 * per-row log-sum-exp kept). q, k, v, o are bf16; lse is float.
 * hd in {32, 64, 128}; any S >= 1. Arithmetic: bf16 products, fp32 accumulation and
 * softmax statistics (row T12: softmax kept in fp32 under bf16); P is rounded to bf16
 * before the P.V product; o is rounded to nearest even.
 */
xattn_status xattn_fwd(const void *q, const void *k, const void *v, int B, int S, int nh,
                       int nkv, int hd, float scale, void *o, float *lse, void *stream);

/*
 * Backward, bf16 (row T14: recompute the scores, D = rowsum(dO * O); row T15: dK/dV
 * summed over each kv head's query group without atomics). Takes the forward's o and
 * lse. Writes dq [B,S,nh,hd], dk and dv [B,S,nkv,hd] in bf16. scale == 0 is taken
 * exactly; a nonzero |scale| below 2^-64 is rejected (XATTN_ERR_BAD_SCALE), because the
 * recompute adds -LSE/scale to the scores inside a tensor-core product.
 * Scratch (xattn_bwd_workspace_bytes) is taken with cudaMallocAsync on `stream` and
 * released with cudaFreeAsync on the same stream; nothing else is allocated.
 * dQ is accumulated across key tiles with fp32 reduce-adds whose order is not fixed,
 * so its last bits may vary from run to run; dK, dV, o and lse are bit-for-bit
 * reproducible. xattn_bwd_deterministic gives a dQ that is reproducible too.
 * hd in {32, 64, 128}. At hd = 128 dV, dK and a dQ accumulator do not fit in the
 * tensor memory together, so xattn_bwd runs xattn_bwd_deterministic (every output
 * reproducible; scratch as described there).
 */
xattn_status xattn_bwd(const void *q, const void *k, const void *v, const void *o,
                       const void *dO, const float *lse, int B, int S, int nh, int nkv,
                       int hd, float scale, void *dq, void *dk, void *dv, void *stream);

/*
 * Which backward xattn_bwd (deterministic == 0) or xattn_bwd_deterministic
 * (deterministic != 0) runs for these sizes; no device work, -1 for sizes they reject:
 *   XATTN_BWD_FUSED_DQ      xattn_bwd at hd 32 / 64: dK/dV key-stationary; dQ added across
 *                           key tiles into an fp32 accumulator with reduce-adds, then
 *                           converted (the three stage calls below); dQ's last bits may vary
 *                           from run to run.
 *   XATTN_BWD_RESIDENT_DQ   xattn_bwd_deterministic on small problems (group * ceil(S / 128)
 *                           * hd <= 64, hd 32 or 64): one CTA per (batch, kv head) takes all
 *                           its key tiles and keeps the head's dQ tiles in tensor memory,
 *                           summed in a fixed order and written once (one kernel after the
 *                           preprocess).
 *   XATTN_BWD_QUERY_DQ      otherwise deterministic (and xattn_bwd at hd 128): dQ from a
 *                           query-stationary recompute.
 * The last two give every output bit-for-bit the same from run to run.
 */
#define XATTN_BWD_FUSED_DQ 0
#define XATTN_BWD_RESIDENT_DQ 1
#define XATTN_BWD_QUERY_DQ 2
int xattn_bwd_dq_mode(int S, int nh, int nkv, int hd, int deterministic);

/*
 * The backward's three steps with a caller-owned workspace, for callers that manage
 * memory themselves (or capture the call in a CUDA graph). xattn_bwd is exactly
 * workspace allocation + these three calls + release.
 *
 * hd in {32, 64} only (hd = 128 has no fused dQ step; use xattn_bwd).
 * workspace: device pointer, 256-byte aligned, at least xattn_bwd_workspace_bytes()
 * bytes. Its contents on entry do not matter; the three steps must run in this order
 * on one stream with the same arguments.
 *   xattn_bwd_preprocess : D_i = dO_i . O_i (fp32); per query row, -LSE_i/scale and
 *                          -D_i as bf16 operand rows of the recompute (each the sum
 *                          of three bf16 terms); a zeroed fp32 dQ accumulator (all
 *                          inside the workspace).
 *   xattn_bwd_main       : the recompute loop; writes dk, dv and adds dS K into the
 *                          dQ accumulator (without the softmax scale).
 *   xattn_bwd_dq_convert : dq = bf16(scale * dQ accumulator); scale is the one given
 *                          to xattn_bwd_main.
 */
size_t xattn_bwd_workspace_bytes(int B, int S, int nh, int hd);
xattn_status xattn_bwd_preprocess(const void *o, const void *dO, const float *lse, int B,
                                  int S, int nh, int hd, float scale, void *workspace,
                                  size_t workspace_bytes, void *stream);
xattn_status xattn_bwd_main(const void *q, const void *k, const void *v, const void *dO,
                            int B, int S, int nh, int nkv, int hd, float scale, void *dk,
                            void *dv, void *workspace, size_t workspace_bytes, void *stream);
xattn_status xattn_bwd_dq_convert(int B, int S, int nh, int hd, float scale, void *dq,
                                  void *workspace, size_t workspace_bytes, void *stream);

/*
 * Backward with a reproducible dQ: the same arguments, results and scale rule as
 * xattn_bwd, but every output is bit-for-bit the same from run to run. dK and dV come
 * from the same key-stationary recompute as in xattn_bwd (without dQ there); dQ comes
 * from a query-stationary recompute that accumulates dQ_i = scale sum_j dS_ij k_j over
 * the key tiles of its query tile in a fixed order, with no atomics (row T14's
 * recompute, done a second time: 7 tensor-core products per tile pair instead of 5).
 * Scratch (D and the recompute's operand rows) is taken with cudaMallocAsync on
 * `stream` and released with cudaFreeAsync on the same stream.
 */
xattn_status xattn_bwd_deterministic(const void *q, const void *k, const void *v,
                                     const void *o, const void *dO, const float *lse, int B,
                                     int S, int nh, int nkv, int hd, float scale, void *dq,
                                     void *dk, void *dv, void *stream);

/*
 * xattn_bwd with no allocation at all. The pages have no counterpart: this entry point
 * exists for callers that may not allocate device memory, such as a loop running under
 * a no-allocation rule once started (cudaFree synchronises the whole device), or a host
 * whose device memory is already fully reserved by its own allocator, so the
 * cudaMallocAsync inside xattn_bwd would fail.
 *
 * Same arguments and results as xattn_bwd, for hd in {32, 64}. The scratch (xattn_bwd_workspace_bytes(B, S,
 * nh, hd) bytes) lives in one fixed device array of XATTN_NOALLOC_SCRATCH_BYTES inside
 * the library. Sizes that need more return XATTN_ERR_SCRATCH_LIMIT before anything is
 * launched (64 MiB fits, e.g., B=8, S=2048, nh=8, hd=64).
 * CUDA loads the library's device code lazily: the first call on a device places the
 * 64 MiB array on that device (looking up its address with cudaGetSymbolAddress), and
 * the device holds it until the process exits. Make that first call before the host's
 * own allocator reserves the device's memory, and before any stream capture on the
 * device. If it fails (XATTN_ERR_CUDA, e.g. no 64 MiB left), the next call tries again.
 * `stream` must belong to the current device (else XATTN_ERR_CUDA, nothing launched).
 * All calls share the one array and each call overwrites all of the scratch it uses, so
 * nothing carries over between calls, but calls whose work overlaps on the GPU (on
 * different streams, or from different threads) race on it and must be serialised by
 * the caller.
 */
#define XATTN_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
xattn_status xattn_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                               const void *dO, const float *lse, int B, int S, int nh, int nkv,
                               int hd, float scale, void *dq, void *dk, void *dv, void *stream);

/*
 * fp32 mode: same parameters and layouts, float tensors, IEEE fp32 arithmetic on the
 * CUDA cores (no TF32). hd in [1, 128]; any S >= 1. No scratch memory.
 */
xattn_status xattn_fwd_f32(const float *q, const float *k, const float *v, int B, int S,
                           int nh, int nkv, int hd, float scale, float *o, float *lse,
                           void *stream);
xattn_status xattn_bwd_f32(const float *q, const float *k, const float *v, const float *o,
                           const float *dO, const float *lse, int B, int S, int nh, int nkv,
                           int hd, float scale, float *dq, float *dk, float *dv,
                           void *stream);

/* Static text for a status code (never NULL). */
/*
 * Decode attention, bf16 (xtrain docs/evolution.md, post-training milestones M2a-M2c):
 * one new query per sequence against that sequence's cached keys and values -- equal to
 * the last row of full causal attention over the T cached positions, which include the
 * query's own (so every cached key is visible; there is no mask). Batch-agnostic: the B
 * sequences are independent and share T.
 *   q      [B, nh, hd]      bf16, the new token's query heads
 *   k, v   [B, T, nkv, hd]  bf16, the caches, row-major like the [B, S, heads, hd]
 *                           tensors of xattn_fwd (position T-1 is the new token)
 *   o      [B, nh, hd]      bf16 out;  lse [B, nh] float out (natural log of the sum of
 *                           exp of the scaled scores, as xattn_fwd's lse)
 * Query head h reads kv head h / (nh / nkv). hd in {32, 64, 128}; nh / nkv <= 16
 * (else XATTN_ERR_GROUP); T >= 1 with B * nkv * ceil(T / C) < 2^31, C = 16384 / hd
 * keys per chunk (else XATTN_ERR_BAD_SHAPE); any finite scale. q, k, v, o 16-byte
 * aligned, lse 4-byte aligned.
 * Arithmetic: tensor-core products on the bf16 inputs with fp32 accumulation (the
 * scores q . k, and the sum over keys of p v with the probabilities p rounded to bf16,
 * as in xattn_fwd); softmax statistics in fp32, merged across chunks online; o rounded
 * to nearest even. Scratch (B * nh * ceil(T / C) * (hd + 2) floats, an upper bound on the
 * per-run records that xattn_decode_runs describes) is taken with cudaMallocAsync on
 * `stream` and released with cudaFreeAsync; nothing else is allocated. The result is
 * bit-for-bit reproducible (fixed reduction order for given sizes and SM count).
 */
xattn_status xattn_decode(const void *q, const void *k_cache, const void *v_cache, int B, int T,
                          int nh, int nkv, int hd, float scale, void *o, float *lse, void *stream);

/*
 * How xattn_decode splits the caches on a GPU with num_sms SMs; no device work, -1 for
 * sizes xattn_decode rejects (or num_sms <= 0). The result R is the number of key runs per
 * (sequence, kv head): each run is one CTA that streams its C-key chunks through shared
 * memory and merges them online.
 *   R == 1  one kernel: a CTA per (sequence, kv head) writes o and lse itself; chosen when
 *           the B * nkv pairs fill the SMs in one wave of resident CTAs;
 *   R > 1   each run writes (maximum, sum, unnormalised output) per query head to the
 *           scratch and a second kernel merges the runs; chosen when B * nkv is below the
 *           SM count (more CTAs for the GPU), and for batches beyond one wave where a split
 *           shortens the waves of CTAs.
 * The split depends only on these sizes and num_sms, so results are reproducible on one
 * GPU model.
 */
int xattn_decode_runs(int B, int T, int nh, int nkv, int hd, int num_sms);

const char *xattn_status_string(xattn_status status);

/*
 * Synchronises `stream`, then reads and clears the current device's status word.
 * Returns XATTN_ERR_DEVICE_TIMEOUT if a kernel gave up on a bounded wait since the
 * last check (XATTN_ERR_DEVICE_BOUNDS if, in a debug build, a bounds check failed first),
 * XATTN_ERR_CUDA if the synchronisation failed, else XATTN_OK.
 */
xattn_status xattn_check_device_status(void *stream);

/*
 * Self-test of failure detection (no counterpart on the pages, which have none for
 * attention). Every wait of this library's kernels is bounded: past the limit the kernel
 * records XATTN_ERR_DEVICE_TIMEOUT in a device status word, stops and frees what it
 * holds, and the context stays usable. This call launches one small kernel whose only
 * work is such a wait on a barrier that nothing completes, with the given limit (1 us to
 * 10 s, else XATTN_ERR_BAD_SHAPE), so a test can see the timeout reported by
 * xattn_check_device_status without any kernel of the attention path failing.
 * Asynchronous on `stream`; returns XATTN_OK once launched.
 */
xattn_status xattn_selftest_wait_timeout(unsigned long long limit_ns, void *stream);

/*
 * Debug build (the library compiled with XATTN_DEBUG; bwd_xattn_fwd_gb300/build.py
 * builds it with `--debug` into its own directory). The tensor-core kernels then check,
 * before each use, the indices they compute -- TMA tile coordinates against the tensor's
 * extents and the 16-byte rule for the innermost coordinate, shared-memory offsets
 * against their tile, tensor-memory columns against their region, and global row offsets
 * of direct stores against the tensor -- and record XATTN_ERR_DEVICE_BOUNDS in the device
 * status word when one fails (no trap; xattn_check_device_status reports it). It stands in
 * for a memory checker; release builds compile the checks out.
 *
 * xattn_build_flags: bit 0 set in a debug build. No device work.
 * xattn_selftest_bounds_check: launches one small kernel whose only work is a bounds check
 * that fails (an index one past the end of a 1-element range, never used for an access),
 * so a test can see XATTN_ERR_DEVICE_BOUNDS reported in a debug build (and nothing in a
 * release build). Asynchronous on `stream`; returns XATTN_OK once launched.
 */
#define XATTN_BUILD_DEVICE_CHECKS 1
int xattn_build_flags(void);
xattn_status xattn_selftest_bounds_check(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* XATTN_H */
