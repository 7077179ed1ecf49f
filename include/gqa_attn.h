/*
 * gqa_attn.h -- C ABI of the GB300 (sm_103a) grouped-query FlashAttention
 * library: forward (O, LSE) and the backward hot path (Delta, dQ, dK, dV, dsink).
 *
 * Sources of the operations (web pages, by title and section):
 *  [P1] tilelang PR #1093 "[GQA] Add regional atomic add to slightly boost
 *       performance" -- Additional comments: dQ slice atomics per KV-block
 *       iteration; dK/dV accumulated locally and added once into kv head
 *       "bx // groups"; Related PRs: TMA-based atomic reduce, varlen GQA bwd.
 *  [P2] tilelang-ascend PR #1638 "[Feat] Add GQA Sink Backward BHSD with
 *       robustness improvements" -- review thread (k1..k5 formulas), "Kernel 9:
 *       Dsink", the 9->6 kernel commit (preprocess + dsink, dual-output
 *       postprocess cast), the 4->2 kernel commit (Phase0 Delta, fp32
 *       atomic_add then cast), Description (BHSD layout, sink + window forward).
 *  [P3] triton issue #4717 "atomic_add slows down attention backwards due to
 *       layout conversions" -- vectorised atomics vs. scalar atomic_add in the
 *       causal fused-attention backward.
 *
 * Conventions shared by every entry point
 *  - Shapes: q, dq [B,Hq,S,Dqk]; k, dk [B,Hkv,S,Dqk]; v, dv [B,Hkv,S,Dv];
 *    o, dout [B,Hq,S,Dv]; lse, delta [B,Hq,S] fp32; sink, dsink [Hq] fp32.  By
 *    default every tensor is dense row-major BHSD ([P2] Description); the 16-bit
 *    ones may instead carry (batch, head, sequence) strides (gqa_stride: BSHD,
 *    packed THD, ...).  Packed variable-length batches use B == 1, S == total
 *    tokens T and cu_seqlens ([P1] Related PRs).
 *  - Element type of q/k/v/o/dout/dq/dk/dv: fp16 or bf16 (params.dtype).
 *    Every accumulation is fp32 ([P2] 4->2 commit: fp16 atomics fail precision).
 *  - Pointers: device pointers unless stated; base addresses of the 16-bit
 *    tensors must be 16-byte aligned.  The caller owns and allocates every
 *    buffer, including the workspace; the library never allocates or frees
 *    device memory.
 *  - Execution: every call is asynchronous on `stream` (a cudaStream_t passed
 *    as void*; NULL = legacy default stream) and never synchronises the host,
 *    except gqa_attn_get_device_error.
 *  - Errors: arguments are validated before anything is launched; an invalid
 *    or unsupported problem returns a negative status and launches nothing.
 *    A failed launch returns GQA_ERR_CUDA.  Device-side problems (a bounded
 *    wait that timed out, a packed sequence longer than max_seqlen) are
 *    recorded in the workspace and reported by gqa_attn_get_device_error.
 */
#ifndef GQA_ATTN_H_
#define GQA_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GQA_OK = 0,
  GQA_ERR_INVALID_ARG = -1,   /* null/misaligned pointer, bad shape, inconsistent flags */
  GQA_ERR_UNSUPPORTED = -2,   /* valid problem outside the supported head dims / dtypes */
  GQA_ERR_WORKSPACE = -3,     /* workspace missing, too small or not 256-byte aligned */
  GQA_ERR_CUDA = -4,          /* a CUDA runtime call or launch failed */
  GQA_ERR_DEVICE_TIMEOUT = -5,/* a kernel's bounded wait gave up (reported after the fact) */
  GQA_ERR_DEVICE_INPUT = -6   /* device-side input check failed, e.g. a sequence > max_seqlen */
} gqa_status;

typedef enum { GQA_F16 = 0, GQA_BF16 = 1 } gqa_dtype;

/* How the per-query-head dK/dV contributions of one kv head are summed ([P1]). */
typedef enum {
  GQA_GROUP_TMEM = 0,   /* one CTA per (kv head, KV tile) loops over all Hq/Hkv query heads;
                           dK/dV stay in tensor memory and are written once, no atomics */
  GQA_GROUP_ATOMIC = 1  /* one CTA per (query head, KV tile); after its Q loop it adds its
                           dK/dV into fp32 accumulators in the workspace with atomics
                           (Hq/Hkv-way contention); gqa_attn_bwd_postprocess casts them */
} gqa_group_mode;

/* How each fp32 atomic accumulation (dQ partials, and dK/dV in GROUP_ATOMIC) is issued ([P1], [P3]). */
typedef enum {
  GQA_RED_V4 = 0,      /* red.global.add.v4.f32: vectorised, 16 bytes per instruction */
  GQA_RED_BULK = 1,    /* cp.reduce.async.bulk ... .add.f32: whole tile rows from shared memory */
  GQA_RED_SCALAR = 2,  /* red.global.add.f32 per element (the slow baseline of [P3]) */
  GQA_RED_NONE = 3     /* BENCHMARK ONLY: partials are stored, not added; dQ (and GROUP_ATOMIC
                          dK/dV) are WRONG.  Mirrors [P3]'s "entirely omit the atomic_add".
                          Where the bulk path exists (dQ of the main kernel) the same bulk copies
                          are issued as stores, so the difference to GQA_RED_BULK is the
                          reduction alone; elsewhere plain per-thread stores. */
} gqa_red_mode;

/* Element strides of one 16-bit [B, H, S, D] tensor along batch, head and sequence; the head-dim
 * stride is 1.  {0, 0, 0} means contiguous BHSD, i.e. {H*S*D, S*D, D}.  Otherwise every stride
 * is a multiple of 8 elements (16 bytes), h and s are >= D, and b may be 0 only when B == 1.
 * Examples: BSHD {S*H*D, D, H*D}; packed varlen THD with B = 1 {0, D, H*D}.  Outputs must not
 * overlap themselves or any input. */
typedef struct {
  int64_t b, h, s;
} gqa_stride;

typedef struct {
  int B, Hq, Hkv;        /* batch, query heads, kv heads; Hq % Hkv == 0 (group size Hq/Hkv) */
  int S;                 /* query rows per batch, or total packed query tokens when cu_seqlens != NULL;
                            also the key rows unless Sk (below) says otherwise */
  int Dqk, Dv;           /* head dims: (64,64), (128,128) or (192,128) */
  gqa_dtype dtype;
  int causal;            /* 1: key j visible to query i iff j <= i + (Lk - Lq) for a sequence of Lq
                            queries and Lk keys: the diagonal aligned at the bottom right, i.e.
                            j <= i when Lq == Lk (query rows that see no key get O = 0, LSE = -inf
                            or the sink alone, and zero gradients) */
  int window;            /* > 0: also require i + (Lk - Lq) - j < window (requires causal or
                            window_right > 0); <= 0: none */
  float scale;           /* softmax scale on Q.K^T, finite and > 0; typically 1/sqrt(Dqk) */
  const int32_t* cu_seqlens; /* DEVICE int32 [nseq+1], cu[0] = 0, non-decreasing, cu[nseq] = S;
                                NULL for dense batches.  Requires B == 1. */
  int nseq;              /* number of packed sequences (cu_seqlens != NULL) */
  int max_seqlen;        /* upper bound on every packed length; sequences longer than it are
                            rejected on the device (GQA_ERR_DEVICE_INPUT); ignored when dense */
  gqa_group_mode group_mode;
  gqa_red_mode red_mode;
  int deterministic;     /* 1: no atomics anywhere; dQ comes from a separate query-stationary
                            pass; results are bit-identical run to run; group_mode/red_mode
                            are ignored */
  /* Memory layouts of the 16-bit tensors (zero-initialised = contiguous BHSD for all of them):
   * inputs q, k, v, o (read by the backward preprocess, written by the forward), dout; outputs
   * dq, dk, dv.  LSE, Delta and dsink stay contiguous fp32 [B, Hq, S] / [Hq]. */
  gqa_stride q_st, k_st, v_st, o_st, do_st, dq_st, dk_st, dv_st;
  /* Keys fewer or more than queries (chunked prefill, a KV cache, cross-attention); all zero /
   * NULL: the same as the queries. */
  int Sk;                /* key rows per batch (k, v, dk, dv are [B,Hkv,Sk,D]), or total packed key
                            tokens; 0: Sk = S */
  const int32_t* cu_seqlens_k; /* DEVICE int32 [nseq+1] key offsets of the packed sequences (same
                                  rules as cu_seqlens, cu[nseq] = Sk), or NULL: the same offsets
                                  as cu_seqlens; requires cu_seqlens */
  int max_seqlen_k;      /* upper bound on every packed key length; 0: max_seqlen */
  int window_right;      /* > 0 (requires causal == 0): also require j - (i + Lk - Lq) < window_right,
                            a local window on the right of the diagonal (with window: two-sided);
                            <= 0: none */
} gqa_attn_params;

/* Bytes of workspace every call below needs for `p` (0 if `p` is invalid).  The
 * workspace holds the error word, the row statistics LSE*log2(e) and Delta in a
 * per-128-row tiled layout, the fp32 dQ accumulator (unless deterministic) and
 * the fp32 dK/dV accumulators (GROUP_ATOMIC).  It must be 256-byte aligned and
 * may be reused across calls on the same stream. */
size_t gqa_attn_workspace_size(const gqa_attn_params* p);

/* sizeof(gqa_attn_params) as this library was compiled: bindings check their mirror of the
 * struct against it. */
size_t gqa_attn_params_size(void);

/* Forward with causal / sliding-window / attention-sink masking ([P2] 4->2
 * commit, "flashattn_fwd: online softmax + sink + window -> O, lse").
 *   q, k, v : inputs (device, dtype).   sink : device fp32 [Hq] or NULL.
 *   o       : output [B,Hq,S,Dv] (device, dtype), laid out as p->o_st says.
 *   lse     : output [B,Hq,S] fp32, natural log, sink included:
 *             lse_i = log(exp(sink_h) + sum_{j visible} exp(scale * q_i . k_j)). */
gqa_status gqa_attn_fwd(const gqa_attn_params* p, const void* q, const void* k, const void* v,
                        const float* sink, void* o, float* lse, void* workspace, size_t ws_bytes,
                        void* stream);

/* Backward preprocess ([P2] 9->6 commit "flashattn_bwd_preprocess"; 4->2 commit
 * "Phase0(Delta) = sum(O*dO)").
 *   o, dout : forward output and its incoming gradient (device, dtype).
 *   lse     : forward LSE (device fp32 [B,Hq,S]).
 *   delta   : output, device fp32 [B,Hq,S], delta_i = sum_d dout_id * o_id.
 * Also fills the workspace's tiled row statistics and zeroes the fp32
 * accumulators that gqa_attn_bwd adds into. */
gqa_status gqa_attn_bwd_preprocess(const gqa_attn_params* p, const void* o, const void* dout,
                                   const float* lse, float* delta, void* workspace, size_t ws_bytes,
                                   void* stream);

/* Backward main kernel(s) ([P2] review thread k1..k5; [P1] Additional comments):
 * recompute S = scale*Q.K^T and P = exp(S - LSE) under the masks, dP = dO.V^T,
 * dS = P*(dP - Delta)*scale, dV = P^T.dO, dK = dS^T.Q, dQ = dS.K, with dK/dV
 * summed over the query heads of each kv head and dQ summed over KV tiles.
 * Needs gqa_attn_bwd_preprocess on the same workspace first.
 *   q, k, v, dout : inputs (device, dtype).
 *   dq            : written here only when deterministic; otherwise by postprocess.
 *   dk, dv        : written here with GQA_GROUP_TMEM (or deterministic);
 *                   otherwise by postprocess. */
gqa_status gqa_attn_bwd(const gqa_attn_params* p, const void* q, const void* k, const void* v,
                        const void* dout, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                        void* stream);

/* Backward postprocess ([P2] 9->6 commit, dual-output cast; 4->2 commit, fp32
 * atomics then cast): dq = dtype(dQaccum) unless deterministic, and with
 * GQA_GROUP_ATOMIC dk = dtype(dKaccum), dv = dtype(dVaccum).  Round to nearest even. */
gqa_status gqa_attn_bwd_postprocess(const gqa_attn_params* p, void* dq, void* dk, void* dv, void* workspace,
                                    size_t ws_bytes, void* stream);

/* Attention-sink gradient ([P2] "Kernel 9: Dsink -- dSink = -exp(sink - lse) * Delta,
 * fp32 output"): dsink_h = - sum_{b,i} exp(sink_h - lse_{b,h,i}) * delta_{b,h,i}.
 *   sink, lse, delta : device fp32 inputs.  dsink : device fp32 [Hq] output.
 * Deterministic (fixed-order reduction); needs no workspace. */
gqa_status gqa_attn_dsink(const gqa_attn_params* p, const float* sink, const float* lse, const float* delta,
                          float* dsink, void* stream);

/* Synchronises `stream`, then reports (and clears) the device error word of
 * `workspace`: GQA_OK, GQA_ERR_DEVICE_TIMEOUT or GQA_ERR_DEVICE_INPUT.  If
 * `site` is non-NULL it receives the raw word (0 if none). */
gqa_status gqa_attn_get_device_error(void* workspace, size_t ws_bytes, void* stream, int* site);

/* Upper bound, in SM clock cycles, on every mbarrier wait of the kernels
 * (process-wide; default about two seconds).  cycles <= 0 restores the default. */
void gqa_attn_set_wait_limit(long long cycles);

/* Launches one CTA that waits on an mbarrier nothing will ever complete, with
 * the current wait limit, so callers can check that a timed-out wait is
 * reported (GQA_ERR_DEVICE_TIMEOUT via gqa_attn_get_device_error) and that
 * the context stays usable.  Needs a workspace of gqa_attn_workspace_size. */
gqa_status gqa_attn_selftest_wait_timeout(void* workspace, size_t ws_bytes, void* stream);

/* No-allocation backward (no counterpart in the pages: a convenience for callers
 * that cannot allocate device memory -- e.g. code running inside a CUDA graph
 * capture that forbids cudaMalloc, or a runtime whose device memory is fixed at
 * start-up).  Runs gqa_attn_bwd_preprocess, gqa_attn_bwd and
 * gqa_attn_bwd_postprocess on `stream` with their scratch in a 16 MiB device
 * array that is part of the library (held on every GPU that loads it until the
 * process exits) instead of a caller workspace.
 *   q, k, v, o, dout, lse : inputs as for the three calls above (device).
 *   delta, dq, dk, dv     : outputs (device), written as by those calls.
 * Returns GQA_ERR_WORKSPACE when gqa_attn_workspace_size(p) exceeds 16 MiB.
 * Allocates nothing.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  All calls share the one array and it keeps the
 * last call's contents: calls that overlap on the GPU (other streams, other
 * threads) race and must be serialised by the caller.  Device-side errors (a
 * packed sequence longer than max_seqlen, a wait that timed out) are recorded in
 * the array's error word, which each call clears first: read them back with
 * gqa_attn_noalloc_get_device_error. */
gqa_status gqa_attn_bwd_noalloc(const gqa_attn_params* p, const void* q, const void* k, const void* v,
                                const void* o, const void* dout, const float* lse, float* delta, void* dq,
                                void* dk, void* dv, void* stream);

/* Companion of gqa_attn_bwd_noalloc (no counterpart in the pages either): synchronises
 * `stream`, then reports and clears the error word of the library's scratch array on the
 * current device -- GQA_OK, GQA_ERR_DEVICE_TIMEOUT or GQA_ERR_DEVICE_INPUT, the raw word in
 * *site if `site` is non-NULL -- as gqa_attn_get_device_error does for a caller workspace.
 * Allocates nothing. */
gqa_status gqa_attn_noalloc_get_device_error(void* stream, int* site);

/* Human-readable name of a status. */
const char* gqa_attn_strerror(gqa_status s);

#ifdef __cplusplus
}
#endif
#endif /* GQA_ATTN_H_ */
