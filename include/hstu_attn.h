/*
 * hstu_attn.h — C ABI of the GB300 (sm_103a) HSTU attention forward.
 *
 * The operation (composable_kernel example 18_hstu_attention README,
 * "Forward computation", "Masking", "Modes of operation", "Split-KV"): for
 * every sequence b, head h, query row i and key row j
 *
 *     s[i,j] = alpha * <q[i,h,:], k[j,h,:]>
 *     s[i,j] = 0 where the functional mask rules (i,j) out
 *     SiLU mode:    o[i,h,:] = attn_scale_g * sum_j SiLU(s[i,j]) * v[j,h,:]
 *     softmax mode: o[i,h,:] = attn_scale_g * sum_j softmax_j(s[i,:]) v[j,h,:]
 *                   over the allowed j only; lse[h,i] = log sum_{allowed j} exp(s[i,j])
 *
 * over jagged sequences laid out [context | UIH | targets] (query side; the key
 * side is the same sequence for self-attention, [context | UIH_kv] for
 * cross-attention, or [context | UIH_kv | targets] for cross-attention with
 * kv_targets: an M-FALCON candidate microbatch over a cached history, "From
 * transformer parallelism to HSTU", section 5.3).  The mask is the composite of the causal, local-window,
 * contextual, min-full and target components of the README's "Masking" table:
 *   - context keys (j < c) are visible to every query;
 *   - a target key is visible only to its own row (target r: query row
 *     c + u + r, key row c + uih_kv + r);
 *   - context rows see context keys and every UIH key;
 *   - UIH and target rows see UIH keys by UIH coordinate x (query UIH row:
 *     x = (i - c) + (uih_kv - uih_q), bottom-right aligned; target row:
 *     x = uih_kv; key: x = j - c): causal keeps x_j <= x_i; a local window
 *     W > 0 keeps |x_i - x_j| <= W unless the row is min-full
 *     (minfull F > 0 and x_i >= uih_kv - F).
 *
 * Every entry point is host-callable and asynchronous on `stream` unless it
 * says otherwise.  The library allocates no device or host memory and keeps no
 * state between calls other than per-device caches of kernel attributes and the
 * fixed scratch of hstu_attn_fwd_static_ws; the caller owns every other buffer,
 * including the workspace.
 */
#ifndef HSTU_ATTN_H_
#define HSTU_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define HSTU_ABI_VERSION 6
#define HSTU_MAX_GROUPS 256
#define HSTU_MAX_SPLITS 16
#define HSTU_RAB_TIME_BUCKETS 11
#define HSTU_RAB_MAX_POS 256

typedef enum hstu_status {
  HSTU_OK = 0,
  HSTU_ERR_INVALID_ARG = 1,  /* a host-checkable argument is wrong (null, negative, misaligned...) */
  HSTU_ERR_UNSUPPORTED = 2,  /* valid but not implemented (head dim, dtype, group count...) */
  HSTU_ERR_WORKSPACE = 3,    /* workspace missing or smaller than hstu_attn_fwd_workspace_size */
  HSTU_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed (no device, launch failure...) */
  HSTU_ERR_DEVICE = 5        /* a device-side check failed (see the HSTU_DEVERR_* bits) */
} hstu_status;

/* Bits of the device error word (hstu_attn_fwd_check). */
#define HSTU_DEVERR_OFFSETS 1     /* offsets not non-decreasing or beyond total_q / total_kv */
#define HSTU_DEVERR_Q_LAYOUT 2    /* a query length < context_len + num_targets */
#define HSTU_DEVERR_KV_LAYOUT 4   /* a cross-attention key length < context_len (+ num_targets with kv_targets) */
#define HSTU_DEVERR_MAXSEQ 8      /* a length exceeds max_seqlen_q / max_seqlen_kv */
#define HSTU_DEVERR_TIMEOUT 16    /* a pipeline wait gave up; outputs are incomplete */

typedef enum hstu_dtype { HSTU_DTYPE_FP16 = 0, HSTU_DTYPE_BF16 = 1 } hstu_dtype;

/*
 * Arguments of one forward call.  Device pointers are marked [dev], host
 * pointers [host]; all are borrowed for the duration of the call (the host
 * arrays are read before hstu_attn_fwd returns).
 */
typedef struct hstu_fwd_args {
  int32_t dtype;          /* hstu_dtype of q, k, v and o (README "Data types": fp16 / bf16) */
  int32_t batch;          /* number of sequences B >= 1 */
  int32_t nhead;          /* heads H >= 1 */
  int32_t hdim_qk;        /* 64, 96, 128 or 256 (the head sizes the README lists as supported) */
  int32_t hdim_v;         /* equal to hdim_qk, or 64 with hdim_qk 96 (asymmetric 96/64) */
  int32_t total_q;        /* rows of q and o (tokens of all sequences) */
  int32_t total_kv;       /* rows of k and v; self-attention: == total_q */
  int32_t max_seqlen_q;   /* upper bound of every physical query length; 0 = total_q */
  int32_t max_seqlen_kv;  /* upper bound of every physical key length; 0 = total_kv */
  int32_t causal;         /* README --causal: 1 = lower-triangular on UIH positions */
  int32_t softmax;        /* 0 = SiLU, 1 = softmax (README --softmax) */
  int32_t num_groups;     /* G >= 1, batch % G == 0, G <= HSTU_MAX_GROUPS; group g = b / (B/G) */
  int32_t num_splits;     /* split-KV: 0 = automatic, 1 = none, n = n splits (<= HSTU_MAX_SPLITS) */
  float alpha;            /* QK scale; 0 = 1/sqrt(hdim_qk) (README -alpha) */
  /* Elements between consecutive tokens; 0 = nhead * hdim (packed).  q/k/v/o
   * are [tokens, nhead, hdim] with unit stride in hdim and nhead*hdim stride
   * between heads within a token.  Row strides * 2 bytes must be multiples of 16. */
  int64_t q_row_stride, k_row_stride, v_row_stride, o_row_stride;
  const void* q;          /* [dev] [total_q, H, hdim_qk], 16-byte aligned */
  const void* k;          /* [dev] [total_kv, H, hdim_qk], 16-byte aligned */
  const void* v;          /* [dev] [total_kv, H, hdim_v], 16-byte aligned */
  void* o;                /* [dev] [total_q, H, hdim_v], 16-byte aligned; rows outside every
                             sequence are left untouched */
  float* lse;             /* [dev] [H, total_q] fp32 natural-log LSE (softmax only) or NULL;
                             a row with no allowed key gets -inf and o = 0 */
  const int32_t* seq_offsets_q;   /* [dev] [B+1] token offsets of the query sequences (README
                                     "Batch modes": jagged; batched = offsets b*S) */
  const int32_t* seq_offsets_kv;  /* [dev] [B+1] key offsets; NULL = self-attention */
  const int32_t* num_targets;     /* [dev] [B] targets at the end of each query sequence; NULL = 0 */
  const int32_t* local_len;       /* [host] [G] local window W (0 = none); NULL = all 0 */
  const int32_t* context_len;     /* [host] [G] context prefix c; NULL = all 0 */
  const int32_t* minfull_len;     /* [host] [G] min-full tail F; NULL = all 0 */
  const int32_t* max_uih_len;     /* [host] [G] max UIH length used by the attn_scale default;
                                     0 / NULL = the largest query UIH length of the group */
  const float* attn_scale;        /* [host] [G] post-nonlinearity scale; 0 / NULL = 1/max_uih_len */
  void* workspace;                /* [dev] caller-owned scratch, 256-byte aligned */
  size_t workspace_bytes;         /* its size, >= hstu_attn_fwd_workspace_size() */
  /* Optional cudaEvent_t handles (NULL = none), recorded on `stream` right
   * before and right after the forward kernel's launch, so a caller can time
   * that kernel alone (the scheduler and combine kernels fall outside). */
  void* event_fwd_begin;
  void* event_fwd_end;
  /* Cross-attention only (seq_offsets_kv set): 1 = each key sequence is
   * [context | UIH_kv | targets] with the same num_targets as its query
   * sequence, the targets' own keys; target r of the queries sees target key r
   * of the keys and no other target key.  0 = [context | UIH_kv]. */
  int32_t kv_targets;
  /* Relative attention bias ("From transformer parallelism to HSTU", sections
   * 2.4 and 3.5), added to alpha * <q, k> before SiLU / softmax:
   *   rab[i,j] = rab_time[h, bucket(|ts_i - ts_j|)] + rab_pos[h, min(|pos_i - j|, P - 1)]
   * Time-gap buckets by lower edge in seconds: 0, 1, 5, 30, 60, 300, 1800,
   * 3600, 86400, 604800, 2.6e6 (the last open-ended).  pos_i is query row i's
   * position in key coordinates: i for a context row, i + (uih_kv - uih_q)
   * for UIH and target rows (the mask's bottom-right alignment).  Gaps are
   * exact unless the 128 keys of one key tile span 2^29 s (17 years) or
   * more.  The bias works at every head-dimension pair the forward
   * supports; everything NULL / 0 = no bias. */
  const int64_t* timestamps_q;    /* [dev] [total_q] seconds; required with rab_time */
  const int64_t* timestamps_kv;   /* [dev] [total_kv]; cross-attention with rab_time (NULL for
                                     self-attention, which uses timestamps_q) */
  const float* rab_time;          /* [dev] [H, HSTU_RAB_TIME_BUCKETS] one scalar per head and bucket */
  const float* rab_pos;           /* [dev] [H, rab_pos_buckets] one scalar per head and clamped distance */
  int32_t rab_pos_buckets;        /* P: 1..HSTU_RAB_MAX_POS with rab_pos, else ignored */
  /* Forward kernel choice where both apply (hdim_qk == hdim_v == 128, no
   * bias, batch <= 128): the CTA-pair kernel runs two query tiles of one
   * (sequence, head) on the two SMs of a TPC as one 256-row tile, each SM
   * loading half of every key and value tile; the single-CTA kernel runs one
   * query tile per SM.  Both compute the same results.
   * 0 = automatic (single CTAs, the faster on every measured workload),
   * 1 = pairs, -1 = single CTAs.  Ignored elsewhere. */
  int32_t cta_pairs;
} hstu_fwd_args;

/* Counters of one call's schedule (hstu_attn_fwd_stats). */
typedef struct hstu_fwd_stats {
  int64_t executed_tiles;   /* (b, h, 128-row query tile, 128-key tile) blocks the kernel runs */
  int64_t allowed_pairs;    /* (b, h, i, j) entries the mask allows: the useful GEMM work */
  int32_t work_units;       /* (b, h, query tile, split) units in the persistent queue */
  int32_t num_splits;       /* KV splits chosen for the call */
  int32_t device_error;     /* HSTU_DEVERR_* bits found by the scheduler */
  int32_t reserved;
} hstu_fwd_stats;

/* Library ABI version (HSTU_ABI_VERSION). */
int32_t hstu_abi_version(void);

/* Static string naming a status; never NULL. */
const char* hstu_status_string(hstu_status status);

/*
 * Workspace bytes a call with these arguments needs (pointer fields are not
 * read).  Depends on batch, nhead, hdim, total_q, the max_seqlen hints and the
 * split count.  Synchronous, host only.  Returns HSTU_ERR_INVALID_ARG /
 * HSTU_ERR_UNSUPPORTED for the same argument errors as hstu_attn_fwd.
 */
hstu_status hstu_attn_fwd_workspace_size(const hstu_fwd_args* args, size_t* bytes);

/*
 * The forward (README "Forward computation").  Launches, on `stream`, the
 * scheduler kernel, the persistent tcgen05 forward kernel and, with split-KV
 * (README "Split-KV"), the combine kernel that merges the splits' fp32
 * partials into o (and lse); returns without synchronising.  Host-checkable errors
 * return before anything is launched and leave o/lse untouched.
 * Data-dependent errors (bad offsets, lengths beyond the hints) make the
 * kernels skip all work and set the device error word, read back by
 * hstu_attn_fwd_check.  Not thread-safe against concurrent calls sharing one
 * workspace.  `stream` is a cudaStream_t (NULL = legacy default stream).
 */
hstu_status hstu_attn_fwd(const hstu_fwd_args* args, void* stream);

/*
 * Synchronises `stream`, then reads the device error word the last forward
 * using `workspace` left there into *device_error (may be NULL).  Returns
 * HSTU_ERR_DEVICE when it is non-zero, HSTU_ERR_CUDA on a CUDA error.
 */
hstu_status hstu_attn_fwd_check(const void* workspace, void* stream, int32_t* device_error);

/*
 * Runs only the scheduler and a pair-count kernel for these arguments (no
 * attention arithmetic; o and lse are not written), synchronises `stream` and
 * fills *stats.  Uses the workspace like hstu_attn_fwd.
 */
hstu_status hstu_attn_fwd_stats(const hstu_fwd_args* args, void* stream, hstu_fwd_stats* stats);

/* Number of streaming multiprocessors of the current device (0 on error). */
int32_t hstu_device_sm_count(void);

/* sizeof(hstu_fwd_args) as compiled into the library (binding layout check). */
size_t hstu_fwd_args_size(void);

/*
 * Self-test of the kernels' time-bounded waits (no counterpart in the README;
 * it exercises this library's failure detection).  Launches one CTA on
 * `stream` that waits on a shared-memory barrier nothing ever arrives on,
 * using the same bounded wait as the forward kernel, for at most timeout_ns
 * nanoseconds; the kernel then stores 1 (gave up, the expected outcome) or 0
 * to *result_dev ([dev] one int32, caller-owned) and returns normally.
 * Synchronises `stream` and copies the flag to *timed_out.
 */
hstu_status hstu_selftest_wait_timeout(int32_t* result_dev, uint64_t timeout_ns, void* stream,
                                       int32_t* timed_out);

/*
 * Arguments of one backward call (the gradients of the forward above): the
 * forward call's own arguments plus the output gradient and the three input
 * gradients, all [dev] and 16-byte aligned, in the storage type of q.
 */
typedef struct hstu_bwd_args {
  /* The forward call's arguments.  Read: every shape, mask, group and scale
   * field, alpha, q, k, v, the offsets and num_targets; softmax mode also reads
   * o and lse as the forward wrote them.  fwd.workspace / fwd.workspace_bytes
   * hold the backward's own workspace (hstu_attn_bwd_workspace_size);
   * num_splits and the two events are ignored. */
  hstu_fwd_args fwd;
  const void* d_o;        /* [dev] [total_q, H, hdim_v] gradient of the loss with respect to o */
  void* dq;               /* [dev] [total_q, H, hdim_qk] written: gradient with respect to q */
  void* dk;               /* [dev] [total_kv, H, hdim_qk] written: gradient with respect to k */
  void* dv;               /* [dev] [total_kv, H, hdim_v] written: gradient with respect to v */
  /* Elements between consecutive tokens; 0 = packed (nhead * hdim).  Row
   * strides * 2 bytes must be multiples of 16. */
  int64_t do_row_stride, dq_row_stride, dk_row_stride, dv_row_stride;
  /* Gradients of the relative attention bias tables ("From transformer
   * parallelism to HSTU" section 3.5: the bias is added to the scaled score,
   * so an entry's gradient is the sum of ds over the (row, key) pairs, of every
   * sequence, that read it).  Optional: NULL = not computed.
   *   d_rab_time [dev] [H, HSTU_RAB_TIME_BUCKETS] fp32, needs fwd.rab_time and
   *              fwd.timestamps_q;
   *   d_rab_pos  [dev] [H, rab_pos_buckets] fp32, needs fwd.rab_pos.
   * Written (overwritten) by the call; 4-byte aligned.  The sums are
   * accumulated with floating-point atomics, so their last bits depend on
   * the order the kernels run in. */
  float* d_rab_time;
  float* d_rab_pos;
} hstu_bwd_args;

/* sizeof(hstu_bwd_args) as compiled into the library (binding layout check). */
size_t hstu_bwd_args_size(void);

/*
 * Workspace bytes of a backward call (pointer fields are not read).
 * Synchronous, host only; same argument errors as hstu_attn_bwd.
 */
hstu_status hstu_attn_bwd_workspace_size(const hstu_bwd_args* args, size_t* bytes);

/*
 * The backward of the forward (the exact derivative of "Forward computation";
 * the README's training mode keeps the softmax LSE for it).  With
 * s = alpha q k^T on the allowed entries, c = attn_scale of the group and
 * g = d_o, per sequence and head:
 *   SiLU:    a = SiLU(s) masked       dv = c a^T g,  ds = (c g v^T) . SiLU'(s) masked
 *   softmax: p = exp(s - lse) masked  dv = c p^T g,  ds = p . (c g v^T - rowsum(g . o))
 *   both:    dq = alpha ds k,  dk = alpha ds^T q
 * Head dimensions: hdim_qk == hdim_v in {64, 96, 128}, or 96 with hdim_v 64
 * (others HSTU_ERR_UNSUPPORTED), with or without a bias.
 * With a relative attention bias in fwd, s includes it and every gradient
 * flows through it; d_rab_time / d_rab_pos (when set) receive the tables'
 * gradients.
 * Launches on `stream` the scheduler, in softmax mode a row-sum kernel, then
 * one persistent tcgen05 kernel per query tile (dq) and one per key tile (dk,
 * dv); returns without synchronising.  Every row of every sequence gets its
 * gradient (0 where the mask allows nothing); rows outside every sequence are
 * left untouched.  Host-checkable errors return before any launch and write
 * nothing; data-dependent errors set the device error word in the workspace,
 * read back by hstu_attn_fwd_check(args->fwd.workspace, ...).  Not thread-safe
 * against concurrent calls sharing one workspace.
 */
hstu_status hstu_attn_bwd(const hstu_bwd_args* args, void* stream);

/* Size of the library's fixed scratch used by hstu_attn_fwd_static_ws. */
#define HSTU_STATIC_WS_BYTES (4u << 20)

/*
 * The forward without a caller workspace (no counterpart in the README; the
 * README's forward has the framework allocate its buffers).  Same arguments,
 * launches and results as hstu_attn_fwd, except that args->workspace and
 * args->workspace_bytes are ignored: the scratch is a fixed array of
 * HSTU_STATIC_WS_BYTES bytes per device, built into this library, and the call
 * makes no cudaMalloc, cudaFree or other allocating call.
 *
 * It is meant for callers that cannot allocate device memory per call: a plain
 * C or C++ host loop without a caching allocator, where cudaFree waits for the
 * whole device and a per-call cudaMalloc would stall other streams; or code
 * that has given all its device memory to a fixed budget up front.
 *
 * Limits and ordering:
 *  - Calls whose hstu_attn_fwd_workspace_size exceeds HSTU_STATIC_WS_BYTES are
 *    rejected with HSTU_ERR_WORKSPACE before anything is launched (typically
 *    split-KV on long batches, whose fp32 partials need more room).
 *  - The first call on a device looks up the array's device address (which
 *    may load this library's kernels into the context) and sets the kernels'
 *    attributes; make that first call before any stream capture begins.  If
 *    the lookup fails the call returns HSTU_ERR_CUDA and the next call tries
 *    it again; only a successful lookup is kept.
 *  - There is one scratch per device.  Calls on one stream run one after
 *    another and are safe; calls in flight at the same time on different
 *    streams or from different host threads race on it and give wrong results.
 *  - Each call first clears the scratch's header (its work counter and device
 *    error word must start at zero) with cudaMemsetAsync on `stream`; the rest
 *    of the scratch is written before it is read.
 *
 * *workspace_used ([host], may be NULL) receives the scratch's device address,
 * for hstu_attn_fwd_check.
 */
hstu_status hstu_attn_fwd_static_ws(const hstu_fwd_args* args, void* stream, const void** workspace_used);

#ifdef __cplusplus
}
#endif

#endif /* HSTU_ATTN_H_ */
