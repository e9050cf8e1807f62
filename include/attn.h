/*
 * attn.h -- C ABI of the GB300 (sm_103a) fused scaled-dot-product attention
 * library: forward (O, LSE) and backward (dQ, dK, dV, dBias).
 *
 * The operations follow the fused-attention forward/backward pair of the
 * TransformerEngine pages: the unified nvte_fused_attn_fwd / nvte_fused_attn_bwd
 * calls that take separate Q/K/V pointers after the packed layouts have been
 * resolved ("[JAX] Make all jax attention calls use non-packed common calls",
 * PR #2358: description and pointer-arithmetic sequence diagram), the backward
 * that turns the saved forward output plus the incoming output gradient into
 * Q/K/V and optional bias gradients ("[JAX] Align fused attn backward output
 * gradient sharding and other test strengthening", PR #3516: diagram), with
 * THD sequences described by segment ids and positions ("[JAX] Fix batcher in
 * FusedAttn primitive ...", PR #2692: Description) or ragged offsets.
 *
 * Mathematics.  For batch row b, query head h, KV head g = h / (Hq / Hkv),
 * query i and key j:
 *   valid(i,j) = id_q[i] == id_kv[j] != 0 && (!causal || pos_kv[j] <= pos_q[i])
 *                (with a band: the band's position test in place of the causal one)
 *   S_ij = scale * Q_i . K_j + bias_ij          (masked pairs: -inf)
 *   P = softmax_j(S),  O_i = sum_j P_ij V_j,  LSE_i = ln sum_j exp(S_ij)
 *   dP_ij = dO_i . V_j,  D_i = dO_i . O_i,  dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i = scale sum_j dS_ij K_j;  dK_j = scale sum_{h in g} sum_i dS_ij Q_i
 *   dV_j = sum_{h in g} sum_i P_ij dO_i;  dBias = dS summed over broadcast axes
 * A query row with no valid key gets O = 0, LSE = -inf (its head's sink
 * logit when sink logits are given) and dQ = 0; gradients of keys no query
 * attends to are exactly 0.
 *
 * Conventions.
 *  - Every tensor is caller-owned device memory (including the workspace).
 *    The library never allocates device memory and never synchronises,
 *    except attn_read_status(), which synchronises the given stream.  Its
 *    only resources are one extra stream and two events per host thread and
 *    device, made by the first deterministic backward with d_qk, d_v <= 128
 *    outside stream capture (see attn_bwd) and kept until the process
 *    exits.
 *  - All work is ordered on the caller's stream (a cudaStream_t passed as
 *    void*; NULL is the legacy default stream); work forked to the extra
 *    stream is joined back before the call returns.
 *  - Arguments are validated on the host before anything is launched; an
 *    invalid call returns a status and launches nothing.  No call aborts.
 *  - Element type of Q/K/V/O/dO/bias and of all gradients: bf16 or fp16
 *    (attn_params_t.dtype; the MMAs take that type, accumulate in fp32, and
 *    P and dS are rounded to it).  LSE: fp32.
 *  - Token-major memory: a BSHD tensor [B, S, H, D] is B*S token rows; a THD
 *    tensor with B rows of S tokens uses the same addressing (row b, token t
 *    is token row b*S + t).  With cu_seqlens, B = 1 and S = total tokens.
 *  - Pointers must be 16-byte aligned.
 */
#ifndef GB300_ATTN_H_
#define GB300_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ATTN_PARAMS_VERSION 6

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,         /* null/misaligned pointer, bad enum, bad size */
  ATTN_ERR_UNSUPPORTED = 2,         /* valid request the library does not implement */
  ATTN_ERR_SHAPE_MISMATCH = 3,      /* segment ids/pos (or Q/KV) shapes disagree */
  ATTN_ERR_WORKSPACE_TOO_SMALL = 4, /* ws_bytes below the *_workspace_size() value */
  ATTN_ERR_CUDA = 5,                /* a CUDA runtime call failed (launch, attribute) */
  ATTN_ERR_DEVICE_TIMEOUT = 6,      /* a kernel wait ran past its limit (read via
                                       attn_read_status) */
  ATTN_ERR_DEVICE_BOUNDS = 7        /* checking build only (attn_build_flags):
                                       a device-side bounds check failed and its
                                       access was skipped (read via
                                       attn_read_status) */
} attn_status_t;

/* Q/K/V memory layouts (PR #2358, NVTE_3HD / NVTE_HD_2HD / NVTE_HD_HD_HD).
 *  3HD:      one buffer, token row = [Hq*d_qk Q | Hkv*d_qk K | Hkv*d_v V]; with
 *            Hq == Hkv and d_qk == d_v this is [T, 3, H, D].  Needs Sq == Skv.
 *            q points at the buffer; k and v are ignored.
 *  HD_2HD:   q [T_q, Hq, d_qk]; k points at a [T_kv, 2, Hkv, d_v] buffer whose
 *            V slice starts Hkv*d_v elements after K.  Needs d_qk == d_v.
 *            v is ignored.
 *  HD_HD_HD: separate q [T_q,Hq,d_qk], k [T_kv,Hkv,d_qk], v [T_kv,Hkv,d_v]. */
typedef enum { ATTN_LAYOUT_3HD = 0, ATTN_LAYOUT_HD_2HD = 1, ATTN_LAYOUT_HD_HD_HD = 2 } attn_layout_t;

/* Sequence description.
 *  BSHD:            dense rows; segment ids optional (0 = padding).
 *  THD_SEGMENTS:    rows packed with segments given by ids [B,S] (0 = padding)
 *                   and positions [B,S] (NULL: derived on the device as the
 *                   offset inside each run of equal ids).
 *  THD_CU_SEQLENS:  B = 1; ragged offsets int32[num_segments+1]; segment k of Q
 *                   pairs with segment k of KV; tokens past the last offset
 *                   are padding. */
typedef enum { ATTN_FMT_BSHD = 0, ATTN_FMT_THD_SEGMENTS = 1, ATTN_FMT_THD_CU_SEQLENS = 2 } attn_format_t;

/* Causal masking compares segment positions (pos_kv <= pos_q); without
 * segments the position is the token index (top-left alignment; see
 * attn_params_t.bottom_right for the other one).  The PADDING variants only
 * document that segment metadata is present; padding (id 0) is always
 * masked.  Sliding windows: attn_params_t.band. */
typedef enum {
  ATTN_MASK_NONE = 0,
  ATTN_MASK_CAUSAL = 1,
  ATTN_MASK_PADDING = 2,
  ATTN_MASK_PADDING_CAUSAL = 3
} attn_mask_t;

/* dQ accumulation: ATOMIC adds fp32 partial products per KV tile into an fp32
 * workspace (run-to-run order may vary in the last bits); DETERMINISTIC runs a
 * separate pass per query tile that visits KV tiles in a fixed order
 * (bit-reproducible).  dK, dV and dBias are bit-reproducible in both modes. */
typedef enum { ATTN_DQ_ATOMIC = 0, ATTN_DQ_DETERMINISTIC = 1 } attn_dq_mode_t;

/* 16-bit element type of Q/K/V/O/dO/bias and of all gradients. */
/* Element types.  ATTN_DTYPE_FP8_E4M3: forward only, Q / K / V hold E4M3
 * codes (one byte each) standing for descale_q * Q, descale_k * K and
 * descale_v * V; O is written in bf16 and LSE in fp32.  Reading (the pages use
 * bf16 only): scores are the exact products of the E4M3 values accumulated in
 * fp32, P enters P V as E4M3(256 p) with p = exp(s - m) against the row's
 * final maximum m, the normaliser l sums the p before rounding, and
 * O = descale_v * sum_j P8_j V_j / (256 l).  Needs d_qk = d_v = 128, no bias,
 * no sink (ATTN_ERR_UNSUPPORTED otherwise, and from attn_bwd and
 * attn_fwd_noalloc). */
typedef enum {
  ATTN_DTYPE_BF16 = 0,
  ATTN_DTYPE_FP16 = 1,
  ATTN_DTYPE_FP8_E4M3 = 2
} attn_dtype_t;

typedef struct {
  int32_t struct_version; /* = ATTN_PARAMS_VERSION */
  int32_t fmt;            /* attn_format_t */
  int32_t layout;         /* attn_layout_t */
  int32_t mask;           /* attn_mask_t */
  int32_t dq_mode;        /* attn_dq_mode_t (backward only) */
  int32_t B, Sq, Skv, Hq, Hkv, d_qk, d_v;
  /* Supported head dims: d_qk in {64, 128, 192}, d_v in {64, 128};
   * Hq a multiple of Hkv and at most 256 (ATTN_ERR_UNSUPPORTED beyond). */
  float scale;  /* softmax scale, applied to Q.K before the bias is added */
  const void* q;
  const void* k;
  const void* v;
  /* Segment metadata, int32 [B,S] each (THD_SEGMENTS, or BSHD with padding).
   * The *_dims pairs state each array's shape as the caller sees it; ids and
   * positions of one side must agree with each other and with (B, S). */
  const int32_t* q_seg_ids;
  const int32_t* q_seg_pos;
  const int32_t* kv_seg_ids;
  const int32_t* kv_seg_pos;
  int64_t q_ids_dims[2], q_pos_dims[2], kv_ids_dims[2], kv_pos_dims[2];
  /* Ragged offsets (THD_CU_SEQLENS): int32[num_segments + 1], non-decreasing,
   * starting at 0, last entry <= Sq (resp. Skv). */
  const int32_t* cu_seqlens_q;
  const int32_t* cu_seqlens_kv;
  int32_t num_segments;
  /* Optional post-scale bias, bf16 [bias_b, bias_h, Sq, Skv] with
   * bias_b in {1, B} and bias_h in {1, Hq}; NULL for none. */
  const void* bias;
  int32_t bias_b, bias_h;
  int32_t force_general_path; /* testing knob: skip the fast metadata path */
  /* Backward only.  Nonzero: the workspace given to attn_bwd already holds the
   * segment metadata that an attn_fwd call wrote into that same buffer for
   * these same parameters and segment arrays, nothing has written its
   * metadata region since, and attn_bwd reuses it instead of recomputing it
   * (one metadata pass per training step instead of two).  Zero: attn_bwd
   * recomputes it.  attn_fwd ignores the field. */
  int32_t metadata_from_forward;
  /* Forward only, optional (NULL: not computed).  fp32 [B, Hq], written by
   * attn_fwd: for each batch row and query head the largest logit
   * S_ij = scale * Q_i.K_j + bias_ij over the (i, j) pairs the mask keeps, in
   * natural units; -inf where no pair is kept.  4-byte aligned.  (Max-logit
   * cases of TransformerEngine PR #3516, Description item 5.1; the page does
   * not define the output, this is the plainest reading.)  attn_bwd ignores
   * the field. */
  float* max_logit;
  /* Optional sink logits, fp32 [Hq] in natural units (NULL: none): each query
   * head's sink joins every softmax row as one more logit that has no value
   * vector, so it only enlarges the normaliser; a row without valid keys then
   * gets O = 0 and LSE = its head's sink.  Read by attn_fwd and attn_bwd.
   * (Sink attention of TransformerEngine PR #2225, linked from PR #2358
   * without a definition; this is the usual reading.) */
  const float* sink;
  /* Backward only, optional (NULL: not computed; needs sink): fp32 [Hq], the
   * gradient of the loss with respect to each sink logit, summed over batch
   * rows and query rows in a fixed order (bit-reproducible). */
  float* dsink;
  /* Band mask: sliding windows and bottom-right alignment (both directions).
   * The pages define neither; this is the usual reading.  Positions are the
   * segment positions (token indices for dense rows), and
   *   shift = Skv - Sq if bottom_right != 0, else 0.
   * band == 0: no window; a causal mask keeps pos_kv[j] <= pos_q[i] + shift.
   * band != 0: key j is kept for query i (in the same nonzero segment) when
   *   -window_left <= pos_kv[j] - (pos_q[i] + shift) <= window_right,
   *   a negative window_left / window_right leaving that side unbounded.  With
   *   a causal mask window_right must be 0 or negative and is taken as 0
   *   (window_left = w - 1 then keeps the last w keys up to the diagonal).
   * ATTN_ERR_INVALID_ARG: a causal mask with window_right > 0. */
  int32_t band;
  int32_t window_left;
  int32_t window_right;
  int32_t bottom_right;
  /* attn_dtype_t of Q, K, V, O, dO, bias and the gradients (zero: bf16).  An
   * adjacent precision of the same computation (the pages use bf16 only);
   * with ATTN_DTYPE_FP8_E4M3, Q / K / V are E4M3 and O is bf16 (see
   * attn_dtype_t).  ATTN_ERR_INVALID_ARG for other values. */
  int32_t dtype;
  /* Testing knob for the failure path (zero in normal use).  Nonzero: the
   * forward kernel for query heads in pairs (even GQA group size, head dims
   * <= 128) hands out no work, so every bounded wait for work runs out
   * (after about 2 s); the kernel records ATTN_ERR_DEVICE_TIMEOUT and the
   * first wait that ran out, frees its tensor memory and exits without
   * writing O or LSE.  attn_read_status reports it; the next call on the
   * workspace starts from a clear status.  No fault, trap or endless wait. */
  int32_t test_wait_timeout;
  /* ATTN_DTYPE_FP8_E4M3 only: the factors the E4M3 Q, K, V codes stand
   * scaled by (the tensors are descale_x times the codes' values); positive
   * and finite (ATTN_ERR_INVALID_ARG otherwise).  Ignored for other types. */
  float descale_q;
  float descale_k;
  float descale_v;
} attn_params_t;

/* Which metadata path the device chose (read back by attn_read_status). */
typedef enum {
  ATTN_PATH_FAST = 0,   /* Q and KV metadata identical with standard positions:
                           masks from segment boundaries only */
  ATTN_PATH_GENERAL = 1 /* per-token id/position comparison */
} attn_path_t;

typedef enum {
  ATTN_REASON_DENSE = 0,             /* BSHD without segment ids */
  ATTN_REASON_METADATA_MATCH = 1,    /* fast: Q/KV ids and positions equal */
  ATTN_REASON_FORCED = 2,            /* general: force_general_path */
  ATTN_REASON_LENGTHS_DIFFER = 3,    /* general: Sq != Skv */
  ATTN_REASON_IDS_DIFFER = 4,        /* general: Q/KV segment ids differ */
  ATTN_REASON_POS_DIFFER = 5,        /* general: Q/KV positions differ */
  ATTN_REASON_POS_NONSTANDARD = 6,   /* general: positions do not restart at 0
                                        and count up inside each segment */
  ATTN_REASON_CU_SEQLENS_DIFFER = 7  /* general: Q/KV ragged offsets differ */
} attn_path_reason_t;

typedef struct {
  int32_t status;        /* attn_status_t of the device side (timeouts, failed
                            bounds checks of the checking build) */
  int32_t path;          /* attn_path_t of the last call using this workspace */
  int32_t reason;        /* attn_path_reason_t */
  int32_t dq_mode;       /* dQ mode actually used by the last backward */
  int64_t tile_pairs;    /* (query tile, KV tile) pairs scheduled by the last call */
  int32_t wait_site;     /* with ATTN_ERR_DEVICE_TIMEOUT: the first bounded wait
                            that ran out (kernel and role code: 0x6.. forward
                            over head pairs, 0x3.. 128-row dK/dV, 0x4.. dQ,
                            0x1.. / 0x2.. the other backward passes, 0x0.. the
                            other forward, 0x30. metadata); with
                            ATTN_ERR_DEVICE_BOUNDS: the first failed check
                            (0x7K.., K the kernel: 0 other forward, 1 forward
                            over head pairs, 2 preprocess and conversions,
                            3 128-row dK/dV, 4 dQ, 5 64-row dK/dV, 6 192-wide
                            dQ, 8 metadata); 0 otherwise */
  int32_t reserved;
} attn_stats_t;

/* Workspace bytes the forward / backward needs for these parameters (0 on
 * invalid parameters).  The workspace must be 256-byte aligned. */
size_t attn_fwd_workspace_size(const attn_params_t* p);
size_t attn_bwd_workspace_size(const attn_params_t* p);

/* Forward.  o: bf16 [B*Sq, Hq, d_v] token-major; lse: fp32 [B, Hq, Sq]
 * (natural log; -inf for rows without a valid key). */
attn_status_t attn_fwd(const attn_params_t* p, void* o, float* lse, void* ws, size_t ws_bytes,
                       void* stream);

/* Backward.  o and lse are the forward's outputs, d_o is bf16 like o.
 * Gradients are written in the input layout:
 *   3HD:      dq -> the packed dQKV buffer (dk, dv ignored);
 *   HD_2HD:   dq [T_q,Hq,d_qk]; dk -> packed dKV [T_kv,2,Hkv,d_v] (dv ignored);
 *   HD_HD_HD: dq, dk, dv separate.
 * dbias: bf16 like the bias (NULL: not computed; must be NULL without bias).
 * Every element of every gradient is written (padding rows get exact 0).
 * Streams: in deterministic mode with d_qk, d_v <= 128 the dQ pass runs on a
 * second stream that the library owns (one per host thread and device, made
 * by the first such call that is not under stream capture), forked from
 * `stream` after the preprocess and joined back before the call returns; the
 * dK/dV pass runs beside it on `stream`.  Everything later on `stream` sees
 * all gradients.  The fork and join are events, so the call can be captured
 * into a CUDA graph.  Under capture before that stream exists, or if it
 * cannot be made, both passes run one after the other on `stream`. */
attn_status_t attn_bwd(const attn_params_t* p, const void* o, const void* d_o, const float* lse,
                       void* dq, void* dk, void* dv, void* dbias, void* ws, size_t ws_bytes,
                       void* stream);

/* Synchronises `stream`, then reads the device-side status and path record of
 * the last call that used `ws`.  stats may be NULL. */
attn_status_t attn_read_status(const void* ws, void* stream, attn_stats_t* stats);

const char* attn_status_string(attn_status_t s);

/* Layout resolution (host only, no device access): element offsets of the K
 * and V slices from the pointers given and the token-row strides, in
 * elements.  Returns ATTN_OK or the validation error of the parameters. */
typedef struct {
  const void* q;
  const void* k;
  const void* v;
  int64_t q_token_stride, k_token_stride, v_token_stride;
  const void* dq;
  const void* dk;
  const void* dv;
} attn_resolved_t;
attn_status_t attn_resolve_layout(const attn_params_t* p, void* dq, void* dk, void* dv,
                                  attn_resolved_t* out);

/* Kernel-level timing (tracing).  `events` points to 2 * ATTN_TRACE_SLOTS
 * cudaEvent_t handles created by the caller (start, end of each slot), or is
 * NULL to switch tracing off.  While set (per host thread), every attn_fwd /
 * attn_bwd call records each slot's start event before the first launch of
 * that stage and its end event after the last one, on the stream the stage
 * runs on (the call's stream, or the dQ pass's second stream).  A
 * slot whose handles are NULL is skipped.  The handles are copied; the caller
 * keeps ownership. */
#define ATTN_TRACE_SLOTS 6
typedef enum {
  ATTN_TRACE_META = 0,     /* segment-metadata kernels */
  ATTN_TRACE_FWD = 1,      /* forward kernel */
  ATTN_TRACE_BWD_PRE = 2,  /* D = rowsum(dO*O), accumulator zeroing */
  ATTN_TRACE_DKDV = 3,     /* dK/dV pass (with atomic dQ) */
  ATTN_TRACE_DQ = 4,       /* deterministic dQ pass or dQ conversion; on the
                              second stream (see attn_bwd) its events span
                              from the end of the preprocess to the end of
                              the dQ pass, overlapping the dK/dV pass */
  ATTN_TRACE_DBIAS = 5     /* not recorded: a broadcast dBias is finished
                              inside the dK/dV pass */
} attn_trace_slot_t;
attn_status_t attn_set_trace_events(void* const* events);

/* Thin wrappers over the CUDA runtime's timing events for callers without a
 * CUDA binding of their own (e.g. ctypes).  attn_event_create makes a timing
 * event on the current device (caller owns it; release with
 * attn_event_destroy).  attn_event_elapsed_ms returns ATTN_ERR_CUDA if either
 * event has not completed or was never recorded. */
attn_status_t attn_event_create(void** event);
attn_status_t attn_event_destroy(void* event);
attn_status_t attn_event_elapsed_ms(const void* start, const void* end, float* ms);

/* Forward with no caller workspace and no allocation.  The pages have no
 * counterpart of this call; it exists for callers that cannot allocate device
 * memory when they run attention: plugin hosts that pass a kernel its inputs
 * and outputs but no workspace, runtimes that plan all device memory at start-up
 * and forbid allocation later, and latency-critical loops that cannot accept
 * cudaMalloc's implicit device synchronisation.
 *
 * Same arguments and outputs as attn_fwd, minus the workspace.  The scratch is
 * a fixed device array of ATTN_FWD_NOALLOC_SCRATCH_BYTES inside this library,
 * held on every GPU that loads the library until the process exits.  Calls
 * whose attn_fwd_workspace_size() exceeds that size return
 * ATTN_ERR_WORKSPACE_TOO_SMALL and launch nothing (the forward needs about
 * 16.5 bytes per query token and per key token, so B*Sq + B*Skv up to roughly
 * 250k tokens fit).
 *  - The first call on each device looks the array's device address up (this
 *    may load the module); make that first call before any stream capture.
 *  - Every call uses the same array.  Calls that overlap on the GPU (e.g. on
 *    two streams without ordering between them) race on it; order them.
 *  - Device-side status (attn_read_status) cannot be read for this call: it
 *    needs the workspace pointer, which the caller does not have.
 * No cudaMalloc/cudaFree or allocating library routine is called. */
#define ATTN_FWD_NOALLOC_SCRATCH_BYTES (4u << 20)
attn_status_t attn_fwd_noalloc(const attn_params_t* p, void* o, float* lse, void* stream);

int32_t attn_abi_version(void);

/* Properties of this build of the library, as bit flags:
 *  ATTN_BUILD_DEVICE_CHECKS  the checking build (libattn_sm103_debug.so,
 *    compiled with ATTN_DEBUG; the pages have no counterpart, it stands in for
 *    a memory checker): before every tensor-map copy and every global store a
 *    kernel checks the copy's coordinates (16-byte-aligned innermost
 *    coordinate, box inside the row, existing head, no store starting at a
 *    negative row) or the store's element range against the tensor's size.
 *    A failed check records ATTN_ERR_DEVICE_BOUNDS and the check's site in
 *    the workspace status and skips the access (no trap); waits that then go
 *    unanswered run out and the kernel unwinds as for a timeout.  Same entry
 *    points and results, slower. */
#define ATTN_BUILD_DEVICE_CHECKS 1
int32_t attn_build_flags(void);

#ifdef __cplusplus
}
#endif
#endif /* GB300_ATTN_H_ */
