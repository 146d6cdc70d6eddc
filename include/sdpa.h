/*
 * sdpa.h -- C ABI of the fused scaled-dot-product attention library for one
 * GB300 (sm_103a) GPU: libsdpa.so.
 *
 * Operation (TransformerEngine PR #3527 "Approach" and PR #3705 "Execution
 * and supported scope" describe the fused kernels this library provides;
 * the arithmetic is standard softmax attention):
 *
 *   forward   S = scale * Q K^T, masked (top-left or bottom-right causal, an
 *             optional (left, right) window), P = softmax(S) row-wise,
 *             O = P V, and LSE = ln sum_j exp(S_ij) per query row, stored as
 *             FP32 natural logarithms in a packed token-major array
 *             (PR #3705: "Stats remain packed token-major FP32 natural
 *             logarithms").
 *   backward  given Q, K, V, O, LSE and dO: recompute P from LSE and return
 *             dQ, dK, dV of the forward above (GQA heads summed into their
 *             shared K/V head).
 *
 * Layouts (PR #3527 "Scope": bshd, sbhd; PR #3705: separate Q/K/V, compact
 * THD with zero-based cumulative sequence lengths). Every tensor is
 * contiguous in its layout:
 *   SDPA_BSHD  [B, S, H, D]
 *   SDPA_SBHD  [S, B, H, D]
 *   SDPA_THD   [T, H, D]; sequence b owns rows cu_seqlens[b] .. cu_seqlens[b+1]-1
 * The "token row" of a position is its index over the leading dimensions:
 * b*S+s (BSHD), s*B+b (SBHD), cu_seqlens[b]+s (THD). LSE is float32
 * [rows_q][Hq] indexed by Q's token row. dq/dk/dv have q/k/v's layout.
 *
 * Supported: dtype bf16 or fp16 (Q, K, V, O, dO, dQ, dK, dV share it);
 * symmetric head_dim 128, 256 or 512, and for the forward alone the
 * asymmetric pair head_dim 192 (Q, K) with head_dim_v 128 (V, O) (PR #3527
 * "Scope": the forward prefill engine lists (192, 128) among its native
 * shapes, the backward requires d_qk == d_v); Hq a multiple of Hkv (q head
 * h reads kv head h / (Hq/Hkv)); every device pointer 16-byte aligned.
 *
 * Ownership: the caller owns every buffer, the workspace and the stream.
 * Pointers marked "device" must be device memory (cudaMalloc or torch);
 * the library never allocates device memory inside sdpa_fwd / sdpa_bwd and
 * never synchronises the stream there. Device-side faults in the inputs
 * (bad cu_seqlens) and bounded-wait timeouts are recorded in a per-device
 * error word that kernels check before writing outputs; read it with
 * sdpa_get_device_error. The first call on each device does a one-time
 * host-side set-up (the error word's device address, kernel attributes); a
 * device reset (cudaDeviceReset) invalidates it, so a process must not call
 * the library on a device it has reset.
 *
 * Errors: every entry point returns an sdpa_status. Host-detectable problems
 * are returned before anything is launched (an explicit decline, never a
 * fallback to another implementation).
 */
#ifndef SDPA_GB300_H
#define SDPA_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SDPA_API __attribute__((visibility("default")))
#else
#define SDPA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SDPA_OK = 0,
  SDPA_ERR_INVALID_ARG = 1,      /* null pointer, negative size, inconsistent geometry */
  SDPA_ERR_UNSUPPORTED = 2,      /* dtype, head_dim, layout or mask/window combination declined */
  SDPA_ERR_ALIGNMENT = 3,        /* a pointer is not 16-byte aligned */
  SDPA_ERR_OVERLAP = 4,          /* an output buffer overlaps an input or another output */
  SDPA_ERR_WORKSPACE_TOO_SMALL = 5,
  SDPA_ERR_BAD_SEQLENS = 6,      /* device-detected: cu_seqlens not compact / out of bounds */
  SDPA_ERR_TIMEOUT = 7,          /* device-detected: a bounded wait inside a kernel gave up */
  SDPA_ERR_CUDA = 8,             /* a CUDA runtime or driver call failed */
  SDPA_ERR_ADDRESS = 9           /* device-detected, address-checked library only: a kernel access
                                    fell outside the call's buffers and was skipped */
} sdpa_status;

typedef enum { SDPA_BSHD = 0, SDPA_SBHD = 1, SDPA_THD = 2 } sdpa_layout;

/* PR #3527 "Scope": mask types no_mask / causal / causal_bottom_right.
 * Top-left: query i's diagonal is key i. Bottom-right: query i's diagonal is
 * key i + Sk - Sq (per sequence for THD). */
typedef enum {
  SDPA_MASK_NONE = 0,
  SDPA_MASK_CAUSAL_TOP_LEFT = 1,
  SDPA_MASK_CAUSAL_BOTTOM_RIGHT = 2
} sdpa_mask;

typedef enum { SDPA_BF16 = 0, SDPA_FP16 = 1 } sdpa_dtype;

typedef struct {
  int layout;       /* sdpa_layout */
  int dtype;        /* sdpa_dtype */
  int mask_type;    /* sdpa_mask */
  int batch;        /* B; THD: number of sequences */
  int seqlen_q;     /* BSHD/SBHD: Sq. THD: the largest per-sequence q length (bounds the grid) */
  int seqlen_kv;    /* BSHD/SBHD: Sk. THD: the largest per-sequence kv length */
  int total_q;      /* THD only: rows of the packed q/o/dO/dq buffers (must equal cu_seqlens_q[B]) */
  int total_kv;     /* THD only: rows of the packed k/v/dk/dv buffers (must equal cu_seqlens_kv[B]) */
  int num_heads_q;  /* Hq */
  int num_heads_kv; /* Hkv, divides Hq */
  int head_dim;     /* D: 128, 256 or 512 */
  int window_left;  /* keys allowed left of the diagonal; -1 = unbounded (PR #3693 window pair) */
  int window_right; /* keys allowed right of the diagonal; -1 = unbounded; causal requires 0 or -1 */
  float softmax_scale; /* multiplies Q K^T before the mask, e.g. 1/sqrt(D) */
  int deterministic;   /* backward only. 0: head_dim 128 accumulates dQ with fp32 reductions (fastest,
                          not bitwise reproducible). 1: every gradient bitwise reproducible run to run
                          (head_dim 128 forms dQ in a separate pass that recomputes S and dP per query
                          tile; head_dim 256/512 are always so). Must be 0 or 1. */
  int head_dim_v;      /* Dv, the width of V and O rows (and of dV, dO): 0 or head_dim = symmetric.
                          The one asymmetric pair is head_dim 192 with head_dim_v 128, forward
                          only; sdpa_bwd and sdpa_bwd_noalloc decline it (SDPA_ERR_UNSUPPORTED). */
  int kv_chunk;        /* backward, head_dim 256/512 only (ignored elsewhere): key positions per
                          chunk of the two-phase backward, a multiple of 128; 0 = the library's
                          choice. The workspace holds the score tiles of one chunk of keys, so it
                          stays bounded however long the keys are (TransformerEngine PR #3527
                          "Known limitations": the prior art's backward workspace grows to 74 GiB
                          at 64k tokens and caps the context). Smaller chunks need less
                          workspace and repeat more per-chunk work. The library's choice keeps one
                          chunk when a bounded (left, right) window already bounds the keys a query
                          tile sees or the tile arrays fit in 512 MiB, else the largest chunk that
                          fits that budget. Negative or not a multiple of 128:
                          SDPA_ERR_INVALID_ARG. */
} sdpa_problem;

/* Bytes of device workspace sdpa_fwd / sdpa_bwd need for this problem
 * (0 when none). Returns 0 as well for a problem the library declines; call
 * sdpa_check_problem to tell the two apart. The workspace is caller-owned and
 * per call (TransformerEngine PR #3527, "Known limitations", where the
 * backward's workspace request is what caps the context length).
 * The forward needs 256 bytes for THD (the metadata guard word) and for
 * head_dim 128 (the tile counter of its persistent kernel, zeroed on the
 * stream by every call), else none. The backward needs per-row statistics
 * (8 bytes per query row and head, padded) plus: head_dim 128, a float32 dQ
 * accumulator (4 * D bytes per query row and head; none with
 * deterministic = 1); head_dim 256/512, the 16-bit P and dS score tiles of one
 * chunk of keys (see kv_chunk: 64 KiB per (query tile, key tile) pair of the
 * chunk) and, when the keys are split into several chunks, the float32 dQ
 * accumulator. It does not
 * grow with the key length beyond one chunk. */
SDPA_API size_t sdpa_fwd_workspace_size(const sdpa_problem* p);
SDPA_API size_t sdpa_bwd_workspace_size(const sdpa_problem* p);

/* Host-side validation only (no CUDA call): SDPA_OK or the reason a call
 * with this problem would be declined (by the forward; the backward declines
 * head_dim_v != head_dim as well). Declined: (head_dim, head_dim_v) not one
 * of (128|256|512, 0 or the same) or (192, 128); Hq % Hkv != 0; a causal mask with window_right > 0; a
 * bounded window on a non-causal mask when seqlen_q != seqlen_kv (PR #3527
 * "Scope": the alignment of such a window is ambiguous, so it is declined
 * rather than guessed). */
SDPA_API int sdpa_check_problem(const sdpa_problem* p);

/* Forward. q [.., Hq, D], k [.., Hkv, D], v [.., Hkv, Dv] (device, read); o [.., Hq, Dv] and
 * lse float32 [rows_q][Hq] (device, written). cu_seqlens_q/kv: device int32
 * [B+1] for THD (checked on the device on every call: cu[0] == 0,
 * non-decreasing, cu[B] == total, every length <= seqlen_q/seqlen_kv, and a
 * non-empty kv sequence wherever the q sequence is non-empty -- PR #3705's
 * compactness promise), NULL otherwise. workspace/ws_bytes: device scratch
 * of at least sdpa_fwd_workspace_size bytes (may be NULL when that is 0).
 * stream: a cudaStream_t (NULL = legacy default stream). Rows whose every
 * key is masked get o = 0 and lse = -inf. */
SDPA_API int sdpa_fwd(const sdpa_problem* p, const void* q, const void* k, const void* v, void* o, float* lse,
             const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv, void* workspace, size_t ws_bytes,
             void* stream);

/* Backward. q, k, v, o, lse, dout as produced/consumed by sdpa_fwd (device,
 * read); dq [.., Hq, D], dk, dv [.., Hkv, D] (device, written, fully
 * overwritten). workspace: device scratch of at least
 * sdpa_bwd_workspace_size bytes (float32 dQ accumulator and per-row
 * statistics). With p->deterministic = 0, head_dim 128 accumulates dQ with
 * float32 reductions, so dQ is not bitwise reproducible run to run (dK and
 * dV are); with 1, every output is. */
SDPA_API int sdpa_bwd(const sdpa_problem* p, const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dout, void* dq, void* dk, void* dv, const int32_t* cu_seqlens_q,
             const int32_t* cu_seqlens_kv, void* workspace, size_t ws_bytes, void* stream);

/* Synchronises `stream`, then returns and clears the current device's error
 * word (SDPA_OK if no kernel recorded an error). The word records what the
 * kernels detect on the device: cu_seqlens that break the compactness
 * promise of TransformerEngine PR #3705 ("Execution and supported scope":
 * zero-based cumulative lengths, checked on the GPU on every execution) as
 * SDPA_ERR_BAD_SEQLENS, and a bounded wait that gave up as SDPA_ERR_TIMEOUT. */
SDPA_API int sdpa_get_device_error(void* stream);

/* Static description of a status code. */
SDPA_API const char* sdpa_error_string(int status);

/* Number of kernels the last successful sdpa_fwd / sdpa_bwd call on this
 * host thread launched. */
SDPA_API int sdpa_last_launch_count(void);

/* Allocation-free backward (no counterpart in the pages: an addition for
 * callers that cannot allocate device memory -- a plugin whose host owns all
 * device allocations, a C caller with no allocator, or a path that cannot
 * afford the device-wide synchronisation of cudaMalloc/cudaFree).
 * Same arguments and results as sdpa_bwd, without the workspace: the scratch
 * comes from a static array of SDPA_BWD_NOALLOC_MAX_BYTES in the library's
 * device memory, which every GPU that loads the library holds until the
 * process exits. Problems whose sdpa_bwd_workspace_size exceeds that maximum
 * are rejected with SDPA_ERR_WORKSPACE_TOO_SMALL before any launch. The first
 * call on a device looks up the array's device address (a one-time host-side
 * set-up); make that first call before any stream capture. A device reset
 * (cudaDeviceReset) unloads the library's device code and with it the array:
 * the address looked up before it is stale, so do not call this entry point
 * (or any other, see the per-device set-up under "Ownership") on a device
 * after resetting it in the same process. Every call shares
 * the array: calls that overlap on the GPU (e.g. on two streams at once) race
 * and must be serialised by the caller. No call allocates memory. */
#define SDPA_BWD_NOALLOC_MAX_BYTES (32u << 20)
SDPA_API int sdpa_bwd_noalloc(const sdpa_problem* p, const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dout, void* dq, void* dk, void* dv,
                              const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv, void* stream);

/* Testing aid, off by default: caps how many CTAs any tcgen05 kernel of the
 * library has in flight at once (0 = no cap, the default; negative:
 * SDPA_ERR_INVALID_ARG). The persistent head_dim 128 forward launches at most
 * max_ctas CTAs, which then take every query tile from the ticket counter;
 * every other attention kernel is launched as successive grids of at most
 * max_ctas CTAs. Results must not depend on the cap (dQ of the head_dim 128
 * backward with deterministic = 0 only up to the order of its fp32
 * reductions): it reschedules the same work, which is how a test shakes out
 * ordering, ticket, queue and barrier-phase assumptions that element-wise
 * parity at one schedule cannot (the sanitizers' race and sync checks are
 * the other route). Process-wide; slow for large problems. */
SDPA_API int sdpa_debug_set_max_ctas(int max_ctas);

/* Address checking (testing aid; a stand-in for a memory checker, which
 * answers the sanitizers' out-of-bounds question that element-wise parity
 * cannot: a stray write can land where no test looks). Only the separately
 * built checked library, libsdpa_checked.so (the same sources compiled with
 * SDPA_ADDR_CHECK), answers these; the normal library returns
 * SDPA_ERR_UNSUPPORTED and checks nothing.
 *
 * In the checked library every entry point registers the byte extents of the
 * buffers it was given (inputs, outputs, cu_seqlens, workspace) in a
 * per-device table, and every kernel load or store at a computed global
 * address -- each access that is not a tensor-map (TMA) copy, which the
 * hardware bounds against its map -- first tests its bytes against those
 * extents. An access outside all of them is skipped (a skipped bulk load still
 * completes its transaction count, so no pipeline waits on it), counted, and
 * its address kept; the call's device error word becomes SDPA_ERR_ADDRESS.
 * The table is per device, so calls on several streams at once share it:
 * check one stream at a time.
 *
 * sdpa_debug_address_report synchronises the current device, stores the
 * number of violations since the last report, the first offending address
 * and its size (any pointer may be NULL), and clears them.
 * sdpa_debug_address_shrink(bytes) pulls the end of every extent registered
 * from then on in by `bytes` (0 restores them): the last bytes of each buffer
 * become out of bounds for the checker while staying valid memory, which
 * tests the checker itself without any access outside a real allocation. */
SDPA_API int sdpa_debug_address_report(unsigned long long* violations, unsigned long long* first_addr,
                                       unsigned long long* first_bytes);
SDPA_API int sdpa_debug_address_shrink(long long bytes);

/* Failure-path self-test of the bounded waits every pipelined kernel uses:
 * launches one thread that waits on a barrier nothing arrives on, gives up
 * after limit_us microseconds (1 .. 1,000,000) and records SDPA_ERR_TIMEOUT
 * in the device error word, as a stalled kernel would. The GPU context stays
 * usable; read and clear the result with sdpa_get_device_error. */
SDPA_API int sdpa_selftest_bounded_wait(unsigned limit_us, void* stream);

/* Merge of partial results over a split of the keys (the context-parallel
 * LSE handling of TransformerEngine PR #3527 "Context parallelism" and
 * PR #3693, which keeps "neutral statistics for empty ragged ring blocks"):
 * for every item (one row of one head)
 *     LSE = ln sum_k exp(LSE_k),   O = sum_k exp(LSE_k - LSE) O_k.
 * A block that saw no keys carries LSE_k = -inf and contributes nothing
 * (its O rows are not read); an item whose blocks are all empty gets O = 0
 * and LSE = -inf, the forward's convention for a row without keys.
 * o_parts: device, n_parts blocks of [items][head_dim] 16-bit values, block
 *   k at element offset k * items * head_dim (e.g. sdpa_fwd outputs over n
 *   key blocks, stacked; items = rows x heads of the generic view).
 * lse_parts: device fp32 [n_parts][items] (natural log, the forward's LSE).
 * o: device [items][head_dim] (dtype), lse: device fp32 [items]; written.
 * All pointers 16-byte aligned; the outputs may not overlap the inputs.
 * Errors: SDPA_ERR_INVALID_ARG (null pointer, n_parts outside 1..64,
 * items < 0), SDPA_ERR_UNSUPPORTED (dtype, head_dim not 128/256/512),
 * SDPA_ERR_ALIGNMENT, SDPA_ERR_OVERLAP, SDPA_ERR_CUDA. Asynchronous on
 * `stream` (a cudaStream_t, NULL = legacy default stream). */
typedef struct {
  int dtype;        /* sdpa_dtype of o_parts and o */
  long long items;  /* rows x heads of one block */
  int head_dim;     /* 128, 256 or 512 */
  int n_parts;      /* number of key blocks, 1..64 */
} sdpa_merge_problem;
SDPA_API int sdpa_merge(const sdpa_merge_problem* p, const void* o_parts, const float* lse_parts, void* o, float* lse,
               void* stream);

/* FP8 E4M3 forward, head_dim 128 or 256 (TransformerEngine PR #3705's closing note
 * on FP8: with E4M3 inputs the softmax output is stored in E4M3 under the
 * fixed scale 448, so no amax of it is needed; PR #3527 "Scope" lists the
 * FP8 fused path at head dims up to 256). Computes, with the decoded values
 * of the codes,
 *   S = softmax_scale * descale_q * descale_k * Q8 K8^T, masked as sdpa_fwd;
 *   m = max_j S_ij, l = sum_j exp(S_ij - m), LSE = m + ln l   (float32,
 *       token-major, as sdpa_fwd);
 *   P8  = E4M3(exp(S - m) * 448)   (round to nearest even; the row's largest
 *         probability is stored as 448, so no amax is needed);
 *   O   = P8 V8 * descale_v / (448 * l)   (written in p->dtype: bf16 or fp16).
 * q8 [.., Hq, D], k8 and v8 [.., Hkv, D]: device E4M3 codes (the finite-
 * only OCP format: bias 7, largest 448, S.1111.111 = NaN), one byte each, in
 * p->layout; o [.., Hq, D] and lse as for sdpa_fwd (device, written).
 * p->head_dim = D must be 128 or 256 (head_dim_v 0 or D), else
 * SDPA_ERR_UNSUPPORTED;
 * p->dtype is O's type. Descales: finite and > 0, else SDPA_ERR_INVALID_ARG.
 * workspace: at least sdpa_fwd_fp8_workspace_size bytes, 256-byte aligned
 * (the THD guard word, the query-tile ticket counter, and V transposed to
 * [Hkv][D][keys], one byte per key, every sequence starting on a 16-byte
 * boundary). Launches (THD guard), the transpose, a 4-byte memset of the ticket
 * counter and the attention kernel on `stream`; errors as sdpa_fwd. */
SDPA_API size_t sdpa_fwd_fp8_workspace_size(const sdpa_problem* p);
SDPA_API int sdpa_fwd_fp8(const sdpa_problem* p, const void* q8, const void* k8, const void* v8, float descale_q,
                          float descale_k, float descale_v, void* o, float* lse, const int32_t* cu_seqlens_q,
                          const int32_t* cu_seqlens_kv, void* workspace, size_t ws_bytes, void* stream);

/* Kernel timing for benchmarks and tracing. Between sdpa_profile_begin and
 * sdpa_profile_end, every sdpa_fwd / sdpa_bwd call made by this host thread
 * (and sdpa_merge) records a pair of CUDA events on its stream around each kernel it
 * launches. sdpa_profile_end synchronises those events and writes, per kernel
 * kind (SDPA_KERNEL_*), the summed milliseconds and the number of launches
 * into arrays of n_kinds entries. At most 65536 launches are recorded. */
typedef enum {
  SDPA_KERNEL_FWD = 0,        /* forward attention kernel */
  SDPA_KERNEL_BWD = 1,        /* backward dK/dV/dQ kernel */
  SDPA_KERNEL_PREPROCESS = 2, /* backward preprocess (delta, LSE rescale, dQ accumulator zeroing) */
  SDPA_KERNEL_DQ_FINALIZE = 3,
  SDPA_KERNEL_GUARD = 4,      /* THD metadata guard */
  SDPA_KERNEL_MERGE = 5,      /* log-sum-exp merge of key-split partial results */
  SDPA_KERNEL_BWD_DQ = 6,     /* deterministic backward: the separate head_dim 128 dQ pass */
  SDPA_KERNEL_V_TRANSPOSE = 7, /* FP8 forward: V transposed into the workspace */
  SDPA_KERNEL_KINDS = 8
} sdpa_kernel_kind;
SDPA_API int sdpa_profile_begin(void);
SDPA_API int sdpa_profile_end(double* ms_by_kind, int* launches_by_kind, int n_kinds);

#ifdef __cplusplus
}
#endif
#endif /* SDPA_GB300_H */
