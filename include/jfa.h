/*
 * jfa.h -- C ABI of the GB300 (sm_103a) Jagged Flash Attention library.
 *
 * Operation.  Exact softmax attention, forward and backward, computed directly on
 * variable-length sequences packed as jagged tensors (values plus int64 offsets),
 * never padded to the longest sequence, with an optional per-head additive bias and
 * unequal query and key/value lengths ("Jagged Flash Attention (JFA)", Definition).
 * "Exact" is the FlashAttention sense: tiling plus online softmax changes only the
 * rounding, never the function ("TLX-Optimized Jagged Flash Attention: Approaching
 * FA4-Level Performance on Blackwell", section "Why Jagged Flash Attention Deserves
 * Attention").  For sequence b, head h, local query row i < Lq_b and key j < Lk_b:
 *
 *   s_ij   = scale * q_i . k_j + beta_h(i, j)
 *   lse_i  = ln sum_j exp(s_ij)                 (over visible j)
 *   out_i  = sum_j exp(s_ij - lse_i) v_j
 *
 * with Lq_b = q_offsets[b+1] - q_offsets[b], Lk_b = kv_offsets[b+1] - kv_offsets[b].
 * Causal: key j is visible to query i iff j <= i + (Lk_b - Lq_b) (bottom-right
 * alignment; equal lengths give the usual j <= i).  A query row with no visible key
 * (Lk_b = 0, or causal with Lq_b > Lk_b) gets out = 0 and lse = -inf, and no gradient.
 *
 * Layout.  q, out, dout, dq: bf16 [total_q, H, d] row-major (token-major, heads
 * contiguous); k, v, dk, dv: bf16 [total_kv, H, d]; lse: fp32 [H, total_q];
 * offsets: int64 [B+1], offsets[0] = 0, non-decreasing, offsets[B] = total.  Empty
 * sequences are allowed.
 *
 * Ownership and execution.  Every pointer is a DEVICE pointer owned by the caller.
 * The library allocates nothing, keeps no state between calls (one process-wide
 * cache of driver entry points aside), and enqueues all work asynchronously on
 * `stream`.  Scratch memory is the caller's `workspace` (size from
 * jfa_workspace_size, 256-byte aligned, and its first 256 bytes zero before its first
 * use -- jfa_check_status keeps them so).  Calls sharing a workspace must not overlap.
 *
 * Errors.  Argument errors detectable on the host are returned synchronously and
 * enqueue nothing.  Errors found on the device (malformed offsets, a bounded
 * pipeline wait that ran out) are recorded in a status word in the workspace, the first
 * one sticking until jfa_check_status (which synchronises the stream) reads and clears
 * it.  On a device error the outputs of that call are unspecified.
 *
 * Requirements.  d in {64, 128}; H >= 1; B >= 1; every tensor pointer 16-byte
 * aligned; an sm_100-family GPU (built for sm_103a).
 */
#ifndef JFA_H_
#define JFA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* jfa_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  JFA_OK = 0,
  JFA_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer */
  JFA_ERR_UNSUPPORTED = 2, /* head_dim not in {64,128}, unsupported bias kind or bias gradient */
  JFA_ERR_WORKSPACE = 3,   /* workspace missing, too small or misaligned */
  JFA_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed (launch, tensor-map encode) */
  JFA_ERR_BAD_OFFSETS = 5, /* device: offsets not 0-based, not monotone, or last != total (also kind-2 bias block offsets) */
  JFA_ERR_TIMEOUT = 6      /* device: a bounded pipeline wait ran out; outputs unspecified */
} jfa_status;

/* Additive attention bias (the user-defined biases of "Jagged Flash Attention
 * (JFA)", Definition).  kind 0 = none.  kind 2 = general jagged bias (below).
 * kind 1 = per-head relative-position table:
 *   beta_h(i, j) = table[h * num_buckets + clamp(j - i + center, 0, num_buckets - 1)]
 * with i, j local 0-based positions; added after scaling.  `table` is a device
 * fp32 [H][num_buckets] array; num_buckets in [1, 8192].
 * `grad` (kind 1, jfa_backward only; NULL = not wanted): a device fp32 [H][num_buckets]
 * array, 4-byte aligned, not overlapping any other argument, that jfa_backward
 * overwrites with the gradient of sum(dout * out) w.r.t. `table`: entry (h, n) is the sum
 * of dS_ij = P_ij (dP_ij - D_i) over every sequence's visible pairs (i, j) whose bucket is
 * n.  It is accumulated with fp32 additions in L2 whose order is not fixed, so repeated
 * calls can differ in the last bits.  jfa_forward ignores it.
 * kind 2 = general jagged bias: beta_h(i, j) = values[h * plane + block_offsets[b] +
 * i * round_up(Lk_b, 8) + j], i.e. one Lq_b x Lk_b matrix per sequence and head, stored
 * row-major with each row padded to a multiple of 8 elements (the padding is never
 * read), the blocks of one head packed into a plane of `plane` elements.  `values` is a
 * device bf16 array [H][plane], 16-byte aligned; `block_offsets` a device int64 array
 * [B+1] with block_offsets[0] = 0 and block_offsets[b+1] - block_offsets[b] =
 * Lq_b * round_up(Lk_b, 8), block_offsets[B] = plane -- checked on the device (a mismatch
 * is JFA_ERR_BAD_OFFSETS and no attention is computed).  Added after scaling, like kind 1.
 * `grad` must be NULL for kind 2; its gradient goes to `values_grad` instead (jfa_backward
 * only; NULL = not wanted): a device bf16 array with the layout of `values`, 16-byte
 * aligned, not overlapping any other argument, overwritten with dS_ij = P_ij (dP_ij - D_i)
 * at each block element (0 for pairs the causal mask hides and for the row padding). */
typedef struct {
  int kind;
  const float* table;
  int num_buckets;
  int center;
  float* grad;
  const void* values;            /* kind 2 */
  const int64_t* block_offsets;  /* kind 2 */
  int64_t plane;                 /* kind 2 */
  void* values_grad;             /* kind 2, jfa_backward */
} jfa_bias;

/* Bytes of workspace jfa_forward (is_backward = 0) or jfa_backward (is_backward = 1)
 * needs for these sizes.  Returns 0 on invalid sizes. */
size_t jfa_workspace_size(int B, int H, int d, int64_t total_q, int64_t total_kv, int is_backward);

/* Forward.  Writes out (bf16 [total_q, H, d]) and lse (fp32 [H, total_q], natural
 * log of the row's sum of exp(s_ij)).  bias may be NULL. */
jfa_status jfa_forward(const void* q, const void* k, const void* v, const int64_t* q_offsets,
                       const int64_t* kv_offsets, int B, int H, int d, int64_t total_q, int64_t total_kv,
                       const jfa_bias* bias, float scale, int causal, void* out, float* lse, void* workspace,
                       size_t workspace_bytes, jfa_stream_t stream);

/* Backward of sum(dout * out) w.r.t. q, k, v (the backward pass listed among JFA's
 * features, "Jagged Flash Attention (JFA)", Definition; split scheme of "Four generations"
 * item 2: dK/dV computed per key/value block, dQ in a separate pass that owns each
 * dQ tile, no atomics).  out and lse must be the forward's results for the same
 * inputs.  dq, dk, dv are bf16 with the shapes of q, k, v and are fully overwritten
 * (rows of keys no query sees get 0).  With a relative-position bias whose `grad` is
 * non-NULL, the table's gradient is written there too (see jfa_bias). */
jfa_status jfa_backward(const void* dout, const void* q, const void* k, const void* v, const void* out,
                        const float* lse, const int64_t* q_offsets, const int64_t* kv_offsets, int B, int H,
                        int d, int64_t total_q, int64_t total_kv, const jfa_bias* bias, float scale,
                        int causal, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                        jfa_stream_t stream);

/* Forward without a workspace, for callers that cannot allocate device memory.  The
 * pages have no counterpart to this entry point.  Hosts such as inference-runtime
 * plugins and services on a fixed, pre-planned memory arena give a kernel library
 * only its inputs and outputs and must not call cudaMalloc on their hot path (it can
 * synchronise the device and breaks the arena's budget); this call runs jfa_forward
 * with its scratch in a file-scope device array of 8 MiB that every GPU loading the
 * library holds until exit.  Arguments and results are those of jfa_forward.
 * - Sizes whose workspace (jfa_workspace_size(..., 0)) exceeds 8 MiB are rejected with
 *   JFA_ERR_WORKSPACE before anything is enqueued.
 * - The first call on a device looks up the array's device address (cudaGetSymbolAddress)
 *   with that device current; make that first call before any stream capture.
 * - Allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 * - Every call on a device shares the one array: calls whose work overlaps on the GPU
 *   (e.g. on two streams) race and must be serialised by the caller.  Each call
 *   rewrites all of the scratch it reads, so no clearing is needed between calls.
 * - Device-detected errors (bad offsets, wait timeout) land in the shared array and are
 *   not reported to the caller; use jfa_forward with a workspace to read them. */
jfa_status jfa_forward_noalloc(const void* q, const void* k, const void* v, const int64_t* q_offsets,
                               const int64_t* kv_offsets, int B, int H, int d, int64_t total_q, int64_t total_kv,
                               const jfa_bias* bias, float scale, int causal, void* out, float* lse,
                               jfa_stream_t stream);

/* Synchronises `stream`, then returns the first device-side error recorded in
 * `workspace` since the previous jfa_check_status (JFA_OK if none; else
 * JFA_ERR_BAD_OFFSETS, JFA_ERR_TIMEOUT or JFA_ERR_WORKSPACE) and clears it. */
jfa_status jfa_check_status(void* workspace, jfa_stream_t stream);

/* Static, NUL-terminated description of a status code. */
const char* jfa_status_string(jfa_status s);

/* Number of kernels the last successful jfa_forward / jfa_backward call on this
 * thread enqueued (for launch accounting). */
int jfa_last_launch_count(void);

/* Description of the last failed CUDA runtime/driver call made by this library on the
 * calling thread (the cause behind a JFA_ERR_CUDA); "" if none.  Thread-local, static. */
const char* jfa_last_error(void);

/* Kernel kinds for per-kernel timing. */
enum { JFA_KERNEL_PLAN = 0, JFA_KERNEL_FORWARD = 1, JFA_KERNEL_BWD_PREPROCESS = 2, JFA_KERNEL_BWD_DKDV = 3,
       JFA_KERNEL_BWD_DQ = 4, JFA_KERNEL_BWD_FUSED = 5, JFA_KERNEL_BWD_NSP = 6, JFA_NUM_KERNEL_KINDS = 7 };

/* Benchmark support (not part of the attention itself).  While enabled (process-wide),
 * every kernel launch is bracketed by two CUDA events recorded on the launch stream.
 * jfa_timing_read waits for the recorded events, adds each kernel's elapsed time (ms)
 * to ms[kind] and its launch count to launches[kind] for kind < n_kinds, then drops
 * the records.  Both return JFA_ERR_CUDA if an event call fails. */
jfa_status jfa_timing_enable(int on);
jfa_status jfa_timing_read(double* ms, int* launches, int n_kinds);

/* Failure-detection self test (not part of the attention itself).  Enqueues one tiny
 * kernel whose single thread waits on a pipeline barrier that nothing ever signals,
 * through the bounded wait every kernel of this library uses; after `timeout_ns`
 * (1 ns .. 2 s) the wait gives up and JFA_ERR_TIMEOUT is recorded in the workspace
 * status word, readable with jfa_check_status.  Nothing faults or hangs; the context
 * stays usable.  `workspace` needs 256 bytes (zeroed status word). */
jfa_status jfa_selftest_wait_timeout(void* workspace, uint64_t timeout_ns, jfa_stream_t stream);

/* Which backward pass takes a sequence of two or more query tiles (128 rows each), for
 * every later jfa_backward call in the process.  Sequences of 2 .. max_tiles query tiles
 * take the non-sequence-parallel pass -- one CTA owns a (sequence, head), forms every tile
 * pair's S, P, dP and dS once and computes dK, dV and dQ from them (five GEMMs per tile
 * pair), summing dQ over key tiles in an fp32 buffer in the workspace with one writer per
 * row ("Jagged Flash Attention (JFA)", "Four generations" item 2, the reading in which
 * the backward is not parallel over a sequence's query tiles); longer sequences take the
 * split passes (dK/dV per key tile, then dQ per query tile: seven GEMMs per tile pair, no
 * sum buffer).  max_tiles in 0 .. 16; below 2 every such sequence takes the split passes
 * (the default, which measured faster on GB300) and jfa_backward launches five kernels, not
 * the pass's sixth.  Both paths give the same results within
 * rounding and are each deterministic.  With max_tiles >= 2 the backward workspace also
 * holds the fp32 dQ sums (4 * total_q * H * d more bytes): jfa_workspace_size reflects the
 * setting at the time it is called, and a workspace sized before the pass was enabled is
 * rejected with JFA_ERR_WORKSPACE.  A negative max_tiles only reads the setting.
 * Returns the previous setting, or -1 (nothing changed) for max_tiles > 16. */
int jfa_set_nsp_max_tiles(int max_tiles);

/* The item hand-off wait limit, in ns, that the kernels use for a launch whose planner
 * found `planned_tile_pairs` 128x128 (query tile, key tile) pairs over all heads, to be
 * shared by `ctas` persistent CTAs, the costliest single work item being
 * `max_item_tile_pairs` pairs (not part of the attention itself; exported so the rule can
 * be checked without a GPU).  A CTA's scheduler waits for its previous items to finish
 * before it claims the next, and its roles wait for the next item to be claimed: such a
 * wait lasting longer ends the CTA with JFA_ERR_TIMEOUT.  The limit is 2 s plus 32 us for
 * each pair of one CTA's share (rounded up) and of the costliest item, capped at 2 s + 1 h;
 * negative arguments count as 0, `ctas` < 1 as 1.  32 us is about 30 times the time one SM
 * takes for a pair, so no hand-off of a correct launch comes near it, whatever the
 * launch's size.  (Waits inside an item's tile pipeline last at most a few tiles' time and
 * keep a fixed 2 s limit.) */
uint64_t jfa_wait_limit_ns(int64_t planned_tile_pairs, int ctas, int64_t max_item_tile_pairs);

/* Developer tracing (not part of the attention itself).  With a non-NULL device buffer,
 * kernels of `kernel_kind` (JFA_KERNEL_*) launched afterwards record the pipeline events
 * of their first CTA: uint64 entries (SM clock << 16 | role << 8 | event id) in five
 * regions of bytes/40 entries, one per warp role (0 streaming TMA producer, 1 MMA issuer,
 * 2 and 3 the two compute warpgroups, 4 resident-tile loader); each launch overwrites
 * them; unused entries are left as they were.  A NULL buffer or a kind outside [0, JFA_NUM_KERNEL_KINDS) turns tracing off.
 * Process-wide; returns JFA_ERR_INVALID_ARG for a buffer too small or not 8-byte aligned. */
jfa_status jfa_trace_configure(void* device_buffer, size_t bytes, int kernel_kind);

#ifdef __cplusplus
}
#endif
#endif /* JFA_H_ */
