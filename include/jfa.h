/*
 * jfa.h - C ABI of the GB300 (sm_103a) jagged flash attention library.
 *
 * Exact softmax attention, forward and backward, over packed, padding-free
 * bf16 Q/K/V whose sequence boundaries are given by an int32 offsets array
 * ("Optimizing Jagged Flash Attention with TLX", pytorch.org, Introduction:
 * sequences are packed contiguously and their boundaries recorded in an
 * offsets tensor; the attention never materialises padded tokens).  The
 * broadcast-Q mode, where one dense Q is shared by every sequence and dQ is
 * summed over the batch, follows section 1 of the same page ("The
 * Challenge", broadcast_q=True).  The per-row math is the softmax attention
 * of "cuTile Kernels - FMHA Implementation" (build.nvidia.com), "Attention
 * Basics" and "Flash Attention Algorithm".
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor pointers are DEVICE pointers on the current CUDA device, row
 *   major and contiguous, 16-byte aligned.  q, k, v, out, dout, dq, dk, dv
 *   hold bf16 (IEEE bfloat16); lse holds fp32; offsets holds int32.
 * - offsets: device int32[B+1], offsets[0] = 0, non-decreasing; sequence b
 *   owns packed rows [offsets[b], offsets[b+1]) of k and v (and of q in
 *   self-attention).  T = offsets[B].  Every length must be <= max_len.
 *   The host never reads offsets; a violation found on the device sets the
 *   device error word (see jfa_sync_and_check) and no output is written.
 * - Self-attention layouts: q, k, v, out, dout, dq, dk, dv are [T, H, D];
 *   lse is [H, T].
 * - Broadcast-Q layouts: q and dq are [q_len, H, D]; k, v, dk, dv are
 *   [T, H, D]; out and dout are [B, q_len, H, D]; lse is [B, H, q_len].
 * - lse is the natural-log log-sum-exp of the scaled scores of each query
 *   row.  A broadcast sequence of length 0 gives out = 0 and lse = -inf and
 *   adds nothing to dq.
 * - causal (self-attention only): query i attends to key j iff j <= i, both
 *   counted from the start of their own sequence.
 * - scale: positive finite softmax scale (normally 1/sqrt(D)).
 * - D must be 64 or 128; 1 <= H <= 32767.
 * - Inputs must be finite.  Rows of neighbouring sequences are read into a
 *   tile's padding and then multiplied by an exact zero, so a non-finite
 *   value in one sequence can leak into its neighbours.
 * - Ownership: the caller owns every buffer.  The library keeps no pointer
 *   after the call returns.  Scratch memory is taken stream-ordered from a
 *   library-owned CUDA memory pool (cudaMallocAsync / cudaFreeAsync on
 *   `stream`), so calls are asynchronous and capturable in a CUDA graph.
 * - Errors: a non-OK status means nothing was enqueued; jfa_last_error()
 *   gives the reason (thread-local).  Errors found by the device (bad
 *   offsets, a bounded wait that ran out) are reported by
 *   jfa_sync_and_check().  With the environment variable JFA_VALIDATE=1
 *   every call synchronises and checks before returning.
 * - Thread safety: calls on different streams may run concurrently, except
 *   jfa_fwd_bq_noalloc, whose calls all share one scratch array (see there).
 * - With the environment variable JFA_KV_PAIR=1 (read on every call) the
 *   backward runs its dK/dV pass on CTA pairs ("Optimizing Jagged Flash
 *   Attention with TLX", "2-CTA collaborative MMA (backward)": clusters of
 *   two CTAs whose cta_group::2 products cover two adjacent key blocks)
 *   where that variant exists (D = 128, no causal mask or window; for
 *   broadcast-Q, the two-pass backward).  Results are bit-identical to the
 *   default single-CTA pass.
 */
#ifndef JFA_H_
#define JFA_H_

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  JFA_OK = 0,
  JFA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size or offsets */
  JFA_ERR_UNSUPPORTED = 2, /* D not in {64,128}; causal or a window with broadcast_q */
  JFA_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
  JFA_ERR_TIMEOUT = 4,     /* a device-side bounded wait ran out */
  JFA_ERR_WORKSPACE = 5    /* scratch allocation failed */
} jfa_status;

/* Forward pass, self-attention (broadcast_q must be 0; use jfa_fwd_bq for
 * broadcast-Q, which needs the dense Q length).  Writes out and lse.
 * Follows "Optimizing Jagged Flash Attention with TLX", section 2.1
 * (persistent, warp-specialised forward) and "cuTile Kernels - FMHA
 * Implementation", "Flash Attention Algorithm" (online softmax). */
jfa_status jfa_fwd(const void* q, const void* k, const void* v, const int32_t* offsets, int B,
                   int H, int D, int max_len, int broadcast_q, int causal, float scale, void* out,
                   float* lse, cudaStream_t stream);

/* Backward pass, self-attention: given out, lse from jfa_fwd and dout,
 * writes dq, dk, dv (gradients of sum(out * dout)).  The products of
 * "Optimizing Jagged Flash Attention with TLX", section "2-CTA
 * collaborative MMA", after a pre-pass (the two work lists and the row
 * statistics LSE*log2(e) and Delta = rowsum(dout * out)), in two passes: a
 * K/V-block-outer pass for dk and dv and a query-tile-outer pass for dq, so
 * that dq accumulates on chip and needs no global fp32 accumulator (the
 * page's "Multi-stage dQ staging" is not needed).  Three kernels: the
 * pre-pass and the two passes. */
jfa_status jfa_bwd(const void* q, const void* k, const void* v, const int32_t* offsets, int B,
                   int H, int D, int max_len, int broadcast_q, int causal, float scale,
                   const void* out, const float* lse, const void* dout, void* dq, void* dk,
                   void* dv, cudaStream_t stream);

/* Same as jfa_fwd / jfa_bwd with the dense Q length `q_len` (>= 1) added.
 * Required when broadcast_q = 1 (q_len is then the row count of q); with
 * broadcast_q = 0 q_len is ignored.  Broadcast-Q: section 1 of "Optimizing
 * Jagged Flash Attention with TLX"; dq is summed over all B sequences. */
jfa_status jfa_fwd_bq(const void* q, const void* k, const void* v, const int32_t* offsets, int B,
                      int H, int D, int max_len, int q_len, int broadcast_q, int causal,
                      float scale, void* out, float* lse, cudaStream_t stream);
jfa_status jfa_bwd_bq(const void* q, const void* k, const void* v, const int32_t* offsets, int B,
                      int H, int D, int max_len, int q_len, int broadcast_q, int causal,
                      float scale, const void* out, const float* lse, const void* dout, void* dq,
                      void* dk, void* dv, cudaStream_t stream);

/* The attention variants that "Optimizing Jagged Flash Attention with TLX"
 * (sections 3 and 4) names as supported by its kernels without defining
 * them: GQA and sliding windows.  Same arguments as jfa_fwd_bq / jfa_bwd_bq
 * plus:
 * - H_kv: heads of k, v, dk, dv (H_kv divides H).  Layouts as above with
 *   H_kv in place of H for k, v, dk, dv ([T, H_kv, D]); q, dq, out, dout and
 *   lse keep H query heads.  Query head h reads K/V head h / (H / H_kv), so
 *   consecutive query heads share one K/V head; dk and dv of a K/V head sum
 *   over its H / H_kv query heads.  H_kv = H is multi-head attention.
 * - window_left, window_right: query i attends to key j iff
 *   i - window_left <= j <= i + window_right, positions counted from the
 *   start of their sequence; -1 leaves that side unbounded (both -1: no
 *   window).  causal = 1 is window_right = 0 (a window_right > 0 with causal
 *   is JFA_ERR_INVALID_ARG).  Windows are self-attention only
 *   (JFA_ERR_UNSUPPORTED with broadcast_q).  Every query row keeps at least
 *   its own key.
 * Key tiles outside a query tile's band are skipped (not loaded, no
 * products), so the work follows the band's area.  Errors and ownership as
 * for the other entry points. */
jfa_status jfa_fwd_ex(const void* q, const void* k, const void* v, const int32_t* offsets, int B,
                      int H, int H_kv, int D, int max_len, int q_len, int broadcast_q, int causal,
                      int window_left, int window_right, float scale, void* out, float* lse,
                      cudaStream_t stream);
jfa_status jfa_bwd_ex(const void* q, const void* k, const void* v, const int32_t* offsets, int B,
                      int H, int H_kv, int D, int max_len, int q_len, int broadcast_q, int causal,
                      int window_left, int window_right, float scale, const void* out,
                      const float* lse, const void* dout, void* dq, void* dk, void* dv,
                      cudaStream_t stream);

/* Block-sparse attention ("Optimizing Jagged Flash Attention with TLX",
 * section 3, "Block-sparse attention"): a cheap scoring step average-pools
 * each Q block and each K block and keeps the top-k K/V blocks per Q block;
 * the attention then runs over the selected blocks only.  GQA as for
 * jfa_fwd_ex; self-attention, or broadcast-Q (broadcast_q = 1, q_len as for
 * jfa_fwd_bq, layouts of broadcast-Q).  The pages keep windowing in the
 * sparse variant: the _ex forms take a causal mask and a sliding window as
 * jfa_fwd_ex does (self-attention only).
 *
 * Blocks: K block j of a sequence = its keys [128 j, 128 j + 128), Q block i
 * = its query rows [256 i, 256 i + 256) (broadcast: rows of the dense Q,
 * the same blocks for every sequence; the last ones ragged).  With
 * nqb = ceil(max_len / 256) (broadcast: ceil(q_len / 256)) and
 * kcap = ceil(max_len / 128):
 * - blocks: device int32 [B, H, nqb, kcap]; entry (b, h, i) lists the K
 *   blocks that query head h of Q block i of sequence b attends to, strictly
 *   ascending, in its first counts[b, h, i] slots;
 * - counts: device int32 [B, H, nqb]; 0 for Q blocks past the sequence and,
 *   in broadcast mode, for sequences without keys.
 *
 * jfa_block_select (stage 1) fills blocks and counts: the score of K block j
 * for Q block i is the dot product (fp32) of the mean of the Q block's rows
 * (query head h) with the mean of the K block's rows (K/V head h / (H /
 * H_kv)); the k = max(1, ceil(permille * n / 1000)) highest scores of the
 * sequence's n K blocks are kept (1 <= permille <= 1000), ties to the lower
 * index; slots after the count are set to -1.  Two kernels that read K and
 * Q once each; scratch: B * H_kv * kcap * D floats from the pool.  max_len
 * must be <= 262144 (kcap <= 2048) and B <= 65535.
 *
 * jfa_fwd_sparse (stage 2) writes out and lse like jfa_fwd / jfa_fwd_bq, with
 * query row r attending only to the keys of the K blocks listed for its Q
 * block r / 256; a row whose list is empty gets out = 0 and lse = -inf.  The
 * lists may come from jfa_block_select or from the caller; they are checked
 * on the device (a count above the sequence's K blocks, or entries not
 * strictly ascending below it, sets the device error word, reported by
 * jfa_sync_and_check as JFA_ERR_INVALID_ARG, and nothing is written).  The
 * forward kernel is the dense one following each item's list instead of all
 * key tiles, so its time scales with the selected fraction.
 *
 * jfa_block_select_ex / jfa_fwd_sparse_ex add causal, window_left and
 * window_right, with the meaning and checks of jfa_fwd_ex; the plain forms
 * are these with causal = 0 and window_left = window_right = -1.  With a
 * local mask (admissible keys [i - wl, i + wr] for row i), the candidates
 * of Q block i are the K blocks that hold an admissible key of one of its
 * rows, and k counts from those candidates instead of all n; the forward
 * keeps a key only when it is both in a listed block and admissible, so a
 * row whose band misses every listed block gets out = 0 and lse = -inf. */
jfa_status jfa_block_select(const void* q, const void* k, const int32_t* offsets, int B, int H,
                            int H_kv, int D, int max_len, int q_len, int broadcast_q,
                            int permille, int32_t* blocks, int32_t* counts, cudaStream_t stream);
jfa_status jfa_fwd_sparse(const void* q, const void* k, const void* v, const int32_t* offsets,
                          int B, int H, int H_kv, int D, int max_len, int q_len, int broadcast_q,
                          float scale, const int32_t* blocks, const int32_t* counts, void* out,
                          float* lse, cudaStream_t stream);
jfa_status jfa_block_select_ex(const void* q, const void* k, const int32_t* offsets, int B, int H,
                               int H_kv, int D, int max_len, int q_len, int broadcast_q,
                               int causal, int window_left, int window_right, int permille,
                               int32_t* blocks, int32_t* counts, cudaStream_t stream);
jfa_status jfa_fwd_sparse_ex(const void* q, const void* k, const void* v, const int32_t* offsets,
                             int B, int H, int H_kv, int D, int max_len, int q_len,
                             int broadcast_q, int causal, int window_left, int window_right,
                             float scale, const int32_t* blocks, const int32_t* counts, void* out,
                             float* lse, cudaStream_t stream);

/* Allocation-free forward pass.  The pages have no counterpart: this entry
 * point exists for callers that must not allocate device memory while the
 * library runs (memory owned and pre-partitioned by a host framework, for
 * example an inference server or plugin host that forbids allocation during
 * execution, or a real-time loop that cannot risk an out-of-memory failure).
 * Same arguments and results as jfa_fwd_bq (broadcast_q = 0 gives
 * self-attention and ignores q_len).  It calls no cudaMalloc, cudaFree or
 * allocating routine: its scratch lives in one 1 MiB device array inside the
 * library, which every GPU that loads the library keeps until the process
 * exits.  Limit: H * B * ceil(L / 256) <= 131040 work items, with L = max_len
 * (self-attention) or q_len (broadcast); larger problems return
 * JFA_ERR_WORKSPACE with nothing enqueued.  The first call on each device
 * looks up the device addresses it needs (no allocation); make that first
 * call before capturing a stream into a CUDA graph.  All calls share the one
 * array, so calls whose GPU work overlaps (different streams, or different
 * host threads) race and give wrong results: serialise them.  Device-side
 * errors set the same device error word that jfa_sync_and_check reads; with
 * JFA_VALIDATE=1 this call, like the others, synchronises and checks that
 * word before returning (still without allocating). */
jfa_status jfa_fwd_bq_noalloc(const void* q, const void* k, const void* v, const int32_t* offsets,
                              int B, int H, int D, int max_len, int q_len, int broadcast_q,
                              int causal, float scale, void* out, float* lse,
                              cudaStream_t stream);

/* Synchronise `stream`, then read and clear the device error word of the
 * current device.  Returns JFA_ERR_INVALID_ARG for offsets found invalid on
 * the device, JFA_ERR_TIMEOUT for a bounded wait that ran out,
 * JFA_ERR_CUDA if the stream reported an error, JFA_OK otherwise. */
jfa_status jfa_sync_and_check(cudaStream_t stream);

/* Message for the last non-OK status returned on this thread ("" if none). */
const char* jfa_last_error(void);

/* Library version string. */
const char* jfa_version(void);

/* ------------------------------------------------------------------------
 * Work-list inspection.  A library facility with no counterpart in the
 * pages (whose tile scheduling, "Optimizing Jagged Flash Attention with
 * TLX", section 2.2 "Scheduling jagged tiles across SMs", sorts work
 * longest-first on the host): it builds one of the device work lists
 * exactly as the named pass does and copies it out, so that a caller can
 * check it.  list: 0 forward (items (b, h, pair of 128-row query tiles),
 * longest sequences first), 1 dK/dV pass ((b, h, 128-key block), most query
 * tiles first), 2 self-attention dQ pass ((b, h, pair), longest first), 3
 * broadcast-Q dQ pass (equal chunks of the key-tile stream).  offsets as for
 * jfa_fwd (device int32[B+1]); q_len as for jfa_fwd_bq.  items: DEVICE
 * int32 buffer of 4 * capacity ints, 16-byte aligned, written with 4 ints
 * per item in list order: lists 0-2 {b, h, tile, 0}; list 3 {h | pair << 16,
 * b, j, n}: n key tiles from tile j of sequence b on, through the following
 * non-empty sequences.  count: DEVICE int32[2]: {number of items (-1 if the
 * device found the offsets invalid), chunks per (head, pair) for list 3 else
 * 0}.  JFA_ERR_INVALID_ARG if capacity is below the list's size bound (the
 * message names it).  Asynchronous on `stream`; scratch as for jfa_fwd.
 * ------------------------------------------------------------------------ */
jfa_status jfa_worklist(const int32_t* offsets, int B, int H, int max_len, int q_len,
                        int broadcast_q, int causal, int list, int32_t* items, int capacity,
                        int32_t* count, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Launch accounting.  A library facility with no counterpart in the pages:
 * it lets a caller count the kernels this library enqueues and time each
 * kind on the stream it runs on.
 * ------------------------------------------------------------------------ */

/* Kernel kinds reported by jfa_profile_read (array index). */
typedef enum {
  JFA_KERNEL_SCHED = 0,     /* forward work-list scheduler */
  JFA_KERNEL_FWD = 1,       /* forward */
  JFA_KERNEL_PREP = 2,      /* backward pre-pass: work lists, LSE*log2e, Delta */
  JFA_KERNEL_BWD_KV = 3,    /* backward dK / dV pass (self-attention and broadcast-Q) */
  JFA_KERNEL_BWD_Q = 4,     /* self-attention backward, dQ pass */
  JFA_KERNEL_BWD_Q_BCAST = 5, /* broadcast-Q backward, dQ pass (per-chunk partials) */
  JFA_KERNEL_FINALIZE = 6,  /* broadcast-Q dQ: sum of the partials, bf16 cast */
  JFA_KERNEL_FILL = 7,      /* outputs of an all-empty broadcast batch */
  JFA_KERNEL_BWD_BCAST_ONEPASS = 8, /* broadcast-Q backward, one pass (D = 64, q_len <= 128) */
  JFA_KERNEL_FWD_COMBINE = 9, /* broadcast-Q forward (q_len <= 128): merge of split sequences */
  JFA_KERNEL_SPARSE_POOL = 10,   /* block-sparse selection: K-block and Q-block means */
  JFA_KERNEL_SPARSE_SELECT = 11, /* block-sparse selection: scores, top-k */
  JFA_KERNEL_BWD_KV_PAIR = 12,   /* backward dK / dV pass on pairs of CTAs (JFA_KV_PAIR=1) */
  JFA_KERNEL_SPARSE_CHECK = 13,  /* block-sparse forward: check of every block list */
  JFA_KERNEL_KINDS = 14
} jfa_kernel_kind;

/* Kernels enqueued by this library since the process started (all threads,
 * devices and streams; a failed launch is not counted).  Never fails. */
long long jfa_launch_count(void);

/* on != 0: every later launch is bracketed by a CUDA event pair recorded on
 * its own stream, until profiling is switched off.  Process-wide.  Do not
 * enable while a stream of this library is being captured into a graph.
 * Always returns JFA_OK. */
jfa_status jfa_profile_enable(int on);

/* Kernel kinds that profiling brackets: bit k of `kinds` selects kind k
 * (1u << JFA_KERNEL_BWD_KV: the dK/dV pass alone); other launches are
 * counted by jfa_launch_count but get no events.  Default: every kind
 * (~0u).  Process-wide; read at each launch.  Always returns JFA_OK. */
jfa_status jfa_profile_select(unsigned int kinds);

/* Waits for every event pair recorded so far, writes per kernel kind the
 * summed device time in milliseconds (ms[kind]) and the number of launches
 * (launches[kind]) for kinds < n, and releases the records.  ms and
 * launches are HOST arrays of n elements owned by the caller (n >= 0; both
 * may be null when n == 0).  JFA_ERR_CUDA if an event could not be read
 * (the remaining records are still released). */
jfa_status jfa_profile_read(double* ms, long long* launches, int n);

#ifdef __cplusplus
}
#endif

#endif /* JFA_H_ */
