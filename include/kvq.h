/*
 * kvq -- attention over a group-wise affine-quantized KV cache, for one
 * NVIDIA GB300 GPU (sm_103a).  C ABI of libkvq.so.
 *
 * The operations are those of one attention layer of the Gemma 4 serving
 * graph shown on the pages of the @mlx-bun/inference package:
 *   - model.ts, "Parity notes" header: SDPA scale 1.0 (q and k are
 *     normalized instead); full-attention layers use K = V (one projection,
 *     v gets an un-scaled RMS norm); proportional RoPE rotates only
 *     partial_rotary_factor * head_dim dims.
 *   - model.ts, attentionTraining: q/k/v reshaped per head, qNorm / kNorm /
 *     vNorm, RoPE at the cache offset, cache.appendWindow(k, v), then
 *     read.attend(q, 1.0).
 *   - gemma4-e4b.ts, Gemma4Layer / LAYERS: each cache is affine quantized
 *     with {bits: 4 | 8, groupSize: 64}; KV-shared layers attend the cache of
 *     the last donor of their type without appending.
 *
 * Conventions for every call
 *   - All tensor pointers are DEVICE pointers owned by the caller; the
 *     library allocates no memory and keeps no reference after the call
 *     returns (attn_mixed creates its streams and events once per device).
 *     `kvq_layer` is read on the host during the call.
 *   - Alignment: k_raw, v_raw and q_raw 16 bytes (read with 128-bit loads);
 *     the workspace 256 bytes; the kvq_seq_cache array 8 bytes; every other
 *     pointer its element size.  The six arrays a kvq_seq_cache points to are
 *     16-byte aligned (copied with the tensor memory accelerator).
 *   - bf16 values are passed as their 16-bit patterns (uint16_t).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and runs asynchronously; no call synchronizes the device.
 *   - A call with no rows (n_rows == 0) enqueues nothing; its workspace,
 *     status word included, is left as it was.
 *   - Arguments are checked on the host first; a bad argument returns a
 *     status other than KVQ_OK and enqueues nothing.  kvq_last_error()
 *     returns a message for the calling thread's last failure.
 *   - Per-sequence fields that live in device memory (kvq_seq_cache) are
 *     checked by the kernels.  A sequence whose cache descriptor is invalid
 *     (bits not 4/8, capacity not a positive multiple of 64, a misaligned
 *     pointer, or a capacity too small for the window) is skipped: nothing of
 *     it is written by kv_quant_append, and its attention outputs are NaN.
 *
 * Cache layout (per sequence of one layer)
 *   k_codes, v_codes  uint32 [n_kv_heads][capacity][head_dim*bits/32]
 *       element e of a row lives in word e*bits/32 at bit (e*bits) % 32,
 *       element 0 in the low bits (little-endian packing).
 *   k_scales, k_biases, v_scales, v_biases  bf16 [n_kv_heads][capacity][head_dim/64]
 *   Position p is stored in slot p % capacity: a full-attention cache uses a
 *   capacity above its largest position (linear), a sliding-window cache a
 *   ring of at least `window` slots (window + rows_per_call - 1 for prompt
 *   chunks).
 *
 * Quantization of one 64-element group of a prepped bf16 row (IEEE fp32):
 *   scale = bf16_rne((max - min) / (2^bits - 1));  bias = min;
 *   code  = clamp(rint_half_even((x - bias) / scale), 0, 2^bits - 1),
 *   all codes 0 when scale == 0.  The pages name the affine {bits, groupSize}
 *   scheme and its (codes, scales, biases) triple but print no formula; this
 *   is the plain min/max affine reading.
 */
#ifndef KVQ_H_
#define KVQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KVQ_OK = 0,
  KVQ_EINVAL = 1,        /* bad argument (null/misaligned pointer, size out of range) */
  KVQ_EUNSUPPORTED = 2,  /* shape this build does not implement (head_dim, group, ratio) */
  KVQ_ECUDA = 3,         /* a CUDA launch failed; kvq_last_error() has the CUDA message */
  KVQ_EWORKSPACE = 4     /* workspace smaller than the matching *_workspace_bytes() */
} kvq_status;

/* Bits of the device status word an attention call leaves in the first 4
 * bytes of its workspace (attn_decode_static: read with kvq_static_status).
 * Errors found while the kernels run cannot be returned by the (asynchronous)
 * call itself; the kernels record them here instead and finish. */
#define KVQ_STATUS_WAIT_TIMEOUT 0x2u  /* a bounded wait on a copy gave up (outputs of that work are not valid) */
#define KVQ_STATUS_SEQ_SKIPPED 0x4u   /* a sequence with an invalid descriptor was skipped (its outputs are NaN) */

/* One sequence's cache of one layer.  An array of these lives in DEVICE
 * memory (kernels read the pointers from it). */
typedef struct {
  uint32_t* k_codes;
  uint32_t* v_codes;
  uint16_t* k_scales;
  uint16_t* k_biases;
  uint16_t* v_scales;
  uint16_t* v_biases;
  int32_t bits;        /* 4 or 8; may differ between sequences */
  int32_t capacity;    /* slots, a positive multiple of 64 */
} kvq_seq_cache;

/* One attention layer (host memory). */
typedef struct {
  int32_t n_q_heads;   /* q heads; a multiple of n_kv_heads, at most 16 per kv head */
  int32_t n_kv_heads;  /* kv heads; q head h reads kv head h / (n_q_heads / n_kv_heads) */
  int32_t head_dim;    /* 64, 128, 256 or 512 */
  int32_t group_size;  /* must be 64 */
  int32_t window;      /* 0 = full causal; W > 0: a query at p sees keys p-W+1 .. p */
  int32_t rope_dims;   /* even, 0..head_dim: dims 0..rope_dims-1 are rotated in pairs
                          (j, j + rope_dims/2) at angle pos * rope_theta^(-2j/head_dim) */
  double rope_theta;   /* > 0 */
  float rms_eps;       /* >= 0; RMSNorm: x / sqrt(mean(x^2) + eps) * w */
  int32_t k_eq_v;      /* 1: V is the un-scaled RMS norm of the raw k rows (no v input) */
  /* NULL, or DEVICE int8[head_dim] of +1 / -1: the deferred TurboQuant read
   * (model.ts, cacheLayers comment: full-attention caches keep their values
   * rotated through the attention and the read un-rotates the output).  The
   * rotation R = diag(rot_signs) H, H the Sylvester Hadamard matrix of order
   * head_dim (entries +-1, H H^T = head_dim I), is taken from outside the
   * pages (the randomized Hadamard transform).  kv_quant_append stores
   * bf16(k_hat R) and bf16(v_hat R); the attention calls rotate q alike
   * (bf16(q_hat R)), score (q R)(k R)^T / head_dim and return O' R^T / head_dim
   * for the output O' over the rotated values.  kv_prepped and q_prepped
   * receive the rotated rows.  The same signs must be given to the append and
   * the attention calls of a cache.  q_hat R is at most head_dim |w| in size:
   * norm weights |w| <= 64 keep the f16 operands finite. */
  const int8_t* rot_signs;
} kvq_layer;

/*
 * kv_quant_append -- prep and quantize-append new K/V rows (the cache's
 * appendWindow in model.ts attentionTraining).
 *
 * For each new row t of sequence s at position p = start_pos[s] + (t - row_offsets[s]):
 *   k_hat = RoPE_p(bf16(RMSNorm(k_raw[t], k_norm_w)))       (rounded to bf16 after each)
 *   v_hat = bf16(RMSNorm(v_raw[t] or k_raw[t] if k_eq_v, no weight))
 * then each is quantized per 64-group and written at slot p % capacity of
 * every kv head.  When a sequence appends more rows than its capacity, only
 * the newest `capacity` rows are written (older ones would be overwritten).
 *
 *   seqs          device kvq_seq_cache[n_seqs]
 *   row_offsets   device int32[n_seqs + 1], non-decreasing, row_offsets[0] = 0,
 *                 row_offsets[n_seqs] = n_rows (rows of sequence s are
 *                 row_offsets[s] .. row_offsets[s+1]-1)
 *   start_pos     device int32[n_seqs], position of each sequence's first new row,
 *                 0 <= p < 2^24
 *   n_rows        host copy of row_offsets[n_seqs]
 *   k_raw         device bf16 [n_rows][n_kv_heads][head_dim]
 *   v_raw         device bf16 [n_rows][n_kv_heads][head_dim]; NULL iff k_eq_v
 *   k_norm_w      device bf16 [head_dim]; |w| <= 256 keeps the attention
 *                 calls' f16 operands (k biases) finite
 *   kv_prepped    NULL, or device bf16 [2][n_rows][n_kv_heads][head_dim] that
 *                 receives k_hat and v_hat (for inspection)
 */
kvq_status kv_quant_append(const kvq_layer* layer, const kvq_seq_cache* seqs, int32_t n_seqs,
                           const int32_t* row_offsets, const int32_t* start_pos, int32_t n_rows,
                           const uint16_t* k_raw, const uint16_t* v_raw, const uint16_t* k_norm_w,
                           uint16_t* kv_prepped, void* stream);

/*
 * attn_decode -- one query token per sequence attends its cache
 * (read.attend(q, 1.0) of model.ts attentionTraining in the decode phase).
 * Call it after kv_quant_append has stored the token's own K/V row (the new
 * row is read back quantized); a KV-shared layer calls it on its donor's
 * caches without appending.
 *
 * For sequence s with query position p = pos[s] and each q head h:
 *   q_hat = RoPE_p(bf16(RMSNorm(q_raw[s][h], q_norm_w)))
 *   out[s][h] = sum_j softmax_j(q_hat . k_hat_j) v_hat_j,  scale 1.0,
 * over keys j = max(0, p-window+1) .. p (0 .. p when window == 0), with
 * k_hat_j, v_hat_j dequantized (code * scale + bias) from the cache.
 *
 *   seqs        device kvq_seq_cache[n_seqs]
 *   pos         device int32[n_seqs], 0 <= pos < 2^24; the cache must hold
 *               every visible key (ring capacity >= window, linear capacity > pos)
 *   max_pos     host upper bound of pos[] (sizes the split over the cache length),
 *               0 <= max_pos < 2^24, else KVQ_EINVAL (and a workspace size of 0)
 *   q_raw       device bf16 [n_seqs][n_q_heads][head_dim]
 *   q_norm_w    device bf16 [head_dim]; q_hat and its per-group sums enter the
 *               MMAs as f16, finite for |w| <= 256 (|q_hat| <= sqrt(head_dim) |w|)
 *   out         device [n_seqs][n_q_heads][head_dim], fp32 if out_is_f32 else bf16
 *   q_prepped   NULL, or device bf16 [n_seqs][n_q_heads][head_dim] receiving q_hat
 *   workspace   device scratch of at least attn_decode_workspace_bytes(...) bytes;
 *               its first 4 bytes receive a device status word (0 = clean,
 *               else KVQ_STATUS_WAIT_TIMEOUT / KVQ_STATUS_SEQ_SKIPPED bits)
 */
kvq_status attn_decode(const kvq_layer* layer, const kvq_seq_cache* seqs, int32_t n_seqs,
                       const int32_t* pos, int32_t max_pos,
                       const uint16_t* q_raw, const uint16_t* q_norm_w,
                       void* out, int32_t out_is_f32, uint16_t* q_prepped,
                       void* workspace, size_t workspace_bytes, void* stream);

size_t attn_decode_workspace_bytes(const kvq_layer* layer, int32_t n_seqs, int32_t max_pos);

/*
 * attn_decode_append -- a donor layer's decode step in one call: each
 * sequence's new K/V row is prepped and quantize-appended at position pos[s]
 * (kv_quant_append with one row per sequence, row s of k_raw / v_raw being
 * sequence s's, start_pos = pos), then query row s attends its cache up to
 * and including that row (attn_decode).  model.ts attentionTraining in the
 * decode phase: cache.appendWindow(k, v), then read.attend(q, 1.0).
 *
 * The outputs are those of the two separate calls, bit for bit: the q prep
 * and the K/V append run side by side in the call's first kernel, and the
 * attention kernel copies the tile holding a sequence's new row only once
 * that kernel is complete.
 *
 *   k_raw, v_raw, k_norm_w, kv_prepped   as for kv_quant_append, with n_rows
 *                                        = n_seqs ([n_seqs][n_kv_heads][head_dim])
 *   kv_prepped                           NULL or device bf16 [2][n_seqs][n_kv_heads][head_dim]
 *   every other argument                 as for attn_decode; the workspace is
 *                                        attn_decode_workspace_bytes(layer, n_seqs, max_pos)
 * Arguments of both halves are checked before anything is enqueued.
 */
kvq_status attn_decode_append(const kvq_layer* layer, const kvq_seq_cache* seqs, int32_t n_seqs,
                              const int32_t* pos, int32_t max_pos,
                              const uint16_t* q_raw, const uint16_t* k_raw, const uint16_t* v_raw,
                              const uint16_t* q_norm_w, const uint16_t* k_norm_w,
                              void* out, int32_t out_is_f32, uint16_t* q_prepped, uint16_t* kv_prepped,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_prefill_chunk -- a chunk of new query rows per sequence attends the
 * cache after kv_quant_append stored the chunk's K/V rows (the "window" phase
 * of the pages: prompt chunks and verify windows).  Row t of sequence s sits
 * at position p = start_pos[s] + (t - row_offsets[s]) and sees keys
 * max(0, p-window+1) .. p (0 .. p when window == 0), including the rows of
 * its own chunk up to itself.  Verify windows (max_rows_per_seq <= 16) run
 * on the attn_decode kernels row by row.  Longer chunks with head_dim <= 256
 * and G dividing 128 run on the tcgen05 tensor cores, 128 (token, head) rows
 * per block.
 * Sliding-window layers: every key the chunk sees is dequantized once into
 * the workspace (k_hat as an f16 pair hi + lo, within ~2^-22 of k_hat; v_hat
 * rounded once to f16), then QK and PV on those.  Full-attention layers: QK
 * as on attn_decode (exact codes, fp32 per-group scale), PV on v_hat = scale
 * * code + bias rounded once to f16.  Other shapes (head_dim 512, a rotated
 * layer) use the attn_decode kernels row by row.
 *
 *   max_rows_per_seq must be >= the rows of every sequence (it sizes the grid).
 *
 *   row_offsets, start_pos, n_rows   as for kv_quant_append
 *   max_rows_per_seq                 host upper bound of rows per sequence
 *   q_raw                            device bf16 [n_rows][n_q_heads][head_dim]
 *   out                              device [n_rows][n_q_heads][head_dim]
 *   q_prepped                        NULL or device bf16 [n_rows][n_q_heads][head_dim]
 *   A ring cache needs capacity >= window + rows_of_the_sequence - 1.
 */
kvq_status attn_prefill_chunk(const kvq_layer* layer, const kvq_seq_cache* seqs, int32_t n_seqs,
                              const int32_t* row_offsets, const int32_t* start_pos, int32_t n_rows,
                              int32_t max_rows_per_seq,
                              const uint16_t* q_raw, const uint16_t* q_norm_w,
                              void* out, int32_t out_is_f32, uint16_t* q_prepped,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_prefill_append -- a prompt chunk's (or verify window's) K/V append and
 * its read in one call: kv_quant_append of the chunk rows (row_offsets,
 * start_pos, n_rows as given), then attn_prefill_chunk of the same rows, bit
 * for bit.  On the tensor-core paths the append runs in the grid of the
 * call's q prep (the two share nothing; on sliding-window layers the append
 * also writes the dequantized keys and values of the rows it stores into the
 * read's workspace scratch, and the key dequantization in the same grid
 * covers only the older keys), and the read follows; on the row
 * path (verify windows, head_dim 512, a rotated layer) the append comes
 * first.  k_raw / v_raw / k_norm_w / kv_prepped as for kv_quant_append
 * (kv_prepped: NULL or device bf16 [2][n_rows][n_kv_heads][head_dim]); every
 * other argument as for attn_prefill_chunk, whose workspace size it takes.
 * Arguments of both halves are checked before anything is enqueued.
 */
kvq_status attn_prefill_append(const kvq_layer* layer, const kvq_seq_cache* seqs, int32_t n_seqs,
                               const int32_t* row_offsets, const int32_t* start_pos, int32_t n_rows,
                               int32_t max_rows_per_seq,
                               const uint16_t* q_raw, const uint16_t* k_raw, const uint16_t* v_raw,
                               const uint16_t* q_norm_w, const uint16_t* k_norm_w,
                               void* out, int32_t out_is_f32, uint16_t* q_prepped, uint16_t* kv_prepped,
                               void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes of an attn_prefill_chunk call (0 for an invalid layer or a
 * negative count). */
size_t attn_prefill_workspace_bytes(const kvq_layer* layer, int32_t n_seqs, int32_t n_rows,
                                    int32_t max_rows_per_seq);

/*
 * attn_mixed -- several groups of query rows of one layer in one call, each
 * in its own phase, as in the mixed forward of the pages (serving-blocks.ts,
 * `#mixed`, and the Gemma `#mixed` scope: each group attends over its own
 * caches at its own positions, in decode or window mode, a verify group in
 * window mode).  A decode group computes the attn_decode call its fields
 * describe, a window group (prompt chunk or verify window) the
 * attn_prefill_chunk call.
 *
 * Schedule: the groups the decode kernels serve -- decode groups, verify
 * windows (at most 16 rows per sequence) and window groups of head shapes no
 * tensor-core kernel takes -- run as ONE grouped launch of each decode-path
 * kernel (q prep, attention, merge), whose grids cover the rows of all of
 * them; each group keeps its own caches, bit widths, positions, q, output and
 * workspace (its status word included), and its keys are cut into its own
 * fixed chunks of a split plan shared by all groups (so its outputs can
 * differ from the separate call's in the last bits, within the attention
 * tolerance).  A group whose workspace holds not even one split of that plan
 * runs on its own.  Prompt chunks on the tensor cores run beside the grouped
 * launch, concurrently on the GPU.  attn_mixed_schedule (below) reports which
 * groups a call would group.
 *
 *   groups      host array of n_groups descriptors (below), 0 <= n_groups <=
 *               KVQ_MAX_MIXED_GROUPS
 *   q_norm_w, out_is_f32, stream   as for attn_decode, shared by every group
 *
 * Every group is checked before anything is enqueued: on any failing group
 * the call returns that status and enqueues nothing.  Work enqueued on
 * `stream` before the call is complete before any group starts; work
 * enqueued on `stream` after it waits for every group.  Groups must not share
 * workspace, out or q_prepped memory (overlapping workspaces are rejected
 * with KVQ_EINVAL).  The groups run on streams and events the library
 * creates once per device on the first call with two or more groups: make
 * that call before any stream capture.  Calls that overlap on one device
 * (several host threads) must be serialised.
 */
#define KVQ_MAX_MIXED_GROUPS 8
enum { KVQ_PHASE_DECODE = 0, KVQ_PHASE_WINDOW = 1 };
typedef struct {
  int32_t phase;                 /* KVQ_PHASE_DECODE or KVQ_PHASE_WINDOW */
  const kvq_seq_cache* seqs;     /* device kvq_seq_cache[n_seqs] */
  int32_t n_seqs;
  const int32_t* row_offsets;    /* window: device int32[n_seqs + 1]; decode: ignored */
  const int32_t* pos;            /* device int32[n_seqs]: decode positions, or window start positions */
  int32_t n_rows;                /* window: rows of the group; decode: ignored (one row per sequence) */
  int32_t max_pos;               /* decode: host upper bound of pos[], below 2^24; window: ignored */
  int32_t max_rows_per_seq;      /* window: host upper bound of rows per sequence; decode: ignored */
  const uint16_t* q_raw;         /* device bf16 [rows][n_q_heads][head_dim] */
  void* out;                     /* device [rows][n_q_heads][head_dim], fp32 if out_is_f32 else bf16 */
  uint16_t* q_prepped;           /* NULL or device bf16 [rows][n_q_heads][head_dim] */
  void* workspace;               /* attn_decode_workspace_bytes / attn_prefill_workspace_bytes of the group */
  size_t workspace_bytes;
} kvq_attn_group;

kvq_status attn_mixed(const kvq_layer* layer, const kvq_attn_group* groups, int32_t n_groups,
                      const uint16_t* q_norm_w, int32_t out_is_f32, void* stream);

/*
 * attn_mixed_schedule -- every check and plan of the same attn_mixed call,
 * with nothing enqueued (host only, no device access): on KVQ_OK,
 * *grouped_mask has bit i set for each group i that would run in the grouped
 * launch (0 when fewer than two groups share it).  Returns what attn_mixed
 * would return for its checks; grouped_mask must not be NULL.
 */
kvq_status attn_mixed_schedule(const kvq_layer* layer, const kvq_attn_group* groups, int32_t n_groups,
                               const uint16_t* q_norm_w, int32_t out_is_f32, uint32_t* grouped_mask);

/*
 * The training forward's stateless read (trainable.ts, trainingCaches and
 * prefixShared.prefixSharedHidden; model.ts, the attentionTraining comment and
 * forwardTrainingHidden).  A training cache stores nothing: each donor layer
 * preps plain (unquantized) bf16 keys and values for the rows of the pass,
 * and every layer -- a KV-sharing one with its donor's keys and values -- reads
 * them under the pass's mask, block-sparse under a prefix-shared layout.
 *
 * Layout (the pages name the prefix-shared layout but do not print it; this
 * is the plain reading): the n_rows packed rows of one training sequence form
 * n_blocks blocks [block_offsets[b], block_offsets[b+1]).  Block 0 is the
 * shared prefix (it may be empty) at positions 0, 1, ...; every other block is
 * a branch continuing the prefix, its row j at position block_offsets[1] + j.
 * A row reads the rows of the prefix and of its own block whose positions are
 * at most its own (and, on a sliding layer, greater than its own - window).
 * One block is the plain causal (or windowed) training read.
 *
 *   block_offsets   device int32[n_blocks + 1]: 0 = block_offsets[0] <= ... <=
 *                   block_offsets[n_blocks] = n_rows (1 <= n_blocks <= 65535,
 *                   n_rows < 2^24).  A layout that breaks this for some block is
 *                   found by the kernels: that block's outputs are not written and
 *                   KVQ_STATUS_SEQ_SKIPPED is set in the status word.
 *   rot_signs of the layer must be NULL (KVQ_EUNSUPPORTED): the training read
 *   has no quantized cache to rotate.
 */

/*
 * kvq_train_kv_prep -- a donor layer's plain keys and values for the rows of
 * the pass: k_hat = RoPE_p(bf16(RMSNorm(k_raw, k_norm_w))) and v_hat =
 * bf16(RMSNorm(v_raw or k_raw if k_eq_v, no weight)), each row at its layout
 * position p.  Nothing is quantized.
 *
 *   k_raw, v_raw      device bf16 [n_rows][n_kv_heads][head_dim]; v_raw NULL iff k_eq_v
 *   k_norm_w          device bf16 [head_dim]
 *   k_hat, v_hat      device bf16 [n_rows][n_kv_heads][head_dim] (16-byte aligned),
 *                     the outputs
 */
kvq_status kvq_train_kv_prep(const kvq_layer* layer, int32_t n_blocks, const int32_t* block_offsets,
                             int32_t n_rows, const uint16_t* k_raw, const uint16_t* v_raw,
                             const uint16_t* k_norm_w, uint16_t* k_hat, uint16_t* v_hat, void* stream);

/*
 * attn_train_forward -- every row's q heads read the keys and values of the
 * rows they see under the layout (above), with SDPA scale 1.0:
 *   q_hat = RoPE_p(bf16(RMSNorm(q_raw, q_norm_w))),
 *   out[r][h] = sum_j softmax_j(q_hat . k_hat_j) v_hat_j.
 * It runs on the tcgen05 tensor cores, 128 (row, head) pairs of one block per
 * CTA (head_dim 512: each CTA half of the output dims): QK with the bf16
 * operands (exact products, fp32 accumulation), PV with P and v_hat as f16.
 * n_q_heads / n_kv_heads must divide 128 (KVQ_EUNSUPPORTED otherwise).
 *
 *   max_block_rows   host upper bound of the rows of every block (sizes the grid),
 *                    1 .. n_rows
 *   q_raw            device bf16 [n_rows][n_q_heads][head_dim]
 *   k_hat, v_hat     device bf16 [n_rows][n_kv_heads][head_dim] (16-byte aligned),
 *                    as written by kvq_train_kv_prep of this layer or its donor
 *   out              device [n_rows][n_q_heads][head_dim], fp32 if out_is_f32 else bf16
 *   q_prepped        NULL or device bf16 [n_rows][n_q_heads][head_dim] receiving q_hat
 *   workspace        device scratch of at least attn_train_workspace_bytes(layer,
 *                    n_rows) bytes; its first 4 bytes receive the status word
 */
kvq_status attn_train_forward(const kvq_layer* layer, int32_t n_blocks, const int32_t* block_offsets,
                              int32_t n_rows, int32_t max_block_rows,
                              const uint16_t* q_raw, const uint16_t* q_norm_w,
                              const uint16_t* k_hat, const uint16_t* v_hat,
                              void* out, int32_t out_is_f32, uint16_t* q_prepped,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_train_donor_forward -- a donor layer's training read in one call:
 * kvq_train_kv_prep of the pass's rows into k_hat / v_hat, then
 * attn_train_forward over them, bit for bit.  The K/V prep runs in the grid
 * of the read's q prep (the two share nothing).  Arguments as for those two
 * calls; k_hat / v_hat are written and kept (the layer's sharers read them).
 */
kvq_status attn_train_donor_forward(const kvq_layer* layer, int32_t n_blocks, const int32_t* block_offsets,
                                    int32_t n_rows, int32_t max_block_rows,
                                    const uint16_t* q_raw, const uint16_t* k_raw, const uint16_t* v_raw,
                                    const uint16_t* q_norm_w, const uint16_t* k_norm_w,
                                    uint16_t* k_hat, uint16_t* v_hat,
                                    void* out, int32_t out_is_f32, uint16_t* q_prepped,
                                    void* workspace, size_t workspace_bytes, void* stream);

size_t attn_train_workspace_bytes(const kvq_layer* layer, int32_t n_rows);

/*
 * attn_decode_static -- attn_decode without a caller-provided workspace, for
 * callers that cannot allocate device memory: code that only receives input
 * and output pointers from a host framework that owns every allocation (a
 * plugin or kernel-library slot with no allocator handle), or a serving loop
 * that reserves all device memory up front and forbids allocation
 * afterwards.  The pages have no counterpart of this call: it exists only
 * because the workspace of attn_decode must otherwise come from the caller.
 *
 * Same arguments and results as attn_decode, minus workspace and
 * workspace_bytes.  The scratch is a static device array of
 * KVQ_STATIC_SCRATCH_BYTES bytes inside libkvq.so; every GPU that loads the
 * library holds it until the process exits.  The call allocates nothing (no
 * cudaMalloc, no cudaFree, no allocating library routine).
 *   - A call whose attn_decode_workspace_bytes(layer, n_seqs, max_pos) exceeds
 *     KVQ_STATIC_SCRATCH_BYTES returns KVQ_EWORKSPACE and enqueues nothing.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Every call shares the one array and leaves its contents behind (the
 *     status word at its start is cleared by each call).  Calls whose work
 *     overlaps on the GPU (different streams, or different host threads on
 *     one device) race on it: serialise them.
 *   - The device status word of the call (see KVQ_STATUS_*) stays in the
 *     array until the next call on the device; kvq_static_status copies it out.
 */
#define KVQ_STATIC_SCRATCH_BYTES (16u << 20)
kvq_status attn_decode_static(const kvq_layer* layer, const kvq_seq_cache* seqs, int32_t n_seqs,
                              const int32_t* pos, int32_t max_pos,
                              const uint16_t* q_raw, const uint16_t* q_norm_w,
                              void* out, int32_t out_is_f32, uint16_t* q_prepped, void* stream);

/*
 * kvq_static_status -- the device status word of the latest attn_decode_static
 * call on the current device (0 = clean, else KVQ_STATUS_* bits), for the same
 * callers: they have no workspace to read it from.  The pages have no
 * counterpart of this call.
 *
 *   status   host or device memory for one uint32 (4-byte aligned).  The copy
 *            is enqueued on `stream`, after the work enqueued there before; read
 *            *status once the stream has synchronized (with pageable host
 *            memory the call itself returns after the copy).  It allocates
 *            nothing and, like attn_decode_static, races with static calls
 *            whose work overlaps it on the GPU.
 */
kvq_status kvq_static_status(uint32_t* status, void* stream);

/*
 * kvq_selftest_wait_timeout -- exercises the failure detection of the
 * attention kernels without faulting the GPU.  Every wait of the kernels (on
 * the mbarriers their bulk copies complete) gives up after a bounded time,
 * sets a status bit and lets the kernel finish, so that a lost completion
 * never hangs the device.  This call launches one small kernel whose wait,
 * on an mbarrier that nothing completes, runs out after limit_ns; it then
 * ORs bit 1 (the "bounded wait gave up" bit of the attention status word)
 * into *status.  Nothing else is touched and no copy is in flight.
 *
 *   status     device uint32 (4-byte aligned), typically cleared beforehand
 *   limit_ns   1e3 .. 1e9
 */
kvq_status kvq_selftest_wait_timeout(uint32_t* status, uint64_t limit_ns, void* stream);

/* Static message for a status code. */
const char* kvq_status_string(kvq_status status);
/*
 * kvq_profile_next_read -- profiling: the calling host thread's next call
 * that reads attention (attn_decode, attn_decode_append, attn_prefill_chunk,
 * attn_prefill_append, attn_train_forward, attn_train_donor_forward; not
 * attn_mixed) records start_event on its stream right before launching its
 * attention kernel and stop_event right after, so that
 * cudaEventElapsedTime gives that kernel's time alone.  Both are
 * cudaEvent_t created with timing enabled, or both NULL (clears).  Inside a
 * stream capture they are recorded as external event nodes.  Recording an
 * event between two kernels of a call removes their programmatic overlap.
 */
kvq_status kvq_profile_next_read(void* start_event, void* stop_event);

/* Message of the calling thread's most recent failing call ("" if none). */
const char* kvq_last_error(void);
/* Library version, major*10000 + minor*100 + patch. */
int32_t kvq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H_ */
