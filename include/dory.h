/*
 * dory.h - C ABI of the GB300 (sm_103a) Dory looped normalized-GPT token forward.
 *
 * The forward is the one the docs.rs source page "cortiq_engine/dory.rs"
 * (cortiq-engine 0.8.78) computes on the host:
 *   - an input block runs once per token (fn stack, input layers);
 *   - a recurrent block runs `loops` times, each pass taking h = (state + input)^
 *     and leaving state = R(h)^ (fn stack, the loop mix);
 *   - an output block and the head follow: logits = (H h) * logit_scale
 *     (fn head).
 * Every sub-layer is an attention or SwiGLU MLP on the unit sphere with the
 * nGPT residual x = (x^ + |alpha| (out^ - x^))^ (fn attn_layer, fn mlp_layer,
 * fn slerp). The KV cache is a sliding ring per (attention layer, loop slot)
 * sized window + 64 + 448 rows (page "src/gpu_metal/dory.rs" 0.8.70, fn run),
 * in per_loop or last_loop mode (fn slot_loop, fn attn_layer's overwrite), with
 * rows stored as f32 or as q8_2f (page "cortiq_engine/kv_cache.rs" 0.8.78,
 * fn quant_row, fn freeze_cols, fn append).
 *
 * Conventions for every entry point:
 *   - The return value is DORY_OK (0) or a negative DORY_E* status. The message
 *     of the last failure on the calling thread is dory_last_error().
 *   - A pointer argument may point to host memory or to device memory of the
 *     handle's GPU (CUDA unified addressing tells them apart) unless its comment
 *     says otherwise. The library never keeps a caller pointer past the call.
 *   - All work is ordered on the stream given to dory_create. Calls that write
 *     to host memory (dory_logits with a host dst, the read hooks) synchronise
 *     that stream before they return; the others return once the work is queued.
 *   - A handle is not thread-safe: one thread at a time.
 */
#ifndef DORY_H
#define DORY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define DORY_OK 0
#define DORY_EINVAL (-1) /* a bad argument or config; nothing changed */
#define DORY_ENOMEM (-2) /* device or host memory could not be allocated */
#define DORY_ECUDA (-3)  /* a CUDA call failed; the handle should be destroyed */
#define DORY_ESTATE (-4) /* the call does not fit the sequence's state (e.g. pos0) */
#define DORY_ERANGE (-5) /* a position past what the rings can hold */
#define DORY_EWAIT (-6)  /* a kernel gave up a bounded wait (the message has its code): the rows
                          * of the steps since the last reported status are undefined; reset
                          * those sequences, the handle itself stays usable. Reported once, by
                          * the next call that synchronises (dory_logits, the read hooks). */

/* KV modes (dory.rs, enum KvMode): per_loop keeps one slot per loop for the
 * recurrent attention layers; last_loop keeps one slot per attention layer and
 * each loop > 0 rewrites the chunk's rows in place. */
#define DORY_KV_PER_LOOP 0
#define DORY_KV_LAST_LOOP 1

/* KV row storage (kv_cache.rs, enum KvMode): f32 rows, or q8_2f: int8 K codes with
 * one f32 scale per 32 channels, int8 V codes with one f32 scale per row, and
 * per-channel RMS fields frozen at the first append that finds 64 stored rows. */
#define DORY_KV_F32 0
#define DORY_KV_Q8_2F 1

/* Weight element type of the matrices (embedding, head, projections). */
#define DORY_W_F32 0
#define DORY_W_BF16 1 /* raw bfloat16 bits, uint16_t per element */

/* Which rows of a prefill chunk get logits (dory.rs, enum Want). */
#define DORY_WANT_NONE 0
#define DORY_WANT_LAST 1
#define DORY_WANT_ALL 2

#define DORY_MAX_LOOPS 16 /* dory.rs, const MAX_LOOPS */
#define DORY_CHUNK_ROWS 64 /* rows of one prefill chunk at most (dory.rs, HOST_CHUNK) */
#define DORY_MAX_BATCH 128 /* sequences of one decode step at most */

typedef struct dory_config {
  int32_t hidden, ffn, vocab; /* model width, MLP width, vocabulary rows */
  int32_t nh, nk, hd;         /* query heads, KV heads (nh % nk == 0), head width: 32, 64 or 128; nh / nk in {1, 2, 4, 8} */
  int32_t window;             /* sliding attention window W: keys [p-W+1, p] */
  int32_t full_window;        /* full layers' window; 0: every earlier row up to max_context */
  int32_t max_context;        /* positions a full layer without full_window can hold */
  int32_t n_in, n_rec, n_out; /* physical sub-layers of the input, recurrent, output blocks */
  const char *layer_pattern;  /* n_in+n_rec+n_out chars: 'S' sliding attention, '*' full, '-' MLP */
  double rope_theta_sliding;  /* RoPE base of sliding layers */
  double rope_theta_full;     /* RoPE base of full layers */
  int32_t max_loops;          /* loop slots of per_loop rings and the loop bound, 1..16 */
  int32_t kv_mode;            /* DORY_KV_PER_LOOP or DORY_KV_LAST_LOOP */
  int32_t kv_quant;           /* DORY_KV_F32 or DORY_KV_Q8_2F */
  int32_t prompt_loops;       /* last_loop: passes of a chunk whose logits are unread; 0: all */
  int32_t max_batch;          /* sequences one decode step may carry, 1..DORY_MAX_BATCH */
  int32_t max_seqs;           /* sequences (KV states) the handle keeps */
  int32_t weight_dtype;       /* DORY_W_F32 or DORY_W_BF16 */
} dory_config;

/* One physical layer's weights. Matrices are row-major [out][in] in the config's
 * weight dtype; vectors are f32. Scales are the effective (folded) values of
 * dory.rs fn from_model: sq = (sqk sqrt(hd)/sigma0)^2, sg = (s_gate sqrt(g0)/sigma0)^2,
 * mlp_sg/mlp_su = suv sqrt(hidden), alpha = |alpha_raw alpha_init/sigma0|. */
typedef struct dory_layer_weights {
  const void *q, *k, *v, *g; /* attention: [nh*hd][hidden], [nk*hd][hidden] x2, [nh*hd][hidden] */
  const void *o;             /* attention: [hidden][nh*hd] */
  const float *sq, *sg;      /* attention: [nh*hd] each */
  const void *gate, *up;     /* MLP: [ffn][hidden] each */
  const void *down;          /* MLP: [hidden][ffn] */
  const float *mlp_sg, *mlp_su; /* MLP: [ffn] each */
  const float *alpha;        /* both kinds: [hidden] */
} dory_layer_weights;

typedef struct dory_weights {
  const void *embed;        /* [vocab][hidden] */
  const void *head;         /* [vocab][hidden] */
  const float *logit_scale; /* [vocab], logit_scale/sigma0 */
  const dory_layer_weights *layers; /* one per char of layer_pattern; unused fields may be NULL */
} dory_weights;

typedef struct dory_handle dory_t;

/* Build a handle: checks the config (nh % nk == 0, 1 <= max_loops <= 16, the pattern's
 * length and chars, hd in {32, 64, 128}, nh / nk in {1, 2, 4, 8}, hidden and ffn multiples
 * of 32, hidden <= 8192, ffn and nh * hd <= 32768, ...), copies every weight into device
 * memory the handle owns (the caller may free its buffers on return), allocates the KV
 * rings of max_seqs sequences and resets them. `stream` is a cudaStream_t (NULL: the
 * legacy default stream) that orders all of the handle's work.
 * Errors: DORY_EINVAL, DORY_ENOMEM, DORY_ECUDA; *out is NULL then. */
int dory_create(const dory_config *cfg, const dory_weights *w, void *stream, dory_t **out);

/* Free everything the handle owns (after synchronising its stream). NULL is a no-op.
 * The handle plays the part of the Metal path's per-model Device (page
 * "src/gpu_metal/dory.rs", fn forward: built on a model's first forward and kept in the
 * DEVICES map); the pages never remove one, so this entry point has no counterpart there
 * beyond dropping that state. */
int dory_destroy(dory_t *d);

/* Empty one sequence's rings and set its position to 0 (gpu_metal/dory.rs fn reset). */
int dory_reset(dory_t *d, int32_t seq);

/* Forget the rows of sequence `seq` from position n on (dory.rs DoryState::rollback, which
 * serves a rejected speculation or a new turn that rewrites the end of the last one): every
 * slot keeps its rows at positions < n and the sequence's position becomes min(pos, n). On
 * q8_2f rings the dropped rows leave the store as kv_cache.rs fn truncate_last drops them: a
 * field that froze stays frozen, and a slot that has not frozen yet counts only the rows it
 * keeps toward the 64 the freeze waits for. A ring keeps window + 64 + 448 rows (page
 * "src/gpu_metal/dory.rs", fn run: the chunk and the REWIND rows), so a rollback may go back
 * as long as every window that reads a row before n still finds its rows: at most
 * rows - window + 1 positions on a sliding ring (513 with the pages' sizes); a full layer
 * without full_window holds every position. n >= the position changes nothing.
 * Errors: DORY_EINVAL (seq, n < 0), DORY_ERANGE (further back than a ring keeps; nothing
 * changed), DORY_ECUDA. */
int dory_rollback(dory_t *d, int32_t seq, int32_t n);

/* One prefill chunk of `n` (1..64) rows of sequence `seq` at positions pos0..pos0+n-1
 * (dory.rs fn forward_host for one chunk): pos0 must equal the sequence's position
 * (DORY_ESTATE otherwise). `ids` [n] int32; an id outside [0, vocab) embeds as a zero
 * row (dory.rs: such a row is left at zero). `loops` 1..max_loops passes of the
 * recurrent block; under last_loop with want == DORY_WANT_NONE and prompt_loops > 0 the
 * chunk runs min(loops, prompt_loops) passes (fn chunk_loops). `want` chooses the rows
 * whose logits dory_logits can read afterwards (none, the last row, every row).
 * Errors: DORY_EINVAL (n, loops, want, seq), DORY_ESTATE (pos0), DORY_ERANGE (a full
 * layer without full_window past max_context), DORY_ECUDA. */
int dory_prefill_chunk(dory_t *d, int32_t seq, const int32_t *ids, int32_t n, int32_t pos0,
                       int32_t loops, int32_t want);

/* A whole prompt of `n` rows of sequence `seq` from position pos0: the same result as
 * dory_prefill_chunk over consecutive chunks of 64 rows from pos0 with `want` on the last
 * chunk and DORY_WANT_NONE on the others (dory.rs fn forward_host; prompt_loops as there).
 * The input and output blocks run once per row, at loop 0, and attend causally to their own
 * rows, so their projections and MLPs run over up to 4096 rows of many chunks at once (dense
 * contractions on the tensor cores, activations rounded to bf16 from 256 rows up; 512 rows
 * with q8_2f rings), while the recurrent block runs chunk by chunk (under last_loop a chunk's
 * rows see earlier chunks at their last pass). Their attention takes pieces of as many rows
 * as the input/output rings hold beyond their window (512 with the pages' sizes); without
 * room for 128 rows, or with f32 weights, the prompt goes chunk by chunk. `want`:
 * DORY_WANT_NONE or DORY_WANT_LAST (one logits row).
 * Errors: as dory_prefill_chunk (n >= 1, want none or last). */
int dory_prefill(dory_t *d, int32_t seq, const int32_t *ids, int32_t n, int32_t pos0, int32_t loops, int32_t want);

/* Prefill chunks of several sequences in one step (the chunk of dory.rs fn forward_host for
 * each, at that sequence's position): sequence seqs[j] takes counts[j] (1..64) rows, ids
 * [sum of counts] holding each sequence's rows in turn. Every projection runs once over all
 * the rows; each sequence's rows attend causally to their own rings. `loops`, `want` and
 * prompt_loops as in dory_prefill_chunk, for every sequence. Logits: want last gives one row
 * per sequence (row j = sequence seqs[j]'s last row), want all every row in the order of
 * `ids`. `seqs` and `counts` must be host pointers; at most max(64, max_batch) rows in all.
 * Errors: DORY_EINVAL (nseq, counts, a duplicate sequence, too many rows, loops, want),
 * DORY_ERANGE, DORY_ECUDA. */
int dory_prefill_batch(dory_t *d, int32_t nseq, const int32_t *seqs, const int32_t *counts, const int32_t *ids,
                       int32_t loops, int32_t want);

/* One decode token for each of `batch` distinct sequences: row b is token ids[b] of
 * sequence seqs[b] at that sequence's position, a one-row chunk whose logits are read
 * (dory.rs fn forward_host with a chunk of t = 1 and Want::Last, once per sequence; the
 * rows of the step share every weight pass). `seqs` must be a host pointer. One loop
 * count for the whole step.
 * Errors: DORY_EINVAL (batch, duplicate or bad seq, loops), DORY_ERANGE, DORY_ECUDA. */
int dory_decode_step(dory_t *d, const int32_t *ids, const int32_t *seqs, int32_t batch, int32_t loops);

/* dory_decode_step with one loop count per sequence: row b runs loops[b] (1..max_loops)
 * passes of the recurrent block, as sequence seqs[b]'s own forward would (dory.rs
 * fn forward_host takes the loop count per call, so each row is that call for its sequence).
 * The step runs the passes of the longest row; pass i computes only the rows with more than
 * i loops, so a row's later passes neither cost weight-streaming rows nor write KV rows.
 * `loops` must be a host pointer [batch]. Logits and hidden rows come back in the caller's
 * order (row b = seqs[b]). Equal counts take dory_decode_step.
 * Errors: as dory_decode_step. */
int dory_decode_ragged(dory_t *d, const int32_t *ids, const int32_t *seqs, int32_t batch, const int32_t *loops);

/* One decode token of one sequence under the Conf(th) early-exit gate (dory.rs enum Gate,
 * fn stack's early-exit block, struct ExitRate, fn top_prob; the Metal path's token gate in
 * page "src/gpu_metal/dory.rs", fn forward's run stages). The sequence's exit rate decides
 * whether the token reads out after its first pass: while the rate of early exits is at least
 * 0.35, and for one token in eight below it. A read-out runs the first pass, the output block
 * and the head, and takes top_prob of the logits (the largest softmax probability, from the
 * entries within 20 of the top); top_prob >= th ends the token there, with those logits. A
 * token that stays (or does not read out) runs a second recurrent pass from the first pass's
 * state and input, then the output block and head again; the second output block rewrites
 * the rows the read-out appended in both KV modes. So a token makes 1 or 2 passes whatever
 * the handle's loop count. `id`: one int32 token id (host or device). *passes gets 1 or 2,
 * *top_prob the read-out's top probability or NaN without a read-out (either may be NULL).
 * The decision needs the probability on the host: a read-out synchronises the stream.
 * dory_reset restores the sequence's exit rate to its start (1.0, no tokens).
 * Errors: DORY_EINVAL (seq, th NaN, max_loops < 2), DORY_ERANGE, DORY_ECUDA. */
int dory_decode_conf(dory_t *d, const int32_t *id, int32_t seq, float th, int32_t *passes, float *top_prob);

/* Copy the logits of row `row` of the last call that produced logits ([vocab] f32,
 * logits = (H h) * logit_scale per vocabulary row, dory.rs fn head) to dst, which has room
 * for `cap` floats. Decode: row = batch index. Prefill: want last gives row 0 only (the
 * chunk's last row, Want::Last), want all rows 0..n-1 (Want::All).
 * Errors: DORY_EINVAL (row, cap < vocab), DORY_ESTATE (no logits yet), DORY_EWAIT (a kernel
 * of the steps since the last check gave up a bounded wait), DORY_ECUDA. */
int dory_logits(dory_t *d, int32_t row, float *dst, size_t cap);

/* Device address of the logits buffer [rows][vocab] of the last call (no copy). */
int dory_logits_device(dory_t *d, const float **out, int32_t *rows);

/* Message of the last failure on this thread ("" if none). Never NULL. */
const char *dory_last_error(void);

/* ---- inspection and test hooks (same library, same rules) ---------------------------- */

/* Final hidden states of the last forward call, [rows][hidden] f32, before the head.
 * Errors: DORY_EINVAL, DORY_EWAIT (as dory_logits), DORY_ECUDA. */
int dory_read_hidden(dory_t *d, float *dst, size_t cap);

/* Geometry of attention layer `ordinal`'s rings: rows per ring, loop slots, and whether
 * the layer is sliding (1) or full (0). */
int dory_slot_info(dory_t *d, int32_t ordinal, int32_t *cap, int32_t *slots, int32_t *sliding);

/* Append n rows [n][nk][hd] of K and V (f32) to slot (ordinal, loop_slot) of `seq` at
 * positions pos0..pos0+n-1 through the same append path a forward uses (quantisation and
 * the 64-row freeze for q8_2f). pos0 must equal the rows the slot has appended so far.
 * The sequence's position is not moved (see dory_set_position). */
int dory_write_kv_rows(dory_t *d, int32_t seq, int32_t ordinal, int32_t loop_slot, int32_t pos0,
                       int32_t n, const float *k, const float *v);

/* Set a sequence's next position (after dory_write_kv_rows built a context). */
int dory_set_position(dory_t *d, int32_t seq, int32_t pos);

/* Read a ring of f32 rows: tags [cap] (the position a ring row holds, -1 if empty) and
 * K, V [nk][cap][hd]. Any output pointer may be NULL. */
int dory_read_kv_f32(dory_t *d, int32_t seq, int32_t ordinal, int32_t loop_slot, int32_t *tags,
                     float *k, float *v);

/* Read a q8_2f ring: tags [cap], K codes [nk][cap][hd], K scales [nk][cap][hd/32],
 * V codes [nk][cap][hd], V scales [nk][cap], fields kcol, vcol [nk][hd] (zeros until
 * frozen), frozen [nk] (0/1). Any output pointer may be NULL. */
int dory_read_kv_q8(dory_t *d, int32_t seq, int32_t ordinal, int32_t loop_slot, int32_t *tags,
                    int8_t *kq, float *ks, int8_t *vq, float *vs, float *kcol, float *vcol,
                    int32_t *frozen);

typedef struct dory_stats {
  uint64_t weight_bytes_device; /* weights resident on the device */
  uint64_t kv_bytes_device;     /* KV rings of all sequences */
  uint64_t weight_bytes;        /* algorithmic weight bytes the last call streamed */
  uint64_t kv_read_bytes;       /* algorithmic KV bytes the last call's attention read */
  uint64_t kv_write_bytes;      /* KV bytes the last call wrote */
  uint64_t launches;            /* kernels the last call launched */
  uint64_t gemm_launches;       /* of which weight-streaming GEMV/GEMM launches */
  uint64_t flops;               /* algorithmic FLOPs of the last call's projections and head (2 x weights x rows) */
} dory_stats;

/* Byte and launch accounting of the handle and of its last call (dory_prefill: the totals
 * over its steps). */
int dory_get_stats(dory_t *d, dory_stats *out);

/* ---- for callers that cannot allocate device memory ---------------------------------- */

/* The pages have no counterpart of this entry point: it serves callers that may not call
 * cudaMalloc (code running inside another runtime's allocator or memory pool, code that
 * runs while a CUDA graph is being captured, plugins that must not grow the process's
 * device memory). It quantises n K and V rows to q8_2f exactly as dory_write_kv_rows
 * appends them to an empty slot: the same codes, scales and frozen fields, bit for bit,
 * without a handle and without allocating anything.
 *   k, v   [n][nk][hd] f32 rows, in memory the current device can read (device, managed or
 *          mapped pinned memory);
 *   kq, vq [nk][n][hd] int8 codes; ks [nk][n][hd/32] and vs [nk][n] f32 scales;
 *   kcol, vcol [nk][hd] f32 fields (all zero when n <= 64: nothing froze) - all outputs in
 *          device memory the caller owns;
 *   stream a cudaStream_t (NULL: the legacy default stream); the call returns once the work
 *          is queued on it.
 * Limits: 1 <= nk <= 16, hd in {32, 64, 128}, n >= 1; anything else is DORY_EINVAL.
 * Working memory: a static device array of about 290 KB inside the library (the row
 * counters and the first 64 rows the freeze reads back), held by every GPU that loads the
 * library until the process exits. The first call on a device looks up that array's device
 * address (cudaGetSymbolAddress) and must come before any stream capture on that device; so
 * must the first call after a cudaDeviceReset of that device, which ends the context the
 * address belonged to (the library notices the new context and looks the address up again).
 * Every call clears the counters it needs at zero; calls share the array, so two calls
 * whose work overlaps on the GPU race and must not be made. Errors: DORY_EINVAL,
 * DORY_ECUDA; the message is dory_last_error(). */
int dory_q8_quantize_noalloc(const float *k, const float *v, int32_t n, int32_t nk, int32_t hd, int8_t *kq,
                             float *ks, int8_t *vq, float *vs, float *kcol, float *vcol, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DORY_H */
