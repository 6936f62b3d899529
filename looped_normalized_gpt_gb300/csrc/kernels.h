// Internal launch interface of the Dory kernels. Host code only passes plain pointers,
// sizes and the small structs below; every launch goes on the given stream.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace dory {

enum WDtype { W_F32 = 0, W_BF16 = 1 };

// GEMM epilogues: Y = X W^T, then
enum Epi {
  EPI_STORE = 0,  // y
  EPI_SCALE = 1,  // y * vec[n]                         (head: logit_scale)
  EPI_SILU = 2,   // silu(g * sg[n]) * (u * su[n])       (SwiGLU; g = row n, u = row n + pair)
};

struct EpiArgs {
  int mode;
  const float *vec;  // EPI_SCALE: [N]; EPI_SILU: sg [N]
  const float *vec2; // EPI_SILU: su [N]
  long pair;         // EPI_SILU: row offset of the `up` rows within W
};

// Where a step's rows sit: row r is sequence seq[r] at position seq_pos[seq[r]] + off[r].
struct Rows {
  const int32_t *seq;
  const int32_t *off;
  const int32_t *seq_pos;
  int n;
};

// Byte layout of one KV slot (one sequence, one attention layer, one loop slot).
struct SlotLayout {
  size_t bytes;
  size_t tags, k, v;                  // f32: tags[cap] i32, K/V [nk][cap][hd] f32
  size_t kq, ks, vq, vs;              // q8: codes [nk][cap][hd] i8, K scales [nk][cap][hd/32], V scales [nk][cap]
  size_t kcol, vcol, meta;            // q8: fields [nk][hd] f32, meta [nk][4] i32 {appended, frozen}
  size_t wpos, wkq, wks, wvq, wvs;    // q8: the first 64 appended rows, [nk][64]...
};

SlotLayout slot_layout(int cap, int nk, int hd, bool q8);

// One attention layer's ring as the kernels see it.
struct Ring {
  char *base;         // device base of all KV memory
  size_t seq_stride;  // bytes per sequence
  size_t off;         // bytes from a sequence's block to this (layer, loop slot)
  SlotLayout L;
  int cap;
  int window;         // keys [p - window + 1, p]; INT32_MAX: every stored row
  int q8;
};

struct Dims {
  int hidden, ffn, vocab, nh, nk, hd;
};

// --- launches -------------------------------------------------------------------------

// Rows kept as f32 and, for the tensor-core projections, as two bf16 halves
// (hi = bf16(x), lo = bf16(x - hi)); hi/lo may be null.
struct Emit {
  __nv_bfloat16 *hi, *lo;
};

// h null: only the RoPE table of the rows (their hidden rows are not touched, ids unused).
cudaError_t launch_embed_rope(const int32_t *ids, const void *E, int wdtype, Dims d, Rows rows,
                              double theta_s, double theta_f, float *h, float *rope, Emit em, cudaStream_t s);

cudaError_t launch_gemm(const void *W, int wdtype, int N, int K, const float *X, int ldx, int T, float *Y,
                        int ldy, EpiArgs ep, cudaStream_t s);

// q, k rotation + per-head justnorm + q*sq; f32 rings get k, v and the tag, q8 rings get
// k, v into the staging rows kst/vst [T][nk][hd].
cudaError_t launch_prep(float *qkvg, int ldq, Dims d, Rows rows, const float *rope, int kind, const float *sq,
                        Ring ring, float *kst, float *vst, cudaStream_t s);

// q8_2f append of staged rows, with the 64-row freeze (one block per (sequence, kv head)).
// Rows of one sequence are consecutive; `rewrite` marks a last_loop rewrite of those rows.
cudaError_t launch_q8_append(const float *kst, const float *vst, int ld_rows, Dims d, Rows rows, Ring ring,
                             int rewrite, cudaStream_t s);

// Rows [n][nk][hd] of one sequence appended at pos0.. to a slot whose field is frozen.
cudaError_t launch_q8_append_frozen(const float *kst, const float *vst, int n, Dims d, int seq, long pos0, Ring ring,
                                    cudaStream_t s);

// Split-KV attention: partials, then the combine with the output gate y * sigmoid(g*sg).
cudaError_t launch_attention(const float *qkvg, int ldq, Dims d, Rows rows, Ring ring, int splits, int keys_per_split,
                             float *part, const float *sg, float *z, cudaStream_t s);

// A prefill chunk's attention: rows 0..T-1 are consecutive positions of one sequence
// (f32 ring, hd 64 or 128); `nkb` = attn_chunk_blocks(window keys, T) key blocks. Writes z
// gated and row-normalised (with its bf16 halves when em.hi is set).
int attn_chunk_blocks(long window_keys, int rows);
cudaError_t launch_attention_chunk(const float *qkvg, int ldq, Dims d, Rows rows, Ring ring, int nkb, float *part,
                                   const float *sg, float *z, Emit em, int *err, cudaStream_t s);

// Rows of any sequences (a batched decode step) over f32 rings (hd 64 or 128) or q8_2f rings
// (hd 128): `splits` blocks
// per (row, kv head) stream consecutive parts of the window in 32-position tiles; writes z
// gated (not row-normalised). splits > 1: part holds rows * nk * splits * REP * (hd + 2)
// floats, ctr rows * nk counters (zero between launches). attn_stream_splits picks splits.
int attn_stream_splits(long window_keys, int rows, int nk, int sms);
cudaError_t launch_attention_stream(const float *qkvg, int ldq, Dims d, Rows rows, Ring ring, const float *sg,
                                    float *z, int *err, int splits, float *part, int *ctr, cudaStream_t s);

cudaError_t launch_rownorm(float *x, int T, int width, int ld, Emit em, cudaStream_t s);

// The loop mix of dory.rs fn stack after a sub-layer: MIX_BEGIN (the input block's end:
// input = state = h, h = (state + input)^), MIX_LOOP (a pass's end: state = h^, then
// h = (state + input)^), MIX_END (the last pass's end: state = h^, h = state), and
// MIX_RESUME, which replaces the sub-layer's output: h = (state + input)^ from the saved
// input and state rows (the second pass of an early-exit gate that decided to stay).
enum Mix { MIX_NONE = 0, MIX_BEGIN = 1, MIX_LOOP = 2, MIX_END = 3, MIX_RESUME = 4 };

// x = (x^ + alpha (out^ - x^))^ per row, then the loop mix (dory.rs fn stack).
cudaError_t launch_residual(float *h, const float *out, const float *alpha, int T, int hidden, int mix,
                            float *input, float *state, int do_residual, Emit em, cudaStream_t s);

// ---- fused decode path (up to 4 rows) -------------------------------------------------

enum InMode { IN_PLAIN = 0, IN_NORM = 1, IN_RESID = 2, IN_EMBED = 3 };

// How a fused GEMV builds its input rows: the source rows as they are, their row norm,
// the nGPT residual of the previous sub-layer (src = its input h, out = its output)
// followed by the loop mix, or the embedding rows of the step's token ids (bf16 table).
// With IN_RESID and IN_EMBED the leading block stores the result to h_dst (and the mix's
// input/state rows).
struct GemvIn {
  int mode;
  const float *src;
  int ld;
  const float *out;
  const float *alpha;  // nullptr: the mix alone
  int mix;
  float *h_dst;
  float *input;
  float *state;
  const int32_t *ids;            // IN_EMBED: token ids [T]; an id outside [0, vocab) gives a zero row
  const __nv_bfloat16 *embed;    // IN_EMBED: table [vocab][K]
  int vocab;
  // Persistent kernel only (zero elsewhere). Rows that earlier stages of the same launch
  // wrote as tagged words (value, tag) are awaited word by word until each carries the
  // producing stage's tag: src_t replaces src, out_t replaces out.
  const unsigned long long *src_t, *out_t;
  uint32_t src_tag, out_tag;
  // 1 + the row of the block's private area that holds src / input (the block wrote it
  // itself earlier in the launch), or 0: read the shared row; hdst_pv / input_pv: also store
  // the new hidden row / the mix's input row there (every block, not only the leading one)
  int src_pv, hdst_pv, input_pv;
};

// Per-head epilogue of the q/k/v/g projection (RoPE, justnorm, s_q^2, ring write).
struct HeadEpi {
  int enabled;
  int *counters;  // one arrival counter per head, zero between launches
  Dims d;
  Rows rows;
  const float *rope;
  int kind;
  const float *sq;
  Ring ring;
  float *kst, *vst;
};

cudaError_t launch_gemv_fused(const void *W, int wdtype, int N, int K, int T, GemvIn in, float *Y, int ldy,
                              EpiArgs ep, HeadEpi he, int *err, bool pdl, cudaStream_t s);

cudaError_t launch_attention_fused(const float *qkvg, int ldq, Dims d, Rows rows, Ring ring, int splits, int kps,
                                   float *part, const float *sg, float *z, int *counters, bool pdl, cudaStream_t s);

// ---- tensor-core projections (tcgen05) for steps of 5+ rows ----------------------------

struct TcGemm {
  CUtensorMap tmW;          // W bf16 [rows][K], boxes of 128 x 64
  CUtensorMap tmXh, tmXl;   // activation halves bf16 [rows][K], boxes of BN x 64
  int N, K, splits;
  long pair_rows;           // SwiGLU: offset of the up rows in W
  float *ws;                // split-K partial tiles
  int *ctr;                 // per-tile arrival counters (zero between launches)
  int *err;                 // set when a bounded wait expires
  unsigned long long *trace;  // null, or [grid.y][grid.x][TC_TRACE_EVENTS] %globaltimer stamps
  // launch_tc_gemm_big's split K: 2 * sms partial tiles of 128 x 256 floats, and ctr_slots
  // per-tile counters (zero between launches)
  float *ws_big = nullptr;
  int *ctr_big = nullptr;
  int ctr_slots = 0, sms = 0;
};
constexpr int TC_TRACE_EVENTS = 12;

int tc_tile_rows(int T);
int make_tmap_bf16(CUtensorMap *map, const void *base, long rows, long cols, int box_rows);
cudaError_t launch_tc_gemm(const TcGemm &g, int T, int t_base, float *Y, int ldy, EpiArgs ep, bool pdl,
                           cudaStream_t s);

// Steps of many rows (a few hundred and up): step rows as the MMA's M side (128 per tile),
// 256 weight rows as N (SwiGLU: 128 gate + 128 up rows), activations as one bf16 operand
// (g.tmXh, boxes of 128 rows x 64), one tile per block. g.tmW: boxes of 128 weight rows.
// K a multiple of 64; SwiGLU: N a multiple of 128.
cudaError_t launch_tc_gemm_big(const TcGemm &g, int T, int t_base, float *Y, int ldy, EpiArgs ep, bool pdl,
                               cudaStream_t s);

// ---- attention over f32 rings with TMA-staged tiles ------------------------------------

int attn_tma_splits(long window_keys);
int make_tmap_kv_f32(CUtensorMap *map, const void *base, size_t bytes, int hd);
cudaError_t launch_attention_tma(const CUtensorMap &map, const float *qkvg, int ldq, Dims d, Rows rows, Ring ring,
                                 int splits, float *part, const float *sg, float *z, int *counters, int *err, bool pdl,
                                 cudaStream_t s);

// q8_2f rings with hd = 128: the KV memory as code rows, K-scale rows and V-scale runs.
struct KvMaps {
  CUtensorMap codes, kscales, vscales;
};
int make_tmap_kv_q8(KvMaps *m, const void *base, size_t bytes);
cudaError_t launch_attention_tma_q8(const KvMaps &m, const float *qkvg, int ldq, Dims d, Rows rows, Ring ring,
                                    int splits, float *part, const float *sg, float *z, int *counters, int *err,
                                    bool pdl, cudaStream_t s);

// ---- persistent batch-1 decode ---------------------------------------------------------

enum MegaKind { MK_GEMV = 0, MK_ATTN = 1 };

// One stage of the persistent decode kernel. Stages run in order in every block. A stage
// waits for the words it reads from earlier stages (tagged with the producing stage), not
// for the other blocks as a whole.
struct MegaStage {
  int kind;
  // MK_GEMV: Y[n] = epilogue(W[n] . x) for n < N, x built from `in`; bf16 W [N(+pair)][K]
  const __nv_bfloat16 *W;
  int N, K;
  int R;          // rows per streamed chunk
  long pair;      // > 0: SwiGLU, up rows at n + pair
  GemvIn in;
  float *Y;
  unsigned long long *Yt;  // non-null: Y goes here instead, each value tagged with the stage (index + 1)
  EpiArgs ep;
  // MK_ATTN: from the raw q/k/v/g row, RoPE + justnorm of q and k, q * s_q^2, the ring
  // write of the new k and v, windowed attention over `ring`, the gate, into z
  Ring ring;
  const unsigned long long *qkvg_t;  // the q/k/v/g row as tagged words of stage qtag - 1
  uint32_t qtag;
  const float *sq;
  int rope_kind;  // 0 sliding, 1 full (which RoPE base)
  const float *sg;
  unsigned long long *zt;  // z as tagged words (the stage's index + 1)
  float *part;    // [nk][maxblk][REP][hd + 2] item partials
  int maxblk;     // items per kv head at most
};

struct MegaArgs {
  const MegaStage *stages;
  int nstages;
  Dims d;
  Rows rows;                // one row
  double theta_s, theta_f;  // RoPE bases of sliding and full layers
  float *rope;              // [2][hd] cos | sin of the row's position
  int *sync;                // [1] RoPE entries ready, [2] blocks done; zero at launch
  int *actr;                // [nk] attention item arrivals; zero at launch
  // item partials of the per-head merges as tagged words (stage + 1): o [nh][MEGA_FLAGS][hd]
  // (query head h, item i), then (m, l) [nh][MEGA_FLAGS][2]; zero at launch
  unsigned long long *tpart;
  int *err;
  int32_t *seq_pos;         // advanced by `adv` once every block is done
  float *priv;              // per block: priv_stride floats of rows only that block reads
  int priv_stride;
  int adv_seq, adv_cnt;
  unsigned long long *trace;  // null, or [nstages][grid][MEGA_TRACE_EVENTS] %globaltimer stamps
  int prefetch_ahead;         // bytes per block the producer asks L2 for ahead of its copies
  int stall_lead;             // ... and up to this many while its slots are all taken
  uint32_t spin_limit;        // polls of a grid counter before a block gives up (error 6)
  int max_inflight;           // weight copies a block keeps in flight at most (0: one per free slot)
};

// Stamps per (stage, block) of the persistent kernel's optional trace: 0 stage entered,
// 1 stage descriptor copied, 2 input row built, 3 chunks or attention items done, 4 stage done;
// from the producer warp: 5 first chunk of the stage issued, 6 last chunk issued; 7 the
// stage's first chunk has landed (consumers); 8..11 SM cycles the first consumer thread
// spent over the stage's chunks waiting for a slot, reducing, at the team barrier, and in
// the epilogue (attention stages: copy wait, compute, arrival, merge); 12, 13 cycles of
// the attention merge until its partials are folded, and until its team sync (GEMV
// stages: the %globaltimer stamp once the input row's words were all in, and the poll
// rounds that took); 14 the stamp when the input row's first poll was issued. Attention
// stages reuse 2, 3, 5, 6, 7 for the block's last item: K/V copies issued, queries
// prepared, tiles landed, scores and values done, arrival counted.
constexpr int MEGA_TRACE_EVENTS = 16;
// Attention items of one kv head that the persistent kernel's per-head merge waits for at most.
constexpr int MEGA_FLAGS = 32;

// Bytes of dynamic shared memory and whether the device runs the kernel (one block per SM,
// cooperative launch).
size_t mega_smem_bytes(int hd);
bool mega_supported(int hd, int sms);
int mega_chunk_rows(int K, bool dual);  // rows (or gate/up row pairs) per streamed chunk; 0: too long
size_t mega_work_floats();              // shared scratch of a block: input row, tiles, merge
size_t mega_park_floats(bool dual);     // ... of it after a GEMV's input row: parked row sums
int mega_consumer_warps();
int mega_max_rows_per_block();          // rows of one GEMV a block takes at most
constexpr int MEGA_AK = 32;             // positions per attention item
cudaError_t launch_mega_decode(const MegaArgs &a, int grid, cudaStream_t s);

cudaError_t launch_advance(int32_t *seq_pos, const int32_t *seq, const int32_t *count, int n, cudaStream_t s);

// A step whose rows run in another order than the caller's: ids_out[r] = ids[perm[r]], and
// dst[perm[r]][.] = src[r][.] for `rows` rows of `width` floats (width a multiple of 4).
cudaError_t launch_gather_ids(const int32_t *ids, const int32_t *perm, int n, int32_t *out, cudaStream_t s);
cudaError_t launch_scatter_rows(const float *src, float *dst, const int32_t *perm, int rows, int width,
                                cudaStream_t s);

// dst[j][.] = src[idx[j]][.] for `rows` rows of `width` floats (width a multiple of 4).
cudaError_t launch_gather_rows(const float *src, float *dst, const int32_t *idx, int rows, int width,
                               cudaStream_t s);

// dory.rs fn top_prob of one row of n logits into *out (one block).
cudaError_t launch_top_prob(const float *logits, int n, float *out, cudaStream_t s);

// Forget the rows at positions >= n in every slot of one sequence: `table` holds per slot
// (tags offset, meta offset, ring rows) as int64 from the sequence's block; dropped[slot]
// gets the rows each slot lost; q8 slots' stored-row counters go down by it.
cudaError_t launch_rollback(char *seq_block, const long long *table, int nslots, int n, int nk, int q8,
                            int32_t *dropped, cudaStream_t s);

cudaError_t launch_ring_write_f32(const float *k, const float *v, int n, int pos0, Dims d, Ring ring, int seq,
                                  cudaStream_t s);

}  // namespace dory
