// The C ABI of include/dory.h: the handle, weight residency, KV rings and the launch
// sequence of one forward step (dory.rs fn forward_host / fn stack for one chunk, or
// one decode row per sequence).
#include <algorithm>
#include <array>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <unordered_map>
#include <vector>

#include "../../include/dory.h"
#include "kernels.h"

using namespace dory;

namespace {

thread_local std::string g_err;

int fail(int code, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

#define CK(call)                                                                          \
  do {                                                                                    \
    cudaError_t e_ = (call);                                                              \
    if (e_ != cudaSuccess) return fail(DORY_ECUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
  } while (0)

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

constexpr int KEYS_PER_SPLIT = 128;
// arrays of a step's row table: seq, off, advance seq, advance count, order, head rows
constexpr int ROW_TABLE = 6;
constexpr int RING_EXTRA = 64 + 448;  // a chunk and the rewind slack (gpu_metal/dory.rs fn run)

struct LayerDev {
  bool attn = false, sliding = false, rec = false, out = false;
  int ordinal = -1;
  void *wqkvg = nullptr, *wo = nullptr, *wgu = nullptr, *wdown = nullptr;
  float *sq = nullptr, *sg = nullptr, *alpha = nullptr, *msg = nullptr, *msu = nullptr;
};

struct TcW {
  CUtensorMap map;
  int N = 0, K = 0, splits = 1;
  long pair = 0;
  unsigned long long *trace = nullptr;  // DORY_TC_TRACE: the last launch's block timeline
  int trace_grid = 0;                   // blocks of that launch
};
constexpr int TC_TRACE_BLOCKS = 1024;

// Steps with at least this many rows take the tensor-core kernel with the step rows as the
// MMA's M side and bf16 activations (below it the weights stream once for a thin row block).
constexpr int TC_BIG_ROWS = 256;
constexpr int TC_BIG_CTRS = 4096;  // tile counters of launch_tc_gemm_big's split K
// Rows of dory_prefill's input/output-block steps over f32 rings when the bf16-activation
// tcgen05 kernel runs their projections (their attention goes in ring-sized pieces).
constexpr int PREFILL_ROWS = 4096;

int bn_index(int bn) { return bn <= 16 ? 0 : bn <= 32 ? 1 : bn <= 64 ? 2 : bn <= 128 ? 3 : 4; }

struct Plan {
  cudaGraphExec_t exec = nullptr;
  uint64_t used = 0;  // the handle's step counter at its last replay (least recently used goes first)
  int32_t *rt = nullptr;  // the captured step's own row table
  MegaStage *stages = nullptr;  // the persistent decode kernel's stage list (device)
  int launches = 0, gemm_launches = 0;
  float *h_last = nullptr;
};

// dory.rs struct ExitRate: the rate of tokens whose first read-out ended them; below 0.35 a
// token goes straight to its second pass, except one token in eight, which still reads out.
// f32 steps as the page writes them (the host code is built without contracted multiply-adds).
struct ExitRate {
  float rate = 1.0f;
  uint32_t tokens = 0;
  bool probe() {
    tokens += 1;  // wraps like the page's u32
    return rate >= 0.35f || tokens % 8 == 0;
  }
  void note(bool exited) {
    const float diff = (exited ? 1.0f : 0.0f) - rate;
    const float step = 0.1f * diff;
    rate = rate + step;
  }
};

struct OrdInfo {
  bool sliding = true, rec = false;
  int cap = 0, window = 0, slots = 1;
  size_t off = 0;  // slot 0 within a sequence block
  SlotLayout L;
};

}  // namespace

struct dory_handle {
  dory_config cfg{};
  std::string pattern;
  Dims dims{};
  int wdtype = 0;
  size_t esz = 4;
  cudaStream_t stream = nullptr;
  int Tmax = 64;          // rows of a step at most (the row table's stride)
  int Tstep = 64;         // ... of a decode or batched-prefill step, and of the logits buffers
  int prefill_rows = 0;   // rows of a whole prompt's input/output-block steps (dory_prefill); 0: chunk by chunk
  int piece_rows = 0;     // rows of such a step that join the rings and attend at once

  char *wmem = nullptr;
  size_t wbytes = 0;
  void *embed = nullptr, *head = nullptr;
  float *logit_scale = nullptr;
  std::vector<LayerDev> layers;
  std::vector<OrdInfo> ords;

  char *kvmem = nullptr;
  size_t seq_stride = 0, kv_bytes = 0;
  int max_splits = 1;

  float *h2 = nullptr, *h_last = nullptr;  // second hidden buffer (fused path), final rows
  int32_t *hctr = nullptr, *actr = nullptr;  // arrival counters of the fused kernels
  bool fused_ok = false;
  // persistent batch-1 decode: one block per SM; zeroed before each launch: counters
  // ([1] RoPE entries, [2] blocks done, [64..) per-kv-head attention item arrivals), then the
  // tagged words that stages hand on (q/k/v/g row, z, out, mlp, attention item partials)
  bool mega_ok = false;
  int sms = 0;
  int32_t *mega_sync = nullptr;
  size_t mega_sync_bytes = 0;
  unsigned long long *mega_tq = nullptr, *mega_tz = nullptr, *mega_to = nullptr, *mega_tm = nullptr;
  unsigned long long *mega_tp = nullptr;  // attention item partials of the per-head merges
  float *mega_priv = nullptr;  // per block: its hidden rows (2) and the loop's input row
  MegaStage *mega_stages = nullptr;  // stage list of the launches issued without graphs
  size_t mega_cap = 0;
  // optional trace of the persistent kernel (DORY_MEGA_TRACE=<file>, written at destroy)
  unsigned long long *mega_trace = nullptr;
  size_t mega_trace_stages = 0;
  std::string mega_trace_path;
  std::vector<int32_t> mega_trace_desc;  // kind, N, K per stage of the last traced step
  // L2 lead of the kernel's weight stream, bytes per block (DORY_MEGA_PREFETCH): about two
  // chunks measured best (1 chunk -0.5%, 5 chunks -1%, none -5%)
  int mega_prefetch = 32768;
  // the L2 lead the producer builds while its slots are all taken, bytes per block
  // (DORY_MEGA_LEAD; 0: no more than mega_prefetch): 256 KB measured 0.6% faster than none,
  // 512 KB the same
  int mega_lead = 262144;
  int mega_inflight = 0;  // cap on a block's weight copies in flight (DORY_MEGA_INFLIGHT)
  // tensor-core projections: weight maps per layer ([0] q/k/v/g or gate/up, [1] o or down)
  bool tc_ok = false;
  bool tc_big = true;  // steps of TC_BIG_ROWS rows and more take launch_tc_gemm_big (DORY_TC_BIG=0: never)
  std::vector<std::array<TcW, 2>> tcw;
  TcW tc_head;
  CUtensorMap xmap[3][2][5];  // activation rows (h, z, y) x (hi, lo) x tile rows 16..256
  Emit em_h{}, em_z{}, em_y{};
  CUtensorMap kvmap;          // f32 KV memory as [rows][hd] for the attention's tile copies
  bool kv_tma = false;
  KvMaps kvq;                 // q8 KV memory (hd = 128) for the attention's tile copies
  bool kv_tma_q8 = false;
  int32_t *dev_err = nullptr;  // set by a kernel whose bounded wait expired
  float *tc_ws = nullptr, *tc_ws_big = nullptr;
  int32_t *tc_ctr = nullptr, *tc_err = nullptr, *tc_ctr_big = nullptr;
  float *h = nullptr, *input = nullptr, *state = nullptr, *qkvg = nullptr, *z = nullptr, *out = nullptr,
        *mlp = nullptr, *logits = nullptr, *rope = nullptr, *part = nullptr, *kst = nullptr, *vst = nullptr;
  float *logits2 = nullptr;  // logits of a reordered step, before they go back to the caller's order
  int32_t *d_ids = nullptr, *d_ids2 = nullptr, *d_seq_pos = nullptr, *d_zero = nullptr;
  char *act = nullptr;
  char *tcmem = nullptr;

  cudaStream_t cap_stream = nullptr;  // graphs are captured here and replayed on `stream`
  bool use_graphs = true;
  std::unordered_map<std::string, Plan> plans;
  size_t max_plans = 256;  // captured steps kept at most (DORY_MAX_PLANS); the least recently used goes
  uint64_t steps = 0;
  int32_t *d_rows = nullptr;  // step table when graphs are off: seq, off, advance seq, count, order

  std::vector<ExitRate> exits;      // per sequence: the Conf gate's exit rate
  float *d_top = nullptr;           // the gate's top probability of the last read-out
  long long *slot_table = nullptr;  // per flat slot: tags offset, meta offset, ring rows (rollback)
  int32_t *dropped = nullptr;       // per flat slot: rows the last rollback dropped
  std::vector<int> seq_pos;     // host mirror of d_seq_pos
  std::vector<int> appended;    // rows appended per (seq, ordinal, slot)
  std::vector<int> slot_index;  // first flat slot index of each ordinal
  int n_flat_slots = 0;
  int logits_rows = 0, last_rows = 0;
  dory_stats st{};

  Ring ring(int ordinal, int slot) const {
    const OrdInfo &o = ords[ordinal];
    Ring r;
    r.base = kvmem;
    r.seq_stride = seq_stride;
    r.off = o.off + (size_t)slot * o.L.bytes;
    r.L = o.L;
    r.cap = o.cap;
    r.window = o.window;
    r.q8 = cfg.kv_quant == DORY_KV_Q8_2F;
    return r;
  }
  int &app(int seq, int ordinal, int slot) {
    return appended[(size_t)seq * n_flat_slots + slot_index[ordinal] + slot];
  }
};

namespace {

// An environment switch set to "0".
bool getenv_off(const char *name) {
  const char *e = getenv(name);
  return e && e[0] == '0';
}

int validate(const dory_config *c, std::string &pat) {
  if (!c) return fail(DORY_EINVAL, "config is NULL");
  if (c->hidden <= 0 || c->ffn <= 0 || c->vocab <= 0 || c->nh <= 0 || c->nk <= 0 || c->hd <= 0)
    return fail(DORY_EINVAL, "dimensions must be positive");
  if (c->nh % c->nk != 0) return fail(DORY_EINVAL, "nh (%d) must be a multiple of nk (%d)", c->nh, c->nk);
  const int rep = c->nh / c->nk;
  if (rep != 1 && rep != 2 && rep != 4 && rep != 8) return fail(DORY_EINVAL, "nh/nk must be 1, 2, 4 or 8");
  if (c->hd != 32 && c->hd != 64 && c->hd != 128) return fail(DORY_EINVAL, "hd must be 32, 64 or 128");
  if (c->hidden % 32 || c->ffn % 32) return fail(DORY_EINVAL, "hidden and ffn must be multiples of 32");
  if (c->hidden > 8192) return fail(DORY_EINVAL, "hidden above 8192");
  if (c->ffn > 32768 || c->nh * c->hd > 32768) return fail(DORY_EINVAL, "ffn or nh*hd above 32768");
  if (c->max_loops < 1 || c->max_loops > DORY_MAX_LOOPS)
    return fail(DORY_EINVAL, "max_loops=%d: want 1..%d", c->max_loops, DORY_MAX_LOOPS);
  if (c->window < 1) return fail(DORY_EINVAL, "window must be positive");
  if (c->full_window < 0) return fail(DORY_EINVAL, "full_window must be >= 0");
  if (c->kv_mode != DORY_KV_PER_LOOP && c->kv_mode != DORY_KV_LAST_LOOP) return fail(DORY_EINVAL, "kv_mode");
  if (c->kv_quant != DORY_KV_F32 && c->kv_quant != DORY_KV_Q8_2F) return fail(DORY_EINVAL, "kv_quant");
  if (c->weight_dtype != DORY_W_F32 && c->weight_dtype != DORY_W_BF16) return fail(DORY_EINVAL, "weight_dtype");
  if (c->max_batch < 1 || c->max_batch > DORY_MAX_BATCH) return fail(DORY_EINVAL, "max_batch 1..%d", DORY_MAX_BATCH);
  if (c->max_seqs < 1) return fail(DORY_EINVAL, "max_seqs must be positive");
  if (c->prompt_loops < 0) return fail(DORY_EINVAL, "prompt_loops must be >= 0");
  if (c->n_in < 0 || c->n_rec < 0 || c->n_out < 0) return fail(DORY_EINVAL, "block sizes must be >= 0");
  if (!c->layer_pattern) return fail(DORY_EINVAL, "layer_pattern is NULL");
  pat = c->layer_pattern;
  if ((int)pat.size() != c->n_in + c->n_rec + c->n_out)
    return fail(DORY_EINVAL, "layer_pattern has %zu layers, blocks give %d", pat.size(), c->n_in + c->n_rec + c->n_out);
  for (char ch : pat)
    if (ch != 'S' && ch != '*' && ch != '-') return fail(DORY_EINVAL, "layer_pattern char '%c'", ch);
  bool has_full = false;
  for (char ch : pat) has_full |= ch == '*';
  if (has_full && c->full_window == 0 && c->max_context < 1) return fail(DORY_EINVAL, "max_context must be positive");
  return DORY_OK;
}

int copy_in(void *dst, const void *src, size_t bytes, const char *what) {
  if (!src) return fail(DORY_EINVAL, "weight %s is NULL", what);
  CK(cudaMemcpy(dst, src, bytes, cudaMemcpyDefault));
  return DORY_OK;
}

void free_all(dory_t *d) {
  for (auto &kv : d->plans) {
    if (kv.second.exec) cudaGraphExecDestroy(kv.second.exec);
    if (kv.second.rt) cudaFree(kv.second.rt);
    if (kv.second.stages) cudaFree(kv.second.stages);
  }
  if (d->mega_stages) cudaFree(d->mega_stages);
  d->mega_stages = nullptr;
  if (d->mega_trace) cudaFree(d->mega_trace);
  if (d->mega_priv) cudaFree(d->mega_priv);
  d->mega_trace = nullptr;
  for (auto &pr : d->tcw)
    for (TcW &w : pr)
      if (w.trace) cudaFree(w.trace), w.trace = nullptr;
  if (d->tc_head.trace) cudaFree(d->tc_head.trace), d->tc_head.trace = nullptr;
  d->mega_cap = 0;
  d->plans.clear();
  if (d->cap_stream) cudaStreamDestroy(d->cap_stream);
  d->cap_stream = nullptr;
  if (d->wmem) cudaFree(d->wmem);
  if (d->kvmem) cudaFree(d->kvmem);
  if (d->act) cudaFree(d->act);
  if (d->tcmem) cudaFree(d->tcmem);
  d->wmem = d->kvmem = d->act = d->tcmem = nullptr;
}

int reset_seq(dory_t *d, int seq) {
  char *blk = d->kvmem + (size_t)seq * d->seq_stride;
  CK(cudaMemsetAsync(blk, 0, d->seq_stride, d->stream));
  for (size_t o = 0; o < d->ords.size(); o++)
    for (int s = 0; s < d->ords[o].slots; s++) {
      Ring r = d->ring((int)o, s);
      CK(cudaMemsetAsync(blk + r.off + r.L.tags, 0xFF, (size_t)r.cap * 4, d->stream));
    }
  CK(cudaMemsetAsync(d->d_seq_pos + seq, 0, 4, d->stream));
  d->seq_pos[seq] = 0;
  if ((size_t)seq < d->exits.size()) d->exits[seq] = ExitRate{};
  for (int i = 0; i < d->n_flat_slots; i++) d->appended[(size_t)seq * d->n_flat_slots + i] = 0;
  return DORY_OK;
}

// The rows of one step: row r is sequence hseq[r] at position seq_pos[hseq[r]] + hoff[r];
// aseq/acnt are the position advances at the step's end. `loops` recurrent passes; logits
// for head_rows rows starting at row head_from.
// `resume`: the second pass of an early-exit gate that stayed (dory.rs fn stack): no
// embedding or input block; h = (state + input)^ from the saved rows, recurrent passes
// first_loop..loops-1, and the output block rewrites the rows its read-out appended.
// `rl`: per-row loop counts (empty: every row runs `loops`), sorted from the most loops down
// so that the rows a pass runs are a prefix; `perm[r]` is the caller's index of row r (ids
// are gathered into this order, logits and hidden rows scattered back).
// `do_in` / `do_out`: run the input block (with the embedding) / the output block; a whole
// prompt runs its input and output blocks over many chunks' rows at once and its recurrent
// block chunk by chunk, each chunk's rows at row offset `h0` of the hidden buffers.
struct StepArgs {
  int T = 0, loops = 1, head_from = 0, head_rows = 0, first_loop = 0, h0 = 0;
  bool resume = false, do_in = true, do_out = true;
  std::vector<int> hseq, hoff, aseq, acnt, rl, perm;
  // rows whose logits are read when they are not one run (the last row of each sequence of a
  // batched prefill): the head covers rows [0, T) and these rows are gathered, in order
  std::vector<int> head_pick;
  // rows that run pass i
  int active(int i) const {
    if (i >= loops) return 0;
    if (rl.empty()) return T;
    int n = 0;
    while (n < T && rl[n] > i) n++;
    return n;
  }
  std::string key() const {
    std::string k = std::to_string(T) + ":" + std::to_string(loops) + ":" + std::to_string(head_from) + ":" +
                    std::to_string(head_rows) + ":" + std::to_string(first_loop) + (resume ? "r" : "") +
                    (do_in ? "i" : "") + (do_out ? "o" : "") + std::to_string(h0) + "|";
    for (int i = 0; i < T; i++) k += std::to_string(hseq[i]) + "," + std::to_string(hoff[i]) + ";";
    if (!rl.empty()) {
      k += "L";
      for (int i = 0; i < T; i++) k += std::to_string(rl[i]) + "," + std::to_string(perm[i]) + ";";
    }
    if (!head_pick.empty()) {
      k += "H";
      for (int x : head_pick) k += std::to_string(x) + ";";
    }
    return k;
  }
};

// Host-side accounting of a step: algorithmic bytes and the rows each slot appends.
void account(dory_t *d, const StepArgs &a) {
  const dory_config &c = d->cfg;
  const Dims dm = d->dims;
  const bool q8 = c.kv_quant == DORY_KV_Q8_2F;
  const size_t kv_row_bytes = q8 ? (size_t)dm.hd * 2 + (dm.hd / 32) * 4 + 4 : (size_t)dm.hd * 8;
  const int q_size = dm.nh * dm.hd, kv_size = dm.nk * dm.hd;
  uint64_t wb = 0, kr = 0, kw = 0, fl = 0;
  auto layer = [&](int li, int loop_i) {
    const LayerDev &L = d->layers[li];
    const int rows = L.rec ? a.active(loop_i) : a.T;
    if (L.attn) {
      const uint64_t params = (uint64_t)(2 * q_size + 2 * kv_size) * dm.hidden + (uint64_t)dm.hidden * q_size;
      wb += params * d->esz;
      fl += 2 * params * rows;
      const int sl = (c.kv_mode == DORY_KV_PER_LOOP && L.rec) ? loop_i : 0;
      const bool rewrite = (c.kv_mode == DORY_KV_LAST_LOOP && (L.rec || L.out) && loop_i > 0) || (a.resume && L.out);
      const OrdInfo &o = d->ords[L.ordinal];
      for (int r = 0; r < rows; r++) {
        const long p = (long)d->seq_pos[a.hseq[r]] + a.hoff[r];
        const long keys = o.window == INT_MAX ? p + 1 : std::min<long>(o.window, p + 1);
        kr += (uint64_t)keys * dm.nk * kv_row_bytes;
        if (!rewrite) d->app(a.hseq[r], L.ordinal, sl)++;
      }
      kw += (uint64_t)rows * dm.nk * kv_row_bytes;
    } else {
      wb += (uint64_t)3 * dm.ffn * dm.hidden * d->esz;
      fl += (uint64_t)6 * dm.ffn * dm.hidden * rows;
    }
  };
  const int n_in = c.n_in, n_rec = c.n_rec, n_all = (int)d->layers.size();
  if (!a.resume && a.do_in)
    for (int li = 0; li < n_in; li++) layer(li, 0);
  for (int i = a.first_loop; i < a.loops; i++)
    for (int li = n_in; li < n_in + n_rec; li++) layer(li, i);
  if (a.do_out)
    for (int li = n_in + n_rec; li < n_all; li++) layer(li, a.resume ? 1 : 0);
  if (a.head_rows > 0) {
    wb += (uint64_t)dm.vocab * dm.hidden * d->esz;
    fl += (uint64_t)2 * dm.vocab * dm.hidden * a.head_rows;
  }
  d->st.weight_bytes = wb;
  d->st.flops = fl;
  d->st.kv_read_bytes = kr;
  d->st.kv_write_bytes = kw;
}

// 64-position blocks the attention of the step's rows covers: the most over the rows.
int tma_splits(dory_t *d, const StepArgs &a, const Ring &ring) {
  int nb = 1;
  for (int r = 0; r < a.T; r++) {
    const long p = (long)d->seq_pos[a.hseq[r]] + a.hoff[r];
    const long lo = ring.window == INT_MAX ? 0 : std::max<long>(p + 1 - ring.window, 0);
    nb = std::max<int>(nb, (int)(p / 64 - lo / 64 + 1));
  }
  return nb;
}

// Issue every launch of one step on stream s. `rt` holds the device row table: seq[Tmax],
// off[Tmax], advance seq[Tmax], advance count[Tmax]. With fixed_splits the attention grids
// cover the whole window whatever the positions (for replayed graphs).
int issue_step(dory_t *d, const StepArgs &a, int32_t *rt, bool fixed_splits, cudaStream_t s, int *launches,
               int *gemm_launches) {
  const dory_config &c = d->cfg;
  const Dims dm = d->dims;
  const int T = a.T;
  // runs of rows that are consecutive positions of one sequence (prefill chunks); when some
  // run has two rows or more, each run's attention takes the chunk kernel
  std::vector<std::pair<int, int>> segs;  // (first row, rows)
  for (int r = 0; r < T; r++) {
    if (r > 0 && a.hseq[r] == a.hseq[r - 1] && a.hoff[r] == a.hoff[r - 1] + 1) segs.back().second++;
    else segs.push_back({r, 1});
  }
  const bool chunk_rows = (int)segs.size() < T && !getenv_off("DORY_CHUNK_ATTN");
  Rows rows;
  rows.seq = rt;
  rows.off = rt + d->Tmax;
  rows.seq_pos = d->d_seq_pos;
  rows.n = T;
  int nl = 0, ng = 0;
  const int q_size = dm.nh * dm.hd, kv_size = dm.nk * dm.hd;
  const int ldq = 2 * q_size + 2 * kv_size;
  long pmax = 0;
  for (int r = 0; r < T; r++) pmax = std::max(pmax, (long)d->seq_pos[a.hseq[r]] + a.hoff[r]);
  const bool q8 = c.kv_quant == DORY_KV_Q8_2F;

  const bool tc = d->tc_ok && T >= 5;
  const bool ragged = !a.rl.empty();
  const int32_t *perm = rt + 4 * d->Tmax;
  const int32_t *ids = d->d_ids;
  if (ragged) {  // the caller's ids in the step's row order
    CK(launch_gather_ids(d->d_ids, perm, T, d->d_ids2, s));
    nl++;
    ids = d->d_ids2;
  }
  // the step's hidden rows: rows h0.. of the hidden, input and state buffers (and of the
  // activations' bf16 halves)
  const size_t ho = (size_t)a.h0 * dm.hidden;
  float *const H = d->h + ho, *const IN = d->input + ho, *const ST = d->state + ho;
  const Emit EH = tc ? Emit{d->em_h.hi + ho, d->em_h.lo + ho} : Emit{nullptr, nullptr};
  const bool embed = a.do_in && !a.resume;
  CK(launch_embed_rope(ids, d->embed, d->wdtype, dm, rows, c.rope_theta_sliding, c.rope_theta_full,
                       embed ? H : nullptr, d->rope, EH, s));
  nl++;
  auto tcg = [&](const TcW &w, int xbuf, int rowsT, int t_base, float *Y, int ldy, EpiArgs ep) -> int {
    TcGemm g;
    g.tmW = w.map;
    if (rowsT >= TC_BIG_ROWS && d->tc_big) {  // a dense contraction: step rows as the MMA's M side
      g.tmXh = d->xmap[xbuf][0][bn_index(128)];
      g.N = w.N;
      g.K = w.K;
      g.pair_rows = w.pair;
      g.err = d->tc_err;
      g.ws_big = d->tc_ws_big;
      g.ctr_big = d->tc_ctr_big;
      g.ctr_slots = TC_BIG_CTRS;
      g.sms = d->sms;
      CK(launch_tc_gemm_big(g, rowsT, t_base, Y, ldy, ep, true, s));
      nl++;
      ng++;
      return DORY_OK;
    }
    const int bi = bn_index(tc_tile_rows(rowsT));
    g.tmXh = d->xmap[xbuf][0][bi];
    g.tmXl = d->xmap[xbuf][1][bi];
    g.N = w.N;
    g.K = w.K;
    g.splits = (rowsT + tc_tile_rows(rowsT) - 1) / tc_tile_rows(rowsT) > 1 ? 1 : w.splits;
    g.pair_rows = w.pair;
    g.ws = d->tc_ws;
    g.ctr = d->tc_ctr;
    g.err = d->tc_err;
    g.trace = w.trace;
    if (w.trace) {
      const int bn = tc_tile_rows(rowsT);
      const_cast<TcW &>(w).trace_grid = ((w.N + 127) / 128) * g.splits * ((rowsT + bn - 1) / bn);
    }
    CK(launch_tc_gemm(g, rowsT, t_base, Y, ldy, ep, true, s));
    nl++;
    ng++;
    return DORY_OK;
  };
  auto gemm = [&](const void *W, int N, int K, const float *X, int ldx, int Tr, float *Y, int ldy,
                  EpiArgs ep) -> int {
    CK(launch_gemm(W, d->wdtype, N, K, X, ldx, Tr, Y, ldy, ep, s));
    nl++;
    ng++;
    return DORY_OK;
  };
  // The residual of rows [0, Tr) with the loop mix `mix` for rows [0, Tsplit) and MIX_END for
  // rows [Tsplit, Tr) (rows whose last pass this is, when loop counts differ per row).
  auto resid = [&](const float *alpha, int mix, int Tr, int Tsplit, int do_res) -> int {
    const Emit em = EH;
    if (Tsplit > 0) {
      CK(launch_residual(H, d->out, alpha, Tsplit, dm.hidden, mix, IN, ST, do_res, em, s));
      nl++;
    }
    if (Tr > Tsplit) {
      const size_t o = (size_t)Tsplit * dm.hidden;
      const Emit e2 = em.hi ? Emit{em.hi + o, em.lo + o} : em;
      CK(launch_residual(H + o, d->out + o, alpha, Tr - Tsplit, dm.hidden, MIX_END, IN + o, ST + o,
                         do_res, e2, s));
      nl++;
    }
    return DORY_OK;
  };
  auto layer = [&](int li, int loop_i, int mix, int Tr, int Tsplit) -> int {
    const LayerDev &L = d->layers[li];
    int rc;
    Rows rows_l = rows;
    rows_l.n = Tr;
    if (L.attn) {
      const int sl = (c.kv_mode == DORY_KV_PER_LOOP && L.rec) ? loop_i : 0;
      const bool rewrite = (c.kv_mode == DORY_KV_LAST_LOOP && (L.rec || L.out) && loop_i > 0) || (a.resume && L.out);
      Ring ring = d->ring(L.ordinal, sl);
      EpiArgs ep{EPI_STORE, nullptr, nullptr, 0};
      if (tc) {
        if ((rc = tcg(d->tcw[li][0], 0, Tr, a.h0, d->qkvg, ldq, ep))) return rc;
      } else if ((rc = gemm(L.wqkvg, ldq, dm.hidden, H, dm.hidden, Tr, d->qkvg, ldq, ep))) {
        return rc;
      }
      // prefill chunks: a chunk's rows share every key block (the merge also row-normalises z);
      // a step of more rows than a ring takes at once prepares and attends piece by piece
      const bool chunked = chunk_rows && Tr == T && !q8 && (dm.hd == 64 || dm.hd == 128);
      const bool pieces = chunked && T > d->piece_rows;
      if (!pieces) {
        CK(launch_prep(d->qkvg, ldq, dm, rows_l, d->rope, L.sliding ? 0 : 1, L.sq, ring, d->kst, d->vst, s));
        nl++;
      }
      if (q8) {
        CK(launch_q8_append(d->kst, d->vst, kv_size, dm, rows_l, ring, rewrite ? 1 : 0, s));
        nl++;
      }
      const long wmax = ring.window == INT_MAX ? (long)ring.cap : std::min<long>(ring.window, ring.cap);
      const long keys = fixed_splits ? wmax : std::min<long>(wmax, pmax + 1);
      const int splits = (int)((keys + KEYS_PER_SPLIT - 1) / KEYS_PER_SPLIT);
      if (splits > d->max_splits) return fail(DORY_ERANGE, "attention needs %d splits (max %d)", splits, d->max_splits);
      bool z_normed = false;
      if (chunked) {
        for (const auto &sg_ : segs)
          for (int r0 = sg_.first; r0 < sg_.first + sg_.second; r0 += d->piece_rows) {
            const int n = std::min(d->piece_rows, sg_.first + sg_.second - r0);
            const int nkb = attn_chunk_blocks(wmax, n);
            if (nkb > d->max_splits) return fail(DORY_ERANGE, "chunk attention needs %d key blocks", nkb);
            Rows rs = rows_l;
            rs.seq = rows_l.seq + r0;
            rs.off = rows_l.off + r0;
            rs.n = n;
            if (pieces) {
              CK(launch_prep(d->qkvg + (size_t)r0 * ldq, ldq, dm, rs, d->rope + (size_t)r0 * 2 * dm.hd,
                             L.sliding ? 0 : 1, L.sq, ring, d->kst, d->vst, s));
              nl++;
            }
            const size_t zo = (size_t)r0 * q_size;
            const Emit ez = tc ? Emit{d->em_z.hi + zo, d->em_z.lo + zo} : Emit{nullptr, nullptr};
            CK(launch_attention_chunk(d->qkvg + (size_t)r0 * ldq, ldq, dm, rs, ring, nkb, d->part, L.sg, d->z + zo,
                                      ez, d->dev_err, s));
            nl += 2;
          }
        z_normed = true;
      } else if ((q8 ? dm.hd == 128 && !getenv_off("DORY_STREAM_Q8") : (dm.hd == 64 || dm.hd == 128)) &&
                 !getenv_off("DORY_STREAM_ATTN")) {
        // rows of separate sequences: each (row, kv head) streams its own window
        int ssp = attn_stream_splits(wmax, Tr, dm.nk, d->sms);
        if (const char *e = getenv("DORY_STREAM_SPLIT")) {  // a fixed split (0 or 1: none)
          const long tiles = (wmax + 31) / 32 + 1;             // 32-position tiles of the window
          ssp = (int)std::max(1L, std::min<long>(atoi(e), tiles / 4));
        }
        ssp = std::min(ssp, d->max_splits);
        CK(launch_attention_stream(d->qkvg, ldq, dm, rows_l, ring, L.sg, d->z, d->dev_err, ssp, d->part, d->actr,
                                   s));
        nl += 1;
      } else if (d->kv_tma || d->kv_tma_q8) {
        const int tsp = fixed_splits ? attn_tma_splits(wmax) : tma_splits(d, a, ring);
        if (d->kv_tma)
          CK(launch_attention_tma(d->kvmap, d->qkvg, ldq, dm, rows_l, ring, tsp, d->part, L.sg, d->z, d->actr,
                                  d->dev_err, true, s));
        else
          CK(launch_attention_tma_q8(d->kvq, d->qkvg, ldq, dm, rows_l, ring, tsp, d->part, L.sg, d->z, d->actr,
                                     d->dev_err, true, s));
        nl += 1;
      } else if (tc) {
        CK(launch_attention_fused(d->qkvg, ldq, dm, rows_l, ring, splits, KEYS_PER_SPLIT, d->part, L.sg, d->z,
                                  d->actr, true, s));
        nl += 1;
      } else {
        CK(launch_attention(d->qkvg, ldq, dm, rows_l, ring, splits, KEYS_PER_SPLIT, d->part, L.sg, d->z, s));
        nl += 2;
      }
      if (!z_normed) {
        CK(launch_rownorm(d->z, Tr, q_size, q_size, tc ? d->em_z : Emit{nullptr, nullptr}, s));
        nl++;
      }
      if (tc) {
        if ((rc = tcg(d->tcw[li][1], 1, Tr, 0, d->out, dm.hidden, ep))) return rc;
      } else if ((rc = gemm(L.wo, dm.hidden, q_size, d->z, q_size, Tr, d->out, dm.hidden, ep))) {
        return rc;
      }
    } else {
      EpiArgs ep{EPI_SILU, L.msg, L.msu, (long)dm.ffn};
      if (tc) {
        if ((rc = tcg(d->tcw[li][0], 0, Tr, a.h0, d->mlp, dm.ffn, ep))) return rc;
      } else if ((rc = gemm(L.wgu, dm.ffn, dm.hidden, H, dm.hidden, Tr, d->mlp, dm.ffn, ep))) {
        return rc;
      }
      CK(launch_rownorm(d->mlp, Tr, dm.ffn, dm.ffn, tc ? d->em_y : Emit{nullptr, nullptr}, s));
      nl++;
      EpiArgs e2{EPI_STORE, nullptr, nullptr, 0};
      if (tc) {
        if ((rc = tcg(d->tcw[li][1], 2, Tr, 0, d->out, dm.hidden, e2))) return rc;
      } else if ((rc = gemm(L.wdown, dm.hidden, dm.ffn, d->mlp, dm.ffn, Tr, d->out, dm.hidden, e2))) {
        return rc;
      }
    }
    return resid(L.alpha, mix, Tr, Tsplit, 1);
  };
  auto mix_only = [&](int mix, int Tr, int Tsplit) -> int { return resid(nullptr, mix, Tr, Tsplit, 0); };

  int rc;
  const int n_in = c.n_in, n_rec = c.n_rec, n_all = (int)d->layers.size();
  if (a.resume) {
    if ((rc = mix_only(MIX_RESUME, T, T))) return rc;
  } else if (a.do_in) {
    for (int li = 0; li < n_in; li++)
      if ((rc = layer(li, 0, li == n_in - 1 ? MIX_BEGIN : MIX_NONE, T, T))) return rc;
    if (n_in == 0 && (rc = mix_only(MIX_BEGIN, T, T))) return rc;
  }
  // pass i runs the rows that still loop (a prefix); at its end those with more passes to go
  // mix for the next pass and the others end (state = h^, h = state)
  for (int i = a.first_loop; i < a.loops; i++) {
    const int Ti = a.active(i), Tn = a.active(i + 1);
    for (int li = n_in; li < n_in + n_rec; li++) {
      const bool last = li == n_in + n_rec - 1;
      if ((rc = layer(li, i, last ? MIX_LOOP : MIX_NONE, Ti, last ? Tn : Ti))) return rc;
    }
    if (n_rec == 0 && (rc = mix_only(MIX_LOOP, Ti, Tn))) return rc;
  }
  if (a.do_out)
    for (int li = n_in + n_rec; li < n_all; li++)
      if ((rc = layer(li, a.resume ? 1 : 0, MIX_NONE, T, T))) return rc;
  if (a.head_rows > 0) {
    EpiArgs ep{EPI_SCALE, d->logit_scale, nullptr, 0};
    const bool pick = !a.head_pick.empty();
    float *lg = ragged || pick ? d->logits2 : d->logits;
    if (tc && a.head_rows >= 5) {
      if ((rc = tcg(d->tc_head, 0, a.head_rows, a.h0 + a.head_from, lg, dm.vocab, ep))) return rc;
    } else {
      CK(launch_gemm(d->head, d->wdtype, dm.vocab, dm.hidden, H + (size_t)a.head_from * dm.hidden, dm.hidden,
                     a.head_rows, lg, dm.vocab, ep, s));
      nl++;
      ng++;
    }
    if (ragged) {  // logits rows back in the caller's order
      CK(launch_scatter_rows(lg, d->logits, perm, T, dm.vocab, s));
      nl++;
    }
    if (pick) {  // the wanted rows, in order
      CK(launch_gather_rows(lg, d->logits, rt + 5 * d->Tmax, (int)a.head_pick.size(), dm.vocab, s));
      nl++;
    }
  }
  if (ragged) {  // and the final hidden rows
    CK(launch_scatter_rows(H, d->h2, perm, T, dm.hidden, s));
    nl++;
    d->h_last = d->h2;
  }
  CK(launch_advance(d->d_seq_pos, rt + 2 * d->Tmax, rt + 3 * d->Tmax, (int)a.aseq.size(), s));
  nl++;
  *launches = nl;
  *gemm_launches = ng;
  return DORY_OK;
}

// The fused launch sequence for steps of up to 4 rows: per attention sub-layer the q/k/v/g
// GEMV (its prologue takes the previous residual and loop mix, its last block per head the
// RoPE/norm/ring write), [the q8 append], attention with the merge and gate, the O GEMV
// (row norm in its prologue); per MLP the gate/up GEMV with SwiGLU and the down GEMV.
// Kernels after the first use programmatic dependent launch.
int issue_step_fused(dory_t *d, const StepArgs &a, int32_t *rt, bool fixed_splits, cudaStream_t s, int *launches,
                     int *gemm_launches) {
  const dory_config &c = d->cfg;
  const Dims dm = d->dims;
  const int T = a.T;
  Rows rows;
  rows.seq = rt;
  rows.off = rt + d->Tmax;
  rows.seq_pos = d->d_seq_pos;
  rows.n = T;
  int nl = 0, ng = 0;
  const int q_size = dm.nh * dm.hd, kv_size = dm.nk * dm.hd;
  const int ldq = 2 * q_size + 2 * kv_size;
  long pmax = 0;
  for (int r = 0; r < T; r++) pmax = std::max(pmax, (long)d->seq_pos[a.hseq[r]] + a.hoff[r]);
  const bool q8 = c.kv_quant == DORY_KV_Q8_2F;
  CK(launch_embed_rope(d->d_ids, d->embed, d->wdtype, dm, rows, c.rope_theta_sliding, c.rope_theta_full, d->h,
                       d->rope, Emit{nullptr, nullptr}, s));
  nl++;
  float *cur = d->h, *other = d->h2;
  struct {
    bool on = false;
    const float *alpha = nullptr;
    int mix = MIX_NONE;
    bool resume = false;
  } pend;
  pend.resume = a.resume;
  auto first_in = [&]() {
    GemvIn g{};
    if (pend.resume) {  // h = (state + input)^ from the saved rows
      g.mode = IN_RESID;
      g.src = d->state;
      g.ld = dm.hidden;
      g.mix = MIX_RESUME;
      g.h_dst = other;
      g.input = d->input;
      g.state = d->state;
      std::swap(cur, other);
      pend.resume = false;
      return g;
    }
    if (!pend.on) {
      g.mode = IN_PLAIN;
      g.src = cur;
      g.ld = dm.hidden;
      return g;
    }
    g.mode = IN_RESID;
    g.src = cur;
    g.ld = dm.hidden;
    g.out = d->out;
    g.alpha = pend.alpha;
    g.mix = pend.mix;
    g.h_dst = other;
    g.input = d->input;
    g.state = d->state;
    std::swap(cur, other);
    pend.on = false;
    return g;
  };
  HeadEpi none{};
  none.enabled = 0;
  auto layer = [&](int li, int loop_i, int mix) -> int {
    const LayerDev &L = d->layers[li];
    if (L.attn) {
      const int sl = (c.kv_mode == DORY_KV_PER_LOOP && L.rec) ? loop_i : 0;
      const bool rewrite = (c.kv_mode == DORY_KV_LAST_LOOP && (L.rec || L.out) && loop_i > 0) || (a.resume && L.out);
      Ring ring = d->ring(L.ordinal, sl);
      HeadEpi he{};
      he.enabled = 1;
      he.counters = d->hctr;
      he.d = dm;
      he.rows = rows;
      he.rope = d->rope;
      he.kind = L.sliding ? 0 : 1;
      he.sq = L.sq;
      he.ring = ring;
      he.kst = d->kst;
      he.vst = d->vst;
      EpiArgs ep{EPI_STORE, nullptr, nullptr, 0};
      CK(launch_gemv_fused(L.wqkvg, d->wdtype, ldq, dm.hidden, T, first_in(), d->qkvg, ldq, ep, he, d->dev_err, true, s));
      nl++;
      ng++;
      if (q8) {
        CK(launch_q8_append(d->kst, d->vst, kv_size, dm, rows, ring, rewrite ? 1 : 0, s));
        nl++;
      }
      const long wmax = ring.window == INT_MAX ? (long)ring.cap : std::min<long>(ring.window, ring.cap);
      const long keys = fixed_splits ? wmax : std::min<long>(wmax, pmax + 1);
      const int splits = (int)((keys + KEYS_PER_SPLIT - 1) / KEYS_PER_SPLIT);
      if (splits > d->max_splits) return fail(DORY_ERANGE, "attention needs %d splits (max %d)", splits, d->max_splits);
      if (d->kv_tma || d->kv_tma_q8) {
        const int tsp = fixed_splits ? attn_tma_splits(wmax) : tma_splits(d, a, ring);
        if (d->kv_tma)
          CK(launch_attention_tma(d->kvmap, d->qkvg, ldq, dm, rows, ring, tsp, d->part, L.sg, d->z, d->actr,
                                  d->dev_err, true, s));
        else
          CK(launch_attention_tma_q8(d->kvq, d->qkvg, ldq, dm, rows, ring, tsp, d->part, L.sg, d->z, d->actr,
                                     d->dev_err, true, s));
      } else {
        CK(launch_attention_fused(d->qkvg, ldq, dm, rows, ring, splits, KEYS_PER_SPLIT, d->part, L.sg, d->z, d->actr,
                                  true, s));
      }
      nl++;
      GemvIn in{};
      in.mode = IN_NORM;
      in.src = d->z;
      in.ld = q_size;
      CK(launch_gemv_fused(L.wo, d->wdtype, dm.hidden, q_size, T, in, d->out, dm.hidden, ep, none, d->dev_err, true, s));
      nl++;
      ng++;
    } else {
      EpiArgs ep{EPI_SILU, L.msg, L.msu, (long)dm.ffn};
      CK(launch_gemv_fused(L.wgu, d->wdtype, dm.ffn, dm.hidden, T, first_in(), d->mlp, dm.ffn, ep, none, d->dev_err, true, s));
      GemvIn in{};
      in.mode = IN_NORM;
      in.src = d->mlp;
      in.ld = dm.ffn;
      EpiArgs e2{EPI_STORE, nullptr, nullptr, 0};
      CK(launch_gemv_fused(L.wdown, d->wdtype, dm.hidden, dm.ffn, T, in, d->out, dm.hidden, e2, none, d->dev_err, true, s));
      nl += 2;
      ng += 2;
    }
    pend.on = true;
    pend.alpha = L.alpha;
    pend.mix = mix;
    return DORY_OK;
  };
  int rc;
  const int n_in = c.n_in, n_rec = c.n_rec, n_all = (int)d->layers.size();
  if (!a.resume)
    for (int li = 0; li < n_in; li++)
      if ((rc = layer(li, 0, li == n_in - 1 ? MIX_BEGIN : MIX_NONE))) return rc;
  for (int i = a.first_loop; i < a.loops; i++) {
    const int m = i == a.loops - 1 ? MIX_END : MIX_LOOP;
    for (int li = n_in; li < n_in + n_rec; li++)
      if ((rc = layer(li, i, li == n_in + n_rec - 1 ? m : MIX_NONE))) return rc;
  }
  for (int li = n_in + n_rec; li < n_all; li++)
    if ((rc = layer(li, a.resume ? 1 : 0, MIX_NONE))) return rc;
  EpiArgs eh{EPI_SCALE, d->logit_scale, nullptr, 0};
  if (a.head_rows == T && a.head_from == 0) {
    CK(launch_gemv_fused(d->head, d->wdtype, dm.vocab, dm.hidden, T, first_in(), d->logits, dm.vocab, eh, none, d->dev_err,
                         true, s));
    nl++;
    ng++;
  } else {
    CK(launch_residual(cur, d->out, pend.alpha, T, dm.hidden, pend.mix, d->input, d->state, 1,
                       Emit{nullptr, nullptr}, s));
    nl++;
    pend.on = false;
    if (a.head_rows > 0) {
      CK(launch_gemm(d->head, d->wdtype, dm.vocab, dm.hidden, cur + (size_t)a.head_from * dm.hidden, dm.hidden,
                     a.head_rows, d->logits, dm.vocab, eh, s));
      nl++;
      ng++;
    }
  }
  d->h_last = cur;
  CK(launch_advance(d->d_seq_pos, rt + 2 * d->Tmax, rt + 3 * d->Tmax, (int)a.aseq.size(), s));
  nl++;
  *launches = nl;
  *gemm_launches = ng;
  return DORY_OK;
}

int issue_any(dory_t *d, const StepArgs &a, int32_t *rt, bool fixed_splits, cudaStream_t s, int *nl, int *ng) {
  if (d->fused_ok && a.T <= 4 && a.rl.empty() && a.head_pick.empty() && a.do_in && a.do_out && a.h0 == 0)
    return issue_step_fused(d, a, rt, fixed_splits, s, nl, ng);
  d->h_last = d->h;
  return issue_step(d, a, rt, fixed_splits, s, nl, ng);
}

// The persistent kernel runs steps of one row that end with that row's logits.
bool use_mega(const dory_t *d, const StepArgs &a) {
  return d->mega_ok && a.T == 1 && a.head_rows == 1 && a.head_from == 0 && a.aseq.size() == 1 && a.do_in &&
         a.do_out && a.h0 == 0;
}

// The stage list of a one-row step, in the order of issue_step_fused's launches.
int mega_build(dory_t *d, const StepArgs &a, int32_t *rt, std::vector<MegaStage> &out, float **h_last) {
  const dory_config &c = d->cfg;
  const Dims dm = d->dims;
  const int q_size = dm.nh * dm.hd, kv_size = dm.nk * dm.hd;
  const int ldq = 2 * q_size + 2 * kv_size;
  (void)rt;  // the row table reaches the kernel through its arguments
  out.clear();
  float *cur = d->h, *other = d->h2;
  bool first = true;
  struct {
    bool on = false;
    const float *alpha = nullptr;
    int mix = MIX_NONE;
  } pend;
  // Stages hand on their outputs as tagged words (tag = the producing stage's index + 1).
  // The hidden rows and the loop's input row, which every block computes alike, go to each
  // block's private rows too (1: h, 2: h2, 3: input) and are read back from there.
  uint32_t tag_q = 0, tag_z = 0, tag_o = 0, tag_m = 0;
  bool input_here = false;  // the input row was written earlier in this launch
  auto pv = [&](const float *p) { return p == d->h ? 1 : p == d->h2 ? 2 : 0; };
  auto first_in = [&]() {
    GemvIn g{};
    g.ld = dm.hidden;
    if (first && a.resume) {  // h = (state + input)^ from the saved rows
      first = false;
      g.mode = IN_RESID;
      g.src = d->state;
      g.mix = MIX_RESUME;
      g.h_dst = other;
      g.hdst_pv = pv(other);
      g.input = d->input;
      g.state = d->state;
      std::swap(cur, other);
      return g;
    }
    if (first) {  // the token's embedding row, stored as the hidden row
      first = false;
      g.mode = IN_EMBED;
      g.ids = d->d_ids;
      g.embed = static_cast<const __nv_bfloat16 *>(d->embed);
      g.vocab = dm.vocab;
      g.h_dst = cur;
      g.hdst_pv = pv(cur);
      return g;
    }
    if (!pend.on) {
      g.mode = IN_PLAIN;
      g.src = cur;
      g.src_pv = pv(cur);
      return g;
    }
    g.mode = IN_RESID;
    g.src = cur;
    g.src_pv = pv(cur);
    g.out = d->out;
    g.out_t = d->mega_to;
    g.out_tag = tag_o;
    g.alpha = pend.alpha;
    g.mix = pend.mix;
    g.h_dst = other;
    g.hdst_pv = pv(other);
    g.input = d->input;
    if (pend.mix == MIX_BEGIN) {
      g.input_pv = 3;
      input_here = true;
    } else if (pend.mix == MIX_LOOP && input_here) {
      g.input_pv = 3;
    }
    g.state = d->state;
    std::swap(cur, other);
    pend.on = false;
    return g;
  };
  auto gemv = [&](const void *W, int N, int K, long pair, const GemvIn &in, float *Y, EpiArgs ep) {
    MegaStage st{};
    st.kind = MK_GEMV;
    st.W = static_cast<const __nv_bfloat16 *>(W);
    st.N = N;
    st.K = K;
    st.pair = pair;
    st.R = mega_chunk_rows(K, pair > 0);
    st.in = in;
    st.Y = Y;
    const uint32_t tag = (uint32_t)out.size() + 1;
    if (Y == d->qkvg) {
      st.Yt = d->mega_tq;
      tag_q = tag;
    } else if (Y == d->out) {
      st.Yt = d->mega_to;
      tag_o = tag;
    } else if (Y == d->mlp) {
      st.Yt = d->mega_tm;
      tag_m = tag;
    }
    st.ep = ep;
    out.push_back(st);
  };
  auto layer = [&](int li, int loop_i, int mix) {
    const LayerDev &L = d->layers[li];
    if (L.attn) {
      const int sl = (c.kv_mode == DORY_KV_PER_LOOP && L.rec) ? loop_i : 0;
      const Ring ring = d->ring(L.ordinal, sl);
      gemv(L.wqkvg, ldq, dm.hidden, 0, first_in(), d->qkvg, EpiArgs{EPI_STORE, nullptr, nullptr, 0});
      MegaStage at{};
      at.kind = MK_ATTN;
      at.ring = ring;
      at.qkvg_t = d->mega_tq;
      at.qtag = tag_q;
      at.sq = L.sq;
      at.rope_kind = L.sliding ? 0 : 1;
      at.sg = L.sg;
      at.zt = d->mega_tz;
      at.part = d->part;
      const long keys = ring.window == INT_MAX ? (long)ring.cap : std::min<long>(ring.window, ring.cap);
      at.maxblk = (int)(keys / MEGA_AK + 2);
      tag_z = (uint32_t)out.size() + 1;
      out.push_back(at);
      GemvIn in{};
      in.mode = IN_NORM;
      in.src = d->z;
      in.src_t = d->mega_tz;
      in.src_tag = tag_z;
      in.ld = q_size;
      gemv(L.wo, dm.hidden, q_size, 0, in, d->out, EpiArgs{EPI_STORE, nullptr, nullptr, 0});
    } else {
      gemv(L.wgu, dm.ffn, dm.hidden, dm.ffn, first_in(), d->mlp, EpiArgs{EPI_SILU, L.msg, L.msu, (long)dm.ffn});
      GemvIn in{};
      in.mode = IN_NORM;
      in.src = d->mlp;
      in.src_t = d->mega_tm;
      in.src_tag = tag_m;
      in.ld = dm.ffn;
      gemv(L.wdown, dm.hidden, dm.ffn, 0, in, d->out, EpiArgs{EPI_STORE, nullptr, nullptr, 0});
    }
    pend.on = true;
    pend.alpha = L.alpha;
    pend.mix = mix;
  };
  const int n_in = c.n_in, n_rec = c.n_rec, n_all = (int)d->layers.size();
  if (!a.resume)
    for (int li = 0; li < n_in; li++) layer(li, 0, li == n_in - 1 ? MIX_BEGIN : MIX_NONE);
  for (int i = a.first_loop; i < a.loops; i++) {
    const int m = i == a.loops - 1 ? MIX_END : MIX_LOOP;
    for (int li = n_in; li < n_in + n_rec; li++) layer(li, i, li == n_in + n_rec - 1 ? m : MIX_NONE);
  }
  for (int li = n_in + n_rec; li < n_all; li++) layer(li, 0, MIX_NONE);  // f32 rings: the same row is rewritten
  gemv(d->head, dm.vocab, dm.hidden, 0, first_in(), d->logits, EpiArgs{EPI_SCALE, d->logit_scale, nullptr, 0});
  *h_last = cur;
  // DORY_MEGA_STALL=1 (tests): the first row-norm input awaits a tag that no stage writes,
  // so that its wait runs out (bounded by DORY_MEGA_SPIN) and the failure path runs
  if (const char *e = getenv("DORY_MEGA_STALL"); e && e[0] == '1')
    for (MegaStage &x : out)
      if (x.kind == MK_GEMV && x.in.mode == IN_NORM) {
        x.in.src_tag = 0xffffffffu;
        break;
      }
  if (d->mega_trace) {
    d->mega_trace_desc.clear();
    for (const MegaStage &x : out) {
      d->mega_trace_desc.push_back(x.kind);
      d->mega_trace_desc.push_back(x.kind == MK_GEMV ? x.N : 0);
      d->mega_trace_desc.push_back(x.kind == MK_GEMV ? x.K : 0);
    }
  }
  return DORY_OK;
}

// Zero the kernel's counters and launch it over the uploaded stage list.
int issue_mega(dory_t *d, const StepArgs &a, int32_t *rt, const MegaStage *stages, int nstages, cudaStream_t s) {
  const dory_config &c = d->cfg;
  CK(cudaMemsetAsync(d->mega_sync, 0, d->mega_sync_bytes, s));
  MegaArgs m{};
  m.stages = stages;
  m.nstages = nstages;
  m.d = d->dims;
  m.rows.seq = rt;
  m.rows.off = rt + d->Tmax;
  m.rows.seq_pos = d->d_seq_pos;
  m.rows.n = 1;
  m.theta_s = c.rope_theta_sliding;
  m.theta_f = c.rope_theta_full;
  m.rope = d->rope;
  m.sync = d->mega_sync;
  m.actr = d->mega_sync + 64;
  m.tpart = d->mega_tp;
  m.err = d->dev_err;
  m.seq_pos = d->d_seq_pos;
  m.priv = d->mega_priv;
  m.priv_stride = 3 * d->dims.hidden;
  m.adv_seq = a.aseq[0];
  m.adv_cnt = a.acnt[0];
  m.trace = (size_t)nstages <= d->mega_trace_stages ? d->mega_trace : nullptr;
  m.prefetch_ahead = d->mega_prefetch;
  m.stall_lead = std::max(d->mega_prefetch, d->mega_lead);
  // DORY_MEGA_SPIN: polls of a grid counter before a block gives up (read at every launch
  // that is not a graph replay, so that a test can make one wait run out)
  m.spin_limit = 1u << 22;
  if (const char *e = getenv("DORY_MEGA_SPIN")) m.spin_limit = (uint32_t)std::max(1, atoi(e));
  m.max_inflight = d->mega_inflight;
  CK(launch_mega_decode(m, d->sms, s));
  return DORY_OK;
}

int count_gemv(const std::vector<MegaStage> &st) {
  int n = 0;
  for (const MegaStage &x : st) n += x.kind == MK_GEMV;
  return n;
}

int upload_table(dory_t *d, const StepArgs &a, int32_t *rt, cudaStream_t s) {
  std::vector<int32_t> t((size_t)ROW_TABLE * d->Tmax, 0);
  for (int i = 0; i < a.T; i++) {
    t[i] = a.hseq[i];
    t[d->Tmax + i] = a.hoff[i];
    t[4 * d->Tmax + i] = a.perm.empty() ? i : a.perm[i];
  }
  for (size_t j = 0; j < a.head_pick.size(); j++) t[5 * d->Tmax + j] = a.head_pick[j];
  for (size_t i = 0; i < a.aseq.size(); i++) {
    t[2 * d->Tmax + i] = a.aseq[i];
    t[3 * d->Tmax + i] = a.acnt[i];
  }
  CK(cudaMemcpyAsync(rt, t.data(), t.size() * 4, cudaMemcpyHostToDevice, s));
  CK(cudaStreamSynchronize(s));
  return DORY_OK;
}

// Run one step: replay its captured graph (captured on first use), or issue the launches.
int do_step(dory_t *d, const StepArgs &a, const int32_t *ids) {
  int rc;
  CK(cudaMemcpyAsync(d->d_ids, ids, (size_t)a.T * 4, cudaMemcpyDefault, d->stream));
  const bool mega = use_mega(d, a);
  if (!d->use_graphs) {
    if ((rc = upload_table(d, a, d->d_rows, d->stream))) return rc;
    int nl = 0, ng = 0;
    if (mega) {
      std::vector<MegaStage> st;
      if ((rc = mega_build(d, a, d->d_rows, st, &d->h_last))) return rc;
      if (st.size() > d->mega_cap) {
        if (d->mega_stages) cudaFree(d->mega_stages);
        d->mega_stages = nullptr;
        d->mega_cap = 0;
        if (cudaMalloc(&d->mega_stages, st.size() * sizeof(MegaStage)) != cudaSuccess) {
          cudaGetLastError();
          return fail(DORY_ENOMEM, "cudaMalloc of a stage list");
        }
        d->mega_cap = st.size();
      }
      CK(cudaMemcpyAsync(d->mega_stages, st.data(), st.size() * sizeof(MegaStage), cudaMemcpyHostToDevice,
                         d->stream));
      if ((rc = issue_mega(d, a, d->d_rows, d->mega_stages, (int)st.size(), d->stream))) return rc;
      CK(cudaStreamSynchronize(d->stream));  // the host stage list is freed on return
      nl = 1;
      ng = count_gemv(st);
    } else if ((rc = issue_any(d, a, d->d_rows, false, d->stream, &nl, &ng))) {
      return rc;
    }
    d->st.launches = nl;
    d->st.gemm_launches = ng;
  } else {
    const std::string key = a.key();
    auto it = d->plans.find(key);
    const bool found = it != d->plans.end();
    if (!found && d->plans.size() >= d->max_plans) {
      // a server whose batches keep changing would grow without bound: drop the plan replayed
      // longest ago (after the work queued so far, which may still replay it)
      auto old = d->plans.begin();
      for (auto j = d->plans.begin(); j != d->plans.end(); ++j)
        if (j->second.used < old->second.used) old = j;
      CK(cudaStreamSynchronize(d->stream));
      cudaGraphExecDestroy(old->second.exec);
      if (old->second.rt) cudaFree(old->second.rt);
      if (old->second.stages) cudaFree(old->second.stages);
      d->plans.erase(old);
    }
    if (!found) {
      Plan p;
      if (cudaMalloc(&p.rt, (size_t)ROW_TABLE * d->Tmax * 4) != cudaSuccess) {
        cudaGetLastError();
        return fail(DORY_ENOMEM, "cudaMalloc of a step table");
      }
      if ((rc = upload_table(d, a, p.rt, d->stream))) {
        cudaFree(p.rt);
        return rc;
      }
      std::vector<MegaStage> st;
      if (mega) {
        if ((rc = mega_build(d, a, p.rt, st, &p.h_last))) {
          cudaFree(p.rt);
          return rc;
        }
        if (cudaMalloc(&p.stages, st.size() * sizeof(MegaStage)) != cudaSuccess) {
          cudaGetLastError();
          cudaFree(p.rt);
          return fail(DORY_ENOMEM, "cudaMalloc of a stage list");
        }
        CK(cudaMemcpy(p.stages, st.data(), st.size() * sizeof(MegaStage), cudaMemcpyHostToDevice));
      }
      cudaGraph_t g = nullptr;
      CK(cudaStreamBeginCapture(d->cap_stream, cudaStreamCaptureModeThreadLocal));
      if (mega) {
        rc = issue_mega(d, a, p.rt, p.stages, (int)st.size(), d->cap_stream);
        p.launches = 1;
        p.gemm_launches = count_gemv(st);
      } else {
        rc = issue_any(d, a, p.rt, true, d->cap_stream, &p.launches, &p.gemm_launches);
        p.h_last = d->h_last;
      }
      cudaError_t ec = cudaStreamEndCapture(d->cap_stream, &g);
      if (rc || ec != cudaSuccess) {
        if (g) cudaGraphDestroy(g);
        cudaFree(p.rt);
        if (p.stages) cudaFree(p.stages);
        cudaGetLastError();
        return rc ? rc : fail(DORY_ECUDA, "graph capture: %s", cudaGetErrorString(ec));
      }
      ec = cudaGraphInstantiate(&p.exec, g, 0);
      cudaGraphDestroy(g);
      if (ec != cudaSuccess) {
        cudaFree(p.rt);
        if (p.stages) cudaFree(p.stages);
        return fail(DORY_ECUDA, "graph instantiate: %s", cudaGetErrorString(ec));
      }
      it = d->plans.emplace(key, p).first;
    }
    it->second.used = ++d->steps;
    CK(cudaGraphLaunch(it->second.exec, d->stream));
    d->h_last = it->second.h_last;
    d->st.launches = it->second.launches;
    d->st.gemm_launches = it->second.gemm_launches;
  }
  account(d, a);
  for (size_t i = 0; i < a.aseq.size(); i++) d->seq_pos[a.aseq[i]] += a.acnt[i];
  d->last_rows = a.T;
  return DORY_OK;
}


// Tensor maps, split counts and buffers of the tensor-core projections (bf16 weights).
int setup_tc(dory_t *d) {
  const Dims dm = d->dims;
  const int q_size = dm.nh * dm.hd, kv_size = dm.nk * dm.hd, ldq = 2 * q_size + 2 * kv_size;
  {
    const char *e = getenv("DORY_TC");
    if (e && e[0] == '0') return DORY_OK;
  }
  if (d->wdtype != W_BF16 || dm.hidden % 64 || dm.ffn % 64 || q_size % 64) return DORY_OK;
  d->tc_big = !getenv_off("DORY_TC_BIG") && dm.ffn % 128 == 0;
  int dev = 0, sms = 148;
  CK(cudaGetDevice(&dev));
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  // rows of the split-activation kernel's steps (larger steps take launch_tc_gemm_big)
  const int small_rows = d->tc_big ? std::min(d->Tmax, TC_BIG_ROWS - 1) : d->Tmax;
  const int bn_max = tc_tile_rows(small_rows);
  // K splits per tile at most: 6 measured best for 64-row steps (batch-64 decode 2.21 ms with 4,
  // 2.16 with 6, 2.48 with 8); DORY_TC_SPLITS changes it
  int max_split = 6;
  if (const char *e = getenv("DORY_TC_SPLITS")) max_split = std::max(1, std::min(8, atoi(e)));
  int per_sm = 1;  // blocks per SM the splits aim at (one: the 64-row rings fill an SM); DORY_TC_PER_SM changes it
  if (const char *e = getenv("DORY_TC_PER_SM")) per_sm = std::max(1, std::min(4, atoi(e)));
  size_t ws_floats = 0;
  int max_tiles = 1;
  auto mk = [&](TcW &w, const void *base, long rows, int K, int N, long pair) -> int {
    if (make_tmap_bf16(&w.map, base, rows, K, 128)) return fail(DORY_ECUDA, "tensor map of a weight matrix");
    w.N = N;
    w.K = K;
    w.pair = pair;
    const int mt = (N + 127) / 128, nkb = K / 64;
    if (getenv("DORY_TC_TRACE") && !w.trace) {
      if (cudaMalloc(&w.trace, (size_t)TC_TRACE_BLOCKS * TC_TRACE_EVENTS * 8) != cudaSuccess) {
        cudaGetLastError();
        w.trace = nullptr;
      }
    }
    w.splits = std::max(1, std::min(std::min(per_sm * sms / mt, max_split), nkb));
    const int t_tiles = (small_rows + bn_max - 1) / bn_max;
    ws_floats = std::max(ws_floats, (size_t)mt * t_tiles * w.splits * (pair ? 2 : 1) * bn_max * 128);
    max_tiles = std::max(max_tiles, mt * t_tiles);
    return DORY_OK;
  };
  d->tcw.assign(d->layers.size(), {});
  int rc;
  for (size_t li = 0; li < d->layers.size(); li++) {
    const LayerDev &L = d->layers[li];
    if (L.attn) {
      if ((rc = mk(d->tcw[li][0], L.wqkvg, ldq, dm.hidden, ldq, 0))) return rc;
      if ((rc = mk(d->tcw[li][1], L.wo, dm.hidden, q_size, dm.hidden, 0))) return rc;
    } else {
      if ((rc = mk(d->tcw[li][0], L.wgu, 2L * dm.ffn, dm.hidden, dm.ffn, dm.ffn))) return rc;
      if ((rc = mk(d->tcw[li][1], L.wdown, dm.hidden, dm.ffn, dm.hidden, 0))) return rc;
    }
  }
  if ((rc = mk(d->tc_head, d->head, dm.vocab, dm.hidden, dm.vocab, 0))) return rc;
  const int XR = std::max(d->Tmax, 256);
  const int widths[3] = {dm.hidden, q_size, dm.ffn};
  size_t off = 0, offs[3][2];
  for (int b = 0; b < 3; b++)
    for (int h = 0; h < 2; h++) {
      offs[b][h] = off;
      off = align256(off + (size_t)XR * widths[b] * 2);
    }
  const size_t o_ws = off;
  off = align256(off + ws_floats * 4);
  const size_t o_ctr = off;
  off = align256(off + (size_t)max_tiles * 4);
  const size_t o_err = off;
  off = align256(off + 4);
  const size_t o_wsb = off;
  if (d->tc_big) off = align256(off + (size_t)2 * sms * 128 * 256 * 4);
  const size_t o_ctrb = off;
  if (d->tc_big) off = align256(off + (size_t)TC_BIG_CTRS * 4);
  if (cudaMalloc(&d->tcmem, off) != cudaSuccess) {
    cudaGetLastError();
    return fail(DORY_ENOMEM, "cudaMalloc of %zu tensor-core bytes", off);
  }
  CK(cudaMemset(d->tcmem, 0, off));
  __nv_bfloat16 *buf[3][2];
  for (int b = 0; b < 3; b++)
    for (int h = 0; h < 2; h++) {
      buf[b][h] = reinterpret_cast<__nv_bfloat16 *>(d->tcmem + offs[b][h]);
      for (int bi = 0; bi < 5; bi++)
        if (make_tmap_bf16(&d->xmap[b][h][bi], buf[b][h], XR, widths[b], 16 << bi))
          return fail(DORY_ECUDA, "tensor map of an activation buffer");
    }
  d->em_h = Emit{buf[0][0], buf[0][1]};
  d->em_z = Emit{buf[1][0], buf[1][1]};
  d->em_y = Emit{buf[2][0], buf[2][1]};
  d->tc_ws = reinterpret_cast<float *>(d->tcmem + o_ws);
  if (d->tc_big) {
    d->tc_ws_big = reinterpret_cast<float *>(d->tcmem + o_wsb);
    d->tc_ctr_big = reinterpret_cast<int32_t *>(d->tcmem + o_ctrb);
  }
  d->tc_ctr = reinterpret_cast<int32_t *>(d->tcmem + o_ctr);
  d->tc_err = d->dev_err;
  (void)o_err;
  d->tc_ok = true;
  return DORY_OK;
}

// A bounded wait of a kernel ran out during the calls since the last check: reported once
// (the flag is cleared), the handle stays usable.
int check_device_error(dory_t *d) {
  if (!d->dev_err) return DORY_OK;
  int32_t e = 0;
  CK(cudaMemcpy(&e, d->dev_err, 4, cudaMemcpyDeviceToHost));
  if (e) {
    CK(cudaMemset(d->dev_err, 0, 4));
    return fail(DORY_EWAIT, "a kernel gave up a bounded wait (code %d): the rows of the steps since the last "
                            "check are undefined; reset their sequences", e);
  }
  return DORY_OK;
}

}  // namespace

namespace dory {
void set_last_error(const char *msg) { g_err = msg; }
}  // namespace dory

extern "C" {

const char *dory_last_error(void) { return g_err.c_str(); }

int dory_create(const dory_config *cfg, const dory_weights *w, void *stream, dory_t **out) {
  if (!out) return fail(DORY_EINVAL, "out is NULL");
  *out = nullptr;
  std::string pat;
  int rc = validate(cfg, pat);
  if (rc) return rc;
  if (!w || !w->layers) return fail(DORY_EINVAL, "weights are NULL");
  dory_t *d = new dory_t();
  d->cfg = *cfg;
  d->pattern = pat;
  d->cfg.layer_pattern = nullptr;
  d->dims = Dims{cfg->hidden, cfg->ffn, cfg->vocab, cfg->nh, cfg->nk, cfg->hd};
  d->wdtype = cfg->weight_dtype == DORY_W_BF16 ? W_BF16 : W_F32;
  d->esz = cfg->weight_dtype == DORY_W_BF16 ? 2 : 4;
  d->stream = static_cast<cudaStream_t>(stream);
  d->Tmax = d->Tstep = std::max(DORY_CHUNK_ROWS, cfg->max_batch);
  {
    // dory_prefill runs the input and output blocks over up to PREFILL_ROWS rows at once. Their
    // attention takes pieces of at most 512 rows: a piece's rows join a ring before any of
    // them attends, so a sliding (or capped full) ring must hold the piece plus the window
    // behind its first row: rows + window - 1 <= ring rows
    long lim = 512;
    for (size_t li = 0; li < pat.size(); li++) {
      const bool io = (int)li < cfg->n_in || (int)li >= cfg->n_in + cfg->n_rec;
      if (!io || pat[li] == '-') continue;
      long cap, win;
      if (pat[li] == 'S') win = cfg->window;
      else if (cfg->full_window > 0) win = cfg->full_window;
      else continue;  // every position from 0 stays in such a ring
      cap = (win + RING_EXTRA + 63) / 64 * 64;
      lim = std::min(lim, cap - win + 1);
    }
    lim = lim / 64 * 64;
    d->piece_rows = (int)lim;
    // f32 rings: the projections and MLPs of the input and output blocks run over many more
    // rows per step (tensor-bound contractions), the attention piece by piece; q8_2f rings
    // attend the step's rows at once
    const int q_sz = cfg->nh * cfg->hd;
    const bool big = cfg->kv_quant != DORY_KV_Q8_2F && cfg->weight_dtype == DORY_W_BF16 && !getenv_off("DORY_TC") &&
                     !getenv_off("DORY_TC_BIG") && cfg->ffn % 128 == 0 && cfg->hidden % 64 == 0 && q_sz % 64 == 0;
    long rows = big ? std::max<long>(lim, PREFILL_ROWS) : lim;
    if (const char *e = getenv("DORY_PREFILL_ROWS")) rows = std::min<long>(rows, std::max(0, atoi(e)));
    rows = rows / 64 * 64;
    d->piece_rows = (int)std::min<long>(d->piece_rows, rows);
    d->prefill_rows = (d->piece_rows >= 128 && cfg->weight_dtype == DORY_W_BF16) ? (int)rows : 0;
    d->Tmax = std::max(d->Tmax, d->prefill_rows);
  }
  const Dims &dm = d->dims;
  const size_t esz = d->esz;
  const int q_size = dm.nh * dm.hd, kv_size = dm.nk * dm.hd;
  auto cleanup = [&](int code) {
    free_all(d);
    delete d;
    return code;
  };

  // ---- weights -----------------------------------------------------------------------
  size_t wb = 0;
  auto reserve = [&](size_t bytes) {
    size_t at = wb;
    wb = align256(wb + bytes);
    return at;
  };
  const size_t o_embed = reserve((size_t)dm.vocab * dm.hidden * esz);
  const size_t o_head = reserve((size_t)dm.vocab * dm.hidden * esz);
  const size_t o_ls = reserve((size_t)dm.vocab * 4);
  struct Offs {
    size_t qkvg, o, sq, sg, gu, down, msg, msu, alpha;
  };
  std::vector<Offs> offs(pat.size());
  for (size_t li = 0; li < pat.size(); li++) {
    Offs &o = offs[li];
    if (pat[li] == '-') {
      o.gu = reserve((size_t)2 * dm.ffn * dm.hidden * esz);
      o.down = reserve((size_t)dm.hidden * dm.ffn * esz);
      o.msg = reserve((size_t)dm.ffn * 4);
      o.msu = reserve((size_t)dm.ffn * 4);
    } else {
      o.qkvg = reserve((size_t)(2 * q_size + 2 * kv_size) * dm.hidden * esz);
      o.o = reserve((size_t)dm.hidden * q_size * esz);
      o.sq = reserve((size_t)q_size * 4);
      o.sg = reserve((size_t)q_size * 4);
    }
    o.alpha = reserve((size_t)dm.hidden * 4);
  }
  if (cudaMalloc(&d->wmem, wb) != cudaSuccess) {
    cudaGetLastError();
    fail(DORY_ENOMEM, "cudaMalloc of %zu weight bytes", wb);
    return cleanup(DORY_ENOMEM);
  }
  d->wbytes = wb;
  char *W = d->wmem;
  d->embed = W + o_embed;
  d->head = W + o_head;
  d->logit_scale = reinterpret_cast<float *>(W + o_ls);
#define COPY(dst, src, bytes, what)                       \
  if ((rc = copy_in((dst), (src), (bytes), (what))) != 0) \
    return cleanup(rc);
  COPY(d->embed, w->embed, (size_t)dm.vocab * dm.hidden * esz, "embed");
  COPY(d->head, w->head, (size_t)dm.vocab * dm.hidden * esz, "head");
  COPY(d->logit_scale, w->logit_scale, (size_t)dm.vocab * 4, "logit_scale");
  d->layers.resize(pat.size());
  int ordinal = 0;
  for (size_t li = 0; li < pat.size(); li++) {
    const dory_layer_weights &lw = w->layers[li];
    const Offs &o = offs[li];
    LayerDev &L = d->layers[li];
    L.rec = (int)li >= cfg->n_in && (int)li < cfg->n_in + cfg->n_rec;
    L.out = (int)li >= cfg->n_in + cfg->n_rec;
    L.alpha = reinterpret_cast<float *>(W + o.alpha);
    COPY(L.alpha, lw.alpha, (size_t)dm.hidden * 4, "alpha");
    if (pat[li] == '-') {
      L.attn = false;
      L.wgu = W + o.gu;
      L.wdown = W + o.down;
      L.msg = reinterpret_cast<float *>(W + o.msg);
      L.msu = reinterpret_cast<float *>(W + o.msu);
      const size_t m = (size_t)dm.ffn * dm.hidden * esz;
      COPY(L.wgu, lw.gate, m, "gate");
      COPY(static_cast<char *>(L.wgu) + m, lw.up, m, "up");
      COPY(L.wdown, lw.down, (size_t)dm.hidden * dm.ffn * esz, "down");
      COPY(L.msg, lw.mlp_sg, (size_t)dm.ffn * 4, "mlp_sg");
      COPY(L.msu, lw.mlp_su, (size_t)dm.ffn * 4, "mlp_su");
    } else {
      L.attn = true;
      L.sliding = pat[li] == 'S';
      L.ordinal = ordinal++;
      L.wqkvg = W + o.qkvg;
      L.wo = W + o.o;
      L.sq = reinterpret_cast<float *>(W + o.sq);
      L.sg = reinterpret_cast<float *>(W + o.sg);
      char *qk = static_cast<char *>(L.wqkvg);
      const size_t qb = (size_t)q_size * dm.hidden * esz, kb = (size_t)kv_size * dm.hidden * esz;
      COPY(qk, lw.q, qb, "q");
      COPY(qk + qb, lw.k, kb, "k");
      COPY(qk + qb + kb, lw.v, kb, "v");
      COPY(qk + qb + 2 * kb, lw.g, qb, "g");
      COPY(L.wo, lw.o, (size_t)dm.hidden * q_size * esz, "o");
      COPY(L.sq, lw.sq, (size_t)q_size * 4, "sq");
      COPY(L.sg, lw.sg, (size_t)q_size * 4, "sg");
    }
  }
#undef COPY

  // ---- KV rings ------------------------------------------------------------------------
  const bool q8 = cfg->kv_quant == DORY_KV_Q8_2F;
  size_t sb = 0;
  d->ords.resize(ordinal);
  d->slot_index.resize(ordinal);
  int flat = 0;
  for (size_t li = 0; li < pat.size(); li++) {
    const LayerDev &L = d->layers[li];
    if (!L.attn) continue;
    OrdInfo &o = d->ords[L.ordinal];
    o.sliding = L.sliding;
    o.rec = L.rec;
    if (L.sliding) {
      o.cap = cfg->window + RING_EXTRA;
      o.window = cfg->window;
    } else if (cfg->full_window > 0) {
      o.cap = cfg->full_window + RING_EXTRA;
      o.window = cfg->full_window;
    } else {
      o.cap = cfg->max_context;
      o.window = INT_MAX;
    }
    o.cap = (o.cap + 63) / 64 * 64;  // whole 64-row blocks: a block of positions is contiguous in the ring
    o.slots = (cfg->kv_mode == DORY_KV_PER_LOOP && L.rec) ? cfg->max_loops : 1;
    o.L = slot_layout(o.cap, dm.nk, dm.hd, q8);
    o.off = sb;
    sb = (sb + (size_t)o.slots * o.L.bytes + 1023) & ~(size_t)1023;
    d->slot_index[L.ordinal] = flat;
    flat += o.slots;
    const long keys = o.window == INT_MAX ? (long)o.cap : std::min<long>(o.window, o.cap);
    d->max_splits = std::max<int>(d->max_splits, (int)((keys + KEYS_PER_SPLIT - 1) / KEYS_PER_SPLIT));
    d->max_splits = std::max<int>(d->max_splits, attn_tma_splits(keys));
    d->max_splits = std::max<int>(d->max_splits, attn_chunk_blocks(keys, std::max(d->Tstep, d->piece_rows)));
    if ((keys + KEYS_PER_SPLIT - 1) / KEYS_PER_SPLIT > 2 * dm.hd) {
      fail(DORY_EINVAL, "a window of %ld keys is more than the attention merge holds for hd %d", keys, dm.hd);
      return cleanup(DORY_EINVAL);
    }
  }
  d->n_flat_slots = flat;
  d->seq_stride = std::max<size_t>(sb, 1024);
  d->kv_bytes = d->seq_stride * cfg->max_seqs;
  if (cudaMalloc(&d->kvmem, d->kv_bytes) != cudaSuccess) {
    cudaGetLastError();
    fail(DORY_ENOMEM, "cudaMalloc of %zu KV bytes", d->kv_bytes);
    return cleanup(DORY_ENOMEM);
  }

  {
    const char *e = getenv("DORY_KV_TMA");
    const bool on = !(e && e[0] == '0');
    if (!q8) d->kv_tma = on && make_tmap_kv_f32(&d->kvmap, d->kvmem, d->kv_bytes, dm.hd) == 0;
    else d->kv_tma_q8 = on && dm.hd == 128 && make_tmap_kv_q8(&d->kvq, d->kvmem, d->kv_bytes) == 0;
  }

  // ---- activations ---------------------------------------------------------------------
  const int T = d->Tmax;
  const int rep = dm.nh / dm.nk;
  size_t ab = 0;
  auto areserve = [&](size_t bytes) {
    size_t at = ab;
    ab = align256(ab + bytes);
    return at;
  };
  const size_t a_h2 = areserve((size_t)T * dm.hidden * 4), a_hc = areserve((size_t)(2 * dm.nh + 2 * dm.nk) * 4),
               a_ac2 = areserve((size_t)T * dm.nk * 4);
  const size_t a_h = areserve((size_t)T * dm.hidden * 4), a_in = areserve((size_t)T * dm.hidden * 4),
               a_st = areserve((size_t)T * dm.hidden * 4),
               a_qkvg = areserve((size_t)T * (2 * q_size + 2 * kv_size) * 4),
               a_z = areserve((size_t)T * q_size * 4), a_out = areserve((size_t)T * dm.hidden * 4),
               a_mlp = areserve((size_t)T * dm.ffn * 4), a_lg = areserve((size_t)d->Tstep * dm.vocab * 4),
               a_rope = areserve((size_t)T * 2 * dm.hd * 4),
               a_part = areserve((size_t)std::max(d->Tstep, d->piece_rows) * dm.nk * d->max_splits * rep *
                                 (dm.hd + 2) * 4),
               a_kst = areserve((size_t)T * kv_size * 4), a_vst = areserve((size_t)T * kv_size * 4),
               a_ids = areserve((size_t)T * 4), a_ids2 = areserve((size_t)T * 4),
               a_lg2 = areserve((size_t)d->Tstep * dm.vocab * 4),
               a_sp = areserve((size_t)cfg->max_seqs * 4), a_rows = areserve((size_t)ROW_TABLE * T * 4),
               a_zero = areserve((size_t)cfg->max_seqs * 4), a_err = areserve(256);
  const size_t ms_ints = ((size_t)(64 + dm.nk) * 4 + 15) & ~(size_t)15;
  const size_t ms_words = (size_t)(2 * q_size + 2 * kv_size) + q_size + dm.hidden + dm.ffn +
                          (size_t)dm.nh * MEGA_FLAGS * (dm.hd + 2);
  const size_t ms_bytes = ms_ints + ms_words * 8, a_ms = areserve(ms_bytes);
  const size_t a_stab = areserve((size_t)d->n_flat_slots * 3 * 8), a_drop = areserve((size_t)d->n_flat_slots * 4),
               a_top = areserve(4);
  if (cudaMalloc(&d->act, ab) != cudaSuccess) {
    cudaGetLastError();
    fail(DORY_ENOMEM, "cudaMalloc of %zu activation bytes", ab);
    return cleanup(DORY_ENOMEM);
  }
  char *A = d->act;
  d->h = reinterpret_cast<float *>(A + a_h);
  d->h2 = reinterpret_cast<float *>(A + a_h2);
  d->h_last = d->h;
  d->hctr = reinterpret_cast<int32_t *>(A + a_hc);
  d->actr = reinterpret_cast<int32_t *>(A + a_ac2);
  {
    const int hdv = dm.hd;
    const size_t kmax = std::max(std::max(dm.hidden, dm.ffn), dm.nh * dm.hd);
    d->fused_ok = (hdv == 64 || hdv == 128) && cfg->n_in >= 1 && cfg->n_rec >= 1 && cfg->n_out >= 1 &&
                  kmax % 8 == 0 && 4 * kmax * 4 <= 96 * 1024;
    const char *e = getenv("DORY_FUSED");
    if (e && e[0] == '0') d->fused_ok = false;
  }
  d->mega_sync = reinterpret_cast<int32_t *>(A + a_ms);
  d->mega_sync_bytes = ms_bytes;
  d->mega_tq = reinterpret_cast<unsigned long long *>(A + a_ms + ms_ints);
  d->mega_tz = d->mega_tq + 2 * q_size + 2 * kv_size;
  d->mega_to = d->mega_tz + q_size;
  d->mega_tm = d->mega_to + dm.hidden;
  d->mega_tp = d->mega_tm + dm.ffn;
  {
    // the persistent decode kernel: bf16 weights, f32 rings, rows that stream as whole
    // 16-byte runs and fit a ring slot, a block's input row and attention scratch within
    // its work area
    int dev = 0;
    CK(cudaGetDevice(&dev));
    CK(cudaDeviceGetAttribute(&d->sms, cudaDevAttrMultiProcessorCount, dev));
    const size_t kmax = std::max(std::max(dm.hidden, dm.ffn), q_size);
    bool ok = d->wdtype == W_BF16 && !q8 && (dm.hd == 64 || dm.hd == 128) && dm.hidden % 8 == 0 &&
              dm.ffn % 8 == 0 && q_size % 8 == 0 && kmax + mega_park_floats(false) <= mega_work_floats() &&
              (size_t)dm.hidden + mega_park_floats(true) <= mega_work_floats() &&
              (size_t)2 * MEGA_AK * dm.hd <= mega_work_floats() && mega_chunk_rows(dm.hidden, true) >= 1 &&
              mega_chunk_rows((int)kmax, false) >= 2;
    // the merge's per-warp partials of a kv head's query heads
    if ((size_t)mega_consumer_warps() * rep * (dm.hd + 2) > mega_work_floats()) ok = false;
    // input rows of at most six float4 chunks a thread, a residual (hidden row) of at most two
    if (dm.hidden > 2048 || dm.ffn > 6144 || q_size > 6144) ok = false;
    const int nmax = std::max(std::max(dm.vocab, dm.ffn), 2 * q_size + 2 * kv_size);
    if (d->sms > 0 && (nmax + d->sms - 1) / d->sms > mega_max_rows_per_block()) ok = false;
    for (const OrdInfo &o : d->ords) {
      const long keys = o.window == INT_MAX ? (long)o.cap : std::min<long>(o.window, o.cap);
      const long maxblk = keys / MEGA_AK + 2;
      if (maxblk > (long)T * d->max_splits) ok = false;  // partials buffer
    }
    const char *e = getenv("DORY_MEGA");
    if (e && e[0] == '0') ok = false;
    d->mega_ok = ok && mega_supported(dm.hd, d->sms);
    if (d->mega_ok && cudaMalloc(&d->mega_priv, (size_t)d->sms * 3 * dm.hidden * 4) != cudaSuccess) {
      cudaGetLastError();
      d->mega_priv = nullptr;
      d->mega_ok = false;
    }
    if (const char *pe = getenv("DORY_MEGA_PREFETCH")) d->mega_prefetch = std::max(0, atoi(pe));
    if (const char *pe = getenv("DORY_MEGA_LEAD")) d->mega_lead = std::max(0, atoi(pe));
    if (const char *pe = getenv("DORY_MEGA_INFLIGHT")) d->mega_inflight = std::max(0, atoi(pe));
    const char *tp = getenv("DORY_MEGA_TRACE");
    if (d->mega_ok && tp && tp[0]) {
      const size_t stages = (size_t)3 * (cfg->n_in + cfg->max_loops * cfg->n_rec + cfg->n_out) + 2;
      const size_t bytes = stages * d->sms * MEGA_TRACE_EVENTS * 8;
      if (cudaMalloc(&d->mega_trace, bytes) == cudaSuccess && cudaMemset(d->mega_trace, 0, bytes) == cudaSuccess) {
        d->mega_trace_stages = stages;
        d->mega_trace_path = tp;
      } else {
        cudaGetLastError();
        d->mega_trace = nullptr;
      }
    }
  }
  d->input = reinterpret_cast<float *>(A + a_in);
  d->state = reinterpret_cast<float *>(A + a_st);
  d->qkvg = reinterpret_cast<float *>(A + a_qkvg);
  d->z = reinterpret_cast<float *>(A + a_z);
  d->out = reinterpret_cast<float *>(A + a_out);
  d->mlp = reinterpret_cast<float *>(A + a_mlp);
  d->logits = reinterpret_cast<float *>(A + a_lg);
  d->rope = reinterpret_cast<float *>(A + a_rope);
  d->part = reinterpret_cast<float *>(A + a_part);
  d->kst = reinterpret_cast<float *>(A + a_kst);
  d->vst = reinterpret_cast<float *>(A + a_vst);
  d->d_ids = reinterpret_cast<int32_t *>(A + a_ids);
  d->d_ids2 = reinterpret_cast<int32_t *>(A + a_ids2);
  d->logits2 = reinterpret_cast<float *>(A + a_lg2);
  d->d_seq_pos = reinterpret_cast<int32_t *>(A + a_sp);
  d->d_rows = reinterpret_cast<int32_t *>(A + a_rows);
  d->d_zero = reinterpret_cast<int32_t *>(A + a_zero);
  d->dev_err = reinterpret_cast<int32_t *>(A + a_err);
  d->slot_table = reinterpret_cast<long long *>(A + a_stab);
  d->dropped = reinterpret_cast<int32_t *>(A + a_drop);
  d->d_top = reinterpret_cast<float *>(A + a_top);
  if (cudaMemsetAsync(d->act, 0, ab, d->stream) != cudaSuccess) return cleanup(fail(DORY_ECUDA, "memset"));
  {
    std::vector<long long> t((size_t)d->n_flat_slots * 3);
    for (size_t o = 0; o < d->ords.size(); o++)
      for (int sl = 0; sl < d->ords[o].slots; sl++) {
        const Ring r = d->ring((int)o, sl);
        long long *e = &t[(size_t)(d->slot_index[o] + sl) * 3];
        e[0] = (long long)(r.off + r.L.tags);
        e[1] = (long long)(r.off + r.L.meta);
        e[2] = r.cap;
      }
    if (cudaMemcpyAsync(d->slot_table, t.data(), t.size() * 8, cudaMemcpyHostToDevice, d->stream) != cudaSuccess ||
        cudaStreamSynchronize(d->stream) != cudaSuccess)
      return cleanup(fail(DORY_ECUDA, "slot table upload"));
  }

  {
    const char *e = getenv("DORY_GRAPHS");
    d->use_graphs = !(e && e[0] == '0');
    if (const char *m = getenv("DORY_MAX_PLANS")) d->max_plans = (size_t)std::max(1, atoi(m));
  }
  if (cudaStreamCreateWithFlags(&d->cap_stream, cudaStreamNonBlocking) != cudaSuccess)
    return cleanup(fail(DORY_ECUDA, "stream create"));
  if ((rc = setup_tc(d))) return cleanup(rc);
  d->seq_pos.assign(cfg->max_seqs, 0);
  d->exits.assign(cfg->max_seqs, ExitRate{});
  d->appended.assign((size_t)cfg->max_seqs * d->n_flat_slots, 0);
  for (int s = 0; s < cfg->max_seqs; s++)
    if ((rc = reset_seq(d, s))) return cleanup(rc);
  if (cudaStreamSynchronize(d->stream) != cudaSuccess) return cleanup(fail(DORY_ECUDA, "sync after create"));
  d->st.weight_bytes_device = wb;
  d->st.kv_bytes_device = d->kv_bytes;
  *out = d;
  g_err.clear();
  return DORY_OK;
}

int dory_destroy(dory_t *d) {
  if (!d) return DORY_OK;
  cudaStreamSynchronize(d->stream);
  if (const char *tp = getenv("DORY_TC_TRACE")) {
    // file: records of int32 (layer, which, N, K, splits, blocks) then u64 [blocks][TC_TRACE_EVENTS]
    if (FILE *f = fopen(tp, "wb")) {
      auto dump = [&](const TcW &w, int li, int which) {
        if (!w.trace || w.trace_grid <= 0) return;
        const int nb = std::min(w.trace_grid, TC_TRACE_BLOCKS);
        std::vector<unsigned long long> t((size_t)nb * TC_TRACE_EVENTS);
        if (cudaMemcpy(t.data(), w.trace, t.size() * 8, cudaMemcpyDeviceToHost) != cudaSuccess) return;
        const int32_t hdr[6] = {li, which, w.N, w.K, w.splits, nb};
        fwrite(hdr, 4, 6, f);
        fwrite(t.data(), 8, t.size(), f);
      };
      for (size_t li = 0; li < d->tcw.size(); li++)
        for (int which = 0; which < 2; which++) dump(d->tcw[li][which], (int)li, which);
      dump(d->tc_head, -1, 0);
      fclose(f);
    }
  }
  if (d->mega_trace && !d->mega_trace_desc.empty()) {
    // file: int32 nstages, grid, events; int32 [nstages][3] (kind, N, K); u64 stamps
    const int32_t hdr[3] = {(int32_t)(d->mega_trace_desc.size() / 3), d->sms, MEGA_TRACE_EVENTS};
    std::vector<unsigned long long> t((size_t)hdr[0] * d->sms * MEGA_TRACE_EVENTS);
    if (cudaMemcpy(t.data(), d->mega_trace, t.size() * 8, cudaMemcpyDeviceToHost) == cudaSuccess) {
      if (FILE *f = fopen(d->mega_trace_path.c_str(), "wb")) {
        fwrite(hdr, 4, 3, f);
        fwrite(d->mega_trace_desc.data(), 4, d->mega_trace_desc.size(), f);
        fwrite(t.data(), 8, t.size(), f);
        fclose(f);
      }
    }
  }
  free_all(d);
  delete d;
  return DORY_OK;
}

int dory_reset(dory_t *d, int32_t seq) {
  if (!d) return fail(DORY_EINVAL, "handle is NULL");
  if (seq < 0 || seq >= d->cfg.max_seqs) return fail(DORY_EINVAL, "seq %d out of range", seq);
  return reset_seq(d, seq);
}

int dory_rollback(dory_t *d, int32_t seq, int32_t n) {
  if (!d) return fail(DORY_EINVAL, "handle is NULL");
  if (seq < 0 || seq >= d->cfg.max_seqs) return fail(DORY_EINVAL, "seq %d out of range", seq);
  if (n < 0) return fail(DORY_EINVAL, "n=%d must be >= 0", n);
  const int pos = d->seq_pos[seq];
  if (n >= pos) return DORY_OK;  // nothing is stored at or past n: the position stays (min(pos, n))
  // every window that reads a row before n must still find its rows in the ring
  for (const OrdInfo &o : d->ords) {
    if (o.window == INT_MAX) continue;  // such a ring holds every position from 0
    const long need = std::max<long>(0, (long)n - o.window + 1), held = std::max<long>(0, (long)pos - o.cap);
    if (need < held)
      return fail(DORY_ERANGE, "rollback of sequence %d from %d to %d: a ring of %d rows with window %d keeps %d "
                               "positions back at most", seq, pos, n, o.cap, o.window, o.cap - o.window + 1);
  }
  CK(launch_rollback(d->kvmem + (size_t)seq * d->seq_stride, d->slot_table, d->n_flat_slots, n, d->dims.nk,
                     d->cfg.kv_quant == DORY_KV_Q8_2F ? 1 : 0, d->dropped, d->stream));
  std::vector<int32_t> dropped(d->n_flat_slots);
  CK(cudaMemcpyAsync(dropped.data(), d->dropped, dropped.size() * 4, cudaMemcpyDeviceToHost, d->stream));
  d->seq_pos[seq] = n;
  CK(cudaMemcpyAsync(d->d_seq_pos + seq, &d->seq_pos[seq], 4, cudaMemcpyHostToDevice, d->stream));
  CK(cudaStreamSynchronize(d->stream));
  for (int i = 0; i < d->n_flat_slots; i++) d->appended[(size_t)seq * d->n_flat_slots + i] -= dropped[i];
  return DORY_OK;
}

static int check_range(dory_t *d, int seq, long last_pos) {
  for (const OrdInfo &o : d->ords)
    if (o.window == INT_MAX && last_pos >= o.cap)
      return fail(DORY_ERANGE, "position %ld of sequence %d is past max_context %d", last_pos, seq, o.cap);
  return DORY_OK;
}

int dory_prefill_chunk(dory_t *d, int32_t seq, const int32_t *ids, int32_t n, int32_t pos0, int32_t loops,
                       int32_t want) {
  if (!d) return fail(DORY_EINVAL, "handle is NULL");
  if (seq < 0 || seq >= d->cfg.max_seqs) return fail(DORY_EINVAL, "seq %d out of range", seq);
  if (n < 1 || n > DORY_CHUNK_ROWS) return fail(DORY_EINVAL, "n=%d: want 1..%d", n, DORY_CHUNK_ROWS);
  if (!ids) return fail(DORY_EINVAL, "ids is NULL");
  if (loops < 1 || loops > d->cfg.max_loops) return fail(DORY_EINVAL, "loops=%d: want 1..%d", loops, d->cfg.max_loops);
  if (want < DORY_WANT_NONE || want > DORY_WANT_ALL) return fail(DORY_EINVAL, "want=%d", want);
  if (pos0 != d->seq_pos[seq])
    return fail(DORY_ESTATE, "pos0=%d but sequence %d is at %d", pos0, seq, d->seq_pos[seq]);
  int rc = check_range(d, seq, (long)pos0 + n - 1);
  if (rc) return rc;
  // dory.rs fn chunk_loops
  int L = loops;
  if (want == DORY_WANT_NONE && d->cfg.prompt_loops > 0 && d->cfg.kv_mode == DORY_KV_LAST_LOOP)
    L = std::min(loops, d->cfg.prompt_loops);
  StepArgs st;
  st.T = n;
  st.loops = L;
  st.hseq.assign(n, seq);
  st.hoff.resize(n);
  for (int i = 0; i < n; i++) st.hoff[i] = i;
  st.aseq.assign(1, seq);
  st.acnt.assign(1, n);
  const int head_rows = want == DORY_WANT_ALL ? n : (want == DORY_WANT_LAST ? 1 : 0);
  st.head_rows = head_rows;
  st.head_from = want == DORY_WANT_ALL ? 0 : n - 1;
  if ((rc = do_step(d, st, ids))) return rc;
  d->logits_rows = head_rows;
  return DORY_OK;
}

int dory_prefill(dory_t *d, int32_t seq, const int32_t *ids, int32_t n, int32_t pos0, int32_t loops, int32_t want) {
  if (!d) return fail(DORY_EINVAL, "handle is NULL");
  if (seq < 0 || seq >= d->cfg.max_seqs) return fail(DORY_EINVAL, "seq %d out of range", seq);
  if (n < 1) return fail(DORY_EINVAL, "n=%d must be positive", n);
  if (!ids) return fail(DORY_EINVAL, "ids is NULL");
  if (loops < 1 || loops > d->cfg.max_loops) return fail(DORY_EINVAL, "loops=%d: want 1..%d", loops, d->cfg.max_loops);
  if (want != DORY_WANT_NONE && want != DORY_WANT_LAST) return fail(DORY_EINVAL, "want=%d: none or last", want);
  if (pos0 != d->seq_pos[seq])
    return fail(DORY_ESTATE, "pos0=%d but sequence %d is at %d", pos0, seq, d->seq_pos[seq]);
  int rc = check_range(d, seq, (long)pos0 + n - 1);
  if (rc) return rc;
  const int S = d->prefill_rows;
  if (S < 128) {  // chunk by chunk
    for (int a0 = 0; a0 < n; a0 += DORY_CHUNK_ROWS) {
      const int m = std::min(DORY_CHUNK_ROWS, n - a0);
      if ((rc = dory_prefill_chunk(d, seq, ids + a0, m, pos0 + a0, loops, a0 + m == n ? want : DORY_WANT_NONE)))
        return rc;
    }
    return DORY_OK;
  }
  auto rows = [&](StepArgs &st, int T, int off0) {
    st.T = T;
    st.hseq.assign(T, seq);
    st.hoff.resize(T);
    for (int i = 0; i < T; i++) st.hoff[i] = off0 + i;
    st.aseq.assign(1, seq);
    st.acnt.assign(1, 0);
  };
  dory_stats sum{};
  auto add = [&]() {
    sum.weight_bytes += d->st.weight_bytes;
    sum.kv_read_bytes += d->st.kv_read_bytes;
    sum.kv_write_bytes += d->st.kv_write_bytes;
    sum.launches += d->st.launches;
    sum.gemm_launches += d->st.gemm_launches;
    sum.flops += d->st.flops;
  };
  for (int a0 = 0; a0 < n; a0 += S) {
    const int Sa = std::min(S, n - a0);
    StepArgs in;  // embedding and input block over the rows (loop slot 0, run once)
    rows(in, Sa, 0);
    in.loops = 0;
    in.do_out = false;
    if ((rc = do_step(d, in, ids + a0))) return rc;
    add();
    for (int c = 0; c < Sa; c += DORY_CHUNK_ROWS) {  // the recurrent block, chunk by chunk
      const int nc = std::min(DORY_CHUNK_ROWS, Sa - c);
      const bool last = a0 + c + nc == n;
      StepArgs r;
      rows(r, nc, c);
      r.h0 = c;
      r.do_in = r.do_out = false;
      r.loops = loops;  // dory.rs fn chunk_loops: a chunk whose logits are unread takes prompt_loops
      if (!(last && want == DORY_WANT_LAST) && d->cfg.prompt_loops > 0 && d->cfg.kv_mode == DORY_KV_LAST_LOOP)
        r.loops = std::min(loops, d->cfg.prompt_loops);
      if ((rc = do_step(d, r, ids + a0 + c))) return rc;
      add();
    }
    StepArgs out;  // output block over the rows' final states, the head of the prompt's last row
    rows(out, Sa, 0);
    out.loops = 0;
    out.do_in = false;
    out.acnt.assign(1, Sa);
    if (a0 + Sa == n && want == DORY_WANT_LAST) {
      out.head_from = Sa - 1;
      out.head_rows = 1;
    }
    if ((rc = do_step(d, out, ids + a0))) return rc;
    add();
  }
  sum.weight_bytes_device = d->st.weight_bytes_device;
  sum.kv_bytes_device = d->st.kv_bytes_device;
  d->st = sum;  // the call's totals over its steps
  d->logits_rows = want == DORY_WANT_LAST ? 1 : 0;
  return DORY_OK;
}

int dory_prefill_batch(dory_t *d, int32_t nseq, const int32_t *seqs, const int32_t *counts, const int32_t *ids,
                       int32_t loops, int32_t want) {
  if (!d) return fail(DORY_EINVAL, "handle is NULL");
  if (!seqs || !counts || !ids) return fail(DORY_EINVAL, "seqs, counts or ids is NULL");
  if (nseq < 1 || nseq > d->Tstep) return fail(DORY_EINVAL, "nseq=%d: want 1..%d", nseq, d->Tstep);
  if (loops < 1 || loops > d->cfg.max_loops) return fail(DORY_EINVAL, "loops=%d: want 1..%d", loops, d->cfg.max_loops);
  if (want < DORY_WANT_NONE || want > DORY_WANT_ALL) return fail(DORY_EINVAL, "want=%d", want);
  std::vector<char> seen(d->cfg.max_seqs, 0);
  int T = 0, rc;
  for (int j = 0; j < nseq; j++) {
    const int sq = seqs[j], n = counts[j];
    if (sq < 0 || sq >= d->cfg.max_seqs) return fail(DORY_EINVAL, "seqs[%d]=%d out of range", j, sq);
    if (seen[sq]) return fail(DORY_EINVAL, "sequence %d appears twice in one step", sq);
    seen[sq] = 1;
    if (n < 1 || n > DORY_CHUNK_ROWS) return fail(DORY_EINVAL, "counts[%d]=%d: want 1..%d", j, n, DORY_CHUNK_ROWS);
    if ((rc = check_range(d, sq, (long)d->seq_pos[sq] + n - 1))) return rc;
    T += n;
  }
  if (T > d->Tstep) return fail(DORY_EINVAL, "%d rows in one step: at most %d (max(64, max_batch))", T, d->Tstep);
  // dory.rs fn chunk_loops
  int L = loops;
  if (want == DORY_WANT_NONE && d->cfg.prompt_loops > 0 && d->cfg.kv_mode == DORY_KV_LAST_LOOP)
    L = std::min(loops, d->cfg.prompt_loops);
  StepArgs st;
  st.T = T;
  st.loops = L;
  for (int j = 0; j < nseq; j++)
    for (int i = 0; i < counts[j]; i++) {
      st.hseq.push_back(seqs[j]);
      st.hoff.push_back(i);
    }
  st.aseq.assign(seqs, seqs + nseq);
  st.acnt.assign(counts, counts + nseq);
  if (want == DORY_WANT_ALL) {
    st.head_from = 0;
    st.head_rows = T;
  } else if (want == DORY_WANT_LAST && nseq == 1) {
    st.head_from = T - 1;
    st.head_rows = 1;
  } else if (want == DORY_WANT_LAST) {
    st.head_from = 0;
    st.head_rows = T;
    for (int j = 0, r = 0; j < nseq; j++) {
      r += counts[j];
      st.head_pick.push_back(r - 1);
    }
  }
  if ((rc = do_step(d, st, ids))) return rc;
  d->logits_rows = want == DORY_WANT_ALL ? T : (want == DORY_WANT_LAST ? nseq : 0);
  return DORY_OK;
}

int dory_decode_step(dory_t *d, const int32_t *ids, const int32_t *seqs, int32_t batch, int32_t loops) {
  if (!d) return fail(DORY_EINVAL, "handle is NULL");
  if (batch < 1 || batch > d->cfg.max_batch) return fail(DORY_EINVAL, "batch=%d: want 1..%d", batch, d->cfg.max_batch);
  if (!ids || !seqs) return fail(DORY_EINVAL, "ids or seqs is NULL");
  if (loops < 1 || loops > d->cfg.max_loops) return fail(DORY_EINVAL, "loops=%d: want 1..%d", loops, d->cfg.max_loops);
  StepArgs st;
  st.T = batch;
  st.loops = loops;
  st.hseq.resize(batch);
  st.hoff.assign(batch, 0);
  st.acnt.assign(batch, 1);
  std::vector<char> seen(d->cfg.max_seqs, 0);
  int rc;
  for (int b = 0; b < batch; b++) {
    const int s = seqs[b];
    if (s < 0 || s >= d->cfg.max_seqs) return fail(DORY_EINVAL, "seqs[%d]=%d out of range", b, s);
    if (seen[s]) return fail(DORY_EINVAL, "sequence %d appears twice in one step", s);
    seen[s] = 1;
    st.hseq[b] = s;
    if ((rc = check_range(d, s, d->seq_pos[s]))) return rc;
  }
  st.aseq = st.hseq;
  st.head_rows = batch;
  st.head_from = 0;
  if ((rc = do_step(d, st, ids))) return rc;
  d->logits_rows = batch;
  return DORY_OK;
}

int dory_decode_ragged(dory_t *d, const int32_t *ids, const int32_t *seqs, int32_t batch, const int32_t *loops) {
  if (!d) return fail(DORY_EINVAL, "handle is NULL");
  if (!loops) return fail(DORY_EINVAL, "loops is NULL");
  if (batch < 1 || batch > d->cfg.max_batch) return fail(DORY_EINVAL, "batch=%d: want 1..%d", batch, d->cfg.max_batch);
  if (!ids || !seqs) return fail(DORY_EINVAL, "ids or seqs is NULL");
  int lmax = 0;
  bool same = true;
  for (int b = 0; b < batch; b++) {
    if (loops[b] < 1 || loops[b] > d->cfg.max_loops)
      return fail(DORY_EINVAL, "loops[%d]=%d: want 1..%d", b, loops[b], d->cfg.max_loops);
    lmax = std::max(lmax, (int)loops[b]);
    same &= loops[b] == loops[0];
  }
  if (same) return dory_decode_step(d, ids, seqs, batch, loops[0]);
  StepArgs st;
  st.T = batch;
  st.loops = lmax;
  std::vector<char> seen(d->cfg.max_seqs, 0);
  int rc;
  for (int b = 0; b < batch; b++) {
    const int s = seqs[b];
    if (s < 0 || s >= d->cfg.max_seqs) return fail(DORY_EINVAL, "seqs[%d]=%d out of range", b, s);
    if (seen[s]) return fail(DORY_EINVAL, "sequence %d appears twice in one step", s);
    seen[s] = 1;
    if ((rc = check_range(d, s, d->seq_pos[s]))) return rc;
  }
  // rows by loop count, most first (stable): the rows of each pass are a prefix
  st.perm.resize(batch);
  for (int b = 0; b < batch; b++) st.perm[b] = b;
  std::stable_sort(st.perm.begin(), st.perm.end(), [&](int x, int y) { return loops[x] > loops[y]; });
  st.rl.resize(batch);
  st.hseq.resize(batch);
  for (int r = 0; r < batch; r++) {
    st.rl[r] = loops[st.perm[r]];
    st.hseq[r] = seqs[st.perm[r]];
  }
  st.hoff.assign(batch, 0);
  st.aseq = st.hseq;
  st.acnt.assign(batch, 1);
  st.head_rows = batch;
  st.head_from = 0;
  if ((rc = do_step(d, st, ids))) return rc;
  d->logits_rows = batch;
  return DORY_OK;
}

int dory_decode_conf(dory_t *d, const int32_t *id, int32_t seq, float th, int32_t *passes, float *top_prob) {
  if (!d) return fail(DORY_EINVAL, "handle is NULL");
  if (!id) return fail(DORY_EINVAL, "id is NULL");
  if (seq < 0 || seq >= d->cfg.max_seqs) return fail(DORY_EINVAL, "seq %d out of range", seq);
  if (d->cfg.max_loops < 2) return fail(DORY_EINVAL, "the gate's second pass needs max_loops >= 2");
  if (!(th == th)) return fail(DORY_EINVAL, "th is NaN");
  int rc = check_range(d, seq, d->seq_pos[seq]);
  if (rc) return rc;
  StepArgs st;
  st.T = 1;
  st.hseq.assign(1, seq);
  st.hoff.assign(1, 0);
  st.aseq.assign(1, seq);
  st.acnt.assign(1, 1);
  st.head_rows = 1;
  ExitRate &ex = d->exits[seq];
  float tp = NAN;
  int np = 2;
  if (!ex.probe()) {  // no read-out: both passes at once
    st.loops = 2;
    if ((rc = do_step(d, st, id))) return rc;
  } else {
    st.loops = 1;  // the first pass, the output block and the head (the read-out)
    if ((rc = do_step(d, st, id))) return rc;
    CK(launch_top_prob(d->logits, d->dims.vocab, d->d_top, d->stream));
    CK(cudaMemcpyAsync(&tp, d->d_top, 4, cudaMemcpyDeviceToHost, d->stream));
    CK(cudaStreamSynchronize(d->stream));
    const bool stay = tp < th;
    ex.note(!stay);
    if (stay) {  // the second pass from the saved rows; the output block rewrites its rows
      StepArgs r = st;
      r.resume = true;
      r.loops = 2;
      r.first_loop = 1;
      r.hoff.assign(1, -1);  // the first step moved the position past the token
      r.acnt.assign(1, 0);
      if ((rc = do_step(d, r, id))) return rc;
    } else {
      np = 1;
    }
  }
  d->logits_rows = 1;
  if (passes) *passes = np;
  if (top_prob) *top_prob = tp;
  return DORY_OK;
}

int dory_logits(dory_t *d, int32_t row, float *dst, size_t cap) {
  if (!d || !dst) return fail(DORY_EINVAL, "NULL argument");
  if (d->logits_rows == 0) return fail(DORY_ESTATE, "the last call produced no logits");
  if (row < 0 || row >= d->logits_rows) return fail(DORY_EINVAL, "row %d of %d", row, d->logits_rows);
  if (cap < (size_t)d->dims.vocab) return fail(DORY_EINVAL, "cap %zu < vocab %d", cap, d->dims.vocab);
  CK(cudaMemcpyAsync(dst, d->logits + (size_t)row * d->dims.vocab, (size_t)d->dims.vocab * 4, cudaMemcpyDefault,
                     d->stream));
  CK(cudaStreamSynchronize(d->stream));
  return check_device_error(d);
}

int dory_logits_device(dory_t *d, const float **out, int32_t *rows) {
  if (!d || !out || !rows) return fail(DORY_EINVAL, "NULL argument");
  *out = d->logits;
  *rows = d->logits_rows;
  return DORY_OK;
}

int dory_read_hidden(dory_t *d, float *dst, size_t cap) {
  if (!d || !dst) return fail(DORY_EINVAL, "NULL argument");
  const size_t n = (size_t)d->last_rows * d->dims.hidden;
  if (cap < n) return fail(DORY_EINVAL, "cap %zu < %zu", cap, n);
  CK(cudaMemcpyAsync(dst, d->h_last, n * 4, cudaMemcpyDefault, d->stream));
  CK(cudaStreamSynchronize(d->stream));
  return check_device_error(d);
}

int dory_slot_info(dory_t *d, int32_t ordinal, int32_t *cap, int32_t *slots, int32_t *sliding) {
  if (!d) return fail(DORY_EINVAL, "handle is NULL");
  if (ordinal < 0 || ordinal >= (int)d->ords.size()) return fail(DORY_EINVAL, "ordinal %d", ordinal);
  const OrdInfo &o = d->ords[ordinal];
  if (cap) *cap = o.cap;
  if (slots) *slots = o.slots;
  if (sliding) *sliding = o.sliding ? 1 : 0;
  return DORY_OK;
}

static int check_slot(dory_t *d, int seq, int ordinal, int slot) {
  if (!d) return fail(DORY_EINVAL, "handle is NULL");
  if (seq < 0 || seq >= d->cfg.max_seqs) return fail(DORY_EINVAL, "seq %d", seq);
  if (ordinal < 0 || ordinal >= (int)d->ords.size()) return fail(DORY_EINVAL, "ordinal %d", ordinal);
  if (slot < 0 || slot >= d->ords[ordinal].slots) return fail(DORY_EINVAL, "slot %d", slot);
  return DORY_OK;
}

int dory_write_kv_rows(dory_t *d, int32_t seq, int32_t ordinal, int32_t loop_slot, int32_t pos0, int32_t n,
                       const float *k, const float *v) {
  int rc = check_slot(d, seq, ordinal, loop_slot);
  if (rc) return rc;
  if (n < 0 || !k || !v) return fail(DORY_EINVAL, "bad rows");
  int &cnt = d->app(seq, ordinal, loop_slot);
  if (pos0 != cnt) return fail(DORY_ESTATE, "pos0=%d but the slot holds %d rows", pos0, cnt);
  const OrdInfo &o = d->ords[ordinal];
  if (o.window == INT_MAX && (long)pos0 + n > o.cap) return fail(DORY_ERANGE, "rows past max_context");
  const Dims dm = d->dims;
  const size_t row = (size_t)dm.nk * dm.hd;
  Ring ring = d->ring(ordinal, loop_slot);
  const bool q8 = d->cfg.kv_quant == DORY_KV_Q8_2F;
  cudaStream_t s = d->stream;
  for (int a = 0; a < n;) {
    // at most a ring's rows per launch: two rows of one launch never share a ring row
    int m = std::min(std::min(n - a, d->Tmax), ring.cap);
    // q8: rows up to and including the freeze go one at a time in order
    const int c = cnt + a;
    int seq_rows = 0;
    if (q8 && c <= 64) seq_rows = std::min(m, 65 - c);
    if (seq_rows > 0) m = seq_rows;
    CK(cudaMemcpyAsync(d->kst, k + (size_t)a * row, (size_t)m * row * 4, cudaMemcpyDefault, s));
    CK(cudaMemcpyAsync(d->vst, v + (size_t)a * row, (size_t)m * row * 4, cudaMemcpyDefault, s));
    if (!q8) {
      CK(launch_ring_write_f32(d->kst, d->vst, m, pos0 + a, dm, ring, seq, s));
    } else if (seq_rows > 0) {
      std::vector<int> hseq(m, seq), hoff(m);
      for (int i = 0; i < m; i++) hoff[i] = pos0 + a + i;
      CK(cudaMemcpyAsync(d->d_rows, hseq.data(), m * 4, cudaMemcpyHostToDevice, s));
      CK(cudaMemcpyAsync(d->d_rows + d->Tmax, hoff.data(), m * 4, cudaMemcpyHostToDevice, s));
      Rows rows;
      rows.seq = d->d_rows;
      rows.off = d->d_rows + d->Tmax;
      rows.seq_pos = d->d_zero;
      rows.n = m;
      CK(launch_q8_append(d->kst, d->vst, (int)row, dm, rows, ring, 0, s));
    } else {
      CK(launch_q8_append_frozen(d->kst, d->vst, m, dm, seq, (long)pos0 + a, ring, s));
    }
    // the staging rows are reused by the next chunk only after these kernels ran
    CK(cudaStreamSynchronize(s));
    a += m;
  }
  cnt += n;
  return DORY_OK;
}

int dory_set_position(dory_t *d, int32_t seq, int32_t pos) {
  if (!d) return fail(DORY_EINVAL, "handle is NULL");
  if (seq < 0 || seq >= d->cfg.max_seqs || pos < 0) return fail(DORY_EINVAL, "seq %d pos %d", seq, pos);
  d->seq_pos[seq] = pos;
  CK(cudaMemcpyAsync(d->d_seq_pos + seq, &d->seq_pos[seq], 4, cudaMemcpyHostToDevice, d->stream));
  CK(cudaStreamSynchronize(d->stream));
  return DORY_OK;
}

int dory_read_kv_f32(dory_t *d, int32_t seq, int32_t ordinal, int32_t loop_slot, int32_t *tags, float *k, float *v) {
  int rc = check_slot(d, seq, ordinal, loop_slot);
  if (rc) return rc;
  if (d->cfg.kv_quant != DORY_KV_F32) return fail(DORY_EINVAL, "the rings hold q8_2f rows");
  Ring r = d->ring(ordinal, loop_slot);
  const char *slot = d->kvmem + (size_t)seq * d->seq_stride + r.off;
  const size_t n = (size_t)d->dims.nk * r.cap * d->dims.hd;
  CK(cudaStreamSynchronize(d->stream));
  if (tags) CK(cudaMemcpy(tags, slot + r.L.tags, (size_t)r.cap * 4, cudaMemcpyDefault));
  if (k) CK(cudaMemcpy(k, slot + r.L.k, n * 4, cudaMemcpyDefault));
  if (v) CK(cudaMemcpy(v, slot + r.L.v, n * 4, cudaMemcpyDefault));
  return DORY_OK;
}

int dory_read_kv_q8(dory_t *d, int32_t seq, int32_t ordinal, int32_t loop_slot, int32_t *tags, int8_t *kq, float *ks,
                    int8_t *vq, float *vs, float *kcol, float *vcol, int32_t *frozen) {
  int rc = check_slot(d, seq, ordinal, loop_slot);
  if (rc) return rc;
  if (d->cfg.kv_quant != DORY_KV_Q8_2F) return fail(DORY_EINVAL, "the rings hold f32 rows");
  Ring r = d->ring(ordinal, loop_slot);
  const char *slot = d->kvmem + (size_t)seq * d->seq_stride + r.off;
  const int nk = d->dims.nk, hd = d->dims.hd;
  const size_t rows = (size_t)nk * r.cap;
  CK(cudaStreamSynchronize(d->stream));
  if (tags) CK(cudaMemcpy(tags, slot + r.L.tags, (size_t)r.cap * 4, cudaMemcpyDefault));
  if (kq) CK(cudaMemcpy(kq, slot + r.L.kq, rows * hd, cudaMemcpyDefault));
  if (ks) CK(cudaMemcpy(ks, slot + r.L.ks, rows * (hd / 32) * 4, cudaMemcpyDefault));
  if (vq) CK(cudaMemcpy(vq, slot + r.L.vq, rows * hd, cudaMemcpyDefault));
  if (vs) CK(cudaMemcpy(vs, slot + r.L.vs, rows * 4, cudaMemcpyDefault));
  if (kcol) CK(cudaMemcpy(kcol, slot + r.L.kcol, (size_t)nk * hd * 4, cudaMemcpyDefault));
  if (vcol) CK(cudaMemcpy(vcol, slot + r.L.vcol, (size_t)nk * hd * 4, cudaMemcpyDefault));
  if (frozen) {
    std::vector<int32_t> meta(nk * 4);
    CK(cudaMemcpy(meta.data(), slot + r.L.meta, (size_t)nk * 16, cudaMemcpyDefault));
    for (int h = 0; h < nk; h++) frozen[h] = meta[h * 4 + 1];
  }
  return DORY_OK;
}

int dory_get_stats(dory_t *d, dory_stats *out) {
  if (!d || !out) return fail(DORY_EINVAL, "NULL argument");
  *out = d->st;
  return DORY_OK;
}

}  // extern "C"
