// Persistent batch-1 decode: one launch runs the whole token forward (dory.rs fn stack:
// the input block, `loops` passes of the recurrent block with the loop mix, the output
// block and the logits) as a list of stages.
//
// One block per SM, launched cooperatively so that every block is resident. Warp 0 is the
// producer: it walks this block's share of every weight matrix (a contiguous range of rows)
// in stage order, asks L2 for the bytes about two chunks ahead (cp.async.bulk.prefetch),
// and copies chunks into a ring of shared-memory slots with cp.async.bulk, completion on one
// mbarrier per slot. It never waits for activations, so HBM keeps streaming the next stages'
// weights while the consumers wait for their inputs or run attention. Warps 1..8 are the
// consumers; each awaits only the chunks that hold its rows, and a chunk's slot is free once
// they have all arrived (the first of them arrives for the consumers without a row).
//
// There is no grid barrier. A stage's outputs (GEMV rows, the attention output z) are
// tagged words: value and the stage's index + 1 in one 64-bit store. A consumer thread loads
// the words it needs and polls again until each carries the tag it expects, so a stage
// starts as soon as its own inputs exist, one L2 round trip after the last of them was
// stored, with no fence and no counter. The words are zeroed before each launch, and a
// buffer is reused only by a stage that depends on every reader of its previous contents.
// Rows that every block computes alike (the hidden row, the loop's input row) are kept in a
// private area per block and read back by the thread that wrote them. Per stage the
// consumers
//   * copy the stage's descriptor into shared memory;
//   * GEMV: build the input row in shared memory (the embedding, a row norm, or the nGPT
//     residual with the loop mix), then take the rows two at a time (or a gate/up pair) per
//     warp (bf16 weights, f32 sums; lanes split the row into 16-byte columns), park the lane
//     sums and reduce them 8 rows at a time, and apply the epilogue (SwiGLU, logit scale);
//   * attention (dory.rs fn attn_layer), in items of 32 positions of one kv head: the K and
//     V rows of an item are contiguous in the ring and arrive with two bulk copies; meanwhile
//     warp h rotates and normalises query head h of the group from the raw projection row
//     (q = s_q^2 q^), and in the item that holds the row's own position one warp rotates and
//     normalises the new key, puts key and value into the tile and writes them (and the
//     position tag) to the ring; warp h then scores (lane = key), takes the item's softmax and
//     value sum (with four query heads a group, warps h and h + 4 share head h, half of its
//     dimensions each); one block per query head (or the last item of a kv head) merges the
//     items and applies the output gate.
// Every wait is bounded. When one runs out the block records error 6, stops at the next
// team-wide check, lets its copies in flight land and returns; the other blocks then give up
// waiting for its words. The last block to finish advances the row's position.
#include <algorithm>
#include <climits>

#include "async.cuh"
#include "common.cuh"
#include "kernels.h"
#include "team.cuh"

namespace dory {

namespace {

constexpr int MW = 8;                             // consumer warps
constexpr int MTHREADS = 32 * (MW + 1);           // and the producer warp
constexpr int NS = 7;                             // weight slots
constexpr uint32_t SLOT = 26 * 1024;              // bytes per slot
constexpr int RMAX = 8;                           // rows (or row pairs) per chunk at most
static_assert(RMAX <= 32, "a chunk's rows fit the parked sums of one warp in whole rounds");
constexpr int EPI_ROWS = 256;                     // a block's rows of one GEMV at most
constexpr uint32_t WORK = 32 * 1024;              // input row, or attention tiles and merge scratch
constexpr int AK = MEGA_AK;                       // positions per attention item
constexpr int ERR_MEGA = 6;                       // dev_err: a wait of the persistent kernel ran out
static_assert(EPI_ROWS == 32 * MW, "a consumer thread holds one row's epilogue scales");
static_assert(sizeof(MegaStage) % 4 == 0 && sizeof(MegaStage) / 4 <= 32 * MW, "stage copy by the team");

struct Ctl {
  volatile int abort;  // a wait ran out somewhere in the block
  int decision;        // team-wide copy of `abort`, written by the team's first thread
  int last;            // this block merges the kv head's items
  int seq;             // the row's sequence and position
  long long p;
};

// Cycle counts of the current stage's phases (trace only; the team's first thread).
__shared__ unsigned long long trace_acc[6];

// The chunk each weight slot was last given (written by the producer before the copy). A
// chunk's warp waits for its number before it waits on the slot's barrier: a slot may still
// hold a chunk several phases older, which a parity wait could not tell apart.
__shared__ volatile int slot_chunk[NS];

// Optional per-stage timestamps (off when the pointer is null).
struct Tracer {
  unsigned long long *p;
  __device__ __forceinline__ void mark(int stage, int event) const {
    if (!p) return;
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    p[((size_t)stage * gridDim.x + blockIdx.x) * MEGA_TRACE_EVENTS + event] = t;
  }
  __device__ __forceinline__ void add(int, int event, long long v) const {
    if (p) trace_acc[event - 8] += (unsigned long long)v;
  }
  __device__ __forceinline__ void zero(int) const {
    if (p)
      for (int e = 0; e < 6; e++) trace_acc[e] = 0;
  }
  __device__ __forceinline__ void flush(int stage, int n = 6) const {
    if (p)
      for (int e = 0; e < n; e++)
        p[((size_t)stage * gridDim.x + blockIdx.x) * MEGA_TRACE_EVENTS + 8 + e] = trace_acc[e];
  }
  __device__ __forceinline__ long long clk() const { return p ? clock64() : 0; }
};

__device__ __forceinline__ void flag_error(Ctl &ctl, int *err) {
  if (!ctl.abort) {
    ctl.abort = 1;
    atomicExch(err, ERR_MEGA);
  }
}

// Team-uniform check of the abort flag (one thread reads it, all see the same value).
__device__ __forceinline__ bool team_ok(const WarpTeam &tm, Ctl &ctl) {
  tm.sync();
  if (tm.tid() == 0) ctl.decision = ctl.abort;
  tm.sync();
  return ctl.decision == 0;
}

// Wait until `*ctr >= target` (the RoPE entries written).
__device__ bool team_wait_counter(const WarpTeam &tm, const int *ctr, int target, Ctl &ctl, int *err,
                                  uint32_t limit) {
  if (tm.tid() == 0) {
    uint32_t i = 0;
    while (ld_acquire_gpu(ctr) < target) {
      if (ctl.abort) break;
      if (++i > limit) {
        flag_error(ctl, err);
        break;
      }
    }
    ctl.decision = ctl.abort;
  }
  tm.sync();
  return ctl.decision == 0;
}


// Words p[off[i]] of a tagged row into v[i], re-polling those that do not carry `tag` yet.
// False when the polls ran out or the block stopped.
template <int N>
__device__ __forceinline__ bool await_words(const unsigned long long *p, const int (&off)[N], uint32_t tag,
                                            float (&v)[N], const Ctl &ctl, uint32_t limit) {
  uint32_t pend = 0;
#pragma unroll
  for (int i = 0; i < N; i++)
    if (!ld_tagged(p + off[i], tag, v[i])) pend |= 1u << i;
  for (uint32_t k = 0; pend && k < limit && !ctl.abort; k++) {
#pragma unroll
    for (int i = 0; i < N; i++)
      if (((pend >> i) & 1u) && ld_tagged(p + off[i], tag, v[i])) pend &= ~(1u << i);
  }
  return pend == 0;
}

// 4 consecutive tagged words p[0..3] (16-byte aligned) into v
__device__ __forceinline__ bool await4(const unsigned long long *p, uint32_t tag, float4 &v, const Ctl &ctl,
                                       uint32_t limit) {
  for (uint32_t k = 0; k <= limit && !ctl.abort; k++)
    if (ld_tagged4(p, tag, v)) return true;
  return false;
}

// ---- producer -----------------------------------------------------------------------------

// A walk over this block's rows of the GEMV stages, chunk by chunk.
struct ChunkWalk {
  int s, r0, re, K, R;
  long pair;
  const __nv_bfloat16 *W;
  bool ok;
  __device__ void seek(const MegaArgs &a, int from) {
    const int G = gridDim.x, b = blockIdx.x;
    for (s = from; s < a.nstages; s++) {
      const MegaStage &st = a.stages[s];
      if (st.kind != MK_GEMV) continue;
      const int rb = (int)((unsigned)st.N * (unsigned)b / (unsigned)G);  // N * G < 2^32 (host limit)
      re = (int)((unsigned)st.N * (unsigned)(b + 1) / (unsigned)G);
      if (rb < re) {
        r0 = rb;
        K = st.K;
        R = st.R;
        pair = st.pair;
        W = st.W;
        ok = true;
        return;
      }
    }
    ok = false;
  }
  __device__ int rows() const { return min(R, re - r0); }
  __device__ void step(const MegaArgs &a) {
    r0 += rows();
    if (r0 >= re) seek(a, s + 1);
  }
};

__device__ void produce(const MegaArgs &a, uint8_t *ring, uint64_t *full, uint64_t *empty, Ctl &ctl) {
  const Tracer tr{a.trace};
  // weights are read once per step: they go through L2 evict-first, so that the step's
  // activations, partials and counters stay there
  const uint64_t pol = l2_evict_first_policy();
  ChunkWalk cp, pf;  // copies, and the L2 prefetch ahead of them
  cp.seek(a, 0);
  pf.seek(a, 0);
  long ahead = 0;  // bytes asked of L2 and not yet copied
  int c = 0;       // chunks issued
  int marked = -1;
  bool ok = true;
  while (cp.ok) {
    while (pf.ok && ahead < a.prefetch_ahead) {
      const uint32_t pb = (uint32_t)pf.rows() * pf.K * 2;
      prefetch_l2_bulk(pf.W + (size_t)pf.r0 * pf.K, pb);
      if (pf.pair > 0) prefetch_l2_bulk(pf.W + (size_t)(pf.r0 + pf.pair) * pf.K, pb);
      ahead += pf.pair > 0 ? 2 * pb : pb;
      pf.step(a);
    }
    const int sl = c % NS;
    if (c >= NS) {
      // wait for the slot; while it is taken (the consumers are at attention or a barrier),
      // keep HBM busy by asking L2 for the next weights, up to a longer lead
      const uint32_t eb = smem_addr(&empty[sl]), par = ((c / NS) - 1) & 1;
      uint32_t polls = 0;
      bool free_ = false;
      while (!(free_ = mbar_test(eb, par))) {
        if (ctl.abort || ++polls > MBAR_WAIT_LIMIT) break;
        if (pf.ok && ahead < a.stall_lead) {
          const uint32_t pb = (uint32_t)pf.rows() * pf.K * 2;
          prefetch_l2_bulk(pf.W + (size_t)pf.r0 * pf.K, pb);
          if (pf.pair > 0) prefetch_l2_bulk(pf.W + (size_t)(pf.r0 + pf.pair) * pf.K, pb);
          ahead += pf.pair > 0 ? 2 * pb : pb;
          pf.step(a);
        }
      }
      if (!free_) {
        ok = false;
        break;
      }
    }
    // with a cap on copies in flight, the copy max_inflight back lands first: bytes queued
    // beyond what keeps HBM busy only delay the step's latency-bound loads
    const int back = c - a.max_inflight;
    if (a.max_inflight > 0 && a.max_inflight < NS && back >= 0 &&
        !mbar_wait(smem_addr(&full[back % NS]), (back / NS) & 1, &ctl.abort)) {
      ok = false;
      break;
    }
    if (cp.s != marked) {
      tr.mark(cp.s, 5);
      marked = cp.s;
    }
    slot_chunk[sl] = c;
    const uint32_t bytes = (uint32_t)cp.rows() * cp.K * 2, bar = smem_addr(&full[sl]);
    const uint32_t dst = smem_addr(ring + (size_t)sl * SLOT);
    mbar_expect_tx(bar, cp.pair > 0 ? 2 * bytes : bytes);
    bulk_g2s_hint(dst, cp.W + (size_t)cp.r0 * cp.K, bytes, bar, pol);
    if (cp.pair > 0) bulk_g2s_hint(dst + bytes, cp.W + (size_t)(cp.r0 + cp.pair) * cp.K, bytes, bar, pol);
    ahead -= cp.pair > 0 ? 2 * bytes : bytes;
    c++;
    const int s_before = cp.s;
    cp.step(a);
    if (!cp.ok || cp.s != s_before) tr.mark(s_before, 6);
  }
  if (!ok) flag_error(ctl, a.err);
  // the block may not exit while a copy into its shared memory is in flight
  for (int k = max(0, c - NS); k < c; k++) mbar_wait(smem_addr(&full[k % NS]), (k / NS) & 1);
}

// ---- GEMV stage ---------------------------------------------------------------------------

// A stage's rows in groups of two (two rows, or one gate/up pair, share each load of the
// input row): group g of the block's rows belongs to consumer warp g mod MW, which awaits only
// the chunks that hold its groups (a chunk holds at most MW groups). The lanes split a row
// into 16-byte columns (lane l: columns l, l + 32, ...) against the input row in shared
// memory, held as two halves (inputs 8u..8u+3 at float4 u of the first, 8u+4..8u+7 of the
// second) so that the loads are conflict-free. A row's 32 lane sums are not reduced at once:
// the warp parks them in shared memory and reduces 8 rows together (lane 4i + q adds 8 of row
// i's sums, two shuffles finish), so that no shuffle chain stands between one row's loads
// and the next; lane 4i then applies the epilogue (SwiGLU, logit scale) and stores.
constexpr int PEND = 8;  // rows a warp parks before it reduces them

// The parked sums of np (<= PEND) rows: reduce, apply the epilogue, store (tagged words, or
// plain floats for the logits). Dual: the gate sums at pg, the up sums at pu, one row each.
__device__ __forceinline__ void flush_rows(const MegaStage &st, bool dual, int rb, int np, const float *pg,
                                           const float *pu, const int *prow, const float (*epi)[EPI_ROWS],
                                           uint32_t tag) {
  const int lane = threadIdx.x & 31, i = lane >> 2, q = lane & 3;
  __syncwarp();
  const float4 *g4 = reinterpret_cast<const float4 *>(pg + i * 32 + q * 8);
  const float4 ga = g4[0], gb = g4[1];
  float g = ((ga.x + ga.y) + (ga.z + ga.w)) + ((gb.x + gb.y) + (gb.z + gb.w)), u = 0.f;
  if (dual) {
    const float4 *u4 = reinterpret_cast<const float4 *>(pu + i * 32 + q * 8);
    const float4 ua = u4[0], ub = u4[1];
    u = ((ua.x + ua.y) + (ua.z + ua.w)) + ((ub.x + ub.y) + (ub.z + ub.w));
  }
  g += __shfl_xor_sync(0xffffffffu, g, 1);
  g += __shfl_xor_sync(0xffffffffu, g, 2);
  u += __shfl_xor_sync(0xffffffffu, u, 1);
  u += __shfl_xor_sync(0xffffffffu, u, 2);
  if (q == 0 && i < np) {
    const int jr = prow[i];
    const int mode = st.ep.mode;
    float y;
    if (mode == EPI_SCALE) {
      y = g * epi[0][jr];
    } else if (mode == EPI_SILU) {
      const float gs = g * epi[0][jr];
      y = gs * sigmoidf_(gs) * (u * epi[1][jr]);
    } else {
      y = g;
    }
    if (st.Yt) st_tagged(st.Yt + rb + jr, y, tag);
    else st.Y[rb + jr] = y;
  }
  __syncwarp();  // the parked sums may be overwritten
}

// One body for every GEMV stage: a group is two weight rows against the shared input row,
// either two consecutive rows of a chunk or (dual) the gate and up rows of one SwiGLU pair,
// so that each load of the input row serves two rows.
__device__ void gemv_rows(const WarpTeam &tm, const MegaStage &st, int rb, int re, int c0, const uint8_t *ring,
                          uint64_t *full, uint64_t *empty, const float *xs, float *park, const float (*epi)[EPI_ROWS],
                          Ctl &ctl, int *err, const Tracer &tr, int s) {
  const bool dual = st.pair > 0;
  const int lane = threadIdx.x & 31, cw = tm.warp();
  const int K = st.K, R = st.R, nu = K / 8;  // 16-byte columns per row
  const int n = re - rb;                     // rows (pairs) of this block
  const int per = dual ? 1 : 2;              // rows (pairs) a group covers; R is a multiple of it
  const int ngroups = (n + per - 1) / per;
  // this warp's parked lane sums [PEND][32] (gate, then up), and their rows
  float *pg = park + cw * (dual ? 2 : 1) * PEND * 32, *pu = pg + PEND * 32;
  __shared__ int prow_all[MW][PEND];
  int *prow = prow_all[cw];
  int np = 0;
  // a 16-byte column of weights against the input row: two chains of paired FMAs
  auto dot8 = [&](const uint4 &wq, const float4 &p, const float4 &q, float2 &a0, float2 &a1) {
    float wv[8];
    unpack8(wq, wv);
    a0 = ffma2(make_float2(wv[0], wv[1]), make_float2(p.x, p.y), a0);
    a1 = ffma2(make_float2(wv[2], wv[3]), make_float2(p.z, p.w), a1);
    a0 = ffma2(make_float2(wv[4], wv[5]), make_float2(q.x, q.y), a0);
    a1 = ffma2(make_float2(wv[6], wv[7]), make_float2(q.z, q.w), a1);
  };
  tr.zero(s);
  for (int gi = cw; gi < ngroups; gi += MW) {  // this warp's groups
    const int x = gi * per / R, c = c0 + x, sl = c % NS;
    long long t0 = tr.clk();
    bool landed = false;
    for (uint32_t i = 0; i < MBAR_WAIT_LIMIT && !ctl.abort; i++)
      if (slot_chunk[sl] == c) {
        landed = mbar_wait(smem_addr(&full[sl]), (c / NS) & 1, &ctl.abort);
        break;
      }
    long long t1 = tr.clk();
    tr.add(s, 8, t1 - t0);
    if (!landed && lane == 0) flag_error(ctl, err);  // the block stops at the stage's end
    const int r0 = x * R, nr = min(R, n - r0), j = gi * per - r0;
    if (landed) {
      // a group's second row past the chunk's last one reads stale slot bytes: not stored
      float2 a0 = make_float2(0.f, 0.f), a1 = a0, b0 = a0, b1 = a0;
      const uint4 *wc = reinterpret_cast<const uint4 *>(ring + (size_t)sl * SLOT);
      const uint4 *w0 = wc + (size_t)j * nu, *w1 = wc + (size_t)(dual ? nr + j : j + 1) * nu;
#pragma unroll 4
      for (int u = lane; u < nu; u += 32) {
        const float4 p = reinterpret_cast<const float4 *>(xs)[u], q = reinterpret_cast<const float4 *>(xs)[nu + u];
        dot8(w0[u], p, q, a0, a1);
        dot8(w1[u], p, q, b0, b1);
      }
      const float sa = (a0.x + a0.y) + (a1.x + a1.y), sb = (b0.x + b0.y) + (b1.x + b1.y);
      pg[np * 32 + lane] = sa;
      if (lane == 0) prow[np] = gi * per;
      if (dual) {
        pu[np * 32 + lane] = sb;
        np++;
      } else if (j + 1 < nr) {
        pg[(np + 1) * 32 + lane] = sb;
        if (lane == 0) prow[np + 1] = gi * per + 1;
        np += 2;
      } else {
        np++;
      }
    }
    // one place reduces and stores: when two more rows might not fit, and after the last group
    if (np > PEND - 2 || (gi + MW >= ngroups && np > 0)) {
      flush_rows(st, dual, rb, np, pg, pu, prow, epi, s + 1);
      np = 0;
    }
    __syncwarp();
    // the slot is free after MW arrivals: one per group of the chunk, the first group's warp
    // also arriving for the warps that hold no group of it
    const int ng = (nr + per - 1) / per;
    if (lane == 0 && !ctl.abort) mbar_arrive_n(smem_addr(&empty[sl]), j == 0 ? MW - ng + 1 : 1);
    tr.add(s, 9, tr.clk() - t1);
  }
  tr.flush(s, 4);  // (12 .. 14 hold the input row's wait)
}

// ---- input rows ---------------------------------------------------------------------------
//
// One row. Thread t owns the float4 chunks t + 256 j (j < KC) and stores them to the shared
// input row as two halves (chunk c at (c & 1) * K/8 + c/2), so that a lane reading the 8
// inputs of a 16-byte weight column reads float4 u of each half: consecutive lanes,
// consecutive addresses. Each kind of input row has its own function, so that a stage runs
// (and fetches) only its own code. All end with a team sync and return false when a tagged
// wait ran out or the block stopped.

// How an input row awaits tagged words: the block's stop flag, the polls of a word before
// it gives up, the block's private rows, and (trace only, or null) where to stamp the time
// the words were all in ([0]), count the poll rounds ([1]) and stamp the first poll ([2]).
struct TagWait {
  const volatile int *abort;
  uint32_t limit;
  float *priv;
  unsigned long long *trace;
};

// Chunks tid + 256 j (< nch) of a row of tagged words into v, polled again (the whole set)
// until every word carries `tag`.
// A failed poll of a row sleeps this long before the next: while a stage waits (the O
// projection during an attention stage), up to 150 blocks poll the same few lines of L2.
constexpr unsigned POLL_SLEEP_NS = 200;

template <int KC>
__device__ __forceinline__ bool await_row(const unsigned long long *src, uint32_t tag, int tid, int nch,
                                          float4 (&v)[KC], const TagWait &tw) {
  if (tw.trace && tid == 0) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    tw.trace[2] = t;
  }
  for (uint32_t i = 0; i <= tw.limit && !*tw.abort; i++) {
    bool all = true;
#pragma unroll
    for (int j = 0; j < KC; j++) {
      const int c = tid + j * 32 * MW;
      if (c < nch) all &= ld_tagged4(src + 4 * (size_t)c, tag, v[j]);
    }
    if (all) {
      if (tw.trace && tid == 0) tw.trace[1] += i + 1;
      return true;
    }
    __nanosleep(POLL_SLEEP_NS);
  }
  return false;
}

__device__ __forceinline__ void stamp_in(const TagWait &tw, int tid) {
  if (tw.trace && tid == 0) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    tw.trace[0] = t;
  }
}

__device__ __forceinline__ float sq4(const float4 &v) { return v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w; }
__device__ __forceinline__ float4 mul4(const float4 &v, float f) {
  return make_float4(v.x * f, v.y * f, v.z * f, v.w * f);
}

__shared__ float red_in[2][TEAM_MAX_WARPS];

// Sums of two values over the consumer warps, out of line: inline, each of the reductions
// of the input rows added about 3.7 KB of code to the stage.
__device__ __noinline__ float2 row_sum2(float a, float b) {
  const WarpTeam tm{1, MW, 1};
  team_sum2(tm, a, b, red_in);
  return make_float2(a, b);
}
__device__ __forceinline__ float row_sum(float a) { return row_sum2(a, 0.f).x; }

__device__ __forceinline__ float4 *xs_chunk(float *xs, int nch, int c) {
  return reinterpret_cast<float4 *>(xs) + (c & 1) * (nch / 2) + (c >> 1);
}

// IN_NORM: x / sqrt(sum x^2 + eps) (dory.rs fn justnorm); IN_PLAIN: x. The row is tagged
// words of an earlier stage, or a row of the block's private area.
template <int KC>
__device__ __forceinline__ bool in_norm(const WarpTeam &tm, const GemvIn &in, int K, float *xs, const TagWait &tw) {
  const int tid = tm.tid(), nch = K / 4;
  float4 x[KC];
#pragma unroll
  for (int j = 0; j < KC; j++) x[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  bool ok = true;
  if (in.src_t) {
    ok = await_row<KC>(in.src_t, in.src_tag, tid, nch, x, tw);
  } else {
    const float4 *src = reinterpret_cast<const float4 *>(in.src_pv ? tw.priv + (size_t)(in.src_pv - 1) * K : in.src);
#pragma unroll
    for (int j = 0; j < KC; j++)
      if (tid + j * 32 * MW < nch) x[j] = src[tid + j * 32 * MW];
  }
  stamp_in(tw, tid);
  if (in.mode == IN_NORM) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < KC; j++) ss += sq4(x[j]);
    const float inv = 1.f / sqrtf(row_sum(ss) + DORY_EPS);
#pragma unroll
    for (int j = 0; j < KC; j++) x[j] = mul4(x[j], inv);
  }
#pragma unroll
  for (int j = 0; j < KC; j++)
    if (tid + j * 32 * MW < nch) *xs_chunk(xs, nch, tid + j * 32 * MW) = x[j];
  tm.sync();
  return ok;
}

// The token's embedding row (bf16 table; an id outside the vocabulary gives zeros), stored
// as the hidden row (K <= 2048: two chunks a thread).
__device__ __forceinline__ bool in_embed(const WarpTeam &tm, const GemvIn &in, int K, float *xs, const TagWait &tw) {
  const int tid = tm.tid(), nch = K / 4;
  const int id = in.ids[0];
  const bool lead = blockIdx.x == 0;
#pragma unroll
  for (int j = 0; j < 2; j++) {
    const int c = tid + j * 32 * MW;
    if (c >= nch) continue;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (id >= 0 && id < in.vocab) {
      const uint2 u = __ldg(reinterpret_cast<const uint2 *>(in.embed + (size_t)id * K) + c);
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
      x = make_float4(a.x, a.y, b.x, b.y);
    }
    *xs_chunk(xs, nch, c) = x;
    if (lead) reinterpret_cast<float4 *>(in.h_dst)[c] = x;
    if (in.hdst_pv) reinterpret_cast<float4 *>(tw.priv + (size_t)(in.hdst_pv - 1) * K)[c] = x;
  }
  tm.sync();
  return true;
}

// IN_RESID (K <= 2048: two chunks a thread): the nGPT residual x = (x^ + alpha (out^ -
// x^))^ (dory.rs fn slerp), then the loop mix (dory.rs fn stack): MIX_LOOP / MIX_END state =
// x^; MIX_BEGIN input = state = x; MIX_BEGIN / MIX_LOOP / MIX_RESUME x = (x + input)^. The
// new hidden row goes to the block's private area, and from the leading block to h_dst; the
// leading block also stores the state and input rows.
__device__ __forceinline__ bool in_resid(const WarpTeam &tm, const GemvIn &in, int K, float *xs, const TagWait &tw) {
  constexpr int KC = 2;
  const int tid = tm.tid(), nch = K / 4;
  const bool lead = blockIdx.x == 0;
  const bool has_in = in.mix == MIX_LOOP || in.mix == MIX_RESUME;
  const float4 *src = reinterpret_cast<const float4 *>(in.src_pv ? tw.priv + (size_t)(in.src_pv - 1) * K : in.src);
  const float4 *inr =
      reinterpret_cast<const float4 *>(in.input_pv ? tw.priv + (size_t)(in.input_pv - 1) * K : in.input);
  float4 x[KC], o[KC], al[KC], inp[KC];
#pragma unroll
  for (int j = 0; j < KC; j++) {
    const int c = tid + j * 32 * MW;
    x[j] = o[j] = al[j] = inp[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c < nch) {
      x[j] = in.src_pv ? src[c] : __ldcg(src + c);
      if (in.alpha) al[j] = __ldg(reinterpret_cast<const float4 *>(in.alpha) + c);
      if (has_in) inp[j] = in.input_pv ? inr[c] : __ldcg(inr + c);
    }
  }
  bool ok = true;
  if (in.alpha) ok = await_row<KC>(in.out_t, in.out_tag, tid, nch, o, tw);
  stamp_in(tw, tid);
  if (in.alpha) {
    float sx = 0.f, so = 0.f;
#pragma unroll
    for (int j = 0; j < KC; j++) {
      sx += sq4(x[j]);
      so += sq4(o[j]);
    }
    const float2 sxo = row_sum2(sx, so);
    sx = sxo.x;
    so = sxo.y;
    const float ix = 1.f / sqrtf(sx + DORY_EPS), io = 1.f / sqrtf(so + DORY_EPS);
    float sr = 0.f;
#pragma unroll
    for (int j = 0; j < KC; j++) {
      const float4 xh = mul4(x[j], ix), oh = mul4(o[j], io);
      x[j] = make_float4(xh.x + al[j].x * (oh.x - xh.x), xh.y + al[j].y * (oh.y - xh.y),
                         xh.z + al[j].z * (oh.z - xh.z), xh.w + al[j].w * (oh.w - xh.w));
      sr += sq4(x[j]);
    }
    const float inv = 1.f / sqrtf(row_sum(sr) + DORY_EPS);
#pragma unroll
    for (int j = 0; j < KC; j++) x[j] = mul4(x[j], inv);
  }
  if (in.mix == MIX_LOOP || in.mix == MIX_END) {  // state = h^
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < KC; j++) ss += sq4(x[j]);
    const float inv = 1.f / sqrtf(row_sum(ss) + DORY_EPS);
#pragma unroll
    for (int j = 0; j < KC; j++) {
      x[j] = mul4(x[j], inv);
      const int c = tid + j * 32 * MW;
      if (lead && c < nch) reinterpret_cast<float4 *>(in.state)[c] = x[j];
    }
  }
  if (in.mix == MIX_BEGIN || in.mix == MIX_LOOP || in.mix == MIX_RESUME) {  // h = (state + input)^
    // (MIX_RESUME: src is the saved state row, taken as it is)
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < KC; j++) {
      const int c = tid + j * 32 * MW;
      if (in.mix == MIX_BEGIN) {
        inp[j] = x[j];
        if (c < nch) {
          if (lead) {
            reinterpret_cast<float4 *>(in.input)[c] = x[j];
            reinterpret_cast<float4 *>(in.state)[c] = x[j];
          }
          if (in.input_pv) reinterpret_cast<float4 *>(tw.priv + (size_t)(in.input_pv - 1) * K)[c] = x[j];
        }
      }
      x[j] = make_float4(x[j].x + inp[j].x, x[j].y + inp[j].y, x[j].z + inp[j].z, x[j].w + inp[j].w);
      ss += sq4(x[j]);
    }
    const float inv = 1.f / sqrtf(row_sum(ss) + DORY_EPS);
#pragma unroll
    for (int j = 0; j < KC; j++) x[j] = mul4(x[j], inv);
  }
#pragma unroll
  for (int j = 0; j < KC; j++) {
    const int c = tid + j * 32 * MW;
    if (c < nch) {
      *xs_chunk(xs, nch, c) = x[j];
      if (lead && in.h_dst) reinterpret_cast<float4 *>(in.h_dst)[c] = x[j];
      if (in.hdst_pv) reinterpret_cast<float4 *>(tw.priv + (size_t)(in.hdst_pv - 1) * K)[c] = x[j];
    }
  }
  tm.sync();
  return ok;
}

// Returns false (team-uniformly) when the block has stopped.
__device__ __noinline__ bool gemv_stage(const WarpTeam &tm, const MegaArgs &a, const MegaStage &st, int s, int &c,
                           const uint8_t *ring, uint64_t *full, uint64_t *empty, float *xs,
                           float (*epi)[EPI_ROWS], Ctl &ctl) {
  ring = in_shared(ring);  // shared-space loads and stores (this function is not inlined)
  xs = in_shared(xs);
  epi = in_shared(epi);
  const Tracer tr{tm.tid() == 0 ? a.trace : nullptr};
  const int G = gridDim.x, b = blockIdx.x;
  const int N = st.N, K = st.K;
  // 32-bit: N * G < 2^32 (the host's limit on rows per block); a 64-bit division is a subroutine
  const int rb = (int)((unsigned)N * (unsigned)b / (unsigned)G);
  const int re = (int)((unsigned)N * (unsigned)(b + 1) / (unsigned)G);
  // the epilogue's per-row scales of this block's rows (re - rb <= EPI_ROWS = team size),
  // held in registers while the input row's loads are in flight, stored to shared memory after
  const int ei = tm.tid();
  const bool has_e = st.ep.mode != EPI_STORE && ei < re - rb;
  float e0 = 0.f, e1 = 0.f;
  if (has_e) {
    e0 = __ldg(st.ep.vec + rb + ei);
    if (st.ep.mode == EPI_SILU) e1 = __ldg(st.ep.vec2 + rb + ei);
  }
  const int kc = (K / 4 + tm.size() - 1) / tm.size();  // float4 chunks per thread
  // K is at most 6144 (the host's limit): 2 or 6 float4 chunks a thread. Two sizes only: with
  // four (2, 4, 6, 8) the stage's register allocation spilled and a token took 4.4% longer;
  // a residual of 6 chunks (two rows of tagged words awaited at once) spilled too, inline or
  // called, so hidden rows (residuals, embeddings) are at most 2048 wide here.
  // trace: events 12 and 13 of a GEMV stage are the time its input words were all in and the poll rounds
  unsigned long long *tw_trace =
      tr.p ? tr.p + ((size_t)s * gridDim.x + blockIdx.x) * MEGA_TRACE_EVENTS + 12 : nullptr;
  if (tw_trace) tw_trace[1] = 0;
  const TagWait tw{&ctl.abort, a.spin_limit, a.priv + (size_t)b * a.priv_stride, tw_trace};
  bool in_ok;
  if (st.in.mode == IN_RESID) in_ok = in_resid(tm, st.in, K, xs, tw);
  else if (st.in.mode == IN_EMBED) in_ok = in_embed(tm, st.in, K, xs, tw);
  else if (kc <= 2) in_ok = in_norm<2>(tm, st.in, K, xs, tw);
  else in_ok = in_norm<6>(tm, st.in, K, xs, tw);
  if (!in_ok) flag_error(ctl, a.err);  // the rows below see the stop and skip their work
  if (st.ep.mode != EPI_STORE) {
    if (has_e) {
      epi[0][ei] = e0;
      epi[1][ei] = e1;
    }
    tm.sync();
  }
  tr.mark(s, 2);
  float *park = xs + K;  // the rows' parked lane sums, after the input row
  gemv_rows(tm, st, rb, re, c, ring, full, empty, xs, park, epi, ctl, a.err, tr, s);
  c += re > rb ? (re - rb + st.R - 1) / st.R : 0;
  const bool ok = team_ok(tm, ctl);
  tr.mark(s, 3);
  return ok;
}

// ---- attention stage ----------------------------------------------------------------------

// Item partials of an attention stage: outputs o [nk][maxblk][rep][hd] (unnormalised),
// then (max, sum) pairs [nk][maxblk][rep][2].
__device__ __forceinline__ float *part_o(const MegaStage &st, int rep, int hd, int kh, int blk, int h) {
  return st.part + (((size_t)kh * st.maxblk + blk) * rep + h) * hd;
}
__device__ __forceinline__ float *part_ml(const MegaStage &st, int nk, int rep, int hd, int kh, int blk, int h) {
  return st.part + (size_t)nk * st.maxblk * rep * hd + (((size_t)kh * st.maxblk + blk) * rep + h) * 2;
}

// Merge the items of kv head kh and gate. Thread t takes the 4 outputs q = t mod nq of the
// group's rep*hd and the items g, g + G, ... (g = t / nq, G = team size / nq groups), loads
// all of their partials at once (IB per round), folds them with a running max; the groups
// meet in shared memory `scr` and the first nq threads finish: y = sum o e^(m - M) / sum l
// e^(m - M), z = y * sigmoid(g * s_g^2).
template <int HD>
__device__ __forceinline__ void merge_items(const WarpTeam &tm, const MegaArgs &a, const MegaStage &st, const Dims &d,
                                            int kh, int nblk, int s, float *scr, Ctl &ctl, const Tracer &tr) {
  const long long t_in = tr.clk();
  constexpr int IB = 9;  // items a thread loads per round
  const int rep = d.nh / d.nk, nq = rep * HD / 4;
  const int groups = tm.size() / nq;
  const size_t col0 = (size_t)kh * rep * HD;
  float4 *Acc = reinterpret_cast<float4 *>(scr);  // [groups][nq]
  float *Ms = scr + 4 * groups * nq, *Ls = Ms + groups * nq;
  {  // nq = rep * hd / 4 <= 256 <= team size (rep <= 8, hd <= 128)
    const int t = tm.tid();
    const int q = t % nq, g = t / nq;
    const bool act = g < groups;
    const int h = act ? (q * 4) / HD : 0, dim = act ? (q * 4) % HD : 0;
    float M = -INFINITY, L = 0.f;
    float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
    // the gate inputs of the thread's outputs, in flight with the partials
    const size_t c = col0 + (size_t)q * 4;
    float4 gr = make_float4(0.f, 0.f, 0.f, 0.f), sg = gr;
    if (g == 0 && act) {
      sg = __ldg(reinterpret_cast<const float4 *>(st.sg + c));
      if (!await4(st.qkvg_t + (size_t)(d.nh + 2 * d.nk) * HD + c, st.qtag, gr, ctl, a.spin_limit))
        flag_error(ctl, a.err);
    }
    for (int i0 = g; act && i0 < nblk; i0 += IB * groups) {
      float4 o[IB];
      float2 ml[IB];
#pragma unroll
      for (int u = 0; u < IB; u++) {
        const int it = i0 + u * groups;
        const bool in = it < nblk;
        o[u] = in ? __ldcg(reinterpret_cast<const float4 *>(part_o(st, rep, HD, kh, it, h) + dim))
                  : make_float4(0.f, 0.f, 0.f, 0.f);
        ml[u] = in ? __ldcg(reinterpret_cast<const float2 *>(part_ml(st, d.nk, rep, HD, kh, it, h)))
                   : make_float2(-INFINITY, 0.f);
      }
#pragma unroll
      for (int u = 0; u < IB; u++) {
        if (ml[u].x == -INFINITY) continue;
        const float nm = fmaxf(M, ml[u].x);
        const float sa = M == -INFINITY ? 0.f : expf(M - nm), sb = expf(ml[u].x - nm);
        L = L * sa + ml[u].y * sb;
        A = make_float4(A.x * sa + o[u].x * sb, A.y * sa + o[u].y * sb, A.z * sa + o[u].z * sb,
                        A.w * sa + o[u].w * sb);
        M = nm;
      }
    }
    if (act) {
      Acc[g * nq + q] = A;
      Ms[g * nq + q] = M;
      Ls[g * nq + q] = L;
    }
    tr.add(0, 12, tr.clk() - t_in);
    tm.sync();
    tr.add(0, 13, tr.clk() - t_in);
    if (g == 0 && act) {
      float Mx = -INFINITY;
      for (int k = 0; k < groups; k++) Mx = fmaxf(Mx, Ms[k * nq + q]);
      float Lx = 0.f;
      float4 Ax = make_float4(0.f, 0.f, 0.f, 0.f);
      if (Mx != -INFINITY)
        for (int k = 0; k < groups; k++) {
          const float mk = Ms[k * nq + q];
          if (mk == -INFINITY) continue;
          const float e = expf(mk - Mx);
          const float4 ak = Acc[k * nq + q];
          Lx += Ls[k * nq + q] * e;
          Ax = make_float4(Ax.x + ak.x * e, Ax.y + ak.y * e, Ax.z + ak.z * e, Ax.w + ak.w * e);
        }
      const float inv = Lx > 0.f ? 1.f / Lx : 0.f;
      float4 z;
      z.x = Ax.x * inv * sigmoidf_(gr.x * sg.x);
      z.y = Ax.y * inv * sigmoidf_(gr.y * sg.y);
      z.z = Ax.z * inv * sigmoidf_(gr.z * sg.z);
      z.w = Ax.w * inv * sigmoidf_(gr.w * sg.w);
      st_tagged4(st.zt + c, z, s + 1);
    }
    tm.sync();
  }
}

// Merge the items of query head h (of kv head kh = h / rep) and gate: thread t takes the 4
// outputs q = t mod HD/4 and the items g, g + G, ... (g = t / (HD/4), G = team size / (HD/4)),
// polls each item's partials (tagged words of this stage) and folds them in item order with
// a running max; the groups meet in shared memory and warp 0
// finishes in group order: y = sum o e^(m - M) / sum l e^(m - M), z = y * sigmoid(g * s_g^2).
// Returns false (team-uniformly) when the block has stopped.
template <int HD>
__device__ __noinline__ bool merge_head(const WarpTeam &tm, const MegaArgs &a, const MegaStage &st, const Dims &d,
                                        int h, int nblk, int s, float *scr, Ctl &ctl) {
  scr = in_shared(scr);
  constexpr int NQ = HD / 4, IB = MEGA_FLAGS / (32 * MW / NQ);  // items a thread holds at most
  const int rep = d.nh / d.nk, kh = h / rep, hh = h % rep;
  const int groups = tm.size() / NQ;
  const int t = tm.tid(), q = t % NQ, g = t / NQ;
  const size_t c = (size_t)h * HD + (size_t)q * 4;
  float4 gr = make_float4(0.f, 0.f, 0.f, 0.f), sg = gr;
  if (g == 0) {  // the gate inputs, while the items finish
    sg = __ldg(reinterpret_cast<const float4 *>(st.sg + c));
    if (!await4(st.qkvg_t + (size_t)(d.nh + 2 * d.nk) * HD + c, st.qtag, gr, ctl, a.spin_limit))
      flag_error(ctl, a.err);
  }
  // each item's partials are tagged words of this stage: the thread's items are polled
  // together, again only those whose words are not all in yet
  const unsigned long long *po = a.tpart + (size_t)h * MEGA_FLAGS * HD + q * 4;
  const unsigned long long *pml = a.tpart + (size_t)d.nh * MEGA_FLAGS * HD + (size_t)h * MEGA_FLAGS * 2;
  const uint32_t tag = s + 1;
  float4 o[IB];
  float2 ml[IB];
  uint32_t pend = 0;
#pragma unroll
  for (int u = 0; u < IB; u++) {
    o[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    ml[u] = make_float2(-INFINITY, 0.f);
    if (g + u * groups < nblk) pend |= 1u << u;
  }
  for (uint32_t polls = 0; pend && !ctl.abort && polls <= a.spin_limit; polls++) {
#pragma unroll
    for (int u = 0; u < IB; u++) {
      if (!((pend >> u) & 1u)) continue;
      const int it = g + u * groups;
      float4 ov;
      float2 mv;
      const bool o_in = ld_tagged4(po + (size_t)it * HD, tag, ov);
      const bool ml_in = ld_tagged2(pml + (size_t)it * 2, tag, mv);
      if (o_in && ml_in) {
        o[u] = ov;
        ml[u] = mv;
        pend &= ~(1u << u);
      }
    }
  }
  if (pend) flag_error(ctl, a.err);
  float M = -INFINITY, L = 0.f;
  float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int u = 0; u < IB; u++) {
    if (ml[u].x == -INFINITY) continue;
    const float nm = fmaxf(M, ml[u].x);
    const float sa = M == -INFINITY ? 0.f : expf(M - nm), sb = expf(ml[u].x - nm);
    L = L * sa + ml[u].y * sb;
    A = make_float4(A.x * sa + o[u].x * sb, A.y * sa + o[u].y * sb, A.z * sa + o[u].z * sb, A.w * sa + o[u].w * sb);
    M = nm;
  }
  float4 *Acc = reinterpret_cast<float4 *>(scr);  // [groups][NQ]
  float *Ms = scr + 4 * groups * NQ, *Ls = Ms + groups * NQ;
  Acc[g * NQ + q] = A;
  Ms[g * NQ + q] = M;
  Ls[g * NQ + q] = L;
  if (!team_ok(tm, ctl)) return false;  // (its first sync publishes the groups' states)
  if (g == 0) {
    float Mx = -INFINITY;
    for (int k = 0; k < groups; k++) Mx = fmaxf(Mx, Ms[k * NQ + q]);
    float Lx = 0.f;
    float4 Ax = make_float4(0.f, 0.f, 0.f, 0.f);
    if (Mx != -INFINITY)
      for (int k = 0; k < groups; k++) {
        const float mk = Ms[k * NQ + q];
        if (mk == -INFINITY) continue;
        const float e = expf(mk - Mx);
        const float4 ak = Acc[k * NQ + q];
        Lx += Ls[k * NQ + q] * e;
        Ax = make_float4(Ax.x + ak.x * e, Ax.y + ak.y * e, Ax.z + ak.z * e, Ax.w + ak.w * e);
      }
    const float inv = Lx > 0.f ? 1.f / Lx : 0.f;
    float4 z;
    z.x = Ax.x * inv * sigmoidf_(gr.x * sg.x);
    z.y = Ax.y * inv * sigmoidf_(gr.y * sg.y);
    z.z = Ax.z * inv * sigmoidf_(gr.z * sg.z);
    z.w = Ax.w * inv * sigmoidf_(gr.w * sg.w);
    st_tagged4(st.zt + c, z, s + 1);
  }
  return true;
}

// Scores of the two halves of a query head's dimensions (split heads), one row per warp.
__shared__ float sc_part[MW][32];

// Warp-wide: query head h of kv head kh against the item's 32 keys (lane = key): scores,
// the item's softmax statistics and its value sum, written as the item's partial. SPLIT = 2:
// two warps share the head, each takes half of its dimensions (half = 0, 1: warps h and
// h + rep); they add their partial scores through shared memory (a team sync: every warp of
// the team is one of the pairs), take the same softmax, and each sums the values of its half.
template <int HD, int SPLIT>
__device__ __forceinline__ void attn_head(const WarpTeam &tm, const MegaStage &st, int nk, const float *Ks,
                                          const float *Vs, const float *q, int tg, long P0, long lo, long p, int kh,
                                          int blk, int rep, int h, int half, unsigned long long *tp, int nh,
                                          uint32_t tag) {
  constexpr int NV = HD / 32 / SPLIT, NC = HD / 4 / SPLIT;  // values a lane sums, float4 chunks scored
  const int lane = threadIdx.x & 31;
  const int d0 = half * (HD / SPLIT);  // this warp's first dimension
  const float scale = 1.f / sqrtf((float)HD);
  const int j = lane;
  const long pe = P0 + j;
  const bool valid = pe >= lo && pe <= p && (tg == (int32_t)pe || pe == p);
  float s0 = 0.f, s1 = 0.f;
  if (valid) {
    const float4 *kr = reinterpret_cast<const float4 *>(Ks + j * HD + d0);
    const float4 *q4 = reinterpret_cast<const float4 *>(q + d0);
#pragma unroll 8
    for (int c = 0; c < NC; c++) {
      const int cc = (c + j) & (NC - 1);  // rotated: the 32 lanes spread over all banks
      const float4 k = kr[cc], qq = q4[cc];
      s0 = fmaf(qq.x, k.x, fmaf(qq.y, k.y, s0));
      s1 = fmaf(qq.z, k.z, fmaf(qq.w, k.w, s1));
    }
  }
  float sp = s0 + s1;
  if constexpr (SPLIT == 2) {
    sc_part[tm.warp()][lane] = sp;
    tm.sync();
    sp = sc_part[h][lane] + sc_part[h + rep][lane];  // the same order in both warps
  }
  const float s = valid ? sp * scale : -INFINITY;
  const float m = warp_max(s);
  const float e = m == -INFINITY ? 0.f : expf(s - m);
  const float l = warp_sum(e);
  float acc[NV], acc_b[NV];  // two chains: even and odd keys
#pragma unroll
  for (int i = 0; i < NV; i++) acc[i] = acc_b[i] = 0.f;
#pragma unroll 4
  for (int jj = 0; jj < AK; jj += 2) {
    const float w0 = __shfl_sync(0xffffffffu, e, jj), w1 = __shfl_sync(0xffffffffu, e, jj + 1);
    const float *v0 = Vs + jj * HD + d0 + lane * NV, *v1 = v0 + HD;
#pragma unroll
    for (int i = 0; i < NV; i++) {
      acc[i] = fmaf(w0, v0[i], acc[i]);
      acc_b[i] = fmaf(w1, v1[i], acc_b[i]);
    }
  }
  if (tp) {  // the per-head merges poll these words
    const size_t qh = (size_t)kh * rep + h;
    unsigned long long *to = tp + (qh * MEGA_FLAGS + blk) * HD + d0 + lane * NV;
    if constexpr (NV == 4)
      st_tagged4(to, make_float4(acc[0] + acc_b[0], acc[1] + acc_b[1], acc[2] + acc_b[2], acc[3] + acc_b[3]), tag);
    else if constexpr (NV == 2)
      st_tagged2(to, acc[0] + acc_b[0], acc[1] + acc_b[1], tag);
    else
      st_tagged(to, acc[0] + acc_b[0], tag);
    if (lane == 0 && half == 0)
      st_tagged2(tp + (size_t)nh * MEGA_FLAGS * HD + (qh * MEGA_FLAGS + blk) * 2, m, l, tag);
    return;
  }
  float *out = part_o(st, rep, HD, kh, blk, h) + d0;
#pragma unroll
  for (int i = 0; i < NV; i++) out[lane * NV + i] = acc[i] + acc_b[i];
  if (lane == 0 && half == 0) *reinterpret_cast<float2 *>(part_ml(st, nk, rep, HD, kh, blk, h)) = make_float2(m, l);
}

// (stages are not inlined: each gets its own register allocation, so the chunk loop does
// not spill)
template <int HD>
__device__ __noinline__ bool attn_stage(const WarpTeam &tm, const MegaArgs &a, const MegaStage &st, int s, float *work,
                                        uint64_t *abar, int &aph, float (*qs)[HD], float (*rope_s)[HD], Ctl &ctl) {
  work = in_shared(work);  // shared-space loads and stores (this function is not inlined)
  qs = in_shared(qs);
  rope_s = in_shared(rope_s);
  const Tracer tr{tm.tid() == 0 ? a.trace : nullptr};
  tr.zero(s);  // trace only: copy wait, compute, arrival, merge cycles
  constexpr int HALF = HD / 2, PP = HALF / 32;  // pairs per lane
  const Dims &d = a.d;
  const int rep = d.nh / d.nk;
  const int cap = st.ring.cap, window = st.ring.window;
  const int seq = ctl.seq;
  const long p = (long)ctl.p;
  const long lo = window == INT_MAX ? 0 : (p + 1 - window > 0 ? p + 1 - window : 0);
  const long blk0 = lo / AK;
  const int nblk = (int)(p / AK - blk0 + 1);
  const int items = d.nk * nblk;
  char *slot = st.ring.base + (size_t)seq * st.ring.seq_stride + st.ring.off;
  int32_t *tags = reinterpret_cast<int32_t *>(slot + st.ring.L.tags);
  float *Kg = reinterpret_cast<float *>(slot + st.ring.L.k), *Vg = reinterpret_cast<float *>(slot + st.ring.L.v);
  const unsigned long long *qkvg = st.qkvg_t;
  float *Ks = work, *Vs = work + AK * HD;
  const int cw = tm.warp(), lane = threadIdx.x & 31;
  const int kw = rep % MW;  // the warp that prepares the new key and value
  const float *rc = rope_s[st.rope_kind], *rsn = rope_s[st.rope_kind] + HALF;
  // With a block for every item and one more for every query head, no block waits for an
  // arrival counter: each item stores its partials as tagged words, and block items + h
  // merges head h.
  const bool per_head = items + d.nh <= (int)gridDim.x && nblk <= MEGA_FLAGS;
  for (int it = blockIdx.x; it < items; it += gridDim.x) {
    const int kh = it / nblk, blk = it % nblk;
    const long P0 = (blk0 + blk) * AK;
    const int rr0 = (int)P0 % cap;  // positions are below 2^31: a 32-bit remainder
    const bool has_p = P0 + AK > p;  // the item that holds the row's own position
    tm.sync();                       // the previous item's tiles and scratch are no longer read
    if (tm.tid() == 0) {
      // Ring rows are not fenced for the async proxy: rows of earlier launches are ordered by
      // the launch boundary, and the one row this launch writes (position p) is replaced in the
      // tile by the item that holds it before anything reads it.
      fence_proxy_async_smem();  // the input row, tiles and merge scratch written before
      const uint32_t bar = smem_addr(abar), bytes = AK * HD * 4;
      mbar_expect_tx(bar, 2 * bytes);
      bulk_g2s(smem_addr(Ks), Kg + ((size_t)kh * cap + rr0) * HD, bytes, bar);
      bulk_g2s(smem_addr(Vs), Vg + ((size_t)kh * cap + rr0) * HD, bytes, bar);
    }
    tr.mark(s, 2);
    aph++;
    const int tg = __ldcg(tags + rr0 + lane);
    // the group's query heads: RoPE on the pairs (j, j + hd/2), justnorm, times s_q^2
    for (int h = cw; h < rep; h += MW) {
      const size_t off = (size_t)(kh * rep + h) * HD;
      float x[PP], y[PP], sx[PP], sy[PP], ss = 0.f;
      int wo[2 * PP];
      float wv[2 * PP];
#pragma unroll
      for (int u = 0; u < PP; u++) {  // the projection and the s_q^2 entries in one round trip
        const int j = lane + 32 * u;
        sx[u] = __ldg(st.sq + off + j);
        sy[u] = __ldg(st.sq + off + j + HALF);
        wo[2 * u] = (int)off + j;
        wo[2 * u + 1] = (int)off + j + HALF;
      }
      if (!await_words(qkvg, wo, st.qtag, wv, ctl, a.spin_limit)) flag_error(ctl, a.err);
#pragma unroll
      for (int u = 0; u < PP; u++) {
        const int j = lane + 32 * u;
        const float a0 = wv[2 * u], b0 = wv[2 * u + 1];
        x[u] = a0 * rc[j] - b0 * rsn[j];
        y[u] = b0 * rc[j] + a0 * rsn[j];
        ss += x[u] * x[u] + y[u] * y[u];
      }
      ss = warp_sum(ss);
      const float inv = 1.f / sqrtf(ss + DORY_EPS);
#pragma unroll
      for (int u = 0; u < PP; u++) {
        const int j = lane + 32 * u;
        qs[h][j] = x[u] * inv * sx[u];
        qs[h][j + HALF] = y[u] * inv * sy[u];
      }
    }
    // the new key (rotated, normalised) and value of kv head kh
    float kx[PP], ky[PP], vx[PP], vy[PP];
    if (has_p && cw == kw) {
      const int ko = (d.nh + kh) * HD, vo = (d.nh + d.nk + kh) * HD;
      float ss = 0.f;
      int wo[4 * PP];
      float wv[4 * PP];
#pragma unroll
      for (int u = 0; u < PP; u++) {
        const int j = lane + 32 * u;
        wo[4 * u] = ko + j;
        wo[4 * u + 1] = ko + j + HALF;
        wo[4 * u + 2] = vo + j;
        wo[4 * u + 3] = vo + j + HALF;
      }
      if (!await_words(qkvg, wo, st.qtag, wv, ctl, a.spin_limit)) flag_error(ctl, a.err);
#pragma unroll
      for (int u = 0; u < PP; u++) {
        const int j = lane + 32 * u;
        const float a0 = wv[4 * u], b0 = wv[4 * u + 1];
        kx[u] = a0 * rc[j] - b0 * rsn[j];
        ky[u] = b0 * rc[j] + a0 * rsn[j];
        ss += kx[u] * kx[u] + ky[u] * ky[u];
        vx[u] = wv[4 * u + 2];
        vy[u] = wv[4 * u + 3];
      }
      ss = warp_sum(ss);
      const float inv = 1.f / sqrtf(ss + DORY_EPS);
#pragma unroll
      for (int u = 0; u < PP; u++) {
        kx[u] *= inv;
        ky[u] *= inv;
      }
    }
    tr.mark(s, 3);
    long long t0 = tr.clk();
    const bool landed = mbar_wait(smem_addr(abar), (aph - 1) & 1, &ctl.abort);
    if (!landed && lane == 0) flag_error(ctl, a.err);
    if (!team_ok(tm, ctl)) return false;
    long long t1 = tr.clk();
    tr.add(s, 8, t1 - t0);
    tr.mark(s, 5);
    if (has_p && cw == kw) {
      // into the tile (it holds the ring's older row there), and into the ring
      const int jp = (int)(p - P0), rr = (int)p % cap;
      float *kg = Kg + ((size_t)kh * cap + rr) * HD, *vg = Vg + ((size_t)kh * cap + rr) * HD;
#pragma unroll
      for (int u = 0; u < PP; u++) {
        const int j = lane + 32 * u;
        Ks[jp * HD + j] = kx[u];
        Ks[jp * HD + j + HALF] = ky[u];
        Vs[jp * HD + j] = vx[u];
        Vs[jp * HD + j + HALF] = vy[u];
        kg[j] = kx[u];
        kg[j + HALF] = ky[u];
        vg[j] = vx[u];
        vg[j + HALF] = vy[u];
      }
      if (kh == 0 && lane == 0) tags[rr] = (int32_t)p;
    }
    tm.sync();
    unsigned long long *tp = per_head ? a.tpart : nullptr;
    if (2 * rep == MW)  // two warps a query head, half of its dimensions each
      attn_head<HD, 2>(tm, st, d.nk, Ks, Vs, qs[cw % rep], tg, P0, lo, p, kh, blk, rep, cw % rep, cw / rep, tp, d.nh,
                       s + 1);
    else
      for (int h = cw; h < rep; h += MW)
        attn_head<HD, 1>(tm, st, d.nk, Ks, Vs, qs[h], tg, P0, lo, p, kh, blk, rep, h, 0, tp, d.nh, s + 1);
    // the last item of this kv head merges the items and gates
    tm.sync();
    t0 = tr.clk();
    tr.add(s, 9, t0 - t1);
    tr.mark(s, 6);
    if (per_head) continue;  // the head merges poll the item's tagged partials
    if (tm.tid() == 0) {
      const int old = atom_add_acq_rel_gpu(a.actr + kh, 1);
      ctl.last = old == nblk - 1;
      if (ctl.last) a.actr[kh] = 0;
    }
    tm.sync();
    t1 = tr.clk();
    tr.add(s, 10, t1 - t0);
    tr.mark(s, 7);
    if (ctl.last) {
      merge_items<HD>(tm, a, st, d, kh, nblk, s, Ks, ctl, tr);
      tr.add(s, 11, tr.clk() - t1);
    }
  }
  if (per_head && (int)blockIdx.x >= items && (int)blockIdx.x < items + d.nh) {
    const long long tm0 = tr.clk();
    if (!merge_head<HD>(tm, a, st, d, (int)blockIdx.x - items, nblk, s, work, ctl)) return false;
    tr.add(s, 11, tr.clk() - tm0);
  }
  tr.flush(s);
  // the merge's last warp may still read the descriptor and the scratch: the next stage
  // copies its descriptor over this one
  tm.sync();
  return true;
}

// The team copies a stage's descriptor into shared memory.
__device__ __forceinline__ void copy_stage(const WarpTeam &tm, const MegaStage *src, MegaStage *dst) {
  constexpr int n = sizeof(MegaStage) / 4;
  const int i = tm.tid();
  if (i < n) reinterpret_cast<int *>(dst)[i] = __ldg(reinterpret_cast<const int *>(src) + i);
}

// ---- the kernel ---------------------------------------------------------------------------

template <int HD>
// 9 warps: at most 3 on an SM sub-partition, so at most 168 registers a thread
__global__ void __launch_bounds__(MTHREADS, 1) mega_decode_kernel(const __grid_constant__ MegaArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *ring = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);  // stays a shared-space pointer
  float *work = reinterpret_cast<float *>(ring + (size_t)NS * SLOT);
  __shared__ __align__(8) uint64_t full[NS], empty[NS], abar;
  __shared__ __align__(16) float qs[8][HD];
  __shared__ __align__(16) float rope_s[2][HD];
  __shared__ __align__(16) MegaStage sst;
  __shared__ float epi[2][EPI_ROWS];
  __shared__ Ctl ctl;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; s++) {
      mbar_init(smem_addr(&full[s]), 1);
      mbar_init(smem_addr(&empty[s]), MW);
      slot_chunk[s] = -1;
    }
    mbar_init(smem_addr(&abar), 1);
    mbar_fence_init();
    ctl.abort = 0;
    ctl.decision = 0;
  }
  __syncthreads();
  if (warp == 0) {
    if (lane == 0) produce(a, ring, full, empty, ctl);
    return;
  }
  const WarpTeam tm{1, MW, 1};
  const int G = gridDim.x, b = blockIdx.x;
  const Dims &d = a.d;
  const Tracer tr{tm.tid() == 0 ? a.trace : nullptr};
  // the row's position, and the RoPE table of it spread over the blocks (f64 angle, f32
  // table; the first attention stage waits for all of it)
  if (tm.tid() == 0) {
    ctl.seq = a.rows.seq[0];
    const long pos = (long)a.rows.seq_pos[ctl.seq] + a.rows.off[0];
    ctl.p = pos;
    const int half = d.hd / 2;
    int n = 0;
    for (int i = b; i < d.hd; i += G, n++) {
      const int kind = i / half, j = i % half;
      const double theta = kind == 0 ? a.theta_s : a.theta_f;
      const float inv = (float)pow((double)(float)theta, -2.0 * (double)j / (double)d.hd);
      double sn, cs;
      sincos((double)pos * (double)inv, &sn, &cs);
      a.rope[kind * d.hd + j] = (float)cs;
      a.rope[kind * d.hd + half + j] = (float)sn;
    }
    if (n) red_release_gpu_add(a.sync + 1, n);
  }
  int c = 0, aph = 0;
  bool ok = true, rope_ready = false;
  for (int s = 0; s < a.nstages && ok; s++) {
    tr.mark(s, 0);
    copy_stage(tm, a.stages + s, &sst);  // (every stage ends with a team sync)
    tm.sync();
    tr.mark(s, 1);
    if (sst.kind == MK_GEMV) {
      ok = gemv_stage(tm, a, sst, s, c, ring, full, empty, work, epi, ctl);
    } else {
      if (!rope_ready) {
        if (!team_wait_counter(tm, a.sync + 1, HD, ctl, a.err, a.spin_limit)) {
          ok = false;
          break;
        }
        for (int i = tm.tid(); i < 2 * HD; i += tm.size()) rope_s[i / HD][i % HD] = __ldcg(a.rope + i);
        tm.sync();
        rope_ready = true;
      }
      ok = attn_stage<HD>(tm, a, sst, s, work, &abar, aph, qs, rope_s, ctl);
    }
    tr.mark(s, 4);
  }
  // an attention copy may still be in flight after a stop
  if (!ok && tm.tid() == 0 && aph > 0) mbar_wait(smem_addr(&abar), (aph - 1) & 1);
  // every block read the position at its start: the last block done advances it
  if (ok && tm.tid() == 0 && atom_add_acq_rel_gpu(a.sync + 2, 1) == G - 1) a.seq_pos[a.adv_seq] += a.adv_cnt;
}

}  // namespace

size_t mega_smem_bytes(int) { return 1024 + (size_t)NS * SLOT + WORK; }

int mega_chunk_rows(int K, bool dual) {  // 0: a row does not fit a slot
  const size_t rb = (size_t)K * 2 * (dual ? 2 : 1);
  const int r = (int)std::min<size_t>(SLOT / rb, RMAX);
  return dual || r < 2 ? r : r & ~1;  // rows go in pairs: an even count per chunk
}

int mega_consumer_warps() { return MW; }

int mega_max_rows_per_block() { return EPI_ROWS; }

size_t mega_work_floats() { return WORK / 4; }

size_t mega_park_floats(bool dual) { return (size_t)(dual ? 2 : 1) * MW * PEND * 32; }

bool mega_supported(int hd, int sms) {
  if (hd != 64 && hd != 128) return false;
  int dev = 0, coop = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop) return false;
  const void *k = hd == 64 ? (const void *)mega_decode_kernel<64> : (const void *)mega_decode_kernel<128>;
  const size_t smem = mega_smem_bytes(hd);
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, MTHREADS, smem) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return per_sm >= 1 && sms >= 1;
}

cudaError_t launch_mega_decode(const MegaArgs &a, int grid, cudaStream_t s) {
  const int hd = a.d.hd;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(MTHREADS);
  cfg.dynamicSmemBytes = mega_smem_bytes(hd);
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;
  at[0].val.cooperative = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (hd == 64) return cudaLaunchKernelEx(&cfg, mega_decode_kernel<64>, a);
  if (hd == 128) return cudaLaunchKernelEx(&cfg, mega_decode_kernel<128>, a);
  return cudaErrorInvalidValue;
}

}  // namespace dory
