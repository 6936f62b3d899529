// Persistent batch-1 decode: one launch runs the whole token forward (dory.rs fn stack:
// the input block, `loops` passes of the recurrent block with the loop mix, the output
// block and the logits) as a list of stages.
//
// One block per SM, launched cooperatively so that every block is resident. Warp 0 is the
// producer: it walks the stages in order and streams this block's share of every weight
// matrix (a contiguous range of rows) into a ring of shared-memory slots with cp.async.bulk,
// completion on one mbarrier per slot. It never waits for activations, so the weights of
// the next stages are already in flight while the consumers wait at a grid barrier or run
// attention. Warps 1..7 are the consumers, and consumer warp w owns slot w: it takes the
// step's chunks w, w + 7, w + 14, ... (each wait on a slot's barrier is then for the phase
// right after the one that warp saw last, never two ahead). Per stage they
//   * wait until every block has finished the stage before (a counter in global memory);
//   * GEMV: build the input row in shared memory (the embedding, a row norm, or the nGPT
//     residual with the loop mix), then each warp takes whole chunks of rows from the ring,
//     reduces them against the input (bf16 weights, f32 sums), applies the epilogue
//     (SwiGLU, logit scale) and frees the slot; in the q/k/v/g projection the block that
//     completes a head does its RoPE + justnorm (+ s_q^2) and the f32 ring write
//     (dory.rs fn attn_layer);
//   * attention: items of 32 positions of one kv head. The K and V rows of an item are
//     contiguous in the ring and arrive with two bulk copies; warp h scores query head h
//     (lane = key), takes the softmax of the item and its value sum; the last item of a kv
//     head merges the items and applies the output gate (dory.rs fn attn_layer).
// Every wait is bounded. When one runs out the block records error 6, stops at the next
// team-wide check, lets its copies in flight land and returns; the other blocks then stop
// at their next grid barrier.
#include <algorithm>
#include <climits>

#include "async.cuh"
#include "common.cuh"
#include "fused_body.cuh"
#include "kernels.h"
#include "team.cuh"

namespace dory {

namespace {

constexpr int MW = 7;                       // consumer warps
constexpr int MTHREADS = 32 * (MW + 1);     // and the producer warp
constexpr int NS = MW;                      // weight slots, one per consumer warp
constexpr uint32_t SLOT = 26 * 1024;        // bytes per slot
static_assert(NS == MW, "a slot's barrier phases are followed by one warp");
constexpr uint32_t WORK = 32 * 1024;        // input row, or attention tiles and merge scratch
constexpr int AK = MEGA_AK;                 // positions per attention item
constexpr uint32_t SPIN_LIMIT = 1u << 22;   // polls of a global counter
constexpr int ERR_MEGA = 6;                 // dev_err: a wait of the persistent kernel ran out
constexpr int MAX_HEADS_PER_BLOCK = 64;

struct Ctl {
  volatile int abort;  // a wait ran out somewhere in the block
  int decision;        // team-wide copy of `abort`, written by the team's first thread
  int nheads;
  int heads[MAX_HEADS_PER_BLOCK];
  int last;
};

// Optional per-stage timestamps (off when the trace pointer is null).
struct Tracer {
  unsigned long long *p;
  __device__ __forceinline__ void mark(int stage, int event) const {
    if (!p) return;
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    p[((size_t)stage * gridDim.x + blockIdx.x) * MEGA_TRACE_EVENTS + event] = t;
  }
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

// Wait until `*ctr >= target` (blocks past a stage, or RoPE entries written).
__device__ bool team_wait_counter(const WarpTeam &tm, const int *ctr, int target, Ctl &ctl, int *err) {
  if (tm.tid() == 0) {
    uint32_t i = 0;
    while (ld_acquire_gpu(ctr) < target) {
      if (ctl.abort) break;
      if (++i > SPIN_LIMIT) {
        flag_error(ctl, err);
        break;
      }
    }
    ctl.decision = ctl.abort;
  }
  tm.sync();
  return ctl.decision == 0;
}

__device__ __forceinline__ void grid_arrive(const WarpTeam &tm, int *ctr) {
  tm.sync();
  if (tm.tid() == 0) {
    __threadfence();
    red_release_gpu_add(ctr, 1);
  }
}

// ---- producer -----------------------------------------------------------------------------

__device__ void produce(const MegaArgs &a, uint8_t *ring, uint64_t *full, uint64_t *empty, Ctl &ctl) {
  const int G = gridDim.x, b = blockIdx.x;
  const Tracer tr{a.trace};
  int c = 0;  // chunks issued
  bool ok = true;
  for (int s = 0; s < a.nstages && ok; s++) {
    const MegaStage &st = a.stages[s];
    if (st.kind != MK_GEMV) continue;
    const int c_first = c;
    const int N = st.N, K = st.K, R = st.R;
    const long pair = st.pair;
    const int rb = (int)((long)N * b / G), re = (int)((long)N * (b + 1) / G);
    const uint32_t row_bytes = (uint32_t)K * 2;
    for (int r0 = rb; r0 < re; r0 += R) {
      const int nr = min(R, re - r0), sl = c % NS;
      if (c >= NS && !mbar_wait(smem_addr(&empty[sl]), ((c / NS) - 1) & 1, &ctl.abort)) {
        ok = false;
        break;
      }
      const uint32_t bytes = (uint32_t)nr * row_bytes, bar = smem_addr(&full[sl]);
      const uint32_t dst = smem_addr(ring + (size_t)sl * SLOT);
      mbar_expect_tx(bar, pair > 0 ? 2 * bytes : bytes);
      bulk_g2s(dst, st.W + (size_t)r0 * K, bytes, bar);
      if (pair > 0) bulk_g2s(dst + bytes, st.W + (size_t)(r0 + pair) * K, bytes, bar);
      if (c == c_first) tr.mark(s, 5);
      c++;
    }
    tr.mark(s, 6);
  }
  if (!ok) flag_error(ctl, a.err);
  // the block may not exit while a copy into its shared memory is in flight
  for (int k = max(0, c - NS); k < c; k++) mbar_wait(smem_addr(&full[k % NS]), (k / NS) & 1);
}

// ---- GEMV stage ---------------------------------------------------------------------------

// The consumer warps' share of a stage's chunks (chunk c goes to warp c mod MW, in slot
// c mod NS = the same warp's slot). KI > 0:
// K = 256 KI and every lane keeps its 8 KI input values in registers; KI = 0: any K with
// K % 8 == 0, the input read from shared memory.
template <int KI>
__device__ void gemv_chunks(const MegaStage &st, int rb, int re, int c0, const uint8_t *ring, uint64_t *full,
                            uint64_t *empty, const float *xs, Ctl &ctl, int *err) {
  const int lane = threadIdx.x & 31, cw = (threadIdx.x >> 5) - 1;
  const int K = st.K, R = st.R;
  const bool dual = st.pair > 0;
  const int mode = st.ep.mode;
  float xr[KI > 0 ? 8 * KI : 1];
  if (KI > 0) {
#pragma unroll
    for (int i = 0; i < KI; i++) {
      const float4 p = *reinterpret_cast<const float4 *>(xs + i * 256 + lane * 8);
      const float4 q = *reinterpret_cast<const float4 *>(xs + i * 256 + lane * 8 + 4);
      xr[8 * i + 0] = p.x; xr[8 * i + 1] = p.y; xr[8 * i + 2] = p.z; xr[8 * i + 3] = p.w;
      xr[8 * i + 4] = q.x; xr[8 * i + 5] = q.y; xr[8 * i + 6] = q.z; xr[8 * i + 7] = q.w;
    }
  }
  const int nch = re > rb ? (re - rb + R - 1) / R : 0;
  for (int i = 0; i < nch; i++) {
    const int c = c0 + i;  // chunk indices run over the whole step
    if (c % MW != cw) continue;
    const int sl = c % NS;
    // decisions stay warp-uniform: the lanes shuffle below
    if (__shfl_sync(0xffffffffu, ctl.abort, 0)) break;
    if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&full[sl]), (c / NS) & 1, &ctl.abort))) {
      if (lane == 0) flag_error(ctl, err);
      break;
    }
    const int r0 = rb + i * R, nr = min(R, re - r0);
    const __nv_bfloat16 *w = reinterpret_cast<const __nv_bfloat16 *>(ring + (size_t)sl * SLOT);
    for (int rr = 0; rr < nr; rr++) {
      const uint4 *w0 = reinterpret_cast<const uint4 *>(w + (size_t)rr * K);
      const uint4 *w1 = reinterpret_cast<const uint4 *>(w + (size_t)(nr + rr) * K);
      float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
      if (KI > 0) {
#pragma unroll
        for (int k = 0; k < KI; k++) {
          float wv[8];
          unpack8(w0[k * 32 + lane], wv);
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            a0 = fmaf(wv[e], xr[8 * k + e], a0);
            a1 = fmaf(wv[e + 1], xr[8 * k + e + 1], a1);
          }
          if (dual) {
            unpack8(w1[k * 32 + lane], wv);
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              b0 = fmaf(wv[e], xr[8 * k + e], b0);
              b1 = fmaf(wv[e + 1], xr[8 * k + e + 1], b1);
            }
          }
        }
      } else {
        for (int k = lane * 8; k < K; k += 256) {
          float wv[8];
          const float4 p = *reinterpret_cast<const float4 *>(xs + k);
          const float4 q = *reinterpret_cast<const float4 *>(xs + k + 4);
          const float xv[8] = {p.x, p.y, p.z, p.w, q.x, q.y, q.z, q.w};
          unpack8(w0[k / 8], wv);
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            a0 = fmaf(wv[e], xv[e], a0);
            a1 = fmaf(wv[e + 1], xv[e + 1], a1);
          }
          if (dual) {
            unpack8(w1[k / 8], wv);
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              b0 = fmaf(wv[e], xv[e], b0);
              b1 = fmaf(wv[e + 1], xv[e + 1], b1);
            }
          }
        }
      }
      const float g = warp_sum(a0 + a1);
      const float u = dual ? warp_sum(b0 + b1) : 0.f;
      if (lane == 0) {
        const int n = r0 + rr;
        float y;
        if (mode == EPI_SCALE) {
          y = g * __ldg(st.ep.vec + n);
        } else if (mode == EPI_SILU) {
          const float gs = g * __ldg(st.ep.vec + n);
          y = gs * sigmoidf_(gs) * (u * __ldg(st.ep.vec2 + n));
        } else {
          y = g;
        }
        st.Y[n] = y;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&empty[sl]));
  }
}

template <int KC>
__device__ __forceinline__ void input_row(const WarpTeam &tm, const GemvIn &in, int K, float *xs) {
  build_input<1, KC>(tm, in, 1, K, xs, blockIdx.x == 0);
}

// Returns false (team-uniformly) when the block has stopped.
__device__ bool gemv_stage(const WarpTeam &tm, const MegaArgs &a, const MegaStage &st, int s, int &c,
                           const uint8_t *ring, uint64_t *full, uint64_t *empty, float *xs, Ctl &ctl) {
  const Tracer tr{tm.tid() == 0 ? a.trace : nullptr};
  const int G = gridDim.x, b = blockIdx.x;
  const int N = st.N, K = st.K;
  const int rb = (int)((long)N * b / G), re = (int)((long)N * (b + 1) / G);
  const int kc = (K / 4 + tm.size() - 1) / tm.size();  // float4 chunks per thread
  if (kc <= 2) input_row<2>(tm, st.in, K, xs);
  else if (kc <= 4) input_row<4>(tm, st.in, K, xs);
  else if (kc <= 6) input_row<6>(tm, st.in, K, xs);
  else input_row<8>(tm, st.in, K, xs);
  tr.mark(s, 2);
  switch (K) {
    case 256: gemv_chunks<1>(st, rb, re, c, ring, full, empty, xs, ctl, a.err); break;
    case 512: gemv_chunks<2>(st, rb, re, c, ring, full, empty, xs, ctl, a.err); break;
    case 1024: gemv_chunks<4>(st, rb, re, c, ring, full, empty, xs, ctl, a.err); break;
    case 2048: gemv_chunks<8>(st, rb, re, c, ring, full, empty, xs, ctl, a.err); break;
    default: gemv_chunks<0>(st, rb, re, c, ring, full, empty, xs, ctl, a.err); break;
  }
  c += re > rb ? (re - rb + st.R - 1) / st.R : 0;
  if (!team_ok(tm, ctl)) return false;
  tr.mark(s, 3);
  if (!st.he.enabled) return true;
  // heads this block finished rows of: the block that completes a head runs its epilogue
  const Dims &d = a.d;
  const int hd = d.hd;
  if (tm.tid() == 0) {
    __threadfence();
    int n = 0;
    for (int h = rb / hd; re > rb && h <= (re - 1) / hd && n < MAX_HEADS_PER_BLOCK; h++) {
      const int cnt = min(re, (h + 1) * hd) - max(rb, h * hd);
      const int old = atomicAdd(&st.he.counters[h], cnt);
      if (old + cnt == hd) {
        st.he.counters[h] = 0;
        ctl.heads[n++] = h;
      }
    }
    ctl.nheads = n;
  }
  tm.sync();
  const int nh = ctl.nheads;
  if (nh > 0 && !team_wait_counter(tm, a.sync + 1, hd, ctl, a.err)) return false;  // RoPE table ready
  for (int i = 0; i < nh; i++) {
    __threadfence();
    head_epilogue(tm, st.he, ctl.heads[i], 1, st.Y, 0);
    fence_proxy_async_global();  // the ring rows are read by bulk copies after the barrier
    tm.sync();
  }
  return true;
}

// ---- attention stage ----------------------------------------------------------------------

template <int HD, int REP>
__device__ __forceinline__ void merge_items(const WarpTeam &tm, const MegaStage &st, const Dims &d, int kh, int nblk,
                                            float *scratch) {
  const size_t col0 = (size_t)kh * REP * HD;
  merge_splits<REP, HD>(tm, st.part + (size_t)kh * st.maxblk * REP * (HD + 2), nblk, scratch,
                        st.qkvg + (size_t)(d.nh + 2 * d.nk) * HD + col0, st.sg + col0, nullptr, st.z + col0);
}

template <int HD>
__device__ bool attn_stage(const WarpTeam &tm, const MegaArgs &a, const MegaStage &st, float *work, uint64_t *abar,
                           int &aph, float (*qs)[HD], Ctl &ctl) {
  constexpr int NV = HD / 32, NC = HD / 4;
  const Dims &d = a.d;
  const int rep = d.nh / d.nk;
  const int cap = st.ring.cap, window = st.ring.window;
  const int seq = a.rows.seq[0];
  const long p = (long)a.rows.seq_pos[seq] + a.rows.off[0];
  const long lo = window == INT_MAX ? 0 : (p + 1 - window > 0 ? p + 1 - window : 0);
  const long blk0 = lo / AK;
  const int nblk = (int)(p / AK - blk0 + 1);
  const int items = d.nk * nblk;
  const char *slot = st.ring.base + (size_t)seq * st.ring.seq_stride + st.ring.off;
  const int32_t *tags = reinterpret_cast<const int32_t *>(slot + st.ring.L.tags);
  const size_t koff = st.ring.L.k, voff = st.ring.L.v;
  float *Ks = work, *Vs = work + AK * HD;
  const int cw = tm.warp(), lane = threadIdx.x & 31;
  const float scale = 1.f / sqrtf((float)HD);
  for (int it = blockIdx.x; it < items; it += gridDim.x) {
    const int kh = it / nblk, blk = it % nblk;
    const long P0 = (blk0 + blk) * AK;
    const int rr0 = (int)(P0 % cap);
    tm.sync();  // the previous item's tiles and scratch are no longer read
    if (tm.tid() == 0) {
      fence_proxy_async_global();  // ring rows written by this launch's head epilogues
      fence_proxy_async_smem();    // the input row, tiles and merge scratch written before
      const uint32_t bar = smem_addr(abar), bytes = AK * HD * 4;
      mbar_expect_tx(bar, 2 * bytes);
      bulk_g2s(smem_addr(Ks), slot + koff + ((size_t)kh * cap + rr0) * HD * 4, bytes, bar);
      bulk_g2s(smem_addr(Vs), slot + voff + ((size_t)kh * cap + rr0) * HD * 4, bytes, bar);
    }
    aph++;
    for (int i = tm.tid(); i < rep * HD; i += tm.size()) qs[i / HD][i % HD] = __ldcg(st.qkvg + (size_t)kh * rep * HD + i);
    const bool landed = mbar_wait(smem_addr(abar), (aph - 1) & 1, &ctl.abort);
    if (!landed && lane == 0) flag_error(ctl, a.err);
    if (!team_ok(tm, ctl)) return false;
    for (int h = cw; h < rep; h += MW) {
      // warp cw: query heads kh * rep + h; lane j: key P0 + j
      const int j = lane;
      const long pe = P0 + j;
      const bool valid = pe >= lo && pe <= p && __ldcg(tags + rr0 + j) == (int32_t)pe;
      float s0 = 0.f, s1 = 0.f;
      if (valid) {
        const float4 *kr = reinterpret_cast<const float4 *>(Ks + j * HD);
        const float4 *q4 = reinterpret_cast<const float4 *>(qs[h]);
#pragma unroll 8
        for (int c = 0; c < NC; c++) {
          const int cc = (c + j) & (NC - 1);  // rotated: the 32 lanes spread over all banks
          const float4 k = kr[cc], q = q4[cc];
          s0 = fmaf(q.x, k.x, fmaf(q.y, k.y, s0));
          s1 = fmaf(q.z, k.z, fmaf(q.w, k.w, s1));
        }
      }
      const float s = valid ? (s0 + s1) * scale : -INFINITY;
      const float m = warp_max(s);
      const float e = m == -INFINITY ? 0.f : expf(s - m);
      const float l = warp_sum(e);
      float acc[NV];
#pragma unroll
      for (int i = 0; i < NV; i++) acc[i] = 0.f;
      for (int jj = 0; jj < AK; jj++) {
        const float wj = __shfl_sync(0xffffffffu, e, jj);
        if (wj == 0.f) continue;
        const float *v = Vs + jj * HD + lane * NV;
#pragma unroll
        for (int i = 0; i < NV; i++) acc[i] = fmaf(wj, v[i], acc[i]);
      }
      float *out = st.part + (((size_t)kh * st.maxblk + blk) * rep + h) * (HD + 2);
#pragma unroll
      for (int i = 0; i < NV; i++) out[lane * NV + i] = acc[i];
      if (lane == 0) {
        out[HD] = m;
        out[HD + 1] = l;
      }
    }
    // the last item of this kv head merges the items and gates
    __threadfence();
    tm.sync();
    if (tm.tid() == 0) {
      const int old = atomicAdd(a.actr + kh, 1);
      ctl.last = old == nblk - 1;
      if (ctl.last) a.actr[kh] = 0;
    }
    tm.sync();
    if (ctl.last) {
      __threadfence();
      switch (rep) {
        case 1: merge_items<HD, 1>(tm, st, d, kh, nblk, Ks); break;
        case 2: merge_items<HD, 2>(tm, st, d, kh, nblk, Ks); break;
        case 4: merge_items<HD, 4>(tm, st, d, kh, nblk, Ks); break;
        default: merge_items<HD, 8>(tm, st, d, kh, nblk, Ks); break;
      }
    }
  }
  return true;
}

// ---- the kernel ---------------------------------------------------------------------------

template <int HD>
__global__ void __launch_bounds__(MTHREADS, 1) mega_decode_kernel(const __grid_constant__ MegaArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  float *work = reinterpret_cast<float *>(ring + (size_t)NS * SLOT);
  __shared__ __align__(8) uint64_t full[NS], empty[NS], abar;
  __shared__ __align__(16) float qs[8][HD];
  __shared__ Ctl ctl;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; s++) {
      mbar_init(smem_addr(&full[s]), 1);
      mbar_init(smem_addr(&empty[s]), 1);
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
  // RoPE table of the row's position, one entry per block (f64 angle, f32 table; the
  // heads' epilogues wait for all of it)
  if (tm.tid() == 0) {
    const long pos = (long)a.rows.seq_pos[a.rows.seq[0]] + a.rows.off[0];
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
    if (n) {
      __threadfence();
      red_release_gpu_add(a.sync + 1, n);
    }
  }
  int c = 0, aph = 0;
  bool ok = true;
  const Tracer tr{tm.tid() == 0 ? a.trace : nullptr};
  for (int s = 0; s < a.nstages && ok; s++) {
    const MegaStage &st = a.stages[s];
    tr.mark(s, 0);
    if (s > 0 && !team_wait_counter(tm, a.sync, s * G, ctl, a.err)) {
      ok = false;
      break;
    }
    tr.mark(s, 1);
    // every reader of the position has passed: the last stage advances it
    if (s == a.nstages - 1 && b == 0 && tm.tid() == 0) a.seq_pos[a.adv_seq] += a.adv_cnt;
    if (st.kind == MK_GEMV) ok = gemv_stage(tm, a, st, s, c, ring, full, empty, work, ctl);
    else ok = attn_stage<HD>(tm, a, st, work, &abar, aph, qs, ctl);
    tr.mark(s, 4);
    if (ok && s + 1 < a.nstages) grid_arrive(tm, a.sync);
  }
  // an attention copy may still be in flight after a stop
  if (!ok && tm.tid() == 0 && aph > 0) mbar_wait(smem_addr(&abar), (aph - 1) & 1);
}

}  // namespace

size_t mega_smem_bytes(int) { return 1024 + (size_t)NS * SLOT + WORK; }

int mega_chunk_rows(int K, bool dual) {  // 0: a row does not fit a slot
  const size_t rb = (size_t)K * 2 * (dual ? 2 : 1);
  return (int)std::min<size_t>(SLOT / rb, 64);
}

int mega_max_heads_per_block() { return MAX_HEADS_PER_BLOCK; }

size_t mega_work_floats() { return WORK / 4; }

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
