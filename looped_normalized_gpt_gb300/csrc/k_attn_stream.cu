// Windowed GQA attention of a batched decode step over f32 rings (dory.rs fn attn_layer):
// one block per (row, kv head) streams the row's window through shared memory.
//
// The window [max(p - W + 1, 0), p] is walked in tiles of 32 positions; a tile's K rows, V
// rows and position tags are contiguous in the ring (capacities are whole multiples of 64)
// and arrive with three bulk copies into one of three stages, completion on the stage's
// mbarrier. Warp w takes positions 4w .. 4w + 3 of every tile for all REP query heads of the
// group, lane l holding dims [l * HD/32, (l + 1) * HD/32) of q (in registers) and of the
// value sums. A position's K row and V row are each read from shared memory once, as one
// vector load per lane: the lane's partial dot products (4 positions x REP heads) are summed
// across the warp by a transpose reduction (recursive halving: at each step a lane keeps half
// of its values and adds its partner's copy of them), after which each lane holds one
// (head, position) score. Each warp keeps its own online softmax per head (running max, sum
// and value sums); the eight warps' states are merged at the end. The last warp to leave a
// stage refills it with the tile three ahead, so no warp waits to issue copies. The output
// y / l is gated, y * sigmoid(g * s_g^2), into z; the row norm follows in its own kernel.
// Waits are bounded; on expiry the block sets error 7, lets its copies land and returns.
// A long window is split over `splits` blocks of consecutive tiles (flash-decoding style)
// when the (row, kv head) blocks alone would leave SMs idle: each block leaves its merged
// softmax state (max, sum, value sums per head) in `part`, and the last block of a (row, kv
// head) to finish (a counter in `ctr`, reset by that block) merges the splits in split order
// and applies the gate.
#include <algorithm>
#include <climits>

#include "async.cuh"
#include "common.cuh"
#include "kernels.h"

namespace dory {

namespace {

constexpr int AS_KEYS = 32;                   // positions per tile
// warps per block: 8 (4 positions a warp per tile) measured 2.8% faster per batch-64 step
// than 4 (8 positions a warp): twice the warps in flight at the same shared memory
constexpr int AS_WARPS_USED = 8;
constexpr int AS_STAGES_F32 = 3;
// q8 tiles are a quarter of the bytes: 8 stages keep about as much in flight per block
constexpr int AS_STAGES_Q8 = 8;
constexpr int ERR_STREAM = 7;

// A stage: K and V rows of a tile (f32, or q8_2f int8 codes), for q8 the K group scales
// [AS_KEYS][HD/32] and V scales [AS_KEYS], then the position tags.
template <int HD, bool Q8 = false>
struct StreamSmem {
  static constexpr int ST = Q8 ? AS_STAGES_Q8 : AS_STAGES_F32;  // stages
  static constexpr int TILE = AS_KEYS * HD * (Q8 ? 1 : 4);   // bytes of K (or V) per tile
  static constexpr int KS = Q8 ? AS_KEYS * (HD / 32) * 4 : 0;
  static constexpr int VS = Q8 ? AS_KEYS * 4 : 0;
  static constexpr int TAGS = 2 * TILE + KS + VS;             // offset of the tags
  static constexpr int STAGE = TAGS + AS_KEYS * 4;
  static constexpr int TOTAL = ST * STAGE + 128;             // + alignment slack
};

template <int DPL>
__device__ __forceinline__ void ld_vec(const float *p, float (&v)[DPL]) {
  if constexpr (DPL == 4) {
    const float4 t = *reinterpret_cast<const float4 *>(p);
    v[0] = t.x, v[1] = t.y, v[2] = t.z, v[3] = t.w;
  } else {
    const float2 t = *reinterpret_cast<const float2 *>(p);
    v[0] = t.x, v[1] = t.y;
  }
}

// Sum NV per-lane values (NV a power of two, at most 32) over the warp. Afterwards every lane
// holds the total of value index lane / (32 / NV); the 32 / NV lanes sharing an index hold
// the same total.
template <int NV>
__device__ __forceinline__ float transpose_sum(float (&v)[NV], int lane) {
#pragma unroll
  for (int cnt = NV, o = 16; cnt > 1; cnt >>= 1, o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < cnt / 2; i++) {
      const float send = up ? v[i] : v[i + cnt / 2];
      const float keep = up ? v[i + cnt / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  float s = v[0];
#pragma unroll
  for (int o = 16 / NV; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

// Q8: q8_2f rings (kv_cache.rs fn attend_group_upto): scores scale * sum_g ks[g] <q * kcol,
// kq>_g, values (sum_j p_j vs_j vq_j) * vcol, the fields applied once the slot has frozen.
template <int HD, int REP, int AS_WARPS, bool Q8 = false>
__global__ void __launch_bounds__(AS_WARPS * 32) attn_stream_kernel(const float *__restrict__ qkvg, int ldq, Dims d,
                                                                    Rows rows, Ring ring, const float *__restrict__ sg,
                                                                    float *__restrict__ z, int *err, int splits,
                                                                    float *__restrict__ part, int *__restrict__ ctr) {
  constexpr int AS_KW = AS_KEYS / AS_WARPS;                   // positions per warp per tile
  constexpr int DPL = HD / 32;                                // dims per lane
  constexpr int NV = REP * AS_KW < 32 ? REP * AS_KW : 32;     // partial scores reduced together
  constexpr int NCH = REP * AS_KW / NV;                       // chunks of heads
  constexpr int HC = NV / AS_KW;                              // heads per chunk
  constexpr int LPI = 32 / NV;                                // lanes holding one reduced score
  constexpr int GRP = AS_KW * LPI;                            // lanes holding one head's scores
  using S = StreamSmem<HD, Q8>;
  constexpr int AS_STAGES = S::ST;
  static_assert(!Q8 || HD == 128, "q8 rows: one 32-bit word of codes per lane");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);  // stays a shared-space pointer
  __shared__ __align__(8) uint64_t full[AS_STAGES];
  __shared__ int done[AS_STAGES], hi, last;
  __shared__ volatile int stop;
  const int rk = blockIdx.x / splits, sp = blockIdx.x % splits;  // (row, kv head), split
  const int r = rk / d.nk, kh = rk % d.nk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seq = rows.seq[r];
  const long p = (long)rows.seq_pos[seq] + rows.off[r];
  const long lo = ring.window == INT_MAX ? 0 : (p + 1 - ring.window > 0 ? p + 1 - ring.window : 0);
  const int nt_all = (int)(p / AS_KEYS - lo / AS_KEYS + 1);
  const int tb = (int)((long)nt_all * sp / splits);               // this split's first tile
  const long t0 = lo / AS_KEYS + tb;
  const int ntiles = (int)((long)nt_all * (sp + 1) / splits) - tb;  // and its tile count (maybe 0)
  const char *slot = ring.base + (size_t)seq * ring.seq_stride + ring.off;
  constexpr int EB = Q8 ? 1 : 4;  // bytes per stored element
  const char *kbase = slot + (Q8 ? ring.L.kq : ring.L.k) + (size_t)kh * ring.cap * HD * EB;
  const char *vbase = slot + (Q8 ? ring.L.vq : ring.L.v) + (size_t)kh * ring.cap * HD * EB;
  const char *ksbase = slot + ring.L.ks + (size_t)kh * ring.cap * (HD / 32) * 4;
  const char *vsbase = slot + ring.L.vs + (size_t)kh * ring.cap * 4;
  const char *tbase = slot + ring.L.tags;
  const bool frozen = Q8 && reinterpret_cast<const int32_t *>(slot + ring.L.meta)[kh * 4 + 1] != 0;

  auto issue = [&](int t) {  // tile t into stage t % AS_STAGES
    const int s = t % AS_STAGES;
    const int rr = (int)(((t0 + t) * AS_KEYS) % ring.cap);
    const uint32_t bar = smem_addr(&full[s]), dst = smem_addr(base + (size_t)s * S::STAGE);
    mbar_expect_tx(bar, S::STAGE);
    bulk_g2s(dst, kbase + (size_t)rr * HD * EB, S::TILE, bar);
    bulk_g2s(dst + S::TILE, vbase + (size_t)rr * HD * EB, S::TILE, bar);
    if constexpr (Q8) {
      bulk_g2s(dst + 2 * S::TILE, ksbase + (size_t)rr * (HD / 32) * 4, S::KS, bar);
      bulk_g2s(dst + 2 * S::TILE + S::KS, vsbase + (size_t)rr * 4, S::VS, bar);
    }
    bulk_g2s(dst + S::TAGS, tbase + (size_t)rr * 4, AS_KEYS * 4, bar);
  };
  if (threadIdx.x == 0) {
    for (int s = 0; s < AS_STAGES; s++) {
      mbar_init(smem_addr(&full[s]), 1);
      done[s] = 0;
    }
    mbar_fence_init();
    stop = 0;
    hi = ntiles < AS_STAGES ? ntiles : AS_STAGES;
    for (int t = 0; t < hi; t++) issue(t);
  }
  // this kv head's query heads, pre-scaled by 1/sqrt(hd) (q8: and by the frozen K field);
  // lane l holds dims l*DPL ..
  const float scale = 1.f / sqrtf((float)HD);
  float kc[DPL], vc[DPL];
#pragma unroll
  for (int i = 0; i < DPL; i++) kc[i] = vc[i] = 1.f;
  if (frozen) {
    ld_vec<DPL>(reinterpret_cast<const float *>(slot + ring.L.kcol) + (size_t)kh * HD + lane * DPL, kc);
    ld_vec<DPL>(reinterpret_cast<const float *>(slot + ring.L.vcol) + (size_t)kh * HD + lane * DPL, vc);
  }
  float q[REP][DPL];
#pragma unroll
  for (int h = 0; h < REP; h++) {
    float t[DPL];
    ld_vec<DPL>(qkvg + (size_t)r * ldq + (size_t)(kh * REP + h) * HD + lane * DPL, t);
#pragma unroll
    for (int i = 0; i < DPL; i++) q[h][i] = t[i] * kc[i] * scale;
  }
  __syncthreads();

  float m[REP], l[REP], acc[REP][DPL];
#pragma unroll
  for (int h = 0; h < REP; h++) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int i = 0; i < DPL; i++) acc[h][i] = 0.f;
  }
  const int own_k = (lane / LPI) % AS_KW, own_hc = lane / GRP;  // the (position, head) a lane scores
  for (int t = 0; t < ntiles; t++) {
    const int s = t % AS_STAGES;
    if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&full[s]), (t / AS_STAGES) & 1, &stop))) {
      if (lane == 0) {
        stop = 1;
        atomicExch(err, ERR_STREAM);
      }
      break;
    }
    const uint8_t *st_base = base + (size_t)s * S::STAGE;
    const float *Kt = reinterpret_cast<const float *>(st_base) + warp * AS_KW * HD;
    const float *Vt = Kt + AS_KEYS * HD;
    const int8_t *Kq = reinterpret_cast<const int8_t *>(st_base) + warp * AS_KW * HD;
    const int8_t *Vq = reinterpret_cast<const int8_t *>(st_base + S::TILE) + warp * AS_KW * HD;
    const float *Ks = reinterpret_cast<const float *>(st_base + 2 * S::TILE) + warp * AS_KW * (HD / 32);
    const float *Vs = reinterpret_cast<const float *>(st_base + 2 * S::TILE + S::KS) + warp * AS_KW;
    const int32_t *tags = reinterpret_cast<const int32_t *>(st_base + S::TAGS);
    const int j = warp * AS_KW + own_k;
    const long pe = (t0 + t) * AS_KEYS + j;
    const bool valid = pe >= lo && pe <= p && tags[j] == (int32_t)pe;
    float e[NCH], fold[REP];
#pragma unroll
    for (int c = 0; c < NCH; c++) {
      float part[NV];
#pragma unroll
      for (int k = 0; k < AS_KW; k++) {
        float kv[DPL];
        float gsc = 1.f;  // q8: the K scale of this lane's 32-channel group
        if constexpr (Q8) {
          const int w4 = *reinterpret_cast<const int *>(Kq + k * HD + lane * 4);
#pragma unroll
          for (int i = 0; i < 4; i++) kv[i] = (float)(int8_t)(w4 >> (8 * i));
          gsc = Ks[k * (HD / 32) + lane / 8];
        } else {
          ld_vec<DPL>(Kt + k * HD + lane * DPL, kv);
        }
#pragma unroll
        for (int hc = 0; hc < HC; hc++) {
          float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
          for (int i = 0; i < DPL; i += 2)
            s2 = ffma2(make_float2(q[c * HC + hc][i], q[c * HC + hc][i + 1]), make_float2(kv[i], kv[i + 1]), s2);
          part[hc * AS_KW + k] = (s2.x + s2.y) * gsc;
        }
      }
      float sc = transpose_sum<NV>(part, lane);
      sc = valid ? sc : -INFINITY;
      float tm = sc;  // this head's maximum over the warp's positions
#pragma unroll
      for (int o = LPI; o < GRP; o <<= 1) tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, o));
      float mown = -INFINITY;
#pragma unroll
      for (int hc = 0; hc < HC; hc++) {
        const int h = c * HC + hc;
        const float mn = fmaxf(m[h], __shfl_sync(0xffffffffu, tm, hc * GRP));
        fold[h] = m[h] == -INFINITY ? 0.f : expf(m[h] - mn);
        m[h] = mn;
        if (hc == own_hc) mown = mn;
      }
      e[c] = sc == -INFINITY ? 0.f : expf(sc - mown);
      float gs = e[c];
#pragma unroll
      for (int o = LPI; o < GRP; o <<= 1) gs += __shfl_xor_sync(0xffffffffu, gs, o);
#pragma unroll
      for (int hc = 0; hc < HC; hc++) {
        const int h = c * HC + hc;
        l[h] = l[h] * fold[h] + __shfl_sync(0xffffffffu, gs, hc * GRP);
      }
    }
#pragma unroll
    for (int h = 0; h < REP; h++)
#pragma unroll
      for (int i = 0; i < DPL; i++) acc[h][i] *= fold[h];
#pragma unroll
    for (int k = 0; k < AS_KW; k++) {
      float vv[DPL];
      if constexpr (Q8) {  // codes times the row's V scale
        const int w4 = *reinterpret_cast<const int *>(Vq + k * HD + lane * 4);
        const float vsk = Vs[k];
#pragma unroll
        for (int i = 0; i < 4; i++) vv[i] = (float)(int8_t)(w4 >> (8 * i)) * vsk;
      } else {
        ld_vec<DPL>(Vt + k * HD + lane * DPL, vv);
      }
#pragma unroll
      for (int c = 0; c < NCH; c++)
#pragma unroll
        for (int hc = 0; hc < HC; hc++) {
          const int h = c * HC + hc;
          const float w = __shfl_sync(0xffffffffu, e[c], (hc * AS_KW + k) * LPI);
#pragma unroll
          for (int i = 0; i < DPL; i += 2) {
            const float2 a = ffma2(make_float2(w, w), make_float2(vv[i], vv[i + 1]), make_float2(acc[h][i], acc[h][i + 1]));
            acc[h][i] = a.x;
            acc[h][i + 1] = a.y;
          }
        }
    }
    // the last warp to leave the stage refills it with the tile three ahead
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      if (atomicAdd(&done[s], 1) == AS_WARPS * (t / AS_STAGES + 1) - 1 && t + AS_STAGES < ntiles && !stop) {
        __threadfence_block();
        atomicMax(&hi, t + AS_STAGES + 1);
        issue(t + AS_STAGES);
      }
    }
  }
  __syncthreads();
  // copies in flight land before the stage memory is reused or the block exits
  if (threadIdx.x == 0)
    for (int t = hi - AS_STAGES < 0 ? 0 : hi - AS_STAGES; t < hi; t++)
      mbar_wait(smem_addr(&full[t % AS_STAGES]), (t / AS_STAGES) & 1);
  __syncthreads();
  if (stop) return;

  // q8: the frozen V field scales every value sum
  if (frozen)
#pragma unroll
    for (int h = 0; h < REP; h++)
#pragma unroll
      for (int i = 0; i < DPL; i++) acc[h][i] *= vc[i];
  // merge the warps' softmax states: m, l per (warp, head), then the value sums
  float *ms = reinterpret_cast<float *>(base), *ls = ms + AS_WARPS * REP, *as = ls + AS_WARPS * REP;
  if (lane == 0)
#pragma unroll
    for (int h = 0; h < REP; h++) {
      ms[warp * REP + h] = m[h];
      ls[warp * REP + h] = l[h];
    }
#pragma unroll
  for (int h = 0; h < REP; h++)
#pragma unroll
    for (int i = 0; i < DPL; i++) as[(warp * REP + h) * HD + lane * DPL + i] = acc[h][i];
  __syncthreads();
  const float *g = qkvg + (size_t)r * ldq + (size_t)(d.nh + 2 * d.nk) * HD;
  // a split's state: [REP] max, [REP] sum, [REP][HD] value sums
  constexpr int PS = REP * (HD + 2);
  float *mine = part + ((size_t)rk * splits + sp) * PS;
  for (int o = threadIdx.x; o < REP * HD; o += blockDim.x) {
    const int h = o / HD, dd = o % HD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < AS_WARPS; w++) M = fmaxf(M, ms[w * REP + h]);
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int w = 0; w < AS_WARPS; w++) {
      const float mw = ms[w * REP + h];
      if (mw == -INFINITY) continue;
      const float f = expf(mw - M);
      num += f * as[(w * REP + h) * HD + dd];
      den += f * ls[w * REP + h];
    }
    const int col = (kh * REP + h) * HD + dd;
    if (splits == 1) {
      z[(size_t)r * d.nh * HD + col] = (den > 0.f ? num / den : 0.f) * sigmoidf_(g[col] * sg[col]);
    } else {
      mine[2 * REP + h * HD + dd] = num;
      if (dd == 0) {
        mine[h] = M;
        mine[REP + h] = den;
      }
    }
  }
  if (splits == 1) return;
  __threadfence();  // this split's state before its count
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(ctr + rk, 1) == splits - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  const float *all = part + (size_t)rk * splits * PS;
  for (int o = threadIdx.x; o < REP * HD; o += blockDim.x) {
    const int h = o / HD, dd = o % HD;
    float M = -INFINITY;
    for (int k = 0; k < splits; k++) M = fmaxf(M, __ldcg(all + (size_t)k * PS + h));
    float num = 0.f, den = 0.f;
    for (int k = 0; k < splits; k++) {  // in split order
      const float mk = __ldcg(all + (size_t)k * PS + h);
      if (mk == -INFINITY) continue;
      const float f = expf(mk - M);
      num += f * __ldcg(all + (size_t)k * PS + 2 * REP + h * HD + dd);
      den += f * __ldcg(all + (size_t)k * PS + REP + h);
    }
    const int col = (kh * REP + h) * HD + dd;
    z[(size_t)r * d.nh * HD + col] = (den > 0.f ? num / den : 0.f) * sigmoidf_(g[col] * sg[col]);
  }
  if (threadIdx.x == 0) ctr[rk] = 0;  // ready for the next launch
}

template <int HD, int REP, int W, bool Q8>
cudaError_t stream_w(const float *qkvg, int ldq, Dims d, Rows rows, Ring ring, const float *sg, float *z, int *err,
                     int splits, float *part, int *ctr, cudaStream_t s) {
  using S = StreamSmem<HD, Q8>;
  // the stages, or the warps' merge scratch after them (m, l and value sums per warp and head)
  constexpr int MERGE = (2 * W * REP + W * REP * HD) * 4 + 128;
  constexpr int SMEM = S::TOTAL > MERGE ? S::TOTAL : MERGE;
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(attn_stream_kernel<HD, REP, W, Q8>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    attr = true;
  }
  attn_stream_kernel<HD, REP, W, Q8><<<rows.n * d.nk * splits, W * 32, SMEM, s>>>(qkvg, ldq, d, rows, ring, sg, z,
                                                                                 err, splits, part, ctr);
  return cudaGetLastError();
}

template <int HD, int REP>
cudaError_t stream_t(const float *qkvg, int ldq, Dims d, Rows rows, Ring ring, const float *sg, float *z, int *err,
                     int splits, float *part, int *ctr, cudaStream_t s) {
  if constexpr (HD == 128)
    if (ring.q8) return stream_w<HD, REP, AS_WARPS_USED, true>(qkvg, ldq, d, rows, ring, sg, z, err, splits, part, ctr, s);
  if (ring.q8) return cudaErrorInvalidValue;
  return stream_w<HD, REP, AS_WARPS_USED, false>(qkvg, ldq, d, rows, ring, sg, z, err, splits, part, ctr, s);
}

}  // namespace

int attn_stream_splits(long window_keys, int rows, int nk, int sms) {
  // only when the (row, kv head) blocks leave SMs idle (at batch 64 x 4 kv heads a split
  // measured slower: 2.22 -> 2.46 ms a step), at least 4 tiles (128 positions) a split. Two
  // blocks fit an SM (the stages take under half its shared memory), so a split's time goes
  // as the rounds of blocks times the tiles a block streams, plus the merge of the splits
  // (half a tile a split): per_loop batch 16 at context 8192 measured 5 splits 2.59 ms a step,
  // 8 2.31, 10 2.42, 12 2.35, 16 2.36 (cost 103, 64, 77, 64, 64 tiles)
  const long units = (long)rows * nk;
  if (units >= sms) return 1;
  const long tiles = (window_keys + AS_KEYS - 1) / AS_KEYS + 1;
  const long most = std::max(1L, std::min(tiles / 4, 64L)), slots = 2L * sms;
  long best = 1;
  double best_cost = 1e30;
  for (long sp = 1; sp <= most; sp++) {
    const long rounds = (units * sp + slots - 1) / slots;
    const double cost = (double)rounds * (double)((tiles + sp - 1) / sp) + 0.5 * (double)sp;
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = sp;
    }
  }
  return (int)best;
}

cudaError_t launch_attention_stream(const float *qkvg, int ldq, Dims d, Rows rows, Ring ring, const float *sg,
                                    float *z, int *err, int splits, float *part, int *ctr, cudaStream_t s) {
  const int rep = d.nh / d.nk;
  if (splits < 1 || (splits > 1 && (!part || !ctr))) return cudaErrorInvalidValue;
#define STREAM(H, R) \
  if (d.hd == H && rep == R) return stream_t<H, R>(qkvg, ldq, d, rows, ring, sg, z, err, splits, part, ctr, s);
  STREAM(64, 1) STREAM(64, 2) STREAM(64, 4) STREAM(64, 8)
  STREAM(128, 1) STREAM(128, 2) STREAM(128, 4) STREAM(128, 8)
#undef STREAM
  return cudaErrorInvalidValue;
}

}  // namespace dory
