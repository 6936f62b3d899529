// Windowed causal GQA attention over the KV rings (dory.rs fn attn_layer; q8_2f rows as in
// kv_cache.rs fn attend_group_upto), split over the keys.
//
// attn_split_kernel: one block per (row, kv head, split of the key range). Row r at
// position p reads positions [max(p - W + 1, 0), p]; a ring row counts only when its tag
// holds that position (per_loop holes are skipped). Each warp takes 32 keys at a time,
// lane j owning key j: the lane scores its key against every query head of the group,
// the warp keeps a running max/sum per head, and the value sum runs over the 32 keys
// with the weights broadcast by shuffles (lane owns hd/32 value dims). q8 keys score as
// scale * sum_g ks[g] <q * kcol, kq>_g and values add (p * vs) * vq.
// attn_combine_kernel: merges the splits, applies vcol (q8, once frozen) and the output
// gate y * sigmoid(g * sg) (dory.rs fn gate_body).
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace dory {

namespace {

constexpr int ATT_WARPS = 4;

template <bool Q8, int REP, int NV>
__global__ void __launch_bounds__(ATT_WARPS * 32) attn_split_kernel(const float *__restrict__ qkvg, int ldq, Dims d,
                                                                    Rows rows, Ring ring, int splits, int ks_len,
                                                                    float *__restrict__ part) {
  constexpr int HD = NV * 32;
  __shared__ float qs[REP][HD];
  __shared__ float wm[ATT_WARPS][REP], wl[ATT_WARPS][REP];
  __shared__ float wo[ATT_WARPS][REP][HD];
  const int r = blockIdx.x / d.nk, kh = blockIdx.x % d.nk, sp = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seq = rows.seq[r];
  const long p = (long)rows.seq_pos[seq] + rows.off[r];
  const long lo = ring.window == INT_MAX ? 0 : (p + 1 - ring.window > 0 ? p + 1 - ring.window : 0);
  const long k0 = lo + (long)sp * ks_len;
  const long k1 = (k0 + ks_len - 1 < p) ? k0 + ks_len - 1 : p;  // inclusive
  const char *slot = ring.base + (size_t)seq * ring.seq_stride + ring.off;
  const int32_t *tags = reinterpret_cast<const int32_t *>(slot + ring.L.tags);
  const float *q = qkvg + (size_t)r * ldq + (size_t)kh * REP * HD;

  const float *kcol = Q8 ? reinterpret_cast<const float *>(slot + ring.L.kcol) + (size_t)kh * HD : nullptr;
  const int frozen = Q8 ? reinterpret_cast<const int32_t *>(slot + ring.L.meta)[kh * 4 + 1] : 0;
  for (int i = threadIdx.x; i < REP * HD; i += blockDim.x) {
    float v = q[i];
    if (Q8 && frozen) v *= kcol[i % HD];
    qs[i / HD][i % HD] = v;
  }
  __syncthreads();

  const float scale = 1.f / sqrtf((float)HD);
  float m[REP], l[REP], acc[REP][NV];
#pragma unroll
  for (int h = 0; h < REP; h++) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int i = 0; i < NV; i++) acc[h][i] = 0.f;
  }
  for (long kb = k0 + warp * 32; kb <= k1; kb += ATT_WARPS * 32) {
    const long pe = kb + lane;
    const int rr = (int)(((pe % ring.cap) + ring.cap) % ring.cap);
    const bool valid = pe <= k1 && tags[rr] == (int32_t)pe;
    float s[REP];
#pragma unroll
    for (int h = 0; h < REP; h++) s[h] = 0.f;
    if (valid) {
      if (!Q8) {
        const float4 *kr = reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(slot + ring.L.k) +
                                                            ((size_t)kh * ring.cap + rr) * HD);
#pragma unroll 4
        for (int c = 0; c < HD / 4; c++) {
          const float4 k4 = __ldg(kr + c);
#pragma unroll
          for (int h = 0; h < REP; h++) {
            const float4 q4 = *reinterpret_cast<const float4 *>(&qs[h][c * 4]);
            s[h] = fmaf(q4.x, k4.x, fmaf(q4.y, k4.y, fmaf(q4.z, k4.z, fmaf(q4.w, k4.w, s[h]))));
          }
        }
      } else {
        const int8_t *kq = reinterpret_cast<const int8_t *>(slot + ring.L.kq) + ((size_t)kh * ring.cap + rr) * HD;
        const float *ksc = reinterpret_cast<const float *>(slot + ring.L.ks) + ((size_t)kh * ring.cap + rr) * (HD / 32);
#pragma unroll
        for (int g = 0; g < HD / 32; g++) {
          float dg[REP];
#pragma unroll
          for (int h = 0; h < REP; h++) dg[h] = 0.f;
#pragma unroll
          for (int c = 0; c < 2; c++) {
            const int4 w = __ldg(reinterpret_cast<const int4 *>(kq + g * 32 + c * 16));
            const int8_t *b = reinterpret_cast<const int8_t *>(&w);
#pragma unroll
            for (int e = 0; e < 16; e++) {
              const float kv = (float)b[e];
#pragma unroll
              for (int h = 0; h < REP; h++) dg[h] = fmaf(qs[h][g * 32 + c * 16 + e], kv, dg[h]);
            }
          }
          const float sg = __ldg(ksc + g);
#pragma unroll
          for (int h = 0; h < REP; h++) s[h] = fmaf(sg, dg[h], s[h]);
        }
      }
    }
    // online softmax over this block of 32 keys, per head
    float pw[REP];
    bool any = false;
#pragma unroll
    for (int h = 0; h < REP; h++) {
      const float sv = valid ? s[h] * scale : -INFINITY;
      const float mb = warp_max(sv);
      if (mb == -INFINITY) {
        pw[h] = 0.f;
        continue;
      }
      any = true;
      const float mn = fmaxf(m[h], mb);
      const float corr = expf(m[h] - mn);  // 0 when m was -inf
      pw[h] = valid ? expf(sv - mn) : 0.f;
      l[h] = l[h] * corr + warp_sum(pw[h]);
#pragma unroll
      for (int i = 0; i < NV; i++) acc[h][i] *= corr;
      m[h] = mn;
    }
    if (!any) continue;
    const unsigned vmask = __ballot_sync(0xffffffffu, valid);
    for (int j = 0; j < 32; j++) {
      if (!((vmask >> j) & 1u)) continue;
      const long pj = kb + j;
      const int rj = (int)(pj % ring.cap);
      float pj_h[REP];
#pragma unroll
      for (int h = 0; h < REP; h++) pj_h[h] = __shfl_sync(0xffffffffu, pw[h], j);
      if (!Q8) {
        const float *vr = reinterpret_cast<const float *>(slot + ring.L.v) + ((size_t)kh * ring.cap + rj) * HD;
#pragma unroll
        for (int i = 0; i < NV; i++) {
          const float vv = __ldg(vr + lane + 32 * i);
#pragma unroll
          for (int h = 0; h < REP; h++) acc[h][i] = fmaf(pj_h[h], vv, acc[h][i]);
        }
      } else {
        const int8_t *vq = reinterpret_cast<const int8_t *>(slot + ring.L.vq) + ((size_t)kh * ring.cap + rj) * HD;
        const float vs = __ldg(reinterpret_cast<const float *>(slot + ring.L.vs) + (size_t)kh * ring.cap + rj);
#pragma unroll
        for (int i = 0; i < NV; i++) {
          const float vv = (float)vq[lane + 32 * i];
#pragma unroll
          for (int h = 0; h < REP; h++) acc[h][i] = fmaf(pj_h[h] * vs, vv, acc[h][i]);
        }
      }
    }
  }
  // merge the warps of the block
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < REP; h++) {
      wm[warp][h] = m[h];
      wl[warp][h] = l[h];
    }
  }
#pragma unroll
  for (int h = 0; h < REP; h++)
#pragma unroll
    for (int i = 0; i < NV; i++) wo[warp][h][lane + 32 * i] = acc[h][i];
  __syncthreads();
  float *out = part + ((size_t)(r * d.nk + kh) * splits + sp) * REP * (HD + 2);
  for (int i = threadIdx.x; i < REP * HD; i += blockDim.x) {
    const int h = i / HD, c = i % HD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < ATT_WARPS; w++) M = fmaxf(M, wm[w][h]);
    float o = 0.f, L = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < ATT_WARPS; w++) {
        const float f = expf(wm[w][h] - M);
        o += wo[w][h][c] * f;
        L += wl[w][h] * f;
      }
    }
    out[h * (HD + 2) + c] = o;
    if (c == 0) {
      out[h * (HD + 2) + HD] = M;
      out[h * (HD + 2) + HD + 1] = L;
    }
  }
}

template <bool Q8, int REP, int NV>
__global__ void attn_combine_kernel(const float *__restrict__ part, int splits, const float *__restrict__ qkvg,
                                    int ldq, Dims d, Rows rows, Ring ring, const float *__restrict__ sg,
                                    float *__restrict__ z) {
  constexpr int HD = NV * 32;
  const int r = blockIdx.x, kh = blockIdx.y, c = threadIdx.x;  // blockDim = HD
  const float *pr = part + (size_t)(r * d.nk + kh) * splits * REP * (HD + 2);
  float vcol = 1.f;
  if (Q8) {
    const int seq = rows.seq[r];
    const char *slot = ring.base + (size_t)seq * ring.seq_stride + ring.off;
    if (reinterpret_cast<const int32_t *>(slot + ring.L.meta)[kh * 4 + 1])
      vcol = reinterpret_cast<const float *>(slot + ring.L.vcol)[kh * HD + c];
  }
  const float *g = qkvg + (size_t)r * ldq + (size_t)(d.nh + 2 * d.nk) * HD;
  for (int h = 0; h < REP; h++) {
    float M = -INFINITY;
    for (int s = 0; s < splits; s++) M = fmaxf(M, pr[(s * REP + h) * (HD + 2) + HD]);
    float o = 0.f, L = 0.f;
    for (int s = 0; s < splits; s++) {
      const float *ps = pr + (s * REP + h) * (HD + 2);
      const float ms = ps[HD];
      if (ms == -INFINITY) continue;
      const float f = expf(ms - M);
      o += ps[c] * f;
      L += ps[HD + 1] * f;
    }
    const int col = (kh * REP + h) * HD + c;
    const float y = (L > 0.f ? o / L : 0.f) * vcol;
    z[(size_t)r * d.nh * HD + col] = y * sigmoidf_(g[col] * sg[col]);
  }
}

template <bool Q8, int REP, int NV>
cudaError_t attn_t(const float *qkvg, int ldq, Dims d, Rows rows, Ring ring, int splits, int kps, float *part,
                   const float *sg, float *z, cudaStream_t s) {
  dim3 g1(rows.n * d.nk, splits);
  attn_split_kernel<Q8, REP, NV><<<g1, ATT_WARPS * 32, 0, s>>>(qkvg, ldq, d, rows, ring, splits, kps, part);
  dim3 g2(rows.n, d.nk);
  attn_combine_kernel<Q8, REP, NV><<<g2, NV * 32, 0, s>>>(part, splits, qkvg, ldq, d, rows, ring, sg, z);
  return cudaGetLastError();
}

template <bool Q8>
cudaError_t attn_q8(const float *qkvg, int ldq, Dims d, Rows rows, Ring ring, int splits, int kps, float *part,
                    const float *sg, float *z, cudaStream_t s) {
  const int rep = d.nh / d.nk, nv = d.hd / 32;
#define DISPATCH(R, N) \
  if (rep == R && nv == N) return attn_t<Q8, R, N>(qkvg, ldq, d, rows, ring, splits, kps, part, sg, z, s);
  DISPATCH(1, 1) DISPATCH(1, 2) DISPATCH(1, 4)
  DISPATCH(2, 1) DISPATCH(2, 2) DISPATCH(2, 4)
  DISPATCH(4, 1) DISPATCH(4, 2) DISPATCH(4, 4)
  DISPATCH(8, 1) DISPATCH(8, 2) DISPATCH(8, 4)
#undef DISPATCH
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_attention(const float *qkvg, int ldq, Dims d, Rows rows, Ring ring, int splits, int kps, float *part,
                             const float *sg, float *z, cudaStream_t s) {
  return ring.q8 ? attn_q8<true>(qkvg, ldq, d, rows, ring, splits, kps, part, sg, z, s)
                 : attn_q8<false>(qkvg, ldq, d, rows, ring, splits, kps, part, sg, z, s);
}

}  // namespace dory
