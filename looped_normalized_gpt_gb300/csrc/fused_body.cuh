// Device bodies shared by the standalone decode kernels and the persistent decode kernel:
// the GEMV input prologue, the per-head epilogue of the q/k/v/g projection, and the merge
// of split attention partials. Each runs on a team of threads (a block, or some warps of
// a block) given as a template parameter.
#pragma once

#include "kernels.h"
#include "team.cuh"

namespace dory {

// Prologue: the team's input rows xs[t][K] from the previous kernels' outputs. Each
// thread owns the float4 chunks tid + j * (team size) of a row (KC of them at most) and loads
// all the vectors it needs for them at once, so a row costs one memory round trip; the
// reductions pair up their sums. `lead`: this team stores the new hidden rows (and the
// mix's input/state rows). HALVES: each row goes to shared memory as two halves, float4
// chunk c at (c & 1) * K / 8 + c / 2, so that a lane reading the 8 inputs of a 16-byte
// weight column reads float4 u of each half: consecutive lanes, consecutive addresses
// (the plain layout puts a lane's two float4 loads 32 bytes apart, two-way bank conflicts).
template <int TT, int KC, typename Team, bool HALVES = false>
__device__ void build_input(const Team &tm, const GemvIn &in, int T, int K, float *xs, bool lead) {
  __shared__ float red[2][TEAM_MAX_WARPS];
  const int tid = tm.tid(), nt = tm.size();
  const int nch = K / 4;
  for (int t = 0; t < T; t++) {
    // rows written earlier in the same launch (persistent kernel) are read from L2
    const float4 *src = reinterpret_cast<const float4 *>(in.src + (size_t)t * in.ld);
    float4 x[KC], o[KC], al[KC], inp[KC];
#pragma unroll
    for (int j = 0; j < KC; j++) {
      const int c = tid + j * nt;
      x[j] = o[j] = al[j] = inp[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c < nch) {
        if (in.mode == IN_EMBED) {
          const int id = in.ids[t];
          if (id >= 0 && id < in.vocab) {
            const uint2 u = __ldg(reinterpret_cast<const uint2 *>(in.embed + (size_t)id * K) + c);
            const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
            const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
            x[j] = make_float4(a.x, a.y, b.x, b.y);
          }
        } else {
          x[j] = __ldcg(src + c);
        }
        if (in.mode == IN_RESID && in.alpha) {
          o[j] = __ldcg(reinterpret_cast<const float4 *>(in.out + (size_t)t * K) + c);
          al[j] = __ldg(reinterpret_cast<const float4 *>(in.alpha) + c);
        }
        if (in.mode == IN_RESID && (in.mix == MIX_LOOP || in.mix == MIX_RESUME))
          inp[j] = __ldcg(reinterpret_cast<const float4 *>(in.input + (size_t)t * K) + c);
      }
    }
    auto sq4 = [](const float4 &v) { return v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w; };
    auto scale4 = [](float4 &v, float f) {
      v.x *= f;
      v.y *= f;
      v.z *= f;
      v.w *= f;
    };
    if (in.mode == IN_NORM) {
      float ss = 0.f, dummy = 0.f;
#pragma unroll
      for (int j = 0; j < KC; j++) ss += sq4(x[j]);
      team_sum2(tm, ss, dummy, red);
      const float inv = 1.f / sqrtf(ss + DORY_EPS);
#pragma unroll
      for (int j = 0; j < KC; j++) scale4(x[j], inv);
    } else if (in.mode == IN_RESID) {
      if (in.alpha) {
        float sx = 0.f, so = 0.f;
#pragma unroll
        for (int j = 0; j < KC; j++) {
          sx += sq4(x[j]);
          so += sq4(o[j]);
        }
        team_sum2(tm, sx, so, red);
        const float ix = 1.f / sqrtf(sx + DORY_EPS), io = 1.f / sqrtf(so + DORY_EPS);
        float sr = 0.f, dummy = 0.f;
#pragma unroll
        for (int j = 0; j < KC; j++) {
          float4 xh = x[j], oh = o[j];
          scale4(xh, ix);
          scale4(oh, io);
          x[j] = make_float4(xh.x + al[j].x * (oh.x - xh.x), xh.y + al[j].y * (oh.y - xh.y),
                             xh.z + al[j].z * (oh.z - xh.z), xh.w + al[j].w * (oh.w - xh.w));
          sr += sq4(x[j]);
        }
        team_sum2(tm, sr, dummy, red);
        const float inv = 1.f / sqrtf(sr + DORY_EPS);
#pragma unroll
        for (int j = 0; j < KC; j++) scale4(x[j], inv);
      }
      if (in.mix == MIX_LOOP || in.mix == MIX_END) {  // state = h^
        float ss = 0.f, dummy = 0.f;
#pragma unroll
        for (int j = 0; j < KC; j++) ss += sq4(x[j]);
        team_sum2(tm, ss, dummy, red);
        const float inv = 1.f / sqrtf(ss + DORY_EPS);
#pragma unroll
        for (int j = 0; j < KC; j++) {
          scale4(x[j], inv);
          const int c = tid + j * nt;
          if (lead && c < nch) reinterpret_cast<float4 *>(in.state + (size_t)t * K)[c] = x[j];
        }
      }
      if (in.mix == MIX_BEGIN || in.mix == MIX_LOOP || in.mix == MIX_RESUME) {  // h = (state + input)^
        // (MIX_RESUME: src is the saved state row, taken as it is)
        float ss = 0.f, dummy = 0.f;
#pragma unroll
        for (int j = 0; j < KC; j++) {
          const int c = tid + j * nt;
          if (in.mix == MIX_BEGIN) {
            inp[j] = x[j];
            if (lead && c < nch) {
              reinterpret_cast<float4 *>(in.input + (size_t)t * K)[c] = x[j];
              reinterpret_cast<float4 *>(in.state + (size_t)t * K)[c] = x[j];
            }
          }
          x[j] = make_float4(x[j].x + inp[j].x, x[j].y + inp[j].y, x[j].z + inp[j].z, x[j].w + inp[j].w);
          ss += sq4(x[j]);
        }
        team_sum2(tm, ss, dummy, red);
        const float inv = 1.f / sqrtf(ss + DORY_EPS);
#pragma unroll
        for (int j = 0; j < KC; j++) scale4(x[j], inv);
      }
    }
#pragma unroll
    for (int j = 0; j < KC; j++) {
      const int c = tid + j * nt;
      if (c < nch) {
        reinterpret_cast<float4 *>(xs + (size_t)t * K)[HALVES ? (c & 1) * (nch / 2) + (c >> 1) : c] = x[j];
        if ((in.mode == IN_RESID || in.mode == IN_EMBED) && lead && in.h_dst)
          reinterpret_cast<float4 *>(in.h_dst + (size_t)t * K)[c] = x[j];
      }
    }
  }
  tm.sync();
}

// The last team of a q/k/v/g head: RoPE + justnorm (+ s_q^2) and the ring write
// (dory.rs fn attn_layer). The team has at least T * hd/2 threads.
template <typename Team>
__device__ void head_epilogue(const Team &tm, const HeadEpi &he, int head, int T, float *Y, int ldy) {
  __shared__ float red2[TEAM_MAX_WARPS];
  const Dims &d = he.d;
  const int hd = d.hd, half = hd / 2;
  const int tid = tm.tid();
  const int t = tid / half, j = tid % half;  // blockDim 256 >= T * half for hd <= 128
  const bool act = t < T;
  const bool is_q = head < d.nh, is_k = head >= d.nh && head < d.nh + d.nk;
  const bool is_v = head >= d.nh + d.nk && head < d.nh + 2 * d.nk;
  if (!(is_q || is_k || is_v)) return;  // gate heads need nothing (block-uniform)
  float a = 0.f, b = 0.f;
  float *row = Y + (size_t)(act ? t : 0) * ldy + head * hd;
  if (act) {
    a = __ldcg(row + j);
    b = __ldcg(row + j + half);
  }
  if (is_q || is_k) {
    if (act) {
      const float *cs = he.rope + ((size_t)t * 2 + he.kind) * hd;
      const float c = __ldcg(cs + j), sn = __ldcg(cs + half + j);
      const float x = a, y = b;
      a = x * c - y * sn;
      b = y * c + x * sn;
    }
    // per-row sums over the row's half threads (two warps when hd = 128)
    float v = act ? a * a + b * b : 0.f;
    v = warp_sum(v);
    const int lane = tid & 31, warp = tid >> 5;
    tm.sync();
    if (lane == 0) red2[warp] = v;
    tm.sync();
    const int wpr = (half + 31) / 32;  // warps per row
    if (act) {
      float s = 0.f;
      for (int w = 0; w < wpr; w++) s += red2[t * wpr + w];
      const float inv = 1.f / sqrtf(s + DORY_EPS);
      a *= inv;
      b *= inv;
    }
  }
  if (!act) return;
  if (is_q) {
    row[j] = a * he.sq[head * hd + j];
    row[j + half] = b * he.sq[head * hd + j + half];
    return;
  }
  const int kh = is_k ? head - d.nh : head - d.nh - d.nk;
  if (is_k) {  // rotated, normalised key back into the projection rows for reference
    row[j] = a;
    row[j + half] = b;
  }
  const Ring &ring = he.ring;
  if (ring.q8) {
    float *dst = (is_k ? he.kst : he.vst) + ((size_t)t * d.nk + kh) * hd;
    dst[j] = a;
    dst[j + half] = b;
    return;
  }
  const int seq = he.rows.seq[t];
  const long pos = (long)he.rows.seq_pos[seq] + he.rows.off[t];
  const int rr = (int)(pos % ring.cap);
  char *slot = ring.base + (size_t)seq * ring.seq_stride + ring.off;
  float *dst = reinterpret_cast<float *>(slot + (is_k ? ring.L.k : ring.L.v)) + ((size_t)kh * ring.cap + rr) * hd;
  dst[j] = a;
  dst[j + half] = b;
  if (is_k && kh == 0 && j == 0) reinterpret_cast<int32_t *>(slot + ring.L.tags)[rr] = (int32_t)pos;
}

// Merge the split-KV partials of one (row, kv head) and apply the output gate.
// Split s left, per query head h of the group, o[HD] (unnormalised) then m and l at
// pr[(s * REP + h) * (HD + 2)]. y = sum_s o_s e^(m_s - M) / sum_s l_s e^(m_s - M), times
// vcol (q8_2f, once frozen), then z = y * sigmoid(g * sg). The maxima and sums of all
// splits go to shared memory first (`sm`, 2 * REP * splits floats), every partial output
// is read with eight independent loads in flight per thread.
template <int REP, int HD, typename Team>
__device__ void merge_splits(const Team &tm, const float *pr, int splits, float *sm, const float *g, const float *sg,
                             const float *vcol, float *zrow) {
  const int lane = threadIdx.x & 31, warp = tm.warp(), nw = tm.nwarps();
  float *fm = sm, *fl = sm + REP * splits;
  for (int i = tm.tid(); i < REP * splits; i += tm.size()) {
    const int sp = i / REP, h = i % REP;
    fm[i] = __ldcg(pr + (size_t)(sp * REP + h) * (HD + 2) + HD);
    fl[i] = __ldcg(pr + (size_t)(sp * REP + h) * (HD + 2) + HD + 1);
  }
  tm.sync();
  for (int h = warp; h < REP; h += nw) {
    float M = -INFINITY;
    for (int sp = lane; sp < splits; sp += 32) M = fmaxf(M, fm[sp * REP + h]);
    M = warp_max(M);
    float L = 0.f;
    for (int sp = lane; sp < splits; sp += 32) {
      const float m = fm[sp * REP + h];
      if (m != -INFINITY) L += fl[sp * REP + h] * expf(m - M);
    }
    L = warp_sum(L);
    __syncwarp();
    for (int sp = lane; sp < splits; sp += 32) {
      const float m = fm[sp * REP + h];
      fm[sp * REP + h] = (m == -INFINITY || !(L > 0.f)) ? 0.f : expf(m - M) / L;
    }
  }
  tm.sync();
  for (int i = tm.tid(); i < REP * HD; i += tm.size()) {
    const int h = i / HD, c = i % HD;
    const float *base = pr + (size_t)h * (HD + 2) + c;
    float o = 0.f;
    int sp = 0;
    for (; sp + 8 <= splits; sp += 8) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; u++) v[u] = __ldcg(base + (size_t)(sp + u) * REP * (HD + 2));
#pragma unroll
      for (int u = 0; u < 8; u++) o = fmaf(v[u], fm[(sp + u) * REP + h], o);
    }
    for (; sp < splits; sp++) o = fmaf(__ldcg(base + (size_t)sp * REP * (HD + 2)), fm[sp * REP + h], o);
    const float y = o * (vcol ? vcol[c] : 1.f);
    zrow[i] = y * sigmoidf_(__ldcg(g + i) * sg[i]);
  }
}

}  // namespace dory
