// Device helpers shared by the Dory kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define DORY_EPS 1e-6f  // justnorm's epsilon (dory.rs, const EPS)

namespace dory {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Sum over the block; every thread gets the result. `red` holds >= 32 floats.
__device__ __forceinline__ float block_sum(float v, float *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = (lane < nw) ? red[lane] : 0.f;
  t = warp_sum(t);
  return t;
}

__device__ __forceinline__ float block_max(float v, float *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = (lane < nw) ? red[lane] : -INFINITY;
  t = warp_max(t);
  return t;
}

// Eight weights from 16 bytes.
__device__ __forceinline__ void unpack8(const uint4 &u, float *w) {
  const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
  for (int i = 0; i < 4; i++) {
    float2 f = __bfloat1622float2(p[i]);
    w[2 * i] = f.x;
    w[2 * i + 1] = f.y;
  }
}

__device__ __forceinline__ float load_w(const float *p, size_t i) { return p[i]; }
__device__ __forceinline__ float load_w(const __nv_bfloat16 *p, size_t i) { return __bfloat162float(p[i]); }

__device__ __forceinline__ float sigmoidf_(float x) { return 1.f / (1.f + expf(-x)); }

}  // namespace dory

namespace dory {

// Merge the split-KV partials of one (row, kv head) and apply the output gate.
// Split s left, per query head h of the group, o[HD] (unnormalised) then m and l at
// pr[(s * REP + h) * (HD + 2)]. y = sum_s o_s e^(m_s - M) / sum_s l_s e^(m_s - M), times
// vcol (q8_2f, once frozen), then z = y * sigmoid(g * sg). The maxima and sums of all
// splits go to shared memory first (`sm`, 2 * REP * splits floats), every partial output
// is read with eight independent loads in flight per thread.
template <int REP, int HD>
__device__ void merge_splits(const float *pr, int splits, float *sm, const float *g, const float *sg,
                             const float *vcol, float *zrow) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  float *fm = sm, *fl = sm + REP * splits;
  for (int i = threadIdx.x; i < REP * splits; i += blockDim.x) {
    const int sp = i / REP, h = i % REP;
    fm[i] = __ldcg(pr + (size_t)(sp * REP + h) * (HD + 2) + HD);
    fl[i] = __ldcg(pr + (size_t)(sp * REP + h) * (HD + 2) + HD + 1);
  }
  __syncthreads();
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
  __syncthreads();
  for (int i = threadIdx.x; i < REP * HD; i += blockDim.x) {
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
    zrow[i] = y * sigmoidf_(g[i] * sg[i]);
  }
}

}  // namespace dory
