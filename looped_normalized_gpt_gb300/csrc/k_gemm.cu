// Weight-streaming projections Y[t][n] = sum_k W[n][k] X[t][k] (dory.rs fn attn_layer's
// q/k/v/g/o matvecs, fn mlp_layer's gate/up/down, fn head) on CUDA cores.
//
// gemv_kernel: up to 4 rows. One warp per output row reads the row with 16-byte loads
// (8 bf16 or 4+4 f32), the rows' activations sit in shared memory, and the epilogue
// fuses the head's logit scale or the SwiGLU activation (warp reads its gate row and
// its up row).
// gemm_simt_kernel: more rows. A 64x64 output tile per block over 32-wide K slices.
#include "common.cuh"
#include "kernels.h"

namespace dory {

namespace {

constexpr int GEMV_WARPS = 8;

template <typename WT>
struct Vec8;

template <>
struct Vec8<__nv_bfloat16> {
  static __device__ __forceinline__ void load(const __nv_bfloat16 *p, float *w) {
    uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    unpack8(u, w);
  }
};

template <>
struct Vec8<float> {
  static __device__ __forceinline__ void load(const float *p, float *w) {
    float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  }
};

template <typename WT, int TT, bool DUAL>
__global__ void __launch_bounds__(GEMV_WARPS * 32) gemv_kernel(const WT *__restrict__ W, int N, int K,
                                                               const float *__restrict__ X, int ldx, int T,
                                                               float *__restrict__ Y, int ldy, EpiArgs ep) {
  extern __shared__ float xs[];  // [TT][K]
  for (int t = 0; t < T; t++)
    for (int i = threadIdx.x; i < K; i += blockDim.x) xs[t * K + i] = X[(size_t)t * ldx + i];
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * GEMV_WARPS + warp;
  if (n >= N) return;
  const WT *w0 = W + (size_t)n * K;
  const WT *w1 = DUAL ? W + (size_t)(n + ep.pair) * K : nullptr;
  float acc0[TT], acc1[TT];
#pragma unroll
  for (int t = 0; t < TT; t++) acc0[t] = acc1[t] = 0.f;
#pragma unroll 4
  for (int k = lane * 8; k < K; k += 256) {
    float w[8], u[8];
    Vec8<WT>::load(w0 + k, w);
    if (DUAL) Vec8<WT>::load(w1 + k, u);
#pragma unroll
    for (int t = 0; t < TT; t++) {
      if (t < T) {
        const float4 xa = *reinterpret_cast<const float4 *>(&xs[t * K + k]);
        const float4 xb = *reinterpret_cast<const float4 *>(&xs[t * K + k + 4]);
        const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
        for (int i = 0; i < 8; i++) {
          acc0[t] = fmaf(w[i], xv[i], acc0[t]);
          if (DUAL) acc1[t] = fmaf(u[i], xv[i], acc1[t]);
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < TT; t++) {
    if (t >= T) break;
    float a = warp_sum(acc0[t]);
    float b = DUAL ? warp_sum(acc1[t]) : 0.f;
    if (lane == 0) {
      float y;
      if (ep.mode == EPI_SCALE) {
        y = a * ep.vec[n];
      } else if (ep.mode == EPI_SILU) {
        const float g = a * ep.vec[n];
        y = g * sigmoidf_(g) * (b * ep.vec2[n]);
      } else {
        y = a;
      }
      Y[(size_t)t * ldy + n] = y;
    }
  }
}

constexpr int BT = 64, BN = 64, BK = 32;

template <typename WT, bool DUAL>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const WT *__restrict__ W, int N, int K,
                                                        const float *__restrict__ X, int ldx, int T,
                                                        float *__restrict__ Y, int ldy, EpiArgs ep) {
  __shared__ float xs[BK][BT + 4];
  __shared__ float ws[BK][BN + 4];
  __shared__ float us[DUAL ? BK : 1][BN + 4];
  const int tid = threadIdx.x;
  const int t0 = blockIdx.y * BT, n0 = blockIdx.x * BN;
  const int tr = (tid / 16) * 4, nc = (tid % 16) * 4;
  float acc[4][4] = {}, accu[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += BK) {
    for (int i = tid; i < BT * BK; i += 256) {
      const int r = i / BK, c = i % BK;
      const int t = t0 + r, k = k0 + c;
      xs[c][r] = (t < T && k < K) ? X[(size_t)t * ldx + k] : 0.f;
      const int n = n0 + r;
      ws[c][r] = (n < N && k < K) ? load_w(W, (size_t)n * K + k) : 0.f;
      if (DUAL) us[c][r] = (n < N && k < K) ? load_w(W, (size_t)(n + ep.pair) * K + k) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int c = 0; c < BK; c++) {
      float xa[4], wa[4], ua[4];
#pragma unroll
      for (int i = 0; i < 4; i++) {
        xa[i] = xs[c][tr + i];
        wa[i] = ws[c][nc + i];
        if (DUAL) ua[i] = us[c][nc + i];
      }
#pragma unroll
      for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < 4; j++) {
          acc[i][j] = fmaf(xa[i], wa[j], acc[i][j]);
          if (DUAL) accu[i][j] = fmaf(xa[i], ua[j], accu[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const int t = t0 + tr + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const int n = n0 + nc + j;
      if (n >= N) continue;
      float y;
      if (ep.mode == EPI_SCALE) {
        y = acc[i][j] * ep.vec[n];
      } else if (ep.mode == EPI_SILU) {
        const float g = acc[i][j] * ep.vec[n];
        y = g * sigmoidf_(g) * (accu[i][j] * ep.vec2[n]);
      } else {
        y = acc[i][j];
      }
      Y[(size_t)t * ldy + n] = y;
    }
  }
}

template <typename WT, bool DUAL>
cudaError_t gemm_t(const WT *W, int N, int K, const float *X, int ldx, int T, float *Y, int ldy, EpiArgs ep,
                   cudaStream_t s) {
  if (T <= 4 && K % 8 == 0 && (size_t)T * K * 4 <= 96 * 1024) {
    const size_t smem = (size_t)T * K * sizeof(float);
    dim3 grid((N + GEMV_WARPS - 1) / GEMV_WARPS);
    switch (T) {
#define CASE(TTv)                                                                                   \
  case TTv: {                                                                                       \
    auto kern = gemv_kernel<WT, TTv, DUAL>;                                                         \
    if (smem > 48 * 1024) cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); \
    kern<<<grid, GEMV_WARPS * 32, smem, s>>>(W, N, K, X, ldx, T, Y, ldy, ep);                       \
    break;                                                                                          \
  }
      CASE(1) CASE(2) CASE(3) CASE(4)
#undef CASE
    }
  } else {
    dim3 grid((N + BN - 1) / BN, (T + BT - 1) / BT);
    gemm_simt_kernel<WT, DUAL><<<grid, 256, 0, s>>>(W, N, K, X, ldx, T, Y, ldy, ep);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm(const void *W, int wdtype, int N, int K, const float *X, int ldx, int T, float *Y, int ldy,
                        EpiArgs ep, cudaStream_t s) {
  const bool dual = ep.mode == EPI_SILU;
  if (wdtype == W_BF16) {
    const __nv_bfloat16 *w = static_cast<const __nv_bfloat16 *>(W);
    return dual ? gemm_t<__nv_bfloat16, true>(w, N, K, X, ldx, T, Y, ldy, ep, s)
                : gemm_t<__nv_bfloat16, false>(w, N, K, X, ldx, T, Y, ldy, ep, s);
  }
  const float *w = static_cast<const float *>(W);
  return dual ? gemm_t<float, true>(w, N, K, X, ldx, T, Y, ldy, ep, s)
              : gemm_t<float, false>(w, N, K, X, ldx, T, Y, ldy, ep, s);
}

}  // namespace dory
