// Fused decode kernels for steps of up to 4 rows (batch-1..4 decode, tiny chunks).
//
// gemv_fused_kernel streams one weight row per warp with 16-byte loads, like gemv_kernel,
// but
//   * issues its first weight loads before griddepcontrol.wait, so under programmatic
//     dependent launch they overlap the previous kernel's tail;
//   * builds its input rows itself (prologue): the nGPT residual of the previous
//     sub-layer with the loop mix after it (dory.rs fn slerp, fn stack), or the row norm
//     of an attention or MLP output (fn attn_layer's justnorm over nh*hd, fn mlp_layer's
//     over ffn); block 0 stores the new hidden rows for the layers after;
//   * for the q/k/v/g projection, the last block to finish a head (an arrival counter per
//     head) does that head's epilogue: RoPE + justnorm (+ s_q^2) for q and k, and the f32
//     ring write (or staging for q8) of k and v (dory.rs fn attn_layer).
// attn_fused_kernel is the split-KV attention of k_attn.cu whose last split block per
// (row, kv head) merges the splits and applies the gate (no second launch).
#include <algorithm>
#include <climits>
#include <cstdlib>

#include "common.cuh"
#include "fused_body.cuh"
#include "kernels.h"

namespace dory {

namespace {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

constexpr int FW = 8;     // warps per block
// 8-element chunks of a row loaded before the dependency wait
template <typename WT>
struct Pre {
  static constexpr int n = sizeof(WT) == 2 ? 8 : 2;
};
constexpr int MAXT = 4;   // rows

template <typename WT>
struct Chunk;
template <>
struct Chunk<__nv_bfloat16> {
  uint4 u;
  __device__ __forceinline__ void load(const __nv_bfloat16 *p) { u = __ldg(reinterpret_cast<const uint4 *>(p)); }
  __device__ __forceinline__ void get(float *w) const { unpack8(u, w); }
};
template <>
struct Chunk<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float *p) {
    a = __ldg(reinterpret_cast<const float4 *>(p));
    b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
  }
  __device__ __forceinline__ void get(float *w) const {
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  }
};

template <typename WT, int TT, bool DUAL, int KC>
__global__ void __launch_bounds__(FW * 32, 2) gemv_fused_kernel(const WT *__restrict__ W, int N, int K, int T,
                                                                GemvIn in, float *__restrict__ Y, int ldy,
                                                                EpiArgs ep, HeadEpi he) {
  extern __shared__ float xs[];  // [T][K]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * FW + warp;
  const bool has_row = n < N;
  const WT *w0 = W + (size_t)(has_row ? n : 0) * K;
  const WT *w1 = DUAL ? W + (size_t)((has_row ? n : 0) + ep.pair) * K : nullptr;
  // weights do not depend on earlier kernels: start them before the wait
  constexpr int PRE = Pre<WT>::n;
  Chunk<WT> pa[PRE], pb[DUAL ? PRE : 1];
  const int nchunks = K / 8;
#pragma unroll
  for (int c = 0; c < PRE; c++) {
    const int ci = lane + 32 * c;
    if (has_row && ci < nchunks) {
      pa[c].load(w0 + ci * 8);
      if (DUAL) pb[c].load(w1 + ci * 8);
    }
  }
  pdl_wait();
  pdl_trigger();
  build_input<TT, KC, BlockTeam, true>(BlockTeam{}, in, T, K, xs, blockIdx.x == 0);

  float acc0[TT], acc1[TT];
#pragma unroll
  for (int t = 0; t < TT; t++) acc0[t] = acc1[t] = 0.f;
  auto fma_chunk = [&](const float *w, const float *u, int ci) {
    const int k = ci * 8;
#pragma unroll
    for (int t = 0; t < TT; t++) {
      if (t < T) {
        const float4 xa = reinterpret_cast<const float4 *>(xs + t * K)[ci];  // halves layout
        const float4 xb = reinterpret_cast<const float4 *>(xs + t * K)[K / 8 + ci];
        const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
        for (int i = 0; i < 8; i++) {
          acc0[t] = fmaf(w[i], xv[i], acc0[t]);
          if (DUAL) acc1[t] = fmaf(u[i], xv[i], acc1[t]);
        }
      }
    }
  };
  if (has_row) {
#pragma unroll
    for (int c = 0; c < PRE; c++) {
      const int ci = lane + 32 * c;
      if (ci < nchunks) {
        float w[8], u[8];
        pa[c].get(w);
        if (DUAL) pb[c].get(u);
        fma_chunk(w, u, ci);
      }
    }
#pragma unroll 4
    for (int ci = lane + 32 * PRE; ci < nchunks; ci += 32) {
      Chunk<WT> x, y;
      x.load(w0 + ci * 8);
      if (DUAL) y.load(w1 + ci * 8);
      float w[8], u[8];
      x.get(w);
      if (DUAL) y.get(u);
      fma_chunk(w, u, ci);
    }
  }
#pragma unroll
  for (int t = 0; t < TT; t++) {
    if (t >= T) break;
    const float a = warp_sum(acc0[t]);
    const float b = DUAL ? warp_sum(acc1[t]) : 0.f;
    if (lane == 0 && has_row) {
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
  if (!he.enabled) return;
  // arrival per head: the last block of a head runs its epilogue
  __shared__ int last;
  __threadfence();
  __syncthreads();
  const int head = (blockIdx.x * FW) / he.d.hd;
  if (threadIdx.x == 0) {
    const int per_head = he.d.hd / FW;
    const int old = atomicAdd(&he.counters[head], 1);
    last = old == per_head - 1;
    if (last) he.counters[head] = 0;  // ready for the next launch
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  head_epilogue(BlockTeam{}, he, head, T, Y, ldy);
}

// ---------------------------------------------------------------------------------------
// attention with the combine in the last split block
// ---------------------------------------------------------------------------------------

constexpr int AW = 4;

template <bool Q8, int REP, int NV>
__global__ void __launch_bounds__(AW * 32) attn_fused_kernel(const float *__restrict__ qkvg, int ldq, Dims d,
                                                             Rows rows, Ring ring, int splits, int ks_len,
                                                             float *__restrict__ part, const float *__restrict__ sg,
                                                             float *__restrict__ z, int *counters) {
  constexpr int HD = NV * 32;
  __shared__ float qs[REP][HD];
  __shared__ float wm[AW][REP], wl[AW][REP];
  __shared__ float wo[AW][REP][HD];
  __shared__ int last;
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x / d.nk, kh = blockIdx.x % d.nk, sp = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seq = rows.seq[r];
  const long p = (long)rows.seq_pos[seq] + rows.off[r];
  const long lo = ring.window == INT_MAX ? 0 : (p + 1 - ring.window > 0 ? p + 1 - ring.window : 0);
  const long k0 = lo + (long)sp * ks_len;
  const long k1 = (k0 + ks_len - 1 < p) ? k0 + ks_len - 1 : p;
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
  for (long kb = k0 + warp * 32; kb <= k1; kb += AW * 32) {
    const long pe = kb + lane;
    const int rr = (int)(pe % ring.cap);
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
            const int8_t *bb = reinterpret_cast<const int8_t *>(&w);
#pragma unroll
            for (int e = 0; e < 16; e++) {
              const float kv = (float)bb[e];
#pragma unroll
              for (int h = 0; h < REP; h++) dg[h] = fmaf(qs[h][g * 32 + c * 16 + e], kv, dg[h]);
            }
          }
          const float sgk = __ldg(ksc + g);
#pragma unroll
          for (int h = 0; h < REP; h++) s[h] = fmaf(sgk, dg[h], s[h]);
        }
      }
    }
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
      const float corr = expf(m[h] - mn);
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
    for (int w = 0; w < AW; w++) M = fmaxf(M, wm[w][h]);
    float o = 0.f, L = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < AW; w++) {
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
  // the last split block of (row, kv head) merges the splits and gates
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    int *ctr = counters + r * d.nk + kh;
    const int old = atomicAdd(ctr, 1);
    last = old == splits - 1;
    if (last) *ctr = 0;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  const float *pr = part + (size_t)(r * d.nk + kh) * splits * REP * (HD + 2);
  const size_t col0 = (size_t)kh * REP * HD;
  const float *vcol = (Q8 && frozen) ? reinterpret_cast<const float *>(slot + ring.L.vcol) + (size_t)kh * HD : nullptr;
  // the warps' partial outputs are no longer needed: their space holds the merge's factors
  merge_splits<REP, HD>(BlockTeam{}, pr, splits, &wo[0][0][0], qkvg + (size_t)r * ldq + (size_t)(d.nh + 2 * d.nk) * HD + col0,
                        sg + col0, vcol, z + (size_t)r * d.nh * HD + col0);
}

template <typename K, typename... Args>
cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, bool pdl, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---------------------------------------------------------------------------------------
// bf16 GEMV with the weights streamed by bulk copies (TMA) into a shared-memory ring
// ---------------------------------------------------------------------------------------
//
// One block per SM takes a contiguous range of output rows. Thread 0 copies chunks of CH
// rows (and, for SwiGLU, the matching up rows) with cp.async.bulk into ST stages; the
// first ST chunks are requested before griddepcontrol.wait, so the weights are in flight
// while the previous kernel finishes and while the prologue builds the input rows. Each
// warp reduces whole rows of a chunk from shared memory. With ~100 KB of shared memory and
// few registers per thread the next kernel's block fits beside this one.

constexpr uint32_t SWAIT = 1u << 20;

__device__ __forceinline__ uint32_t s_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ bool s_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < SWAIT; i++) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  return false;
}

__device__ __forceinline__ void bulk_copy(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

template <int TT, bool DUAL, int KC>
__global__ void __launch_bounds__(FW * 32) gemv_stream_kernel(const __nv_bfloat16 *__restrict__ W, int N, int K,
                                                              int T, int CH, int ST, GemvIn in,
                                                              float *__restrict__ Y, int ldy, EpiArgs ep, HeadEpi he,
                                                              int *err) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[8];
  __shared__ int last_sh, fail_sh;
  float *xs = reinterpret_cast<float *>(smem_raw);  // [T][K]
  const uint32_t wbase = (s_u32(smem_raw) + (uint32_t)T * K * 4 + 127) & ~127u;
  const int rb = (int)((long)N * blockIdx.x / gridDim.x), re = (int)((long)N * (blockIdx.x + 1) / gridDim.x);
  const int nchunks = (re - rb + CH - 1) / CH;
  const uint32_t row_bytes = (uint32_t)K * 2;
  const uint32_t stage_bytes = (uint32_t)CH * row_bytes * (DUAL ? 2 : 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  auto issue = [&](int c) {
    const int s = c % ST;
    const int r0 = rb + c * CH, nr = min(CH, re - r0);
    const uint32_t bar = s_u32(&full[s]);
    const uint32_t bytes = (uint32_t)nr * row_bytes;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes * (DUAL ? 2 : 1))
                 : "memory");
    bulk_copy(wbase + s * stage_bytes, W + (size_t)r0 * K, bytes, bar);
    if (DUAL) bulk_copy(wbase + s * stage_bytes + CH * row_bytes, W + (size_t)(r0 + ep.pair) * K, bytes, bar);
  };
  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; s++) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(s_u32(&full[s])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fail_sh = 0;
    for (int c = 0; c < ST && c < nchunks; c++) issue(c);  // weights only: before the wait
  }
  pdl_wait();
  pdl_trigger();
  build_input<TT, KC, BlockTeam, true>(BlockTeam{}, in, T, K, xs, blockIdx.x == 0);  // ends with __syncthreads

  for (int c = 0; c < nchunks; c++) {
    const int s = c % ST;
    if (!s_wait(s_u32(&full[s]), (c / ST) & 1)) {
      if (lane == 0) atomicExch(err, 5);
      fail_sh = 1;
    }
    __syncthreads();
    if (fail_sh) break;
    const int r0 = rb + c * CH, nr = min(CH, re - r0);
    const __nv_bfloat16 *ws = reinterpret_cast<const __nv_bfloat16 *>(smem_raw + (wbase - s_u32(smem_raw)) +
                                                                      (size_t)s * stage_bytes);
    for (int rr = warp; rr < nr; rr += FW) {
      const __nv_bfloat16 *w0 = ws + (size_t)rr * K;
      const __nv_bfloat16 *w1 = DUAL ? ws + (size_t)(CH + rr) * K : nullptr;
      float acc0[TT], acc1[TT];
#pragma unroll
      for (int t = 0; t < TT; t++) acc0[t] = acc1[t] = 0.f;
#pragma unroll 4
      for (int k = lane * 8; k < K; k += 256) {
        float w[8], u[8];
        unpack8(*reinterpret_cast<const uint4 *>(w0 + k), w);
        if (DUAL) unpack8(*reinterpret_cast<const uint4 *>(w1 + k), u);
#pragma unroll
        for (int t = 0; t < TT; t++) {
          if (t < T) {
            const float4 xa = reinterpret_cast<const float4 *>(xs + t * K)[k / 8];  // halves layout
            const float4 xb = reinterpret_cast<const float4 *>(xs + t * K)[K / 8 + k / 8];
            const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
            for (int i = 0; i < 8; i++) {
              acc0[t] = fmaf(w[i], xv[i], acc0[t]);
              if (DUAL) acc1[t] = fmaf(u[i], xv[i], acc1[t]);
            }
          }
        }
      }
      const int n = r0 + rr;
#pragma unroll
      for (int t = 0; t < TT; t++) {
        if (t >= T) break;
        const float a = warp_sum(acc0[t]);
        const float b = DUAL ? warp_sum(acc1[t]) : 0.f;
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
    __syncthreads();  // the stage is free again
    if (threadIdx.x == 0 && c + ST < nchunks) issue(c + ST);
  }
  if (!he.enabled || fail_sh) return;
  // heads this block finished rows of: the block that completes a head runs its epilogue
  __threadfence();
  __syncthreads();
  const int hd = he.d.hd;
  for (int h = rb / hd; h <= (re - 1) / hd && re > rb; h++) {
    if (threadIdx.x == 0) {
      const int cnt = min(re, (h + 1) * hd) - max(rb, h * hd);
      const int old = atomicAdd(&he.counters[h], cnt);
      last_sh = old + cnt == hd;
      if (last_sh) he.counters[h] = 0;
    }
    __syncthreads();
    if (last_sh) {
      __threadfence();
      head_epilogue(BlockTeam{}, he, h, T, Y, ldy);
    }
    __syncthreads();
  }
}

template <int TT, bool DUAL, int KC>
cudaError_t gemv_stream_k(const void *W, int N, int K, int T, GemvIn in, float *Y, int ldy, EpiArgs ep, HeadEpi he,
                          int *err, bool pdl, cudaStream_t s) {
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
  }
  const size_t row_bytes = (size_t)K * 2 * (DUAL ? 2 : 1);
  const size_t xs_bytes = (size_t)T * K * 4;
  const size_t budget = 110 * 1024;
  if (xs_bytes + 128 + 2 * row_bytes > 200 * 1024) return cudaErrorInvalidValue;
  const size_t wbudget = budget > xs_bytes + 128 + 2 * row_bytes ? budget - xs_bytes - 128 : 2 * row_bytes;
  int CH = (int)std::min<size_t>(32, std::max<size_t>(1, (wbudget / 3) / row_bytes));
  int ST = (int)std::min<size_t>(8, std::max<size_t>(2, wbudget / (CH * row_bytes)));
  const int rows_per_block = (N + sms - 1) / sms;
  if (CH > rows_per_block) CH = rows_per_block;
  ST = (int)std::min<size_t>(ST, std::max<size_t>(2, wbudget / (CH * row_bytes)));
  ST = std::min(ST, 8);
  const size_t smem = xs_bytes + 128 + (size_t)ST * CH * row_bytes;
  auto kern = gemv_stream_kernel<TT, DUAL, KC>;
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    attr = true;
  }
  const int grid = std::min(sms, N);
  return launch_pdl(kern, dim3(grid), dim3(FW * 32), smem, pdl, s, static_cast<const __nv_bfloat16 *>(W), N, K, T, CH,
                    ST, in, Y, ldy, ep, he, err);
}

template <int TT, bool DUAL>
cudaError_t gemv_stream_t(const void *W, int N, int K, int T, GemvIn in, float *Y, int ldy, EpiArgs ep, HeadEpi he,
                          int *err, bool pdl, cudaStream_t s) {
  const int kc = (K / 4 + FW * 32 - 1) / (FW * 32);
  if (kc <= 2) return gemv_stream_k<TT, DUAL, 2>(W, N, K, T, in, Y, ldy, ep, he, err, pdl, s);
  if (kc <= 4) return gemv_stream_k<TT, DUAL, 4>(W, N, K, T, in, Y, ldy, ep, he, err, pdl, s);
  if (kc <= 6) return gemv_stream_k<TT, DUAL, 6>(W, N, K, T, in, Y, ldy, ep, he, err, pdl, s);
  return gemv_stream_k<TT, DUAL, 8>(W, N, K, T, in, Y, ldy, ep, he, err, pdl, s);
}

template <bool DUAL>
cudaError_t gemv_stream_d(const void *W, int N, int K, int T, GemvIn in, float *Y, int ldy, EpiArgs ep, HeadEpi he,
                          int *err, bool pdl, cudaStream_t s) {
  switch (T) {
    case 1: return gemv_stream_t<1, DUAL>(W, N, K, T, in, Y, ldy, ep, he, err, pdl, s);
    case 2: return gemv_stream_t<2, DUAL>(W, N, K, T, in, Y, ldy, ep, he, err, pdl, s);
    default: return gemv_stream_t<4, DUAL>(W, N, K, T, in, Y, ldy, ep, he, err, pdl, s);
  }
}

template <typename WT, int TT, bool DUAL, int KC>
cudaError_t gemv_fused_k(const void *W, int N, int K, int T, GemvIn in, float *Y, int ldy, EpiArgs ep, HeadEpi he,
                         bool pdl, cudaStream_t s) {
  auto kern = gemv_fused_kernel<WT, TT, DUAL, KC>;
  const size_t smem = (size_t)T * K * sizeof(float);
  static bool attr_done = false;
  if (!attr_done) {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
    attr_done = true;
  }
  dim3 grid((N + FW - 1) / FW);
  return launch_pdl(kern, grid, dim3(FW * 32), smem, pdl, s, static_cast<const WT *>(W), N, K, T, in, Y, ldy, ep, he);
}

template <typename WT, int TT, bool DUAL>
cudaError_t gemv_fused_t(const void *W, int N, int K, int T, GemvIn in, float *Y, int ldy, EpiArgs ep, HeadEpi he,
                         bool pdl, cudaStream_t s) {
  const int kc = (K / 4 + FW * 32 - 1) / (FW * 32);
  if (kc <= 2) return gemv_fused_k<WT, TT, DUAL, 2>(W, N, K, T, in, Y, ldy, ep, he, pdl, s);
  if (kc <= 4) return gemv_fused_k<WT, TT, DUAL, 4>(W, N, K, T, in, Y, ldy, ep, he, pdl, s);
  if (kc <= 6) return gemv_fused_k<WT, TT, DUAL, 6>(W, N, K, T, in, Y, ldy, ep, he, pdl, s);
  return gemv_fused_k<WT, TT, DUAL, 8>(W, N, K, T, in, Y, ldy, ep, he, pdl, s);
}

template <typename WT, bool DUAL>
cudaError_t gemv_fused_d(const void *W, int N, int K, int T, GemvIn in, float *Y, int ldy, EpiArgs ep, HeadEpi he,
                         bool pdl, cudaStream_t s) {
  switch (T) {
    case 1: return gemv_fused_t<WT, 1, DUAL>(W, N, K, T, in, Y, ldy, ep, he, pdl, s);
    case 2: return gemv_fused_t<WT, 2, DUAL>(W, N, K, T, in, Y, ldy, ep, he, pdl, s);
    default: return gemv_fused_t<WT, 4, DUAL>(W, N, K, T, in, Y, ldy, ep, he, pdl, s);
  }
}

template <bool Q8, int REP, int NV>
cudaError_t attn_fused_t(const float *qkvg, int ldq, Dims d, Rows rows, Ring ring, int splits, int kps, float *part,
                         const float *sg, float *z, int *counters, bool pdl, cudaStream_t s) {
  dim3 grid(rows.n * d.nk, splits);
  return launch_pdl(attn_fused_kernel<Q8, REP, NV>, grid, dim3(AW * 32), 0, pdl, s, qkvg, ldq, d, rows, ring, splits,
                    kps, part, sg, z, counters);
}

template <bool Q8>
cudaError_t attn_fused_q(const float *qkvg, int ldq, Dims d, Rows rows, Ring ring, int splits, int kps, float *part,
                         const float *sg, float *z, int *counters, bool pdl, cudaStream_t s) {
  const int rep = d.nh / d.nk, nv = d.hd / 32;
#define DISPATCH(R, N)       \
  if (rep == R && nv == N) \
    return attn_fused_t<Q8, R, N>(qkvg, ldq, d, rows, ring, splits, kps, part, sg, z, counters, pdl, s);
  DISPATCH(1, 1) DISPATCH(1, 2) DISPATCH(1, 4)
  DISPATCH(2, 1) DISPATCH(2, 2) DISPATCH(2, 4)
  DISPATCH(4, 1) DISPATCH(4, 2) DISPATCH(4, 4)
  DISPATCH(8, 1) DISPATCH(8, 2) DISPATCH(8, 4)
#undef DISPATCH
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_gemv_fused(const void *W, int wdtype, int N, int K, int T, GemvIn in, float *Y, int ldy,
                              EpiArgs ep, HeadEpi he, int *err, bool pdl, cudaStream_t s) {
  if (T < 1 || T > MAXT || K % 8 != 0 || K > 8192 || (size_t)T * K * 4 > 96 * 1024) return cudaErrorInvalidValue;
  if (he.enabled && ((he.d.hd / 2) % 32 != 0 || T * (he.d.hd / 2) > FW * 32)) return cudaErrorInvalidValue;
  const bool dual = ep.mode == EPI_SILU;
  static const bool stream_off = [] {
    const char *e = getenv("DORY_GEMV_STREAM");
    return e && e[0] == '0';
  }();
  if (wdtype == W_BF16 && !stream_off)
    return dual ? gemv_stream_d<true>(W, N, K, T, in, Y, ldy, ep, he, err, pdl, s)
                : gemv_stream_d<false>(W, N, K, T, in, Y, ldy, ep, he, err, pdl, s);
  if (wdtype == W_BF16)
    return dual ? gemv_fused_d<__nv_bfloat16, true>(W, N, K, T, in, Y, ldy, ep, he, pdl, s)
                : gemv_fused_d<__nv_bfloat16, false>(W, N, K, T, in, Y, ldy, ep, he, pdl, s);
  return dual ? gemv_fused_d<float, true>(W, N, K, T, in, Y, ldy, ep, he, pdl, s)
              : gemv_fused_d<float, false>(W, N, K, T, in, Y, ldy, ep, he, pdl, s);
}

cudaError_t launch_attention_fused(const float *qkvg, int ldq, Dims d, Rows rows, Ring ring, int splits, int kps,
                                   float *part, const float *sg, float *z, int *counters, bool pdl, cudaStream_t s) {
  return ring.q8 ? attn_fused_q<true>(qkvg, ldq, d, rows, ring, splits, kps, part, sg, z, counters, pdl, s)
                 : attn_fused_q<false>(qkvg, ldq, d, rows, ring, splits, kps, part, sg, z, counters, pdl, s);
}

}  // namespace dory
