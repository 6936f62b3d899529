// Windowed GQA attention of a batched decode step over f32 rings (dory.rs fn attn_layer):
// one block per (row, kv head) streams the row's window through shared memory.
//
// The window [max(p - W + 1, 0), p] is walked in tiles of 32 positions; a tile's K rows, V
// rows and position tags are contiguous in the ring (capacities are whole multiples of 64)
// and arrive with three bulk copies into one of three stages, completion on the stage's
// mbarrier. Warp h takes query head h of the group (more heads than warps: h, h + 4, ...):
// lane j scores key j (rotated chunk order, so the 32 lanes spread over the banks), then an
// online softmax keeps the running max and sum, and the value sum runs with lane l owning
// hd/32 dims and the weights broadcast by shuffles. A stage is refilled once every warp has
// left it (an arrival per warp on the stage's second mbarrier). The output y / l is gated,
// y * sigmoid(g * s_g^2), into z; the row norm follows in its own kernel. With two blocks
// per SM about 190 KB of K/V are in flight per SM. Waits are bounded; on expiry the block
// sets error 7, lets its copies land and returns.
#include <climits>

#include "async.cuh"
#include "common.cuh"
#include "kernels.h"

namespace dory {

namespace {

constexpr int AS_WARPS = 4;
constexpr int AS_KEYS = 32;   // positions per tile
constexpr int AS_STAGES = 3;
constexpr int ERR_STREAM = 7;

template <int HD>
struct StreamSmem {
  static constexpr int TILE = AS_KEYS * HD * 4;              // bytes of K (or V) per tile
  static constexpr int STAGE = 2 * TILE + AS_KEYS * 4;       // K, V, tags
  static constexpr int TOTAL = AS_STAGES * STAGE + 128;      // + alignment slack
};

template <int HD, int REP>
__global__ void __launch_bounds__(AS_WARPS * 32) attn_stream_kernel(const float *__restrict__ qkvg, int ldq, Dims d,
                                                                    Rows rows, Ring ring, const float *__restrict__ sg,
                                                                    float *__restrict__ z, int *err) {
  constexpr int NV = HD / 32, NC = HD / 4;
  using S = StreamSmem<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~(uintptr_t)127);
  __shared__ __align__(8) uint64_t full[AS_STAGES], empty[AS_STAGES];
  __shared__ __align__(16) float qs[REP][HD];
  __shared__ volatile int stop;
  const int r = blockIdx.x / d.nk, kh = blockIdx.x % d.nk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seq = rows.seq[r];
  const long p = (long)rows.seq_pos[seq] + rows.off[r];
  const long lo = ring.window == INT_MAX ? 0 : (p + 1 - ring.window > 0 ? p + 1 - ring.window : 0);
  const long t0 = lo / AS_KEYS;
  const int ntiles = (int)(p / AS_KEYS - t0 + 1);
  const char *slot = ring.base + (size_t)seq * ring.seq_stride + ring.off;
  const char *kbase = slot + ring.L.k + (size_t)kh * ring.cap * HD * 4;
  const char *vbase = slot + ring.L.v + (size_t)kh * ring.cap * HD * 4;
  const char *tbase = slot + ring.L.tags;

  auto issue = [&](int t) {  // tile t into stage t % AS_STAGES
    const int s = t % AS_STAGES;
    const int rr = (int)(((t0 + t) * AS_KEYS) % ring.cap);
    const uint32_t bar = smem_addr(&full[s]), dst = smem_addr(base + (size_t)s * S::STAGE);
    mbar_expect_tx(bar, S::STAGE);
    bulk_g2s(dst, kbase + (size_t)rr * HD * 4, S::TILE, bar);
    bulk_g2s(dst + S::TILE, vbase + (size_t)rr * HD * 4, S::TILE, bar);
    bulk_g2s(dst + 2 * S::TILE, tbase + (size_t)rr * 4, AS_KEYS * 4, bar);
  };
  if (threadIdx.x == 0) {
    for (int s = 0; s < AS_STAGES; s++) {
      mbar_init(smem_addr(&full[s]), 1);
      mbar_init(smem_addr(&empty[s]), AS_WARPS);
    }
    mbar_fence_init();
    stop = 0;
    for (int t = 0; t < AS_STAGES && t < ntiles; t++) issue(t);
  }
  for (int i = threadIdx.x; i < REP * HD; i += blockDim.x)
    qs[i / HD][i % HD] = qkvg[(size_t)r * ldq + (size_t)kh * REP * HD + i];
  __syncthreads();

  const float scale = 1.f / sqrtf((float)HD);
  float m[(REP + AS_WARPS - 1) / AS_WARPS], l[(REP + AS_WARPS - 1) / AS_WARPS];
  float acc[(REP + AS_WARPS - 1) / AS_WARPS][NV];
#pragma unroll
  for (int u = 0; u < (REP + AS_WARPS - 1) / AS_WARPS; u++) {
    m[u] = -INFINITY;
    l[u] = 0.f;
#pragma unroll
    for (int i = 0; i < NV; i++) acc[u][i] = 0.f;
  }
  int issued = ntiles < AS_STAGES ? ntiles : AS_STAGES;
  bool ok = true;
  for (int t = 0; t < ntiles; t++) {
    const int s = t % AS_STAGES;
    if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&full[s]), (t / AS_STAGES) & 1, &stop))) {
      if (lane == 0) {
        stop = 1;
        atomicExch(err, ERR_STREAM);
      }
      ok = false;
      break;
    }
    const float *Kt = reinterpret_cast<const float *>(base + (size_t)s * S::STAGE);
    const float *Vt = Kt + AS_KEYS * HD;
    const int32_t *tags = reinterpret_cast<const int32_t *>(Vt + AS_KEYS * HD);
    const long pe = (t0 + t) * AS_KEYS + lane;
    const bool valid = pe >= lo && pe <= p && tags[lane] == (int32_t)pe;
#pragma unroll
    for (int u = 0; u < (REP + AS_WARPS - 1) / AS_WARPS; u++) {
      const int h = warp + u * AS_WARPS;
      if (h >= REP) break;
      float2 s2 = make_float2(0.f, 0.f);
      if (valid) {
        const float4 *kr = reinterpret_cast<const float4 *>(Kt + lane * HD);
        const float4 *q4 = reinterpret_cast<const float4 *>(qs[h]);
#pragma unroll 8
        for (int c = 0; c < NC; c++) {
          const int cc = (c + lane) & (NC - 1);
          const float4 k = kr[cc], q = q4[cc];
          s2 = ffma2(make_float2(q.y, q.w), make_float2(k.y, k.w), s2);
          s2 = ffma2(make_float2(q.x, q.z), make_float2(k.x, k.z), s2);
        }
      }
      const float sc = valid ? (s2.x + s2.y) * scale : -INFINITY;
      const float mt = warp_max(sc);
      const float mn = fmaxf(m[u], mt);
      if (mn == -INFINITY) continue;  // nothing valid yet (warp-uniform)
      const float fold = m[u] == -INFINITY ? 0.f : expf(m[u] - mn);
      const float e = sc == -INFINITY ? 0.f : expf(sc - mn);
      l[u] = l[u] * fold + warp_sum(e);
      m[u] = mn;
      float a0[NV], a1[NV];
#pragma unroll
      for (int i = 0; i < NV; i++) {
        a0[i] = acc[u][i] * fold;
        a1[i] = 0.f;
      }
#pragma unroll 4
      for (int j = 0; j < AS_KEYS; j += 2) {
        const float w0 = __shfl_sync(0xffffffffu, e, j), w1 = __shfl_sync(0xffffffffu, e, j + 1);
        const float *v0 = Vt + j * HD + lane * NV, *v1 = v0 + HD;
#pragma unroll
        for (int i = 0; i < NV; i += 2) {
          const float2 r0 = ffma2(make_float2(w0, w0), make_float2(v0[i], v0[i + 1]), make_float2(a0[i], a0[i + 1]));
          const float2 r1 = ffma2(make_float2(w1, w1), make_float2(v1[i], v1[i + 1]), make_float2(a1[i], a1[i + 1]));
          a0[i] = r0.x;
          a0[i + 1] = r0.y;
          a1[i] = r1.x;
          a1[i + 1] = r1.y;
        }
      }
#pragma unroll
      for (int i = 0; i < NV; i++) acc[u][i] = a0[i] + a1[i];
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
    // thread 0 refills the stage once every warp has left it
    if (threadIdx.x == 0 && issued < ntiles) {
      if (!mbar_wait(smem_addr(&empty[s]), (t / AS_STAGES) & 1, &stop)) {
        stop = 1;
        atomicExch(err, ERR_STREAM);
      } else {
        issue(issued);
        issued++;
      }
    }
  }
  // copies in flight land before the block may exit
  if (threadIdx.x == 0)
    for (int t = issued - AS_STAGES < 0 ? 0 : issued - AS_STAGES; t < issued; t++)
      mbar_wait(smem_addr(&full[t % AS_STAGES]), (t / AS_STAGES) & 1);
  if (!ok || stop) return;
  const float *g = qkvg + (size_t)r * ldq + (size_t)(d.nh + 2 * d.nk) * HD;
#pragma unroll
  for (int u = 0; u < (REP + AS_WARPS - 1) / AS_WARPS; u++) {
    const int h = warp + u * AS_WARPS;
    if (h >= REP) break;
    const float inv = l[u] > 0.f ? 1.f / l[u] : 0.f;
#pragma unroll
    for (int i = 0; i < NV; i++) {
      const int col = (kh * REP + h) * HD + lane * NV + i;
      z[(size_t)r * d.nh * HD + col] = acc[u][i] * inv * sigmoidf_(g[col] * sg[col]);
    }
  }
}

template <int HD, int REP>
cudaError_t stream_t(const float *qkvg, int ldq, Dims d, Rows rows, Ring ring, const float *sg, float *z, int *err,
                     cudaStream_t s) {
  using S = StreamSmem<HD>;
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(attn_stream_kernel<HD, REP>, cudaFuncAttributeMaxDynamicSharedMemorySize, S::TOTAL);
    attr = true;
  }
  attn_stream_kernel<HD, REP><<<rows.n * d.nk, AS_WARPS * 32, S::TOTAL, s>>>(qkvg, ldq, d, rows, ring, sg, z, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention_stream(const float *qkvg, int ldq, Dims d, Rows rows, Ring ring, const float *sg,
                                    float *z, int *err, cudaStream_t s) {
  const int rep = d.nh / d.nk;
#define STREAM(H, R) \
  if (d.hd == H && rep == R) return stream_t<H, R>(qkvg, ldq, d, rows, ring, sg, z, err, s);
  STREAM(64, 1) STREAM(64, 2) STREAM(64, 4) STREAM(64, 8)
  STREAM(128, 1) STREAM(128, 2) STREAM(128, 4) STREAM(128, 8)
#undef STREAM
  return cudaErrorInvalidValue;
}

}  // namespace dory
