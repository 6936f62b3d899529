// Windowed GQA attention over f32 rings with TMA-staged K/V tiles (dory.rs fn attn_layer).
//
// One block per (row, kv head, block of 64 positions). Ring capacities are whole multiples
// of 64 rows, so the 64 positions [64 b, 64 b + 64) sit in 64 consecutive ring rows; one
// elected thread loads that block's K and V rows with 2D tensor copies (boxes of 64 rows x
// 32 floats, 128-byte swizzle) into shared memory, completion on an mbarrier. Scores: lane
// j of warp w owns key 32 w + j and reads its row chunk by chunk; the swizzle spreads the
// 32 lanes' 16-byte reads over all banks. A position counts when it lies in
// [max(p - W + 1, 0), p] and the ring row's tag holds it (per_loop holes are skipped).
// Softmax statistics per head over the block, then the value sum with lane l owning hd/32
// dims of one head per warp. Each block leaves (max, sum, partial output) per head; the
// last block of a (row, kv head) merges them and applies the gate y * sigmoid(g * s_g^2).
#include <climits>

#include "common.cuh"
#include "fused_body.cuh"
#include "kernels.h"

namespace dory {

namespace {

constexpr int AB = 64;  // positions per block
constexpr uint32_t WAIT_LIMIT = 1u << 20;

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < WAIT_LIMIT; i++) {
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

// float4 chunk c (0..7) of row j (0..63) of column box cb in a [box][64][32] swizzled tile
__device__ __forceinline__ const float4 *tile_chunk(const float *tile, int cb, int j, int c) {
  return reinterpret_cast<const float4 *>(tile + (cb * AB + j) * 32 + ((c ^ (j & 7)) << 2));
}

template <int REP, int NV>
__global__ void __launch_bounds__(128) attn_tma_kernel(const __grid_constant__ CUtensorMap kvmap,
                                                       const float *__restrict__ qkvg, int ldq, Dims d, Rows rows,
                                                       Ring ring, int splits, float *__restrict__ part,
                                                       const float *__restrict__ sg, float *__restrict__ z,
                                                       int *counters, int *err) {
  constexpr int HD = NV * 32;
  constexpr int NB = HD / 32;  // column boxes per tile
  extern __shared__ uint8_t smem_raw[];
  float *Ks = reinterpret_cast<float *>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
  float *Vs = Ks + NB * AB * 32;
  __shared__ float qs[REP][HD];
  __shared__ float ps[REP][AB];
  __shared__ float mh[REP], lh[REP];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int last, ok_sh;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int r = blockIdx.x / d.nk, kh = blockIdx.x % d.nk, sp = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seq = rows.seq[r];
  const long p = (long)rows.seq_pos[seq] + rows.off[r];
  const long lo = ring.window == INT_MAX ? 0 : (p + 1 - ring.window > 0 ? p + 1 - ring.window : 0);
  const long P0 = (lo / AB + sp) * AB;  // first position of this block
  const bool active = P0 <= p;
  const char *slot = ring.base + (size_t)seq * ring.seq_stride + ring.off;
  const int32_t *tags = reinterpret_cast<const int32_t *>(slot + ring.L.tags);
  const int rr0 = (int)(P0 % ring.cap);

  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    ok_sh = 1;
  }
  __syncthreads();
  if (active && threadIdx.x == 0) {
    const uint32_t b = smem_u32(&bar);
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(2 * NB * AB * 32 * 4)
                 : "memory");
    // row index of ring row rr0 of head kh in the KV memory seen as [rows][HD] f32
    const size_t rowK = ((size_t)(slot - ring.base) + ring.L.k) / (HD * 4) + (size_t)kh * ring.cap + rr0;
    const size_t rowV = ((size_t)(slot - ring.base) + ring.L.v) / (HD * 4) + (size_t)kh * ring.cap + rr0;
#pragma unroll
    for (int cb = 0; cb < NB; cb++) {
      asm volatile(
          "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
              smem_u32(Ks + cb * AB * 32)),
          "l"(reinterpret_cast<uint64_t>(&kvmap)), "r"(cb * 32), "r"((int)rowK), "r"(b)
          : "memory");
      asm volatile(
          "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
              smem_u32(Vs + cb * AB * 32)),
          "l"(reinterpret_cast<uint64_t>(&kvmap)), "r"(cb * 32), "r"((int)rowV), "r"(b)
          : "memory");
    }
  }
  const float *q = qkvg + (size_t)r * ldq + (size_t)kh * REP * HD;
  for (int i = threadIdx.x; i < REP * HD; i += blockDim.x) qs[i / HD][i % HD] = q[i];
  __syncthreads();
  if (active) {
    if (!mbar_wait(smem_u32(&bar), 0)) {
      atomicExch(err, 4);
      ok_sh = 0;
    }
  }
  __syncthreads();
  const bool run = active && ok_sh;

  // scores: warps 0 and 1, lane = key
  const float scale = 1.f / sqrtf((float)HD);
  if (run && warp < 2) {
    const int j = warp * 32 + lane;
    const long pe = P0 + j;
    const bool valid = pe >= lo && pe <= p && tags[rr0 + j] == (int32_t)pe;
    float s[REP];
#pragma unroll
    for (int h = 0; h < REP; h++) s[h] = 0.f;
    if (valid) {
#pragma unroll
      for (int cb = 0; cb < NB; cb++)
#pragma unroll
        for (int c = 0; c < 8; c++) {
          const float4 k4 = *tile_chunk(Ks, cb, j, c);
#pragma unroll
          for (int h = 0; h < REP; h++) {
            const float4 q4 = *reinterpret_cast<const float4 *>(&qs[h][cb * 32 + c * 4]);
            s[h] = fmaf(q4.x, k4.x, fmaf(q4.y, k4.y, fmaf(q4.z, k4.z, fmaf(q4.w, k4.w, s[h]))));
          }
        }
    }
#pragma unroll
    for (int h = 0; h < REP; h++) ps[h][j] = valid ? s[h] * scale : -INFINITY;
  }
  __syncthreads();
  // per-head max and sum over the block; weights p = exp(s - m)
  for (int h = warp; h < REP; h += 4) {
    if (!run) break;
    const float a = ps[h][lane], b = ps[h][lane + 32];
    const float m = warp_max(fmaxf(a, b));
    const float ea = m == -INFINITY ? 0.f : expf(a - m), eb = m == -INFINITY ? 0.f : expf(b - m);
    const float l = warp_sum(ea + eb);
    ps[h][lane] = ea;
    ps[h][lane + 32] = eb;
    if (lane == 0) {
      mh[h] = m;
      lh[h] = l;
    }
  }
  __syncthreads();
  float *out = part + ((size_t)(r * d.nk + kh) * splits + sp) * REP * (HD + 2);
  for (int h = warp; h < REP; h += 4) {
    float acc[NV];
#pragma unroll
    for (int i = 0; i < NV; i++) acc[i] = 0.f;
    if (run) {
      // lane owns dims [NV*lane, NV*lane + NV): box lane*NV/32, chunk (lane*NV%32)/4
      const int dim0 = lane * NV;
      const int cb = dim0 / 32, c = (dim0 % 32) / 4, sub = dim0 % 4;
      for (int j = 0; j < AB; j++) {
        const float w = ps[h][j];
        if (w == 0.f) continue;
        const float *v = reinterpret_cast<const float *>(tile_chunk(Vs, cb, j, c)) + sub;
#pragma unroll
        for (int i = 0; i < NV; i++) acc[i] = fmaf(w, v[i], acc[i]);
      }
    }
#pragma unroll
    for (int i = 0; i < NV; i++) out[h * (HD + 2) + lane * NV + i] = acc[i];
    if (lane == 0) {
      out[h * (HD + 2) + HD] = run ? mh[h] : -INFINITY;
      out[h * (HD + 2) + HD + 1] = run ? lh[h] : 0.f;
    }
  }
  // the last block of (row, kv head) merges the blocks and gates
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
  merge_splits<REP, HD>(BlockTeam{}, pr, splits, Ks, qkvg + (size_t)r * ldq + (size_t)(d.nh + 2 * d.nk) * HD + col0, sg + col0,
                        nullptr, z + (size_t)r * d.nh * HD + col0);
}

template <int REP, int NV>
cudaError_t attn_tma_t(const CUtensorMap &map, const float *qkvg, int ldq, Dims d, Rows rows, Ring ring, int splits,
                       float *part, const float *sg, float *z, int *counters, int *err, bool pdl, cudaStream_t s) {
  constexpr int HD = NV * 32;
  const size_t smem = 2 * (HD / 32) * AB * 32 * 4 + 1024;
  auto kern = attn_tma_kernel<REP, NV>;
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    attr = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(rows.n * d.nk, splits);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, map, qkvg, ldq, d, rows, ring, splits, part, sg, z, counters, err);
}


// q8_2f rings (hd = 128): per 64-position block, tensor copies of the K and V code tiles
// (64 rows x 128 bytes, 128-byte swizzle), the K scales (64 rows x 4 floats) and the V
// scales (64 floats). Scores s = scale * sum_g ks[g] <q * kcol, kq>_g; values
// sum_j (p_j vs_j) vq_j, times vcol in the merge (kv_cache.rs fn attend_group_upto).
template <int REP>
__global__ void __launch_bounds__(128) attn_tma_q8_kernel(const __grid_constant__ CUtensorMap codes,
                                                          const __grid_constant__ CUtensorMap kscales,
                                                          const __grid_constant__ CUtensorMap vscales,
                                                          const float *__restrict__ qkvg, int ldq, Dims d, Rows rows,
                                                          Ring ring, int splits, float *__restrict__ part,
                                                          const float *__restrict__ sg, float *__restrict__ z,
                                                          int *counters, int *err) {
  constexpr int HD = 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *Kq = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t *Vq = Kq + AB * HD;
  float *Ksc = reinterpret_cast<float *>(Vq + AB * HD);  // [64][4]
  float *Vsc = Ksc + AB * 4;                             // [64]
  __shared__ float qs[REP][HD];
  __shared__ float ps[REP][AB];
  __shared__ float mh[REP], lh[REP];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int last, ok_sh;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int r = blockIdx.x / d.nk, kh = blockIdx.x % d.nk, sp = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seq = rows.seq[r];
  const long p = (long)rows.seq_pos[seq] + rows.off[r];
  const long lo = ring.window == INT_MAX ? 0 : (p + 1 - ring.window > 0 ? p + 1 - ring.window : 0);
  const long P0 = (lo / AB + sp) * AB;
  const bool active = P0 <= p;
  const char *slot = ring.base + (size_t)seq * ring.seq_stride + ring.off;
  const int32_t *tags = reinterpret_cast<const int32_t *>(slot + ring.L.tags);
  const int rr0 = (int)(P0 % ring.cap);
  const int frozen = reinterpret_cast<const int32_t *>(slot + ring.L.meta)[kh * 4 + 1];
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    ok_sh = 1;
  }
  __syncthreads();
  if (active && threadIdx.x == 0) {
    const uint32_t b = smem_u32(&bar);
    const uint32_t bytes = 2 * AB * HD + AB * 4 * 4 + AB * 4;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(bytes) : "memory");
    const size_t so = (size_t)(slot - ring.base);
    const size_t row = (size_t)kh * ring.cap + rr0;
    const int rk = (int)((so + ring.L.kq) / HD + row), rv = (int)((so + ring.L.vq) / HD + row);
    const int rs = (int)((so + ring.L.ks) / 16 + row);
    const int rvs = (int)((so + ring.L.vs + row * 4) / (AB * 4));
    const uint64_t mc = reinterpret_cast<uint64_t>(&codes), mk = reinterpret_cast<uint64_t>(&kscales),
                   mv = reinterpret_cast<uint64_t>(&vscales);
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(Kq)), "l"(mc), "r"(0), "r"(rk), "r"(b) : "memory");
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(Vq)), "l"(mc), "r"(0), "r"(rv), "r"(b) : "memory");
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(Ksc)), "l"(mk), "r"(0), "r"(rs), "r"(b) : "memory");
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(Vsc)), "l"(mv), "r"(0), "r"(rvs), "r"(b) : "memory");
  }
  const float *q = qkvg + (size_t)r * ldq + (size_t)kh * REP * HD;
  const float *kcol = reinterpret_cast<const float *>(slot + ring.L.kcol) + (size_t)kh * HD;
  for (int i = threadIdx.x; i < REP * HD; i += blockDim.x) {
    float v = q[i];
    if (frozen) v *= kcol[i % HD];
    qs[i / HD][i % HD] = v;
  }
  __syncthreads();
  if (active && !mbar_wait(smem_u32(&bar), 0)) {
    atomicExch(err, 6);
    ok_sh = 0;
  }
  __syncthreads();
  const bool run = active && ok_sh;
  const float scale = 1.f / sqrtf((float)HD);
  if (run && warp < 2) {
    const int j = warp * 32 + lane;
    const long pe = P0 + j;
    const bool valid = pe >= lo && pe <= p && tags[rr0 + j] == (int32_t)pe;
    float s[REP];
#pragma unroll
    for (int h = 0; h < REP; h++) s[h] = 0.f;
    if (valid) {
#pragma unroll
      for (int g = 0; g < HD / 32; g++) {
        float dg[REP];
#pragma unroll
        for (int h = 0; h < REP; h++) dg[h] = 0.f;
#pragma unroll
        for (int c2 = 0; c2 < 2; c2++) {
          const int c = g * 2 + c2;  // 16-byte chunk of the row
          const int4 w = *reinterpret_cast<const int4 *>(Kq + j * HD + ((c ^ (j & 7)) << 4));
          const int8_t *bb = reinterpret_cast<const int8_t *>(&w);
#pragma unroll
          for (int e = 0; e < 16; e++) {
            const float kv = (float)bb[e];
#pragma unroll
            for (int h = 0; h < REP; h++) dg[h] = fmaf(qs[h][c * 16 + e], kv, dg[h]);
          }
        }
        const float ksg = Ksc[j * 4 + g];
#pragma unroll
        for (int h = 0; h < REP; h++) s[h] = fmaf(ksg, dg[h], s[h]);
      }
    }
#pragma unroll
    for (int h = 0; h < REP; h++) ps[h][j] = valid ? s[h] * scale : -INFINITY;
  }
  __syncthreads();
  for (int h = warp; h < REP; h += 4) {
    if (!run) break;
    const float a = ps[h][lane], b = ps[h][lane + 32];
    const float m = warp_max(fmaxf(a, b));
    const float ea = m == -INFINITY ? 0.f : expf(a - m), eb = m == -INFINITY ? 0.f : expf(b - m);
    const float l = warp_sum(ea + eb);
    ps[h][lane] = ea;
    ps[h][lane + 32] = eb;
    if (lane == 0) {
      mh[h] = m;
      lh[h] = l;
    }
  }
  __syncthreads();
  float *out = part + ((size_t)(r * d.nk + kh) * splits + sp) * REP * (HD + 2);
  for (int h = warp; h < REP; h += 4) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (run) {
      const int c = lane >> 2, sub = (lane & 3) * 4;  // lane owns dims 4 lane .. 4 lane + 3
      for (int j = 0; j < AB; j++) {
        const float w = ps[h][j];
        if (w == 0.f) continue;
        const float wv = w * Vsc[j];
        const char4 v4 = *reinterpret_cast<const char4 *>(Vq + j * HD + ((c ^ (j & 7)) << 4) + sub);
        acc[0] = fmaf(wv, (float)v4.x, acc[0]);
        acc[1] = fmaf(wv, (float)v4.y, acc[1]);
        acc[2] = fmaf(wv, (float)v4.z, acc[2]);
        acc[3] = fmaf(wv, (float)v4.w, acc[3]);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; i++) out[h * (HD + 2) + lane * 4 + i] = acc[i];
    if (lane == 0) {
      out[h * (HD + 2) + HD] = run ? mh[h] : -INFINITY;
      out[h * (HD + 2) + HD + 1] = run ? lh[h] : 0.f;
    }
  }
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
  const float *vcol = reinterpret_cast<const float *>(slot + ring.L.vcol) + (size_t)kh * HD;
  const size_t col0 = (size_t)kh * REP * HD;
  merge_splits<REP, HD>(BlockTeam{}, pr, splits, reinterpret_cast<float *>(Kq), qkvg + (size_t)r * ldq +
                        (size_t)(d.nh + 2 * d.nk) * HD + col0, sg + col0, frozen ? vcol : nullptr,
                        z + (size_t)r * d.nh * HD + col0);
}

template <int REP>
cudaError_t attn_tma_q8_t(const KvMaps &m, const float *qkvg, int ldq, Dims d, Rows rows, Ring ring, int splits,
                          float *part, const float *sg, float *z, int *counters, int *err, bool pdl, cudaStream_t s) {
  const size_t smem = 2 * AB * 128 + AB * 4 * 4 + AB * 4 + 1024;
  auto kern = attn_tma_q8_kernel<REP>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(rows.n * d.nk, splits);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, m.codes, m.kscales, m.vscales, qkvg, ldq, d, rows, ring, splits, part, sg, z,
                            counters, err);
}
}  // namespace

int attn_tma_splits(long window_keys) { return (int)((window_keys + AB - 1) / AB) + 1; }

cudaError_t launch_attention_tma(const CUtensorMap &map, const float *qkvg, int ldq, Dims d, Rows rows, Ring ring,
                                 int splits, float *part, const float *sg, float *z, int *counters, int *err, bool pdl,
                                 cudaStream_t s) {
  const int rep = d.nh / d.nk, nv = d.hd / 32;
#define DISPATCH(R, N) \
  if (rep == R && nv == N) return attn_tma_t<R, N>(map, qkvg, ldq, d, rows, ring, splits, part, sg, z, counters, err, pdl, s);
  DISPATCH(1, 2) DISPATCH(1, 4) DISPATCH(2, 2) DISPATCH(2, 4) DISPATCH(4, 2) DISPATCH(4, 4) DISPATCH(8, 2) DISPATCH(8, 4)
#undef DISPATCH
  return cudaErrorInvalidValue;
}

cudaError_t launch_attention_tma_q8(const KvMaps &m, const float *qkvg, int ldq, Dims d, Rows rows, Ring ring,
                                    int splits, float *part, const float *sg, float *z, int *counters, int *err,
                                    bool pdl, cudaStream_t s) {
  const int rep = d.nh / d.nk;
  if (d.hd != 128) return cudaErrorInvalidValue;
  switch (rep) {
    case 1: return attn_tma_q8_t<1>(m, qkvg, ldq, d, rows, ring, splits, part, sg, z, counters, err, pdl, s);
    case 2: return attn_tma_q8_t<2>(m, qkvg, ldq, d, rows, ring, splits, part, sg, z, counters, err, pdl, s);
    case 4: return attn_tma_q8_t<4>(m, qkvg, ldq, d, rows, ring, splits, part, sg, z, counters, err, pdl, s);
    case 8: return attn_tma_q8_t<8>(m, qkvg, ldq, d, rows, ring, splits, part, sg, z, counters, err, pdl, s);
  }
  return cudaErrorInvalidValue;
}

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encoder() {
  static EncodeTiledFn encode = nullptr;
  if (!encode) {
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  return encode;
}

// rows of `width` elements of `dt` over [base, base + bytes), boxes of box_w x box_h
int kv_map(CUtensorMap *map, CUtensorMapDataType dt, int esz, const void *base, size_t bytes, int width, int box_w,
           int box_h, CUtensorMapSwizzle sw) {
  EncodeTiledFn enc = encoder();
  if (!enc) return -1;
  cuuint64_t dims[2] = {(cuuint64_t)width, (cuuint64_t)(bytes / ((size_t)width * esz))};
  cuuint64_t strides[1] = {(cuuint64_t)width * esz};
  cuuint32_t box[2] = {(cuuint32_t)box_w, (cuuint32_t)box_h};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? 0
             : -2;
}
}  // namespace

// The q8 KV memory seen three ways: 128-byte code rows, 16-byte K-scale rows, 256-byte
// runs of V scales.
int make_tmap_kv_q8(KvMaps *m, const void *base, size_t bytes) {
  if (kv_map(&m->codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base, bytes, 128, 128, AB, CU_TENSOR_MAP_SWIZZLE_128B))
    return -1;
  if (kv_map(&m->kscales, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, bytes, 4, 4, AB, CU_TENSOR_MAP_SWIZZLE_NONE))
    return -1;
  if (kv_map(&m->vscales, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, bytes, AB, AB, 1, CU_TENSOR_MAP_SWIZZLE_NONE))
    return -1;
  return 0;
}

// The KV memory as rows of hd f32 values, read in boxes of 64 rows x 32 floats.
int make_tmap_kv_f32(CUtensorMap *map, const void *base, size_t bytes, int hd) {
  typedef CUresult (*EncodeTiled)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static EncodeTiled encode = nullptr;
  if (!encode) {
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return -1;
    encode = reinterpret_cast<EncodeTiled>(fn);
  }
  cuuint64_t dims[2] = {(cuuint64_t)hd, (cuuint64_t)(bytes / ((size_t)hd * 4))};
  cuuint64_t strides[1] = {(cuuint64_t)hd * 4};
  cuuint32_t box[2] = {32, (cuuint32_t)AB};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -2;
}

}  // namespace dory
