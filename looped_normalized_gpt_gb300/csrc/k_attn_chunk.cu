// Windowed causal GQA attention of a prefill chunk: T consecutive positions p0 .. p0+T-1 of
// one sequence over an f32 ring (dory.rs fn attn_layer; the chunk form of the pages'
// attend_chunk).
//
// One block per (kv head, group of RG rows, block of 64 key positions). The group's
// RG x REP query vectors (64 of them) share the key block: its K and V rows (64 ring rows,
// contiguous since ring capacities are whole multiples of 64) are read once into shared
// memory, rows padded to hd + 4 floats so that eight different rows hit eight different
// bank groups. Scores: thread (tq, tk) owns queries tq + 16a and keys tk + 16b (a, b < 4), a
// 4 x 4 register tile, and sums over the head width a float4 at a time. A key counts for
// the row at p when it lies in [max(p - W + 1, 0), p] and its ring row's tag holds it. Then
// the block's softmax statistics per query (four threads per query), and the value sum with
// the same 4 x (hd/16) register tiling. Each block leaves (output, max, sum) per query in
// the split-KV layout of k_attn.cu; the combine kernel there merges the key blocks and
// applies the gate.
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace dory {

namespace {

constexpr int CK_THREADS = 256;
constexpr int CK_KEYS = 64;    // key positions per block
constexpr int CK_QUERIES = 64; // query vectors per block (rows x query heads of the group)

template <int HD>
struct ChunkSmem {
  static constexpr int LD = HD + 4;  // padded row
  float q[CK_QUERIES][LD];
  float k[CK_KEYS][LD];
  float v[CK_KEYS][LD];
  float s[CK_QUERIES][CK_KEYS + 1];
  float m[CK_QUERIES], l[CK_QUERIES];
  int32_t tag[CK_KEYS];
};

template <int HD, int REP>
__global__ void __launch_bounds__(CK_THREADS) attn_chunk_kernel(const float *__restrict__ qkvg, int ldq, Dims d,
                                                                Rows rows, Ring ring, int nkb,
                                                                float *__restrict__ part) {
  constexpr int RG = CK_QUERIES / REP;  // rows per group
  constexpr int NC = HD / 4;            // float4 chunks per row
  constexpr int NG = HD / 64;           // value float4 groups per thread
  extern __shared__ __align__(16) uint8_t smem_raw[];
  ChunkSmem<HD> &S = *reinterpret_cast<ChunkSmem<HD> *>(smem_raw);
  const int T = rows.n;
  const int nrg = (T + RG - 1) / RG;
  const int kh = blockIdx.x / nrg, rg = blockIdx.x % nrg, sb = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seq = rows.seq[0];
  const long p0 = (long)rows.seq_pos[seq] + rows.off[0];
  const long lo0 = ring.window == INT_MAX ? 0 : (p0 + 1 - ring.window > 0 ? p0 + 1 - ring.window : 0);
  const long P0 = (lo0 / CK_KEYS + sb) * CK_KEYS;  // first position of this key block
  const int r_first = rg * RG, r_end = min(T, r_first + RG);
  const long p_last = p0 + r_end - 1;
  const long lo_first = ring.window == INT_MAX ? 0 : max(p0 + r_first + 1 - (long)ring.window, 0L);
  const bool any = P0 <= p_last && P0 + CK_KEYS - 1 >= lo_first;
  const char *slot = ring.base + (size_t)seq * ring.seq_stride + ring.off;
  const int rr0 = (int)(P0 % ring.cap);

  if (any) {
    const float4 *kg = reinterpret_cast<const float4 *>(slot + ring.L.k) + ((size_t)kh * ring.cap + rr0) * NC;
    const float4 *vg = reinterpret_cast<const float4 *>(slot + ring.L.v) + ((size_t)kh * ring.cap + rr0) * NC;
    for (int i = tid; i < CK_KEYS * NC; i += CK_THREADS) {
      const int j = i / NC, c = i % NC;
      *reinterpret_cast<float4 *>(&S.k[j][c * 4]) = kg[i];
      *reinterpret_cast<float4 *>(&S.v[j][c * 4]) = vg[i];
    }
    for (int i = tid; i < CK_QUERIES * NC; i += CK_THREADS) {
      const int qi = i / NC, c = i % NC;  // query qi = row i * REP + head
      const int r = r_first + qi / REP, h = qi % REP;
      float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
      if (r < T) x = *reinterpret_cast<const float4 *>(qkvg + (size_t)r * ldq + (size_t)(kh * REP + h) * HD + c * 4);
      *reinterpret_cast<float4 *>(&S.q[qi][c * 4]) = x;
    }
    if (tid < CK_KEYS) S.tag[tid] = reinterpret_cast<const int32_t *>(slot + ring.L.tags)[rr0 + tid];
  }
  __syncthreads();

  // scores: thread (tq, tk) owns queries tq + 16a and keys tk + 16b
  const int tq = (warp & 1) * 8 + (lane & 7), tk = (warp >> 1) * 4 + (lane >> 3);
  float acc[4][4];
#pragma unroll
  for (int a = 0; a < 4; a++)
#pragma unroll
    for (int b = 0; b < 4; b++) acc[a][b] = 0.f;
  if (any) {
#pragma unroll 4
    for (int c = 0; c < NC; c++) {
      float4 qv[4], kv[4];
#pragma unroll
      for (int a = 0; a < 4; a++) qv[a] = *reinterpret_cast<const float4 *>(&S.q[tq + 16 * a][c * 4]);
#pragma unroll
      for (int b = 0; b < 4; b++) kv[b] = *reinterpret_cast<const float4 *>(&S.k[tk + 16 * b][c * 4]);
#pragma unroll
      for (int a = 0; a < 4; a++)
#pragma unroll
        for (int b = 0; b < 4; b++)
          acc[a][b] = fmaf(qv[a].x, kv[b].x, fmaf(qv[a].y, kv[b].y, fmaf(qv[a].z, kv[b].z, fmaf(qv[a].w, kv[b].w, acc[a][b]))));
    }
  }
  const float scale = 1.f / sqrtf((float)HD);
#pragma unroll
  for (int a = 0; a < 4; a++) {
    const int qi = tq + 16 * a, r = r_first + qi / REP;
    const long p = p0 + r;
    const long lo = ring.window == INT_MAX ? 0 : (p + 1 - ring.window > 0 ? p + 1 - ring.window : 0);
#pragma unroll
    for (int b = 0; b < 4; b++) {
      const int kj = tk + 16 * b;
      const long pk = P0 + kj;
      const bool valid = any && r < T && pk >= lo && pk <= p && S.tag[kj] == (int32_t)pk;
      S.s[qi][kj] = valid ? acc[a][b] * scale : -INFINITY;
    }
  }
  __syncthreads();
  {  // softmax statistics of the block: four threads per query, 16 keys each
    const int qi = tid >> 2, k0 = (tid & 3) * 16;
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < 16; j++) m = fmaxf(m, S.s[qi][k0 + j]);
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    float l = 0.f;
#pragma unroll
    for (int j = 0; j < 16; j++) {
      const float e = m == -INFINITY ? 0.f : expf(S.s[qi][k0 + j] - m);
      S.s[qi][k0 + j] = e;
      l += e;
    }
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    if ((tid & 3) == 0) {
      S.m[qi] = m;
      S.l[qi] = l;
    }
  }
  __syncthreads();
  // value sum: queries tq + 16a, dims tk*4 + 64g
  float o[4][NG][4];
#pragma unroll
  for (int a = 0; a < 4; a++)
#pragma unroll
    for (int g = 0; g < NG; g++)
#pragma unroll
      for (int i = 0; i < 4; i++) o[a][g][i] = 0.f;
  if (any) {
#pragma unroll 4
    for (int k = 0; k < CK_KEYS; k++) {
      float pv[4];
      float4 vv[NG];
#pragma unroll
      for (int a = 0; a < 4; a++) pv[a] = S.s[tq + 16 * a][k];
#pragma unroll
      for (int g = 0; g < NG; g++) vv[g] = *reinterpret_cast<const float4 *>(&S.v[k][tk * 4 + 64 * g]);
#pragma unroll
      for (int a = 0; a < 4; a++)
#pragma unroll
        for (int g = 0; g < NG; g++) {
          o[a][g][0] = fmaf(pv[a], vv[g].x, o[a][g][0]);
          o[a][g][1] = fmaf(pv[a], vv[g].y, o[a][g][1]);
          o[a][g][2] = fmaf(pv[a], vv[g].z, o[a][g][2]);
          o[a][g][3] = fmaf(pv[a], vv[g].w, o[a][g][3]);
        }
    }
  }
#pragma unroll
  for (int a = 0; a < 4; a++) {
    const int qi = tq + 16 * a, r = r_first + qi / REP, h = qi % REP;
    if (r >= T) continue;
    float *out = part + ((((size_t)r * d.nk + kh) * nkb + sb) * REP + h) * (HD + 2);
#pragma unroll
    for (int g = 0; g < NG; g++)
#pragma unroll
      for (int i = 0; i < 4; i++) out[tk * 4 + 64 * g + i] = o[a][g][i];
    if (tk == 0) {
      out[HD] = S.m[qi];
      out[HD + 1] = S.l[qi];
    }
  }
}

template <int HD, int REP>
cudaError_t chunk_t(const float *qkvg, int ldq, Dims d, Rows rows, Ring ring, int nkb, float *part, cudaStream_t s) {
  const size_t smem = sizeof(ChunkSmem<HD>);
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(attn_chunk_kernel<HD, REP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    attr = true;
  }
  constexpr int RG = CK_QUERIES / REP;
  const int nrg = (rows.n + RG - 1) / RG;
  attn_chunk_kernel<HD, REP><<<dim3(d.nk * nrg, nkb), CK_THREADS, smem, s>>>(qkvg, ldq, d, rows, ring, nkb, part);
  return cudaGetLastError();
}

}  // namespace

int attn_chunk_blocks(long window_keys, int rows) {
  return (int)((window_keys + rows - 1 + CK_KEYS - 1) / CK_KEYS) + 1;
}

cudaError_t launch_attention_chunk(const float *qkvg, int ldq, Dims d, Rows rows, Ring ring, int nkb, float *part,
                                   const float *sg, float *z, cudaStream_t s) {
  const int rep = d.nh / d.nk;
  cudaError_t e = cudaErrorInvalidValue;
#define CHUNK(H, R) \
  if (d.hd == H && rep == R) e = chunk_t<H, R>(qkvg, ldq, d, rows, ring, nkb, part, s);
  CHUNK(64, 1) CHUNK(64, 2) CHUNK(64, 4) CHUNK(64, 8)
  CHUNK(128, 1) CHUNK(128, 2) CHUNK(128, 4) CHUNK(128, 8)
#undef CHUNK
  if (e != cudaSuccess) return e;
  return launch_attention_combine(part, nkb, qkvg, ldq, d, rows, ring, sg, z, s);
}

}  // namespace dory
