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
// the same 4 x (hd/16) register tiling. Each block leaves per query its unnormalised output
// o[hd] and (max, sum). A second kernel, one block per row, merges the key blocks of every
// head (all partials requested at once), applies the output gate y * sigmoid(g * s_g^2),
// justnorms the row over nh * hd and writes it with its two bf16 halves for the O
// projection (dory.rs fn attn_layer).
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
    const size_t pi = (((size_t)r * d.nk + kh) * nkb + sb) * REP + h;  // partial index
    float *out = part + pi * HD;
#pragma unroll
    for (int g = 0; g < NG; g++)
      *reinterpret_cast<float4 *>(out + tk * 4 + 64 * g) = make_float4(o[a][g][0], o[a][g][1], o[a][g][2], o[a][g][3]);
    if (tk == 0)
      *reinterpret_cast<float2 *>(part + (size_t)T * d.nk * nkb * REP * HD + pi * 2) = make_float2(S.m[qi], S.l[qi]);
  }
}

__device__ __forceinline__ void emit4(const Emit &em, size_t i, float4 v) {
  if (!em.hi) return;
  const float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int u = 0; u < 4; u++) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x[u]);
    em.hi[i + u] = h;
    em.lo[i + u] = __float2bfloat16_rn(x[u] - __bfloat162float(h));
  }
}

// One block per row, thread i owns z[4i .. 4i+4) (head (4i)/hd).
template <int HD, int REP>
__global__ void attn_chunk_merge_kernel(const float *__restrict__ part, int nkb, const float *__restrict__ qkvg,
                                        int ldq, Dims d, const float *__restrict__ sg, float *__restrict__ z,
                                        Emit em) {
  constexpr int MB = 12;  // key blocks requested at once
  __shared__ float red[32];
  const int r = blockIdx.x, T = gridDim.x, i = threadIdx.x;
  const int hg = (4 * i) / HD, kh = hg / REP, h = hg % REP, dim = (4 * i) % HD;
  const float4 graw = *reinterpret_cast<const float4 *>(qkvg + (size_t)r * ldq + (size_t)(d.nh + 2 * d.nk) * HD + 4 * i);
  const float4 sgv = __ldg(reinterpret_cast<const float4 *>(sg + 4 * i));
  const size_t p0 = ((size_t)r * d.nk + kh) * nkb * REP + h;  // partial index of key block 0
  const float2 *ml = reinterpret_cast<const float2 *>(part + (size_t)T * d.nk * nkb * REP * HD);
  float M = -INFINITY, L = 0.f;
  float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int b0 = 0; b0 < nkb; b0 += MB) {
    float4 o[MB];
    float2 m[MB];
#pragma unroll
    for (int u = 0; u < MB; u++) {
      const bool in = b0 + u < nkb;
      const size_t pi = p0 + (size_t)(b0 + u) * REP;
      o[u] = in ? *reinterpret_cast<const float4 *>(part + pi * HD + dim) : make_float4(0.f, 0.f, 0.f, 0.f);
      m[u] = in ? ml[pi] : make_float2(-INFINITY, 0.f);
    }
#pragma unroll
    for (int u = 0; u < MB; u++) {
      if (m[u].x == -INFINITY) continue;
      const float nm = fmaxf(M, m[u].x);
      const float sa = M == -INFINITY ? 0.f : expf(M - nm), sb = expf(m[u].x - nm);
      L = L * sa + m[u].y * sb;
      A = make_float4(A.x * sa + o[u].x * sb, A.y * sa + o[u].y * sb, A.z * sa + o[u].z * sb, A.w * sa + o[u].w * sb);
      M = nm;
    }
  }
  const float inv_l = L > 0.f ? 1.f / L : 0.f;
  float4 y = make_float4(A.x * inv_l * sigmoidf_(graw.x * sgv.x), A.y * inv_l * sigmoidf_(graw.y * sgv.y),
                         A.z * inv_l * sigmoidf_(graw.z * sgv.z), A.w * inv_l * sigmoidf_(graw.w * sgv.w));
  const float ss = block_sum(y.x * y.x + y.y * y.y + y.z * y.z + y.w * y.w, red);
  const float inv = 1.f / sqrtf(ss + DORY_EPS);
  y = make_float4(y.x * inv, y.y * inv, y.z * inv, y.w * inv);
  const size_t zi = (size_t)r * d.nh * HD + 4 * i;
  *reinterpret_cast<float4 *>(z + zi) = y;
  emit4(em, zi, y);
}

template <int HD, int REP>
cudaError_t chunk_t(const float *qkvg, int ldq, Dims d, Rows rows, Ring ring, int nkb, float *part, const float *sg,
                    float *z, Emit em, cudaStream_t s) {
  const size_t smem = sizeof(ChunkSmem<HD>);
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(attn_chunk_kernel<HD, REP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    attr = true;
  }
  constexpr int RG = CK_QUERIES / REP;
  const int nrg = (rows.n + RG - 1) / RG;
  attn_chunk_kernel<HD, REP><<<dim3(d.nk * nrg, nkb), CK_THREADS, smem, s>>>(qkvg, ldq, d, rows, ring, nkb, part);
  attn_chunk_merge_kernel<HD, REP><<<rows.n, d.nh * HD / 4, 0, s>>>(part, nkb, qkvg, ldq, d, sg, z, em);
  return cudaGetLastError();
}

}  // namespace

int attn_chunk_blocks(long window_keys, int rows) {
  return (int)((window_keys + rows - 1 + CK_KEYS - 1) / CK_KEYS) + 1;
}

cudaError_t launch_attention_chunk(const float *qkvg, int ldq, Dims d, Rows rows, Ring ring, int nkb, float *part,
                                   const float *sg, float *z, Emit em, cudaStream_t s) {
  const int rep = d.nh / d.nk;
  if (d.nh * d.hd / 4 > 1024) return cudaErrorInvalidValue;  // one thread per 4 outputs of a row
#define CHUNK(H, R) \
  if (d.hd == H && rep == R) return chunk_t<H, R>(qkvg, ldq, d, rows, ring, nkb, part, sg, z, em, s);
  CHUNK(64, 1) CHUNK(64, 2) CHUNK(64, 4) CHUNK(64, 8)
  CHUNK(128, 1) CHUNK(128, 2) CHUNK(128, 4) CHUNK(128, 8)
#undef CHUNK
  return cudaErrorInvalidValue;
}

}  // namespace dory
