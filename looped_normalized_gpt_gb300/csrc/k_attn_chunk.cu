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
#include <cstdlib>

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

// ---- the same partials on the tensor cores (tcgen05, TMEM) ----------------------------
//
// One block per (kv head, tile of 128 query vectors, block of 64 key positions), 128 threads;
// a thread is one query (one TMEM lane). Q, the key block and the value block are split into
// bf16 halves (x = hi + lo, hi = bf16(x), lo = bf16(x - hi)) and written to shared memory in
// the MMA's K-major layout with 128-byte swizzle (V transposed: its K side is the keys).
// S = Q K^T is three MMAs per K step of 16 (hi.hi + hi.lo + lo.hi: the products keep about
// 16 mantissa bits, the sums f32 in TMEM); each thread reads its query's 64 scores, masks
// them (window and tag), and leaves exp(s - m), split into halves, as the A operand of
// O = P V (three MMAs per K step again). The block writes the same unnormalised output and
// (max, sum) per query as attn_chunk_kernel, for the same merge kernel.
constexpr int CT_Q = 128;      // query vectors per block (MMA M)
constexpr int CT_THREADS = 128;

__device__ __forceinline__ uint32_t ct_smem(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Byte offset of element (row, k) of a K-major bf16 tile whose K side is cut into atoms of 64
// elements ([rows][64] each, 128 bytes a row, 16-byte chunks swizzled by row mod 8).
__device__ __forceinline__ uint32_t ct_off(int row, int k, int rows) {
  const int atom = k >> 6, kk = k & 63;
  return (uint32_t)(atom * rows * 128 + row * 128 + ((((kk >> 3) ^ (row & 7))) << 4) + ((kk & 7) << 1));
}

__device__ __forceinline__ uint64_t ct_desc(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFF) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;  // 8 rows x 128 B
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;            // 128-byte swizzle
  return d;
}

__host__ __device__ constexpr uint32_t ct_idesc(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void ct_mma(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ bool ct_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < (1u << 20); i++) {
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

__device__ __forceinline__ void ct_ld16(uint32_t taddr, float *v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void ct_split(float x, __nv_bfloat16 &h, __nv_bfloat16 &l) {
  h = __float2bfloat16_rn(x);
  l = __float2bfloat16_rn(x - __bfloat162float(h));
}

template <int HD>
struct CtSmem {
  static constexpr int Q = CT_Q * HD * 2;   // one half of Q
  static constexpr int K = CK_KEYS * HD * 2;
  static constexpr int V = HD * CK_KEYS * 2;
  static constexpr int P = CT_Q * CK_KEYS * 2;
  static constexpr int QH = 0, QL = QH + Q, KH = QL + Q, KL = KH + K, VH = KL + K, VL = VH + V, PH = VL + V,
                       PL = PH + P, VF = PH;  // the f32 value block, staged where P goes later
  static constexpr int BYTES = PL + P > VF + CK_KEYS * HD * 4 ? PL + P : VF + CK_KEYS * HD * 4;
  static constexpr int TOTAL = BYTES + 1024;
};

template <int HD, int REP>
__global__ void __launch_bounds__(CT_THREADS, 1)
    attn_chunk_tc_kernel(const float *__restrict__ qkvg, int ldq, Dims d, Rows rows, Ring ring, int nkb,
                         float *__restrict__ part, int *__restrict__ err) {
  using L = CtSmem<HD>;
  constexpr int RGT = CT_Q / REP;  // rows per query tile
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_sh;
  __shared__ int32_t tag[CK_KEYS];
  const int T = rows.n;
  const int nrg = (T + RGT - 1) / RGT;
  const int kh = blockIdx.x / nrg, rg = blockIdx.x % nrg, sb = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seq = rows.seq[0];
  const long p0 = (long)rows.seq_pos[seq] + rows.off[0];
  const long lo0 = ring.window == INT_MAX ? 0 : (p0 + 1 - ring.window > 0 ? p0 + 1 - ring.window : 0);
  const long P0 = (lo0 / CK_KEYS + sb) * CK_KEYS;
  const int r_first = rg * RGT, r_end = min(T, r_first + RGT);
  const long p_last = p0 + r_end - 1;
  const long lo_first = ring.window == INT_MAX ? 0 : max(p0 + r_first + 1 - (long)ring.window, 0L);
  const bool any = P0 <= p_last && P0 + CK_KEYS - 1 >= lo_first;
  // this thread's query: row r, head h of the kv head's group
  const int qi = tid, r = r_first + qi / REP, h = qi % REP;
  if (!any) {  // no key of the block is in a window of the tile's rows
    if (r < T) {
      const size_t pi = (((size_t)r * d.nk + kh) * nkb + sb) * REP + h;
      float *out = part + pi * HD;
      for (int i = 0; i < HD; i += 4) *reinterpret_cast<float4 *>(out + i) = make_float4(0.f, 0.f, 0.f, 0.f);
      *reinterpret_cast<float2 *>(part + (size_t)T * d.nk * nkb * REP * HD + pi * 2) = make_float2(-INFINITY, 0.f);
    }
    return;
  }
  const uint32_t base = (ct_smem(smem_raw) + 1023) & ~1023u;
  uint8_t *sm = smem_raw + (base - ct_smem(smem_raw));
  const char *slot = ring.base + (size_t)seq * ring.seq_stride + ring.off;
  const int rr0 = (int)(P0 % ring.cap);
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(ct_smem(&bar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;" ::"r"(ct_smem(&tmem_sh))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // operands into shared memory, split into bf16 halves; loads go out UL at a time per thread
  // (one L2 round trip for UL float4s instead of one each)
  constexpr int NC = HD / 4, UL = 8;
  auto put = [&](uint32_t hoff, uint32_t loff, uint32_t o, const float4 &x) {
    __nv_bfloat16 hv[4], lv[4];
    ct_split(x.x, hv[0], lv[0]);
    ct_split(x.y, hv[1], lv[1]);
    ct_split(x.z, hv[2], lv[2]);
    ct_split(x.w, hv[3], lv[3]);
    *reinterpret_cast<uint2 *>(sm + hoff + o) = *reinterpret_cast<const uint2 *>(hv);
    *reinterpret_cast<uint2 *>(sm + loff + o) = *reinterpret_cast<const uint2 *>(lv);
  };
  static_assert((CT_Q * NC) % (CT_THREADS * UL) == 0 && (CK_KEYS * NC) % (CT_THREADS * UL) == 0, "whole rounds");
  for (int i0 = tid; i0 < CT_Q * NC; i0 += CT_THREADS * UL) {
    float4 x[UL];
#pragma unroll
    for (int u = 0; u < UL; u++) {
      const int i = i0 + u * CT_THREADS, q = i / NC, c = i % NC, rq = r_first + q / REP, hq = q % REP;
      x[u] = rq < T ? *reinterpret_cast<const float4 *>(qkvg + (size_t)rq * ldq + (size_t)(kh * REP + hq) * HD + c * 4)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < UL; u++) {
      const int i = i0 + u * CT_THREADS, q = i / NC, c = i % NC;
      put(L::QH, L::QL, ct_off(q, c * 4, CT_Q), x[u]);
    }
  }
  const float4 *kg = reinterpret_cast<const float4 *>(slot + ring.L.k) + ((size_t)kh * ring.cap + rr0) * NC;
  const float4 *vg = reinterpret_cast<const float4 *>(slot + ring.L.v) + ((size_t)kh * ring.cap + rr0) * NC;
  float *vf = reinterpret_cast<float *>(sm + L::VF);
  for (int i0 = tid; i0 < CK_KEYS * NC; i0 += CT_THREADS * UL) {
    float4 x[UL], y[UL];
#pragma unroll
    for (int u = 0; u < UL; u++) {
      x[u] = kg[i0 + u * CT_THREADS];
      y[u] = vg[i0 + u * CT_THREADS];
    }
#pragma unroll
    for (int u = 0; u < UL; u++) {
      const int i = i0 + u * CT_THREADS, j = i / NC, c = i % NC;
      put(L::KH, L::KL, ct_off(j, c * 4, CK_KEYS), x[u]);
      *reinterpret_cast<float4 *>(vf + (size_t)j * HD + c * 4) = y[u];
    }
  }
  if (tid < CK_KEYS) tag[tid] = reinterpret_cast<const int32_t *>(slot + ring.L.tags)[rr0 + tid];
  __syncthreads();
  // V transposed: row = dimension, K side = the 64 keys; a thread writes 8 keys of one dimension
  for (int i = tid; i < HD * (CK_KEYS / 8); i += CT_THREADS) {
    const int dm = i / (CK_KEYS / 8), j0 = (i % (CK_KEYS / 8)) * 8;
    __nv_bfloat16 hv[8], lv[8];
#pragma unroll
    for (int u = 0; u < 8; u++) ct_split(vf[(size_t)(j0 + u) * HD + dm], hv[u], lv[u]);
    const uint32_t o = ct_off(dm, j0, HD);
    *reinterpret_cast<uint4 *>(sm + L::VH + o) = *reinterpret_cast<const uint4 *>(hv);
    *reinterpret_cast<uint4 *>(sm + L::VL + o) = *reinterpret_cast<const uint4 *>(lv);
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> the MMA's reads
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_sh;
  const uint32_t t_s = tmem, t_o = tmem + 128;  // S: 64 columns, O: HD columns
  bool ok = true;
  if (tid == 0) {
    constexpr uint32_t id_s = ct_idesc(CT_Q, CK_KEYS);
#pragma unroll
    for (int kk = 0; kk < HD / 16; kk++) {
      const uint32_t step = (uint32_t)((kk & 3) * 32);  // K offset within a 64-element atom
      const uint32_t qa = (uint32_t)((kk >> 2) * CT_Q * 128) + step, ka = (uint32_t)((kk >> 2) * CK_KEYS * 128) + step;
      ct_mma(t_s, ct_desc(base + L::QH + qa), ct_desc(base + L::KH + ka), id_s, kk > 0 ? 1u : 0u);
      ct_mma(t_s, ct_desc(base + L::QH + qa), ct_desc(base + L::KL + ka), id_s, 1u);
      ct_mma(t_s, ct_desc(base + L::QL + qa), ct_desc(base + L::KH + ka), id_s, 1u);
    }
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(ct_smem(&bar))
                 : "memory");
  }
  __syncwarp();
  ok = ct_wait(ct_smem(&bar), 0);
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  // this query's scores: mask, softmax statistics, exp(s - m) as the A operand of P V
  const long p = p0 + r;
  const long lo = ring.window == INT_MAX ? 0 : (p + 1 - ring.window > 0 ? p + 1 - ring.window : 0);
  const float scale = 1.f / sqrtf((float)HD);
  float sc[CK_KEYS];
#pragma unroll
  for (int c0 = 0; c0 < CK_KEYS; c0 += 16) ct_ld16(t_s + ((uint32_t)(warp * 32) << 16) + c0, sc + c0);
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < CK_KEYS; j++) {
    const long pk = P0 + j;
    const bool valid = ok && r < T && pk >= lo && pk <= p && tag[j] == (int32_t)pk;
    sc[j] = valid ? sc[j] * scale : -INFINITY;
    m = fmaxf(m, sc[j]);
  }
  float l = 0.f;
#pragma unroll
  for (int j = 0; j < CK_KEYS; j += 8) {
    __nv_bfloat16 hv[8], lv[8];
#pragma unroll
    for (int u = 0; u < 8; u++) {
      const float e = m == -INFINITY ? 0.f : expf(sc[j + u] - m);
      l += e;
      ct_split(e, hv[u], lv[u]);
    }
    const uint32_t o = ct_off(qi, j, CT_Q);
    *reinterpret_cast<uint4 *>(sm + L::PH + o) = *reinterpret_cast<const uint4 *>(hv);
    *reinterpret_cast<uint4 *>(sm + L::PL + o) = *reinterpret_cast<const uint4 *>(lv);
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (tid == 0 && ok) {
    constexpr uint32_t id_o = ct_idesc(CT_Q, HD);
#pragma unroll
    for (int kk = 0; kk < CK_KEYS / 16; kk++) {
      const uint32_t step = (uint32_t)(kk * 32);
      ct_mma(t_o, ct_desc(base + L::PH + step), ct_desc(base + L::VH + step), id_o, kk > 0 ? 1u : 0u);
      ct_mma(t_o, ct_desc(base + L::PH + step), ct_desc(base + L::VL + step), id_o, 1u);
      ct_mma(t_o, ct_desc(base + L::PL + step), ct_desc(base + L::VH + step), id_o, 1u);
    }
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(ct_smem(&bar))
                 : "memory");
  }
  __syncwarp();
  const bool ok2 = ok && ct_wait(ct_smem(&bar), 1);
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (!ok2 && tid == 0) atomicExch(err, 21);
  // every lane takes part in the warp's TMEM loads; lanes of rows past the step store nothing
  const size_t pi = (((size_t)r * d.nk + kh) * nkb + sb) * REP + h;
  float *out = part + pi * HD;
#pragma unroll
  for (int c0 = 0; c0 < HD; c0 += 16) {
    float v[16];
    ct_ld16(t_o + ((uint32_t)(warp * 32) << 16) + c0, v);
    if (r < T) {
#pragma unroll
      for (int u = 0; u < 16; u += 4)
        *reinterpret_cast<float4 *>(out + c0 + u) =
            ok2 ? make_float4(v[u], v[u + 1], v[u + 2], v[u + 3]) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  if (r < T)
    *reinterpret_cast<float2 *>(part + (size_t)T * d.nk * nkb * REP * HD + pi * 2) =
        ok2 ? make_float2(m, l) : make_float2(-INFINITY, 0.f);
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;" ::"r"(tmem) : "memory");
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

// DORY_CHUNK_TC=0: the partials on the f32 pipe (attn_chunk_kernel) instead of the tensor cores
bool chunk_tc_on() {
  static const bool on = [] {
    const char *e = getenv("DORY_CHUNK_TC");
    return !(e && e[0] == '0');
  }();
  return on;
}

template <int HD, int REP>
cudaError_t chunk_t(const float *qkvg, int ldq, Dims d, Rows rows, Ring ring, int nkb, float *part, const float *sg,
                    float *z, Emit em, int *err, cudaStream_t s) {
  if (chunk_tc_on()) {
    using L = CtSmem<HD>;
    static bool attr_tc = false;
    if (!attr_tc) {
      cudaFuncSetAttribute(attn_chunk_tc_kernel<HD, REP>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
      attr_tc = true;
    }
    constexpr int RGT = CT_Q / REP;
    const int nrg = (rows.n + RGT - 1) / RGT;
    attn_chunk_tc_kernel<HD, REP><<<dim3(d.nk * nrg, nkb), CT_THREADS, L::TOTAL, s>>>(qkvg, ldq, d, rows, ring, nkb,
                                                                                     part, err);
    attn_chunk_merge_kernel<HD, REP><<<rows.n, d.nh * HD / 4, 0, s>>>(part, nkb, qkvg, ldq, d, sg, z, em);
    return cudaGetLastError();
  }
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
                                   const float *sg, float *z, Emit em, int *err, cudaStream_t s) {
  const int rep = d.nh / d.nk;
  if (d.nh * d.hd / 4 > 1024) return cudaErrorInvalidValue;  // one thread per 4 outputs of a row
#define CHUNK(H, R) \
  if (d.hd == H && rep == R) return chunk_t<H, R>(qkvg, ldq, d, rows, ring, nkb, part, sg, z, em, err, s);
  CHUNK(64, 1) CHUNK(64, 2) CHUNK(64, 4) CHUNK(64, 8)
  CHUNK(128, 1) CHUNK(128, 2) CHUNK(128, 4) CHUNK(128, 8)
#undef CHUNK
  return cudaErrorInvalidValue;
}

}  // namespace dory
