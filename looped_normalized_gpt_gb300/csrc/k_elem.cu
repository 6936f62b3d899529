// Row kernels of the Dory forward: embedding + RoPE table, the fused norm/RoPE/s_q^2
// prep with the f32 ring writer, row norms, the nGPT residual with the loop mix.
#include <algorithm>
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace dory {

static size_t align1k(size_t x) { return (x + 1023) & ~(size_t)1023; }

// Every sub-array starts on a 1024-byte boundary, so a ring row of hd f32 values sits at a
// whole row index of the KV memory seen as [rows][hd] (the attention's tensor map).
SlotLayout slot_layout(int cap, int nk, int hd, bool q8) {
  SlotLayout L = {};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align1k(o + bytes);
    return at;
  };
  const size_t rows = (size_t)nk * cap;
  L.tags = take((size_t)cap * 4);
  if (!q8) {
    L.k = take(rows * hd * 4);
    L.v = take(rows * hd * 4);
  } else {
    L.kq = take(rows * hd);
    L.ks = take(rows * (hd / 32) * 4);
    L.vq = take(rows * hd);
    L.vs = take(rows * 4);
    L.kcol = take((size_t)nk * hd * 4);
    L.vcol = take((size_t)nk * hd * 4);
    L.meta = take((size_t)nk * 4 * 4);
    L.wpos = take((size_t)nk * 64 * 4);
    L.wkq = take((size_t)nk * 64 * hd);
    L.wks = take((size_t)nk * 64 * (hd / 32) * 4);
    L.wvq = take((size_t)nk * 64 * hd);
    L.wvs = take((size_t)nk * 64 * 4);
  }
  L.bytes = o;
  return L;
}

namespace {

__device__ __forceinline__ void emit(const Emit &em, size_t i, float x) {
  if (em.hi) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    em.hi[i] = h;
    em.lo[i] = __float2bfloat16_rn(x - __bfloat162float(h));
  }
}

__device__ __forceinline__ void pdl_trigger_() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// h[r] = E[id] (zero for an id outside the vocabulary: dory.rs fn forward_host leaves the
// row at zero), and the row's RoPE table for both layer kinds: angle pos*inv[j] in f64,
// inv[j] = theta^(-2j/hd) rounded to f32, cos/sin stored as f32 (dory.rs fn stack).
template <typename WT>
__global__ void embed_rope_kernel(const int32_t *__restrict__ ids, const WT *__restrict__ E, Dims d, Rows rows,
                                  double theta_s, double theta_f, float *__restrict__ h,
                                  float *__restrict__ rope, Emit em) {
  const int r = blockIdx.x;
  const int id = h ? ids[r] : -1;
  float *hr = h ? h + (size_t)r * d.hidden : nullptr;
  if (!h) {
    // the RoPE table alone (rows that continue from saved hidden rows)
  } else if (id >= 0 && id < d.vocab) {
    const WT *er = E + (size_t)id * d.hidden;
    for (int i = threadIdx.x; i < d.hidden; i += blockDim.x) {
      const float x = load_w(er, i);
      hr[i] = x;
      emit(em, (size_t)r * d.hidden + i, x);
    }
  } else {
    for (int i = threadIdx.x; i < d.hidden; i += blockDim.x) {
      hr[i] = 0.f;
      emit(em, (size_t)r * d.hidden + i, 0.f);
    }
  }
  const int half = d.hd / 2;
  const long pos = (long)rows.seq_pos[rows.seq[r]] + rows.off[r];
  for (int i = threadIdx.x; i < 2 * half; i += blockDim.x) {
    const int kind = i / half, j = i % half;
    const double theta = kind == 0 ? theta_s : theta_f;
    const float inv = (float)pow((double)(float)theta, -2.0 * (double)j / (double)d.hd);
    double sn, cs;
    sincos((double)pos * (double)inv, &sn, &cs);
    float *t = rope + ((size_t)r * 2 + kind) * d.hd;
    t[j] = (float)cs;
    t[half + j] = (float)sn;
  }
}

// One block per (row, head): heads 0..nh-1 are queries, nh..nh+nk-1 keys. Rotate the
// pairs (j, j + hd/2) with a' = x cos - y sin, b' = y cos + x sin, justnorm the head,
// multiply queries by s_q^2 (dory.rs fn attn_layer). Keys and raw values go to the ring
// row pos mod cap (f32) or to the staging rows (q8, quantised by the q8 kernel).
__global__ void prep_kernel(float *__restrict__ qkvg, int ldq, Dims d, Rows rows, const float *__restrict__ rope,
                            int kind, const float *__restrict__ sq, Ring ring, float *__restrict__ kst,
                            float *__restrict__ vst) {
  __shared__ float red[32];
  pdl_trigger_();
  const int r = blockIdx.x, head = blockIdx.y;
  const int half = d.hd / 2;
  const bool is_q = head < d.nh;
  const int kh = head - d.nh;
  float *row = qkvg + (size_t)r * ldq + (is_q ? head * d.hd : d.nh * d.hd + kh * d.hd);
  const float *cs = rope + ((size_t)r * 2 + kind) * d.hd;
  const float *sn = cs + half;
  float a = 0.f, b = 0.f;
  const int j = threadIdx.x;
  if (j < half) {
    const float x = row[j], y = row[j + half];
    a = x * cs[j] - y * sn[j];
    b = y * cs[j] + x * sn[j];
  }
  const float ss = block_sum(a * a + b * b, red);
  const float inv = 1.f / sqrtf(ss + DORY_EPS);
  a *= inv;
  b *= inv;
  if (is_q) {
    if (j < half) {
      row[j] = a * sq[head * d.hd + j];
      row[j + half] = b * sq[head * d.hd + j + half];
    }
    return;
  }
  const float *vrow = qkvg + (size_t)r * ldq + d.nh * d.hd + d.nk * d.hd + kh * d.hd;
  if (ring.q8) {
    if (j < half) {
      float *ks = kst + ((size_t)r * d.nk + kh) * d.hd;
      float *vs = vst + ((size_t)r * d.nk + kh) * d.hd;
      ks[j] = a;
      ks[j + half] = b;
      vs[j] = vrow[j];
      vs[j + half] = vrow[j + half];
    }
    return;
  }
  const int seq = rows.seq[r];
  const long pos = (long)rows.seq_pos[seq] + rows.off[r];
  const int rr = (int)(pos % ring.cap);
  char *slot = ring.base + (size_t)seq * ring.seq_stride + ring.off;
  float *K = reinterpret_cast<float *>(slot + ring.L.k) + ((size_t)kh * ring.cap + rr) * d.hd;
  float *V = reinterpret_cast<float *>(slot + ring.L.v) + ((size_t)kh * ring.cap + rr) * d.hd;
  if (j < half) {
    K[j] = a;
    K[j + half] = b;
    V[j] = vrow[j];
    V[j + half] = vrow[j + half];
  }
  if (kh == 0 && j == 0) reinterpret_cast<int32_t *>(slot + ring.L.tags)[rr] = (int32_t)pos;
}

// x / sqrt(sum x^2 + eps) per row, in place (dory.rs fn justnorm).
// The row stays in registers between the sum of squares and the scaling (one read of x).
template <int MAXV>
__global__ void rownorm_kernel(float *__restrict__ x, int width, int ld, Emit em) {
  __shared__ float red[32];
  pdl_trigger_();
  float *row = x + (size_t)blockIdx.x * ld;
  float v[MAXV];
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < MAXV; j++) {
    const int i = threadIdx.x + j * blockDim.x;
    v[j] = i < width ? row[i] : 0.f;
    s += v[j] * v[j];
  }
  s = block_sum(s, red);
  const float inv = 1.f / sqrtf(s + DORY_EPS);
#pragma unroll
  for (int j = 0; j < MAXV; j++) {
    const int i = threadIdx.x + j * blockDim.x;
    if (i < width) {
      const float y = v[j] * inv;
      row[i] = y;
      emit(em, (size_t)blockIdx.x * width + i, y);
    }
  }
}

// The nGPT residual (dory.rs fn slerp) and the loop mix that follows the input block
// (MIX_BEGIN: input = state = x, h = (state + input)^), a recurrent pass that another
// follows (MIX_LOOP: state = x^, h = (state + input)^) or the last pass (MIX_END:
// h = state = x^). Without the residual the mix applies to h as it is.
template <int MAXV>
__global__ void residual_kernel(float *__restrict__ h, const float *__restrict__ out,
                                const float *__restrict__ alpha, int hidden, int mix, float *__restrict__ input,
                                float *__restrict__ state, int do_residual, Emit em) {
  __shared__ float red[64];
  pdl_trigger_();
  const int r = blockIdx.x;
  float *hr = h + (size_t)r * hidden;
  const float *orow = out + (size_t)r * hidden;
  float x[MAXV], o[MAXV], al[MAXV], ip[MAXV];  // every row the kernel reads, loaded at once
  const int nper = (hidden + blockDim.x - 1) / blockDim.x;
  float *in_r = input + (size_t)r * hidden, *st_r = state + (size_t)r * hidden;
  const bool read_in = mix == MIX_LOOP || mix == MIX_RESUME;
  float sx = 0.f, so = 0.f;
#pragma unroll
  for (int i = 0; i < MAXV; i++) {
    const int c = threadIdx.x + i * blockDim.x;
    x[i] = o[i] = al[i] = ip[i] = 0.f;
    if (i < nper && c < hidden) {
      x[i] = mix == MIX_RESUME ? st_r[c] : hr[c];
      if (do_residual) {
        o[i] = orow[c];
        al[i] = alpha[c];
      }
      if (read_in) ip[i] = in_r[c];
    }
  }
  if (do_residual) {
#pragma unroll
    for (int i = 0; i < MAXV; i++) {
      sx += x[i] * x[i];
      so += o[i] * o[i];
    }
    block_sum2(sx, so, red);
    const float ix = 1.f / sqrtf(sx + DORY_EPS), io = 1.f / sqrtf(so + DORY_EPS);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < MAXV; i++) {
      const int c = threadIdx.x + i * blockDim.x;
      if (i < nper && c < hidden) {
        const float xh = x[i] * ix, oh = o[i] * io;
        x[i] = xh + al[i] * (oh - xh);
        s += x[i] * x[i];
      }
    }
    s = block_sum(s, red);
    const float inv = 1.f / sqrtf(s + DORY_EPS);
#pragma unroll
    for (int i = 0; i < MAXV; i++) x[i] *= inv;
  }
  if (mix == MIX_LOOP || mix == MIX_END) {  // state = justnorm(h)
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < MAXV; i++) s += x[i] * x[i];
    s = block_sum(s, red);
    const float inv = 1.f / sqrtf(s + DORY_EPS);
#pragma unroll
    for (int i = 0; i < MAXV; i++) x[i] *= inv;
  }
  if (mix == MIX_BEGIN || mix == MIX_LOOP || mix == MIX_RESUME) {
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < MAXV; i++) {
      const int c = threadIdx.x + i * blockDim.x;
      if (i < nper && c < hidden) {
        float inp;
        if (mix == MIX_BEGIN) {
          inp = x[i];
          in_r[c] = inp;
        } else {
          inp = ip[i];
        }
        if (mix != MIX_RESUME) st_r[c] = x[i];
        x[i] = x[i] + inp;
        s += x[i] * x[i];
      }
    }
    s = block_sum(s, red);
    const float inv = 1.f / sqrtf(s + DORY_EPS);
#pragma unroll
    for (int i = 0; i < MAXV; i++) x[i] *= inv;
  } else if (mix == MIX_END) {
#pragma unroll
    for (int i = 0; i < MAXV; i++) {
      const int c = threadIdx.x + i * blockDim.x;
      if (i < nper && c < hidden) st_r[c] = x[i];
    }
  }
#pragma unroll
  for (int i = 0; i < MAXV; i++) {
    const int c = threadIdx.x + i * blockDim.x;
    if (i < nper && c < hidden) {
      hr[c] = x[i];
      emit(em, (size_t)r * hidden + c, x[i]);
    }
  }
}

__global__ void advance_kernel(int32_t *seq_pos, const int32_t *seq, const int32_t *count, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) seq_pos[seq[i]] += count[i];
}

// Synthetic rows [n][nk][hd] into an f32 ring at positions pos0.. (the append path of a
// forward writes the same bytes through prep_kernel).
__global__ void ring_write_f32_kernel(const float *__restrict__ k, const float *__restrict__ v, int n, int pos0,
                                      Dims d, Ring ring, int seq) {
  const int r = blockIdx.x, kh = blockIdx.y;
  const long pos = (long)pos0 + r;
  const int rr = (int)(pos % ring.cap);
  char *slot = ring.base + (size_t)seq * ring.seq_stride + ring.off;
  float *K = reinterpret_cast<float *>(slot + ring.L.k) + ((size_t)kh * ring.cap + rr) * d.hd;
  float *V = reinterpret_cast<float *>(slot + ring.L.v) + ((size_t)kh * ring.cap + rr) * d.hd;
  const float *ks = k + ((size_t)r * d.nk + kh) * d.hd;
  const float *vs = v + ((size_t)r * d.nk + kh) * d.hd;
  for (int j = threadIdx.x; j < d.hd; j += blockDim.x) {
    K[j] = ks[j];
    V[j] = vs[j];
  }
  if (kh == 0 && threadIdx.x == 0) reinterpret_cast<int32_t *>(slot + ring.L.tags)[rr] = (int32_t)pos;
}

// Rollback of one sequence to position n (dory.rs DoryState::rollback; kv_cache.rs
// fn truncate_last on q8 rings): one block per slot of the sequence. Every ring row whose tag
// is a position >= n becomes empty (-1); the count of such rows is what the slot drops, and a
// q8 slot's stored-row counters (one per kv head) go down by it. The frozen flag and fields
// stay as they are. Rows still to be dropped are all in the ring: a rollback never reaches
// further back than a ring holds (the host checks it).
__global__ void rollback_kernel(char *seq_block, const long long *table, int n, int nk, int q8, int32_t *dropped) {
  __shared__ int red[32];
  const long long *t = table + 3 * blockIdx.x;  // tags offset, meta offset, rows
  int32_t *tags = reinterpret_cast<int32_t *>(seq_block + t[0]);
  const int cap = (int)t[2];
  int cnt = 0;
  for (int r = threadIdx.x; r < cap; r += blockDim.x)
    if (tags[r] >= n) {
      tags[r] = -1;
      cnt++;
    }
  cnt = __reduce_add_sync(0xffffffffu, cnt);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = cnt;
  __syncthreads();
  if (threadIdx.x == 0) {
    int total = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); w++) total += red[w];
    dropped[blockIdx.x] = total;
    if (q8) {
      int32_t *meta = reinterpret_cast<int32_t *>(seq_block + t[1]);
      for (int kh = 0; kh < nk; kh++) meta[kh * 4 + 0] -= total;
    }
  }
}

// dory.rs fn top_prob on one row of logits: the largest softmax probability, from the
// entries within 20 of the top only. top = max (f32); den = sum of exp(x - top) over the x
// with x - top > -20, the difference taken in f32, exp and sum in f64; 1 / den as f32.
__global__ void top_prob_kernel(const float *__restrict__ lg, int n, float *out) {
  __shared__ float red[32];
  __shared__ double dred[32];
  float m = -INFINITY;
  for (int i = threadIdx.x; i < n; i += blockDim.x) m = fmaxf(m, lg[i]);
  m = block_max(m, red);
  double den = 0.0;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const float t = __fsub_rn(lg[i], m);
    if (t > -20.f) den += exp((double)t);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  if (lane == 0) dred[warp] = den;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int w = 0; w < nw; w++) t += dred[w];
    *out = (float)(1.0 / t);
  }
}

// Rows of a step in another order: ids_out[r] = ids[perm[r]] (the token ids in the step's
// row order), and dst[perm[r]] = src[r] for rows of `width` floats (results back in the
// caller's order).
__global__ void gather_ids_kernel(const int32_t *__restrict__ ids, const int32_t *__restrict__ perm, int n,
                                  int32_t *__restrict__ out) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r < n) out[r] = ids[perm[r]];
}

__global__ void scatter_rows_kernel(const float *__restrict__ src, float *__restrict__ dst,
                                    const int32_t *__restrict__ perm, int width) {
  const int r = blockIdx.y;
  const float4 *s4 = reinterpret_cast<const float4 *>(src + (size_t)r * width);
  float4 *d4 = reinterpret_cast<float4 *>(dst + (size_t)perm[r] * width);
  for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < width / 4; c += gridDim.x * blockDim.x) d4[c] = s4[c];
}

// dst[j][.] = src[idx[j]][.] for `rows` rows of `width` floats.
__global__ void gather_rows_kernel(const float *__restrict__ src, float *__restrict__ dst,
                                   const int32_t *__restrict__ idx, int width) {
  const int j = blockIdx.y;
  const float4 *s4 = reinterpret_cast<const float4 *>(src + (size_t)idx[j] * width);
  float4 *d4 = reinterpret_cast<float4 *>(dst + (size_t)j * width);
  for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < width / 4; c += gridDim.x * blockDim.x) d4[c] = s4[c];
}

}  // namespace

cudaError_t launch_gather_rows(const float *src, float *dst, const int32_t *idx, int rows, int width,
                               cudaStream_t s) {
  if (width % 4) return cudaErrorInvalidValue;
  const int per_row = std::min(64, (width / 4 + 255) / 256);
  gather_rows_kernel<<<dim3(per_row, rows), 256, 0, s>>>(src, dst, idx, width);
  return cudaGetLastError();
}

cudaError_t launch_gather_ids(const int32_t *ids, const int32_t *perm, int n, int32_t *out, cudaStream_t s) {
  gather_ids_kernel<<<(n + 127) / 128, 128, 0, s>>>(ids, perm, n, out);
  return cudaGetLastError();
}

cudaError_t launch_scatter_rows(const float *src, float *dst, const int32_t *perm, int rows, int width,
                                cudaStream_t s) {
  if (width % 4) return cudaErrorInvalidValue;
  const int per_row = std::min(64, (width / 4 + 255) / 256);
  scatter_rows_kernel<<<dim3(per_row, rows), 256, 0, s>>>(src, dst, perm, width);
  return cudaGetLastError();
}

cudaError_t launch_top_prob(const float *logits, int n, float *out, cudaStream_t s) {
  top_prob_kernel<<<1, 1024, 0, s>>>(logits, n, out);
  return cudaGetLastError();
}

cudaError_t launch_rollback(char *seq_block, const long long *table, int nslots, int n, int nk, int q8,
                            int32_t *dropped, cudaStream_t s) {
  rollback_kernel<<<nslots, 256, 0, s>>>(seq_block, table, n, nk, q8, dropped);
  return cudaGetLastError();
}

cudaError_t launch_embed_rope(const int32_t *ids, const void *E, int wdtype, Dims d, Rows rows, double theta_s,
                              double theta_f, float *h, float *rope, Emit em, cudaStream_t s) {
  if (wdtype == W_BF16)
    embed_rope_kernel<__nv_bfloat16><<<rows.n, 256, 0, s>>>(ids, static_cast<const __nv_bfloat16 *>(E), d, rows,
                                                             theta_s, theta_f, h, rope, em);
  else
    embed_rope_kernel<float><<<rows.n, 256, 0, s>>>(ids, static_cast<const float *>(E), d, rows, theta_s, theta_f,
                                                     h, rope, em);
  return cudaGetLastError();
}

cudaError_t launch_prep(float *qkvg, int ldq, Dims d, Rows rows, const float *rope, int kind, const float *sq,
                        Ring ring, float *kst, float *vst, cudaStream_t s) {
  dim3 grid(rows.n, d.nh + d.nk);
  const int threads = ((d.hd / 2 + 31) / 32) * 32;
  prep_kernel<<<grid, threads, 0, s>>>(qkvg, ldq, d, rows, rope, kind, sq, ring, kst, vst);
  return cudaGetLastError();
}

cudaError_t launch_rownorm(float *x, int T, int width, int ld, Emit em, cudaStream_t s) {
  const int per = (width + 511) / 512;
  if (per <= 4) rownorm_kernel<4><<<T, 512, 0, s>>>(x, width, ld, em);
  else if (per <= 16) rownorm_kernel<16><<<T, 512, 0, s>>>(x, width, ld, em);
  else if (per <= 64) rownorm_kernel<64><<<T, 512, 0, s>>>(x, width, ld, em);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_residual(float *h, const float *out, const float *alpha, int T, int hidden, int mix, float *input,
                            float *state, int do_residual, Emit em, cudaStream_t s) {
  const int threads = 512;
  const int nper = (hidden + threads - 1) / threads;
  if (nper <= 4)
    residual_kernel<4><<<T, threads, 0, s>>>(h, out, alpha, hidden, mix, input, state, do_residual, em);
  else if (nper <= 16)
    residual_kernel<16><<<T, threads, 0, s>>>(h, out, alpha, hidden, mix, input, state, do_residual, em);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_advance(int32_t *seq_pos, const int32_t *seq, const int32_t *count, int n, cudaStream_t s) {
  advance_kernel<<<(n + 127) / 128, 128, 0, s>>>(seq_pos, seq, count, n);
  return cudaGetLastError();
}

cudaError_t launch_ring_write_f32(const float *k, const float *v, int n, int pos0, Dims d, Ring ring, int seq,
                                  cudaStream_t s) {
  dim3 grid(n, d.nk);
  ring_write_f32_kernel<<<grid, 128, 0, s>>>(k, v, n, pos0, d, ring, seq);
  return cudaGetLastError();
}

}  // namespace dory
