// q8_2f KV append (kv_cache.rs fn append, fn quant_row, fn freeze_cols).
//
// One block per (sequence, kv head), one thread per channel; the rows of the sequence
// are appended in order. A row is quantised against the per-channel field (1 until it
// is frozen): r = x / col, one scale per 32 channels for K and one per row for V,
// s = max(absmax / 127, 1e-12), q = clamp(round_half_away(r / s), -127, 127). At the
// first append that finds 64 stored rows the field is frozen: the stored rows are
// dequantised (x = q s), col[d] = max(sqrt(sum_p x_pd^2 / n), 1e-6) with the sum taken
// sequentially in row order, and every stored row is quantised again against col.
// All of it in float32 with IEEE-rounded operations and no contraction (__f*_rn), so
// codes and scales match the reference bit for bit on identical input rows.
//
// The first 64 appended rows of a slot are also kept in a side buffer so that the freeze
// sees every stored row even if a per_loop slot with holes has spread them over more
// positions than its ring holds.
#include "common.cuh"
#include "kernels.h"

namespace dory {

namespace {

constexpr int WARM = 64;  // kv_cache.rs, const KV_COL_WARMUP

struct Q8Slot {
  int32_t *tags, *meta, *wpos;
  int8_t *kq, *vq, *wkq, *wvq;
  float *ks, *vs, *kcol, *vcol, *wks, *wvs;
};

__device__ __forceinline__ Q8Slot q8_slot(const Ring &ring, int seq) {
  char *s = ring.base + (size_t)seq * ring.seq_stride + ring.off;
  Q8Slot q;
  q.tags = reinterpret_cast<int32_t *>(s + ring.L.tags);
  q.meta = reinterpret_cast<int32_t *>(s + ring.L.meta);
  q.wpos = reinterpret_cast<int32_t *>(s + ring.L.wpos);
  q.kq = reinterpret_cast<int8_t *>(s + ring.L.kq);
  q.vq = reinterpret_cast<int8_t *>(s + ring.L.vq);
  q.wkq = reinterpret_cast<int8_t *>(s + ring.L.wkq);
  q.wvq = reinterpret_cast<int8_t *>(s + ring.L.wvq);
  q.ks = reinterpret_cast<float *>(s + ring.L.ks);
  q.vs = reinterpret_cast<float *>(s + ring.L.vs);
  q.kcol = reinterpret_cast<float *>(s + ring.L.kcol);
  q.vcol = reinterpret_cast<float *>(s + ring.L.vcol);
  q.wks = reinterpret_cast<float *>(s + ring.L.wks);
  q.wvs = reinterpret_cast<float *>(s + ring.L.wvs);
  return q;
}

// Quantise one channel value; the group is a warp (32 channels) or the whole block.
__device__ __forceinline__ int8_t quant_warp(float r, float *scale_out) {
  const float amax = warp_max(fabsf(r));
  const float s = fmaxf(__fdiv_rn(amax, 127.f), 1e-12f);
  *scale_out = s;
  float q = roundf(__fdiv_rn(r, s));  // roundf: half away from zero
  q = fminf(fmaxf(q, -127.f), 127.f);
  return (int8_t)q;
}

__device__ __forceinline__ int8_t quant_block(float r, float *red, float *scale_out) {
  const float amax = block_max(fabsf(r), red);
  const float s = fmaxf(__fdiv_rn(amax, 127.f), 1e-12f);
  *scale_out = s;
  float q = roundf(__fdiv_rn(r, s));
  q = fminf(fmaxf(q, -127.f), 127.f);
  return (int8_t)q;
}

// Quantise channel d of a K and a V row against the field (if frozen) and store them.
__device__ void put_row(const Q8Slot &q, int kh, int hd, int cap, long pos, float kx, float vx, bool frozen,
                        int warm_at, float *red) {
  const int d = threadIdx.x;
  const float kr = frozen ? __fdiv_rn(kx, q.kcol[kh * hd + d]) : kx;
  const float vr = frozen ? __fdiv_rn(vx, q.vcol[kh * hd + d]) : vx;
  float ksc, vsc;
  const int8_t kc = quant_warp(kr, &ksc);
  const int8_t vc = quant_block(vr, red, &vsc);
  const int rr = (int)(pos % cap);
  const size_t row = (size_t)kh * cap + rr;
  q.kq[row * hd + d] = kc;
  q.vq[row * hd + d] = vc;
  if ((d & 31) == 0) q.ks[row * (hd / 32) + d / 32] = ksc;
  if (d == 0) {
    q.vs[row] = vsc;
    if (kh == 0) q.tags[rr] = (int32_t)pos;
  }
  if (warm_at >= 0) {
    const size_t w = (size_t)kh * WARM + warm_at;
    q.wkq[w * hd + d] = kc;
    q.wvq[w * hd + d] = vc;
    if ((d & 31) == 0) q.wks[w * (hd / 32) + d / 32] = ksc;
    if (d == 0) {
      q.wvs[w] = vsc;
      q.wpos[w] = (int32_t)pos;
    }
  }
}

// kv_cache.rs fn freeze_cols for one head over the n stored rows (kept in the side buffer).
__device__ void freeze(const Q8Slot &q, int kh, int hd, int cap, int n, float *red) {
  const int d = threadIdx.x;
  float sk = 0.f, sv = 0.f;
  for (int i = 0; i < n; i++) {
    const size_t w = (size_t)kh * WARM + i;
    const float xk = __fmul_rn((float)q.wkq[w * hd + d], q.wks[w * (hd / 32) + d / 32]);
    const float xv = __fmul_rn((float)q.wvq[w * hd + d], q.wvs[w]);
    sk = __fadd_rn(sk, __fmul_rn(xk, xk));
    sv = __fadd_rn(sv, __fmul_rn(xv, xv));
  }
  const float nf = (float)n;
  const float ck = fmaxf(__fsqrt_rn(__fdiv_rn(sk, nf)), 1e-6f);
  const float cv = fmaxf(__fsqrt_rn(__fdiv_rn(sv, nf)), 1e-6f);
  q.kcol[kh * hd + d] = ck;
  q.vcol[kh * hd + d] = cv;
  __syncthreads();
  for (int i = 0; i < n; i++) {
    const size_t w = (size_t)kh * WARM + i;
    const float xk = __fmul_rn((float)q.wkq[w * hd + d], q.wks[w * (hd / 32) + d / 32]);
    const float xv = __fmul_rn((float)q.wvq[w * hd + d], q.wvs[w]);
    const long pos = q.wpos[w];
    const int rr = (int)(pos % cap);
    const bool held = q.tags[rr] == (int32_t)pos;
    __syncthreads();  // every thread has read the tag before a rewrite of this row
    float ksc, vsc;
    const int8_t kc = quant_warp(__fdiv_rn(xk, ck), &ksc);
    const int8_t vc = quant_block(__fdiv_rn(xv, cv), red, &vsc);
    if (held) {
      const size_t row = (size_t)kh * cap + rr;
      q.kq[row * hd + d] = kc;
      q.vq[row * hd + d] = vc;
      if ((d & 31) == 0) q.ks[row * (hd / 32) + d / 32] = ksc;
      if (d == 0) q.vs[row] = vsc;
    }
  }
  if (d == 0) q.meta[kh * 4 + 1] = 1;
  __syncthreads();
}

__device__ __forceinline__ long row_pos(const Rows &rows, int r) {
  return (long)rows.seq_pos[rows.seq[r]] + rows.off[r];
}

// Sequential append of a run of rows of one sequence (blockDim = hd).
__global__ void q8_append_kernel(const float *__restrict__ kst, const float *__restrict__ vst, Dims d, Rows rows,
                                 Ring ring, int rewrite) {
  __shared__ float red[32];
  const int r0 = blockIdx.x, kh = blockIdx.y;
  const int seq = rows.seq[r0];
  if (r0 > 0 && rows.seq[r0 - 1] == seq) return;  // not the first row of its run
  int run = 1;
  while (r0 + run < rows.n && rows.seq[r0 + run] == seq) run++;
  const Q8Slot q = q8_slot(ring, seq);
  const int hd = d.hd, dch = threadIdx.x;
  int count = q.meta[kh * 4 + 0];
  int frozen = q.meta[kh * 4 + 1];
  __syncthreads();
  for (int i = 0; i < run; i++) {
    const int r = r0 + i;
    const int stored = rewrite ? count - run + i : count;
    if (stored >= WARM && !frozen) {
      freeze(q, kh, hd, ring.cap, WARM, red);
      frozen = 1;
    }
    const float kx = kst[((size_t)r * d.nk + kh) * hd + dch];
    const float vx = vst[((size_t)r * d.nk + kh) * hd + dch];
    put_row(q, kh, hd, ring.cap, row_pos(rows, r), kx, vx, frozen, stored < WARM ? stored : -1, red);
    if (!rewrite) count++;
    __syncthreads();
  }
  if (dch == 0) q.meta[kh * 4 + 0] = count;
}

// Rows of one sequence appended to a slot whose field is already frozen: independent rows.
__global__ void q8_append_frozen_kernel(const float *__restrict__ kst, const float *__restrict__ vst, Dims d,
                                        int seq, long pos0, Ring ring) {
  __shared__ float red[32];
  const int r = blockIdx.x, kh = blockIdx.y;
  const Q8Slot q = q8_slot(ring, seq);
  const int hd = d.hd, dch = threadIdx.x;
  const float kx = kst[((size_t)r * d.nk + kh) * hd + dch];
  const float vx = vst[((size_t)r * d.nk + kh) * hd + dch];
  put_row(q, kh, hd, ring.cap, pos0 + r, kx, vx, true, -1, red);
}

__global__ void q8_add_count_kernel(Ring ring, int seq, int nk, int n) {
  const Q8Slot q = q8_slot(ring, seq);
  for (int kh = threadIdx.x; kh < nk; kh += blockDim.x) q.meta[kh * 4 + 0] += n;
}

}  // namespace

cudaError_t launch_q8_append(const float *kst, const float *vst, int ld_rows, Dims d, Rows rows, Ring ring, int rewrite,
                             cudaStream_t s) {
  (void)ld_rows;
  dim3 grid(rows.n, d.nk);
  q8_append_kernel<<<grid, d.hd, 0, s>>>(kst, vst, d, rows, ring, rewrite);
  return cudaGetLastError();
}

cudaError_t launch_q8_append_frozen(const float *kst, const float *vst, int n, Dims d, int seq, long pos0, Ring ring,
                                    cudaStream_t s) {
  dim3 grid(n, d.nk);
  q8_append_frozen_kernel<<<grid, d.hd, 0, s>>>(kst, vst, d, seq, pos0, ring);
  q8_add_count_kernel<<<1, 32, 0, s>>>(ring, seq, d.nk, n);
  return cudaGetLastError();
}

}  // namespace dory
