// dory_q8_quantize_noalloc: the q8_2f append of rows into an empty slot, for callers that
// cannot allocate device memory.
//
// Some callers run where cudaMalloc is not theirs to call: code inside another runtime's
// memory pool or allocator (a framework that owns all device memory), code that runs
// while a CUDA graph is being captured (an allocation there breaks the capture), and
// plugins that must not change the process's device-memory footprint. This entry point
// quantises K/V rows exactly as dory_write_kv_rows does for an empty slot (the same codes,
// scales and frozen fields, bit for bit) without a handle and without allocating: the
// caller passes the input rows and the output arrays, and the kernel's only other memory,
// the counters and the copy of the first 64 rows that the freeze reads back, sits in a
// file-scope static device array of a fixed size (about 290 KB, for up to 16 KV heads of
// up to 128 channels).
//
// That array belongs to the library image: every GPU that loads the library holds it until
// the process exits, and every call shares it. Each call clears the part that must start
// at zero (the counters), so a call does not depend on the one before; calls whose work
// overlaps on the GPU (different streams, or different host threads without ordering)
// race on the array and must not be made.
#include <cuda.h>

#include <mutex>

#include "../../include/dory.h"
#include "common.cuh"

namespace dory {
void set_last_error(const char *msg);  // the message dory_last_error() returns on this thread
}

namespace {

constexpr int NA_MAX_NK = 16;
constexpr int NA_MAX_HD = 128;
constexpr int NA_WARM = 64;  // rows before the freeze (kv_cache.rs, KV_COL_WARMUP)

struct NaScratch {
  int32_t meta[NA_MAX_NK][4];  // appended rows, frozen
  float wks[NA_MAX_NK][NA_WARM][NA_MAX_HD / 32];
  float wvs[NA_MAX_NK][NA_WARM];
  int8_t wkq[NA_MAX_NK][NA_WARM][NA_MAX_HD];
  int8_t wvq[NA_MAX_NK][NA_WARM][NA_MAX_HD];
};

static __device__ __align__(256) unsigned char g_q8_scratch[sizeof(NaScratch)];

// In host code `g_q8_scratch` names a host-side stand-in, not device memory: the device
// address comes from cudaGetSymbolAddress, once per device (per primary context: a
// cudaDeviceReset ends the context and the module with it, so a new context, told apart by
// its process-unique id, looks the address up again), with that device current.
constexpr int NA_MAX_DEVICES = 64;
std::mutex g_na_mu;
NaScratch *g_na_ptr[NA_MAX_DEVICES] = {};
unsigned long long g_na_ctx[NA_MAX_DEVICES] = {};

// The process-unique id of the calling thread's current context, or 0 if none is current
// (driver calls reached through the runtime, so the library loads without libcuda).
unsigned long long na_context_id() {
  using GetCurrent = CUresult (*)(CUcontext *);
  using GetId = CUresult (*)(CUcontext, unsigned long long *);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  if (!get_current || !get_id) {
    void *f1 = nullptr, *f2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) != cudaSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess || !f1 || !f2) {
      cudaGetLastError();
      return 0;
    }
    get_current = reinterpret_cast<GetCurrent>(f1);
    get_id = reinterpret_cast<GetId>(f2);
  }
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (get_current(&c) != CUDA_SUCCESS || !c || get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

int na_fail(int code, const char *msg) {
  dory::set_last_error(msg);
  return code;
}

struct NaOut {
  const float *k, *v;
  int8_t *kq, *vq;
  float *ks, *vs, *kcol, *vcol;
  int n, nk, hd;
};

__device__ __forceinline__ float na_warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float na_block_max(float v, float *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = na_warp_max(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = lane < nw ? red[lane] : -INFINITY;
  return na_warp_max(t);
}

// One channel of a row: r / s with s = max(absmax / 127, 1e-12) over its group (a warp of
// 32 channels for K, the block for V), rounded half away from zero and clamped to +-127.
__device__ __forceinline__ int8_t na_quant(float r, float amax, float *scale) {
  const float s = fmaxf(__fdiv_rn(amax, 127.f), 1e-12f);
  *scale = s;
  float q = roundf(__fdiv_rn(r, s));
  return (int8_t)fminf(fmaxf(q, -127.f), 127.f);
}

__device__ void na_put(const NaOut &o, NaScratch *sc, int kh, int row, float kx, float vx, bool frozen, float *red) {
  const int d = threadIdx.x, hd = o.hd;
  const float kr = frozen ? __fdiv_rn(kx, o.kcol[kh * hd + d]) : kx;
  const float vr = frozen ? __fdiv_rn(vx, o.vcol[kh * hd + d]) : vx;
  float ksc, vsc;
  const int8_t kc = na_quant(kr, na_warp_max(fabsf(kr)), &ksc);
  const int8_t vc = na_quant(vr, na_block_max(fabsf(vr), red), &vsc);
  const size_t at = (size_t)kh * o.n + row;
  o.kq[at * hd + d] = kc;
  o.vq[at * hd + d] = vc;
  if ((d & 31) == 0) o.ks[at * (hd / 32) + d / 32] = ksc;
  if (d == 0) o.vs[at] = vsc;
  if (row < NA_WARM) {
    sc->wkq[kh][row][d] = kc;
    sc->wvq[kh][row][d] = vc;
    if ((d & 31) == 0) sc->wks[kh][row][d / 32] = ksc;
    if (d == 0) sc->wvs[kh][row] = vsc;
  }
}

// The freeze over the 64 rows kept in the scratch: col = max(sqrt(sum x^2 / 64), 1e-6)
// summed in row order, then every row quantised again against col.
__device__ void na_freeze(const NaOut &o, NaScratch *sc, int kh, float *red) {
  const int d = threadIdx.x, hd = o.hd;
  float sk = 0.f, sv = 0.f;
  for (int i = 0; i < NA_WARM; i++) {
    const float xk = __fmul_rn((float)sc->wkq[kh][i][d], sc->wks[kh][i][d / 32]);
    const float xv = __fmul_rn((float)sc->wvq[kh][i][d], sc->wvs[kh][i]);
    sk = __fadd_rn(sk, __fmul_rn(xk, xk));
    sv = __fadd_rn(sv, __fmul_rn(xv, xv));
  }
  const float ck = fmaxf(__fsqrt_rn(__fdiv_rn(sk, (float)NA_WARM)), 1e-6f);
  const float cv = fmaxf(__fsqrt_rn(__fdiv_rn(sv, (float)NA_WARM)), 1e-6f);
  o.kcol[kh * hd + d] = ck;
  o.vcol[kh * hd + d] = cv;
  for (int i = 0; i < NA_WARM; i++) {
    const float xk = __fmul_rn((float)sc->wkq[kh][i][d], sc->wks[kh][i][d / 32]);
    const float xv = __fmul_rn((float)sc->wvq[kh][i][d], sc->wvs[kh][i]);
    const float rk = __fdiv_rn(xk, ck), rv = __fdiv_rn(xv, cv);
    float ksc, vsc;
    const int8_t kc = na_quant(rk, na_warp_max(fabsf(rk)), &ksc);
    const int8_t vc = na_quant(rv, na_block_max(fabsf(rv), red), &vsc);
    const size_t at = (size_t)kh * o.n + i;
    o.kq[at * hd + d] = kc;
    o.vq[at * hd + d] = vc;
    if ((d & 31) == 0) o.ks[at * (hd / 32) + d / 32] = ksc;
    if (d == 0) o.vs[at] = vsc;
  }
  if (d == 0) sc->meta[kh][1] = 1;
  __syncthreads();
}

// Rows 0..min(n, 65)-1 in order (the freeze comes at the 65th), one block per KV head.
__global__ void na_q8_seq_kernel(NaOut o, NaScratch *sc) {
  __shared__ float red[32];
  const int kh = blockIdx.x, d = threadIdx.x;
  const int m = o.n < NA_WARM + 1 ? o.n : NA_WARM + 1;
  for (int i = 0; i < m; i++) {
    const int stored = sc->meta[kh][0];
    bool frozen = sc->meta[kh][1] != 0;
    __syncthreads();
    if (stored >= NA_WARM && !frozen) {
      na_freeze(o, sc, kh, red);
      frozen = true;
    }
    const size_t src = ((size_t)i * o.nk + kh) * o.hd + d;
    na_put(o, sc, kh, i, o.k[src], o.v[src], frozen, red);
    __syncthreads();
    if (d == 0) sc->meta[kh][0] = stored + 1;
    __syncthreads();
  }
}

// Rows past the freeze: independent of each other once the fields are frozen.
__global__ void na_q8_frozen_kernel(NaOut o, NaScratch *sc) {
  __shared__ float red[32];
  const int row = NA_WARM + 1 + blockIdx.x, kh = blockIdx.y, d = threadIdx.x;
  const size_t src = ((size_t)row * o.nk + kh) * o.hd + d;
  na_put(o, sc, kh, row, o.k[src], o.v[src], true, red);
}

}  // namespace

extern "C" int dory_q8_quantize_noalloc(const float *k, const float *v, int32_t n, int32_t nk, int32_t hd,
                                        int8_t *kq, float *ks, int8_t *vq, float *vs, float *kcol, float *vcol,
                                        void *stream) {
  if (!k || !v || !kq || !ks || !vq || !vs || !kcol || !vcol) return na_fail(DORY_EINVAL, "a pointer is NULL");
  if (n < 1) return na_fail(DORY_EINVAL, "n must be positive");
  if (nk < 1 || nk > NA_MAX_NK) return na_fail(DORY_EINVAL, "nk above the scratch's 16 KV heads");
  if (hd != 32 && hd != 64 && hd != 128) return na_fail(DORY_EINVAL, "hd must be 32, 64 or 128");
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= NA_MAX_DEVICES)
    return na_fail(DORY_ECUDA, "no current device");
  NaScratch *sc;
  {
    std::lock_guard<std::mutex> lock(g_na_mu);
    const unsigned long long ctx = na_context_id();
    if (!g_na_ptr[dev] || ctx == 0 || ctx != g_na_ctx[dev]) {
      void *p = nullptr;
      if (cudaGetSymbolAddress(&p, g_q8_scratch) != cudaSuccess || !p) {
        cudaGetLastError();
        return na_fail(DORY_ECUDA, "cudaGetSymbolAddress of the static scratch failed");
      }
      g_na_ptr[dev] = static_cast<NaScratch *>(p);
      g_na_ctx[dev] = na_context_id();  // the lookup made the primary context current
    }
    sc = g_na_ptr[dev];
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(sc->meta, 0, sizeof(sc->meta), s) != cudaSuccess ||
      cudaMemsetAsync(kcol, 0, (size_t)nk * hd * 4, s) != cudaSuccess ||
      cudaMemsetAsync(vcol, 0, (size_t)nk * hd * 4, s) != cudaSuccess) {
    cudaGetLastError();
    return na_fail(DORY_ECUDA, "clearing the counters failed");
  }
  NaOut o{k, v, kq, vq, ks, vs, kcol, vcol, n, nk, hd};
  na_q8_seq_kernel<<<nk, hd, 0, s>>>(o, sc);
  if (n > NA_WARM + 1) na_q8_frozen_kernel<<<dim3(n - NA_WARM - 1, nk), hd, 0, s>>>(o, sc);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return na_fail(DORY_ECUDA, cudaGetErrorString(e));
  dory::set_last_error("");
  return DORY_OK;
}
