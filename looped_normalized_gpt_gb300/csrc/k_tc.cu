// Tensor-core projections for steps of 5 or more rows on sm_103a (tcgen05 + TMEM + TMA).
//
// Y[t][n] = sum_k W[n][k] X[t][k] with W bf16 [N][K] (weights stream from HBM) and X the
// step's activation rows, held as two bf16 halves X = Xhi + Xlo (Xhi = bf16(X),
// Xlo = bf16(X - Xhi)) so the product keeps about 16 mantissa bits of the activations.
// Swap-AB: the MMA's M side is 128 weight rows, its N side the step's rows (a tile of BN
// rows, 16 <= BN <= 256), K steps of 16.
//
// Block roles (192 threads): warp 0 lane 0 drives TMA (128B-swizzled tiles into a ring of
// shared-memory stages, completion on mbarriers), warp 1 allocates TMEM and lane 0 issues
// tcgen05.mma (two per K step: Xhi and Xlo; gate and up for SwiGLU) and tcgen05.commit,
// warps 2..5 read the accumulator back with tcgen05.ld. K is split over the blocks of a
// cluster when the weight tiles alone would not fill the GPU: once every block's MMAs are
// done, each block pushes its partial sums of the step rows a rank owns into that rank's
// shared memory (remote stores), and each rank adds the splits in split order and applies
// the epilogue (plain, logit scale, or SwiGLU).
// Every mbarrier wait is bounded: on expiry the block records an error code, stops
// issuing work, waits (bounded) for its own copies and MMAs, frees TMEM and returns.
#include <cuda.h>

#include <cstdlib>

#include "common.cuh"
#include "kernels.h"

namespace dory {

namespace {

constexpr int TC_THREADS = 192;
constexpr int BM = 128;  // weight rows per tile (MMA M)
constexpr int BK = 64;   // K elements per stage (one 128-byte swizzle row)
constexpr uint32_t WAIT_LIMIT = 1u << 20;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// Wait for the phase with the given parity to complete; false after the bound.
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

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// tcgen05 shared-memory matrix descriptor: K-major operand in 128-byte swizzled rows,
// 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFF) >> 4);
  d |= (uint64_t)1 << 16;             // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;   // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;             // descriptor version
  d |= (uint64_t)2 << 61;             // 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16: bf16 x bf16 -> f32, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// 16 columns of this warp's 32 TMEM lanes, without waiting (tmem_wait completes them)
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t *r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ void cluster_sync() {
  __syncwarp();  // the .aligned barrier wants the whole warp converged
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// float4 into shared memory at a local address of block `rank` of the cluster
__device__ __forceinline__ void st_cluster4(uint32_t local, uint32_t rank, float4 v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(remote), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w)
               : "memory");
}

template <int BN, bool DUAL, int ST>
struct TcSmem {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE = A_BYTES * (DUAL ? 2 : 1) + 2 * B_BYTES;  // A (gate, up), B hi and lo
  static constexpr int TOTAL = ST * STAGE + 1024;                     // + alignment slack
  static constexpr int TMEM_COLS = (DUAL ? 2 : 1) * BN <= 32    ? 32
                                   : (DUAL ? 2 : 1) * BN <= 64  ? 64
                                   : (DUAL ? 2 : 1) * BN <= 128 ? 128
                                   : (DUAL ? 2 : 1) * BN <= 256 ? 256
                                                                : 512;
};

template <int BN, bool DUAL, int ST>
__global__ void __launch_bounds__(TC_THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmXh,
                   const __grid_constant__ CUtensorMap tmXl, int N, int K, int T, int t_base, int splits,
                   long pair_rows, float *__restrict__ ws, int *__restrict__ tile_ctr, float *__restrict__ Y, int ldy,
                   EpiArgs ep, int *__restrict__ err, unsigned long long *__restrict__ trace, int late_trigger) {
  using S = TcSmem<BN, DUAL, ST>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_full[ST], bar_empty[ST], bar_acc;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int is_last, failed;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // optional timeline: 0 start, 1 set up, 2 past the dependency wait, 3 first stage landed,
  // 4 last MMA issued, 5 accumulator ready, 6 epilogue entered, 7 done; split K: 8 first
  // cluster barrier passed, 9 partials pushed, 10 second barrier passed, 11 rows stored
  auto mark = [&](int e) {
    if (!trace) return;
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    trace[((size_t)blockIdx.y * gridDim.x + blockIdx.x) * TC_TRACE_EVENTS + e] = t;
  };
  if (threadIdx.x == 0) mark(0);
  const int tile = blockIdx.x / splits, split = blockIdx.x % splits;
  const int n0 = tile * BM;
  const int t0 = blockIdx.y * BN;
  const int nkb = K / BK;
  const int kb0 = (int)((long)nkb * split / splits), kb1 = (int)((long)nkb * (split + 1) / splits);
  const int nk = kb1 - kb0;
  const uint32_t base = (smem_u32(smem_raw) + 1023) & ~1023u;
  auto a_addr = [&](int s, int half) { return base + s * S::STAGE + half * S::A_BYTES; };
  auto b_addr = [&](int s, int lo) {
    return base + s * S::STAGE + (DUAL ? 2 : 1) * S::A_BYTES + lo * S::B_BYTES;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; s++) {
      mbar_init(smem_u32(&bar_full[s]), 1);
      mbar_init(smem_u32(&bar_empty[s]), 1);
    }
    mbar_init(smem_u32(&bar_acc), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    failed = 0;
    is_last = 0;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_sh)),
                 "r"(S::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (threadIdx.x == 0) mark(1);
  const uint32_t tmem = tmem_base_sh;
  const uint32_t tx = (uint32_t)(S::A_BYTES * (DUAL ? 2 : 1) + 2 * S::B_BYTES);

  if (warp == 0) {
    if (lane == 0) {
      // weight tiles do not depend on earlier kernels: issue the first stages' before the wait
      const int pre = nk < ST ? nk : ST;
      for (int i = 0; i < pre; i++) {
        const uint32_t fb = smem_u32(&bar_full[i]);
        mbar_expect_tx(fb, tx);
        const int kc = (kb0 + i) * BK;
        tma_load_2d(a_addr(i, 0), &tmW, kc, n0, fb);
        if (DUAL) tma_load_2d(a_addr(i, 1), &tmW, kc, (int)(n0 + pair_rows), fb);
      }
      pdl_wait();
      mark(2);
      for (int i = 0; i < pre; i++) {
        const uint32_t fb = smem_u32(&bar_full[i]);
        const int kc = (kb0 + i) * BK;
        tma_load_2d(b_addr(i, 0), &tmXh, kc, t_base + t0, fb);
        tma_load_2d(b_addr(i, 1), &tmXl, kc, t_base + t0, fb);
      }
      for (int i = pre; i < nk; i++) {
        const int s = i % ST;
        if (!mbar_wait(smem_u32(&bar_empty[s]), ((i / ST) - 1) & 1)) {
          atomicExch(err, 1);
          failed = 1;
          break;
        }
        const uint32_t fb = smem_u32(&bar_full[s]);
        mbar_expect_tx(fb, tx);
        const int kc = (kb0 + i) * BK;
        tma_load_2d(a_addr(s, 0), &tmW, kc, n0, fb);
        if (DUAL) tma_load_2d(a_addr(s, 1), &tmW, kc, (int)(n0 + pair_rows), fb);
        tma_load_2d(b_addr(s, 0), &tmXh, kc, t_base + t0, fb);
        tma_load_2d(b_addr(s, 1), &tmXl, kc, t_base + t0, fb);
      }
    }
  } else if (warp == 1) {
    pdl_wait();
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(BM, BN);
      for (int i = 0; i < nk; i++) {
        const int s = i % ST;
        if (!mbar_wait(smem_u32(&bar_full[s]), (i / ST) & 1)) {
          atomicExch(err, 2);
          failed = 1;
          break;
        }
        if (i == 0) mark(3);
        fence_after();
#pragma unroll
        for (int kk = 0; kk < BK / 16; kk++) {
          const uint64_t ad = sw128_desc(a_addr(s, 0) + kk * 32);
          const uint64_t bh = sw128_desc(b_addr(s, 0) + kk * 32);
          const uint64_t bl = sw128_desc(b_addr(s, 1) + kk * 32);
          const uint32_t first = (i == 0 && kk == 0) ? 0u : 1u;
          mma_bf16(tmem, ad, bh, idesc, first);
          mma_bf16(tmem, ad, bl, idesc, 1u);
          if (DUAL) {
            const uint64_t au = sw128_desc(a_addr(s, 1) + kk * 32);
            mma_bf16(tmem + BN, au, bh, idesc, first);
            mma_bf16(tmem + BN, au, bl, idesc, 1u);
          }
        }
        mma_commit(smem_u32(&bar_empty[s]));
      }
      mark(4);
      mma_commit(smem_u32(&bar_acc));
    }
  } else {
    pdl_wait();
  }
  if (!late_trigger) pdl_trigger();

  // epilogue: warps 2..5, warp w reads TMEM lanes 32*(w % 4) ..
  // With split K the blocks of a tile form a cluster; their stage memory (drained once every
  // block's MMAs are done) receives the partial sums, see below.
  float *P = reinterpret_cast<float *>(smem_raw + (base - smem_u32(smem_raw)));
  const int tcount = (T - t0) < BN ? (T - t0) : BN;  // valid step rows in this tile
  // A thread's output column n is fixed, so its scales are read once, before any Y store (which
  // the compiler would otherwise have to assume may overwrite them).
  float sv1 = 1.f, sv2 = 1.f;
  if (warp >= 2 && n0 + (warp & 3) * 32 + lane < N) {
    const int n = n0 + (warp & 3) * 32 + lane;
    if (ep.mode != EPI_STORE) sv1 = __ldg(ep.vec + n);
    if (ep.mode == EPI_SILU) sv2 = __ldg(ep.vec2 + n);
  }
  const int mode = ep.mode;
  auto epi = [&](float a, float b, int) {
    if (mode == EPI_SCALE) return a * sv1;
    if (mode == EPI_SILU) {
      const float g = a * sv1;
      return g * sigmoidf_(g) * (b * sv2);
    }
    return a;
  };
  // accumulator columns read per round: all of a 64-column row (one wait for every load)
  constexpr int RB = BN < 64 ? BN : 64;
  auto read_row = [&](uint32_t lane_base, int c0, uint32_t *v, uint32_t *u) {
#pragma unroll
    for (int c = 0; c < RB; c += 16) {
      tmem_ld16_async(lane_base + c0 + c, v + c);
      if (DUAL) tmem_ld16_async(lane_base + BN + c0 + c, u + c);
    }
    tmem_wait();
  };
  bool good = false;  // this warp's accumulator is complete
  if (warp >= 2) {
    const int q = warp & 3;
    const int m = q * 32 + lane;  // row within the tile
    const int n = n0 + m;
    bool ok = mbar_wait(smem_u32(&bar_acc), 0);
    if (!ok) {
      atomicExch(err, 3);
      failed = 1;
    }
    if (threadIdx.x == 64) mark(5);
    fence_after();
    good = ok && !failed;
    if (good && splits == 1) {
      for (int c0 = 0; c0 < BN; c0 += RB) {
        uint32_t v[RB], u[DUAL ? RB : 1];
        read_row(tmem + ((uint32_t)(q * 32) << 16), c0, v, u);
#pragma unroll
        for (int i = 0; i < RB; i++) {
          const int t = c0 + i;
          if (t < tcount && n < N)
            Y[(size_t)(t0 + t) * ldy + n] = epi(__uint_as_float(v[i]), DUAL ? __uint_as_float(u[i]) : 0.f, n);
        }
      }
    }
  }
  if (threadIdx.x == 64) mark(6);
  if (splits > 1) {
    // Rank r of the cluster owns step rows [r * per, (r + 1) * per) of the tile. Every block
    // pushes its partial sums of each rank's rows into that rank's receive buffer
    // R[split][row m (gate, then up)][PL] with remote stores; the rank then adds the splits
    // in split order from its own shared memory.
    const int per = ((tcount + splits - 1) / splits + 3) & ~3;  // rows per rank, whole float4s
    const int PL = per + 4;                                      // padded: conflict-free float4s
    const uint32_t rank = cluster_rank();                        // = this block's split
    cluster_sync();  // every block's MMAs are done: all stage memory may be overwritten
    if (threadIdx.x == 64) mark(8);
    if (warp >= 2 && good) {
      const int q = warp & 3, m = q * 32 + lane;
      const uint32_t rg = smem_u32(P + ((size_t)rank * (DUAL ? 2 : 1) * BM + m) * PL);
      const uint32_t ru = smem_u32(P + ((size_t)rank * 2 * BM + BM + m) * PL);
      for (int c0 = 0; c0 < BN; c0 += RB) {
        uint32_t v[RB], u[DUAL ? RB : 1];
        read_row(tmem + ((uint32_t)(q * 32) << 16), c0, v, u);
#pragma unroll
        for (int g4 = 0; g4 < RB; g4 += 4) {
          const int t = c0 + g4;
          if (t >= tcount) break;
          const uint32_t r = (uint32_t)(t / per), tt = (uint32_t)(t - (int)r * per);
          st_cluster4(rg + tt * 4, r,
                      make_float4(__uint_as_float(v[g4]), __uint_as_float(v[g4 + 1]), __uint_as_float(v[g4 + 2]),
                                  __uint_as_float(v[g4 + 3])));
          if (DUAL)
            st_cluster4(ru + tt * 4, r,
                        make_float4(__uint_as_float(u[g4]), __uint_as_float(u[g4 + 1]), __uint_as_float(u[g4 + 2]),
                                    __uint_as_float(u[g4 + 3])));
        }
      }
    }
    if (threadIdx.x == 64) mark(9);
    cluster_sync();  // this rank's rows from every split are in place (nothing remote after)
    if (threadIdx.x == 64) mark(10);
    if (warp >= 2) {
      const int q = warp & 3, m = q * 32 + lane, n = n0 + m;
      const int ta = (int)rank * per, tb = min(tcount, ta + per);
      for (int t = ta; t < tb; t += 4) {
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
        for (int sp = 0; sp < splits; sp++) {
          const float4 x = *reinterpret_cast<const float4 *>(P + ((size_t)sp * (DUAL ? 2 : 1) * BM + m) * PL + (t - ta));
          a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
          if (DUAL) {
            const float4 y = *reinterpret_cast<const float4 *>(P + ((size_t)sp * 2 * BM + BM + m) * PL + (t - ta));
            b.x += y.x; b.y += y.y; b.z += y.z; b.w += y.w;
          }
        }
        if (n < N) {
          const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
          for (int u = 0; u < 4; u++)
            if (t + u < tb) Y[(size_t)(t0 + t + u) * ldy + n] = epi(av[u], bv[u], n);
        }
      }
    }
    if (threadIdx.x == 64) mark(11);
  }
  fence_before();
  __syncthreads();
  if (failed && threadIdx.x == 64) {
    // let copies and MMAs already issued land before TMEM is freed
    mbar_wait(smem_u32(&bar_acc), 0);
  }
  __syncthreads();
  fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(S::TMEM_COLS) : "memory");
  if (late_trigger) pdl_trigger();
  if (threadIdx.x == 64) mark(7);
}

// ---- many step rows: tokens as the MMA's M side ---------------------------------------
//
// When a step has hundreds of rows (prefill rows of several chunks or sequences at once)
// the projections are dense contractions bound by the tensor pipe, not weight streams. Then
// the MMA's M side is 128 step rows and its N side 256 weight rows (SwiGLU: 128 gate rows and
// the matching 128 up rows), K steps of 16; the activations enter as one bf16 operand (the
// rows rounded to bf16: one MMA per K step). A 4-stage ring of 48 KB stages (activation tile
// 128 x 64, weight tile 256 x 64, both 128B-swizzled, loaded by TMA) feeds one issuing thread;
// the accumulator is 256 TMEM columns; warps 2..5 read a token row per lane and store it with
// the epilogue. One tile per block, grid = weight tiles x token tiles.
constexpr int BT = 128;   // step rows per tile (MMA M)
constexpr int BW = 256;   // weight rows per tile (MMA N)
constexpr int BIG_ST = 4;
constexpr int BIG_A = BT * BK * 2;               // 16 KB
constexpr int BIG_B = BW * BK * 2;               // 32 KB
constexpr int BIG_STAGE = BIG_A + BIG_B;         // 48 KB
constexpr int BIG_SMEM = BIG_ST * BIG_STAGE + 1024;

// With `splits` > 1 (blockIdx.z) the blocks of a tile take consecutive K ranges, store their
// partial tiles to `ws` and count in on the tile's counter; the last one adds the partials
// in split order (the same order whichever block finishes last), applies the epilogue,
// and resets the counter.
template <bool DUAL>
__global__ void __launch_bounds__(TC_THREADS, 1)
    tcb_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, int N, int K,
                    int T, int t_base, long pair_rows, float *__restrict__ Y, int ldy, EpiArgs ep,
                    int *__restrict__ err, int splits, float *__restrict__ ws, int *__restrict__ ctr) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_full[BIG_ST], bar_empty[BIG_ST], bar_acc;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int failed, is_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int OUT = DUAL ? BW / 2 : BW;  // output columns of a tile
  const int n0 = blockIdx.x * OUT;         // first output column (SwiGLU: gate row)
  const int t0 = blockIdx.y * BT;
  const int kb_all = K / BK, split = blockIdx.z;
  const int kb0 = (int)((long)kb_all * split / splits), nk = (int)((long)kb_all * (split + 1) / splits) - kb0;
  const uint32_t base = (smem_u32(smem_raw) + 1023) & ~1023u;
  auto a_addr = [&](int st) { return base + st * BIG_STAGE; };
  auto b_addr = [&](int st) { return base + st * BIG_STAGE + BIG_A; };
  // the two 128-row halves of the weight tile
  const int w_lo = n0, w_hi = DUAL ? (int)(n0 + pair_rows) : n0 + BW / 2;

  if (threadIdx.x == 0) {
    for (int st = 0; st < BIG_ST; st++) {
      mbar_init(smem_u32(&bar_full[st]), 1);
      mbar_init(smem_u32(&bar_empty[st]), 1);
    }
    mbar_init(smem_u32(&bar_acc), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    failed = 0;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_sh)),
                 "r"(BW)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    if (lane == 0) {
      // weight tiles do not depend on earlier kernels: the first stages' go before the wait
      const int pre = nk < BIG_ST ? nk : BIG_ST;
      for (int i = 0; i < pre; i++) {
        const uint32_t fb = smem_u32(&bar_full[i]);
        mbar_expect_tx(fb, BIG_STAGE);
        tma_load_2d(b_addr(i), &tmW, (kb0 + i) * BK, w_lo, fb);
        tma_load_2d(b_addr(i) + BIG_B / 2, &tmW, (kb0 + i) * BK, w_hi, fb);
      }
      pdl_wait();
      for (int i = 0; i < pre; i++)
        tma_load_2d(a_addr(i), &tmX, (kb0 + i) * BK, t_base + t0, smem_u32(&bar_full[i]));
      for (int i = pre; i < nk; i++) {
        const int st = i % BIG_ST;
        if (!mbar_wait(smem_u32(&bar_empty[st]), ((i / BIG_ST) - 1) & 1)) {
          atomicExch(err, 11);
          failed = 1;
          break;
        }
        const uint32_t fb = smem_u32(&bar_full[st]);
        mbar_expect_tx(fb, BIG_STAGE);
        tma_load_2d(b_addr(st), &tmW, (kb0 + i) * BK, w_lo, fb);
        tma_load_2d(b_addr(st) + BIG_B / 2, &tmW, (kb0 + i) * BK, w_hi, fb);
        tma_load_2d(a_addr(st), &tmX, (kb0 + i) * BK, t_base + t0, fb);
      }
    }
  } else if (warp == 1) {
    pdl_wait();
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(BT, BW);
      for (int i = 0; i < nk; i++) {
        const int st = i % BIG_ST;
        if (!mbar_wait(smem_u32(&bar_full[st]), (i / BIG_ST) & 1)) {
          atomicExch(err, 12);
          failed = 1;
          break;
        }
        fence_after();
#pragma unroll
        for (int kk = 0; kk < BK / 16; kk++)
          mma_bf16(tmem, sw128_desc(a_addr(st) + kk * 32), sw128_desc(b_addr(st) + kk * 32), idesc,
                   (i == 0 && kk == 0) ? 0u : 1u);
        mma_commit(smem_u32(&bar_empty[st]));
      }
      mma_commit(smem_u32(&bar_acc));
    }
  } else {
    pdl_wait();
  }
  pdl_trigger();

  const int q = warp & 3, m = q * 32 + lane;  // epilogue warps: this lane's row of the tile
  const int t = t0 + m;                        // and its step row
  const int mode = ep.mode;
  // the epilogue of 16 columns of this lane's row: v (and the up half u) to Y
  auto emit16 = [&](int c0, const float *v, const float *u) {
    if (t >= T) return;
    float o[16];
#pragma unroll
    for (int j = 0; j < 16; j++) {
      const int n = n0 + c0 + j;
      const float a = v[j];
      if (mode == EPI_SCALE) {
        o[j] = n < N ? a * __ldg(ep.vec + n) : 0.f;
      } else if (mode == EPI_SILU) {
        const float g = a * (n < N ? __ldg(ep.vec + n) : 0.f);
        o[j] = g * sigmoidf_(g) * (u[j] * (n < N ? __ldg(ep.vec2 + n) : 0.f));
      } else {
        o[j] = a;
      }
    }
    float *yrow = Y + (size_t)t * ldy + n0 + c0;
    if (n0 + c0 + 16 <= N) {
#pragma unroll
      for (int j = 0; j < 16; j += 4) *reinterpret_cast<float4 *>(yrow + j) = make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]);
    } else {
#pragma unroll
      for (int j = 0; j < 16; j++)
        if (n0 + c0 + j < N) yrow[j] = o[j];
    }
  };
  const size_t tile = (size_t)blockIdx.y * gridDim.x + blockIdx.x;
  if (warp >= 2) {
    bool ok = mbar_wait(smem_u32(&bar_acc), 0);
    if (!ok) {
      atomicExch(err, 13);
      failed = 1;
    }
    fence_after();
    if (ok && !failed) {
      const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
      for (int c0 = 0; c0 < OUT; c0 += 16) {
        uint32_t v[16], u[16];
        tmem_ld16_async(lane_base + c0, v);
        if (DUAL) tmem_ld16_async(lane_base + BW / 2 + c0, u);
        tmem_wait();
        if (splits == 1) {
          emit16(c0, reinterpret_cast<const float *>(v), reinterpret_cast<const float *>(u));
        } else {  // this split's partial sums of the row to the workspace
          float *w = ws + ((tile * splits + split) * BT + m) * BW;
#pragma unroll
          for (int j = 0; j < 16; j += 4) {
            *reinterpret_cast<float4 *>(w + c0 + j) = make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                                                  __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
            if (DUAL)
              *reinterpret_cast<float4 *>(w + BW / 2 + c0 + j) =
                  make_float4(__uint_as_float(u[j]), __uint_as_float(u[j + 1]), __uint_as_float(u[j + 2]),
                              __uint_as_float(u[j + 3]));
          }
        }
      }
    }
  }
  if (splits > 1) {
    __threadfence();  // this block's partials before its count
    __syncthreads();
    if (threadIdx.x == 64) is_last = atomicAdd(ctr + tile, 1) == splits - 1;
    __syncthreads();
    if (is_last) {
      __threadfence();
      if (warp >= 2 && !failed) {
        for (int c0 = 0; c0 < OUT; c0 += 16) {
          float v[16], u[16];
#pragma unroll
          for (int j = 0; j < 16; j++) v[j] = u[j] = 0.f;
          for (int sp = 0; sp < splits; sp++) {
            const float *w = ws + ((tile * splits + sp) * BT + m) * BW;
#pragma unroll
            for (int j = 0; j < 16; j += 4) {
              const float4 a = __ldcg(reinterpret_cast<const float4 *>(w + c0 + j));
              v[j] += a.x, v[j + 1] += a.y, v[j + 2] += a.z, v[j + 3] += a.w;
              if (DUAL) {
                const float4 b = __ldcg(reinterpret_cast<const float4 *>(w + BW / 2 + c0 + j));
                u[j] += b.x, u[j + 1] += b.y, u[j + 2] += b.z, u[j + 3] += b.w;
              }
            }
          }
          emit16(c0, v, u);
        }
      }
      if (threadIdx.x == 64) ctr[tile] = 0;  // ready for the next launch
    }
  }
  fence_before();
  __syncthreads();
  if (failed && threadIdx.x == 64) mbar_wait(smem_u32(&bar_acc), 0);  // let issued copies and MMAs land
  __syncthreads();
  fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(BW) : "memory");
}

template <bool DUAL>
cudaError_t tcb_launch(const TcGemm &g, int T, int t_base, float *Y, int ldy, EpiArgs ep, bool pdl, cudaStream_t s) {
  auto kern = tcb_gemm_kernel<DUAL>;
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, BIG_SMEM);
    attr = true;
  }
  constexpr int OUT = DUAL ? BW / 2 : BW;
  const int gx = (g.N + OUT - 1) / OUT, gy = (T + BT - 1) / BT, tiles = gx * gy;
  // K splits while the blocks still fit one wave (one block per SM: a second wave of a few
  // blocks would double the time): at most 4, at least 8 K blocks each
  int splits = 1;
  while (splits < 4 && tiles * 2 * splits <= g.sms && (g.K / BK) / (2 * splits) >= 8 && tiles <= g.ctr_slots &&
         g.ws_big)
    splits *= 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(gx, gy, splits);
  cfg.blockDim = dim3(TC_THREADS);
  cfg.dynamicSmemBytes = BIG_SMEM;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, g.tmW, g.tmXh, g.N, g.K, T, t_base, g.pair_rows, Y, ldy, ep, g.err, splits,
                            g.ws_big, g.ctr_big);
}

// DORY_TC_TRIGGER=late: let the next kernel launch only once this one's epilogue is done
int late_trigger() {
  static const int v = [] {
    const char *e = getenv("DORY_TC_TRIGGER");
    return e && e[0] == 'l' ? 1 : 0;
  }();
  return v;
}

template <int BN, bool DUAL, int ST>
cudaError_t tc_launch(const TcGemm &g, int T, int t_base, float *Y, int ldy, EpiArgs ep, bool pdl, cudaStream_t s) {
  using S = TcSmem<BN, DUAL, ST>;
  auto kern = tc_gemm_kernel<BN, DUAL, ST>;
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::TOTAL);
    attr = true;
  }
  const int m_tiles = (g.N + BM - 1) / BM;
  const int t_tiles = (T + BN - 1) / BN;
  int splits = g.splits;
  // the partial tile of a split must fit the stage memory it reuses
  const int per = ((BN + splits - 1) / splits + 3) & ~3;  // step rows a rank receives at most
  if ((size_t)splits * (DUAL ? 2 : 1) * BM * (per + 4) * 4 > (size_t)ST * S::STAGE || t_tiles > 1) splits = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(m_tiles * splits, t_tiles);
  cfg.blockDim = dim3(TC_THREADS);
  cfg.dynamicSmemBytes = S::TOTAL;
  cfg.stream = s;
  cudaLaunchAttribute attr1[2];
  int na = 0;
  if (pdl) {
    attr1[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr1[na].val.programmaticStreamSerializationAllowed = 1;
    na++;
  }
  if (splits > 1) {
    attr1[na].id = cudaLaunchAttributeClusterDimension;
    attr1[na].val.clusterDim.x = splits;
    attr1[na].val.clusterDim.y = 1;
    attr1[na].val.clusterDim.z = 1;
    na++;
  }
  cfg.attrs = attr1;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, g.tmW, g.tmXh, g.tmXl, g.N, g.K, T, t_base, splits, g.pair_rows, g.ws,
                            g.ctr, Y, ldy, ep, g.err, g.trace, late_trigger());
}

}  // namespace

int tc_tile_rows(int T) {
  if (T <= 16) return 16;
  if (T <= 32) return 32;
  if (T <= 64) return 64;
  if (T <= 128) return 128;
  return 256;
}

cudaError_t launch_tc_gemm_big(const TcGemm &g, int T, int t_base, float *Y, int ldy, EpiArgs ep, bool pdl,
                               cudaStream_t s) {
  if (g.K % BK || (ep.mode == EPI_SILU ? g.N % (BW / 2) : 0) || ldy % 4) return cudaErrorInvalidValue;
  if (ep.mode == EPI_SILU) return tcb_launch<true>(g, T, t_base, Y, ldy, ep, pdl, s);
  return tcb_launch<false>(g, T, t_base, Y, ldy, ep, pdl, s);
}

cudaError_t launch_tc_gemm(const TcGemm &g, int T, int t_base, float *Y, int ldy, EpiArgs ep, bool pdl,
                           cudaStream_t s) {
  const bool dual = ep.mode == EPI_SILU;
  const int bn = tc_tile_rows(T);
  static const bool deep = [] {
    const char *e = getenv("DORY_TC_DEEP");
    return !(e && e[0] == '0');
  }();
  if (deep && bn == 64) {  // one block per SM with a deeper stage ring (measured faster at 64 rows)
    if (dual) return tc_launch<64, true, 4>(g, T, t_base, Y, ldy, ep, pdl, s);
    return tc_launch<64, false, 6>(g, T, t_base, Y, ldy, ep, pdl, s);
  }
#define TCL(B, D, ST)                                                      \
  if (bn == B && dual == D) return tc_launch<B, D, ST>(g, T, t_base, Y, ldy, ep, pdl, s);
  TCL(16, false, 4) TCL(32, false, 4) TCL(64, false, 3) TCL(128, false, 3) TCL(256, false, 2)
  TCL(16, true, 4) TCL(32, true, 3) TCL(64, true, 2) TCL(128, true, 2) TCL(256, true, 1)
#undef TCL
  return cudaErrorInvalidValue;
}

// Tensor map of a row-major bf16 matrix [rows][cols] read in boxes of box_rows x 64.
int make_tmap_bf16(CUtensorMap *map, const void *base, long rows, long cols, int box_rows) {
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
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -2;
}

}  // namespace dory
