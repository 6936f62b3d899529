// Groups of threads that work together on one piece of a step: a whole block, or a set of
// consecutive warps of a block that synchronise on a named barrier (the persistent decode
// kernel's consumer warps, or a part of them, while its producer warp streams weights).
#pragma once

#include "common.cuh"

namespace dory {

struct BlockTeam {
  __device__ __forceinline__ int tid() const { return threadIdx.x; }
  __device__ __forceinline__ int size() const { return blockDim.x; }
  __device__ __forceinline__ int warp() const { return threadIdx.x >> 5; }
  __device__ __forceinline__ int nwarps() const { return blockDim.x >> 5; }
  __device__ __forceinline__ void sync() const { __syncthreads(); }
};

// warps [w0, w0 + nw) of the block, synchronising on named barrier `id` (1..15)
struct WarpTeam {
  int w0, nw, id;
  __device__ __forceinline__ int tid() const { return (int)threadIdx.x - 32 * w0; }
  __device__ __forceinline__ int size() const { return 32 * nw; }
  __device__ __forceinline__ int warp() const { return ((int)threadIdx.x >> 5) - w0; }
  __device__ __forceinline__ int nwarps() const { return nw; }
  __device__ __forceinline__ void sync() const {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(32 * nw) : "memory");
  }
};

constexpr int TEAM_MAX_WARPS = 16;

// Sums of two values over the team (every thread gets both). `red` holds 2 x 16 floats.
template <typename Team>
__device__ __forceinline__ void team_sum2(const Team &tm, float &a, float &b, float (*red)[TEAM_MAX_WARPS]) {
  const int lane = threadIdx.x & 31, w = tm.warp();
  a = warp_sum(a);
  b = warp_sum(b);
  tm.sync();
  if (lane == 0) {
    red[0][w] = a;
    red[1][w] = b;
  }
  tm.sync();
  a = b = 0.f;
  for (int i = 0; i < tm.nwarps(); i++) {
    a += red[0][i];
    b += red[1][i];
  }
}

}  // namespace dory
