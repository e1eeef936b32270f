// Shared device-side definitions of libprecond (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/precond.h"

namespace precond {

// Per-root bookkeeping, one entry per root of the current call.  A root is
// one Gram (left or right of a weight matrix) or one given SPD matrix.
struct RootStat {
  double trace;        // tr of the source (unnormalised) matrix
  double frob2;        // ||source||_F^2
  double minc;         // Minc row-sum bound of A_hat (max over rows)
  double c;            // start scale: 1.01 * min(Wolkowicz-Styan, Minc) of A_hat
  double resid_acc;    // sum of (M - I)^2 of the iteration in flight
  double resid;        // last ||M - I||_F / sqrt(d)
  double resid_prev;
  int iters;           // iterations executed
  int status;          // PRECOND_OK / ENOTCONV / ENONFINITE
  int done;            // 1: skip further iterations
  int kfinal;          // iteration index whose X is the result (X buffer kfinal & 1)
  unsigned int arrivals;  // tiles of the M product finished (cumulative over iterations)
  int nonfinite;       // NaN/Inf seen in the input or the Gram
  float sac;           // start: 1 / (2 tr c)   (M_0 = (A + A^T) sac + eps / c I)
  float seps;          // start: eps / c
  float fin;           // finish: c^(-1/p)
  int pad;
  double sac_d;        // the start scalars in fp64 (M_0 is formed to more than fp32 precision:
  double seps_d;       // its smallest eigenvalues are eps / c, far below its largest)
};

// Convergence control of the Newton-Schulz stage (same for every root of a call).
struct IterCtl {
  int p;               // 2 or 4
  int kmin;            // stagnation test only after kmin iterations
  int kmax;            // iteration cap
  float tol;           // ||M - I||_F / sqrt(d) <= tol  -> converged
};

__device__ __forceinline__ bool finite_d(double x) { return isfinite(x); }

__device__ __forceinline__ void atomic_max_nonneg(double* addr, double v) {
  // non-negative doubles order like their bit patterns as signed 64-bit ints
  atomicMax(reinterpret_cast<long long*>(addr), __double_as_longlong(v));
}
__device__ __forceinline__ void atomic_max_nonneg(float* addr, float v) {
  atomicMax(reinterpret_cast<int*>(addr), __float_as_int(v));
}

template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
template <typename T>
__device__ __forceinline__ T warp_max(T v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmax(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide sum (blockDim.x multiple of 32, <= 1024); result valid in thread 0.
template <typename T>
__device__ T block_sum(T v) {
  __shared__ T red[32];
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  T r = 0;
  if (w == 0) {
    r = (l < (int)(blockDim.x >> 5)) ? red[l] : T(0);
    r = warp_sum(r);
  }
  return r;
}

__device__ __forceinline__ float load_grad(const void* g, int dtype, long long idx) {
  if (dtype == PRECOND_BF16)
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(g)[idx]);
  return reinterpret_cast<const float*>(g)[idx];
}

}  // namespace precond
