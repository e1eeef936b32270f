// Batched GEMM of the small-matrix engine: C_b = A_b . B_b^T on fp64 planes.
//
// Small Grams (d <= a few hundred) are latency-bound, and their roots are the
// most sensitive to rounding: with eps = 1e-6 on a unit-trace Gram the
// regularised null space sits at 1e-6 of the spectrum, below what fp32
// products resolve.  This engine keeps every work matrix in fp64.
//
// GB300's fp64 pipe is narrow (about 2 fused multiply-adds per clock per SM),
// so the products run on the fp32 pipes in double-float arithmetic instead: each
// operand is split into fp32 hi + lo (hi = fp32(x), lo = fp32(x - hi)), each
// product a_k b_k is formed exactly in its leading part (hi = ah bh, error by a
// fused multiply-add) plus the cross terms ah bl + al bh, and the dot product is
// accumulated as a compensated sum (TwoSum of the leading parts, errors summed
// apart; Ogita, Rump and Oishi 2005).  The result carries about 44 bits, far
// more than the 1e-3 bar needs and than the digit engine's 27, for about a
// dozen fp32 operations per multiply-add.  Tiles of 16 x 16 outputs, one per
// thread, spread even a 128 x 128 product over 64 CTAs.
#pragma once

#include "engine.cuh"

namespace precond {

struct GemmF64Args {
  const double* A; long long a_bstride; int lda;   // A_b: rows x K
  const double* B; long long b_bstride; int ldb;   // B_b: cols x K
  const int* a_index;    // optional: batch entry -> slot of A (null: identity)
  const int* b_index;    // optional: batch entry -> slot of B
  int M, N, K;
};

constexpr int DF_BM = 16, DF_BN = 16, DF_BK = 64;

// x as an unevaluated fp32 pair hi + lo.
__device__ __forceinline__ float2 split_df(double x) {
  const float hi = __double2float_rn(x);
  return make_float2(hi, __double2float_rn(x - (double)hi));
}

__global__ void __launch_bounds__(256)
gemm_f64_kernel(GemmF64Args g, Epi e) {
  const int b = blockIdx.z;
  if (epi_skip(e, b)) return;
  const int tile_m = blockIdx.y * DF_BM, tile_n = blockIdx.x * DF_BN;
  const double* A = g.A + (long long)(g.a_index ? g.a_index[b] : b) * g.a_bstride;
  const double* B = g.B + (long long)(g.b_index ? g.b_index[b] : b) * g.b_bstride;

  __shared__ float2 As[DF_BK][DF_BM + 1];
  __shared__ float2 Bs[DF_BK][DF_BN + 1];
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  float s = 0.f, c = 0.f;        // compensated sum: leading part and accumulated errors

  for (int k0 = 0; k0 < g.K; k0 += DF_BK) {
    // 16 x 64 tiles of A and B: 1024 elements each, 4 per thread; k fastest for coalescing
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int idx = tid + q * 256;
      const int r = idx >> 6, kk = idx & 63;
      const int gk = k0 + kk;
      const int gr = tile_m + r, gc = tile_n + r;
      As[kk][r] = split_df((gr < g.M && gk < g.K) ? A[(long long)gr * g.lda + gk] : 0.0);
      Bs[kk][r] = split_df((gc < g.N && gk < g.K) ? B[(long long)gc * g.ldb + gk] : 0.0);
    }
    __syncthreads();
#pragma unroll 16
    for (int kk = 0; kk < DF_BK; ++kk) {
      const float2 a = As[kk][ty], bb = Bs[kk][tx];
      // the _rn intrinsics are never contracted into fused operations, which the
      // error-free transformations rely on
      const float p = __fmul_rn(a.x, bb.x);
      float err = fmaf(a.x, bb.x, -p);            // exact error of the leading product
      err = fmaf(a.x, bb.y, err);
      err = fmaf(a.y, bb.x, err);
      const float t = __fadd_rn(s, p);            // TwoSum(s, p)
      const float z = __fsub_rn(t, s);
      const float e2 = __fadd_rn(__fsub_rn(s, __fsub_rn(t, z)), __fsub_rn(p, z));
      c = __fadd_rn(c, __fadd_rn(e2, err));
      s = t;
    }
    __syncthreads();
  }

  double part = 0.0;
  const int r = tile_m + ty, col = tile_n + tx;
  if (r < g.M && col < g.N) {
    const double v = epi_apply_f64(e, b, r, col, (double)s + (double)c);
    if (e.kind == EPI_M) part = v;
  }
  if (e.kind == EPI_M) {
    part = block_sum(part);
    if (threadIdx.x < 32) epi_m_finish(e, b, part, g.M, blockIdx.y * gridDim.x + blockIdx.x);
  }
}

}  // namespace precond
