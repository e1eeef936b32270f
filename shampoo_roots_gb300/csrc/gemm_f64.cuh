// fp64 SIMT batched GEMM of the small-matrix engine: C_b = A_b . B_b^T.
//
// Small Grams (d <= a few hundred) are latency-bound, and their roots are the
// most sensitive to rounding: with eps = 1e-6 on a unit-trace Gram the
// regularised null space sits at 1e-6 of the spectrum, below what fp32
// products resolve.  This engine keeps every work matrix in fp64.
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

constexpr int F64_BM = 64, F64_BN = 64, F64_BK = 16;

__global__ void __launch_bounds__(256)
gemm_f64_kernel(GemmF64Args g, Epi e) {
  const int b = blockIdx.z;
  if (epi_skip(e, b)) return;
  const int tile_m = blockIdx.y * F64_BM, tile_n = blockIdx.x * F64_BN;
  const double* A = g.A + (long long)(g.a_index ? g.a_index[b] : b) * g.a_bstride;
  const double* B = g.B + (long long)(g.b_index ? g.b_index[b] : b) * g.b_bstride;

  __shared__ double As[F64_BK][F64_BM + 1];
  __shared__ double Bs[F64_BK][F64_BN + 1];
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  double acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0;

  for (int k0 = 0; k0 < g.K; k0 += F64_BK) {
    // 64 x 16 tiles: 1024 elements, 4 per thread; k fastest for coalescing
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int idx = tid + q * 256;
      const int r = idx >> 4, kk = idx & 15;
      const int gr = tile_m + r, gk = k0 + kk;
      As[kk][r] = (gr < g.M && gk < g.K) ? A[(long long)gr * g.lda + gk] : 0.0;
      const int gc = tile_n + r;
      Bs[kk][r] = (gc < g.N && gk < g.K) ? B[(long long)gc * g.ldb + gk] : 0.0;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < F64_BK; ++kk) {
      double a[4], bb[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bb[j] = Bs[kk][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fma(a[i], bb[j], acc[i][j]);
    }
    __syncthreads();
  }

  double part = 0.0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = tile_m + ty + 16 * i;
    if (r >= g.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = tile_n + tx + 16 * j;
      if (c >= g.N) continue;
      const double v = epi_apply_f64(e, b, r, c, acc[i][j]);
      if (e.kind == EPI_M) part += v;
    }
  }
  if (e.kind == EPI_M) {
    part = block_sum(part);
    if (threadIdx.x < 32) epi_m_finish(e, b, part, g.M, blockIdx.y * gridDim.x + blockIdx.x);
  }
}

}  // namespace precond
