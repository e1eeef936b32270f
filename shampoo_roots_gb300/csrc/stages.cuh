// Element-wise and reduction stages of the preconditioner step:
// gradient preparation, Gram statistics, the largest-eigenvalue bound, the
// start of the iteration and its finish.  All O(d^2), HBM-bound.
//
// The tcgen05 engine's kernels work on (row, 128-column block) units: one warp
// owns a row's block, forms its values, takes the block maximum for the scale
// and writes the digits (engine.cuh).
#pragma once

#include "engine.cuh"

namespace precond {

// ---------------------------------------------------------------------------
// Gradient preparation
// ---------------------------------------------------------------------------
struct PrepArgs {
  const void* const* g;   // per batch entry: caller's gradient (m x n)
  int dtype;
  int m, n;
  const int* roots2;      // per batch entry: the two root ids (left, right)
  RootStat* stats;
  Plane G, GT;            // engine copies of G (m x n) and G^T (n x m)
};

// fp64 engine: 32 x 32 tiles, double copies of G and G^T and the non-finite check.
__global__ void __launch_bounds__(256) prep_f64_kernel(PrepArgs a) {
  __shared__ double tile[32][33];
  const int b = blockIdx.z;
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  const void* g = a.g[b];
  int bad = 0;
  for (int q = ty; q < 32; q += 8) {
    const int r = r0 + q, c = c0 + tx;
    double v = 0.0;
    if (r < a.m && c < a.n) {
      const float f = load_grad(g, a.dtype, (long long)r * a.n + c);
      if (!isfinite(f)) bad = 1;
      v = (double)f;
      f64_store(a.G, b, r, c, v);
    }
    tile[q][tx] = v;
  }
  __syncthreads();
  for (int q = ty; q < 32; q += 8) {
    const int c = c0 + q, r = r0 + tx;
    if (c < a.n && r < a.m) f64_store(a.GT, b, c, r, tile[tx][q]);
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) {
    a.stats[a.roots2[2 * b]].nonfinite = 1;
    a.stats[a.roots2[2 * b + 1]].nonfinite = 1;
  }
}

// tcgen05 engine: one 128 x 128 tile of G per block (staged in shared memory),
// written as digits of G (rows of the tile, one block) and of G^T (columns of
// the tile become rows, one block), plus the non-finite check.
constexpr int PREP_LD = 129;
constexpr int PREP_SMEM = 128 * PREP_LD * 4;

__global__ void __launch_bounds__(256) prep_tc_kernel(PrepArgs a) {
  extern __shared__ float tile[];   // [128][PREP_LD]
  const int b = blockIdx.z;
  const int r0 = blockIdx.y * 128, c0 = blockIdx.x * 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const void* g = a.g[b];
  int bad = 0;
  for (int i = warp; i < 128; i += 8) {
    const int r = r0 + i;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c0 + lane + 32 * u;
      float v = 0.f;
      if (r < a.m && c < a.n) {
        v = load_grad(g, a.dtype, (long long)r * a.n + c);
        if (!isfinite(v)) bad = 1;
      }
      tile[i * PREP_LD + lane + 32 * u] = v;
    }
  }
  __syncthreads();
  for (int i = warp; i < 128; i += 8) {
    float v[4];
    if (r0 + i < a.m) {
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = tile[i * PREP_LD + lane + 32 * u];
      tc_store_row128(a.G, b, r0 + i, c0, a.n, v);
    }
    if (c0 + i < a.n) {
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = tile[(lane + 32 * u) * PREP_LD + i];
      tc_store_row128(a.GT, b, c0 + i, r0, a.m, v);
    }
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) {
    a.stats[a.roots2[2 * b]].nonfinite = 1;
    a.stats[a.roots2[2 * b + 1]].nonfinite = 1;
  }
}

// ---------------------------------------------------------------------------
// Statistics of each root's source matrix (the Gram after the EMA, or a given
// SPD matrix): trace, squared Frobenius norm, absolute row sums.
// ---------------------------------------------------------------------------
struct RootArgs {
  const float* const* src;   // per batch entry: fp32 d x d source (caller's L / R / A)
  const int* root_of;        // batch entry -> root id
  RootStat* stats;
  double* rowabs;            // [b][d]  sum_j |src_ij|
  double* diag;              // [b][d]  src_ii
  double* rowsq;             // [b][d]  sum_j src_ij^2
  float* rvec;               // [b][d]  absolute row sums of A_hat
  int d;
  float eps;
  IterCtl ctl;
  double alpha0, beta0;      // first step polynomial T_0 = alpha0 I - beta0 M_0 (linear first step)
  int write_x1;              // 1: the start also writes X_1 = T_0 (linear first step)
  // engine planes
  Plane M0, X1;              // start outputs
  Plane X[2];                // finish input (X buffer kfinal & 1)
  Plane Xf;                  // finish output in engine format (step), or unused
  float* const* dst;         // finish output to caller fp32 (inv_root), or null
  int packed;                // 1: src is the upper triangle packed row by row
};

// Element (r, c) of a root's source matrix: full row-major, or packed upper triangle.
__device__ __forceinline__ float src_at(const float* A, long long r, long long c, int d, int packed) {
  if (!packed) return A[r * d + c];
  return r <= c ? A[packed_offset(r, c, d)] : A[packed_offset(c, r, d)];
}

__global__ void __launch_bounds__(256) root_stats_kernel(RootArgs a) {
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* A = a.src[b];
  RootStat* st = &a.stats[a.root_of[b]];
  int bad = 0;
  for (int r = blockIdx.x * 8 + warp; r < a.d; r += gridDim.x * 8) {
    // per-lane fp32 partials (at most d/32 terms each), summed across the warp in
    // fixed order in fp64: the sums feed bounds used with a 1.01 margin
    float p1 = 0.f, p2 = 0.f;
    for (int c = lane; c < a.d; c += 32) {
      const float v = src_at(A, r, c, a.d, a.packed);
      if (!isfinite(v)) bad = 1;
      p1 += fabsf(v);
      p2 = fmaf(v, v, p2);
    }
    const double s1 = warp_sum((double)p1);
    const double s2 = warp_sum((double)p2);
    if (lane == 0) {
      const long long o = (long long)b * a.d + r;
      a.rowabs[o] = s1;
      a.rowsq[o] = s2;
      a.diag[o] = src_at(A, r, r, a.d, a.packed);
    }
  }
  bad = __any_sync(0xffffffffu, bad);
  if (lane == 0 && bad) st->nonfinite = 1;
}

// Fixed-order (deterministic) sum of a per-row vector by one block.
__device__ double block_vec_sum(const double* v, int n) {
  double s = 0.0;
  for (int i = threadIdx.x; i < n; i += blockDim.x) s += v[i];
  s = block_sum(s);
  __shared__ double out;
  if (threadIdx.x == 0) out = s;
  __syncthreads();
  return out;
}

// Per root (one block): trace and squared Frobenius norm in a fixed order, and
// the absolute row sums of A_hat = src / tr + eps I,
// r_c = sum_j |A_hat_cj| = (rowabs_c - |src_cc|) / tr + |src_cc / tr + eps|.
__global__ void __launch_bounds__(256) root_trace_kernel(RootArgs a) {
  const int b = blockIdx.x;
  RootStat* st = &a.stats[a.root_of[b]];
  const double t = block_vec_sum(a.diag + (long long)b * a.d, a.d);
  const double f2 = block_vec_sum(a.rowsq + (long long)b * a.d, a.d);
  if (threadIdx.x == 0) {
    st->trace = t;
    st->frob2 = f2;
  }
  const double it = (t > 0.0 && isfinite(t)) ? 1.0 / t : 0.0, eps = (double)a.eps;
  for (int c = threadIdx.x; c < a.d; c += blockDim.x) {
    const double dc = a.diag[(long long)b * a.d + c];
    const double rc = (a.rowabs[(long long)b * a.d + c] - fabs(dc)) * it + fabs(dc * it + eps);
    a.rvec[(long long)b * a.d + c] = (float)fmax(rc, 1e-12);
  }
}

// Minc's bound on A_hat:  max_i (|A_hat| r)_i / r_i  (fp32: it is an upper
// bound used with a 1.01 margin; the sums' rounding is far below that margin).
__global__ void __launch_bounds__(256) root_bound_kernel(RootArgs a) {
  extern __shared__ float rsh[];
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* A = a.src[b];
  RootStat* st = &a.stats[a.root_of[b]];
  const double t = st->trace;
  if (!(t > 0.0) || !isfinite(t)) return;
  const float it = (float)(1.0 / t), eps = a.eps;
  const float* rv = a.rvec + (long long)b * a.d;
  const bool in_smem = a.d <= 12288;           // 48 KB of dynamic shared memory
  if (in_smem) {
    for (int c = threadIdx.x; c < a.d; c += blockDim.x) rsh[c] = rv[c];
    __syncthreads();
  }
  const float* rs = in_smem ? rsh : rv;
  float best = 0.f;
  for (int r = blockIdx.x * 8 + warp; r < a.d; r += gridDim.x * 8) {
    float y = 0.f;
    for (int c = lane; c < a.d; c += 32) y = fmaf(fabsf(src_at(A, r, c, a.d, a.packed)), rs[c], y);
    y = warp_sum(y);
    const float arr = src_at(A, r, r, a.d, a.packed);
    y = y * it - fabsf(arr) * it * rs[r] + fabsf(arr * it + eps) * rs[r];   // the diagonal carries + eps
    best = fmaxf(best, y / rs[r]);
  }
  if (lane == 0 && isfinite(best)) atomic_max_nonneg(&st->minc, (double)best);
}

__device__ __forceinline__ double root_scale(const RootStat& st, int d, double eps) {
  // Wolkowicz-Styan on A_hat: mu = tr/d, s^2 = ||A_hat||_F^2/d - mu^2, mu + s sqrt(d-1)
  const double t = st.trace;
  const double fro2 = st.frob2 / (t * t) + 2.0 * eps + (double)d * eps * eps;
  const double mu = (1.0 + (double)d * eps) / (double)d;
  const double s2 = fmax(fro2 / (double)d - mu * mu, 0.0);
  const double ws = mu + sqrt(s2) * sqrt((double)(d - 1));
  return 1.01 * fmin(ws, st.minc);
}

// Per-root scalars of the start and the finish, one thread per root: the start
// scale c, the flags, 1 / (2 tr c), eps / c and c^(-1/p) (fp64 is slow on this
// part, so the tile kernels only read these).
__global__ void root_scalar_kernel(RootArgs a, int nb) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= nb) return;
  RootStat* st = &a.stats[a.root_of[b]];
  const double eps = (double)a.eps;
  const double t = st->trace;
  const double c = root_scale(*st, a.d, eps);
  const bool bad = st->nonfinite || !(t > 0.0) || !isfinite(t) || !isfinite(c) || !(c > 0.0);
  st->c = c;
  st->resid = 1e300;
  st->iters = 0;
  st->kfinal = 0;
  st->done = bad ? 1 : 0;
  st->status = bad ? PRECOND_ENONFINITE : PRECOND_OK;
  st->sac = bad ? 0.f : (float)(0.5 / (t * c));
  st->seps = bad ? 0.f : (float)(eps / c);
  st->sac_d = bad ? 0.0 : 0.5 / (t * c);
  st->seps_d = bad ? 0.0 : eps / c;
  st->fin = bad ? 0.f : (float)pow(c, -1.0 / (double)a.ctl.p);
}

// ---------------------------------------------------------------------------
// Start: M_0 = A_hat / c (exactly symmetric: (A + A^T)/2 / tr / c + eps / c I)
// and, for a linear first step, X_1 = X_0 T_0 = T_0 = alpha0 I - beta0 M_0.
// ---------------------------------------------------------------------------
// fp64 engine: a block owns 32-row strips and walks their 32 x 32 tiles.
__global__ void __launch_bounds__(256) root_init_f64_kernel(RootArgs a) {
  const int b = blockIdx.z;
  const RootStat* st = &a.stats[a.root_of[b]];
  if (st->done) return;                         // non-finite input or trace
  const double s_ac = st->sac_d, s_eps = st->seps_d;
  const double al = a.alpha0, be = a.beta0;
  const float* A = a.src[b];
  __shared__ float tt[32][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int T = (a.d + 31) / 32;
  for (int strip = blockIdx.x; strip < T; strip += gridDim.x) {
    const int r0 = strip * 32;
    for (int c0 = 0; c0 < a.d; c0 += 32) {
      __syncthreads();
      for (int q = ty; q < 32; q += 8) {
        const int rm = c0 + q, cm = r0 + tx;    // mirrored tile (rows c0.., cols r0..)
        tt[q][tx] = (rm < a.d && cm < a.d) ? src_at(A, rm, cm, a.d, a.packed) : 0.f;
      }
      __syncthreads();
      for (int q = ty; q < 32; q += 8) {
        const int r = r0 + q, col = c0 + tx;
        if (r < a.d && col < a.d) {
          const bool dgl = (r == col);
          const double m0 = ((double)src_at(A, r, col, a.d, a.packed) + (double)tt[tx][q]) * s_ac + (dgl ? s_eps : 0.0);
          f64_store(a.M0, b, r, col, m0);
          if (a.write_x1) f64_store(a.X1, b, r, col, (dgl ? al : 0.0) - be * m0);
        }
      }
    }
  }
}

// tcgen05 engine: block (column block J, 32-row strip, root); each warp owns 4
// rows of the strip and the strip's transposed source block sits in shared memory.
// M_0 is formed as an unevaluated fp32 pair hi + lo (exact sum of the two source
// entries, product with the two-term scalar, fused error terms): its digits then
// hold it to the 27 bits of the representation instead of fp32's 24, which is
// what resolves eigenvalues at eps / c next to ones near 1.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}

__global__ void __launch_bounds__(256) root_init_tc_kernel(RootArgs a) {
  const int b = blockIdx.z;
  const RootStat* st = &a.stats[a.root_of[b]];
  if (st->done) return;
  const float sh = (float)st->sac_d, sl = (float)(st->sac_d - (double)sh);
  const float eh = (float)st->seps_d, el = (float)(st->seps_d - (double)eh);
  const float al = (float)a.alpha0, be = (float)a.beta0;
  const float* A = a.src[b];
  __shared__ float tt[128][33];                 // A[c0 + i][r0 + j]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c0 = blockIdx.x * 128, r0 = blockIdx.y * 32;
  for (int i = warp; i < 128; i += 8) {
    const int rm = c0 + i, cm = r0 + lane;
    tt[i][lane] = (rm < a.d && cm < a.d) ? src_at(A, rm, cm, a.d, a.packed) : 0.f;
  }
  __syncthreads();
  for (int q = warp; q < 32; q += 8) {
    const int r = r0 + q;
    if (r >= a.d) break;
    float mh[4], ml[4], x1[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int cl = lane + 32 * u, col = c0 + cl;
      const bool dgl = (r == col);
      const float av = (col < a.d) ? src_at(A, r, col, a.d, a.packed) : 0.f;
      float s, e;
      two_sum(av, tt[cl][q], s, e);                 // A_rc + A_cr exactly
      const float p = s * sh;
      float lo = fmaf(s, sl, fmaf(e, sh, fmaf(s, sh, -p)));
      float hi = p;
      if (dgl) {
        float s2, e2;
        two_sum(p, eh, s2, e2);
        hi = s2;
        lo += e2 + el;
      }
      mh[u] = hi;
      ml[u] = lo;
      x1[u] = (dgl ? al : 0.f) - be * (hi + lo);
    }
    tc_store_row128_pair(a.M0, b, r, c0, a.d, mh, ml);
    if (a.write_x1) tc_store_row128(a.X1, b, r, c0, a.d, x1);
  }
}

// ---------------------------------------------------------------------------
// Finish: result = sym(X_kfinal) c^(-1/p), to the engine plane Xf (step) or
// the caller's fp32 (inv_root).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) root_finish_f64_kernel(RootArgs a) {
  __shared__ float tile[32][33];
  const int b = blockIdx.z;
  const RootStat* st = &a.stats[a.root_of[b]];
  if (st->status == PRECOND_ENONFINITE || st->kfinal < 1) return;
  const Plane& X = a.X[st->kfinal & 1];
  const float f = st->fin;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int T = (a.d + 31) / 32;
  for (int strip = blockIdx.x; strip < T; strip += gridDim.x) {
    const int r0 = strip * 32;
    for (int c0 = 0; c0 < a.d; c0 += 32) {
      __syncthreads();
      for (int q = ty; q < 32; q += 8) {
        const int rm = c0 + q, cm = r0 + tx;
        tile[q][tx] = (rm < a.d && cm < a.d) ? (float)f64_load(X, b, rm, cm) : 0.f;
      }
      __syncthreads();
      for (int q = ty; q < 32; q += 8) {
        const int r = r0 + q, col = c0 + tx;
        if (r < a.d && col < a.d) {
          const float v = 0.5f * ((float)f64_load(X, b, r, col) + tile[tx][q]) * f;
          if (a.dst) a.dst[b][(long long)r * a.d + col] = v;
          else f64_store(a.Xf, b, r, col, (double)v);
        }
      }
    }
  }
}

__global__ void __launch_bounds__(256) root_finish_tc_kernel(RootArgs a) {
  const int b = blockIdx.z;
  const RootStat* st = &a.stats[a.root_of[b]];
  if (st->status == PRECOND_ENONFINITE || st->kfinal < 1) return;
  const Plane& X = a.X[st->kfinal & 1];
  const float f = st->fin;
  __shared__ float tt[128][33];                 // X[c0 + i][r0 + j]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c0 = blockIdx.x * 128, r0 = blockIdx.y * 32;
  for (int i = warp; i < 128; i += 8) {
    const int rm = c0 + i, cm = r0 + lane;
    tt[i][lane] = (rm < a.d && cm < a.d) ? tc_load(X, b, rm, cm) : 0.f;
  }
  __syncthreads();
  for (int q = warp; q < 32; q += 8) {
    const int r = r0 + q;
    if (r >= a.d) break;
    float x[4];
    tc_load_row128(X, b, r, c0, a.d, x);
#pragma unroll
    for (int u = 0; u < 4; ++u) x[u] = 0.5f * (x[u] + tt[lane + 32 * u][q]) * f;
    if (a.dst) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int col = c0 + lane + 32 * u;
        if (col < a.d) a.dst[b][(long long)r * a.d + col] = x[u];
      }
    } else {
      tc_store_row128(a.Xf, b, r, c0, a.d, x);
    }
  }
}

// ---------------------------------------------------------------------------
// X_1 = X_0 T_0 = alpha I + E_0 (X_0 = I) for quadratic steps, E_0 = T_0 - alpha I.
// Converged or failed roots skip.
// ---------------------------------------------------------------------------
struct ShiftArgs {
  Plane src, dst;
  const int* root_of;
  const RootStat* stats;
  int d;
  float alpha;
};

__global__ void __launch_bounds__(256) shift_identity_f64_kernel(ShiftArgs a) {
  const int b = blockIdx.y;
  if (a.stats[a.root_of[b]].done) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int r = blockIdx.x * 8 + warp; r < a.d; r += gridDim.x * 8)
    for (int c = lane; c < a.d; c += 32)
      f64_store(a.dst, b, r, c, f64_load(a.src, b, r, c) + (r == c ? (double)a.alpha : 0.0));
}

// tcgen05 engine: one warp per (row, 128-column block).  Blocks away from the
// diagonal are the same matrix: digits and scale are copied bit for bit; the
// diagonal block is rebuilt with alpha added and a fresh scale.
__global__ void __launch_bounds__(256) shift_identity_tc_kernel(ShiftArgs a) {
  const int b = blockIdx.z;
  if (a.stats[a.root_of[b]].done) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c0 = blockIdx.x * 128;
  const int r = blockIdx.y * 8 + warp;
  if (r >= a.d) return;
  if (r >= c0 && r < c0 + 128) {
    float v[4];
    tc_load_row128(a.src, b, r, c0, a.d, v);
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (c0 + lane + 32 * u == r) v[u] += a.alpha;
    tc_store_row128(a.dst, b, r, c0, a.d, v);
  } else {
    const long long so = (long long)b * a.src.bstride + (long long)r * a.src.ld;
    const long long dof = (long long)b * a.dst.bstride + (long long)r * a.dst.ld;
    const uint16_t* s = reinterpret_cast<const uint16_t*>(a.src.hi);
    uint16_t* dd = reinterpret_cast<uint16_t*>(a.dst.hi);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c0 + lane + 32 * u;
      if (c < a.d)
#pragma unroll
        for (int p = 0; p < 3; ++p) dd[dof + p * a.dst.pstride + c] = s[so + p * a.src.pstride + c];
    }
    if (lane == 0) *tc_scale_ptr(a.dst, b, c0 / DIG_BLK, r) = *tc_scale_ptr(a.src, b, c0 / DIG_BLK, r);
  }
}

// ---------------------------------------------------------------------------
// Conversions for the self-test and the read-backs
// ---------------------------------------------------------------------------
// Caller fp32 (rows x cols, dense) -> digits: one warp per (row, block).
__global__ void __launch_bounds__(256) f32_to_tc_kernel(const float* src, Plane p, int rows, int cols) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c0 = blockIdx.x * 128;
  const int r = blockIdx.y * 8 + warp;
  if (r >= rows) return;
  float v[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int c = c0 + lane + 32 * u;
    v[u] = c < cols ? src[(long long)r * cols + c] : 0.f;
  }
  tc_store_row128(p, 0, r, c0, cols, v);
}

__global__ void f32_to_f64_kernel(const float* src, Plane p, int rows, int cols) {
  const long long n = (long long)rows * cols;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    f64_store(p, 0, i / cols, i % cols, (double)src[i]);
}

// Engine plane -> caller fp32 (debug / test read-back of a root).
template <int E>
__global__ void plane_to_f32_kernel(Plane p, int b, int rows, int cols, float* dst) {
  const long long n = (long long)rows * cols;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const long long r = i / cols, c = i % cols;
    dst[i] = (E == ENGINE_F64) ? (float)f64_load(p, b, r, c) : tc_load(p, b, r, c);
  }
}

}  // namespace precond
