// Element-wise and reduction stages of the preconditioner step:
// gradient preparation, Gram statistics, the largest-eigenvalue bound, the
// start of the iteration and its finish.  All O(d^2), HBM-bound.
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
  MatStat* mstat;
  // fp64 engine outputs
  double* Gd; double* GTd;            // [b][m][n], [b][n][m]
  // tcgen05 engine outputs: fp32 copies (rows padded to ld) and row maxima
  float* Gf; int ldn;                 // [b][m][ldn]
  float* GTf; int ldm;                // [b][n][ldm]
  float* rowmax_G;                    // [b][m]   max_j |G_ij|
  float* rowmax_GT;                   // [b][n]   max_i |G_ij|
};

__device__ __forceinline__ float pow2_scale(float target, float maxabs) {
  // largest power of two s with maxabs * s <= target (1 when maxabs is 0)
  if (!(maxabs > 0.0f) || !isfinite(maxabs)) return 1.0f;
  int e;
  frexpf(target / maxabs, &e);     // target/maxabs = f * 2^e, f in [0.5, 1)
  return ldexpf(1.0f, e - 1);
}

// Per batch entry: max |G|, max row sum of squares, non-finite check.
__global__ void __launch_bounds__(256) prep_reduce_kernel(PrepArgs a) {
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const void* g = a.g[b];
  float gmax = 0.f, rmax = 0.f;
  int bad = 0;
  for (int r = blockIdx.x * 8 + warp; r < a.m; r += gridDim.x * 8) {
    float s2 = 0.f, mx = 0.f;
    for (int c = lane; c < a.n; c += 32) {
      const float v = load_grad(g, a.dtype, (long long)r * a.n + c);
      if (!isfinite(v)) bad = 1;
      s2 = fmaf(v, v, s2);
      mx = fmaxf(mx, fabsf(v));
    }
    s2 = warp_sum(s2);
    mx = warp_max(mx);
    rmax = fmaxf(rmax, s2);
    gmax = fmaxf(gmax, mx);
    if (a.rowmax_G && lane == 0) a.rowmax_G[(long long)b * a.m + r] = isfinite(mx) ? mx : 0.f;
  }
  bad = __any_sync(0xffffffffu, bad);
  if (lane == 0) {
    if (isfinite(gmax)) atomic_max_nonneg(&a.mstat[b].gmax, gmax);
    if (isfinite(rmax)) atomic_max_nonneg(&a.mstat[b].rownorm2_max, rmax);
    if (bad) {
      a.stats[a.roots2[2 * b]].nonfinite = 1;
      a.stats[a.roots2[2 * b + 1]].nonfinite = 1;
    }
  }
}

// 32 x 32 tiles: writes the engine copies of G and G^T.
template <int E>
__global__ void __launch_bounds__(256) prep_split_kernel(PrepArgs a) {
  __shared__ float tile[32][33];
  __shared__ float cmax[8][32];
  const int b = blockIdx.z;
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  const void* g = a.g[b];
  float cm = 0.f;
  for (int q = ty; q < 32; q += 8) {
    const int r = r0 + q, c = c0 + tx;
    float v = 0.f;
    if (r < a.m && c < a.n) {
      v = load_grad(g, a.dtype, (long long)r * a.n + c);
      if constexpr (E == ENGINE_F64) a.Gd[((long long)b * a.m + r) * a.n + c] = (double)v;
      else a.Gf[((long long)b * a.m + r) * a.ldn + c] = v;
    }
    tile[q][tx] = v;
    if (isfinite(v)) cm = fmaxf(cm, fabsf(v));
  }
  if constexpr (E == ENGINE_TC) {
    cmax[ty][tx] = cm;
    __syncthreads();
    if (ty == 0 && c0 + tx < a.n) {
      float m = cmax[0][tx];
      for (int q = 1; q < 8; ++q) m = fmaxf(m, cmax[q][tx]);
      atomic_max_nonneg(&a.rowmax_GT[(long long)b * a.n + c0 + tx], m);
    }
  }
  __syncthreads();
  for (int q = ty; q < 32; q += 8) {
    const int c = c0 + q, r = r0 + tx;   // output row c of G^T, column r
    if (c < a.n && r < a.m) {
      const float v = tile[tx][q];
      if constexpr (E == ENGINE_F64) a.GTd[((long long)b * a.n + c) * a.m + r] = (double)v;
      else a.GTf[((long long)b * a.n + c) * a.ldm + r] = v;
    }
  }
}

// fp32 rows -> per-row-scaled digits: sigma_i = smallest power of two >= max_j |x_ij|.
struct SliceArgs {
  const float* src; long long src_bstride; int src_ld;
  const int* root_of;       // may be null; else batch entry -> root id, and converged roots are skipped
  const RootStat* stats;
  const float* rowmax;      // [b][rows]
  float* rowscale;          // [b][rows] out
  Plane dst;                // digit form (scale unused)
  int rows, cols;
};

__device__ __forceinline__ float pow2_ceil(float x) {
  if (!(x > 0.f) || !isfinite(x)) return 1.f;
  int e;
  const float f = frexpf(x, &e);          // x = f 2^e, f in [0.5, 1)
  return f == 0.5f ? x : ldexpf(1.f, e);
}

__device__ __forceinline__ void digits4(float v, float inv, float (&d)[4]) {
  float r = v * inv * 128.0f;
  float w = 1.0f;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const float q = rintf(r);
    d[s] = q * w;                // exact: |q| <= 129, power-of-two weight
    r = (r - q) * 128.0f;
    w *= 0.0078125f;
  }
}

__global__ void __launch_bounds__(256) slice_rows_kernel(SliceArgs a) {
  const int b = blockIdx.y;
  if (a.root_of && a.stats[a.root_of[b]].done) return;   // no further product reads these digits
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int r = blockIdx.x * 8 + warp; r < a.rows; r += gridDim.x * 8) {
    const float sigma = pow2_ceil(a.rowmax[(long long)b * a.rows + r]);
    if (lane == 0) a.rowscale[(long long)b * a.rows + r] = sigma;
    const float inv = 1.0f / sigma;          // exact: sigma is a power of two
    const float* src = a.src + (long long)b * a.src_bstride + (long long)r * a.src_ld;
    const long long o = (long long)b * a.dst.bstride + (long long)r * a.dst.ld;
    __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(a.dst.hi) + o;
    const int nv = (a.cols / 4) * 4;
    // 4 columns per lane (16 B in, 8 B out per plane), two such groups per
    // iteration with both loads issued before any store, so that each lane keeps
    // 32 B in flight
    for (int c = lane * 4; c < nv; c += 256) {
      float4 v[2];
      const bool two = c + 128 < nv;
      v[0] = *reinterpret_cast<const float4*>(src + c);
      if (two) v[1] = *reinterpret_cast<const float4*>(src + c + 128);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (h == 1 && !two) break;
        const int cc = c + h * 128;
        float d0[4], d1[4], d2[4], d3[4];
        digits4(v[h].x, inv, d0);
        digits4(v[h].y, inv, d1);
        digits4(v[h].z, inv, d2);
        digits4(v[h].w, inv, d3);
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          if (s < a.dst.S) {
            __nv_bfloat162 lo2 = __floats2bfloat162_rn(d0[s], d1[s]);
            __nv_bfloat162 hi2 = __floats2bfloat162_rn(d2[s], d3[s]);
            uint2 pk;
            pk.x = *reinterpret_cast<uint32_t*>(&lo2);
            pk.y = *reinterpret_cast<uint32_t*>(&hi2);
            *reinterpret_cast<uint2*>(dst + s * a.dst.pstride + cc) = pk;
          }
        }
      }
    }
    for (int c = nv + lane; c < a.cols; c += 32) digits_store(a.dst, o + c, src[c], inv);
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
  double alpha0, beta0;      // first step polynomial T_0 = alpha0 I - beta0 M_0
  // engine planes
  Plane M0, X1;              // start outputs (fp32 form in the tcgen05 engine)
  Plane X[2];                // finalize input (X buffer kfinal & 1)
  Plane Xf;                  // finalize output in engine format (step), or unused
  float* const* dst;         // finalize output to caller fp32 (inv_root), or null
};

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
      const float v = A[(long long)r * a.d + c];
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
      a.diag[o] = A[(long long)r * a.d + r];
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
    const float* row = A + (long long)r * a.d;
    float y = 0.f;
    for (int c = lane; c < a.d; c += 32) y = fmaf(fabsf(row[c]), rs[c], y);
    y = warp_sum(y);
    const float arr = row[r];
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
  st->fin = bad ? 0.f : (float)pow(c, -1.0 / (double)a.ctl.p);
}

// M_0 = A_hat / c and X_1 = X_0 T_0 = T_0 = alpha0 I - beta0 M_0.  A block owns
// 32-row strips of one root and walks their 32 x 32 tiles, so it holds the
// strips' row maxima itself and stores them once (no atomics).
template <int E>
__global__ void __launch_bounds__(256) root_init_kernel(RootArgs a) {
  const int b = blockIdx.z;
  const RootStat* st = &a.stats[a.root_of[b]];
  if (st->done) return;                         // non-finite input or trace
  const float s_ac = st->sac, s_eps = st->seps;
  const float al = (float)a.alpha0, be = (float)a.beta0;
  const float* A = a.src[b];
  __shared__ float tt[2][32][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int T = (a.d + 31) / 32;
  for (int strip = blockIdx.x; strip < T; strip += gridDim.x) {
    const int r0 = strip * 32;
    float mx[4] = {0.f, 0.f, 0.f, 0.f}, xx[4] = {0.f, 0.f, 0.f, 0.f};   // rows r0 + ty + 8 j
    for (int c0 = 0; c0 < a.d; c0 += 64) {     // two 32-column tiles per pass, loads first
      __syncthreads();                          // the previous pass's reads of tt are done
      float av[2][4];
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int q = ty + 8 * j;
          const int rm = c0 + 32 * t + q, cm = r0 + tx;             // mirrored tile (rows c0.., cols r0..)
          tt[t][q][tx] = (rm < a.d && cm < a.d) ? A[(long long)rm * a.d + cm] : 0.f;
          const int r = r0 + q, col = c0 + 32 * t + tx;             // this strip's own elements
          av[t][j] = (r < a.d && col < a.d) ? A[(long long)r * a.d + col] : 0.f;
        }
      __syncthreads();
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int q = ty + 8 * j;
          const int r = r0 + q, col = c0 + 32 * t + tx;
          if (r < a.d && col < a.d) {
            const bool dgl = (r == col);
            // M_0 = ((A + A^T)/2 / tr + eps I) / c, exactly symmetric
            const float m0 = fmaf(av[t][j] + tt[t][tx][q], s_ac, dgl ? s_eps : 0.f);
            const float x1 = (dgl ? al : 0.f) - be * m0;
            plane_store<E>(a.M0, b, r, col, m0);
            plane_store<E>(a.X1, b, r, col, x1);
            mx[j] = fmaxf(mx[j], fabsf(m0));
            xx[j] = fmaxf(xx[j], fabsf(x1));
          }
        }
    }
    if (E == ENGINE_TC) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = r0 + ty + 8 * j;
        const float m = warp_max(mx[j]), x = warp_max(xx[j]);
        if (tx == 0 && r < a.d) {
          a.M0.rowmax[(long long)b * a.d + r] = m;
          a.X1.rowmax[(long long)b * a.d + r] = x;
        }
      }
    }
  }
}

// Result = sym(X_kfinal) * c^(-1/p): to the engine plane Xf (step) or caller fp32
// (inv_root).  Blocks own 32-row strips, as in the start.
template <int E>
__global__ void __launch_bounds__(256) root_finish_kernel(RootArgs a) {
  __shared__ float tile[2][32][33];
  const int b = blockIdx.z;
  const RootStat* st = &a.stats[a.root_of[b]];
  if (st->status == PRECOND_ENONFINITE || st->kfinal < 1) return;
  const Plane& X = a.X[st->kfinal & 1];
  const float f = st->fin;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int T = (a.d + 31) / 32;
  for (int strip = blockIdx.x; strip < T; strip += gridDim.x) {
    const int r0 = strip * 32;
    float mx[4] = {0.f, 0.f, 0.f, 0.f};
    for (int c0 = 0; c0 < a.d; c0 += 64) {     // two 32-column tiles per pass, loads first
      __syncthreads();                          // the previous pass's reads are done
      float xv[2][4];
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int q = ty + 8 * j;
          const int rm = c0 + 32 * t + q, cm = r0 + tx;             // transposed tile (rows c0.., cols r0..)
          tile[t][q][tx] = (rm < a.d && cm < a.d) ? (float)plane_load<E>(X, b, rm, cm) : 0.f;
          const int r = r0 + q, col = c0 + 32 * t + tx;
          xv[t][j] = (r < a.d && col < a.d) ? (float)plane_load<E>(X, b, r, col) : 0.f;
        }
      __syncthreads();
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int q = ty + 8 * j;
          const int r = r0 + q, col = c0 + 32 * t + tx;
          if (r < a.d && col < a.d) {
            const float v = 0.5f * (xv[t][j] + tile[t][tx][q]) * f;
            if (a.dst) a.dst[b][(long long)r * a.d + col] = v;
            else plane_store<E>(a.Xf, b, r, col, (double)v);
            mx[j] = fmaxf(mx[j], fabsf(v));
          }
        }
    }
    if (E == ENGINE_TC && !a.dst) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = r0 + ty + 8 * j;
        const float m = warp_max(mx[j]);
        if (tx == 0 && r < a.d) a.Xf.rowmax[(long long)b * a.d + r] = m;
      }
    }
  }
}

// X_1 = X_0 T_0 = alpha I + E_0 (X_0 = I) for quadratic steps, E_0 = T_0 - alpha I:
// one warp per row, row maxima stored directly.  Converged or failed roots skip.
struct ShiftArgs {
  Plane src, dst;
  const int* root_of;
  const RootStat* stats;
  int d;
  float alpha;
};

template <int E>
__global__ void __launch_bounds__(256) shift_identity_kernel(ShiftArgs a) {
  const int b = blockIdx.y;
  if (a.stats[a.root_of[b]].done) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int r = blockIdx.x * 8 + warp; r < a.d; r += gridDim.x * 8) {
    float mx = 0.f;
    int c0 = 0;
    if (E == ENGINE_TC) {
      // fp32 rows start 256 B aligned (ld is a multiple of 64): 16-byte vectors, two in flight
      const float* src = a.src.f32 + (long long)b * a.src.bstride + (long long)r * a.src.ld;
      float* dst = a.dst.f32 + (long long)b * a.dst.bstride + (long long)r * a.dst.ld;
      const int nv = (a.d / 4) * 4;
      for (int c = lane * 4; c < nv; c += 256) {
        float4 v[2];
        const bool two = c + 128 < nv;
        v[0] = *reinterpret_cast<const float4*>(src + c);
        if (two) v[1] = *reinterpret_cast<const float4*>(src + c + 128);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (h == 1 && !two) break;
          const int cc = c + h * 128;
          float4 w = v[h];
          if (r >= cc && r < cc + 4) (&w.x)[r - cc] += a.alpha;
          *reinterpret_cast<float4*>(dst + cc) = w;
          mx = fmaxf(mx, fmaxf(fmaxf(fabsf(w.x), fabsf(w.y)), fmaxf(fabsf(w.z), fabsf(w.w))));
        }
      }
      c0 = nv;
    }
    for (int c = c0 + lane; c < a.d; c += 32) {
      const float v = (float)plane_load<E>(a.src, b, r, c) + (r == c ? a.alpha : 0.f);
      plane_store<E>(a.dst, b, r, c, (double)v);
      mx = fmaxf(mx, fabsf(v));
    }
    if (E == ENGINE_TC) {
      mx = warp_max(mx);
      if (lane == 0) a.dst.rowmax[(long long)b * a.d + r] = mx;
    }
  }
}

// Caller fp32 -> engine plane (GEMM self-test inputs).
template <int E>
__global__ void f32_to_plane_kernel(const float* src, Plane p, int rows, int cols) {
  const long long n = (long long)rows * cols;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    plane_store<E>(p, 0, i / cols, i % cols, (double)src[i]);
    if (E == ENGINE_TC && p.rowmax) atomic_max_nonneg(&p.rowmax[i / cols], fabsf(src[i]));
  }
}


// Engine plane -> caller fp32 (debug / test read-back of a root).
template <int E>
__global__ void plane_to_f32_kernel(Plane p, int b, int rows, int cols, float* dst) {
  const long long n = (long long)rows * cols;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const long long r = i / cols, c = i % cols;
    dst[i] = (float)plane_load<E>(p, b, r, c);
  }
}

}  // namespace precond
