// Matrix storage of the two root engines and the epilogues of their GEMMs.
//
//  * fp64 engine (small matrices, cross-check): every work matrix is a double
//    plane.
//  * tcgen05 engine: every work matrix is held as three bf16 "digit planes"
//    and one power-of-two scale per (row, 128-column block):
//
//      x_ij = sigma_i,J / 256 * (P1_ij + P2_ij + P3_ij),   J = j / 128,
//      P1 = d1, P2 = d2 / 2^9, P3 = d3 / 2^18,  integers |d_s| <= 256,
//
//    sigma_i,J the smallest power of two >= max over the block of |x_ij|.
//    Every P_s is exact in bf16 (a 9-bit signed integer times a power of
//    two), the three digits hold 27 bits below sigma (the representation
//    error is at most sigma * 2^-27), and no fp32 copy of the matrix exists.
//    The block of 128 columns is the K chunk of the GEMM (gemm_tc.cuh), whose
//    products of one chunk are summed exactly on the tensor cores.
#pragma once

#include "common.cuh"

namespace precond {

enum Engine { ENGINE_F64 = 0, ENGINE_TC = 1 };

constexpr int DIG_BLK = 128;      // columns per scale block (= the GEMM's K chunk)
constexpr int DIGITS = 3;

// A batch of row-major matrices in engine format.
struct Plane {
  void* hi;             // fp64: the double plane; tcgen05: digit plane 1 (plane s at hi + s * pstride)
  long long pstride;    // tcgen05: elements between digit planes
  long long bstride;    // elements between consecutive batch entries
  int ld;               // leading dimension in elements (tcgen05: a multiple of 64)
  float* scale;         // tcgen05: block scales [b][block][srows]
  long long sbstride;   // tcgen05: scale elements between batch entries (blocks * srows)
  int srows;            // tcgen05: scale row stride (rows rounded up to 128)
  int rows;
};

// ---------------------------------------------------------------- digit arithmetic
// Smallest power of two >= m (m >= 0); at least 2^-100 so that 1 / sigma is finite.
__device__ __forceinline__ float pow2_ceil_scale(float m) {
  if (!(m > 7.8886e-31f)) return 7.8886090522101181e-31f;   // 2^-100 (also for NaN: digits become 0 / NaN-free)
  if (!(m < 1.7014118e38f)) return 1.7014118346046923e38f;  // 2^127
  uint32_t u = __float_as_uint(m);
  if (u & 0x7FFFFFu) u = (u & 0x7F800000u) + 0x00800000u;
  return __uint_as_float(u & 0x7F800000u);
}

// Digits of v with 1 / sigma = inv (a power of two): y = v inv 256, d1 = rint(y),
// y <- (y - d1) 512, d2 = rint(y), ...  Every step is exact in fp32 (y - rint(y)
// needs no more bits than y; the products are by powers of two).
__device__ __forceinline__ void digits3(float v, float inv, float& p1, float& p2, float& p3) {
  float y = v * inv * 256.0f;
  const float d1 = rintf(y);
  y = (y - d1) * 512.0f;
  const float d2 = rintf(y);
  y = (y - d2) * 512.0f;
  const float d3 = rintf(y);
  p1 = d1;
  p2 = d2 * 0.001953125f;            // 2^-9
  p3 = d3 * 3.814697265625e-06f;     // 2^-18
}

__device__ __forceinline__ float recon3(float sigma, float p1, float p2, float p3) {
  return sigma * 0.00390625f * (p1 + (p2 + p3));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 t = __floats2bfloat162_rn(a, b);   // exact: every digit is a bf16 number
  return *reinterpret_cast<uint32_t*>(&t);
}

__device__ __forceinline__ float* tc_scale_ptr(const Plane& p, int b, long long blk, long long row) {
  return p.scale + (long long)b * p.sbstride + blk * p.srows + row;
}

// One element of a tcgen05-engine matrix (read-backs and small kernels).
__device__ __forceinline__ float tc_load(const Plane& p, int b, long long i, long long j) {
  const long long o = (long long)b * p.bstride + i * p.ld + j;
  const __nv_bfloat16* base = reinterpret_cast<const __nv_bfloat16*>(p.hi) + o;
  const float s = *tc_scale_ptr(p, b, j / DIG_BLK, i);
  return recon3(s, __bfloat162float(base[0]), __bfloat162float(base[p.pstride]),
                __bfloat162float(base[2 * p.pstride]));
}

// A warp stores columns col0 .. col0 + 127 (col0 a multiple of 128) of row
// `row` as digits with the block's scale; lane holds columns col0 + lane + 32 u
// in v[u] (coalesced accesses); columns >= ncols are neither counted nor written.
__device__ __forceinline__ void tc_store_row128(const Plane& p, int b, long long row, int col0, int ncols,
                                                const float (&v)[4]) {
  const int lane = threadIdx.x & 31;
  float m = 0.f;
#pragma unroll
  for (int u = 0; u < 4; ++u)
    if (col0 + lane + 32 * u < ncols) m = fmaxf(m, fabsf(v[u]));
  m = warp_max(m);
  const float sigma = pow2_ceil_scale(m);
  const float inv = 1.0f / sigma;    // exact: a power of two
  if (lane == 0) *tc_scale_ptr(p, b, col0 / DIG_BLK, row) = sigma;
  __nv_bfloat16* base = reinterpret_cast<__nv_bfloat16*>(p.hi) + (long long)b * p.bstride + row * p.ld;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int c = col0 + lane + 32 * u;
    if (c < ncols) {
      float d1, d2, d3;
      digits3(v[u], inv, d1, d2, d3);
      base[c] = __float2bfloat16_rn(d1);
      base[p.pstride + c] = __float2bfloat16_rn(d2);
      base[2 * p.pstride + c] = __float2bfloat16_rn(d3);
    }
  }
}

// The same for values given as unevaluated fp32 pairs hi + lo (|lo| far below
// |hi|): d1 = rint(y + z) with y, z the scaled parts, and the remainder
// (y - d1) + z carried on, so the digits hold the pair to their own 27 bits.
__device__ __forceinline__ void tc_store_row128_pair(const Plane& p, int b, long long row, int col0, int ncols,
                                                     const float (&hi)[4], const float (&lo)[4]) {
  const int lane = threadIdx.x & 31;
  float m = 0.f;
#pragma unroll
  for (int u = 0; u < 4; ++u)
    if (col0 + lane + 32 * u < ncols) m = fmaxf(m, fabsf(hi[u]));
  m = warp_max(m);
  const float sigma = pow2_ceil_scale(m);
  const float inv = 256.0f / sigma;  // exact: a power of two
  if (lane == 0) *tc_scale_ptr(p, b, col0 / DIG_BLK, row) = sigma;
  __nv_bfloat16* base = reinterpret_cast<__nv_bfloat16*>(p.hi) + (long long)b * p.bstride + row * p.ld;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int c = col0 + lane + 32 * u;
    if (c < ncols) {
      const float y = hi[u] * inv, z = lo[u] * inv;
      const float d1 = rintf(y + z);
      float r = ((y - d1) + z) * 512.0f;
      const float d2 = rintf(r);
      r = (r - d2) * 512.0f;
      const float d3 = rintf(r);
      base[c] = __float2bfloat16_rn(d1);
      base[p.pstride + c] = __float2bfloat16_rn(d2 * 0.001953125f);
      base[2 * p.pstride + c] = __float2bfloat16_rn(d3 * 3.814697265625e-06f);
    }
  }
}

// A warp reads columns col0 + lane + 32 u (u < 4) of row `row` (0 beyond ncols).
__device__ __forceinline__ void tc_load_row128(const Plane& p, int b, long long row, int col0, int ncols,
                                               float (&v)[4]) {
  const int lane = threadIdx.x & 31;
  const float s = *tc_scale_ptr(p, b, col0 / DIG_BLK, row);
  const __nv_bfloat16* base = reinterpret_cast<const __nv_bfloat16*>(p.hi) + (long long)b * p.bstride + row * p.ld;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int c = col0 + lane + 32 * u;
    v[u] = (c < ncols) ? recon3(s, __bfloat162float(base[c]), __bfloat162float(base[p.pstride + c]),
                                __bfloat162float(base[2 * p.pstride + c]))
                       : 0.f;
  }
}

// fp64 engine element access.
__device__ __forceinline__ void f64_store(const Plane& p, int b, long long i, long long j, double v) {
  reinterpret_cast<double*>(p.hi)[(long long)b * p.bstride + i * p.ld + j] = v;
}
__device__ __forceinline__ double f64_load(const Plane& p, int b, long long i, long long j) {
  return reinterpret_cast<const double*>(p.hi)[(long long)b * p.bstride + i * p.ld + j];
}

// ---------------------------------------------------------------------------
// GEMM epilogues.  A GEMM of a launch computes, for every batch entry b,
// acc = A_b . B_b^T (both operands row-major, K contiguous) and hands each
// element to one of these.
// ---------------------------------------------------------------------------
enum EpiKind {
  EPI_STORE = 0,  // f32out_b = acc (fp32, row-major, ld = cols)
  EPI_M     = 1,  // M'_b = acc + beta In_b, residual ||M' - I||, convergence
  EPI_GRAM  = 2,  // state_b = beta state_b + (1-beta) acc   (caller's fp32 L or R)
  EPI_VT    = 3,  // C_b^T = acc   (V = G X_R stored transposed for the second product)
  EPI_U     = 4,  // out_b = acc   (caller's fp32 out or the gradient in place)
  EPI_AFF   = 5,  // C_b = alpha acc + beta In_b + gamma I
};

// Offset of element (i, j), i <= j, of a d x d symmetric matrix stored as its
// upper triangle packed row by row.
__host__ __device__ __forceinline__ long long packed_offset(long long i, long long j, long long d) {
  return i * d - i * (i - 1) / 2 + (j - i);
}

struct Epi {
  int kind;
  int rows, cols;            // output extent (M x N of the GEMM)
  Plane C;                   // EPI_M / EPI_VT / EPI_AFF output
  Plane In;                  // EPI_M / EPI_AFF element-wise input (same shape as C)
  double alpha, beta_in, gamma;
  // root bookkeeping (EPI_M / EPI_AFF): batch entry -> root id; skip done roots
  const int* root_of;        // may be null (no skipping)
  RootStat* stats;
  IterCtl ctl;
  int k;                     // iteration index (EPI_M)
  unsigned int tiles_per_entry;
  double* partials;          // EPI_M: per root, per tile residual parts
  long long partials_stride;
  // EPI_GRAM
  float* const* state;       // per batch entry: caller's fp32 state matrix (rows x cols)
  int state_packed;          // 1: the state is the upper triangle packed row by row (rows == cols)
  float beta;
  // EPI_U
  void* const* out;          // per batch entry: destination (rows x cols)
  int out_dtype;             // PRECOND_F32 or PRECOND_BF16
  const int* nonfinite_of;   // per batch entry: two root ids whose status gates the write
  // EPI_STORE
  float* f32out;
};

// Per-element epilogue of the fp64 engine.  Returns the contribution to the residual sum (EPI_M).
__device__ __forceinline__ double epi_apply_f64(const Epi& e, int b, long long i, long long j, double acc) {
  switch (e.kind) {
    case EPI_STORE:
      e.f32out[(long long)b * e.rows * e.cols + i * e.cols + j] = (float)acc;
      return 0.0;
    case EPI_AFF: {
      const double v = e.alpha * acc + e.beta_in * f64_load(e.In, b, i, j) + (i == j ? e.gamma : 0.0);
      f64_store(e.C, b, i, j, v);
      return 0.0;
    }
    case EPI_M: {
      const double v = acc + e.beta_in * f64_load(e.In, b, i, j);
      f64_store(e.C, b, i, j, v);
      const double r = v - ((i == j) ? 1.0 : 0.0);
      return r * r;
    }
    case EPI_GRAM: {
      if (e.state_packed && i > j) return 0.0;   // the lower triangle is not stored
      float* s = e.state[b];
      const long long o = e.state_packed ? packed_offset(i, j, e.cols) : i * e.cols + j;
      s[o] = (float)((double)e.beta * (double)s[o] + (1.0 - (double)e.beta) * acc);
      return 0.0;
    }
    case EPI_VT:
      f64_store(e.C, b, j, i, acc);
      return 0.0;
    case EPI_U: {
      const long long o = i * e.cols + j;
      if (e.out_dtype == PRECOND_BF16)
        reinterpret_cast<__nv_bfloat16*>(e.out[b])[o] = __float2bfloat16_rn((float)acc);
      else
        reinterpret_cast<float*>(e.out[b])[o] = (float)acc;
      return 0.0;
    }
  }
  return 0.0;
}

// Should this batch entry be skipped?  (root converged, or input non-finite)
__device__ __forceinline__ bool epi_skip(const Epi& e, int b) {
  if (e.kind == EPI_GRAM) {   // leave the state untouched when the gradient is not finite
    if (e.nonfinite_of) {
      const int r0 = e.nonfinite_of[2 * b], r1 = e.nonfinite_of[2 * b + 1];
      if (e.stats[r0].nonfinite || e.stats[r1].nonfinite) return true;
    }
    return false;
  }
  if (e.kind == EPI_U) {
    if (e.nonfinite_of) {
      const int r0 = e.nonfinite_of[2 * b], r1 = e.nonfinite_of[2 * b + 1];
      if (e.stats[r0].status == PRECOND_ENONFINITE || e.stats[r1].status == PRECOND_ENONFINITE) return true;
    }
    return false;
  }
  if (e.root_of == nullptr) return false;
  return e.stats[e.root_of[b]].done != 0;
}

// Called by one full warp of every CTA after its tile of an EPI_M product:
// stores the CTA's residual part and, in the last CTA of the batch entry,
// sums the parts in a fixed order (deterministic) and decides convergence.
__device__ __forceinline__ void epi_m_finish(const Epi& e, int b, double part, int d, unsigned int tile) {
  const int lane = threadIdx.x & 31;
  const int root = e.root_of[b];
  RootStat* st = &e.stats[root];
  double* parts = e.partials + (long long)root * e.partials_stride;
  unsigned int last = 0;
  if (lane == 0) {
    parts[tile] = part;
    __threadfence();
    const unsigned int target = e.tiles_per_entry * (unsigned int)(e.k + 1);
    const unsigned int prev = atomicAdd(&st->arrivals, 1u);
    last = (prev + 1 == target);
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  __threadfence();
  double acc = 0.0;
  for (unsigned int i = lane; i < e.tiles_per_entry; i += 32) acc += *((volatile double*)&parts[i]);
  acc = warp_sum(acc);
  if (lane != 0) return;
  // the stop decision needs no fp64 root (slow, long code on this GPU): fp32 of the fp64 sum
  const double r = (double)sqrtf((float)(acc / (double)d));
  const int kdone = e.k + 1;
  st->iters = kdone;
  st->kfinal = kdone;
  const double prevr = st->resid;
  st->resid_prev = prevr;
  st->resid = r;
  if (!isfinite(r)) {
    st->status = PRECOND_ENONFINITE;
    st->done = 1;
  } else if (r <= (double)e.ctl.tol) {
    st->status = PRECOND_OK;
    st->done = 1;
  } else if (kdone >= e.ctl.kmin && r < 1e-3 && r > 0.5 * prevr) {
    // quadratic phase stopped improving: rounding floor reached above tol
    st->status = PRECOND_ENOTCONV;
    st->done = 1;
  } else if (kdone >= e.ctl.kmax) {
    st->status = PRECOND_ENOTCONV;
    st->done = 1;
  }
}

}  // namespace precond
