// Matrix storage of the two root engines and the epilogues shared by their GEMMs.
//
//  * fp64 engine (small matrices): every work matrix is a double plane.
//  * tcgen05 engine (large matrices): every work matrix is a pair of fp16
//    planes (hi, lo) holding value * scale ~= hi + lo, scale a power of two
//    chosen from a bound on the matrix's entries, so that the fp16 split keeps
//    about 22 significant bits.
#pragma once

#include "common.cuh"

namespace precond {

enum Engine { ENGINE_F64 = 0, ENGINE_TC = 1 };

// A batch of row-major matrices in engine format.
//  fp64 engine: `hi` is a double plane.
//  tcgen05 engine, digit form: `hi` is the first of S bf16 digit planes
//    (plane s at hi + s * pstride) holding x = scale * 2^-7 * sum_s P_s with a
//    fixed power-of-two scale >= max |x| (see gemm_tc.cuh);
//  tcgen05 engine, fp32 form (f32 != null): an fp32 copy plus a per-row
//    max |x| (atomic max), sliced into per-row-scaled digits afterwards.
struct Plane {
  void* hi;
  long long pstride;    // elements between digit planes
  long long bstride;    // elements between consecutive batch entries
  int ld;               // leading dimension in elements
  float scale;          // digit form: fixed power-of-two scale
  int S;                // digit form: digits written
  float* f32;           // fp32 form: values [b][rows][ld]
  float* rowmax;        // fp32 form: per-row max |x|  [b][rows]
  int rows;             // rows per batch entry (rowmax stride)
};

// Digits of an fp32 value: y = v / sigma * 2^7 (exact: sigma is a power of
// two), d_1 = rint(y), y <- (y - d_1) * 2^7 (exact: y - rint(y) needs no more
// bits than y), ...  All steps are exact in fp32, so S = 4 digits (28 bits)
// hold every fp32 value of the row whose magnitude is within 2^-4 of sigma.
__device__ __forceinline__ void digits_store(const Plane& p, long long o, float v, float inv_sigma) {
  float r = v * inv_sigma * 128.0f;
  __nv_bfloat16* base = reinterpret_cast<__nv_bfloat16*>(p.hi) + o;
  float w = 1.0f;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    if (s < p.S) {
      const float d = rintf(r);
      base[s * p.pstride] = __float2bfloat16_rn(d * w);   // exact: |d| <= 129, power-of-two weight
      r = (r - d) * 128.0f;
      w *= 0.0078125f;
    }
  }
}

template <int E>
__device__ __forceinline__ void plane_store(const Plane& p, int b, long long i, long long j, double v) {
  const long long o = (long long)b * p.bstride + i * p.ld + j;
  if constexpr (E == ENGINE_F64) {
    reinterpret_cast<double*>(p.hi)[o] = v;
  } else {
    if (p.f32) p.f32[o] = (float)v;
    else digits_store(p, o, (float)v, 1.0f / p.scale);
  }
}

template <int E>
__device__ __forceinline__ double plane_load(const Plane& p, int b, long long i, long long j) {
  const long long o = (long long)b * p.bstride + i * p.ld + j;
  if constexpr (E == ENGINE_F64) {
    return reinterpret_cast<const double*>(p.hi)[o];
  } else {
    if (p.f32) return (double)p.f32[o];
    const __nv_bfloat16* base = reinterpret_cast<const __nv_bfloat16*>(p.hi) + o;
    double acc = 0.0;
    for (int s = p.S - 1; s >= 0; --s) acc += (double)__bfloat162float(base[s * p.pstride]);
    return acc * (double)p.scale * 0.0078125;
  }
}

// ---------------------------------------------------------------------------
// GEMM epilogues.  A GEMM of a launch computes, for every batch entry b,
// acc = A_b . B_b^T (both operands row-major, K contiguous), already divided
// by the operands' scales, and hands each element to one of these.
// ---------------------------------------------------------------------------
enum EpiKind {
  EPI_STORE = 0,  // C_b = acc
  EPI_M     = 1,  // M'_b = acc + beta In_b, residual ||M' - I||, convergence
  EPI_GRAM  = 2,  // state_b = beta state_b + (1-beta) acc   (caller's fp32 L or R)
  EPI_VT    = 3,  // C_b^T = acc   (V = G X_R stored transposed for the second product)
  EPI_U     = 4,  // out_b = acc   (caller's fp32 out or the gradient in place)
  EPI_AFF   = 5,  // C_b = alpha acc + beta In_b + gamma I
};

struct Epi {
  int kind;
  int rows, cols;            // output extent (M x N of the GEMM)
  Plane C;                   // EPI_STORE / EPI_M / EPI_VT / EPI_AFF output
  Plane In;                  // EPI_M / EPI_AFF element-wise input (same shape as C)
  double alpha, beta_in, gamma;
  // root bookkeeping (EPI_STORE / EPI_M / EPI_AFF): batch entry -> root id; skip done roots
  const int* root_of;        // may be null (no skipping)
  RootStat* stats;
  IterCtl ctl;
  int k;                     // iteration index (EPI_M)
  unsigned int tiles_per_entry;
  double* partials;          // EPI_M: per root, per tile residual parts
  long long partials_stride;
  // EPI_GRAM
  float* const* state;       // per batch entry: caller's fp32 state matrix (rows x cols)
  float beta;
  // EPI_U
  void* const* out;          // per batch entry: destination (rows x cols)
  int out_dtype;             // PRECOND_F32 or PRECOND_BF16
  const int* nonfinite_of;   // per batch entry: two root ids whose status gates the write
  float inv_scale;           // constant factor on acc
  const MatStat* mstat;
  int scale_mode;
};

__device__ __forceinline__ double epi_matrix_scale(const Epi& e, int b) { return 1.0; }

// Per-element epilogue.  Returns the contribution to the residual sum (EPI_M).
template <int E>
__device__ __forceinline__ double epi_apply(const Epi& e, int b, long long i, long long j, double acc) {
  switch (e.kind) {
    case EPI_STORE:
      plane_store<E>(e.C, b, i, j, acc);
      return 0.0;
    case EPI_AFF: {
      const double v = e.alpha * acc + e.beta_in * plane_load<E>(e.In, b, i, j) + (i == j ? e.gamma : 0.0);
      plane_store<E>(e.C, b, i, j, v);
      return fabs(v);        // row-max tracking (tcgen05 engine)
    }
    case EPI_M: {
      const double v = acc + e.beta_in * plane_load<E>(e.In, b, i, j);
      plane_store<E>(e.C, b, i, j, v);
      const double r = v - ((i == j) ? 1.0 : 0.0);
      return r * r;
    }
    case EPI_GRAM: {
      float* s = e.state[b];
      const long long o = i * e.cols + j;
      s[o] = (float)((double)e.beta * (double)s[o] + (1.0 - (double)e.beta) * acc);
      return 0.0;
    }
    case EPI_VT:
      plane_store<E>(e.C, b, j, i, acc);
      if (E == ENGINE_TC && e.C.rowmax) atomic_max_nonneg(&e.C.rowmax[(long long)b * e.C.rows + j], (float)fabs(acc));
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

// The same epilogues in fp32 for the tcgen05 engine (its outputs are fp32, and
// fp64 arithmetic is slow on this GPU).  Returns the residual part (EPI_M) or
// |value| (for row maxima).
__device__ __forceinline__ float epi_apply_tc(const Epi& e, int b, long long i, long long j, float acc) {
  switch (e.kind) {
    case EPI_STORE: {
      const long long o = (long long)b * e.C.bstride + i * e.C.ld + j;
      e.C.f32[o] = acc;
      return fabsf(acc);
    }
    case EPI_AFF: {
      const long long o = (long long)b * e.C.bstride + i * e.C.ld + j;
      const float in = e.In.f32[(long long)b * e.In.bstride + i * e.In.ld + j];
      float v = fmaf((float)e.alpha, acc, (float)e.beta_in * in);
      if (i == j) v += (float)e.gamma;
      e.C.f32[o] = v;
      return fabsf(v);
    }
    case EPI_M: {
      const long long o = (long long)b * e.C.bstride + i * e.C.ld + j;
      const float in = e.In.f32[(long long)b * e.In.bstride + i * e.In.ld + j];
      const float v = fmaf((float)e.beta_in, in, acc);
      e.C.f32[o] = v;
      const float r = v - ((i == j) ? 1.0f : 0.0f);
      return r * r;
    }
    case EPI_GRAM: {
      float* s = e.state[b];
      const long long o = i * e.cols + j;
      s[o] = fmaf(e.beta, s[o], (1.0f - e.beta) * acc);
      return 0.f;
    }
    case EPI_U: {
      const long long o = i * e.cols + j;
      if (e.out_dtype == PRECOND_BF16)
        reinterpret_cast<__nv_bfloat16*>(e.out[b])[o] = __float2bfloat16_rn(acc);
      else
        reinterpret_cast<float*>(e.out[b])[o] = acc;
      return 0.f;
    }
  }
  return 0.f;
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
  const double r = sqrt(acc) / sqrt((double)d);
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
