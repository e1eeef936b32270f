// libprecond host side: the C ABI of include/precond.h.
//
// A call is planned into classes:
//  * shape classes: weight matrices of the same (m, n) and engine, batched in
//    the preparation, Gram and apply launches;
//  * root classes: roots (left / right Grams, or given SPD matrices) of the
//    same side d and engine, batched in the bound, start, iteration and finish
//    launches.
// Matrices with max(m, n) <= small_dim use the fp64 engine, the others
// the tcgen05 engine (three bf16 digit planes per matrix with per-(row,
// 128-column block) scales, exact digit products on the tensor cores).
// Everything is enqueued on the caller's stream; the only host <-> device
// traffic of a call is one upload of its pointer / index tables.

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <list>
#include <map>
#include <mutex>
#include <sstream>
#include <string>
#include <vector>

#include "common.cuh"
#include "engine.cuh"
#include "gemm_f64.cuh"
#include "gemm_tc.cuh"
#include "stages.cuh"

using namespace precond;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

constexpr size_t ALIGN = 1024;
inline size_t align_up(size_t x, size_t a = ALIGN) { return (x + a - 1) / a * a; }
inline int ld16(int cols) { return (int)align_up((size_t)cols, 64); }   // 16-bit planes: rows padded to 128 B

struct Slab {   // an engine-format matrix batch inside the workspace
  size_t off = 0;        // double plane (fp64 engine) or first bf16 digit plane (tcgen05 engine)
  long long pstride = 0; // elements between digit planes
  int rows = 0, cols = 0, ld = 0, batch = 0;
  size_t scale = 0;      // tcgen05: block scales [batch][nblk][srows]
  int nblk = 0, srows = 0;
};

struct StepPoly {       // per-iteration step polynomials T_k = alpha_k I - beta_k M + gamma_k M^2
  std::vector<double> alpha, beta, gamma;
  std::vector<double> lo;   // bottom of the interval [lo_k, 1] holding M_k's spectrum
};

struct RootClass {
  int d = 0, eng = 0;
  std::vector<int> roots;              // global root ids
  std::vector<const float*> src;       // per entry: source matrix (caller)
  std::vector<float*> dst;             // per entry: caller output (inv_root)
  Slab X[2], M[2], D, F, Xf;   // per-row-scaled (tcgen05) or double planes
  size_t rowabs = 0, diag = 0, rowsq = 0, rvec = 0, partials = 0;
  long long tiles = 0;
  size_t t_root = 0, t_src = 0, t_dst = 0;   // device tables (offsets)
  int kmax = 0;
  int tc_ord = -1;                     // ordinal among the tcgen05 root classes (scratch regions)
  StepPoly steps;                      // per-iteration step polynomial coefficients
};

struct ShapeClass {
  int m = 0, n = 0, eng = 0;
  std::vector<int> mats;
  int lrc = -1, rrc = -1;
  std::vector<int> lslot, rslot;
  Slab Gd, GTd, VTd;                    // fp64 engine
  Slab Gq, GTq, VTq;                    // tcgen05 engine: digits with block scales
  size_t t_g = 0, t_L = 0, t_R = 0, t_out = 0, t_roots2 = 0, t_lslot = 0, t_rslot = 0;
};

struct Plan {
  bool step = true;
  int count = 0, nroots = 0, p = 4, dtype = PRECOND_F32;
  bool out_f32 = false;
  std::vector<ShapeClass> sc;
  std::vector<RootClass> rc;
  size_t stats = 0, err = 0, partials = 0, meta = 0, meta_bytes = 0, total = 0;
  size_t scratch = 0, scratch_slot_bytes = 0;   // tcgen05 GEMM tile hand-over slots, one region per stream
  int scratch_slots = 0;
  long long scratch_ctas = 0;                    // CTAs a region serves (the largest tcgen05 grid)
  long long max_tiles = 0;
  std::vector<uint8_t> meta_host;
};

}  // namespace

struct precond_ctx {
  int device = -1;
  double tol = 1e-4;
  int max_iter = 0, min_iter = 4, engine = 0, small_dim = 64, timing = 0, use_graph = 1;
  int classical = 0;                   // 1: classical Newton step polynomial at every iteration
  double fold = 0.3;                   // minimax step: T(1) >= fold * T(l)
  std::map<std::string, StepPoly> schedules;   // step schedules already computed (keyed by l0, p, fold, degree)
  int step_degree = 2;                 // 2: quadratic step polynomials at p = 4; 1: linear
  int packed = 0;                      // 1: precond_step's EMA state is the packed upper triangle
  int tile_split = 4;                  // most CTAs that share one tile of a small tcgen05 launch
  double ws_max = 0;
  void* ws = nullptr;
  size_t ws_cap = 0;
  size_t planned_bytes = 0;   // workspace bytes of the last validated plan
  void* pinned = nullptr;
  size_t pinned_cap = 0;
  cudaEvent_t upload_done = nullptr;
  bool upload_pending = false;
  cudaEvent_t ev[5] = {};
  bool events = false;
  cudaStream_t last_stream = nullptr;
  int last_nroots = 0;
  int last_p = 4;
  bool have_last = false;
  std::vector<int> last_root_d;       // per root: d
  std::vector<int> last_root_class, last_root_slot;
  Plan last_plan;
  int64_t launches = 0;
  int64_t ns_launches = 0;
  bool in_ns = false;                  // timing: inside the iteration stage
  std::vector<cudaEvent_t> gemm_ev;    // timing: start/stop pairs around iteration-stage GEMMs
  size_t gemm_ev_used = 0;
  EncodeTiledFn encode = nullptr;
  bool tc_attr_set = false;
  int num_sms = 152;                   // a GB300's; a device handle reads its device's count
  // CUDA graph of the last plan (replayed on an internal stream joined to the caller's by events)
  struct Graph {                       // one captured plan
    std::string key;
    cudaGraphExec_t exec = nullptr;
    void* ws = nullptr;                // the workspace its kernels point into
    int64_t kernels = 0, ns_launches = 0;
    size_t gemm_ev = 0;
  };
  std::list<Graph> graphs;             // most recently used first, at most kMaxGraphs
  cudaStream_t gstream = nullptr;
  cudaEvent_t gev_in = nullptr, gev_out = nullptr;
  bool branches = true;                // false: the iteration stage stays on the call's stream
  std::vector<cudaStream_t> side;      // iteration-stage branches (two per root class)
  std::vector<cudaEvent_t> sev;        // their fork / join events
  bool capturing = false;              // timing events become event-record nodes of the graph
};

namespace {

#define CK(call)                                                                 \
  do {                                                                           \
    cudaError_t e_ = (call);                                                     \
    if (e_ != cudaSuccess) {                                                     \
      fprintf(stderr, "libprecond: %s failed: %s\n", #call, cudaGetErrorString(e_)); \
      return PRECOND_ECUDA;                                                      \
    }                                                                            \
  } while (0)

int iter_cap(double eps, int d, int p, double tol, int user_max) {
  if (user_max > 0) return user_max;
  // scalar model of the iteration on the smallest scaled eigenvalue
  double m = eps / (1.01 * (1.0 + d * eps));
  int k = 0;
  while (std::fabs(m - 1.0) >= tol * 0.1 && k < 200) {
    m = m * std::pow((p + 1 - m) / p, p);
    ++k;
  }
  return std::min(k + 3, 60);
}


// Step polynomials of the iteration.  Every step uses T_k = alpha_k I - beta_k M_k
// (X <- X T, M <- T^p M keep M = X^p M_0 for ANY such polynomial).  The
// classical choice is alpha = (p+1)/p, beta = 1/p.  Here each step is the
// minimax choice for the interval [l_k, 1] that holds M_k's spectrum: among
// g(m) = m (a - m)^p, a in (1, p+1], take the one maximising
// min(g(l), g(1)) / max_[l,1] g, then scale so the image's top is 1; the image
// [l_{k+1}, 1] is the next interval (the idea of the Chebyshev-optimised
// coefficients of "Online KL Shampoo" section 2.3, computed here for
// any p from the interval alone).  From l_0 = 1e-6 it needs 10 steps at p = 4
// where the classical step needs 20.
static double step_ratio(double l, double a, int p, double* gmax_out) {
  auto g = [&](double m) { return m * std::pow(a - m, p); };
  const double ms = a / (p + 1);
  double gmax = std::max(g(l), g(1.0));
  if (ms > l && ms < 1.0) gmax = std::max(gmax, g(ms));
  if (gmax_out) *gmax_out = gmax;
  return std::min(g(l), g(1.0)) / gmax;
}

// `fold` caps how far a step may push the top of the interval below its
// bottom: T(1) >= fold * T(l), i.e. a - 1 >= fold (a - l).  A deep fold
// stores directions at tiny magnitudes for a step and costs accuracy; with
// fold = 0.3 the step count at p = 4 is unchanged (10 from l = 1e-6).
static StepPoly step_schedule(double l0, int p, int max_steps, double fold) {
  StepPoly sp;
  double l = l0;
  for (int k = 0; k < max_steps; ++k) {
    const double amin = std::max(1.0 + 1e-12, (1.0 - fold * l) / (1.0 - fold));
    double best_a = p + 1.0, best_r = step_ratio(l, best_a, p, nullptr);
    for (int i = 0; i <= 600; ++i) {      // coarse search on log(a - amin)
      const double a = amin + std::pow(10.0, -10.0 + 10.0 * i / 600.0) * (p + 1.0 - amin);
      if (a > p + 1.0) break;
      const double r = step_ratio(l, a, p, nullptr);
      if (r > best_r) { best_r = r; best_a = a; }
    }
    double lo = std::max(amin, amin + (best_a - amin) * 0.9), hi = std::min(p + 1.0, amin + (best_a - amin) * 1.1 + 1e-12);
    for (int it = 0; it < 200; ++it) {    // golden refinement
      const double m1 = lo + (hi - lo) * 0.381966, m2 = hi - (hi - lo) * 0.381966;
      if (step_ratio(l, m1, p, nullptr) < step_ratio(l, m2, p, nullptr)) lo = m1; else hi = m2;
    }
    const double a = 0.5 * (lo + hi);
    double gmax;
    const double r = step_ratio(l, a, p, &gmax);
    const double sc = std::pow(gmax, -1.0 / p);
    sp.alpha.push_back(a * sc);
    sp.beta.push_back(sc);
    sp.gamma.push_back(0.0);
    sp.lo.push_back(l);
    l = r;
    if (1.0 - l < 1e-9) break;
  }
  return sp;
}

// Quadratic steps T(m) = s (1 + u m + v m^2).  The map g(m) = m T(m)^p on [l, 1]
// has its extrema at l, 1 and the roots of  1 + (p+1) u m + (2p+1) v m^2 = 0
// (where T + p m T' vanishes), so its range is exact.  Returns min g / max g, or
// 0 when T is not positive on [l, 1] or folds (min T < fold max T).
static double quad_ratio(double l, double u, double v, int p, double fold, double* gmax_out) {
  auto T = [&](double m) { return 1.0 + u * m + v * m * m; };
  double tmin = std::min(T(l), T(1.0)), tmax = std::max(T(l), T(1.0));
  if (v != 0.0) {
    const double ms = -u / (2.0 * v);
    if (ms > l && ms < 1.0) { tmin = std::min(tmin, T(ms)); tmax = std::max(tmax, T(ms)); }
  }
  if (!(tmin > 0.0) || tmin < fold * tmax) return 0.0;
  auto g = [&](double m) { return m * std::pow(T(m), p); };
  double gmin = std::min(g(l), g(1.0)), gmax = std::max(g(l), g(1.0));
  const double A = (2.0 * p + 1.0) * v, B = (p + 1.0) * u, C = 1.0;
  double roots[2];
  int nr = 0;
  if (A == 0.0) {
    if (B != 0.0) roots[nr++] = -C / B;
  } else {
    const double disc = B * B - 4.0 * A * C;
    if (disc >= 0.0) {
      const double q = -0.5 * (B + std::copysign(std::sqrt(disc), B));
      if (q != 0.0) roots[nr++] = q / A;
      if (q != 0.0) roots[nr++] = C / q;
    }
  }
  for (int i = 0; i < nr; ++i)
    if (roots[i] > l && roots[i] < 1.0) { gmin = std::min(gmin, g(roots[i])); gmax = std::max(gmax, g(roots[i])); }
  if (gmax_out) *gmax_out = gmax;
  return gmin / gmax;
}

// Nelder-Mead on (u, v) maximising quad_ratio, from a few fixed starts and the
// previous step's optimum; deterministic.
static void quad_best(double l, int p, double fold, double& u, double& v) {
  const double starts[][2] = {{u, v}, {-2.06, 1.52}, {-1.8, 1.3}, {-0.8, 0.38}, {-0.4, 0.111}, {-1.2, 0.6}};
  double bu = u, bv = v, br = quad_ratio(l, u, v, p, fold, nullptr);
  for (const auto& st : starts) {
    double x[3][2] = {{st[0], st[1]}, {st[0] + 0.05, st[1]}, {st[0], st[1] + 0.05}};
    double f[3];
    for (int i = 0; i < 3; ++i) f[i] = -quad_ratio(l, x[i][0], x[i][1], p, fold, nullptr);
    for (int it = 0; it < 600; ++it) {
      int o[3] = {0, 1, 2};
      std::sort(o, o + 3, [&](int a, int b) { return f[a] < f[b]; });
      const int b0 = o[0], b1 = o[1], w = o[2];
      const double cx = 0.5 * (x[b0][0] + x[b1][0]), cy = 0.5 * (x[b0][1] + x[b1][1]);
      auto eval = [&](double t, double* px) {
        px[0] = cx + t * (x[w][0] - cx);
        px[1] = cy + t * (x[w][1] - cy);
        return -quad_ratio(l, px[0], px[1], p, fold, nullptr);
      };
      double xr[2], xe[2], xc[2];
      const double fr = eval(-1.0, xr);
      if (fr < f[b0]) {
        const double fe = eval(-2.0, xe);
        if (fe < fr) { x[w][0] = xe[0]; x[w][1] = xe[1]; f[w] = fe; }
        else { x[w][0] = xr[0]; x[w][1] = xr[1]; f[w] = fr; }
      } else if (fr < f[b1]) {
        x[w][0] = xr[0]; x[w][1] = xr[1]; f[w] = fr;
      } else {
        const double fc = eval(0.5, xc);
        if (fc < f[w]) { x[w][0] = xc[0]; x[w][1] = xc[1]; f[w] = fc; }
        else {
          for (int i = 0; i < 3; ++i) {
            if (i == b0) continue;
            x[i][0] = 0.5 * (x[i][0] + x[b0][0]);
            x[i][1] = 0.5 * (x[i][1] + x[b0][1]);
            f[i] = -quad_ratio(l, x[i][0], x[i][1], p, fold, nullptr);
          }
        }
      }
      if (std::fabs(x[0][0] - x[1][0]) + std::fabs(x[0][1] - x[2][1]) + std::fabs(x[1][0] - x[2][0]) < 1e-13) break;
    }
    for (int i = 0; i < 3; ++i)
      if (-f[i] > br) { br = -f[i]; bu = x[i][0]; bv = x[i][1]; }
  }
  u = bu;
  v = bv;
}

// Per-step quadratic minimax schedule (see step_schedule for the linear one).
static StepPoly step_schedule_quad(double l0, int p, int max_steps, double fold) {
  StepPoly sp;
  double l = l0, u = -2.06, v = 1.52;
  for (int k = 0; k < max_steps; ++k) {
    quad_best(l, p, fold, u, v);
    double gmax;
    const double r = quad_ratio(l, u, v, p, fold, &gmax);
    if (!(r > 0.0)) break;
    const double sc = std::pow(gmax, -1.0 / p);
    sp.alpha.push_back(sc);
    sp.beta.push_back(-sc * u);
    sp.gamma.push_back(sc * v);
    sp.lo.push_back(l);
    l = r;
    if (1.0 - l < 1e-9) break;
  }
  return sp;
}

struct Layout {
  size_t top = 0;
  size_t take(size_t bytes) {
    size_t o = top;
    top = align_up(top + std::max<size_t>(bytes, 1));
    return o;
  }
};

Slab make_slab(Layout& L, int eng, int batch, int rows, int cols) {
  Slab s;
  s.rows = rows;
  s.cols = cols;
  s.batch = batch;
  if (eng == ENGINE_F64) {
    s.ld = cols;
    s.off = L.take((size_t)batch * rows * cols * sizeof(double));
  } else {
    s.ld = ld16(cols);
    s.pstride = (long long)batch * rows * s.ld;
    s.off = L.take((size_t)s.pstride * 2 * DIGITS);
    s.nblk = (cols + DIG_BLK - 1) / DIG_BLK;
    s.srows = (int)align_up((size_t)rows, 128);
    s.scale = L.take((size_t)batch * s.nblk * s.srows * sizeof(float));
  }
  return s;
}


struct MetaWriter {
  std::vector<uint8_t>& buf;
  size_t base;   // workspace offset of the meta region
  explicit MetaWriter(std::vector<uint8_t>& b, size_t base_) : buf(b), base(base_) {}
  template <typename T>
  size_t put(const std::vector<T>& v) {
    size_t o = align_up(buf.size(), 16);
    buf.resize(o + std::max<size_t>(v.size() * sizeof(T), 16));
    if (!v.empty()) memcpy(buf.data() + o, v.data(), v.size() * sizeof(T));
    return base + o;
  }
};

int check_power(float power, int* p) {
  if (power == -0.25f) { *p = 4; return PRECOND_OK; }
  if (power == -0.5f) { *p = 2; return PRECOND_OK; }
  return PRECOND_EINVAL;
}

int pick_engine(const precond_ctx* h, int64_t maxdim) {
  if (h->engine == 1) return ENGINE_F64;
  if (h->engine == 2) return ENGINE_TC;
  return maxdim <= h->small_dim ? ENGINE_F64 : ENGINE_TC;
}

// Root-class planes.  The iteration is written without identity offsets in
// any product operand (see launch_iterations), so every tcgen05 operand holds
// its own information in its digits.
void layout_root_class(Layout& L, RootClass& r, int p) {
  const int nb = (int)r.roots.size(), d = r.d, e = r.eng;
  for (int i = 0; i < 2; ++i) {
    r.X[i] = make_slab(L, e, nb, d, d);
    r.M[i] = make_slab(L, e, nb, d, d);
  }
  r.D = make_slab(L, e, nb, d, d);
  if (p == 4) r.F = make_slab(L, e, nb, d, d);
  r.Xf = r.D;   // D is free once the iteration ends; the finished root takes its place
  r.rowabs = L.take((size_t)nb * d * sizeof(double));
  r.diag = L.take((size_t)nb * d * sizeof(double));
  r.rowsq = L.take((size_t)nb * d * sizeof(double));
  r.rvec = L.take((size_t)nb * d * sizeof(float));
}

int build_plan(precond_ctx* h, Plan& P, bool step, int count, const int64_t* dims2, int dtype, float eps,
               int p, void* const* grads, float* const* Ls, float* const* Rs, float* const* outs,
               const float* const* As, float* const* Xs) {
  P = Plan();
  P.step = step;
  P.count = count;
  P.p = p;
  P.dtype = dtype;
  P.out_f32 = outs != nullptr;
  std::map<std::pair<int, int>, int> rc_index;
  auto root_class = [&](int d, int eng) {
    auto key = std::make_pair(d, eng);
    auto it = rc_index.find(key);
    if (it != rc_index.end()) return it->second;
    RootClass r;
    r.d = d;
    r.eng = eng;
    P.rc.push_back(r);
    rc_index[key] = (int)P.rc.size() - 1;
    return (int)P.rc.size() - 1;
  };
  if (step) {
    std::map<std::pair<int, int>, int> sc_index;
    P.nroots = 2 * count;
    for (int i = 0; i < count; ++i) {
      const int m = (int)dims2[2 * i], n = (int)dims2[2 * i + 1];
      auto key = std::make_pair(m, n);
      auto it = sc_index.find(key);
      int s;
      if (it == sc_index.end()) {
        ShapeClass c;
        c.m = m;
        c.n = n;
        c.eng = pick_engine(h, std::max(m, n));
        P.sc.push_back(c);
        s = (int)P.sc.size() - 1;
        sc_index[key] = s;
      } else {
        s = it->second;
      }
      P.sc[s].mats.push_back(i);
    }
    for (auto& c : P.sc) {
      c.lrc = root_class(c.m, c.eng);
      c.rrc = root_class(c.n, c.eng);
      for (int i : c.mats) {
        RootClass& l = P.rc[c.lrc];
        c.lslot.push_back((int)l.roots.size());
        l.roots.push_back(2 * i);
        l.src.push_back(Ls ? Ls[i] : nullptr);
        l.dst.push_back(nullptr);
        RootClass& r = P.rc[c.rrc];
        c.rslot.push_back((int)r.roots.size());
        r.roots.push_back(2 * i + 1);
        r.src.push_back(Rs ? Rs[i] : nullptr);
        r.dst.push_back(nullptr);
      }
    }
  } else {
    P.nroots = count;
    for (int i = 0; i < count; ++i) {
      const int d = (int)dims2[i];
      const int r = root_class(d, pick_engine(h, d));
      P.rc[r].roots.push_back(i);
      P.rc[r].src.push_back(As ? As[i] : nullptr);
      P.rc[r].dst.push_back(Xs ? Xs[i] : nullptr);
    }
  }

  Layout L;
  P.stats = L.take(sizeof(RootStat) * P.nroots);
  P.err = L.take(64);
  for (auto& r : P.rc) {
    layout_root_class(L, r, p);
    // interval of M_0's spectrum: [eps / c_max, 1], c_max = 1.01 tr(A_hat) >= c
    {
      const double l0 = eps / (1.01 * (1.0 + r.d * eps));
      // quadratic steps pay off at p = 4 (7 steps of 5 products instead of 10 of 4);
      // at p = 2 both degrees need 36 products, so p = 2 keeps linear steps
      const int deg = (p == 4 && !h->classical) ? h->step_degree : 1;
      char key[96];
      snprintf(key, sizeof(key), "%.17g %d %.17g %d", l0, p, h->fold, deg);
      auto it = h->schedules.find(key);
      if (it == h->schedules.end())
        it = h->schedules.emplace(key, deg == 2 ? step_schedule_quad(l0, p, 60, h->fold)
                                                : step_schedule(l0, p, 60, h->fold)).first;
      r.steps = it->second;
    }
    if (h->classical) {
      r.steps.alpha.assign(r.steps.alpha.size(), (p + 1.0) / p);
      r.steps.beta.assign(r.steps.beta.size(), 1.0 / p);
      r.steps.gamma.assign(r.steps.gamma.size(), 0.0);
    }
    const int planned = h->classical ? iter_cap(eps, r.d, p, h->tol, 0) : (int)r.steps.alpha.size() + 3;
    r.kmax = h->max_iter > 0 ? h->max_iter : std::min(planned, 60);
    while ((int)r.steps.alpha.size() < std::max(r.kmax, 1)) {   // then Newton steps
      r.steps.alpha.push_back((p + 1.0) / p);
      r.steps.beta.push_back(1.0 / p);
      r.steps.gamma.push_back(0.0);
      r.steps.lo.push_back(1.0);
    }
    const long long t = r.eng == ENGINE_F64
        ? (long long)((r.d + DF_BM - 1) / DF_BM) * ((r.d + DF_BN - 1) / DF_BN)
        : (long long)((r.d + TC_BM - 1) / TC_BM) * ((r.d + TC_BN - 1) / TC_BN);
    P.max_tiles = std::max(P.max_tiles, t);
  }
  P.partials = L.take(sizeof(double) * P.max_tiles * P.nroots);
  for (auto& c : P.sc) {
    const int nb = (int)c.mats.size();
    if (c.eng == ENGINE_F64) {
      c.Gd = make_slab(L, ENGINE_F64, nb, c.m, c.n);
      c.GTd = make_slab(L, ENGINE_F64, nb, c.n, c.m);
      c.VTd = make_slab(L, ENGINE_F64, nb, c.n, c.m);
    } else {
      c.Gq = make_slab(L, ENGINE_TC, nb, c.m, c.n);
      c.GTq = make_slab(L, ENGINE_TC, nb, c.n, c.m);
      c.VTq = make_slab(L, ENGINE_TC, nb, c.n, c.m);
    }
  }
  // hand-over slots of the tcgen05 GEMM: two 128 x 128 fp32 tiles per CTA (at most one CTA per
  // SM), one region for the call's stream and one for each side stream the iteration stage may fork
  {
    auto tiles = [](long long rows, long long cols) { return ((rows + TC_BM - 1) / TC_BM) * ((cols + TC_BN - 1) / TC_BN); };
    int tc_classes = 0;
    long long most = 0;
    for (auto& r : P.rc)
      if (r.eng == ENGINE_TC) {
        r.tc_ord = tc_classes++;
        most = std::max(most, tiles(r.d, r.d) * (long long)r.roots.size());
      }
    for (const auto& c : P.sc)
      if (c.eng == ENGINE_TC)
        most = std::max(most, std::max(tiles(c.m, c.m), std::max(tiles(c.n, c.n), tiles(c.m, c.n))) *
                                  (long long)c.mats.size());
    if (most > 0) {
      // a launch of fewer tiles may spread each over up to tile_split CTAs (tc_split)
      P.scratch_ctas = std::min<long long>(most * h->tile_split, h->num_sms);
      P.scratch_slots = 1 + 2 * tc_classes;
      P.scratch_slot_bytes = (size_t)P.scratch_ctas * 2 * TC_BM * TC_BN * sizeof(float);
      P.scratch = L.take(P.scratch_slot_bytes * P.scratch_slots);
    }
  }
  // meta tables
  P.meta = L.top;
  MetaWriter W(P.meta_host, P.meta);
  for (auto& r : P.rc) {
    std::vector<int> ro(r.roots.begin(), r.roots.end());
    r.t_root = W.put(ro);
    r.t_src = W.put(r.src);
    r.t_dst = W.put(r.dst);
  }
  for (auto& c : P.sc) {
    std::vector<const void*> g;
    std::vector<float*> l, rr;
    std::vector<void*> o;
    std::vector<int> roots2;
    for (int i : c.mats) {
      g.push_back(grads ? grads[i] : nullptr);
      l.push_back(Ls ? Ls[i] : nullptr);
      rr.push_back(Rs ? Rs[i] : nullptr);
      o.push_back(outs ? (void*)outs[i] : (grads ? grads[i] : nullptr));
      roots2.push_back(2 * i);
      roots2.push_back(2 * i + 1);
    }
    c.t_g = W.put(g);
    c.t_L = W.put(l);
    c.t_R = W.put(rr);
    c.t_out = W.put(o);
    c.t_roots2 = W.put(roots2);
    c.t_lslot = W.put(c.lslot);
    c.t_rslot = W.put(c.rslot);
  }
  P.meta_bytes = align_up(P.meta_host.size(), 16);
  P.meta_host.resize(P.meta_bytes);
  P.total = align_up(P.meta + P.meta_bytes);
  return PRECOND_OK;
}

void drop_graph(precond_ctx* h);

// Timing event record; under capture it becomes a node of the graph, so the
// events still fire (and can be timed) on every replay.
cudaError_t record_event(precond_ctx* h, cudaEvent_t ev, cudaStream_t st) {
  return h->capturing ? cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal) : cudaEventRecord(ev, st);
}

int ensure_workspace(precond_ctx* h, size_t bytes) {
  if (h->ws_max > 0 && (double)bytes > h->ws_max) return PRECOND_ENOMEM;
  if (bytes <= h->ws_cap) return PRECOND_OK;
  CK(cudaDeviceSynchronize());
  drop_graph(h);
  if (h->ws) cudaFree(h->ws);
  h->ws = nullptr;
  h->ws_cap = 0;
  if (cudaMalloc(&h->ws, bytes) != cudaSuccess) {
    cudaGetLastError();
    return PRECOND_ENOMEM;
  }
  h->ws_cap = bytes;
  return PRECOND_OK;
}

int upload_meta(precond_ctx* h, const Plan& P, cudaStream_t st) {
  if (h->upload_pending) {
    CK(cudaEventSynchronize(h->upload_done));
    h->upload_pending = false;
  }
  if (P.meta_bytes > h->pinned_cap) {
    if (h->pinned) cudaFreeHost(h->pinned);
    h->pinned = nullptr;
    h->pinned_cap = 0;
    CK(cudaMallocHost(&h->pinned, P.meta_bytes));
    h->pinned_cap = P.meta_bytes;
  }
  memcpy(h->pinned, P.meta_host.data(), P.meta_bytes);
  CK(cudaMemcpyAsync((char*)h->ws + P.meta, h->pinned, P.meta_bytes, cudaMemcpyHostToDevice, st));
  CK(cudaEventRecord(h->upload_done, st));
  h->upload_pending = true;
  return PRECOND_OK;
}

// --------------------------------------------------------------------------- launch helpers
Plane slab_plane(char* ws, const Slab& s) {
  Plane p;
  memset(&p, 0, sizeof(p));
  p.hi = ws + s.off;
  p.pstride = s.pstride;
  p.bstride = (long long)s.rows * s.ld;
  p.ld = s.ld;
  p.rows = s.rows;
  if (s.nblk) {
    p.scale = reinterpret_cast<float*>(ws + s.scale);
    p.sbstride = (long long)s.nblk * s.srows;
    p.srows = s.srows;
  }
  return p;
}

struct Ctx {
  precond_ctx* h;
  const Plan& P;
  char* ws;
  cudaStream_t st;
  int sslot = 0;         // scratch region of the stream (0: the call's stream, 1 + i: side stream i)
  template <typename T>
  T* at(size_t off) const { return reinterpret_cast<T*>(ws + off); }
  RootStat* stats() const { return at<RootStat>(P.stats); }
  unsigned int* err() const { return at<unsigned int>(P.err); }
  Plane plane(const Slab& s) const { return slab_plane(ws, s); }
};

Epi base_epi(const Ctx& c, int kind, int rows, int cols) {
  Epi e;
  memset(&e, 0, sizeof(e));
  e.kind = kind;
  e.rows = rows;
  e.cols = cols;
  e.stats = c.stats();
  e.alpha = 1.0;
  return e;
}

// Tensor map of one digit plane of a slab: operand boxes {K block 32, 128 rows}
// with 64-byte swizzle (the MMA operand layout).
int encode_map(precond_ctx* h, CUtensorMap* map, void* base, const Slab& s, int box_rows) {
  cuuint64_t dims[3] = {(cuuint64_t)s.cols, (cuuint64_t)s.rows, (cuuint64_t)s.batch};
  cuuint64_t strides[2] = {(cuuint64_t)s.ld * 2, (cuuint64_t)s.ld * 2 * s.rows};
  cuuint32_t box[3] = {(cuuint32_t)TC_BK, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = h->encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    fprintf(stderr, "libprecond: cuTensorMapEncodeTiled failed (%d)\n", (int)r);
    return PRECOND_ECUDA;
  }
  return PRECOND_OK;
}

// Batched product C_b = A_b B_b^T in the engine of the operands.
// Ins: the slab of the element-wise input (EPI_AFF, EPI_M) of the tcgen05
// engine, which must be A itself (the epilogue reads it from the operand ring).
// CTAs per tile of a tcgen05 launch of `work` tiles: the largest of 4, 2, 1 (at most
// max_split) whose CTAs still fit on the GPU at one per SM.  A lone tile's latency is
// mostly its output pass, which the split divides; the MMAs it repeats are cheap there.
int tc_split(long long work, int num_sms, int max_split) {
  for (int s = 4; s > 1; s >>= 1)
    if (s <= max_split && work * s <= num_sms) return s;
  return 1;
}

int gemm(const Ctx& c, int eng, const Slab& A, const Slab& B, int M, int N, int K, const int* aidx,
         const int* bidx, const Epi& e0, int batch, bool sym = false, const Slab* Ins = nullptr) {
  Epi e = e0;
  if (eng == ENGINE_F64) {
    GemmF64Args g;
    g.A = c.at<double>(A.off);
    g.a_bstride = (long long)A.rows * A.ld;
    g.lda = A.ld;
    g.B = c.at<double>(B.off);
    g.b_bstride = (long long)B.rows * B.ld;
    g.ldb = B.ld;
    g.a_index = aidx;
    g.b_index = bidx;
    g.M = M;
    g.N = N;
    g.K = K;
    dim3 grid((N + DF_BN - 1) / DF_BN, (M + DF_BM - 1) / DF_BM, batch);
    e.tiles_per_entry = grid.x * grid.y;
    gemm_f64_kernel<<<grid, 256, 0, c.st>>>(g, e);
  } else {
    // the epilogue takes its element-wise input from the operand ring: it must be A itself
    if (Ins && (Ins->off != A.off || e.kind == EPI_AFF && e.alpha == 0.0)) return PRECOND_EINVAL;
    TcMaps maps;
    memset(&maps, 0, sizeof(maps));
    int rc;
    for (int q = 0; q < DIGITS; ++q) {
      if ((rc = encode_map(c.h, &maps.a[q], c.ws + A.off + (size_t)q * A.pstride * 2, A, TC_BM))) return rc;
      if ((rc = encode_map(c.h, &maps.b[q], c.ws + B.off + (size_t)q * B.pstride * 2, B, TC_BN))) return rc;
    }
    TcGemmArgs g;
    memset(&g, 0, sizeof(g));
    g.scratch = c.at<float>(c.P.scratch + (size_t)c.sslot * c.P.scratch_slot_bytes);
    g.M = M;
    g.N = N;
    g.K = K;
    g.a_index = aidx;
    g.b_index = bidx;
    g.a_scale = c.at<const float>(A.scale);
    g.a_sbstride = (long long)A.nblk * A.srows;
    g.a_srows = A.srows;
    g.b_scale = c.at<const float>(B.scale);
    g.b_sbstride = (long long)B.nblk * B.srows;
    g.b_srows = B.srows;
    g.err = c.err();
    g.batch = batch;
    g.sym = (sym && M == N) ? 1 : 0;
    const long long tn = (N + TC_BN - 1) / TC_BN;
    const long long tiles = g.sym ? tn * (tn + 1) / 2 : tn * ((M + TC_BM - 1) / TC_BM);
    e.tiles_per_entry = (unsigned int)tiles;
    g.split = tc_split(tiles * batch, c.h->num_sms, c.h->tile_split);
    dim3 grid((unsigned int)std::min<long long>(tiles * batch * g.split, (long long)c.h->num_sms), 1, 1);
    // every CTA needs its two hand-over slots in the stream's scratch region
    if (c.sslot >= c.P.scratch_slots || (long long)grid.x > c.P.scratch_ctas) return PRECOND_EINVAL;
    const bool timed = c.h->timing == 1 && c.h->events && c.h->in_ns;   // per-launch events: mode 1 only
    // iteration-stage products count the MMA work they issue (converged roots' tiles are skipped on the device)
    g.issued = c.h->in_ns ? reinterpret_cast<unsigned long long*>(c.err() + 2) : nullptr;
    if (timed) {
      while (c.h->gemm_ev.size() < c.h->gemm_ev_used + 2) {
        cudaEvent_t ev;
        CK(cudaEventCreate(&ev));
        c.h->gemm_ev.push_back(ev);
      }
      CK(record_event(c.h, c.h->gemm_ev[c.h->gemm_ev_used], c.st));
    }
    gemm_tc_kernel<<<grid, TC_THREADS, TcSmem::BYTES, c.st>>>(maps, g, e);
    if (timed) {
      CK(record_event(c.h, c.h->gemm_ev[c.h->gemm_ev_used + 1], c.st));
      c.h->gemm_ev_used += 2;
    }
  }
  c.h->launches++;
  CK(cudaGetLastError());
  return PRECOND_OK;
}

// Blocks per root of the fp64 start / finish kernels: one per 32-row strip.
unsigned int tile_blocks(int d) { return (unsigned int)((d + 31) / 32); }

RootArgs root_args(const Ctx& c, const RootClass& r, float eps) {
  RootArgs a;
  memset(&a, 0, sizeof(a));
  a.src = c.at<const float* const>(r.t_src);
  a.root_of = c.at<const int>(r.t_root);
  a.stats = c.stats();
  a.rowabs = c.at<double>(r.rowabs);
  a.diag = c.at<double>(r.diag);
  a.rowsq = c.at<double>(r.rowsq);
  a.rvec = c.at<float>(r.rvec);
  a.d = r.d;
  a.eps = eps;
  a.ctl.p = c.P.p;
  a.ctl.kmin = c.h->min_iter;
  a.ctl.kmax = r.kmax;
  a.ctl.tol = (float)c.h->tol;
  a.M0 = c.plane(r.M[0]);
  a.X1 = c.plane(r.X[1]);
  a.alpha0 = r.steps.alpha[0];
  a.beta0 = r.steps.beta[0];
  a.write_x1 = r.steps.gamma[0] == 0.0 ? 1 : 0;   // quadratic first steps form X_1 from E_0
  a.X[0] = c.plane(r.X[0]);
  a.X[1] = c.plane(r.X[1]);
  a.Xf = c.plane(r.Xf);
  a.dst = c.P.step ? nullptr : c.at<float* const>(r.t_dst);
  a.packed = c.P.step ? c.h->packed : 0;
  return a;
}

int launch_roots_start(const Ctx& c0, float eps, bool br) {
  for (size_t ri = 0; ri < c0.P.rc.size(); ++ri) {
    const RootClass& r = c0.P.rc[ri];
    const Ctx c{c0.h, c0.P, c0.ws, br ? c0.h->side[2 * ri] : c0.st};     // one class per branch
    const int nb = (int)r.roots.size();
    RootArgs a = root_args(c, r, eps);
    const int rb = std::min((r.d + 7) / 8, 512);
    root_stats_kernel<<<dim3(rb, nb), 256, 0, c.st>>>(a);
    root_trace_kernel<<<nb, 256, 0, c.st>>>(a);
    root_bound_kernel<<<dim3(rb, nb), 256, r.d <= 12288 ? r.d * sizeof(float) : 0, c.st>>>(a);
    root_scalar_kernel<<<(nb + 127) / 128, 128, 0, c.st>>>(a, nb);
    if (r.eng == ENGINE_F64)
      root_init_f64_kernel<<<dim3(tile_blocks(r.d), 1, nb), 256, 0, c.st>>>(a);
    else
      root_init_tc_kernel<<<dim3((r.d + 127) / 128, (r.d + 31) / 32, nb), 256, 0, c.st>>>(a);
    c.h->launches += 5;
    CK(cudaGetLastError());
  }
  return PRECOND_OK;
}

// Streams and events for the iteration stage's branches (created on first use,
// reused by every later call; events recorded under capture become graph edges).
int side_streams(precond_ctx* h, size_t n) {
  while (h->side.size() < n) {
    cudaStream_t s;
    CK(cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking));
    h->side.push_back(s);
  }
  return PRECOND_OK;
}

int next_event(precond_ctx* h, size_t& used, cudaEvent_t* out) {
  if (used == h->sev.size()) {
    cudaEvent_t e;
    CK(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
    h->sev.push_back(e);
  }
  *out = h->sev[used++];
  return PRECOND_OK;
}

// Whether a plan's stages fork onto the handle's side streams: only when no root
// class's products fill the GPU (fewer 128 x 128 tiles than SMs); with full
// products the branches would only compete for the same SMs.  Two streams per
// root class (at least two), created on first use.
int branch_plan(const Ctx& c, bool* br) {
  *br = c.h->branches;
  for (const auto& r : c.P.rc) {
    const long long tn = (r.d + TC_BN - 1) / TC_BN;
    if ((long long)r.roots.size() * tn * (tn + 1) / 2 >= c.h->num_sms) *br = false;
  }
  if (*br) return side_streams(c.h, std::max<size_t>(2, 2 * c.P.rc.size()));
  return PRECOND_OK;
}

// Side streams 0 .. n-1 wait for all work issued so far on the call's stream.
int fork_sides(const Ctx& c, size_t& used, size_t n, cudaEvent_t* ev = nullptr) {
  cudaEvent_t f;
  int rc;
  if ((rc = next_event(c.h, used, &f))) return rc;
  CK(cudaEventRecord(f, c.st));
  for (size_t i = 0; i < n; ++i) CK(cudaStreamWaitEvent(c.h->side[i], f, 0));
  if (ev) *ev = f;
  return PRECOND_OK;
}

// The call's stream waits for all work issued so far on side streams 0 .. n-1.
int join_sides(const Ctx& c, size_t& used, size_t n) {
  for (size_t i = 0; i < n; ++i) {
    cudaEvent_t j;
    int rc;
    if ((rc = next_event(c.h, used, &j))) return rc;
    CK(cudaEventRecord(j, c.h->side[i]));
    CK(cudaStreamWaitEvent(c.st, j, 0));
  }
  return PRECOND_OK;
}

// Newton-Schulz iterations of every root class.  When the products are too small
// to fill the GPU, each class runs on two streams of its own: the M chain (D, F, M') and the X chain (X' = X T).  The X
// update of iteration k waits for M_k (its operand) and the M' product of
// iteration k waits for that X update, so the X product overlaps D and F, the
// convergence flags that M' sets are never seen early by an X update, and the
// classes (different d) overlap one another.
int launch_iterations(const Ctx& c, bool br, size_t& used) {
  c.h->in_ns = true;
  c.h->gemm_ev_used = 0;
  struct Guard { precond_ctx* h; ~Guard() { h->in_ns = false; } } guard{c.h};
  const int p = c.P.p;
  const size_t ncls = c.P.rc.size();
  int kall = 0;
  for (const auto& r : c.P.rc) kall = std::max(kall, r.kmax);
  int rcode;
  cudaEvent_t fork = nullptr;
  if (br && (rcode = fork_sides(c, used, 2 * ncls, &fork))) return rcode;
  std::vector<cudaEvent_t> mready(ncls, fork);     // per class: M_k sliced
  int64_t n = 0;
  for (int k = 0; k < kall; ++k) {
    for (size_t ri = 0; ri < ncls; ++ri) {
      const RootClass& r = c.P.rc[ri];
      if (k >= r.kmax) continue;
      const int so = (br && r.tc_ord >= 0) ? 1 + 2 * r.tc_ord : 0;       // scratch regions of the side streams
      const Ctx cm{c.h, c.P, c.ws, br ? c.h->side[2 * ri] : c.st, so};           // M chain
      const Ctx cx{c.h, c.P, c.ws, br ? c.h->side[2 * ri + 1] : c.st, so ? so + 1 : 0};   // X chain
      const int nb = (int)r.roots.size(), d = r.d, eng = r.eng;
      const int* root_of = c.at<const int>(r.t_root);
      const int cur = k & 1, nxt = (k + 1) & 1;
      Epi e = base_epi(c, EPI_STORE, d, d);
      e.root_of = root_of;
      e.partials = c.at<double>(c.P.partials);
      e.partials_stride = c.P.max_tiles;
      e.ctl.p = p;
      e.ctl.kmin = c.h->min_iter;
      e.ctl.kmax = r.kmax;
      e.ctl.tol = (float)c.h->tol;
      e.k = k;
      // Identity-free form of  T = tau I - M/p,  tau = (p+1)/p:
      //   p = 2:  T^2 = tau^2 I + D,   D = M M / p^2 - (2 tau / p) M,   M' = tau^2 M + D M
      //   p = 4:  T^2 = tau^2 I + D,   T^4 = tau^4 I + F,   F = D D + 2 tau^2 D,   M' = tau^4 M + F M
      //   X' = X T = tau X - X M / p
      // so every product operand (M, D, F, X) keeps its information in its own
      // digits instead of next to a dominant identity.
      const double al = r.steps.alpha[k], be = r.steps.beta[k];
      auto aff = [&](const Ctx& cc, const Slab& A, const Slab& B, const Slab& In, const Slab& C, double alpha,
                     double beta_in) -> int {
        Epi ea = e;
        ea.kind = EPI_AFF;
        ea.C = cc.plane(C);
        ea.In = cc.plane(In);
        ea.alpha = alpha;
        ea.beta_in = beta_in;
        ea.gamma = 0.0;
        int rc2;
        if ((rc2 = gemm(cc, eng, A, B, d, d, d, nullptr, nullptr, ea, nb, true, &In))) return rc2;
        ++n;
        return PRECOND_OK;
      };
      // T = al I - be M:  T^2 = al^2 I + D, D = be^2 M M - 2 al be M;  T^4 = al^4 I + F,
      // F = D D + 2 al^2 D;  M' = al^p M + (D or F) M;  X' = X T = al X - be X M
      cudaEvent_t xdone = nullptr;
      const double ga = r.steps.gamma[k];
      const Slab* Pk = &r.D;
      if (ga == 0.0) {
        // linear step T = al I - be M
        if (k >= 1) {
          if (br) CK(cudaStreamWaitEvent(cx.st, mready[ri], 0));
          if ((rcode = aff(cx, r.X[cur], r.M[cur], r.X[cur], r.X[nxt], -be, al))) return rcode;
          if (br) {
            if ((rcode = next_event(c.h, used, &xdone))) return rcode;
            CK(cudaEventRecord(xdone, cx.st));
          }
        }
        if ((rcode = aff(cm, r.M[cur], r.M[cur], r.M[cur], r.D, be * be, -2.0 * al * be))) return rcode;
        if (p == 4) {
          if ((rcode = aff(cm, r.D, r.D, r.D, r.F, 1.0, 2.0 * al * al))) return rcode;
          Pk = &r.F;
        }
      } else {
        // quadratic step T = al I + E, E = ga M M - be M (p = 4):  X' = al X + X E,
        // D = E E + 2 al E (= T^2 - al^2 I), F = D D + 2 al^2 D (= T^4 - al^4 I).
        // E lives in F's slab: F is written after the last reads of E.
        const Slab& E = r.F;
        if ((rcode = aff(cm, r.M[cur], r.M[cur], r.M[cur], E, ga, -be))) return rcode;
        if (br) {
          cudaEvent_t eready;
          if ((rcode = next_event(c.h, used, &eready))) return rcode;
          CK(cudaEventRecord(eready, cm.st));
          CK(cudaStreamWaitEvent(cx.st, eready, 0));
        }
        if (k == 0) {            // X_0 = I: X_1 = al I + E_0
          ShiftArgs sa;
          sa.src = cx.plane(E);
          sa.dst = cx.plane(r.X[nxt]);
          sa.root_of = root_of;
          sa.stats = c.stats();
          sa.d = d;
          sa.alpha = (float)al;
          if (eng == ENGINE_F64)
            shift_identity_f64_kernel<<<dim3((unsigned int)std::min((d + 7) / 8, 1024), (unsigned int)nb), 256, 0,
                                        cx.st>>>(sa);
          else
            shift_identity_tc_kernel<<<dim3((d + 127) / 128, (d + 7) / 8, nb), 256, 0, cx.st>>>(sa);
          c.h->launches++;
          CK(cudaGetLastError());
        } else if ((rcode = aff(cx, r.X[cur], E, r.X[cur], r.X[nxt], 1.0, al))) {
          return rcode;
        }
        if (br) {
          if ((rcode = next_event(c.h, used, &xdone))) return rcode;
          CK(cudaEventRecord(xdone, cx.st));
        }
        if ((rcode = aff(cm, E, E, E, r.D, 1.0, 2.0 * al))) return rcode;
        if (xdone) CK(cudaStreamWaitEvent(cm.st, xdone, 0));     // F overwrites E
        if ((rcode = aff(cm, r.D, r.D, r.D, r.F, 1.0, 2.0 * al * al))) return rcode;
        Pk = &r.F;
      }
      Epi em = e;     // M_{k+1} = tau^p M_k + P M_k, residual, convergence
      em.kind = EPI_M;
      em.C = c.plane(r.M[nxt]);
      em.In = c.plane(r.M[cur]);
      em.beta_in = std::pow(al, p);
      if (xdone) CK(cudaStreamWaitEvent(cm.st, xdone, 0));
      // symmetric product (upper-triangle tiles mirrored): M' is exactly symmetric,
      // which also removes the antisymmetric mode the iteration would amplify
      // M' = M P (P = D or F, a polynomial in M: it commits with M), so that the element-wise
      // input M is the product's first operand
      if ((rcode = gemm(cm, eng, r.M[cur], *Pk, d, d, d, nullptr, nullptr, em, nb, true, &r.M[cur])))
        return rcode;
      ++n;
      if (br) {
        if ((rcode = next_event(c.h, used, &mready[ri]))) return rcode;
        CK(cudaEventRecord(mready[ri], cm.st));
      }
    }
  }
  // join every branch back into the caller's stream
  if (br && (rcode = join_sides(c, used, 2 * ncls))) return rcode;
  c.h->ns_launches = n;
  return PRECOND_OK;
}

int launch_finish(const Ctx& c0, float eps, bool br) {
  for (size_t ri = 0; ri < c0.P.rc.size(); ++ri) {
    const RootClass& r = c0.P.rc[ri];
    const Ctx c{c0.h, c0.P, c0.ws, br ? c0.h->side[2 * ri] : c0.st};
    const int nb = (int)r.roots.size();
    RootArgs a = root_args(c, r, eps);
    if (r.eng == ENGINE_F64)
      root_finish_f64_kernel<<<dim3(tile_blocks(r.d), 1, nb), 256, 0, c.st>>>(a);
    else
      root_finish_tc_kernel<<<dim3((r.d + 127) / 128, (r.d + 31) / 32, nb), 256, 0, c.st>>>(a);
    c.h->launches++;
    CK(cudaGetLastError());
  }
  return PRECOND_OK;
}

int record(precond_ctx* h, int i, cudaStream_t st) {
  if (h->timing && h->events) CK(record_event(h, h->ev[i], st));
  return PRECOND_OK;
}

// Start, iterations and finish of every root class, between the stage events 1 and 3.
// With branches each class's start and finish kernels run on its own side stream,
// joined back into the call's stream at the end of each stage.
int run_roots(const Ctx& c, float eps, bool br, size_t& used) {
  const size_t nside = 2 * c.P.rc.size();
  int rc;
  if (br && (rc = fork_sides(c, used, nside))) return rc;
  if ((rc = launch_roots_start(c, eps, br))) return rc;
  if (br && (rc = join_sides(c, used, nside))) return rc;
  if ((rc = record(c.h, 2, c.st))) return rc;
  if ((rc = launch_iterations(c, br, used))) return rc;
  if ((rc = record(c.h, 3, c.st))) return rc;
  if (br && (rc = fork_sides(c, used, nside))) return rc;
  if ((rc = launch_finish(c, eps, br))) return rc;
  if (br && (rc = join_sides(c, used, nside))) return rc;
  return PRECOND_OK;
}

int run_step(precond_ctx* h, const Plan& P, float beta, float eps, cudaStream_t st) {
  Ctx c{h, P, (char*)h->ws, st};
  int rc;
  bool br;
  size_t used = 0;
  if ((rc = branch_plan(c, &br))) return rc;
  // the Gram products fork by side onto side streams 0 and 1, which own scratch regions 1
  // and 2 (a tcgen05 Gram implies a tcgen05 root class, hence those regions)
  const bool gram_br = br && P.scratch_slots >= 3;
  CK(cudaMemsetAsync(c.ws + P.stats, 0, sizeof(RootStat) * P.nroots, st));
  CK(cudaMemsetAsync(c.ws + P.err, 0, 64, st));
  if ((rc = record(h, 0, st))) return rc;
  // ---- preparation + Gram EMA
  for (const auto& s : P.sc) {
    const int nb = (int)s.mats.size();
    PrepArgs a;
    memset(&a, 0, sizeof(a));
    a.g = c.at<const void* const>(s.t_g);
    a.dtype = P.dtype;
    a.m = s.m;
    a.n = s.n;
    a.roots2 = c.at<const int>(s.t_roots2);
    a.stats = c.stats();
    const bool tc = s.eng == ENGINE_TC;
    if (tc) {
      a.G = c.plane(s.Gq);
      a.GT = c.plane(s.GTq);
      prep_tc_kernel<<<dim3((s.n + 127) / 128, (s.m + 127) / 128, nb), 256, PREP_SMEM, st>>>(a);
    } else {
      a.G = c.plane(s.Gd);
      a.GT = c.plane(s.GTd);
      prep_f64_kernel<<<dim3((s.n + 31) / 32, (s.m + 31) / 32, nb), 256, 0, st>>>(a);
    }
    h->launches++;
    CK(cudaGetLastError());
  }
  if (gram_br && (rc = fork_sides(c, used, 2))) return rc;
  for (const auto& s : P.sc) {
    const int nb = (int)s.mats.size();
    const bool tc = s.eng == ENGINE_TC;
    for (int side = 0; side < 2; ++side) {
      const Ctx cg{h, P, c.ws, gram_br ? h->side[side] : st, gram_br ? 1 + side : 0};
      const int dim = side == 0 ? s.m : s.n, K = side == 0 ? s.n : s.m;
      Epi e = base_epi(c, EPI_GRAM, dim, dim);
      e.state = c.at<float* const>(side == 0 ? s.t_L : s.t_R);
      e.state_packed = h->packed;
      e.beta = beta;
      e.nonfinite_of = c.at<const int>(s.t_roots2);
      const Slab& G = tc ? (side == 0 ? s.Gq : s.GTq) : (side == 0 ? s.Gd : s.GTd);
      if ((rc = gemm(cg, s.eng, G, G, dim, dim, K, nullptr, nullptr, e, nb, true))) return rc;
    }
  }
  if (gram_br && (rc = join_sides(c, used, 2))) return rc;
  if ((rc = record(h, 1, st))) return rc;
  if ((rc = run_roots(c, eps, br, used))) return rc;
  // ---- apply: V = G X_R (stored transposed), U = X_L V
  for (const auto& s : P.sc) {
    const int nb = (int)s.mats.size();
    const RootClass& l = P.rc[s.lrc];
    const RootClass& r = P.rc[s.rrc];
    Epi ev = base_epi(c, EPI_VT, s.m, s.n);
    Epi eu = base_epi(c, EPI_U, s.m, s.n);
    eu.out = c.at<void* const>(s.t_out);
    eu.out_dtype = P.out_f32 ? PRECOND_F32 : P.dtype;
    eu.nonfinite_of = c.at<const int>(s.t_roots2);
    const int* lsl = c.at<const int>(s.t_lslot);
    const int* rsl = c.at<const int>(s.t_rslot);
    const bool tc = s.eng == ENGINE_TC;
    const Slab& G = tc ? s.Gq : s.Gd;
    const Slab& VT = tc ? s.VTq : s.VTd;
    ev.C = c.plane(VT);
    if ((rc = gemm(c, s.eng, G, r.Xf, s.m, s.n, s.n, nullptr, rsl, ev, nb, false))) return rc;
    if ((rc = gemm(c, s.eng, l.Xf, VT, s.m, s.n, s.m, lsl, nullptr, eu, nb))) return rc;
  }
  if ((rc = record(h, 4, st))) return rc;
  return PRECOND_OK;
}

int run_inv_root(precond_ctx* h, const Plan& P, float eps, cudaStream_t st) {
  Ctx c{h, P, (char*)h->ws, st};
  int rc;
  bool br;
  size_t used = 0;
  if ((rc = branch_plan(c, &br))) return rc;
  CK(cudaMemsetAsync(c.ws + P.stats, 0, sizeof(RootStat) * P.nroots, st));
  CK(cudaMemsetAsync(c.ws + P.err, 0, 64, st));
  if ((rc = record(h, 0, st))) return rc;
  if ((rc = record(h, 1, st))) return rc;
  if ((rc = run_roots(c, eps, br, used))) return rc;
  if ((rc = record(h, 4, st))) return rc;
  return PRECOND_OK;
}

int prepare_device(precond_ctx* h) {
  CK(cudaSetDevice(h->device));
  if (!h->tc_attr_set) {
    CK(cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, TcSmem::BYTES));
    CK(cudaFuncSetAttribute(prep_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PREP_SMEM));
    CK(cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device));
    h->tc_attr_set = true;
  }
  return PRECOND_OK;
}

void remember(precond_ctx* h, const Plan& P, cudaStream_t st) {
  h->last_stream = st;
  h->last_nroots = P.nroots;
  h->last_p = P.p;
  h->have_last = true;
  h->last_root_d.assign(P.nroots, 0);
  h->last_root_class.assign(P.nroots, -1);
  h->last_root_slot.assign(P.nroots, -1);
  for (size_t ci = 0; ci < P.rc.size(); ++ci)
    for (size_t j = 0; j < P.rc[ci].roots.size(); ++j) {
      const int r = P.rc[ci].roots[j];
      h->last_root_d[r] = P.rc[ci].d;
      h->last_root_class[r] = (int)ci;
      h->last_root_slot[r] = (int)j;
    }
  h->last_plan = P;
}

// Everything a captured step's kernel parameters depend on, except the
// caller's pointers (those live in the uploaded tables).
std::string plan_key(const precond_ctx* h, const Plan& P, float beta, float eps) {
  std::ostringstream k;
  k << P.step << ' ' << P.count << ' ' << P.nroots << ' ' << P.p << ' ' << P.dtype << ' ' << P.out_f32 << ' '
    << P.total << ' ' << P.meta << ' ' << P.meta_bytes << ' ' << P.max_tiles << ' ' << beta << ' ' << eps << ' '
    << h->tol << ' ' << h->min_iter << ' ' << h->timing << ' ' << h->branches << ' ' << h->step_degree << ' ' << h->packed << ' ' << h->tile_split << ' ' << h->ws;
  for (const auto& r : P.rc) {
    k << " r" << r.d << ',' << r.eng << ',' << r.roots.size() << ',' << r.kmax;
    for (size_t i = 0; i < r.steps.alpha.size(); ++i)
      k << ',' << r.steps.alpha[i] << ':' << r.steps.beta[i] << ':' << r.steps.gamma[i];
  }
  for (const auto& c : P.sc) k << " s" << c.m << ',' << c.n << ',' << c.eng << ',' << c.mats.size();
  return k.str();
}

void drop_graph(precond_ctx* h) {
  for (auto& g : h->graphs) cudaGraphExecDestroy(g.exec);
  h->graphs.clear();
}

constexpr size_t kMaxGraphs = 4;     // plans a handle keeps captured (callers with a few parameter groups)

// Run `fn(stream)` for plan P: directly on the caller's stream, or (graphs on)
// as a replay of a graph captured once per plan on the handle's own stream,
// ordered after the caller's earlier work and before its later work.
template <typename Fn>
int run_planned(precond_ctx* h, const Plan& P, float beta, float eps, cudaStream_t st, Fn fn) {
  int rc;
  if (!h->use_graph) {
    if ((rc = upload_meta(h, P, st))) return rc;
    return fn(st);
  }
  if (!h->gstream) {
    CK(cudaStreamCreateWithFlags(&h->gstream, cudaStreamNonBlocking));
    CK(cudaEventCreateWithFlags(&h->gev_in, cudaEventDisableTiming));
    CK(cudaEventCreateWithFlags(&h->gev_out, cudaEventDisableTiming));
  }
  CK(cudaEventRecord(h->gev_in, st));
  CK(cudaStreamWaitEvent(h->gstream, h->gev_in, 0));
  if ((rc = upload_meta(h, P, h->gstream))) return rc;
  const std::string key = plan_key(h, P, beta, eps);
  auto it = h->graphs.begin();
  while (it != h->graphs.end() && !(it->key == key && it->ws == h->ws)) ++it;
  if (it != h->graphs.end()) {
    h->graphs.splice(h->graphs.begin(), h->graphs, it);      // most recently used first
  } else {
    const int64_t l0 = h->launches;
    CK(cudaStreamBeginCapture(h->gstream, cudaStreamCaptureModeThreadLocal));
    h->capturing = true;
    rc = fn(h->gstream);
    h->capturing = false;
    cudaGraph_t g = nullptr;
    const cudaError_t e = cudaStreamEndCapture(h->gstream, &g);
    if (rc || e != cudaSuccess) {
      if (g) cudaGraphDestroy(g);
      cudaGetLastError();
      h->launches = l0;
      return rc ? rc : PRECOND_ECUDA;
    }
    precond_ctx::Graph ge;
    const cudaError_t ei = cudaGraphInstantiate(&ge.exec, g, 0);
    cudaGraphDestroy(g);
    if (ei != cudaSuccess) return PRECOND_ECUDA;
    ge.key = key;
    ge.ws = h->ws;
    ge.kernels = h->launches - l0;
    h->launches = l0;
    ge.ns_launches = h->ns_launches;
    ge.gemm_ev = h->gemm_ev_used;
    h->graphs.push_front(ge);
    while (h->graphs.size() > kMaxGraphs) {
      cudaGraphExecDestroy(h->graphs.back().exec);
      h->graphs.pop_back();
    }
  }
  const precond_ctx::Graph& gr = h->graphs.front();
  CK(cudaGraphLaunch(gr.exec, h->gstream));
  h->launches += gr.kernels;
  h->ns_launches = gr.ns_launches;
  h->gemm_ev_used = gr.gemm_ev;
  CK(cudaEventRecord(h->gev_out, h->gstream));
  CK(cudaStreamWaitEvent(st, h->gev_out, 0));
  return PRECOND_OK;
}

}  // namespace

// =========================================================================== C ABI
extern "C" {

int precond_create(precond_t* out, int cuda_device) {
  if (!out || cuda_device < -1) return PRECOND_EINVAL;
  *out = nullptr;
  precond_ctx* h = new precond_ctx();
  h->device = cuda_device;
  if (cuda_device >= 0) {
    int n = 0;
    if (cudaGetDeviceCount(&n) != cudaSuccess || cuda_device >= n) {
      cudaGetLastError();
      delete h;
      return PRECOND_ECUDA;
    }
    // the SM count sizes the plans' persistent grids and their scratch regions from the first call on
    if (cudaSetDevice(cuda_device) != cudaSuccess ||
        cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, cuda_device) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->upload_done, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      delete h;
      return PRECOND_ECUDA;
    }
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
      cudaGetLastError();
      cudaEventDestroy(h->upload_done);
      delete h;
      return PRECOND_ECUDA;
    }
    h->encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  *out = h;
  return PRECOND_OK;
}

int precond_destroy(precond_t h) {
  if (!h) return PRECOND_OK;
  if (h->device >= 0) {
    cudaSetDevice(h->device);
    cudaDeviceSynchronize();
    if (h->ws) cudaFree(h->ws);
    if (h->pinned) cudaFreeHost(h->pinned);
    if (h->upload_done) cudaEventDestroy(h->upload_done);
    if (h->events)
      for (auto& e : h->ev) cudaEventDestroy(e);
    for (auto& e : h->gemm_ev) cudaEventDestroy(e);
    drop_graph(h);
    for (auto& x : h->side) cudaStreamDestroy(x);
    for (auto& x : h->sev) cudaEventDestroy(x);
    if (h->gstream) cudaStreamDestroy(h->gstream);
    if (h->gev_in) cudaEventDestroy(h->gev_in);
    if (h->gev_out) cudaEventDestroy(h->gev_out);
  }
  delete h;
  return PRECOND_OK;
}

int precond_set_option(precond_t h, int key, double v) {
  if (!h) return PRECOND_EINVAL;
  switch (key) {
    case PRECOND_OPT_TOL:
      if (!(v > 0) || !std::isfinite(v)) return PRECOND_EINVAL;
      h->tol = v;
      return PRECOND_OK;
    case PRECOND_OPT_MAX_ITER:
      if (v < 0 || v > 1000 || v != std::floor(v)) return PRECOND_EINVAL;
      h->max_iter = (int)v;
      return PRECOND_OK;
    case PRECOND_OPT_MIN_ITER:
      if (v < 1 || v > 1000 || v != std::floor(v)) return PRECOND_EINVAL;
      h->min_iter = (int)v;
      return PRECOND_OK;
    case PRECOND_OPT_ENGINE:
      if (v != 0 && v != 1 && v != 2) return PRECOND_EINVAL;
      h->engine = (int)v;
      return PRECOND_OK;
    case PRECOND_OPT_SMALL_DIM:
      if (v < 0 || v > 1e9 || v != std::floor(v)) return PRECOND_EINVAL;
      h->small_dim = (int)v;
      return PRECOND_OK;
    case PRECOND_OPT_WORKSPACE_MAX:
      if (v < 0 || !std::isfinite(v)) return PRECOND_EINVAL;
      h->ws_max = v;
      return PRECOND_OK;
    case PRECOND_OPT_TIMING:
      if (v != 0 && v != 1 && v != 2) return PRECOND_EINVAL;
      if (v != 0 && h->device >= 0 && !h->events) {
        for (auto& e : h->ev)
          if (cudaEventCreate(&e) != cudaSuccess) return PRECOND_ECUDA;
        h->events = true;
      }
      h->timing = (int)v;
      return PRECOND_OK;
    case PRECOND_OPT_FOLD:
      if (!(v >= 0.0 && v < 1.0)) return PRECOND_EINVAL;
      h->fold = v;
      return PRECOND_OK;
    case PRECOND_OPT_CLASSICAL:
      if (v != 0 && v != 1) return PRECOND_EINVAL;
      h->classical = (int)v;
      return PRECOND_OK;
    case PRECOND_OPT_USE_GRAPH:
      if (v != 0 && v != 1) return PRECOND_EINVAL;
      h->use_graph = (int)v;
      return PRECOND_OK;
    case PRECOND_OPT_PACKED_STATE:
      if (v != 0 && v != 1) return PRECOND_EINVAL;
      h->packed = (int)v;
      return PRECOND_OK;
    case PRECOND_OPT_STEP_DEGREE:
      if (v != 1 && v != 2) return PRECOND_EINVAL;
      h->step_degree = (int)v;
      return PRECOND_OK;
    case PRECOND_OPT_BRANCHES:
      if (v != 0 && v != 1) return PRECOND_EINVAL;
      h->branches = v != 0;
      return PRECOND_OK;
    case PRECOND_OPT_TILE_SPLIT:
      if (v != 1 && v != 2 && v != 4) return PRECOND_EINVAL;
      h->tile_split = (int)v;
      return PRECOND_OK;
  }
  return PRECOND_EINVAL;
}

int precond_step(precond_t h, int count, void* const grads[], int grad_dtype, const int64_t shapes[],
                 float* const L[], float* const R[], float beta, float eps, float power,
                 float* const out_f32[], void* stream) {
  if (!h || count < 1 || !grads || !shapes || !L || !R) return PRECOND_EINVAL;
  if (grad_dtype != PRECOND_F32 && grad_dtype != PRECOND_BF16) return PRECOND_EINVAL;
  if (!(beta >= 0.f && beta < 1.f)) return PRECOND_EINVAL;
  if (!(eps > 0.f) || !std::isfinite(eps)) return PRECOND_EINVAL;
  int p;
  if (check_power(power, &p)) return PRECOND_EINVAL;
  std::vector<const void*> state;
  for (int i = 0; i < count; ++i) {
    if (shapes[2 * i] < 1 || shapes[2 * i + 1] < 1 || shapes[2 * i] > (1 << 20) || shapes[2 * i + 1] > (1 << 20))
      return PRECOND_EINVAL;
    if (!grads[i] || !L[i] || !R[i] || (out_f32 && !out_f32[i])) return PRECOND_EINVAL;
    state.push_back(L[i]);
    state.push_back(R[i]);
  }
  std::vector<const void*> sorted = state;
  std::sort(sorted.begin(), sorted.end());
  if (std::adjacent_find(sorted.begin(), sorted.end()) != sorted.end()) return PRECOND_EINVAL;
  Plan P;
  int rc = build_plan(h, P, true, count, shapes, grad_dtype, eps, p, grads, L, R, out_f32, nullptr, nullptr);
  if (rc) return rc;
  h->planned_bytes = P.total;
  if (h->ws_max > 0 && (double)P.total > h->ws_max) return PRECOND_ENOMEM;
  if (h->device < 0) return PRECOND_ENODEV;
  if ((rc = prepare_device(h))) return rc;
  if ((rc = ensure_workspace(h, P.total))) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  if ((rc = run_planned(h, P, beta, eps, st, [&](cudaStream_t s2) { return run_step(h, P, beta, eps, s2); })))
    return rc;
  remember(h, P, st);
  return PRECOND_OK;
}

int precond_inv_root(precond_t h, int count, const float* const A[], const int64_t dims[], float eps,
                     float power, float* const X[], void* stream) {
  if (!h || count < 1 || !A || !dims || !X) return PRECOND_EINVAL;
  if (!(eps > 0.f) || !std::isfinite(eps)) return PRECOND_EINVAL;
  int p;
  if (check_power(power, &p)) return PRECOND_EINVAL;
  for (int i = 0; i < count; ++i) {
    if (dims[i] < 1 || dims[i] > (1 << 20) || !A[i] || !X[i]) return PRECOND_EINVAL;
    if ((const void*)A[i] == (const void*)X[i]) return PRECOND_EINVAL;
  }
  Plan P;
  int rc = build_plan(h, P, false, count, dims, PRECOND_F32, eps, p, nullptr, nullptr, nullptr, nullptr, A, X);
  if (rc) return rc;
  h->planned_bytes = P.total;
  if (h->ws_max > 0 && (double)P.total > h->ws_max) return PRECOND_ENOMEM;
  if (h->device < 0) return PRECOND_ENODEV;
  if ((rc = prepare_device(h))) return rc;
  if ((rc = ensure_workspace(h, P.total))) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  if ((rc = run_planned(h, P, 0.f, eps, st, [&](cudaStream_t s2) { return run_inv_root(h, P, eps, s2); })))
    return rc;
  remember(h, P, st);
  return PRECOND_OK;
}

int precond_get_stats(precond_t h, int nroots, int iters[], float resid[], int status[], float scale[]) {
  if (!h) return PRECOND_EINVAL;
  if (h->device < 0) return PRECOND_ENODEV;
  if (!h->have_last || nroots != h->last_nroots) return PRECOND_EINVAL;
  CK(cudaSetDevice(h->device));
  CK(cudaStreamSynchronize(h->last_stream));
  std::vector<RootStat> st(nroots);
  unsigned int err = 0;
  CK(cudaMemcpy(st.data(), (char*)h->ws + h->last_plan.stats, sizeof(RootStat) * nroots, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(&err, (char*)h->ws + h->last_plan.err, sizeof(err), cudaMemcpyDeviceToHost));
  for (int r = 0; r < nroots; ++r) {
    if (iters) iters[r] = st[r].iters;
    if (resid) resid[r] = (float)st[r].resid;
    if (status) status[r] = st[r].status;
    if (scale) scale[r] = (float)st[r].c;
  }
  if (err) {
    fprintf(stderr, "libprecond: a device wait timed out (error word %u)\n", err);
    return PRECOND_ECUDA;
  }
  return PRECOND_OK;
}

int precond_get_timing(precond_t h, double ms[4], int64_t* ns_gemm_launches, double* ns_flops) {
  if (!h) return PRECOND_EINVAL;
  if (h->device < 0) return PRECOND_ENODEV;
  if (!h->have_last || !h->timing || !h->events) return PRECOND_EINVAL;
  CK(cudaEventSynchronize(h->ev[4]));
  if (ms)
    for (int i = 0; i < 4; ++i) {
      float t = 0.f;
      CK(cudaEventElapsedTime(&t, h->ev[i], h->ev[i + 1]));
      ms[i] = t;
    }
  if (ns_gemm_launches) *ns_gemm_launches = h->ns_launches;
  if (ns_flops) {
    std::vector<RootStat> st(h->last_nroots);
    CK(cudaMemcpy(st.data(), (char*)h->ws + h->last_plan.stats, sizeof(RootStat) * h->last_nroots,
                  cudaMemcpyDeviceToHost));
    // products per iteration: 3 (p = 2) or 4 (p = 4) for a linear step, 5 for a
    // quadratic one; iteration 0 has one fewer (X_1 is formed element-wise)
    const int g = h->last_p == 4 ? 4 : 3;
    double f = 0;
    for (int r = 0; r < h->last_nroots; ++r) {
      const double d = h->last_root_d[r];
      const StepPoly& sp = h->last_plan.rc[h->last_root_class[r]].steps;
      long long prods = 0;
      for (int k = 0; k < st[r].iters && k < (int)sp.gamma.size(); ++k)
        prods += (sp.gamma[k] != 0.0 ? 5 : g) - (k == 0 ? 1 : 0);
      f += 2.0 * d * d * d * (double)prods;
    }
    *ns_flops = f;
  }
  return PRECOND_OK;
}

int64_t precond_launch_count(precond_t h) { return h ? h->launches : -1; }

int precond_get_workspace(precond_t h, int64_t* planned, int64_t* allocated) {
  if (!h) return PRECOND_EINVAL;
  if (planned) *planned = (int64_t)h->planned_bytes;
  if (allocated) *allocated = (int64_t)h->ws_cap;
  return PRECOND_OK;
}

int precond_get_gemm_timing(precond_t h, double* ms_total, int64_t* launches, double* issued_flops) {
  if (!h) return PRECOND_EINVAL;
  if (h->device < 0) return PRECOND_ENODEV;
  if (!h->have_last || !h->timing || !h->events) return PRECOND_EINVAL;
  CK(cudaEventSynchronize(h->ev[4]));
  double t = -1.0;                  // mode 2: no per-launch events
  if (h->timing == 1) {
    t = 0.0;
    for (size_t i = 0; i + 1 < h->gemm_ev_used; i += 2) {
      float x = 0.f;
      CK(cudaEventElapsedTime(&x, h->gemm_ev[i], h->gemm_ev[i + 1]));
      t += x;
    }
  }
  if (ms_total) *ms_total = t;
  if (launches) *launches = h->timing == 1 ? (int64_t)(h->gemm_ev_used / 2) : (int64_t)h->ns_launches;
  if (issued_flops) {
    unsigned long long n = 0;   // (K blocks x digit pairs) of the computed tiles, counted on the device
    CK(cudaMemcpy(&n, (char*)h->ws + h->last_plan.err + 8, sizeof(n), cudaMemcpyDeviceToHost));
    *issued_flops = (double)n * 2.0 * TC_BM * TC_BN * TC_BK;
  }
  return PRECOND_OK;
}

int precond_step_schedule(int p, double l0, double fold, int degree, int max_steps, double* alpha, double* beta,
                          double* gamma, double* lo, int* nsteps) {
  if ((p != 2 && p != 4) || (degree != 1 && degree != 2) || !(l0 > 0.0 && l0 < 1.0) || !(fold >= 0.0 && fold < 1.0) ||
      max_steps < 1 || !alpha || !beta || !gamma || !lo || !nsteps)
    return PRECOND_EINVAL;
  const StepPoly sp = degree == 2 ? step_schedule_quad(l0, p, max_steps, fold) : step_schedule(l0, p, max_steps, fold);
  const int n = std::min((int)sp.alpha.size(), max_steps);
  for (int i = 0; i < n; ++i) {
    alpha[i] = sp.alpha[i];
    beta[i] = sp.beta[i];
    gamma[i] = sp.gamma[i];
    lo[i] = sp.lo[i];
  }
  *nsteps = n;
  return PRECOND_OK;
}

const char* precond_error_string(int code) {
  switch (code) {
    case PRECOND_OK: return "ok";
    case PRECOND_EINVAL: return "invalid argument";
    case PRECOND_ENOMEM: return "workspace allocation failed or exceeds the limit";
    case PRECOND_ECUDA: return "CUDA error";
    case PRECOND_ENODEV: return "host-only handle: no device";
    case PRECOND_ENOTCONV: return "iteration did not reach the tolerance";
    case PRECOND_ENONFINITE: return "non-finite input";
  }
  return "unknown status";
}

// Test / debug read-back: the fp32 root of root `r` of the last step call
// (X_L for root 2i, X_R for root 2i+1) into a d x d device buffer.
int precond_get_root(precond_t h, int r, float* dst, void* stream) {
  if (!h || !dst) return PRECOND_EINVAL;
  if (h->device < 0) return PRECOND_ENODEV;
  if (!h->have_last || r < 0 || r >= h->last_nroots) return PRECOND_EINVAL;
  const RootClass& rc = h->last_plan.rc[h->last_root_class[r]];
  const int slot = h->last_root_slot[r];
  Plane p = slab_plane((char*)h->ws, rc.Xf);
  cudaStream_t st = (cudaStream_t)stream;
  if (rc.eng == ENGINE_F64) plane_to_f32_kernel<ENGINE_F64><<<256, 256, 0, st>>>(p, slot, rc.d, rc.d, dst);
  else plane_to_f32_kernel<ENGINE_TC><<<256, 256, 0, st>>>(p, slot, rc.d, rc.d, dst);
  h->launches++;
  CK(cudaGetLastError());
  return PRECOND_OK;
}

// Diagnostic read-back of a work matrix of root `r` of the last call:
// which = 0/1 X[0]/X[1], 2/3 M[0]/M[1], 4 D, 5 F, 8 final X.
int precond_debug_plane(precond_t h, int r, int which, float* dst, void* stream) {
  if (!h || !dst || which < 0 || which > 8 || which == 6 || which == 7) return PRECOND_EINVAL;
  if (h->device < 0) return PRECOND_ENODEV;
  if (!h->have_last || r < 0 || r >= h->last_nroots) return PRECOND_EINVAL;
  const RootClass& rc = h->last_plan.rc[h->last_root_class[r]];
  const Slab* sl[9] = {&rc.X[0], &rc.X[1], &rc.M[0], &rc.M[1], &rc.D, &rc.F, nullptr, nullptr, &rc.Xf};
  const Slab& S = *sl[which];
  if (S.batch == 0) return PRECOND_EINVAL;
  Plane p = slab_plane((char*)h->ws, S);
  cudaStream_t st = (cudaStream_t)stream;
  const int slot = h->last_root_slot[r];
  if (rc.eng == ENGINE_F64) plane_to_f32_kernel<ENGINE_F64><<<256, 256, 0, st>>>(p, slot, rc.d, rc.d, dst);
  else plane_to_f32_kernel<ENGINE_TC><<<256, 256, 0, st>>>(p, slot, rc.d, rc.d, dst);
  CK(cudaGetLastError());
  return PRECOND_OK;
}

// Self-test of the GEMM core: C = A . B^T (A: M x K, B: N x K, C: M x N, fp32
// device buffers) through one engine's batched GEMM with a plain store.
int precond_gemm_selftest(precond_t h, int engine, int M, int N, int K, const float* A, const float* B, float* C,
                          int passes, void* stream) {
  if (!h || !A || !B || !C || M < 1 || N < 1 || K < 1 || (engine != 1 && engine != 2)) return PRECOND_EINVAL;
  if (engine == 2 && passes != DIGITS) return PRECOND_EINVAL;
  if (h->device < 0) return PRECOND_ENODEV;
  int rc;
  if ((rc = prepare_device(h))) return rc;
  const int eng = engine == 1 ? ENGINE_F64 : ENGINE_TC;
  Layout L;
  Plan P;
  P.stats = L.take(sizeof(RootStat));
  P.err = L.take(64);
  Slab sa = make_slab(L, eng, 1, M, K), sb = make_slab(L, eng, 1, N, K);
  if (eng == ENGINE_TC) {
    P.scratch_slots = 1;
    P.scratch_ctas = std::min<long long>((long long)((M + TC_BM - 1) / TC_BM) * ((N + TC_BN - 1) / TC_BN) * h->tile_split,
                                         h->num_sms);
    P.scratch_slot_bytes = (size_t)P.scratch_ctas * 2 * TC_BM * TC_BN * sizeof(float);
    P.scratch = L.take(P.scratch_slot_bytes);
  }
  if ((rc = ensure_workspace(h, L.top))) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  Ctx c{h, P, (char*)h->ws, st};
  CK(cudaMemsetAsync(c.ws + P.stats, 0, sizeof(RootStat), st));
  CK(cudaMemsetAsync(c.ws + P.err, 0, 64, st));
  if (eng == ENGINE_F64) {
    f32_to_f64_kernel<<<256, 256, 0, st>>>(A, c.plane(sa), M, K);
    f32_to_f64_kernel<<<256, 256, 0, st>>>(B, c.plane(sb), N, K);
  } else {
    f32_to_tc_kernel<<<dim3((K + 127) / 128, (M + 7) / 8), 256, 0, st>>>(A, c.plane(sa), M, K);
    f32_to_tc_kernel<<<dim3((K + 127) / 128, (N + 7) / 8), 256, 0, st>>>(B, c.plane(sb), N, K);
  }
  Epi e = base_epi(c, EPI_STORE, M, N);
  e.f32out = C;
  if ((rc = gemm(c, eng, sa, sb, M, N, K, nullptr, nullptr, e, 1))) return rc;
  CK(cudaGetLastError());
  CK(cudaStreamSynchronize(st));
  unsigned int err = 0;
  CK(cudaMemcpy(&err, c.ws + P.err, sizeof(err), cudaMemcpyDeviceToHost));
  return err ? PRECOND_ECUDA : PRECOND_OK;
}

}  // extern "C"

// ===========================================================================
// Allocation-free inverse root.
//
// Some callers cannot allocate device memory at the point where they need a
// root: code running inside a pool-allocator hook, a host callback, or an
// embedding runtime that forbids cudaMalloc after start-up (it would
// synchronise the device or break a memory budget fixed in advance).  For
// them, precond_inv_root_noalloc runs the fp64-engine inverse root of ONE
// matrix (side d <= PRECOND_NOALLOC_MAX_D) with all scratch in a fixed
// file-scope device array, so the call itself allocates nothing.
// ===========================================================================
namespace {
constexpr size_t NOALLOC_BYTES = (size_t)4 << 20;   // 4 MiB, held by every GPU that loads the library
constexpr int NOALLOC_MAX_DEVICES = 64;
}  // namespace

// The scratch itself.  In host code this name is only a host-side stand-in:
// its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_BYTES];

namespace {
struct NoAllocSlots {
  std::mutex mu;
  void* addr[NOALLOC_MAX_DEVICES] = {};
};
NoAllocSlots& noalloc_slots() {
  static NoAllocSlots s;
  return s;
}

struct MetaBlob {   // the call's pointer / index tables, passed by value (no staging buffer)
  unsigned char bytes[512];
  int n;
};
__global__ void noalloc_meta_kernel(MetaBlob blob, unsigned char* dst) {
  for (int i = threadIdx.x; i < blob.n; i += blockDim.x) dst[i] = blob.bytes[i];
}
}  // namespace

extern "C" int precond_inv_root_noalloc(const float* A, int64_t d, float eps, float power, float* X,
                                        void* stream, int* status) {
  if (!A || !X || (const void*)A == (const void*)X || d < 1) return PRECOND_EINVAL;
  if (d > PRECOND_NOALLOC_MAX_D) {
    fprintf(stderr, "libprecond: precond_inv_root_noalloc: d = %lld exceeds the fixed scratch limit %d\n",
            (long long)d, PRECOND_NOALLOC_MAX_D);
    return PRECOND_EINVAL;
  }
  if (!(eps > 0.f) || !std::isfinite(eps)) return PRECOND_EINVAL;
  int p;
  if (check_power(power, &p)) return PRECOND_EINVAL;
  int dev = -1;
  CK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return PRECOND_ECUDA;
  // One-time set-up per device (with that device current): the device address
  // of the scratch array.  This first call must not be made during a stream capture.
  void* scratch = nullptr;
  {
    NoAllocSlots& s = noalloc_slots();
    std::lock_guard<std::mutex> lock(s.mu);
    if (!s.addr[dev]) {
      void* ptr = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
      if (e != cudaSuccess || !ptr) {
        fprintf(stderr, "libprecond: cudaGetSymbolAddress of the scratch failed: %s\n", cudaGetErrorString(e));
        return PRECOND_ECUDA;
      }
      s.addr[dev] = ptr;
    }
    scratch = s.addr[dev];
  }
  precond_ctx h;          // options only; its workspace points at the scratch
  h.device = dev;
  h.engine = 1;           // fp64 engine
  h.branches = false;     // no streams or events of its own: everything on the call's stream
  Plan P;
  const int64_t dims[1] = {d};
  const float* As[1] = {A};
  float* Xs[1] = {X};
  int rc = build_plan(&h, P, false, 1, dims, PRECOND_F32, eps, p, nullptr, nullptr, nullptr, nullptr, As, Xs);
  if (rc) return rc;
  if (P.total > NOALLOC_BYTES || P.meta_bytes > sizeof(MetaBlob::bytes)) return PRECOND_ENOMEM;
  h.ws = scratch;
  h.ws_cap = NOALLOC_BYTES;
  cudaStream_t st = (cudaStream_t)stream;
  MetaBlob blob;
  memcpy(blob.bytes, P.meta_host.data(), P.meta_bytes);
  blob.n = (int)P.meta_bytes;
  noalloc_meta_kernel<<<1, 128, 0, st>>>(blob, (unsigned char*)scratch + P.meta);
  CK(cudaGetLastError());
  rc = run_inv_root(&h, P, eps, st);   // clears the per-root state it accumulates into
  h.ws = nullptr;
  if (rc) return rc;
  if (status) {
    CK(cudaStreamSynchronize(st));
    RootStat rs;
    unsigned int err = 0;
    CK(cudaMemcpy(&rs, (char*)scratch + P.stats, sizeof(rs), cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(&err, (char*)scratch + P.err, sizeof(err), cudaMemcpyDeviceToHost));
    *status = rs.status;
    if (err) return PRECOND_ECUDA;
  }
  return PRECOND_OK;
}
