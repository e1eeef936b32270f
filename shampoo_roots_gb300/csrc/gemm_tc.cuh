// tcgen05 batched GEMM of the large-matrix engine (sm_103a):  C_b = A_b . B_b^T
//
// Operands are in the engine's digit form (engine.cuh): three bf16 planes
// P1 + P2 + P3 and a power-of-two scale per (row, 128-column block).  For one
// K chunk c (the 128 columns of scale block c) and one output element,
//
//   sum_{k in c} a_ik b_jk = sigma_A(i,c) sigma_B(j,c) 2^-16 (S0 + S1),
//   S0 = sum P1 Q1,   S1 = sum (P1 Q2 + P2 Q1) + (P1 Q3 + P2 Q2 + P3 Q1).
//
// Every digit product is exact in bf16 x bf16 -> fp32.  S0 is a sum of 128
// integers of magnitude <= 2^16, so it stays below 2^24 and its fp32
// tensor-memory accumulation is EXACT (on this GPU the accumulation truncates,
// which would otherwise bias a long chain); S1 lies 2^-9 below S0 and its own
// rounding is about 2^-33 of the chunk's scale.  Pairs with s + t > 4 (2^-27
// of the scale and below) are dropped: 6 MMAs per K step.  Two tensor-memory
// buffers hold (S0, S1) of two chunks; the drain warps read a finished chunk
// back (tcgen05.ld), weight it with sigma_A(i,c) sigma_B(j,c) and add it to fp32
// sums in registers while the MMAs of the next chunk run.
//
// Pipeline: TMA (3-D tensor maps {K, rows, batch}, 64-byte swizzle, K block 32)
// into a 3-stage shared-memory ring; one elected thread issues tcgen05.mma
// (kind::f16, bf16, M = N = 128, K = 16).  Warp roles (320 threads): warp 0 TMA
// producer, warp 1 TMEM owner and MMA issuer, warps 2..9 drain and epilogue (two
// per tensor-memory lane quadrant, 64 columns each).
//
// The epilogue forms the output element (the product plus the element-wise
// terms) and writes it in its consumer's format: digits with the tile's
// per-(row, block) scales for products that feed further products (and the
// mirrored tile for symmetric products, so results are exactly symmetric), the
// caller's fp32 state for the Gram EMA, or the caller's update.  Digit tiles go
// in and out through one 32 KB shared staging tile, one digit plane at a time,
// moved by TMA (128-byte swizzle): the element-wise input is loaded by TMA
// (prefetched into L2 when the tile starts) and every output plane is stored by
// TMA, so no warp issues row-scattered global accesses.
//
// Every mbarrier wait is bounded.  On a time-out the kernel records an error
// word and raises a shared abort flag: every other wait then gives up at once,
// the roles leave their loops together, and the kernel returns.
#pragma once

#include <cuda.h>
#include "engine.cuh"

namespace precond {

constexpr int TC_BM = 128, TC_BN = 128, TC_BK = 32;
constexpr int TC_CHUNK_KB = DIG_BLK / TC_BK;       // K blocks per chunk (4)
constexpr int TC_PAIRS = 6;                        // digit products per K step
constexpr int EPI_WARPS = 8;                       // two per tensor-memory lane quadrant
constexpr int TC_THREADS = 64 + 32 * EPI_WARPS;    // producer warp, MMA warp, epilogue warps
constexpr unsigned long long TC_WAIT_CYCLES = 4000000000ull;   // ~2 s at 2 GHz

struct TcGemmArgs {
  int M, N, K;
  int batch;             // batch entries (z extent of the tile space)
  int sym;               // 1: the product is symmetric (M == N): compute tiles with row block <=
                         //    column block only and write each off-diagonal tile mirrored too
  const int* a_index;    // batch entry -> z coordinate of A (null: b)
  const int* b_index;    // batch entry -> z coordinate of B (null: b)
  // operand block scales [z][chunk][srows] (A rows = output rows, B rows = output columns)
  const float* a_scale; long long a_sbstride; int a_srows;
  const float* b_scale; long long b_sbstride; int b_srows;
  unsigned int* err;     // error word (bit 0: a wait timed out)
  unsigned long long* issued;   // may be null: += (K blocks x digit pairs) of every tile computed
};

struct TcSmem {
  static constexpr int PLANE_BYTES = TC_BM * TC_BK * 2;                 // 8 KB (A and B tiles alike)
  static constexpr int STAGE_BYTES = 2 * DIGITS * PLANE_BYTES;          // 48 KB
  static constexpr int STAGES = 3;
  static constexpr int RING = STAGES * STAGE_BYTES;
  static constexpr int OFF_STG = RING;                                  // staging: 3 planes x 2 boxes of 64 x 64 bf16
  static constexpr int STG_BYTES = DIGITS * TC_BM * 64 * 2;             // 48 KB: half a tile, all planes
  static constexpr int XP_LD = 17;                                      // transpose scratch row (floats)
  static constexpr int XP_FLOATS = 32 * XP_LD;                          // per epilogue warp
  static constexpr int OFF_XP = OFF_STG + STG_BYTES;
  static constexpr int OFF_SB = OFF_XP + EPI_WARPS * XP_FLOATS * 4;     // per warp: B scales of 2 chunks
  static constexpr int OFF_RMAX = OFF_SB + EPI_WARPS * 128 * 4;         // [2 halves][128 rows]
  static constexpr int OFF_CMAX = OFF_RMAX + 2 * TC_BM * 4;             // [4 quadrants][128 columns]
  static constexpr int OFF_RED = OFF_CMAX + 4 * TC_BN * 4;              // [8] doubles
  static constexpr int OFF_BAR = OFF_RED + EPI_WARPS * 8;
  static constexpr int BAR_BYTES = 256;
  static constexpr int BYTES = 1024 /*align*/ + OFF_BAR + BAR_BYTES;
  static constexpr int TMEM_COLS = 512;                                 // 2 chunk buffers x (S0, S1) x 128
};

// ----------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}
// Bounded wait; gives up at once when another role has aborted, and on its own
// time-out flags `err` and the abort word.  Returns false when it gave up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned int* err, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > TC_WAIT_CYCLES) {
      if (err) atomicOr(err, 1u);
      *abort_flag = 1;
      return false;
    }
  }
  return true;
}
// Bounded wait with no abort check: for work that completes by itself (bulk
// copies and MMAs already issued) and must end before the kernel exits.
__device__ __forceinline__ bool mbar_wait_own(uint32_t bar, uint32_t parity, unsigned int* err) {
  const unsigned long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > TC_WAIT_CYCLES) {
      if (err) atomicOr(err, 1u);
      return false;
    }
  }
  return true;
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}
// TMA store of a box from shared memory (bulk group), its commit and waits.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(x), "r"(y), "r"(z) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Order this thread's generic shared-memory accesses before later async-proxy (TMA) ones.
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global [%0, {%1, %2, %3}];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z) : "memory");
}
// Staging area of one epilogue round: digit plane p, box bx (two TMA boxes of
// {64 columns, 64 rows} per plane, 8 KB each), row rr < 64 of the box; the
// 16-byte chunks of a 128-byte row are XOR-swizzled by rr % 8 (the layout of a
// TMA box with 128-byte swizzle).  Offset of the chunk holding column cc < 64.
__device__ __forceinline__ uint32_t stg_chunk(int p, int bx, int rr, int cc) {
  return (uint32_t)(p * 16384 + bx * 8192 + rr * 128 + (((cc >> 3) ^ (rr & 7)) << 4));
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Shared-memory matrix descriptor: K-major, 64-byte swizzle (rows of 64 B),
// 8-row groups 512 B apart.
__device__ __forceinline__ uint64_t sw64_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);          // start address
  d |= (uint64_t)1 << 16;                           // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(512 >> 4) << 32;                  // stride byte offset
  d |= (uint64_t)1 << 46;                           // descriptor version (tcgen05)
  d |= (uint64_t)4 << 61;                           // swizzle mode: 64 B
  return d;
}
// Instruction descriptor, kind::f16 with bf16 A and B: fp32 accumulate,
// K-major A and B, M = 128, N = 128.
__host__ __device__ constexpr uint32_t tc_idesc() {
  return (1u << 4)                                  // D format f32
       | (1u << 7) | (1u << 10)                     // A, B format bf16
       | ((uint32_t)(TC_BN >> 3) << 17)             // N / 8
       | ((uint32_t)(TC_BM >> 4) << 24);            // M / 16
}
__device__ __forceinline__ void tc_mma(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
      ::"r"(tmem_d), "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32"
      " {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// 16 consecutive fp32 columns of this warp's 32 lanes.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32"
      " {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// The value of x, opaque to the compiler: keeps per-round work inside its round
// (otherwise the digits of all 64 values of a thread are hoisted out of the
// round loop and held at once, far beyond the register budget).
__device__ __forceinline__ float opaque(float x) {
  float y;
  asm volatile("mov.b32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }   // the 8 epilogue warps
// Barrier of the 8 epilogue warps that also returns the OR of `v` over them (a
// decision every epilogue thread takes the same way).
__device__ __forceinline__ bool epi_bar_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n"
      " bar.red.or.pred p, 1, 256, q;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r) : "r"((uint32_t)v) : "memory");
  return r != 0;
}

// Digit-pair schedule (0-based digit indices): pair 0 is level 0 (accumulator
// S0), pairs 1..5 are levels 1 and 2 (accumulator S1).
__host__ __device__ constexpr int pair_a(int i) { return i == 0 ? 0 : i == 1 ? 0 : i == 2 ? 1 : i == 3 ? 0 : i == 4 ? 1 : 2; }
__host__ __device__ constexpr int pair_b(int i) { return i == 0 ? 0 : i == 1 ? 1 : i == 2 ? 0 : i == 3 ? 2 : i == 4 ? 1 : 0; }

// ----------------------------------------------------------------- kernel
// Tensor maps: digit plane s of A is a[s], of B is b[s] (boxes {32, 128}, 64-byte
// swizzle); of the output c[s] and of the element-wise input in[s] (boxes
// {64, 128}, 128-byte swizzle; zero when the epilogue has none).
struct TcMaps {
  CUtensorMap a[DIGITS];
  CUtensorMap b[DIGITS];
  CUtensorMap c[DIGITS];
  CUtensorMap in[DIGITS];
};

// Tile order within one batch entry: groups of TC_GROUP tile-rows, and inside a
// group column by column (rows fastest), so that the tiles in flight at once
// (one per SM) share a few row panels and column panels that stay in L2.
// Symmetric products enumerate the upper triangle (ti <= tj) only; the group's
// diagonal block comes first (column c holds c + 1 of its rows), then full
// columns of the group's rows.
constexpr int TC_GROUP = 8;

__host__ __device__ __forceinline__ void tile_coords(int tl, int tiles_m, int tiles_n, int sym, int& ti, int& tj) {
  if (!sym) {
    const int per_group = TC_GROUP * tiles_n;
    const int g = tl / per_group, first = g * TC_GROUP;
    const int gm = min(tiles_m - first, TC_GROUP);
    const int loc = tl - g * per_group;
    ti = first + loc % gm;
    tj = loc / gm;
    return;
  }
  int first = 0;
  for (;;) {                                   // find the group holding tl
    const int gm = min(tiles_n - first, TC_GROUP);
    const int diag = gm * (gm + 1) / 2;
    const int count = diag + (tiles_n - first - gm) * gm;
    if (tl < count) {
      if (tl < diag) {
        int c = 0;
        while ((c + 1) * (c + 2) / 2 <= tl) ++c;
        tj = first + c;
        ti = first + (tl - c * (c + 1) / 2);
      } else {
        const int loc = tl - diag;
        tj = first + gm + loc / gm;
        ti = first + loc % gm;
      }
      return;
    }
    tl -= count;
    first += gm;
  }
}

// Digit p (0, 1, 2) of v with 1 / sigma = inv (engine.cuh digits3), selected without indexing.
__device__ __forceinline__ float digit_p(float v, float inv, int p) {
  float d1, d2, d3;
  digits3(v, inv, d1, d2, d3);
  return p == 0 ? d1 : (p == 1 ? d2 : d3);
}

// 16 bf16 words (8 x uint32) -> 16 floats.
__device__ __forceinline__ void unpack16(const uint4 (&w)[2], float (&f)[16]) {
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const uint32_t x = (u < 4) ? (&w[0].x)[u] : (&w[1].x)[u - 4];
    f[2 * u] = __uint_as_float(x << 16);
    f[2 * u + 1] = __uint_as_float(x & 0xFFFF0000u);
  }
}

// Write 16 consecutive values of one output row as digits (scale `inv` = 1/sigma):
// full 32-byte pieces per plane, or element by element where `mask` excludes some.
__device__ __forceinline__ void store_digits16(const Plane& p, long long o, const float (&v)[16], float inv,
                                               uint32_t mask) {
  float d[3][16];
#pragma unroll
  for (int i = 0; i < 16; ++i) digits3(v[i], inv, d[0][i], d[1][i], d[2][i]);
  __nv_bfloat16* base = reinterpret_cast<__nv_bfloat16*>(p.hi) + o;
  if (mask == 0xFFFFu) {
#pragma unroll
    for (int s = 0; s < 3; ++s) {
      uint4 w0, w1;
      w0.x = pack_bf16x2(d[s][0], d[s][1]);   w0.y = pack_bf16x2(d[s][2], d[s][3]);
      w0.z = pack_bf16x2(d[s][4], d[s][5]);   w0.w = pack_bf16x2(d[s][6], d[s][7]);
      w1.x = pack_bf16x2(d[s][8], d[s][9]);   w1.y = pack_bf16x2(d[s][10], d[s][11]);
      w1.z = pack_bf16x2(d[s][12], d[s][13]); w1.w = pack_bf16x2(d[s][14], d[s][15]);
      uint4* q = reinterpret_cast<uint4*>(base + s * p.pstride);   // 32-byte aligned: o is a multiple of 16
      q[0] = w0;
      q[1] = w1;
    }
  } else if (mask) {
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (mask & (1u << i))
#pragma unroll
        for (int s = 0; s < 3; ++s) base[s * p.pstride + i] = __float2bfloat16_rn(d[s][i]);
  }
}

// Persistent: CTA c takes tiles c, c + gridDim.x, ... of every batch entry.
__global__ void __launch_bounds__(TC_THREADS, 1)
gemm_tc_kernel(const __grid_constant__ TcMaps maps, TcGemmArgs g, Epi e) {
  using SM = TcSmem;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  uint8_t* stg = gbase + SM::OFF_STG;
  const uint32_t stg_s = base + SM::OFF_STG;
  float* xp_all = reinterpret_cast<float*>(gbase + SM::OFF_XP);
  float* sb_all = reinterpret_cast<float*>(gbase + SM::OFF_SB);
  float* rmax = reinterpret_cast<float*>(gbase + SM::OFF_RMAX);     // [2][128]
  float* cmax = reinterpret_cast<float*>(gbase + SM::OFF_CMAX);     // [4][128]
  double* red = reinterpret_cast<double*>(gbase + SM::OFF_RED);
  uint8_t* tail = gbase + SM::OFF_BAR;
  const uint32_t bars = smem_u32(tail);
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (SM::STAGES + s); };
  auto chunk_full = [&](uint32_t b) { return bars + 8u * (2 * SM::STAGES + b); };
  auto chunk_empty = [&](uint32_t b) { return bars + 8u * (2 * SM::STAGES + 2 + b); };
  const uint32_t final_bar = bars + 8u * (2 * SM::STAGES + 4);
  const uint32_t in_bar = bars + 8u * (2 * SM::STAGES + 5);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tail + 8 * (2 * SM::STAGES + 6));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tail + 8 * (2 * SM::STAGES + 6) + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool need_in = (e.kind == EPI_AFF || e.kind == EPI_M);
  const bool digits_out = (e.kind == EPI_AFF || e.kind == EPI_M || e.kind == EPI_VT);
  if (threadIdx.x == 0) {
    for (int s = 0; s < SM::STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(chunk_full(b), 1);
      mbar_init(chunk_empty(b), EPI_WARPS);
    }
    mbar_init(final_bar, 1);
    mbar_init(in_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(tmem_slot)), "r"((uint32_t)SM::TMEM_COLS) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int tiles_m = (g.M + TC_BM - 1) / TC_BM, tiles_n = (g.N + TC_BN - 1) / TC_BN;
  const int tiles_per_entry = g.sym ? tiles_n * (tiles_n + 1) / 2 : tiles_m * tiles_n;
  const int total = tiles_per_entry * g.batch;
  const int nk = (g.K + TC_BK - 1) / TC_BK;
  const int nchunks = (nk + TC_CHUNK_KB - 1) / TC_CHUNK_KB;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t q = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const int b = t / tiles_per_entry, tl = t % tiles_per_entry;
        if (epi_skip(e, b)) continue;
        int ti, tj;
        tile_coords(tl, tiles_m, tiles_n, g.sym, ti, tj);
        const int tile_m = ti * TC_BM, tile_n = tj * TC_BN;
        const int za = g.a_index ? g.a_index[b] : b;
        const int zb = g.b_index ? g.b_index[b] : b;
        if (need_in) {            // the epilogue's input tile, into L2 while the products run
#pragma unroll
          for (int p = 0; p < DIGITS; ++p) {
            tma_prefetch_3d(&maps.in[p], tile_n, tile_m, b);
            tma_prefetch_3d(&maps.in[p], tile_n + 64, tile_m, b);
          }
        }
        for (int kb = 0; kb < nk; ++kb) {
          const int s = q % SM::STAGES;
          const uint32_t round = q / SM::STAGES;
          if (q >= (uint32_t)SM::STAGES && !mbar_wait(empty_bar(s), (round - 1) & 1, g.err, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t st = base + s * SM::STAGE_BYTES;
          mbar_expect_tx(full_bar(s), SM::STAGE_BYTES);
          const int kx = kb * TC_BK;
#pragma unroll
          for (int p = 0; p < DIGITS; ++p) {
            tma_load_3d(st + p * SM::PLANE_BYTES, &maps.a[p], full_bar(s), kx, tile_m, za);
            tma_load_3d(st + (DIGITS + p) * SM::PLANE_BYTES, &maps.b[p], full_bar(s), kx, tile_n, zb);
          }
          ++q;
        }
      }
      // every bulk copy issued has landed before the CTA may exit
      for (uint32_t i = (q > (uint32_t)SM::STAGES ? q - SM::STAGES : 0u); i < q; ++i)
        mbar_wait_own(full_bar(i % SM::STAGES), (i / SM::STAGES) & 1, g.err);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = tc_idesc();
      uint32_t q = 0, cq = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const int b = t / tiles_per_entry;
        if (epi_skip(e, b)) continue;
        for (int kb = 0; kb < nk; ++kb) {
          const int kc = kb % TC_CHUNK_KB;
          const uint32_t buf = cq & 1;
          if (kc == 0) {
            // the chunk buffer's previous contents (chunk cq - 2) have been drained
            if (cq >= 2 && !mbar_wait(chunk_empty(buf), ((cq >> 1) - 1) & 1, g.err, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          const int s = q % SM::STAGES;
          const uint32_t round = q / SM::STAGES;
          if (!mbar_wait(full_bar(s), round & 1, g.err, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = base + s * SM::STAGE_BYTES;
          const uint32_t d0 = tmem + buf * 256u, d1 = d0 + 128u;
#pragma unroll
          for (int k = 0; k < TC_BK / 16; ++k) {
            const uint32_t koff = k * 32;   // 16 bf16 = 32 bytes inside the 64 B swizzle row
#pragma unroll
            for (int i = 0; i < TC_PAIRS; ++i) {
              const bool first = (kc == 0 && k == 0) && (i <= 1);
              tc_mma(i == 0 ? d0 : d1, sw64_desc(st + pair_a(i) * SM::PLANE_BYTES + koff),
                     sw64_desc(st + (DIGITS + pair_b(i)) * SM::PLANE_BYTES + koff), idesc, first ? 0u : 1u);
            }
          }
          tc_commit(empty_bar(s));
          ++q;
          if (kc == TC_CHUNK_KB - 1 || kb == nk - 1) {
            tc_commit(chunk_full(buf));
            ++cq;
          }
        }
        if (ok && g.issued) atomicAdd(g.issued, (unsigned long long)nk * TC_PAIRS);
      }
      // every MMA issued has completed before tensor memory is released
      tc_commit(final_bar);
      mbar_wait_own(final_bar, 0, g.err);
    }
  } else {
    // ------------------------------------------------ drain + epilogue (warps 2..9)
    // Warps w and w + 4 share a tensor-memory lane quadrant: the first owns the
    // tile's columns 0..63, the second 64..127, of the quadrant's 32 rows.
    const int qd = warp & 3;                // TMEM lane quadrant (tile rows qd*32 ..)
    const int ew = warp - 2;                // epilogue warp index 0..7
    const int own = ew >> 2;                // column half
    const int et = threadIdx.x - 64;        // epilogue thread 0..255
    const int r = qd * 32 + lane;           // tile row of this thread
    float* xp = xp_all + ew * SM::XP_FLOATS;
    float* sbw = sb_all + ew * 128;
    const uint32_t tlane = tmem + ((uint32_t)(qd * 32) << 16) + (uint32_t)(own * 64);
    const float alpha16 = (float)((e.kind == EPI_AFF ? e.alpha : 1.0) * (1.0 / 65536.0));
    uint32_t cq = 0, in_phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const int b = t / tiles_per_entry, tl = t % tiles_per_entry;
      if (epi_skip(e, b)) continue;
      int ti, tj;
      tile_coords(tl, tiles_m, tiles_n, g.sym, ti, tj);
      const int tile_m = ti * TC_BM, tile_n = tj * TC_BN;
      const bool mirror = g.sym && ti != tj;
      const bool diag = g.sym && ti == tj;
      const bool transposed = mirror || diag || e.kind == EPI_VT;
      const int za = g.a_index ? g.a_index[b] : b;
      const int zb = g.b_index ? g.b_index[b] : b;
      const long long gr = tile_m + r;
      const bool rv = gr < g.M;
      const int c0 = tile_n + own * 64;      // first global column of this thread's half
      const bool hv = c0 < g.N;              // the half holds at least one column of the output
      const float* sa_ptr = g.a_scale + (long long)za * g.a_sbstride + gr;
      const float* sb_ptr = g.b_scale + (long long)zb * g.b_sbstride + c0 + lane;
      const bool cv0 = c0 + lane < g.N, cv1 = c0 + 32 + lane < g.N;
      float sa_next = rv ? sa_ptr[0] : 0.f;
      float sb_next0 = cv0 ? sb_ptr[0] : 0.f, sb_next1 = cv1 ? sb_ptr[32] : 0.f;
      float acc[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) acc[j] = 0.f;
      bool ok = true;
      // ---- drain: one K chunk at a time
      for (int c = 0; c < nchunks; ++c, ++cq) {
        const uint32_t buf = cq & 1;
        const float sa = sa_next;
        float* sbc = sbw + (c & 1) * 64;
        sbc[lane] = sb_next0;
        sbc[32 + lane] = sb_next1;
        __syncwarp();
        if (c + 1 < nchunks) {
          const long long o = (long long)(c + 1);
          sa_next = rv ? sa_ptr[o * g.a_srows] : 0.f;
          sb_next0 = cv0 ? sb_ptr[o * g.b_srows] : 0.f;
          sb_next1 = cv1 ? sb_ptr[o * g.b_srows + 32] : 0.f;
        }
        const bool okc = mbar_wait(chunk_full(buf), (cq >> 1) & 1, g.err, abort_flag);
        tc_fence_after();
        if (okc) {
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            float v0[16], v1[16];
            tmem_ld16(tlane + buf * 256u + h * 16, v0);
            tmem_ld16(tlane + buf * 256u + 128u + h * 16, v1);
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[h * 16 + j] = fmaf((v0[j] + v1[j]) * sbc[h * 16 + j], sa, acc[h * 16 + j]);
          }
        } else {
          ok = false;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(chunk_empty(buf));
      }
      // ---- element values: v = alpha acc 2^-16 + beta In (+ gamma on the diagonal)
#pragma unroll
      for (int j = 0; j < 64; ++j) acc[j] *= alpha16;
      if (need_in) {
        // the input tile through the staging area: round h loads its column half (all three
        // planes) and the warps owning that half read it
        const float sin = (rv && hv) ? *tc_scale_ptr(e.In, b, tj, gr) * 0.00390625f * (float)e.beta_in : 0.f;
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          if (et == 0) {
            fence_async_smem();              // earlier reads of the staging area precede the load
            mbar_expect_tx(in_bar, SM::STG_BYTES);
#pragma unroll
            for (int p = 0; p < DIGITS; ++p)
#pragma unroll
              for (int bx = 0; bx < 2; ++bx)
                tma_load_3d(stg_s + p * 16384 + bx * 8192, &maps.in[p], in_bar, tile_n + 64 * h, tile_m + 64 * bx, b);
          }
          const bool okl = mbar_wait(in_bar, in_phase & 1, g.err, abort_flag);
          ++in_phase;
          if (!okl) ok = false;
          if (own == h && rv && hv && ok) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              uint4 w[3];
#pragma unroll
              for (int p = 0; p < DIGITS; ++p) w[p] = *reinterpret_cast<const uint4*>(stg + stg_chunk(p, r >> 6, r & 63, 8 * k));
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const int j = 8 * k + u;
                float f[3];
#pragma unroll
                for (int p = 0; p < DIGITS; ++p) {
                  const uint32_t x = (&w[p].x)[u >> 1];
                  f[p] = __uint_as_float((u & 1) ? (x & 0xFFFF0000u) : (x << 16));
                }
                if (c0 + j < g.N) acc[j] = fmaf(sin, f[0] + (f[1] + f[2]), acc[j]);
              }
            }
          }
          epi_bar();                         // the half is read before the staging area is reused
        }
      }
      if (e.kind == EPI_AFF && e.gamma != 0.0 && rv) {
        const long long jd = gr - c0;
        if (jd >= 0 && jd < 64) {
#pragma unroll
          for (int j = 0; j < 64; ++j)
            if (j == jd) acc[j] += (float)e.gamma;
        }
      }
      // ---- maxima: the row over this half (elements the direct write keeps) and, for the
      // transposed write, each column over this warp's 32 rows (elements it keeps)
      float part = 0.f;
      {
        float m = 0.f;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const int cl = own * 64 + j;
          const bool valid = rv && (c0 + j < g.N) && !(diag && cl < r);
          if (valid) m = fmaxf(m, fabsf(acc[j]));
          if (e.kind == EPI_M && valid) {
            const float rd = acc[j] - ((tile_n + cl == gr) ? 1.0f : 0.0f);
            part += (mirror || (diag && cl > r)) ? 2.f * (rd * rd) : rd * rd;
          }
        }
        rmax[own * TC_BM + r] = m;
      }
      if (transposed && digits_out) {
#pragma unroll
        for (int h = 0; h < 4; ++h) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int cl = own * 64 + h * 16 + i;
            const bool valid = rv && (c0 + h * 16 + i < g.N) && !(diag && cl <= r);
            xp[lane * SM::XP_LD + i] = valid ? fabsf(acc[h * 16 + i]) : 0.f;
          }
          __syncwarp();
          const int jj = lane & 15, rh = lane >> 4;
          float m = 0.f;
#pragma unroll
          for (int i = 0; i < 16; ++i) m = fmaxf(m, xp[(rh * 16 + i) * SM::XP_LD + jj]);
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
          if (lane < 16) cmax[qd * TC_BN + own * 64 + h * 16 + jj] = m;
          __syncwarp();
        }
      }
      if (e.kind == EPI_M) {
        const double pd = warp_sum((double)part);
        if (lane == 0) red[ew] = pd;
      }
      epi_bar();                                       // maxima of the whole tile visible
      if (digits_out) {
        // ---- digit planes of the output: staged one column half (all planes) per round, TMA stores
        float inv_r = 1.f;
        if (e.kind != EPI_VT) {
          float m = fmaxf(rmax[r], rmax[TC_BM + r]);
          if (diag) m = fmaxf(m, fmaxf(fmaxf(cmax[r], cmax[TC_BN + r]), fmaxf(cmax[2 * TC_BN + r], cmax[3 * TC_BN + r])));
          const float sigma = pow2_ceil_scale(m);
          inv_r = 1.0f / sigma;
          if (own == 0 && rv && ok) *tc_scale_ptr(e.C, b, tj, gr) = sigma;
        }
        // direct (and diagonal) rounds: output columns tile_n + 64 h .., all 128 rows
        if (e.kind != EPI_VT) {
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            if (own == h && rv && hv) {
              const float inv_h = opaque(inv_r);
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                uint32_t wv[3][4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  float a[3], c[3];
                  digits3(acc[8 * k + 2 * u], inv_h, a[0], a[1], a[2]);
                  digits3(acc[8 * k + 2 * u + 1], inv_h, c[0], c[1], c[2]);
#pragma unroll
                  for (int p = 0; p < DIGITS; ++p) wv[p][u] = pack_bf16x2(a[p], c[p]);
                }
#pragma unroll
                for (int p = 0; p < DIGITS; ++p)
                  *reinterpret_cast<uint4*>(stg + stg_chunk(p, r >> 6, r & 63, 8 * k)) =
                      make_uint4(wv[p][0], wv[p][1], wv[p][2], wv[p][3]);
              }
            }
            if (diag) {
              // a diagonal tile's lower part comes from its upper part: element (lc, cl), lc < cl,
              // of the tile becomes (cl, lc); lc lies in this round's half, so the writers are the
              // warps of the quadrants 2h, 2h + 1
              epi_bar();                             // the direct values of the half are in place
              if ((qd >> 1) == h) {
#pragma unroll
                for (int hb = 0; hb < 4; ++hb) {
#pragma unroll
                  for (int i = 0; i < 16; ++i) xp[lane * SM::XP_LD + i] = acc[hb * 16 + i];
                  __syncwarp();
                  const int jj = lane & 15, rh = lane >> 4;
                  const int cl = own * 64 + hb * 16 + jj, lc0 = qd * 32 + rh * 16;
                  float v16[16];
#pragma unroll
                  for (int i = 0; i < 16; ++i) v16[i] = xp[(rh * 16 + i) * SM::XP_LD + jj];
                  __syncwarp();
                  float m = fmaxf(fmaxf(cmax[cl], cmax[TC_BN + cl]), fmaxf(cmax[2 * TC_BN + cl], cmax[3 * TC_BN + cl]));
                  m = fmaxf(m, fmaxf(rmax[cl], rmax[TC_BM + cl]));
                  const float inv = opaque(1.0f / pow2_ceil_scale(m));
#pragma unroll
                  for (int i = 0; i < 16; ++i) {
                    const int lc = lc0 + i;
                    if (lc < cl) {
                      float d[3];
                      digits3(v16[i], inv, d[0], d[1], d[2]);
                      const int cc = lc - 64 * h;
#pragma unroll
                      for (int p = 0; p < DIGITS; ++p)
                        *reinterpret_cast<__nv_bfloat16*>(stg + stg_chunk(p, cl >> 6, cl & 63, cc) + ((cc & 7) << 1)) =
                            __float2bfloat16_rn(d[p]);
                    }
                  }
                }
              }
            }
            fence_async_smem();
            epi_bar();
            if (et == 0) {
#pragma unroll
              for (int p = 0; p < DIGITS; ++p)
#pragma unroll
                for (int bx = 0; bx < 2; ++bx)
                  tma_store_3d(&maps.c[p], stg_s + p * 16384 + bx * 8192, tile_n + 64 * h, tile_m + 64 * bx, b);
              bulk_commit();
              bulk_wait_read0();                       // the staging area may be rewritten
            }
            epi_bar();
          }
        }
        // transposed rounds (mirrored tile, or V^T): tile column cl becomes output row tile_n + cl,
        // round h takes the tile's columns 64 h .. (the warps of that half), all 128 tile rows
        if (mirror || e.kind == EPI_VT) {
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            if (own == h) {
#pragma unroll
              for (int hb = 0; hb < 4; ++hb) {
#pragma unroll
                for (int i = 0; i < 16; ++i) xp[lane * SM::XP_LD + i] = acc[hb * 16 + i];
                __syncwarp();
                const int jj = lane & 15, rh = lane >> 4;
                const int ol = hb * 16 + jj;              // output row within the round (cl - 64 h)
                const int cl = own * 64 + ol, lc0 = qd * 32 + rh * 16;
                float v16[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) v16[i] = xp[(rh * 16 + i) * SM::XP_LD + jj];
                __syncwarp();
                const float m = fmaxf(fmaxf(cmax[cl], cmax[TC_BN + cl]), fmaxf(cmax[2 * TC_BN + cl], cmax[3 * TC_BN + cl]));
                const float sigma = pow2_ceil_scale(m);
                const float inv = opaque(1.0f / sigma);
                if (qd == 0 && rh == 0 && tile_n + cl < g.N && ok) *tc_scale_ptr(e.C, b, ti, tile_n + cl) = sigma;
#pragma unroll
                for (int half8 = 0; half8 < 2; ++half8) {
                  uint32_t wv[3][4];
#pragma unroll
                  for (int u = 0; u < 4; ++u) {
                    float a[3], c[3];
                    digits3(v16[8 * half8 + 2 * u], inv, a[0], a[1], a[2]);
                    digits3(v16[8 * half8 + 2 * u + 1], inv, c[0], c[1], c[2]);
#pragma unroll
                    for (int p = 0; p < DIGITS; ++p) wv[p][u] = pack_bf16x2(a[p], c[p]);
                  }
                  const int cc = (lc0 & 63) + 8 * half8;
#pragma unroll
                  for (int p = 0; p < DIGITS; ++p)
                    *reinterpret_cast<uint4*>(stg + stg_chunk(p, lc0 >> 6, ol, cc)) =
                        make_uint4(wv[p][0], wv[p][1], wv[p][2], wv[p][3]);
                }
              }
            }
            fence_async_smem();
            epi_bar();
            if (et == 0) {
#pragma unroll
              for (int p = 0; p < DIGITS; ++p)
#pragma unroll
                for (int bx = 0; bx < 2; ++bx)
                  tma_store_3d(&maps.c[p], stg_s + p * 16384 + bx * 8192, tile_m + 64 * bx, tile_n + 64 * h, b);
              bulk_commit();
              bulk_wait_read0();
            }
            epi_bar();
          }
        }
      } else if (rv && hv && ok) {
        // ---- fp32 results: the caller's state (Gram EMA), update, or a plain store
        if (e.kind == EPI_GRAM) {
          float* srow = e.state[b] + gr * (long long)e.cols;
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const int cl = own * 64 + j;
            if (c0 + j < g.N && !(diag && cl < r)) srow[c0 + j] = fmaf(e.beta, srow[c0 + j], (1.0f - e.beta) * acc[j]);
          }
        } else if (e.kind == EPI_U) {
          const long long o = gr * (long long)e.cols + c0;
          if (e.out_dtype == PRECOND_BF16) {
            __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(e.out[b]) + o;
#pragma unroll
            for (int j = 0; j < 64; ++j)
              if (c0 + j < g.N) dst[j] = __float2bfloat16_rn(acc[j]);
          } else {
            float* dst = reinterpret_cast<float*>(e.out[b]) + o;
#pragma unroll
            for (int j = 0; j < 64; ++j)
              if (c0 + j < g.N) dst[j] = acc[j];
          }
        } else if (e.kind == EPI_STORE) {
          float* dst = e.f32out + (long long)b * e.rows * e.cols + gr * (long long)e.cols + c0;
#pragma unroll
          for (int j = 0; j < 64; ++j)
            if (c0 + j < g.N) dst[j] = acc[j];
        }
      }
      if (e.kind == EPI_GRAM && transposed) {
        // the state's mirrored tile: column cl of the tile is row tile_n + cl of the state
        epi_bar();
#pragma unroll
        for (int h = 0; h < 4; ++h) {
#pragma unroll
          for (int i = 0; i < 16; ++i) xp[lane * SM::XP_LD + i] = acc[h * 16 + i];
          __syncwarp();
          const int jj = lane & 15, rh = lane >> 4;
          const int cl = own * 64 + h * 16 + jj, lc0 = qd * 32 + rh * 16;
          const long long orow = tile_n + cl;
          float v16[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) v16[i] = xp[(rh * 16 + i) * SM::XP_LD + jj];
          __syncwarp();
          if (orow < g.N && ok) {
            float* srow = e.state[b] + orow * (long long)e.cols + tile_m + lc0;
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (tile_m + lc0 + i < g.M && !(diag && lc0 + i >= cl)) srow[i] = fmaf(e.beta, srow[i], (1.0f - e.beta) * v16[i]);
          }
        }
      }
      if (e.kind == EPI_M && ew == 0) {
        double sum = 0.0;
#pragma unroll
        for (int w = 0; w < EPI_WARPS; ++w) sum += red[w];     // fixed order: deterministic
        if (ok) epi_m_finish(e, b, sum, g.M, tl);
      }
      // shared scratch free for the next tile; leave together once any role has aborted
      if (epi_bar_or(*abort_flag != 0)) break;
    }
    if (et == 0) {
      bulk_wait0();                              // every output store has completed
      if (in_phase > 0) mbar_wait_own(in_bar, (in_phase - 1) & 1, g.err);   // and the last input load
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 ::"r"(tmem), "r"((uint32_t)SM::TMEM_COLS) : "memory");
  }
}

}  // namespace precond
