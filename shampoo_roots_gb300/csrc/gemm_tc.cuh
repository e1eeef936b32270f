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
// into a 4-stage shared-memory ring (48 KB per stage: three planes of A and B);
// one elected thread issues tcgen05.mma (kind::f16, bf16, M = N = 128, K = 16).
// Warp roles (576 threads): warp 0 TMA producer, warp 1 TMEM owner and MMA
// issuer, warps 2..9 drain (two per tensor-memory lane quadrant, 64 columns
// each), warps 10..17 output (32 rows x 64 columns each).
//
// After a tile's last chunk the drain warps hand its sums to the output warps
// through one of the CTA's two hand-over slots in L2 and go on with the next
// tile.  The output warps form the output element (the product plus the
// element-wise terms; that input is the A operand itself for every product of
// the iteration, so the drain warps add it from the operand ring as the K loop
// passes the tile's diagonal columns) and write it in its consumer's format:
// digits with the tile's per-(row, block) scales for products that feed
// further products (and the mirrored tile for symmetric products, so results
// are exactly symmetric), the caller's fp32 state for the Gram EMA, or the
// caller's update.  A first pass over the slot takes the row maxima (direct
// scales) and column maxima (mirrored scales); a second writes the digit
// planes in 16-byte vectors staged through a per-warp shared scratch.
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
constexpr int EPI_WARPS = 8;                       // drain warps: two per tensor-memory lane quadrant
constexpr int OUT_WARPS = 8;                       // output warps: 32 tile rows x 64 columns each
constexpr int TC_THREADS = 64 + 32 * (EPI_WARPS + OUT_WARPS);   // producer, MMA, drain, output warps
constexpr unsigned long long TC_WAIT_CYCLES = 4000000000ull;   // ~2 s at 2 GHz

struct TcGemmArgs {
  int M, N, K;
  int batch;             // batch entries (z extent of the tile space)
  int split;             // CTAs per tile (1, 2 or 4; launches with few tiles): each computes the
                         //    whole tile and writes 4 / split of every output warp's four
                         //    16-column groups, part 0 also the scales and the residual
  int sym;               // 1: the product is symmetric (M == N): compute tiles with row block <=
                         //    column block only and write each off-diagonal tile mirrored too
  const int* a_index;    // batch entry -> z coordinate of A (null: b)
  const int* b_index;    // batch entry -> z coordinate of B (null: b)
  // operand block scales [z][chunk][srows] (A rows = output rows, B rows = output columns)
  const float* a_scale; long long a_sbstride; int a_srows;
  const float* b_scale; long long b_sbstride; int b_srows;
  unsigned int* err;     // error word (bit 0: a wait timed out)
  unsigned long long* issued;   // may be null: += (K blocks x digit pairs) of every tile computed
  float* scratch;        // per CTA two 128 x 128 fp32 slots: finished tiles from the drain to the output warps
};

struct TcSmem {
  static constexpr int PLANE_BYTES = TC_BM * TC_BK * 2;                 // 8 KB (A and B tiles alike)
  static constexpr int STAGE_BYTES = 2 * DIGITS * PLANE_BYTES;          // 48 KB
  static constexpr int STAGES = 4;
  static constexpr int RING = STAGES * STAGE_BYTES;
  static constexpr int XS_LD = 17;                                      // per-warp scratch row (32-bit words)
  static constexpr int OFF_XS = RING;                                   // per output warp: 32 rows x 17 words
  static constexpr int OFF_SB = OFF_XS + OUT_WARPS * 32 * XS_LD * 4;    // per drain warp: B scales of 2 chunks
  // per hand-over slot: [2 column halves][128 rows] row maxima, [4 row quarters][128
  // columns] column maxima, [8] residual parts (doubles)
  static constexpr int OFF_RMAX = OFF_SB + EPI_WARPS * 128 * 4;
  static constexpr int OFF_CMAX = OFF_RMAX + 2 * 2 * TC_BM * 4;
  static constexpr int OFF_INV = OFF_CMAX + 2 * 4 * TC_BN * 4;          // [128] row and [128] column 1/sigma
  static constexpr int OFF_RED = OFF_INV + (TC_BM + TC_BN) * 4;
  static constexpr int OFF_BAR = OFF_RED + 2 * EPI_WARPS * 8;
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
// Byte offset of element (row, k), k < 32, of a ring operand tile (TMA box {32, 128},
// 64-byte swizzle: the 16-byte chunk index XOR (row / 2) % 4).
__device__ __forceinline__ uint32_t ring_off(int row, int k) {
  return (uint32_t)(row * 64 + ((((k >> 3) ^ ((row >> 1) & 3)) << 4) | ((k & 7) << 1)));
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
// 8 consecutive fp32 columns of this warp's 32 lanes.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
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
__device__ __forceinline__ void out_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }   // the 8 output warps
// Barrier of the 8 output warps that also returns the OR of `v` over them (a
// decision every output thread takes the same way).
__device__ __forceinline__ bool out_bar_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n"
      " bar.red.or.pred p, 1, 256, q;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r) : "r"((uint32_t)v) : "memory");
  return r != 0;
}
// Columns 16 gi .. 16 gi + 15 of tile row r from a scratch slot laid out as
// [32 column quads][128 rows][4] (L2 only: the slot is rewritten by other warps).
__device__ __forceinline__ void load_row16(const float4* sp, int gi, int r, float (&v)[16]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float4 x = __ldcg(sp + (4 * gi + k) * TC_BM + r);
    v[4 * k] = x.x;
    v[4 * k + 1] = x.y;
    v[4 * k + 2] = x.z;
    v[4 * k + 3] = x.w;
  }
}

// Digit-pair schedule (0-based digit indices): pair 0 is level 0 (accumulator
// S0), pairs 1..5 are levels 1 and 2 (accumulator S1).
__host__ __device__ constexpr int pair_a(int i) { return i == 0 ? 0 : i == 1 ? 0 : i == 2 ? 1 : i == 3 ? 0 : i == 4 ? 1 : 2; }
__host__ __device__ constexpr int pair_b(int i) { return i == 0 ? 0 : i == 1 ? 1 : i == 2 ? 0 : i == 3 ? 2 : i == 4 ? 1 : 0; }

// ----------------------------------------------------------------- kernel
// Tensor maps: digit plane s of A is a[s], of B is b[s] (boxes {32, 128}, 64-byte swizzle).
struct TcMaps {
  CUtensorMap a[DIGITS];
  CUtensorMap b[DIGITS];
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

// The three digits of two values at once (engine.cuh digits3) with packed fp32
// pair arithmetic: half the instructions.  rint(y) for |y| <= 2^22 is
// (y + 1.5 2^23) - 1.5 2^23 in round-to-nearest-even, the rounding rintf uses;
// here |y| <= 256.  Every other step is exact, as in digits3.
__device__ __forceinline__ unsigned long long f2_pack(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long f2_sub(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ void digits3x2(float va, float vb, float ia, float ib, float (&da)[3], float (&db)[3]) {
  const unsigned long long magic = f2_pack(12582912.0f, 12582912.0f);        // 1.5 2^23
  const unsigned long long s512 = f2_pack(512.0f, 512.0f);
  unsigned long long y = f2_mul(f2_pack(va, vb), f2_pack(ia * 256.0f, ib * 256.0f));
  const unsigned long long d1 = f2_sub(f2_add(y, magic), magic);
  y = f2_mul(f2_sub(y, d1), s512);
  const unsigned long long d2 = f2_sub(f2_add(y, magic), magic);
  y = f2_mul(f2_sub(y, d2), s512);
  const unsigned long long d3 = f2_sub(f2_add(y, magic), magic);
  const unsigned long long p2 = f2_mul(d2, f2_pack(0.001953125f, 0.001953125f));          // 2^-9
  const unsigned long long p3 = f2_mul(d3, f2_pack(3.814697265625e-06f, 3.814697265625e-06f));   // 2^-18
  f2_unpack(d1, da[0], db[0]);
  f2_unpack(p2, da[1], db[1]);
  f2_unpack(p3, da[2], db[2]);
}

// Persistent: CTA c takes tiles c, c + gridDim.x, ... of every batch entry.  A
// launch with few tiles gives each tile to `split` adjacent CTAs instead: all of
// them compute it (the MMAs are cheap at that size), and each writes a share of
// its outputs, which cuts the output pass that bounds a lone tile's latency.
//
// Element-wise input.  Every product with one (EPI_AFF, EPI_M) is launched with
// that input equal to its first operand A, so the input tile (rows tile_m..,
// columns tile_n..) is A's K chunk tj, which passes through the operand ring
// anyway: the drain warps read it from the ring stages of that chunk and add
// it to their sums, and the producer refills those stages only after they have
// (barrier in_done).
__global__ void __launch_bounds__(TC_THREADS, 1)
gemm_tc_kernel(const __grid_constant__ TcMaps maps, TcGemmArgs g, Epi e) {
  using SM = TcSmem;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  uint32_t* xs_all = reinterpret_cast<uint32_t*>(gbase + SM::OFF_XS);
  float* sb_all = reinterpret_cast<float*>(gbase + SM::OFF_SB);
  float* rmax_all = reinterpret_cast<float*>(gbase + SM::OFF_RMAX);     // [2 slots][2][128]
  float* cmax_all = reinterpret_cast<float*>(gbase + SM::OFF_CMAX);     // [2 slots][4][128]
  float* invr = reinterpret_cast<float*>(gbase + SM::OFF_INV);      // [128] 1 / sigma of the output rows
  float* invc = invr + TC_BM;                                       // [128] of the mirrored tile's rows
  double* red_all = reinterpret_cast<double*>(gbase + SM::OFF_RED);   // [2 slots][8]
  uint8_t* tail = gbase + SM::OFF_BAR;
  const uint32_t bars = smem_u32(tail);
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (SM::STAGES + s); };
  auto chunk_full = [&](uint32_t b) { return bars + 8u * (2 * SM::STAGES + b); };
  auto chunk_empty = [&](uint32_t b) { return bars + 8u * (2 * SM::STAGES + 2 + b); };
  const uint32_t final_bar = bars + 8u * (2 * SM::STAGES + 4);
  auto slot_full = [&](uint32_t b) { return bars + 8u * (2 * SM::STAGES + 6 + b); };
  auto slot_empty = [&](uint32_t b) { return bars + 8u * (2 * SM::STAGES + 8 + b); };
  // K block k of a tile's input chunk has been read by the four drain warps of its column half
  auto in_done = [&](uint32_t k) { return bars + 8u * (2 * SM::STAGES + 10 + k); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tail + 8 * (2 * SM::STAGES + 14));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tail + 8 * (2 * SM::STAGES + 14) + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool need_in = (e.kind == EPI_AFF || e.kind == EPI_M);
  const bool digits_out = (e.kind == EPI_AFF || e.kind == EPI_M || e.kind == EPI_VT);
  if (threadIdx.x == 0) {
    // fetch the six tensor maps while the barriers and tensor memory are set up
#pragma unroll
    for (int p = 0; p < DIGITS; ++p) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.a[p])) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.b[p])) : "memory");
    }
    for (int s = 0; s < SM::STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(chunk_full(b), 1);
      mbar_init(chunk_empty(b), EPI_WARPS);
    }
    mbar_init(final_bar, 1);
    for (int k = 0; k < TC_CHUNK_KB; ++k) mbar_init(in_done(k), EPI_WARPS / 2);
    for (int b = 0; b < 2; ++b) {
      mbar_init(slot_full(b), EPI_WARPS);
      mbar_init(slot_empty(b), OUT_WARPS);
    }
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
  const int items = total * g.split;          // (tile, part) pairs, the parts of a tile adjacent
  const int nk = (g.K + TC_BK - 1) / TC_BK;
  const int nchunks = (nk + TC_CHUNK_KB - 1) / TC_CHUNK_KB;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t q = 0, nin = 0;
      long long in_cur = -1, in_prev = -1;      // first ring K block of the input chunk of the
      uint32_t par_cur = 0, par_prev = 0;        // current and the previous tile, and its in_done phase
      bool ok = true;
      for (int u = blockIdx.x; u < items && ok; u += gridDim.x) {
        const int t = u / g.split;
        const int b = t / tiles_per_entry, tl = t % tiles_per_entry;
        if (epi_skip(e, b)) continue;
        int ti, tj;
        tile_coords(tl, tiles_m, tiles_n, g.sym, ti, tj);
        const int tile_m = ti * TC_BM, tile_n = tj * TC_BN;
        const int za = g.a_index ? g.a_index[b] : b;
        const int zb = g.b_index ? g.b_index[b] : b;
        if (need_in) {
          in_prev = in_cur;
          par_prev = par_cur;
          in_cur = (long long)q + (long long)TC_CHUNK_KB * tj;
          par_cur = nin & 1;
          ++nin;
        }
        for (int kb = 0; kb < nk; ++kb) {
          const int s = q % SM::STAGES;
          const uint32_t round = q / SM::STAGES;
          if (q >= (uint32_t)SM::STAGES && !mbar_wait(empty_bar(s), (round - 1) & 1, g.err, abort_flag)) {
            ok = false;
            break;
          }
          if (need_in) {
            // the stage held K block q - STAGES: if that was part of a tile's input chunk, the
            // drain warps must have read it
            const long long old = (long long)q - SM::STAGES;
            const bool in_c = old >= in_cur && old < in_cur + TC_CHUNK_KB;
            const bool in_p = in_prev >= 0 && old >= in_prev && old < in_prev + TC_CHUNK_KB;
            if ((in_c || in_p) && !mbar_wait(in_done((uint32_t)(old - (in_c ? in_cur : in_prev))),
                                             in_c ? par_cur : par_prev, g.err, abort_flag)) {
              ok = false;
              break;
            }
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
      for (int u = blockIdx.x; u < items && ok; u += gridDim.x) {
        const int t = u / g.split;
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
  } else if (warp < 2 + EPI_WARPS) {
    // ------------------------------------------------ drain (warps 2..9)
    // Warps w and w + 4 share a tensor-memory lane quadrant: the first owns the
    // tile's columns 0..63, the second 64..127, of the quadrant's 32 rows.  After
    // a tile's last chunk they hand its sums to the output warps through this
    // CTA's scratch slot and go on with the next tile at once.
    const int qd = warp & 3;                // TMEM lane quadrant (tile rows qd*32 ..)
    const int ew = warp - 2;                // drain warp index 0..7
    const int own = ew >> 2;                // column half
    const int r = qd * 32 + lane;           // tile row of this thread
    float* sbw = sb_all + ew * 128;
    const uint32_t tlane = tmem + ((uint32_t)(qd * 32) << 16) + (uint32_t)(own * 64);
    const double alpha_eff = (e.kind == EPI_AFF) ? e.alpha : 1.0;
    const float alpha16 = (float)(alpha_eff * (1.0 / 65536.0));
    // input term in the sums' units: (beta / alpha) 2^16 sigma / 256 (P1 + P2 + P3)
    const float in_unit = need_in ? (float)(e.beta_in / alpha_eff * 256.0) : 0.f;
    uint32_t cq = 0, q = 0, lt = 0;
    for (int u = blockIdx.x; u < items; u += gridDim.x) {
      const int t = u / g.split;
      const int b = t / tiles_per_entry, tl = t % tiles_per_entry;
      if (epi_skip(e, b)) continue;
      int ti, tj;
      tile_coords(tl, tiles_m, tiles_n, g.sym, ti, tj);
      const int tile_m = ti * TC_BM, tile_n = tj * TC_BN;
      const int za = g.a_index ? g.a_index[b] : b;
      const int zb = g.b_index ? g.b_index[b] : b;
      const long long gr = tile_m + r;
      const bool rv = gr < g.M;
      const int c0 = tile_n + own * 64;      // first global column of this thread's half
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
        if (need_in && c == tj) {
          // the input: this thread's 64 columns are the K blocks 4 tj + 2 own (+1) of A's
          // chunk tj, row r, all three planes, resident in the ring; group gi = 16 columns
          const float iu = in_unit * sa;
          bool okr = true;
#pragma unroll
          for (int gi = 0; gi < 4; ++gi) {
            const int kb = TC_CHUNK_KB * tj + 2 * own + (gi >> 1);
            if (kb < nk) {
              const uint32_t qq = q + (uint32_t)kb;
              const int s = qq % SM::STAGES;
              if (mbar_wait(full_bar(s), (qq / SM::STAGES) & 1, g.err, abort_flag)) {
                if (rv) {
                  const uint8_t* tp = gbase + s * SM::STAGE_BYTES;
#pragma unroll
                  for (int h8 = 0; h8 < 2; ++h8) {
                    uint4 w[3];
#pragma unroll
                    for (int p = 0; p < DIGITS; ++p)
                      w[p] = *reinterpret_cast<const uint4*>(tp + p * SM::PLANE_BYTES + ring_off(r, 16 * (gi & 1) + 8 * h8));
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                      float f[3];
#pragma unroll
                      for (int p = 0; p < DIGITS; ++p) {
                        const uint32_t x = (&w[p].x)[i >> 1];
                        f[p] = __uint_as_float((i & 1) ? (x & 0xFFFF0000u) : (x << 16));
                      }
                      acc[16 * gi + 8 * h8 + i] = fmaf(iu, f[0] + (f[1] + f[2]), acc[16 * gi + 8 * h8 + i]);
                    }
                  }
                }
              } else {
                okr = false;
              }
            }
            if (gi & 1) {                         // both groups of this K block read: it may be refilled
              __syncwarp();
              if (lane == 0) mbar_arrive(in_done(2 * own + (gi >> 1)));
            }
          }
          if (!okr) ok = false;
        }
        const bool okc = mbar_wait(chunk_full(buf), (cq >> 1) & 1, g.err, abort_flag);
        tc_fence_after();
        if (okc) {
#pragma unroll
          for (int h = 0; h < 8; ++h) {
            float v0[8], v1[8];
            tmem_ld8(tlane + buf * 256u + h * 8, v0);
            tmem_ld8(tlane + buf * 256u + 128u + h * 8, v1);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[h * 8 + j] = fmaf((v0[j] + v1[j]) * sbc[h * 8 + j], sa, acc[h * 8 + j]);
          }
        } else {
          ok = false;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(chunk_empty(buf));
      }
      q += (uint32_t)nk;
      if (!ok) break;                        // a role gave up: leave (every other wait does too)
      // the tile's sums in the output's units
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        acc[j] *= alpha16;
        if (e.kind == EPI_AFF && c0 + j == gr) acc[j] += (float)e.gamma;
      }
      const uint32_t slot = lt & 1;
      if (lt >= 2 && !mbar_wait(slot_empty(slot), ((lt >> 1) - 1) & 1, g.err, abort_flag)) break;
      float4* sp = reinterpret_cast<float4*>(g.scratch + ((size_t)blockIdx.x * 2 + slot) * (TC_BM * TC_BN));
      // A split launch (few tiles: its latency is the output pass) takes the maxima of the
      // finished tile here, one 16-column group at a time while the sums are in registers
      // (each group is stored right after): row maxima (the direct write's scales), column
      // maxima by warp butterflies (the mirrored write's) and the residual of an M product.
      // A diagonal tile counts its upper part (with the diagonal) for the rows and its strict
      // upper part, mirrored, for the columns.  Launches of many tiles leave this to the
      // output warps, which have time to spare there, while the drain does not.
      const bool drain_max = digits_out && g.split > 1;
      const bool diag = g.sym && ti == tj, mirror = g.sym && ti != tj;
      const bool want_cmax = drain_max && (mirror || diag || e.kind == EPI_VT);
      float* cmx = cmax_all + slot * (4 * TC_BN) + qd * TC_BN + own * 64;
      float part = 0.f, mrow = 0.f;
      // bounds on this thread's column index j (tile column own * 64 + j): columns inside
      // the output are j < jn; a diagonal tile counts j >= jr for the rows and j > jr for the
      // columns (and twice, mirrored, in the residual); jd is the identity's column
      const int jn = rv ? min(64, g.N - tile_n - own * 64) : 0;
      const int jr = r - own * 64;
      const int jlo = diag ? jr : 0, jmlo = diag ? jr + 1 : 0;
      const int jtwo = mirror ? 0 : (diag ? jr + 1 : 64);
      const int jd = (int)(gr - tile_n) - own * 64;
#pragma unroll
      for (int gi = 0; gi < 4; ++gi) {
        if (drain_max) {
          float m[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int j = 16 * gi + i;
            const float v = acc[j];
            const bool valid = j >= jlo && j < jn;
            if (valid) mrow = fmaxf(mrow, fabsf(v));
            if (e.kind == EPI_M && valid) {
              const float rd = v - (j == jd ? 1.0f : 0.0f);
              part += (j >= jtwo) ? 2.f * (rd * rd) : rd * rd;
            }
            m[i] = (j >= jmlo && j < jn) ? fabsf(v) : 0.f;
          }
          if (want_cmax) {
            // after the exchanges lane L holds column L % 16 of the group
#pragma unroll
            for (int w = 8; w >= 1; w >>= 1) {
              const bool up = (lane & w) != 0;
#pragma unroll
              for (int i = 0; i < w; ++i) {
                const float send = up ? m[i] : m[i + w];
                const float keep = up ? m[i + w] : m[i];
                m[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, w));
              }
            }
            m[0] = fmaxf(m[0], __shfl_xor_sync(0xffffffffu, m[0], 16));
            if (lane < 16) cmx[16 * gi + lane] = m[0];
          }
        }
        // the group's sums to the scratch slot: [32 column quads][128 rows][4]
#pragma unroll
        for (int k4 = 4 * gi; k4 < 4 * gi + 4; ++k4)
          __stcg(sp + (own * 16 + k4) * TC_BM + r,
                 make_float4(acc[4 * k4], acc[4 * k4 + 1], acc[4 * k4 + 2], acc[4 * k4 + 3]));
      }
      if (drain_max) {
        rmax_all[slot * (2 * TC_BM) + own * TC_BM + r] = mrow;
        if (e.kind == EPI_M) {
          const float pd = warp_sum(part);
          if (lane == 0) red_all[slot * EPI_WARPS + qd + 4 * own] = (double)pd;   // the output warps' order
        }
      }
      __threadfence_block();
      __syncwarp();
      if (lane == 0) mbar_arrive(slot_full(slot));
      ++lt;
    }
  } else {
    // ------------------------------------------------ output warps (10..17)
    // Warp ow owns tile rows oq*32 .. +31 (one row per lane) and columns
    // oh*64 .. +63 of the tiles the drain hands over, in the same order.  Pass 1
    // takes the row maxima (the direct write's scales), the column maxima (the
    // mirrored write's) and the residual; pass 2 writes the digits of both, or
    // the fp32 results.
    const int ow = warp - 2 - EPI_WARPS;
    const int oq = ow & 3, oh = ow >> 2;    // row quarter, column half
    const int r = oq * 32 + lane;           // tile row of this thread
    const int cb = oh * 64;                 // first tile column of this thread
    uint32_t* xs = xs_all + ow * 32 * SM::XS_LD;
    uint8_t* xb = reinterpret_cast<uint8_t*>(xs);
    uint32_t lt = 0;
    for (int u = blockIdx.x; u < items; u += gridDim.x) {
      const int t = u / g.split;
      const int b = t / tiles_per_entry, tl = t % tiles_per_entry;
      if (epi_skip(e, b)) continue;
      int ti, tj;
      tile_coords(tl, tiles_m, tiles_n, g.sym, ti, tj);
      const int tile_m = ti * TC_BM, tile_n = tj * TC_BN;
      // this CTA's part of the tile's writes: column groups g_lo .. g_hi - 1 of every warp
      const int share = u - t * g.split;
      const int g_lo = share * (4 / g.split), g_hi = g_lo + 4 / g.split;
      const bool mirror = g.sym && ti != tj;
      const bool diag = g.sym && ti == tj;
      const bool transposed = mirror || diag || e.kind == EPI_VT;
      const long long gr = tile_m + r;
      const bool rv = gr < g.M;
      const uint32_t slot = lt & 1;
      const bool got = mbar_wait(slot_full(slot), (lt >> 1) & 1, g.err, abort_flag);
      if (out_bar_or(!got || *abort_flag != 0)) break;
      const float4* sp = reinterpret_cast<const float4*>(g.scratch + ((size_t)blockIdx.x * 2 + slot) * (TC_BM * TC_BN));
      float* rmax = rmax_all + slot * (2 * TC_BM);
      float* cmax = cmax_all + slot * (4 * TC_BN);
      if (g.split == 1) {
        // ---- pass 1: maxima (and the residual of an M product); fp32 results need neither.
        // (A split launch's drain took them; they are visible since slot_full.)
        float part = 0.f, mrow = 0.f;
        const bool want_cmax = transposed && digits_out;
        float vn[16];
        if (digits_out) load_row16(sp, 4 * oh, r, vn);
#pragma unroll 1
        for (int gi = 0; gi < (digits_out ? 4 : 0); ++gi) {
          float v[16], m[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = vn[i];
          if (gi + 1 < 4) load_row16(sp, 4 * oh + gi + 1, r, vn);     // next group in flight
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int cl = cb + 16 * gi + i;
            const bool vcol = rv && (tile_n + cl < g.N);
            const bool valid = vcol && !(diag && cl < r);
            if (valid) mrow = fmaxf(mrow, fabsf(v[i]));
            if (e.kind == EPI_M && valid) {
              const float rd = v[i] - ((tile_n + cl == gr) ? 1.0f : 0.0f);
              part += (mirror || (diag && cl > r)) ? 2.f * (rd * rd) : rd * rd;
            }
            m[i] = (vcol && !(diag && cl <= r)) ? fabsf(v[i]) : 0.f;
          }
          if (want_cmax) {
            // butterfly over the warp: after the exchanges lane L holds column L % 16 of the group
#pragma unroll
            for (int w = 8; w >= 1; w >>= 1) {
              const bool up = (lane & w) != 0;
#pragma unroll
              for (int i = 0; i < w; ++i) {
                const float send = up ? m[i] : m[i + w];
                const float keep = up ? m[i + w] : m[i];
                m[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, w));
              }
            }
            m[0] = fmaxf(m[0], __shfl_xor_sync(0xffffffffu, m[0], 16));
            if (lane < 16) cmax[oq * TC_BN + cb + 16 * gi + lane] = m[0];
          }
        }
        rmax[oh * TC_BM + r] = mrow;
        if (e.kind == EPI_M) {
          const float pd = warp_sum(part);
          if (lane == 0) red_all[slot * EPI_WARPS + ow] = (double)pd;
        }
        out_bar();                                     // column maxima and residual parts visible
      }
      if (digits_out) {
        // output scales: the first column half's threads take row r of this tile (and, for a
        // diagonal tile, its lower part mirrored in), the second half's row r of the mirrored
        // tile / of V^T (tile column r)
        if (oh == 0) {
          float m = fmaxf(rmax[r], rmax[TC_BM + r]);
          if (diag) m = fmaxf(m, fmaxf(fmaxf(cmax[r], cmax[TC_BN + r]), fmaxf(cmax[2 * TC_BN + r], cmax[3 * TC_BN + r])));
          const float sigma = pow2_ceil_scale(m);
          invr[r] = 1.0f / sigma;
          if (e.kind != EPI_VT && rv && share == 0) *tc_scale_ptr(e.C, b, tj, gr) = sigma;
        } else if (mirror || e.kind == EPI_VT) {
          const float m = fmaxf(fmaxf(cmax[r], cmax[TC_BN + r]), fmaxf(cmax[2 * TC_BN + r], cmax[3 * TC_BN + r]));
          const float sigma = pow2_ceil_scale(m);
          invc[r] = 1.0f / sigma;
          if (tile_n + r < g.N && share == 0) *tc_scale_ptr(e.C, b, ti, tile_n + r) = sigma;
        }
        out_bar();
        const float ih = invr[r];
        const long long rbase = (long long)tile_m + oq * 32;
#pragma unroll 1
        for (int gi = g_lo; gi < g_hi; ++gi) {
          if (tile_n + cb + 16 * gi >= g.N) break;     // this and later groups lie beyond the output
          float v[16];
          load_row16(sp, 4 * oh + gi, r, v);
          // ---- direct tile: digits of row r with its scale.  Per plane each lane puts its row's
          // 32 bytes into the warp's scratch (rows 48 bytes apart), then the lanes store 16-byte
          // pieces: two per lane, 32 rows x 32 bytes.  A diagonal tile keeps columns >= row only.
          if (e.kind != EPI_VT) {
            uint32_t wv[3][8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              float a[3], c[3];
              digits3x2(v[2 * u], v[2 * u + 1], ih, ih, a, c);
#pragma unroll
              for (int p = 0; p < DIGITS; ++p) wv[p][u] = pack_bf16x2(a[p], c[p]);
            }
#pragma unroll
            for (int p = 0; p < DIGITS; ++p) {
              *reinterpret_cast<uint4*>(xb + lane * 48) = make_uint4(wv[p][0], wv[p][1], wv[p][2], wv[p][3]);
              *reinterpret_cast<uint4*>(xb + lane * 48 + 16) = make_uint4(wv[p][4], wv[p][5], wv[p][6], wv[p][7]);
              __syncwarp();
              __nv_bfloat16* plane = reinterpret_cast<__nv_bfloat16*>(e.C.hi) + (long long)b * e.C.bstride + p * e.C.pstride;
#pragma unroll
              for (int tt = 0; tt < 2; ++tt) {
                const int cidx = lane + 32 * tt, R = cidx >> 1, hh = cidx & 1;
                const int lc = cb + 16 * gi + 8 * hh;     // first tile column of the piece
                const int lr = oq * 32 + R;               // its tile row
                if (rbase + R < g.M) {
                  __nv_bfloat16* dst = plane + (rbase + R) * e.C.ld + tile_n + lc;
                  if (!diag || lc >= lr) {
                    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(xb + R * 48 + hh * 16);
                  } else if (lc + 7 >= lr) {
                    const __nv_bfloat16* src = reinterpret_cast<const __nv_bfloat16*>(xb + R * 48 + hh * 16);
                    for (int i = lr - lc; i < 8; ++i) dst[i] = src[i];
                  }
                }
              }
              __syncwarp();
            }
          }
          // ---- mirrored tile (a diagonal tile's strict lower part, and V^T): element (r, cl) goes
          // to output row tile_n + cl, column tile_m + r.  Per plane each lane writes its 16 values
          // into the scratch column-major (16 output rows x 32 output columns), then the lanes
          // store 16-byte pieces of 8 output columns: two per lane.
          if (transposed) {
            __nv_bfloat16* xh = reinterpret_cast<__nv_bfloat16*>(xs);
            float inv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) inv[i] = diag ? invr[cb + 16 * gi + i] : invc[cb + 16 * gi + i];
#pragma unroll
            for (int p = 0; p < DIGITS; ++p) {
#pragma unroll
              for (int i = 0; i < 16; i += 2) {
                float da[3], db[3];
                digits3x2(v[i], v[i + 1], inv[i], inv[i + 1], da, db);
                xh[i * 32 + lane] = __float2bfloat16_rn(p == 0 ? da[0] : (p == 1 ? da[1] : da[2]));
                xh[(i + 1) * 32 + lane] = __float2bfloat16_rn(p == 0 ? db[0] : (p == 1 ? db[1] : db[2]));
              }
              __syncwarp();
              __nv_bfloat16* plane = reinterpret_cast<__nv_bfloat16*>(e.C.hi) + (long long)b * e.C.bstride + p * e.C.pstride;
#pragma unroll
              for (int tt = 0; tt < 2; ++tt) {
                const int cidx = lane + 32 * tt, jj = cidx >> 2, k = cidx & 3;
                const int cl = cb + 16 * gi + jj;           // tile column = output row offset
                const int lc = oq * 32 + 8 * k;             // first tile row = output column offset
                const long long orow = tile_n + cl, ocol = (long long)tile_m + lc;
                if (orow < g.N && ocol < g.M) {
                  __nv_bfloat16* dst = plane + orow * e.C.ld + ocol;
                  if (!diag || lc + 7 < cl) {
                    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(xh + jj * 32 + 8 * k);
                  } else if (lc < cl) {
                    // a diagonal tile's piece crossing the diagonal: only rows above it
                    for (int i = 0; i < cl - lc; ++i) dst[i] = xh[jj * 32 + 8 * k + i];
                  }
                }
              }
              __syncwarp();
            }
          }
        }
      } else {
        // ---- fp32 results: the caller's state (Gram EMA, and its mirrored tile), the update, or
        // a plain store.  Row-major stores pass through the warp's scratch: lanes store 2 rows x
        // 16 columns per instruction (64-byte runs); the mirrored Gram tile is stored directly
        // (for a fixed column the warp's lanes are consecutive addresses).
        const long long rbase = (long long)tile_m + oq * 32;
#pragma unroll 1
        for (int gi = g_lo; gi < g_hi; ++gi) {
          if (tile_n + cb + 16 * gi >= g.N) break;
          float v[16];
          load_row16(sp, 4 * oh + gi, r, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) xs[lane * SM::XS_LD + i] = __float_as_uint(v[i]);
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int R = 2 * k + (lane >> 4), w = lane & 15;
            const long long row = rbase + R;
            const int cl = cb + 16 * gi + w;
            const int col = tile_n + cl;
            if (row < g.M && col < g.N) {
              const float x = __uint_as_float(xs[R * SM::XS_LD + w]);
              const long long o = row * (long long)e.cols + col;
              if (e.kind == EPI_GRAM) {
                // the direct tile is upper (diagonal tiles: from the diagonal on); a packed
                // state stores exactly that part
                const long long os = e.state_packed ? packed_offset(row, col, e.cols) : o;
                if (!(diag && cl < oq * 32 + R)) e.state[b][os] = fmaf(e.beta, e.state[b][os], (1.0f - e.beta) * x);
              } else if (e.kind == EPI_U) {
                if (e.out_dtype == PRECOND_BF16) reinterpret_cast<__nv_bfloat16*>(e.out[b])[o] = __float2bfloat16_rn(x);
                else reinterpret_cast<float*>(e.out[b])[o] = x;
              } else if (e.kind == EPI_STORE) {
                e.f32out[(long long)b * e.rows * e.cols + o] = x;
              }
            }
          }
          __syncwarp();
          if (e.kind == EPI_GRAM && transposed && rv && !e.state_packed) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int cl = cb + 16 * gi + i;
              if (tile_n + cl < g.N && !(diag && cl <= r)) {
                float* stp = e.state[b] + (long long)(tile_n + cl) * e.cols + gr;
                *stp = fmaf(e.beta, *stp, (1.0f - e.beta) * v[i]);
              }
            }
          }
        }
      }
      if (e.kind == EPI_M && ow == 0 && share == 0) {
        double sum = 0.0;
#pragma unroll
        for (int w = 0; w < EPI_WARPS; ++w) sum += red_all[slot * EPI_WARPS + w];     // fixed order: deterministic
        epi_m_finish(e, b, sum, g.M, tl);
      }
      // the slot's data is dead: drop its L2 lines without writing them back (the slot is
      // rewritten two tiles later), then hand it back; leave together once any role has aborted
      out_bar();
      {
        const char* lines = reinterpret_cast<const char*>(sp) + (size_t)(threadIdx.x - 32 * (2 + EPI_WARPS)) * 256;
        asm volatile("discard.global.L2 [%0], 128;" ::"l"(lines) : "memory");
        asm volatile("discard.global.L2 [%0], 128;" ::"l"(lines + 128) : "memory");
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(slot_empty(slot));
      ++lt;
      if (out_bar_or(*abort_flag != 0)) break;
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
