// tcgen05 batched GEMM of the large-matrix engine (sm_103a):  C_b = A_b . B_b^T
//
// Exact-digit split.  Each operand row is held as S bf16 "digit planes":
//   x = sigma * 2^-b * (P_1 + P_2 + ... + P_S),   P_s = d_s * 2^(-b (s-1)),
// with sigma a power of two >= max |x| of the row (a per-row scale, or one
// bound for the whole matrix), b = 7 and integer digits |d_1| <= 2^b,
// |d_s| <= 2^(b-1).  Digit products are exact in bf16 x bf16 -> fp32, and the
// two leading product levels are sums of integers (level 2: P_1 Q_1; level 3:
// P_1 Q_2 + P_2 Q_1 in units of 2^-b) below 2^24 for K <= 1024 (and for
// non-coherent rows well beyond), so their fp32 tensor-memory accumulation is
// EXACT: no rounding, and none of the truncation bias of a long fp32 chain.
// The remaining levels (s + t >= 4) go to a third accumulator whose rounding
// is 2^-14 below the result.  Products with s + t > S + 1 are dropped.
//   S = 4: 10 MMAs per K step, ~2^-29 relative to the row scales;
//   S = 3:  6 MMAs per K step, ~2^-22.
// The epilogue forms C_ij = 2^-2b sigma_A(i) sigma_B(j) (acc0 + acc1 + acc2).
//
// Pipeline: TMA (3-D tensor maps {K, rows, batch}, 64-byte swizzle, K block
// 32) into a 3-4 stage shared-memory ring; one elected thread issues
// tcgen05.mma (kind::f16, bf16, M = 128, N = 128, K = 16) into three fp32
// accumulators in tensor memory; eight epilogue warps (two per tensor-memory
// lane quadrant) read them back with tcgen05.ld.  Warp roles (320 threads):
// warp 0 TMA producer, warp 1 TMEM owner and MMA issuer, warps 2..9 epilogue.
// Every mbarrier wait is bounded; on time-out the kernel records an error word
// and leaves the tile.
#pragma once

#include <cuda.h>
#include "engine.cuh"

namespace precond {

constexpr int TC_BM = 128, TC_BN = 128, TC_BK = 32;
constexpr int EPI_WARPS = 8;                       // two per tensor-memory lane quadrant
constexpr int TC_THREADS = 64 + 32 * EPI_WARPS;    // producer warp, MMA warp, epilogue warps
constexpr int DIGIT_BITS = 7;
constexpr unsigned long long TC_WAIT_CYCLES = 4000000000ull;   // ~2 s at 2 GHz

struct TcGemmArgs {
  int M, N, K;
  int batch;             // batch entries (z extent of the tile space)
  int sym;               // 1: the product is symmetric (M == N): compute tiles with row block <=
                         //    column block only and write each off-diagonal tile mirrored too
  const int* a_index;    // batch entry -> z coordinate of A (null: b)
  const int* b_index;    // batch entry -> z coordinate of B (null: b)
  // operand scales: per-row arrays [z][rows] (A rows = output rows, B rows = output cols) or constants
  const float* a_rowscale; long long a_rs_stride; float a_scale;
  const float* b_rowscale; long long b_rs_stride; float b_scale;
  unsigned int* err;     // error word (bit 0: a wait timed out)
  unsigned long long* issued;   // may be null: += (K blocks x digit pairs) of every tile computed
};

template <int S>
struct TcSmem {
  static constexpr int A_BYTES = TC_BM * TC_BK * 2;            // 8 KB per digit plane
  static constexpr int B_BYTES = TC_BN * TC_BK * 2;            // 8 KB
  static constexpr int STAGE_BYTES = S * (A_BYTES + B_BYTES);
  static constexpr int STAGES = (S == 4) ? 3 : 4;
  static constexpr int STG_LD = TC_BN / 2 + 1;                  // staging: half a tile's columns, row stride
                                                                // (floats) bank-conflict free
  static constexpr int STAGING_BYTES = TC_BM * STG_LD * 4;
  static constexpr int TMEM_COLS = 512;                        // 3 x 128 accumulators + 128 parking columns
  static constexpr int PARK_COL = 384;                         // drained second half of a tile waits here
  static constexpr int BYTES = STAGES * STAGE_BYTES + STAGING_BYTES + 1024 /*align*/ + 1024 /*barriers, scales*/;
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
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}
// Bounded wait; returns false (and flags `err`) on time-out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned int* err) {
  if (mbar_try_wait(bar, parity)) return true;
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
// Store 32 consecutive fp32 columns of this warp's 32 lanes into tensor memory.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])), "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Digit-pair schedule (0-based digit indices), ordered by level s + t; the
// first 6 pairs are the S = 3 schedule.  Accumulator: level 0 -> 0, level 1 -> 1,
// level >= 2 -> 2.
__host__ __device__ constexpr int pair_a(int i) {
  return i == 0 ? 0 : i == 1 ? 0 : i == 2 ? 1 : i == 3 ? 0 : i == 4 ? 1 : i == 5 ? 2 : i == 6 ? 0 : i == 7 ? 1 : i == 8 ? 2 : 3;
}
__host__ __device__ constexpr int pair_b(int i) {
  return i == 0 ? 0 : i == 1 ? 1 : i == 2 ? 0 : i == 3 ? 2 : i == 4 ? 1 : i == 5 ? 0 : i == 6 ? 3 : i == 7 ? 2 : i == 8 ? 1 : 0;
}
template <int S>
struct Pairs { static constexpr int N = (S == 4) ? 10 : 6; };
__host__ __device__ constexpr int pair_acc(int s, int t) { return (s + t) >= 2 ? 2 : (s + t); }

// ----------------------------------------------------------------- kernel
// Tensor maps: digit plane s of A is map_a[s] (only the first S are used).
struct TcMaps {
  CUtensorMap a[4];
  CUtensorMap b[4];
};

// Tile `tl` of a batch entry -> (row block, column block); symmetric products
// enumerate the upper triangle row by row.
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

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }   // the 8 epilogue warps

// Persistent: CTA c takes tiles c, c + gridDim.x, ...; tile t = (entry, row block,
// column block) with the column block fastest.  The producer and the MMA
// issuer run ahead through the shared-memory ring; the epilogue drains the
// tensor-memory accumulators of a tile into a shared staging tile, releases
// tensor memory (the next tile's MMAs start), then runs the element-wise
// epilogue from shared memory with coalesced global accesses.
constexpr int EPI_RB = 8;   // epilogue rows per load batch

template <int S>
__global__ void __launch_bounds__(TC_THREADS, 1)
gemm_tc_kernel(const __grid_constant__ TcMaps maps, TcGemmArgs g, Epi e) {
  using SM = TcSmem<S>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  float* staging = reinterpret_cast<float*>(gbase + SM::STAGES * SM::STAGE_BYTES);
  uint8_t* tail = gbase + SM::STAGES * SM::STAGE_BYTES + SM::STAGING_BYTES;
  const uint32_t bars = smem_u32(tail);
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (SM::STAGES + s); };
  const uint32_t accum_bar = bars + 8u * (2 * SM::STAGES);
  const uint32_t tmem_empty_bar = accum_bar + 8u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tail + 8 * (2 * SM::STAGES + 2));
  float* colscale = reinterpret_cast<float*>(tail + 512);      // 128 floats
  __shared__ double red[EPI_WARPS];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < SM::STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(accum_bar, 1);
    mbar_init(tmem_empty_bar, 1);
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
        for (int kb = 0; kb < nk; ++kb, ++q) {
          const int s = q % SM::STAGES;
          const uint32_t round = q / SM::STAGES;
          if (q >= (uint32_t)SM::STAGES && !mbar_wait(empty_bar(s), (round - 1) & 1, g.err)) { ok = false; break; }
          const uint32_t st = base + s * SM::STAGE_BYTES;
          mbar_expect_tx(full_bar(s), SM::STAGE_BYTES);
          const int kx = kb * TC_BK;
#pragma unroll
          for (int p = 0; p < S; ++p) {
            tma_load_3d(st + p * SM::A_BYTES, &maps.a[p], full_bar(s), kx, tile_m, za);
            tma_load_3d(st + S * SM::A_BYTES + p * SM::B_BYTES, &maps.b[p], full_bar(s), kx, tile_n, zb);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = tc_idesc();
      uint32_t q = 0, it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const int b = t / tiles_per_entry;
        if (epi_skip(e, b)) continue;
        if (it > 0 && !mbar_wait(tmem_empty_bar, (it - 1) & 1, g.err)) { ok = false; break; }
        tc_fence_after();
        for (int kb = 0; kb < nk; ++kb, ++q) {
          const int s = q % SM::STAGES;
          const uint32_t round = q / SM::STAGES;
          if (!mbar_wait(full_bar(s), round & 1, g.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t st = base + s * SM::STAGE_BYTES;
#pragma unroll
          for (int k = 0; k < TC_BK / 16; ++k) {
            const uint32_t koff = k * 32;   // 16 bf16 = 32 bytes inside the 64 B swizzle row
#pragma unroll
            for (int i = 0; i < Pairs<S>::N; ++i) {
              const int pa = pair_a(i), pb = pair_b(i);
              const int acc_id = pair_acc(pa, pb);
              const bool first = (kb == 0 && k == 0) && (i == 0 || i == 1 || i == 3);
              tc_mma(tmem + 128u * acc_id, sw64_desc(st + pa * SM::A_BYTES + koff),
                     sw64_desc(st + S * SM::A_BYTES + pb * SM::B_BYTES + koff), idesc, first ? 0u : 1u);
            }
          }
          tc_commit(empty_bar(s));
        }
        tc_commit(accum_bar);
        if (ok && g.issued) atomicAdd(g.issued, (unsigned long long)nk * Pairs<S>::N);
        ++it;
      }
    }
  } else {
    // ------------------------------------------------ epilogue (warps 2..9)
    // Warps w and w + 4 share a tensor-memory lane quadrant: the first drains the
    // tile's columns 0..63 (to the staging tile), the second columns 64..127 (held
    // in registers until the second half); both then split the element-wise work.
    const int q = warp & 3;                 // TMEM lane quadrant of this warp (rows q*32 ..)
    const int ew = warp - 2;                // epilogue warp index 0..7
    const int own = ew >> 2;                // column half this warp drains
    const int et = threadIdx.x - 64;        // epilogue thread index 0..255
    const double c0 = (double)e.inv_scale * ldexp(1.0, -2 * DIGIT_BITS);
    uint32_t it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const int b = t / tiles_per_entry, tl = t % tiles_per_entry;
      if (epi_skip(e, b)) continue;
      int ti, tj;
      tile_coords(tl, tiles_m, tiles_n, g.sym, ti, tj);
      const int tile_m = ti * TC_BM, tile_n = tj * TC_BN;
      const bool mirror = g.sym && ti != tj;
      const int za = g.a_index ? g.a_index[b] : b;
      const int zb = g.b_index ? g.b_index[b] : b;
      // column scales of this tile
      if (et < TC_BN) {
        const long long gc = tile_n + et;
        colscale[et] = (gc < g.N) ? (g.b_rowscale ? g.b_rowscale[(long long)zb * g.b_rs_stride + gc] : g.b_scale) : 0.f;
      }
      const bool ok = mbar_wait(accum_bar, it & 1, g.err);
      tc_fence_after();
      epi_bar();
      // ---- drain: tensor memory -> columns 0..63 to staging, 64..127 to registers (scaled fp32),
      // after which tensor memory is free for the next tile's products
      const int row = q * 32 + lane;
      const long long gr = tile_m + row;
      const double sa = (gr < g.M) ? (g.a_rowscale ? (double)g.a_rowscale[(long long)za * g.a_rs_stride + gr]
                                                    : (double)g.a_scale) : 0.0;
      const float rs = (float)(c0 * sa);
      float* srow = staging + row * SM::STG_LD;
      const uint32_t tlane = tmem + ((uint32_t)(q * 32) << 16);
#pragma unroll
      for (int cc = 0; cc < TC_BN / 64; ++cc) {
        const int ch = own * (TC_BN / 64) + cc;
        float v0[32], v1[32];
        const uint32_t taddr = tlane + (uint32_t)(ch * 32);
        tmem_ld32(taddr, v0);
        tmem_ld32(taddr + 128, v1);
#pragma unroll
        for (int j = 0; j < 32; ++j) v0[j] += v1[j];
        tmem_ld32(taddr + 256, v1);
#pragma unroll
        for (int j = 0; j < 32; ++j) v0[j] = (v0[j] + v1[j]) * rs * colscale[ch * 32 + j];
        if (own == 0) {
#pragma unroll
          for (int j = 0; j < 32; ++j) srow[cc * 32 + j] = v0[j];
        } else {
          tmem_st32(tlane + SM::PARK_COL + cc * 32, v0);   // outside the accumulators
        }
      }
      tc_fence_before();
      epi_bar();
      if (et == 0) mbar_arrive(tmem_empty_bar);    // tensor memory may take the next tile
      // ---- element-wise epilogue, one half of the tile's columns at a time.  Every
      // barrier below is reached by all 256 epilogue threads (work is guarded, not the barriers).
      float part = 0.f;
      const bool track = (e.kind == EPI_AFF || e.kind == EPI_M) && e.C.rowmax;
      const bool need_in = (e.kind == EPI_AFF || e.kind == EPI_M || e.kind == EPI_GRAM);
      // diagonal tile of a symmetric product: the strict upper triangle is computed and written
      // to both triangles, so the result is exactly symmetric (the iteration amplifies any
      // antisymmetric part while M is far from I)
      const bool diag_fix = g.sym && !mirror && (e.kind == EPI_AFF || e.kind == EPI_M);
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        const int hc = h * (TC_BN / 2);             // first tile column of this half
        if (h == 1) {
          epi_bar();                                // the first half's staging is read
          if (own == 1) {
#pragma unroll
            for (int cc = 0; cc < TC_BN / 64; ++cc) {
              float v[32];
              tmem_ld32(tlane + SM::PARK_COL + cc * 32, v);
#pragma unroll
              for (int j = 0; j < 32; ++j) srow[cc * 32 + j] = v[j];
            }
          }
          epi_bar();
        }
        if (e.kind == EPI_VT) {
          // transposed output: warp ew takes 8 of the half's columns, lanes run over rows
          for (int cc = 0; cc < TC_BN / 2 / EPI_WARPS; ++cc) {
            const int cl = ew * (TC_BN / 2 / EPI_WARPS) + cc;
            const long long gc = tile_n + hc + cl;
            float mx = 0.f;
            if (ok && gc < g.N) {
#pragma unroll
              for (int r4 = 0; r4 < 4; ++r4) {
                const int r = r4 * 32 + lane;
                const long long grr = tile_m + r;
                if (grr < g.M) {
                  const float v = staging[r * SM::STG_LD + cl];
                  e.C.f32[(long long)b * e.C.bstride + gc * e.C.ld + grr] = v;
                  mx = fmaxf(mx, fabsf(v));
                }
              }
            }
            mx = warp_max(mx);
            if (ok && lane == 0 && gc < g.N && e.C.rowmax) atomic_max_nonneg(&e.C.rowmax[(long long)b * e.C.rows + gc], mx);
          }
          continue;
        }
        float colmx[2] = {0.f, 0.f};   // diag_fix: per lane column, max |v| of the strict upper part
        // Rows go in groups of EPI_RB: the group's global inputs are loaded first, so
        // their latencies overlap instead of adding up row by row (the whole cost of a
        // product when the grid has only a few tiles).
#pragma unroll 1
        for (int r0 = 0; r0 < TC_BM / EPI_WARPS; r0 += EPI_RB) {
          float in[EPI_RB][2];
#pragma unroll
          for (int u = 0; u < EPI_RB; ++u) {
            const int r = ew * (TC_BM / EPI_WARPS) + r0 + u;
            const long long grr = tile_m + r;
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
              const int c = hc + c2 * 32 + lane;
              const long long gc = tile_n + c;
              in[u][c2] = 0.f;
              if (ok && need_in && grr < g.M && gc < g.N && !(diag_fix && c < r)) {
                if (e.kind == EPI_GRAM)
                  in[u][c2] = e.state[b][grr * e.cols + gc];
                else
                  in[u][c2] = e.In.f32[(long long)b * e.In.bstride + grr * e.In.ld + gc];
              }
            }
          }
#pragma unroll
          for (int u = 0; u < EPI_RB; ++u) {
            const int r = ew * (TC_BM / EPI_WARPS) + r0 + u;
            const long long grr = tile_m + r;
            float mx = 0.f;
            if (ok && grr < g.M) {
#pragma unroll
              for (int c2 = 0; c2 < 2; ++c2) {
                const int cl = c2 * 32 + lane;
                const int c = hc + cl;
                const long long gc = tile_n + c;
                if (gc < g.N && !(diag_fix && c < r)) {
                  float* sp = &staging[r * SM::STG_LD + cl];
                  const float acc = *sp;
                  const long long o = (long long)b * e.C.bstride + grr * e.C.ld + gc;
                  const bool up = diag_fix && c > r;     // also written at the transposed position
                  switch (e.kind) {
                    case EPI_STORE:
                      e.C.f32[o] = acc;
                      break;
                    case EPI_AFF: {
                      float v = fmaf((float)e.alpha, acc, (float)e.beta_in * in[u][c2]);
                      if (grr == gc) v += (float)e.gamma;
                      e.C.f32[o] = v;
                      if (up) {
                        e.C.f32[(long long)b * e.C.bstride + gc * e.C.ld + grr] = v;
                        colmx[c2] = fmaxf(colmx[c2], fabsf(v));
                      }
                      mx = fmaxf(mx, fabsf(v));
                      *sp = v;
                      break;
                    }
                    case EPI_M: {
                      const float v = fmaf((float)e.beta_in, in[u][c2], acc);
                      e.C.f32[o] = v;
                      const float rd = v - ((grr == gc) ? 1.0f : 0.0f);
                      if (up) {
                        e.C.f32[(long long)b * e.C.bstride + gc * e.C.ld + grr] = v;
                        colmx[c2] = fmaxf(colmx[c2], fabsf(v));
                      }
                      part += (mirror || up) ? 2.f * (rd * rd) : rd * rd;
                      mx = fmaxf(mx, fabsf(v));
                      *sp = v;
                      break;
                    }
                    case EPI_GRAM:
                      e.state[b][grr * e.cols + gc] = fmaf(e.beta, in[u][c2], (1.0f - e.beta) * acc);
                      break;
                    case EPI_U: {
                      const long long ou = grr * e.cols + gc;
                      if (e.out_dtype == PRECOND_BF16)
                        reinterpret_cast<__nv_bfloat16*>(e.out[b])[ou] = __float2bfloat16_rn(acc);
                      else
                        reinterpret_cast<float*>(e.out[b])[ou] = acc;
                      break;
                    }
                  }
                }
              }
            }
            if (track) {
              mx = warp_max(mx);
              if (ok && lane == 0 && grr < g.M) atomic_max_nonneg(&e.C.rowmax[(long long)b * e.C.rows + grr], mx);
            }
          }
        }
        if (diag_fix && track && ok) {
          // rows of the lower triangle: their entries are the upper triangle's columns
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) {
            const long long gc = tile_n + hc + c2 * 32 + lane;
            if (gc < g.N && colmx[c2] > 0.f) atomic_max_nonneg(&e.C.rowmax[(long long)b * e.C.rows + gc], colmx[c2]);
          }
        }
        if (mirror) {
          // the mirrored tile (rows tile_n.., columns tile_m..) = transpose of this one
          __syncwarp();
          epi_bar();
#pragma unroll 1
          for (int c0 = 0; c0 < TC_BN / 2 / EPI_WARPS; c0 += EPI_RB) {
            float st_in[EPI_RB][4];
#pragma unroll
            for (int u = 0; u < EPI_RB; ++u) {
              const long long gc = tile_n + hc + ew * (TC_BN / 2 / EPI_WARPS) + c0 + u;
#pragma unroll
              for (int r4 = 0; r4 < 4; ++r4) {
                const long long grr = tile_m + r4 * 32 + lane;
                st_in[u][r4] = (ok && e.kind == EPI_GRAM && gc < g.N && grr < g.M) ? e.state[b][gc * e.cols + grr] : 0.f;
              }
            }
#pragma unroll
            for (int u = 0; u < EPI_RB; ++u) {
              const int cl = ew * (TC_BN / 2 / EPI_WARPS) + c0 + u;   // tile column (in this half) = mirrored row
              const long long gc = tile_n + hc + cl;
              float mx = 0.f;
              if (ok && gc < g.N) {
#pragma unroll
                for (int r4 = 0; r4 < 4; ++r4) {
                  const int r = r4 * 32 + lane;             // tile row = mirrored column
                  const long long grr = tile_m + r;
                  if (grr < g.M) {
                    const float v = staging[r * SM::STG_LD + cl];
                    if (e.kind == EPI_GRAM) {
                      e.state[b][gc * e.cols + grr] = fmaf(e.beta, st_in[u][r4], (1.0f - e.beta) * v);
                    } else {
                      e.C.f32[(long long)b * e.C.bstride + gc * e.C.ld + grr] = v;
                      mx = fmaxf(mx, fabsf(v));
                    }
                  }
                }
              }
              if (track) {
                mx = warp_max(mx);
                if (ok && lane == 0 && gc < g.N) atomic_max_nonneg(&e.C.rowmax[(long long)b * e.C.rows + gc], mx);
              }
            }
          }
        }
      }
      if (e.kind == EPI_M) {
        const double pd = warp_sum((double)part);
        if (lane == 0) red[ew] = pd;
      }
      epi_bar();                          // staging free; residual parts visible
      if (e.kind == EPI_M && ew == 0) {
        double sum = 0.0;
#pragma unroll
        for (int w = 0; w < EPI_WARPS; ++w) sum += red[w];     // fixed order: deterministic
        epi_m_finish(e, b, sum, g.M, tl);
      }
      ++it;
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
