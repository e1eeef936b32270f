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
// accumulators in tensor memory; four epilogue warps read them back with
// tcgen05.ld.  Warp roles (192 threads): warp 0 TMA producer, warp 1 TMEM
// owner and MMA issuer, warps 2..5 epilogue.  Every mbarrier wait is
// bounded; on time-out the kernel records an error word and leaves the tile.
#pragma once

#include <cuda.h>
#include "engine.cuh"

namespace precond {

constexpr int TC_BM = 128, TC_BN = 128, TC_BK = 32;
constexpr int TC_THREADS = 192;
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
};

template <int S>
struct TcSmem {
  static constexpr int A_BYTES = TC_BM * TC_BK * 2;            // 8 KB per digit plane
  static constexpr int B_BYTES = TC_BN * TC_BK * 2;            // 8 KB
  static constexpr int STAGE_BYTES = S * (A_BYTES + B_BYTES);
  static constexpr int STAGES = (S == 4) ? 2 : 3;
  static constexpr int STG_LD = TC_BN + 1;                      // staging row stride (floats), bank-conflict free
  static constexpr int STAGING_BYTES = TC_BM * STG_LD * 4;
  static constexpr int TMEM_COLS = 512;                        // 3 x 128 used
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
__device__ __forceinline__ void tile_coords(int tl, int tiles_n, int sym, int& ti, int& tj) {
  if (!sym) {
    ti = tl / tiles_n;
    tj = tl % tiles_n;
    return;
  }
  int r = 0;
  while (tl >= tiles_n - r) {
    tl -= tiles_n - r;
    ++r;
  }
  ti = r;
  tj = r + tl;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Persistent: CTA c takes tiles c, c + gridDim.x, ...; tile t = (entry, row block,
// column block) with the column block fastest.  The producer and the MMA
// issuer run ahead through the shared-memory ring; the epilogue drains the
// tensor-memory accumulators of a tile into a shared staging tile, releases
// tensor memory (the next tile's MMAs start), then runs the element-wise
// epilogue from shared memory with coalesced global accesses.
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
  __shared__ double red[4];

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
        tile_coords(tl, tiles_n, g.sym, ti, tj);
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
        ++it;
      }
    }
  } else {
    // ------------------------------------------------ epilogue (warps 2..5)
    const int q = warp & 3;                 // TMEM lane quadrant of this warp (rows q*32 ..)
    const int ew = warp - 2;                // epilogue warp index 0..3
    const int et = threadIdx.x - 64;        // epilogue thread index 0..127
    const double c0 = (double)e.inv_scale * ldexp(1.0, -2 * DIGIT_BITS);
    uint32_t it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const int b = t / tiles_per_entry, tl = t % tiles_per_entry;
      if (epi_skip(e, b)) continue;
      int ti, tj;
      tile_coords(tl, tiles_n, g.sym, ti, tj);
      const int tile_m = ti * TC_BM, tile_n = tj * TC_BN;
      const bool mirror = g.sym && ti != tj;
      const int za = g.a_index ? g.a_index[b] : b;
      const int zb = g.b_index ? g.b_index[b] : b;
      // column scales of this tile
      {
        const long long gc = tile_n + et;
        colscale[et] = (gc < g.N) ? (g.b_rowscale ? g.b_rowscale[(long long)zb * g.b_rs_stride + gc] : g.b_scale) : 0.f;
      }
      const bool ok = mbar_wait(accum_bar, it & 1, g.err);
      tc_fence_after();
      epi_bar();
      // ---- drain: tensor memory -> staging (scaled fp32)
      const int row = q * 32 + lane;
      const long long gr = tile_m + row;
      const double sa = (gr < g.M) ? (g.a_rowscale ? (double)g.a_rowscale[(long long)za * g.a_rs_stride + gr]
                                                    : (double)g.a_scale) : 0.0;
      const float rs = (float)(c0 * sa);
      float* srow = staging + row * SM::STG_LD;
#pragma unroll 1
      for (int ch = 0; ch < TC_BN / 32; ++ch) {
        float v0[32], v1[32], v2[32];
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(ch * 32);
        tmem_ld32(taddr, v0);
        tmem_ld32(taddr + 128, v1);
        tmem_ld32(taddr + 256, v2);
#pragma unroll
        for (int j = 0; j < 32; ++j) srow[ch * 32 + j] = ((v0[j] + v1[j]) + v2[j]) * rs * colscale[ch * 32 + j];
      }
      tc_fence_before();
      epi_bar();
      if (et == 0) mbar_arrive(tmem_empty_bar);    // tensor memory may take the next tile
      // ---- element-wise epilogue from staging
      float part = 0.f;
      if (ok) {
        if (e.kind == EPI_VT) {
          // transposed output: warp ew takes tile columns ew*32.., lanes run over rows
          for (int cc = 0; cc < 32; ++cc) {
            const int c = ew * 32 + cc;
            const long long gc = tile_n + c;
            float mx = 0.f;
            if (gc < g.N) {
#pragma unroll
              for (int r4 = 0; r4 < 4; ++r4) {
                const int r = r4 * 32 + lane;
                const long long grr = tile_m + r;
                if (grr < g.M) {
                  const float v = staging[r * SM::STG_LD + c];
                  e.C.f32[(long long)b * e.C.bstride + gc * e.C.ld + grr] = v;
                  mx = fmaxf(mx, fabsf(v));
                }
              }
            }
            mx = warp_max(mx);
            if (lane == 0 && gc < g.N && e.C.rowmax) atomic_max_nonneg(&e.C.rowmax[(long long)b * e.C.rows + gc], mx);
          }
        } else {
          const bool track = (e.kind == EPI_AFF || e.kind == EPI_M) && e.C.rowmax;
          for (int rr = 0; rr < 32; ++rr) {
            const int r = ew * 32 + rr;
            const long long grr = tile_m + r;
            float mx = 0.f;
            if (grr < g.M) {
#pragma unroll
              for (int c4 = 0; c4 < 4; ++c4) {
                const int c = c4 * 32 + lane;
                const long long gc = tile_n + c;
                if (gc < g.N) {
                  float* sp = &staging[r * SM::STG_LD + c];
                  const float acc = *sp;
                  const float v = epi_apply_tc(e, b, grr, gc, acc);
                  if (e.kind == EPI_M) {
                    part += mirror ? 2.f * v : v;
                    const long long o = (long long)b * e.C.bstride + grr * e.C.ld + gc;
                    mx = fmaxf(mx, fabsf(e.C.f32[o]));
                    if (g.sym) *sp = e.C.f32[o];
                  } else {
                    mx = fmaxf(mx, v);
                    if (g.sym && e.kind != EPI_GRAM) *sp = e.C.f32[(long long)b * e.C.bstride + grr * e.C.ld + gc];
                  }
                }
              }
            }
            if (track) {
              mx = warp_max(mx);
              if (lane == 0 && grr < g.M) atomic_max_nonneg(&e.C.rowmax[(long long)b * e.C.rows + grr], mx);
            }
          }
          if (g.sym && !mirror && (e.kind == EPI_AFF || e.kind == EPI_M)) {
            // diagonal tile: its lower triangle takes the upper triangle's values, so
            // the result is exactly symmetric (the iteration amplifies any
            // antisymmetric part while M is far from I)
            epi_bar();
            for (int rr = 0; rr < 32; ++rr) {
              const int r = ew * 32 + rr;
              const long long grr = tile_m + r;
              if (grr >= g.M) continue;
#pragma unroll
              for (int c4 = 0; c4 < 4; ++c4) {
                const int c = c4 * 32 + lane;
                const long long gc = tile_n + c;
                if (c < r && gc < g.N)
                  e.C.f32[(long long)b * e.C.bstride + grr * e.C.ld + gc] = staging[c * SM::STG_LD + r];
              }
            }
          }
          if (mirror) {
            // the mirrored tile (rows tile_n.., columns tile_m..) = transpose of this one
            __syncwarp();
            epi_bar();
            for (int cc = 0; cc < 32; ++cc) {
              const int c = ew * 32 + cc;                 // tile column = mirrored row
              const long long gc = tile_n + c;
              float mx = 0.f;
              if (gc < g.N) {
#pragma unroll
                for (int r4 = 0; r4 < 4; ++r4) {
                  const int r = r4 * 32 + lane;            // tile row = mirrored column
                  const long long grr = tile_m + r;
                  if (grr < g.M) {
                    const float v = staging[r * SM::STG_LD + c];
                    if (e.kind == EPI_GRAM) {
                      float* st = e.state[b];
                      const long long o = gc * e.cols + grr;
                      st[o] = fmaf(e.beta, st[o], (1.0f - e.beta) * v);
                    } else {
                      e.C.f32[(long long)b * e.C.bstride + gc * e.C.ld + grr] = v;
                      mx = fmaxf(mx, fabsf(v));
                    }
                  }
                }
              }
              if (track) {
                mx = warp_max(mx);
                if (lane == 0 && gc < g.N) atomic_max_nonneg(&e.C.rowmax[(long long)b * e.C.rows + gc], mx);
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
      if (e.kind == EPI_M && ew == 0) epi_m_finish(e, b, red[0] + red[1] + red[2] + red[3], g.M, tl);
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
