// moe_gemm.cu -- persistent grouped GEMM on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in tensor memory), fed by TMA through an mbarrier
// pipeline, with the routed-expert epilogues fused:
//
//   W13 FPROP  + SwiGLU            ("Dist-MoE" note, "What it is selling": W13 -> SwiGLU;
//   W2  FPROP  x routing score      nvfp4moe README, "MoE layer": FC1 + gated activation,
//   DGRAD W2   + SwiGLU backward    FC2, probability weighting; "Training": input, weight
//              + score-grad partials and router gradients)
//   DGRAD W13
//   WGRAD      (fp32 in-place accumulation, "What it is selling")
//
// Tile: 128 rows (M) x BN columns (N), K in stages of 64 bf16 (one 128-byte
// swizzle atom).  One CTA per SM, 10 warps:
//   warp 0      TMA producer (one lane issues)
//   warp 1      TMEM allocator and MMA issuer (one lane issues)
//   warps 2..9  epilogue: warp w reads TMEM lanes 32*(w%4)..+31, i.e. one output
//               row per thread, through tcgen05.ld; warps 2..5 take the first
//               half of the tile's columns, warps 6..9 the second
// The accumulator is double buffered in TMEM (2 x BN fp32 columns) so the
// epilogue of tile i overlaps the main loop of tile i+1.
//
// Every mbarrier wait is bounded (moe::mbar_wait); a wait that gives up records
// MOE_ERR_TIMEOUT, all roles leave their loops, outstanding copies and MMAs are
// drained with bounded waits, and TMEM is freed before the CTA exits.

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

// warp 0 TMA producer, warp 1 MMA issuer, warps 2..9 epilogue (two warps per
// TMEM lane quarter, each taking half of the tile's columns)
constexpr int kThreads = 320;
constexpr int kEpiThreads = 256;
constexpr int kBoxBytes = 64 * 64 * 2;  // every TMA box is 64 x 64 bf16 = 8 KB

struct TileInfo {
  int e;        // expert
  int m0;       // first output row of the tile (padded row, or weight row in wgrad mode)
  int n0;       // first output column
  int nt;       // n tile index
  int kb;       // number of 64-wide K blocks
  int krow0;    // wgrad mode: first routed row of the K range
};

__device__ __forceinline__ int count_tiles(const GemmArgs& a) {
  if (a.wgrad) return (*a.num_nonempty) * a.m_tiles * a.n_tiles;
  return (*a.num_mtiles) * a.n_tiles;
}

template <int BN>
__device__ __forceinline__ TileInfo decode_tile(const GemmArgs& a, int tile) {
  TileInfo ti;
  if (a.wgrad) {
    const int per_e = a.m_tiles * a.n_tiles;
    const int q = tile / per_e;
    const int rem = tile - q * per_e;
    ti.e = a.expert_order[q];
    const int mt = rem / a.n_tiles;
    ti.nt = rem - mt * a.n_tiles;
    ti.m0 = mt * kBM;
    ti.n0 = ti.nt * BN;
    ti.krow0 = a.off_pad[ti.e];
    ti.kb = (a.off_pad[ti.e + 1] - ti.krow0) / kBK;
  } else {
    const int mt = tile / a.n_tiles;
    ti.nt = tile - mt * a.n_tiles;
    ti.e = a.tile_expert ? a.tile_expert[mt] : 0;
    ti.m0 = mt * kBM;
    ti.n0 = ti.nt * BN;
    ti.kb = a.k_blocks;
    ti.krow0 = 0;
  }
  return ti;
}

// Bounded wait that ignores the abort flag (used only while draining).
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 200000000ull) return false;  // 200 ms
  }
  return true;
}

// AND of `v` over the 256 epilogue threads (named barrier 1).
__device__ __forceinline__ int epi_bar_and(int v) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.s32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 256, p;\n\t"
      "selp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(v)
      : "memory");
  return r;
}

__device__ __forceinline__ float swiglu_fwd(float G, float U, float L) {
  if (L > 0.f) {
    G = fminf(fmaxf(G, -L), L);
    U = fminf(fmaxf(U, -L), L);
  }
  const float silu = G / (1.0f + expf(-G));
  return silu * U;
}

__device__ __forceinline__ void store16_bf16(uint16_t* dst, const float (&v)[16]) {
  uint4 lo, hi;
  lo.x = pack_bf2(v[0], v[1]);   lo.y = pack_bf2(v[2], v[3]);
  lo.z = pack_bf2(v[4], v[5]);   lo.w = pack_bf2(v[6], v[7]);
  hi.x = pack_bf2(v[8], v[9]);   hi.y = pack_bf2(v[10], v[11]);
  hi.z = pack_bf2(v[12], v[13]); hi.w = pack_bf2(v[14], v[15]);
  reinterpret_cast<uint4*>(dst)[0] = lo;
  reinterpret_cast<uint4*>(dst)[1] = hi;
}

__device__ __forceinline__ void load16_bf16(const uint16_t* src, float (&v)[16]) {
  const uint4 lo = reinterpret_cast<const uint4*>(src)[0];
  const uint4 hi = reinterpret_cast<const uint4*>(src)[1];
  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// ---------------------------------------------------------------------------
// epilogues: one thread owns one output row (`row` within the tile) and reads
// its accumulator columns from TMEM at `tbase` (lane quarter already folded in).

// MXFP8 W13 epilogue: like the bf16 one (R1, SwiGLU, R2), then h is quantised
// along I in 32-column blocks (codes to a.hq, tiled E8M0 scales to a.hsf) as the
// A operand of the block-scaled W2 GEMM; the bf16 h is kept for inspection.
template <int BN>
__device__ __forceinline__ void epilogue_swiglu_mx(const GemmArgs& a, const TileInfo& ti, int row,
                                                   uint32_t tbase, int half) {
  constexpr int BNH = BN / 2;
  constexpr int W = BNH / 2;             // columns of this thread's half
  const long long grow = (long long)ti.m0 + row;
  const int c0 = ti.nt * BNH;
  uint16_t* h = static_cast<uint16_t*>(a.out0) + grow * a.ld0 + c0;
  uint8_t* hq = a.hq + grow * a.ld0 + c0;
  uint32_t g0[16], g1[16], u0[16], u1[16];
#pragma unroll 1
  for (int c = half * W; c < (half + 1) * W; c += 32) {
    tmem_ld16(tbase + c, g0);
    tmem_ld16(tbase + c + 16, g1);
    tmem_ld16(tbase + BNH + c, u0);
    tmem_ld16(tbase + BNH + c + 16, u1);
    tmem_ld_wait();
    float hv[32];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const float G0 = bf2f(f2bf(__uint_as_float(g0[q]))), U0 = bf2f(f2bf(__uint_as_float(u0[q])));
      const float G1 = bf2f(f2bf(__uint_as_float(g1[q]))), U1 = bf2f(f2bf(__uint_as_float(u1[q])));
      hv[q] = bf2f(f2bf(swiglu_fwd(G0, U0, a.clamp)));            // R2
      hv[16 + q] = bf2f(f2bf(swiglu_fwd(G1, U1, a.clamp)));
    }
    float lo[16], hi[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      lo[q] = hv[q];
      hi[q] = hv[16 + q];
    }
    store16_bf16(h + c, lo);
    store16_bf16(h + c + 16, hi);
    uint32_t w[8];
    const uint8_t sc = mx_quant32(hv, w);
    reinterpret_cast<uint4*>(hq + c)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4*>(hq + c)[1] = make_uint4(w[4], w[5], w[6], w[7]);
    a.hsf[mx_sf_offset(grow >> 7, (int)(grow & 127), (c0 + c) >> 5, a.hsf_ngr)] = sc;
  }
}

template <int BN, int EPI>
__device__ __forceinline__ void epilogue(const GemmArgs& a, const TileInfo& ti, int row,
                                         uint32_t tbase, int half) {
  const long long grow = (long long)ti.m0 + row;
  uint32_t r0[16], r1[16];
  constexpr int W = BN / 2;              // columns of this thread's half (BN-wide epilogues)
  if constexpr (EPI == EPI_SWIGLU) {
    constexpr int BNH = BN / 2;          // gate columns [0,BNH), up columns [BNH,BN)
    constexpr int WH = BNH / 2;
    const int c0 = ti.nt * BNH;          // first intermediate column of this tile
    uint16_t* h = static_cast<uint16_t*>(a.out0) + grow * a.ld0 + c0;
    uint16_t* av = static_cast<uint16_t*>(a.out1) + grow * a.ld1 + c0;
#pragma unroll 1
    for (int c = half * WH; c < (half + 1) * WH; c += 16) {
      tmem_ld16(tbase + c, r0);
      tmem_ld16(tbase + BNH + c, r1);
      tmem_ld_wait();
      float G[16], U[16], hv[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        G[q] = bf2f(f2bf(__uint_as_float(r0[q])));   // R1
        U[q] = bf2f(f2bf(__uint_as_float(r1[q])));
        hv[q] = swiglu_fwd(G[q], U[q], a.clamp);      // R2 on store
      }
      store16_bf16(h + c, hv);
      if (a.save) {
        store16_bf16(av + c, G);
        store16_bf16(av + a.I + c, U);
      }
    }
  } else if constexpr (EPI == EPI_SCORE) {
    const float s = a.row_scale[grow];
    uint16_t* out = static_cast<uint16_t*>(a.out0) + grow * a.ld0 + ti.n0;
#pragma unroll 1
    for (int c = half * W; c < (half + 1) * W; c += 16) {
      tmem_ld16(tbase + c, r0);
      tmem_ld_wait();
      float v[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) v[q] = s * __uint_as_float(r0[q]);   // R3 on store
      store16_bf16(out + c, v);
    }
  } else if constexpr (EPI == EPI_STORE) {
    uint16_t* out = static_cast<uint16_t*>(a.out0) + grow * a.ld0 + ti.n0;
#pragma unroll 1
    for (int c = half * W; c < (half + 1) * W; c += 16) {
      tmem_ld16(tbase + c, r0);
      tmem_ld_wait();
      float v[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) v[q] = __uint_as_float(r0[q]);
      store16_bf16(out + c, v);
    }
  } else if constexpr (EPI == EPI_DGRAD2) {
    // acc = g (columns = intermediate index i).  in0 = h [rows, I], in1 = a [rows, 2I],
    // out0 = dA [rows, 2I], out1 = hs [rows, I].
    const float s = a.row_scale[grow];
    const float L = a.clamp;
    const uint16_t* hrow = static_cast<const uint16_t*>(a.in0) + grow * a.ldi0 + ti.n0;
    const uint16_t* arow = static_cast<const uint16_t*>(a.in1) + grow * a.ldi1 + ti.n0;
    uint16_t* darow = static_cast<uint16_t*>(a.out0) + grow * a.ld0 + ti.n0;
    uint16_t* hsrow = static_cast<uint16_t*>(a.out1) + grow * a.ld1 + ti.n0;
    float part = 0.f;
#pragma unroll 1
    for (int c = half * W; c < (half + 1) * W; c += 16) {
      tmem_ld16(tbase + c, r0);
      float hv[16], ag[16], au[16];
      load16_bf16(hrow + c, hv);
      load16_bf16(arow + c, ag);
      load16_bf16(arow + a.I + c, au);
      tmem_ld_wait();
      float dg[16], du[16], hs[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float g = __uint_as_float(r0[q]);
        part += hv[q] * g;
        float G = ag[q], U = au[q], mg = 1.f, mu = 1.f;
        if (L > 0.f) {
          if (G < -L || G > L) mg = 0.f;
          if (U < -L || U > L) mu = 0.f;
          G = fminf(fmaxf(G, -L), L);
          U = fminf(fmaxf(U, -L), L);
        }
        const float dh = s * g;
        const float sig = 1.0f / (1.0f + expf(-G));
        const float silu = G * sig;
        const float dsilu = sig * (1.0f + G * (1.0f - sig));
        dg[q] = dh * U * dsilu * mg;       // R4 on store
        du[q] = dh * silu * mu;
        hs[q] = s * hv[q];                 // R7 on store
      }
      store16_bf16(darow + c, dg);
      store16_bf16(darow + a.I + c, du);
      store16_bf16(hsrow + c, hs);
    }
    // one partial per (n tile, column half), in column order
    a.pdscore[grow * (2 * a.n_tiles) + 2 * ti.nt + half] = part;
  }
}

// WGRAD epilogue: the accumulator tile is written, 32 columns at a time, into one
// of kWgradBufs 16 KB shared-memory buffers (128 rows x 32 fp32, 128-byte swizzle, the
// layout of the fp32 tensor map), and the TMA unit adds each buffer into the
// fp32 gradient in global memory (cp.reduce.async.bulk.tensor .add).  The
// read-modify-write then happens in L2 with many bytes in flight, instead of
// through per-thread loads and stores.
constexpr int kWgradBufs = 5;   // fp32 staging buffers of 16 KB (adds in flight per SM)

template <int BN>
__device__ __forceinline__ void epilogue_wgrad(const GemmArgs& a, const CUtensorMap* tmC,
                                               const TileInfo& ti, int row, uint32_t tbase,
                                               uint32_t stage_smem, int et, int half, int& sub) {
  if (ti.kb == 0) return;
  const int ybase = ti.e * a.m_tiles * kBM + ti.m0;
  uint32_t r0[16];
#pragma unroll 1
  for (int c = 0; c < BN; c += 32) {
    const uint32_t buf = stage_smem + (uint32_t)(sub % kWgradBufs) * 16384u;
    if (et == 0) bulk_wait_read<kWgradBufs - 1>();   // this buffer's previous add has read it
    named_bar_sync(1, kEpiThreads);
    // this thread's half: 16 of the sub-tile's 32 columns (16-byte chunks 4h..4h+3)
    tmem_ld16(tbase + c + 16 * half, r0);
    tmem_ld_wait();
    const uint32_t rbase = buf + (uint32_t)row * 128u;
    const uint32_t sw = (uint32_t)(row & 7);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      st_shared_v4(rbase + (((uint32_t)(q + 4 * half) ^ sw) << 4), __uint_as_float(r0[4 * q]),
                   __uint_as_float(r0[4 * q + 1]), __uint_as_float(r0[4 * q + 2]),
                   __uint_as_float(r0[4 * q + 3]));
    fence_proxy_async_smem();
    named_bar_sync(1, kEpiThreads);
    if (et == 0) {
      tma_reduce_add_2d(tmC, buf, ti.n0 + c, ybase);
      bulk_commit();
    }
    ++sub;
  }
}

template <int BN, int EPI, bool MX>
struct GemmShape {
  // A stage holds 128 rows (A) and BN rows (B) of 128 bytes of K: 64 bf16 or
  // 128 E4M3 elements; MXFP8 stages also carry the 512-byte scale chunks of A
  // and of B for those 128 K-elements (padded to keep stages 1024-aligned).
  static constexpr int A_BYTES = kBM * 128;                    // 16 KB
  static constexpr int B_BYTES = BN * 128;
  static constexpr int SF_STAGE_BYTES = MX ? 1024 : 0;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SF_STAGE_BYTES;
  // WGRAD keeps 64 KB for its four fp32 staging buffers and needs few stages
  // (its K loop is one expert's rows and it is bound by the gradient traffic).
  static constexpr int OUT_BYTES = EPI == EPI_WGRAD ? kWgradBufs * 16384 : 0;
  static constexpr int STAGE_BUDGET = (EPI == EPI_WGRAD ? 226 : 208) * 1024 - OUT_BYTES;
  static constexpr int STAGES = STAGE_BUDGET / STAGE_BYTES > 8 ? 8 : STAGE_BUDGET / STAGE_BYTES;
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + OUT_BYTES + BAR_BYTES + 1024;
  // accumulators (2 x BN columns), then for MXFP8 eight scale columns per stage
  // (4 for A, 4 for B)
  static constexpr uint32_t SF_COL0 = 2 * BN;
  static constexpr uint32_t TMEM_COLS = MX ? 512 : 2 * BN;
  static_assert(!MX || SF_COL0 + 8 * STAGES <= 512, "TMEM budget");
};

template <int BN, bool A_MN, bool B_MN, int EPI, bool MX>
__global__ void __launch_bounds__(kThreads, 1)
    k_grouped_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const GemmArgs args) {
  using S = GemmShape<BN, EPI, MX>;
  constexpr int STAGES = S::STAGES;
  constexpr uint32_t IDESC = MX ? idesc_mxf8(kBM, BN) : idesc_bf16(kBM, BN, A_MN, B_MN);
  constexpr int KE = MX ? 128 : kBK;     // K elements per stage (128 bytes per row)
  static_assert(!MX || (!A_MN && !B_MN && BN == 128), "MXFP8: K-major operands, BN = 128");
  static_assert(S::SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN");

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t tmem_holder;
  __shared__ int num_tiles_s;
  __shared__ volatile int abort_s;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * S::STAGE_BYTES + S::OUT_BYTES);
  // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], drain
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t wlim = args.wait_limit_ns ? args.wait_limit_ns : kWaitLimitNs;

  if (threadIdx.x == 0) {
    num_tiles_s = count_tiles(args);
    abort_s = 0;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), kEpiThreads);
    }
    mbar_init(drain_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int num_tiles = num_tiles_s;
  if ((int)blockIdx.x >= num_tiles) return;  // whole CTA leaves before touching TMEM

  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_holder), S::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (EPI == EPI_WGRAD) tma_prefetch_desc(&tmC);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_holder;
  const uint32_t stage0 = smem_u32(smem);


  if (warp == 0) {
    // ---------------- TMA producer ----------------
    int stage = 0;
    uint32_t phase = 0;
    int issued_parity[STAGES];
#pragma unroll
    for (int s = 0; s < STAGES; ++s) issued_parity[s] = -1;
    bool ok = true;
    for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
      const TileInfo ti = decode_tile<BN>(args, tile);
      for (int kb = 0; kb < ti.kb; ++kb) {
        int w = 1;
        if (lane == 0) w = mbar_wait(empty_bar(stage), phase ^ 1u, &abort_s, args.err, 1, wlim);
        ok = __shfl_sync(0xffffffffu, w, 0) != 0;
        if (!ok) break;
        if (lane == 0) {
          const uint32_t fb = full_bar(stage);
          const uint32_t sa = stage0 + stage * S::STAGE_BYTES;
          const uint32_t sb = sa + S::A_BYTES;
          mbar_arrive_expect_tx(fb, S::STAGE_BYTES);
          if constexpr (MX) {
            // the 512-byte scale chunks of this K group: A's row block, B's row block
            const uint32_t ssf = sb + S::B_BYTES;
            const long long ga = ((long long)(ti.m0 >> 7) * args.sf_ngr + kb) * 512;
            const long long gb =
                (((long long)ti.e * args.b_blocks_per_expert + ti.nt) * args.sf_ngr + kb) * 512;
            bulk_g2s(ssf, args.sfa + ga, 512u, fb);
            bulk_g2s(ssf + 512u, args.sfb + gb, 512u, fb);
          }
          // A: 128 rows x 64 K
          if (A_MN) {
            // tensor [rows(K), M]: boxes cover 64 M columns x 64 K rows
            tma_load_2d(sa, &tmA, ti.m0, ti.krow0 + kb * kBK, fb);
            tma_load_2d(sa + kBoxBytes, &tmA, ti.m0 + 64, ti.krow0 + kb * kBK, fb);
          } else {
            // tensor [rows, K]: boxes cover 128 bytes of K x 64 rows
            tma_load_2d(sa, &tmA, kb * KE, ti.m0, fb);
            tma_load_2d(sa + kBoxBytes, &tmA, kb * KE, ti.m0 + 64, fb);
          }
          // B: BN rows (N) x 64 K
#pragma unroll
          for (int b = 0; b < BN / 64; ++b) {
            if (args.wgrad) {
              tma_load_2d(sb + b * kBoxBytes, &tmB, ti.n0 + 64 * b, ti.krow0 + kb * kBK, fb);
            } else if (B_MN) {
              // tensor [E*K, N]: 64 N columns x 64 K rows of expert e
              tma_load_2d(sb + b * kBoxBytes, &tmB, ti.n0 + 64 * b,
                          ti.e * args.b_expert_rows + kb * kBK, fb);
            } else if (EPI == EPI_SWIGLU) {
              // tensor [E*2I, d]: gate rows then up rows of this tile's columns
              constexpr int NB2 = BN / 128;   // boxes per half
              const int half = b / (NB2 > 0 ? NB2 : 1);
              const int bi = b - half * NB2;
              const int row = ti.e * args.b_expert_rows + half * args.b_half_rows +
                              ti.nt * (BN / 2) + 64 * bi;
              tma_load_2d(sb + b * kBoxBytes, &tmB, kb * KE, row, fb);
            } else {
              // tensor [E*N, K]
              tma_load_2d(sb + b * kBoxBytes, &tmB, kb * KE,
                          ti.e * args.b_expert_rows + ti.n0 + 64 * b, fb);
            }
          }
          issued_parity[stage] = (int)phase;
        }
        __syncwarp();
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (lane == 0) {
      if (!abort_s) {
        // producer tail: every issued stage has been released by the MMA commits
        for (int s = 0; s < STAGES; ++s) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, &abort_s, args.err, 2, wlim)) break;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (abort_s) {
        // drain: let every issued copy land before the CTA can exit
        for (int s = 0; s < STAGES; ++s)
          if (issued_parity[s] >= 0) mbar_wait_drain(full_bar(s), (uint32_t)issued_parity[s]);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
      const TileInfo ti = decode_tile<BN>(args, tile);
      int w = 1;
      if (lane == 0) w = mbar_wait(tempty_bar(acc), acc_phase ^ 1u, &abort_s, args.err, 3, wlim);
      // failure-path test: wait on the drain barrier, which nothing has arrived at
      if (args.stall_mma && lane == 0 && w) w = mbar_wait(drain_bar, 0, &abort_s, args.err, 9, wlim);
      ok = __shfl_sync(0xffffffffu, w, 0) != 0;
      if (!ok) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
      for (int kb = 0; kb < ti.kb; ++kb) {
        w = 1;
        if (lane == 0) w = mbar_wait(full_bar(stage), phase, &abort_s, args.err, 4, wlim);
        ok = __shfl_sync(0xffffffffu, w, 0) != 0;
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t sa = stage0 + stage * S::STAGE_BYTES;
          const uint32_t sb = sa + S::A_BYTES;
          if constexpr (MX) {
            // this stage's scales -> its own 8 TMEM columns (reused only after the
            // stage is released, i.e. after these MMAs have completed); then four
            // 32-element K steps, step j reading scale byte j
            const uint32_t ssf = sb + S::B_BYTES;
            const uint32_t sfa_t = tmem_base + S::SF_COL0 + 8u * (uint32_t)stage;
            const uint32_t sfb_t = sfa_t + 4u;
            tmem_cp_32x128b_x4(sfa_t, smem_desc_noswz(ssf, 512u, 128u));
            tmem_cp_32x128b_x4(sfb_t, smem_desc_noswz(ssf + 512u, 512u, 128u));
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint64_t adesc = smem_desc_sw128(sa + j * 32, 16, 1024);
              const uint64_t bdesc = smem_desc_sw128(sb + j * 32, 16, 1024);
              umma_mxf8(d_tmem, adesc, bdesc, idesc_sf_ids(IDESC, (uint32_t)j, (uint32_t)j),
                        sfa_t, sfb_t, (kb | j) != 0 ? 1u : 0u);
            }
          } else {
#pragma unroll
          for (int k16 = 0; k16 < kBK / 16; ++k16) {
            // K-major: rows of 128 B, 8-row groups 1024 B apart; K step = 32 B.
            // MN-major: 64-wide MN atoms 8 KB apart (LBO), 8-row K groups 1024 B
            // apart (SBO); K step of 16 rows = 2048 B.
            const uint64_t adesc = A_MN ? smem_desc_sw128(sa + k16 * 2048, 8192, 1024)
                                        : smem_desc_sw128(sa + k16 * 32, 16, 1024);
            const uint64_t bdesc = B_MN ? smem_desc_sw128(sb + k16 * 2048, 8192, 1024)
                                        : smem_desc_sw128(sb + k16 * 32, 16, 1024);
            umma_f16(d_tmem, adesc, bdesc, IDESC, (kb | k16) != 0 ? 1u : 0u);
          }
          }
          umma_commit(empty_bar(stage));
        }
        __syncwarp();
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) umma_commit(tfull_bar(acc));
      __syncwarp();
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (abort_s && lane == 0) {
      // drain: wait for every MMA issued so far before TMEM is freed
      umma_commit(drain_bar);
      mbar_wait_drain(drain_bar, 0);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int et = threadIdx.x - 64;          // 0..255 over the epilogue warps
    const int half = (warp - 2) >> 2;         // warps 2..5: columns' first half, 6..9: second
    int acc = 0;
    uint32_t acc_phase = 0;
    int sub = 0;                              // WGRAD staging-buffer sequence number
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      const TileInfo ti = decode_tile<BN>(args, tile);
      int w = 1;
      if (lane == 0) w = mbar_wait(tfull_bar(acc), acc_phase, &abort_s, args.err, 5, wlim);
      // all eight epilogue warps leave together, so their named barriers stay matched
      const int ok_warp = __shfl_sync(0xffffffffu, w, 0);
      if (EPI == EPI_WGRAD) {
        if (epi_bar_and(ok_warp) == 0) break;
      } else if (ok_warp == 0) {
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
      if constexpr (EPI == EPI_WGRAD)
        epilogue_wgrad<BN>(args, &tmC, ti, row, tbase, stage0 + STAGES * S::STAGE_BYTES, et, half,
                           sub);
      else if constexpr (MX && EPI == EPI_SWIGLU)
        epilogue_swiglu_mx<BN>(args, ti, row, tbase, half);
      else
        epilogue<BN, EPI>(args, ti, row, tbase, half);
      tc_fence_before();
      mbar_arrive(tempty_bar(acc));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (EPI == EPI_WGRAD && et == 0) bulk_wait_all();   // every gradient add has landed
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, S::TMEM_COLS);
  }
}

template <int BN, bool A_MN, bool B_MN, int EPI, bool MX>
cudaError_t launch_one(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                       const GemmArgs& args, int grid, cudaStream_t stream) {
  auto kern = k_grouped_gemm<BN, A_MN, B_MN, EPI, MX>;
  const int smem = GemmShape<BN, EPI, MX>::SMEM_BYTES;
  static bool configured = false;   // attribute set once per process (same device image)
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  kern<<<grid, kThreads, smem, stream>>>(ta, tb, tc, args);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm(int epi, int bn, bool a_mn, bool b_mn, const CUtensorMap& ta,
                        const CUtensorMap& tb, const CUtensorMap& tc, const GemmArgs& args,
                        int grid, cudaStream_t stream, bool mx) {
  if (mx) {
    if (epi == EPI_SWIGLU && bn == 128 && !a_mn && !b_mn)
      return launch_one<128, false, false, EPI_SWIGLU, true>(ta, tb, tc, args, grid, stream);
    if (epi == EPI_SCORE && bn == 128 && !a_mn && !b_mn)
      return launch_one<128, false, false, EPI_SCORE, true>(ta, tb, tc, args, grid, stream);
    return cudaErrorInvalidValue;
  }
#define MOE_CASE(EPI_, BN_, AMN_, BMN_)                                     \
  if (epi == EPI_ && bn == BN_ && a_mn == AMN_ && b_mn == BMN_)             \
    return launch_one<BN_, AMN_, BMN_, EPI_, false>(ta, tb, tc, args, grid, stream);
  MOE_CASE(EPI_SWIGLU, 128, false, false)
  MOE_CASE(EPI_SWIGLU, 256, false, false)
  MOE_CASE(EPI_SCORE, 128, false, false)
  MOE_CASE(EPI_SCORE, 256, false, false)
  MOE_CASE(EPI_STORE, 64, false, false)
  MOE_CASE(EPI_STORE, 128, false, false)
  MOE_CASE(EPI_STORE, 256, false, false)
  MOE_CASE(EPI_STORE, 64, false, true)
  MOE_CASE(EPI_STORE, 128, false, true)
  MOE_CASE(EPI_STORE, 256, false, true)
  MOE_CASE(EPI_DGRAD2, 64, false, true)
  MOE_CASE(EPI_DGRAD2, 128, false, true)
  MOE_CASE(EPI_DGRAD2, 256, false, true)
  MOE_CASE(EPI_WGRAD, 64, true, true)
  MOE_CASE(EPI_WGRAD, 128, true, true)
  MOE_CASE(EPI_WGRAD, 256, true, true)
#undef MOE_CASE
  return cudaErrorInvalidValue;
}

}  // namespace moe
