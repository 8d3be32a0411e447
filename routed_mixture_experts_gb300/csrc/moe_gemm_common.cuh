// moe_gemm_common.cuh -- pieces shared by the grouped-GEMM kernels (one-CTA and
// CTA-pair variants): tile decoding, bounded waits used while draining, and the
// fused epilogues that turn a TMEM accumulator row into the routed-expert
// outputs.
#pragma once

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace gemm {

// warp 0 TMA producer, warp 1 MMA issuer, warps 2..9 epilogue (two warps per
// TMEM lane quarter, each taking half of the tile's columns)
constexpr int kThreads = 320;
constexpr int kEpiThreads = 256;

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

// Staging of bf16 outputs: the epilogue threads write one 128-row x 64-column
// sub-tile (16 KB) into a shared-memory buffer in the 128-byte-swizzled layout of
// a 64 x 128 tensor-map box (each of the two warps of a lane quarter writes 32 of
// the 64 columns of its row), then one thread stores it with TMA.  Two buffers
// alternate; a buffer is rewritten only once its previous store has read it.
constexpr int kEpiStageBufs = 2;

__device__ __forceinline__ void epi_stage_store(const CUtensorMap* tm, uint32_t out0, int& seq,
                                                int et, int row, int half, const float (&v)[32],
                                                int x, int y) {
  const uint32_t buf = out0 + (uint32_t)(seq % kEpiStageBufs) * 16384u;
  if (et == 0) bulk_wait_read<kEpiStageBufs - 1>();
  named_bar_sync(1, kEpiThreads);
  const uint32_t rbase = buf + (uint32_t)row * 128u;
  const uint32_t sw = (uint32_t)(row & 7);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    st_shared_v4_u32(rbase + (((uint32_t)(4 * half + q) ^ sw) << 4),
                     pack_bf2(v[8 * q], v[8 * q + 1]), pack_bf2(v[8 * q + 2], v[8 * q + 3]),
                     pack_bf2(v[8 * q + 4], v[8 * q + 5]), pack_bf2(v[8 * q + 6], v[8 * q + 7]));
  fence_proxy_async_smem();
  named_bar_sync(1, kEpiThreads);
  if (et == 0) {
    tma_store_2d(tm, buf, x, y);
    bulk_commit();
  }
  ++seq;
}

__device__ __forceinline__ void load32_bf16(const uint16_t* src, float (&v)[32]) {
  float a[16], b[16];
  load16_bf16(src, a);
  load16_bf16(src + 16, b);
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    v[q] = a[q];
    v[16 + q] = b[q];
  }
}

// bf16-output epilogues.  One-output epilogues (W2 x score, plain store) walk
// the tile in 64-column sub-tiles, the thread owning row `row` handling columns
// [32*half, 32*half+32) of each, and leave through epi_stage_store (tmO0: the
// output tensor's map).  The three-output epilogues (SwiGLU: h and a; SwiGLU
// backward: dA and hs) store their rows directly, each thread taking one half
// of the tile's columns: staging three outputs through two buffers serialises
// them on the buffer reuse.
template <int BN, int EPI>
__device__ __forceinline__ void epilogue(const GemmArgs& a, const TileInfo& ti, int row,
                                         uint32_t tbase, int half, const CUtensorMap* tmO0,
                                         const CUtensorMap* tmO1, uint32_t out0, int et,
                                         int& seq) {
  const long long grow = (long long)ti.m0 + row;
  uint32_t r0[16], r1[16];
  const int ch = 32 * half;
  if constexpr (EPI == EPI_SWIGLU) {
    // direct row stores (three outputs per column block: h and both halves of a)
    constexpr int BNH = BN / 2;          // gate columns [0,BNH), up columns [BNH,BN)
    constexpr int WH = BNH / 2;          // this thread's half of them
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
  } else if constexpr (EPI == EPI_SCORE || EPI == EPI_STORE) {
    const float s = EPI == EPI_SCORE ? a.row_scale[grow] : 1.0f;
#pragma unroll 1
    for (int c = 0; c < BN; c += 64) {
      tmem_ld16(tbase + c + ch, r0);
      tmem_ld16(tbase + c + ch + 16, r1);
      tmem_ld_wait();
      float v[32];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        v[q] = s * __uint_as_float(r0[q]);         // R3 (score) or R5 on store
        v[16 + q] = s * __uint_as_float(r1[q]);
      }
      epi_stage_store(tmO0, out0, seq, et, row, half, v, ti.n0 + c, ti.m0);
    }
  } else if constexpr (EPI == EPI_DGRAD2) {
    // acc = g (columns = intermediate index i).  in0 = h [rows, I], in1 = a [rows, 2I],
    // out0 = dA [rows, 2I], out1 = hs [rows, I]; direct row stores.
    constexpr int W = BN / 2;
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

}  // namespace gemm
}  // namespace moe
