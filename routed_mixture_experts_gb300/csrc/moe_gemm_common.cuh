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
  return (a.mtile_list ? *a.list_count : *a.num_mtiles) * a.n_tiles;
}

// The r-th tile of this CTA (persistent kernels: every role of a CTA walks the
// same sequence).  Round-robin over the grid; weight-gradient tiles, which come
// longest expert first and so shrink from one round to the next, alternate the
// direction of each round (tile r*G + b, then r*G + G-1-b, ...), so the CTAs that
// drew the longest tiles of one round draw the shortest of the next.  Only the
// last round can hold tiles past the end, so the sequence ends at the first one.
__device__ __forceinline__ int cta_tile(const GemmArgs& a, int r) {
  const int G = (int)gridDim.x, b = (int)blockIdx.x;
  return r * G + ((a.wgrad && (r & 1)) ? G - 1 - b : b);
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
    ti.kb = (a.off_pad[ti.e + 1] - ti.krow0) / (a.wgrad_kstep ? a.wgrad_kstep : kBK);
  } else {
    const int q = tile / a.n_tiles;
    ti.nt = tile - q * a.n_tiles;
    const int mt = a.mtile_list ? a.mtile_list[q] : q;
    ti.e = a.tile_expert ? a.tile_expert[mt] : 0;
    ti.m0 = mt * kBM;
    ti.n0 = ti.nt * BN;
    ti.kb = a.k_blocks;
    ti.krow0 = 0;
  }
  return ti;
}

// The order in which a CTA's MMA issuer consumes K stages, as segments: a run
// of K blocks [k0, k1) of one tile on one accumulator; `last` ends the tile, and
// the tiles' epilogues run in the order their last segments come.  Every role
// of the CTA (producer, MMA issuer, epilogue, gradient-chunk loads) walks the
// same sequence.
//
// Plain order: the CTA's tiles (cta_tile) whole, accumulators alternating.
//
// Two streams (weight gradients with `wgrad_long_kb` set): a tile of a heavy
// expert runs a long K loop and finishes with one read-modify-write, while the
// many tiles of light experts are bound by their read-modify-writes.  One after
// the other on an SM, the first keep the tensor pipe busy with DRAM idle and the
// second the reverse.  Here the CTA's long tiles (K blocks > wgrad_long_kb: a
// prefix of its sequence, which is longest first) run on accumulator 0 in
// pieces of G blocks, with a whole short tile on accumulator 1 after each piece
// (and right after a long tile ends), G spreading the long blocks evenly over
// the short tiles: the short tiles' read-modify-writes overlap the long main
// loops.  When one stream runs out, the other continues with alternating
// accumulators (an open long tile first finishes on accumulator 0).  A tile
// starts on an accumulator only after the previous tile on it has ended in
// this order, and epilogues run in this order, so no wait can cycle.  The
// split changes only which K blocks run back to back, not any sum.
struct Seg {
  TileInfo ti;
  int tile;
  int k0, k1;   // K blocks [k0, k1) of the tile
  int acc;      // accumulator
  bool last;    // the tile's last segment
};

template <int BN, int NACC>
struct SegIter {
  int n;          // this CTA's tiles
  int nL;         // long tiles (rounds [0, nL)); 0: plain order
  int G;          // long-tile K blocks between two short tiles
  int iL, pL;     // next long tile, K blocks done of the open one
  int iS;         // next short tile (round)
  int since;      // long-tile K blocks since the last short tile
  int last_acc;   // accumulator of the most recent tile
  TileInfo curL;  // the open long tile
  int curL_tile;

  __device__ __forceinline__ void init(const GemmArgs& a, int num_tiles) {
    n = 0;
    while (cta_tile(a, n) < num_tiles) ++n;
    nL = 0;
    long long sumL = 0;
    if (NACC == 2 && a.wgrad && a.wgrad_long_kb > 0) {
      while (nL < n) {
        const int kb = decode_tile<BN>(a, cta_tile(a, nL)).kb;
        if (kb <= a.wgrad_long_kb) break;
        sumL += kb;
        ++nL;
      }
      if (nL == n) nL = 0;   // no short tiles: plain order
    }
    G = nL ? (int)((sumL + (n - nL) - 1) / (n - nL)) : 0;
    iL = 0;
    pL = 0;
    iS = nL;
    since = 0;
    last_acc = 1;
    if (nL) {
      curL_tile = cta_tile(a, 0);
      curL = decode_tile<BN>(a, curL_tile);
    }
  }

  __device__ __forceinline__ void open_next_long(const GemmArgs& a) {
    ++iL;
    pL = 0;
    if (iL < nL) {
      curL_tile = cta_tile(a, iL);
      curL = decode_tile<BN>(a, curL_tile);
    }
  }

  __device__ __forceinline__ void whole(const GemmArgs& a, int r, int acc, Seg& s) {
    s.tile = cta_tile(a, r);
    s.ti = decode_tile<BN>(a, s.tile);
    s.k0 = 0;
    s.k1 = s.ti.kb;
    s.acc = acc;
    s.last = true;
    last_acc = acc;
  }

  __device__ __forceinline__ bool next(const GemmArgs& a, Seg& s) {
    if (iL < nL && iS < n) {
      if (since >= G) {
        whole(a, iS++, 1, s);
        since = 0;
        return true;
      }
      const int m = min(G - since, curL.kb - pL);
      s.ti = curL;
      s.tile = curL_tile;
      s.k0 = pL;
      s.k1 = pL + m;
      s.acc = 0;
      s.last = s.k1 == curL.kb;
      last_acc = 0;
      pL += m;
      since += m;
      if (s.last) {
        open_next_long(a);
        since = G;   // a short tile next, while this one's epilogue runs
      }
      return true;
    }
    if (iL < nL) {
      if (pL > 0) {
        // the open long tile finishes on its accumulator
        s.ti = curL;
        s.tile = curL_tile;
        s.k0 = pL;
        s.k1 = curL.kb;
        s.acc = 0;
        s.last = true;
        last_acc = 0;
        open_next_long(a);
        return true;
      }
      whole(a, iL, NACC == 2 ? last_acc ^ 1 : 0, s);
      open_next_long(a);
      return true;
    }
    if (iS < n) {
      whole(a, iS++, NACC == 2 ? last_acc ^ 1 : 0, s);
      return true;
    }
    return false;
  }
};

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

// logistic sigmoid with the hardware exponential and reciprocal (CUDA's __expf
// and __fdividef intrinsics, a few ulp of fp32): far below the bf16 rounding
// the SwiGLU outputs go through.  Large negative G gives exp = inf and sig = 0.
// The forward (swiglu_fwd) and the backward's recomputation of h use this one
// function, so both see the same h.
__device__ __forceinline__ float sigmoid_fast(float G) {
  return __fdividef(1.0f, 1.0f + __expf(-G));
}

__device__ __forceinline__ float swiglu_fwd(float G, float U, float L) {
  if (L > 0.f) {
    G = fminf(fmaxf(G, -L), L);
    U = fminf(fmaxf(U, -L), L);
  }
  const float silu = G * sigmoid_fast(G);
  return silu * U;
}

// SwiGLU backward of one element.  g: the DGRAD-W2 accumulator (dh before the
// routing score s); G, U: the saved gate and up values (bf16, R1); L: clamp
// limit (0 = plain).  Returns h * g (the score-gradient term, h as the forward
// stored it, R2) and sets dgate, dup and hs = s * h, all before their bf16
// rounding (R4, R7).
__device__ __forceinline__ float swiglu_bwd(float g, float G, float U, float s, float L,
                                            float& dgate, float& dup, float& hs) {
  float mg = 1.f, mu = 1.f;
  if (L > 0.f) {
    if (G < -L || G > L) mg = 0.f;
    if (U < -L || U > L) mu = 0.f;
    G = fminf(fmaxf(G, -L), L);
    U = fminf(fmaxf(U, -L), L);
  }
  const float sig = sigmoid_fast(G);
  const float silu = G * sig;                   // as in swiglu_fwd
  const float hv = bf2f(f2bf(silu * U));        // h (R2)
  const float dh = s * g;
  const float dsilu = sig * (1.0f + G * (1.0f - sig));
  dgate = dh * U * dsilu * mg;
  dup = dh * silu * mu;
  hs = s * hv;
  return hv * g;
}

// ---------------------------------------------------------------------------
// epilogues: one thread owns one output row (`row` within the tile) and reads
// its accumulator columns from TMEM at `tbase` (lane quarter already folded in).

__device__ __forceinline__ void pack32(const float (&v)[32], uint32_t (&pk)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) pk[i] = pack_bf2(v[2 * i], v[2 * i + 1]);
}


// Staging of bf16 outputs: the epilogue threads write one 128-row x 64-column
// sub-tile (16 KB) into a shared-memory buffer in the 128-byte-swizzled layout of
// a 64 x 128 tensor-map box (each of the two warps of a lane quarter writes 32 of
// the 64 columns of its row), then one thread stores it with TMA.  Two buffers
// alternate; a buffer is rewritten only once its previous store has read it.
constexpr int kEpiStageBufs = 2;
// 16 KB staging buffers of the three-output epilogues (SwiGLU forward: h, a gate,
// a up; backward: dA gate, dA up, hs): two, which leaves room for four 48 KB
// operand stages.  Both main loops are bound by load latency, so the fourth
// stage is worth more than a buffer per output (SwiGLU backward 0.293 -> 0.284 ms
// on the E = 128 training shapes).
template <int EPI>
__host__ __device__ constexpr int tri_bufs() { return 2; }

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

// One packed bf16 sub-tile (this thread's 32 columns as 16 bf16 pairs) through
// the two alternating staging buffers of epi_stage_store: a buffer is rewritten
// once the store issued two sub-tiles earlier has read it, so a thread block
// never waits for the store it has just issued.
__device__ __forceinline__ void epi_stage_packed(const CUtensorMap* tm, uint32_t out0, int& seq,
                                                 int et, int row, int half,
                                                 const uint32_t (&pk)[16], int x, int y) {
  const uint32_t buf = out0 + (uint32_t)(seq % kEpiStageBufs) * 16384u;
  if (et == 0) bulk_wait_read<kEpiStageBufs - 1>();
  named_bar_sync(1, kEpiThreads);
  const uint32_t rbase = buf + (uint32_t)row * 128u;
  const uint32_t sw = (uint32_t)(row & 7);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    st_shared_v4_u32(rbase + (((uint32_t)(4 * half + q) ^ sw) << 4), pk[4 * q], pk[4 * q + 1],
                     pk[4 * q + 2], pk[4 * q + 3]);
  fence_proxy_async_smem();
  named_bar_sync(1, kEpiThreads);
  if (et == 0) {
    tma_store_2d(tm, buf, x, y);
    bulk_commit();
  }
  ++seq;
}

// Batched staging for epilogues with several outputs: NOUT sub-tiles of one
// 64-column chunk (this thread's 32 columns of each, already packed to bf16
// pairs) go to NOUT consecutive 16 KB buffers from `buf` and leave as NOUT TMA
// stores under one pair of barriers.  Buffers are reused only after the previous
// batch's stores have read them; the caller computes the next chunk before
// calling, so that wait overlaps the previous stores.
template <int NOUT>
__device__ __forceinline__ void epi_stage_batch(const CUtensorMap* const (&tms)[NOUT],
                                                uint32_t buf, int et, int row, int half,
                                                const uint32_t (&pk)[NOUT][16],
                                                const int (&xs)[NOUT], int y) {
  if (et == 0) bulk_wait_read<0>();
  named_bar_sync(1, kEpiThreads);
  const uint32_t sw = (uint32_t)(row & 7);
#pragma unroll
  for (int o = 0; o < NOUT; ++o) {
    const uint32_t rbase = buf + (uint32_t)o * 16384u + (uint32_t)row * 128u;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      st_shared_v4_u32(rbase + (((uint32_t)(4 * half + q) ^ sw) << 4), pk[o][4 * q],
                       pk[o][4 * q + 1], pk[o][4 * q + 2], pk[o][4 * q + 3]);
  }
  fence_proxy_async_smem();
  named_bar_sync(1, kEpiThreads);
  if (et == 0) {
#pragma unroll
    for (int o = 0; o < NOUT; ++o) tma_store_2d(tms[o], buf + (uint32_t)o * 16384u, xs[o], y);
    bulk_commit();
  }
}

// The three sub-tiles of a chunk (SwiGLU forward: h, a gate, a up; backward:
// dA gate, dA up, hs) leave as one batch through three buffers, else as a batch
// of the first two and then the third, through two.
template <int NBUF>
__device__ __forceinline__ void epi_stage_three(const CUtensorMap* t0, const CUtensorMap* t1,
                                                const CUtensorMap* t2, uint32_t buf, int et,
                                                int row, int half, const uint32_t (&pk)[3][16],
                                                int x0, int x1, int x2, int y) {
  if constexpr (NBUF >= 3) {
    const CUtensorMap* const tms[3] = {t0, t1, t2};
    const int xs[3] = {x0, x1, x2};
    epi_stage_batch<3>(tms, buf, et, row, half, pk, xs, y);
  } else {
    const CUtensorMap* const tms2[2] = {t0, t1};
    const int xs2[2] = {x0, x1};
    const uint32_t(&pk2)[2][16] = *reinterpret_cast<const uint32_t(*)[2][16]>(&pk[0]);
    epi_stage_batch<2>(tms2, buf, et, row, half, pk2, xs2, y);
    const CUtensorMap* const tms1[1] = {t2};
    const int xs1[1] = {x2};
    const uint32_t(&pk1)[1][16] = *reinterpret_cast<const uint32_t(*)[1][16]>(&pk[2]);
    epi_stage_batch<1>(tms1, buf, et, row, half, pk1, xs1, y);
  }
}

// Staging for the 256-wide MXFP8 epilogues: thread (row, half) owns 64
// consecutive output columns of its row (32 packed bf16 pairs), written in the
// 128-byte-swizzled layout of a 64 x 128 box and stored with TMA, half 0's at
// column x0 and half 1's at x1.  With two 16 KB buffers both halves write at
// once (buffer `half`); with one, half 0's sub-tile goes first.  A buffer is
// rewritten only once the previous store has read it.  MXFP8: one buffer; the
// 16 KB it frees give the operand ring a fourth stage, which is worth more (W13
// 0.272 -> 0.233 ms, W2 0.161 -> 0.137 ms on the E = 128 training shapes).
// NVFP4 (54 KB stages): three stages either way, so two buffers.
template <bool NV>
__host__ __device__ constexpr int wide_bufs() { return NV ? 2 : 1; }

template <int NBUF>
__device__ __forceinline__ void epi_stage_wide(const CUtensorMap* tm, uint32_t out0, int et,
                                               int row, int half, const uint32_t (&pk)[32],
                                               int x0, int x1, int y) {
  const uint32_t sw = (uint32_t)(row & 7);
#pragma unroll
  for (int r = 0; r < 3 - NBUF; ++r) {
    if (et == 0) bulk_wait_read<0>();
    named_bar_sync(1, kEpiThreads);
    if (NBUF == 2 || half == r) {
      const uint32_t rbase = out0 + (uint32_t)(NBUF == 2 ? half : 0) * 16384u +
                             (uint32_t)row * 128u;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        st_shared_v4_u32(rbase + (((uint32_t)q ^ sw) << 4), pk[4 * q], pk[4 * q + 1],
                         pk[4 * q + 2], pk[4 * q + 3]);
    }
    fence_proxy_async_smem();
    named_bar_sync(1, kEpiThreads);
    if (et == 0) {
      if (NBUF == 2) {
        tma_store_2d(tm, out0, x0, y);
        tma_store_2d(tm, out0 + 16384u, x1, y);
      } else {
        tma_store_2d(tm, out0, r == 0 ? x0 : x1, y);
      }
      bulk_commit();
    }
  }
}

// Epilogues of the 256-wide MXFP8 tiles, which have one accumulator: each thread
// reads its 128 accumulator columns [128*half, 128*half + 128) into registers and
// releases the accumulator (arrive on `release`, so the next tile's MMAs can
// start) before it computes and writes its outputs.
//   W13 + SwiGLU: the B tile's rows are two 64-row blocks, each the gate rows of
//     64 intermediate columns followed by the same up rows, so the thread holds
//     the gate (first 64) and up (last 64) values of the intermediate columns
//     c0 = 128*nt + 64*half ...: R1, SwiGLU, R2, then h is quantised along I in
//     32-column blocks (codes to a.hq, tiled E8M0 scales to a.hsf) as the A
//     operand of the block-scaled W2 GEMM; with a.save, a (gate and up, bf16)
//     leaves through shared-memory staging and TMA stores (tmO1).
//   W2 x score (R3) and the plain store (R5): output columns n0 + 128*half ...,
//     in two 64-column sub-tiles through staging (tmO0).
//   NVFP4 (NV): the accumulator is first multiplied by alpha = act_scale *
//     w_scale[e]; h is quantised to NVFP4 along I (16-element blocks, encode
//     scale h_enc: 32 code bytes and one word of four scale bytes per thread).
template <int EPI, bool NV = false>
__device__ __forceinline__ void epilogue_mx_wide(const GemmArgs& a, const TileInfo& ti, int row,
                                                 uint32_t tbase, int half,
                                                 const CUtensorMap* tmO0,
                                                 const CUtensorMap* tmO1, uint32_t out0, int et,
                                                 uint32_t release) {
  uint32_t v[8][16];
#pragma unroll
  for (int i = 0; i < 8; ++i) tmem_ld16(tbase + 128 * half + 16 * i, v[i]);
  tmem_ld_wait();
  tc_fence_before();
  mbar_arrive(release);
  const long long grow = (long long)ti.m0 + row;
  if constexpr (NV) {
    const float alpha = a.act_scale * a.w_scale[ti.e];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int q = 0; q < 16; ++q) v[i][q] = __float_as_uint(__uint_as_float(v[i][q]) * alpha);
  }
  if constexpr (NV && EPI == EPI_SWIGLU) {
    const int c0 = ti.nt * 128 + 64 * half;
    uint32_t sc = 0;
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      float hv[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int c = 32 * s + i;
        const float G = bf2f(f2bf(__uint_as_float(v[c >> 4][c & 15])));          // R1
        const float U = bf2f(f2bf(__uint_as_float(v[4 + (c >> 4)][c & 15])));
        hv[i] = bf2f(f2bf(swiglu_fwd(G, U, a.clamp)));                              // R2
      }
      uint32_t w[4];
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        float f[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) f[i] = hv[16 * b + i];
        uint32_t q[2];
        sc |= (uint32_t)nv_quant16(f, a.h_enc, q) << (16 * s + 8 * b);
        w[2 * b] = q[0];
        w[2 * b + 1] = q[1];
      }
      *reinterpret_cast<uint4*>(a.hq + grow * a.ld0 + (c0 + 32 * s) / 2) =
          make_uint4(w[0], w[1], w[2], w[3]);
    }
    *reinterpret_cast<uint32_t*>(a.hsf + mx_sf_offset(grow >> 7, (int)(grow & 127), c0 >> 4,
                                                      a.hsf_ngr)) = sc;
  } else if constexpr (EPI == EPI_SWIGLU) {
    const int c0 = ti.nt * 128 + 64 * half;
    // R1 first: gate and up to bf16 pairs (a's values), which frees the fp32 copies
    uint32_t pg[32], pu[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int c = 2 * i;
      pg[i] = pack_bf2(__uint_as_float(v[c >> 4][c & 15]), __uint_as_float(v[c >> 4][(c & 15) + 1]));
      pu[i] = pack_bf2(__uint_as_float(v[4 + (c >> 4)][c & 15]),
                       __uint_as_float(v[4 + (c >> 4)][(c & 15) + 1]));
    }
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      float hv[32];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t g2 = pg[16 * s + i], u2 = pu[16 * s + i];
        hv[2 * i] = bf2f(f2bf(swiglu_fwd(__uint_as_float(g2 << 16), __uint_as_float(u2 << 16),
                                         a.clamp)));                                // R2
        hv[2 * i + 1] = bf2f(f2bf(swiglu_fwd(__uint_as_float(g2 & 0xFFFF0000u),
                                             __uint_as_float(u2 & 0xFFFF0000u), a.clamp)));
      }
      uint32_t w[8];
      const uint8_t sc = mx_quant32(hv, w);
      uint8_t* hq = a.hq + grow * a.ld0 + c0 + 32 * s;
      reinterpret_cast<uint4*>(hq)[0] = make_uint4(w[0], w[1], w[2], w[3]);
      reinterpret_cast<uint4*>(hq)[1] = make_uint4(w[4], w[5], w[6], w[7]);
      a.hsf[mx_sf_offset(grow >> 7, (int)(grow & 127), (c0 + 32 * s) >> 5, a.hsf_ngr)] = sc;
    }
    if (a.save) {
      const int xg = ti.nt * 128;        // buffer 0: half 0's columns, buffer 1: half 1's
      epi_stage_wide<wide_bufs<NV>()>(tmO1, out0, et, row, half, pg, xg, xg + 64, ti.m0);
      epi_stage_wide<wide_bufs<NV>()>(tmO1, out0, et, row, half, pu, a.I + xg, a.I + xg + 64,
                                      ti.m0);
    }
  } else {
    static_assert(EPI == EPI_SCORE || EPI == EPI_STORE, "256-wide MXFP8 epilogues");
    const float s = EPI == EPI_SCORE && a.row_scale ? a.row_scale[grow] : 1.0f;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int c = 64 * j + 2 * i;
        pk[i] = pack_bf2(s * __uint_as_float(v[c >> 4][c & 15]),            // R3 / R5 on store
                         s * __uint_as_float(v[(c + 1) >> 4][(c + 1) & 15]));
      }
      const int x = ti.n0 + 64 * j;      // buffer 0: half 0's sub-tile, buffer 1: half 1's
      epi_stage_wide<wide_bufs<NV>()>(tmO0, out0, et, row, half, pk, x, x + 128, ti.m0);
    }
  }
}

// bf16-output epilogues.  The tile is walked in 64-column sub-tiles, the thread
// owning row `row` handling columns [32*half, 32*half+32) of each; outputs leave
// through shared-memory staging and TMA stores (tmO0 / tmO1: the output tensors'
// maps): one-output epilogues (W2 x score, plain store) through two alternating
// buffers, the three-output ones (SwiGLU: h and a; SwiGLU backward: dA and hs)
// as batches of three buffers per chunk.
template <int BN, int EPI>
__device__ __forceinline__ void epilogue(const GemmArgs& a, const TileInfo& ti, int row,
                                         uint32_t tbase, int half, const CUtensorMap* tmO0,
                                         const CUtensorMap* tmO1, uint32_t out0, int et,
                                         int& seq) {
  const long long grow = (long long)ti.m0 + row;
  uint32_t r0[16], r1[16];
  const int ch = 32 * half;
  if constexpr (EPI == EPI_SWIGLU) {
    // per 64-column chunk: h, and (training) the gate and up halves of a
    constexpr int BNH = BN / 2;          // gate columns [0,BNH), up columns [BNH,BN)
    const int c0 = ti.nt * BNH;          // first intermediate column of this tile
#pragma unroll 1
    for (int c = 0; c < BNH; c += 64) {
      float G[32], U[32], hv[32];
      tmem_ld16(tbase + c + ch, r0);
      tmem_ld16(tbase + c + ch + 16, r1);
      tmem_ld_wait();
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        G[q] = bf2f(f2bf(__uint_as_float(r0[q])));   // R1
        G[16 + q] = bf2f(f2bf(__uint_as_float(r1[q])));
      }
      tmem_ld16(tbase + BNH + c + ch, r0);
      tmem_ld16(tbase + BNH + c + ch + 16, r1);
      tmem_ld_wait();
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        U[q] = bf2f(f2bf(__uint_as_float(r0[q])));
        U[16 + q] = bf2f(f2bf(__uint_as_float(r1[q])));
      }
#pragma unroll
      for (int q = 0; q < 32; ++q) hv[q] = swiglu_fwd(G[q], U[q], a.clamp);   // R2 on store
      if (a.save) {
        uint32_t pk[3][16];
        pack32(hv, pk[0]);
        pack32(G, pk[1]);
        pack32(U, pk[2]);
        epi_stage_three<tri_bufs<EPI_SWIGLU>()>(tmO0, tmO1, tmO1, out0, et, row, half, pk, c0 + c, c0 + c,
                                  a.I + c0 + c, ti.m0);
      } else {
        epi_stage_store(tmO0, out0, seq, et, row, half, hv, c0 + c, ti.m0);
      }
    }
  } else if constexpr (EPI == EPI_SCORE || EPI == EPI_STORE) {
    const float s = EPI == EPI_SCORE && a.row_scale ? a.row_scale[grow] : 1.0f;
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
    // acc = g (columns = intermediate index i).  in1 = a [rows, 2I]; per 64-column
    // chunk: dA gate, dA up (tmO0 = dA [rows, 2I]) and hs (tmO1 = hs).  h is not
    // read back: it is recomputed from a with the forward's own arithmetic
    // (swiglu_fwd), which gives the bf16 value the forward stored (R2).
    const float s = a.row_scale[grow];
    const float L = a.clamp;
    const uint16_t* arow = static_cast<const uint16_t*>(a.in1) + grow * a.ldi1 + ti.n0;
    float part = 0.f;
    // the saved gate/up values of the next 16 columns are fetched one round ahead
    uint4 nx[4];
    auto fetch = [&](int cc) {
      const uint4* gp = reinterpret_cast<const uint4*>(arow + cc);
      const uint4* up = reinterpret_cast<const uint4*>(arow + a.I + cc);
      nx[0] = gp[0]; nx[1] = gp[1]; nx[2] = up[0]; nx[3] = up[1];
    };
    fetch(ch);
#pragma unroll 1
    for (int c = 0; c < BN; c += 64) {
      uint32_t pk[3][16];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {            // two 16-column halves of this thread's 32
        const int cc = c + ch + 16 * hh;
        const uint4 cur[4] = {nx[0], nx[1], nx[2], nx[3]};
        if (hh == 0) fetch(cc + 16);
        else if (c + 64 < BN) fetch(c + 64 + ch);
        tmem_ld16(tbase + cc, r0);
        float ag[16], au[16];
        {
          const uint32_t w[16] = {cur[0].x, cur[0].y, cur[0].z, cur[0].w, cur[1].x, cur[1].y,
                                  cur[1].z, cur[1].w, cur[2].x, cur[2].y, cur[2].z, cur[2].w,
                                  cur[3].x, cur[3].y, cur[3].z, cur[3].w};
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            ag[2 * i] = __uint_as_float(w[i] << 16);
            ag[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            au[2 * i] = __uint_as_float(w[8 + i] << 16);
            au[2 * i + 1] = __uint_as_float(w[8 + i] & 0xFFFF0000u);
          }
        }
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 16; q += 2) {
          float dg2[2], du2[2], hs2[2];
#pragma unroll
          for (int u = 0; u < 2; ++u)
            part += swiglu_bwd(__uint_as_float(r0[q + u]), ag[q + u], au[q + u], s, L, dg2[u],
                               du2[u], hs2[u]);
          pk[0][8 * hh + q / 2] = pack_bf2(dg2[0], dg2[1]);   // R4
          pk[1][8 * hh + q / 2] = pack_bf2(du2[0], du2[1]);
          pk[2][8 * hh + q / 2] = pack_bf2(hs2[0], hs2[1]);   // R7
        }
      }
      // dA gate, dA up, hs: one sub-tile at a time through the two buffers
      epi_stage_packed(tmO0, out0, seq, et, row, half, pk[0], ti.n0 + c, ti.m0);
      epi_stage_packed(tmO0, out0, seq, et, row, half, pk[1], a.I + ti.n0 + c, ti.m0);
      epi_stage_packed(tmO1, out0, seq, et, row, half, pk[2], ti.n0 + c, ti.m0);
    }
    // one partial per (n tile, column half)
    a.pdscore[grow * (2 * a.n_tiles) + 2 * ti.nt + half] = part;
  }
}

// DGRAD-W2 epilogue of the MXFP8 backward.  The SwiGLU backward as in
// `epilogue`, but dA and hs leave only as E4M3 codes with E8M0 scales (their
// bf16 values, R4 and R7, quantised; nothing reads bf16 copies):
//  - dA along 2I: each thread quantises the 32-column blocks of its row;
//  - dA and hs along the rows, transposed: a warp's 32 rows are one block.  The
//    warp stages each 32 x 32 block of bf16 values in its own 4 KB of shared
//    memory, each lane quantises one column of it, and the codes (32 bytes per
//    column) go back through the same staging, so that the stores are
//    coalesced.
// Thread (row, half) takes columns [64c + 32*half, +32) of each 64-column chunk.
constexpr int kD2ValLd = 80;    // staged bf16 row (64 bytes + 16: conflict-free 16-byte stores)
constexpr int kD2CodeLd = 48;   // staged code row (32 bytes + 16)
constexpr int kD2WarpBytes = 32 * kD2ValLd + 32 * kD2CodeLd;
static_assert(kD2WarpBytes == 4096, "4 KB of staging per epilogue warp");

template <int BN>
__device__ __forceinline__ void epilogue_dgrad2_mx(const GemmArgs& a, const TileInfo& ti, int row,
                                                   uint32_t tbase, int half, uint8_t* stg, int et) {
  const int lane = row & 31;
  const long long grow = (long long)ti.m0 + row;
  const long long r32 = (long long)ti.m0 + (row & ~31);     // the warp's first row
  uint8_t* vals = stg + (et >> 5) * kD2WarpBytes;              // [32 rows][kD2ValLd]
  uint8_t* codes = vals + 32 * kD2ValLd;                       // [32 columns][kD2CodeLd]
  const float s = a.row_scale[grow];
  const float L = a.clamp;
  const uint16_t* arow = static_cast<const uint16_t*>(a.in1) + grow * a.ldi1 + ti.n0;
  float part = 0.f;
#pragma unroll 1
  for (int c = 0; c < BN; c += 64) {
    const int cc0 = c + 32 * half;                             // this thread's 32 columns
    uint32_t pw[3][16];                                        // bf16 pairs: dA gate, dA up, hs
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int cc = cc0 + 16 * hh;
      uint32_t r0[16];
      tmem_ld16(tbase + cc, r0);
      const uint4* gp = reinterpret_cast<const uint4*>(arow + cc);
      const uint4* up = reinterpret_cast<const uint4*>(arow + a.I + cc);
      const uint4 g0 = gp[0], g1 = gp[1], u0 = up[0], u1 = up[1];
      const uint32_t wg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
      const uint32_t wu[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float dg2[2], du2[2], hs2[2];
        part += swiglu_bwd(__uint_as_float(r0[2 * i]), __uint_as_float(wg[i] << 16),
                           __uint_as_float(wu[i] << 16), s, L, dg2[0], du2[0], hs2[0]);
        part += swiglu_bwd(__uint_as_float(r0[2 * i + 1]), __uint_as_float(wg[i] & 0xFFFF0000u),
                           __uint_as_float(wu[i] & 0xFFFF0000u), s, L, dg2[1], du2[1], hs2[1]);
        pw[0][8 * hh + i] = pack_bf2(dg2[0], dg2[1]);   // R4
        pw[1][8 * hh + i] = pack_bf2(du2[0], du2[1]);
        pw[2][8 * hh + i] = pack_bf2(hs2[0], hs2[1]);   // R7
      }
    }
    // dA along 2I: this row's 32-column block of the gate half and of the up half
#pragma unroll
    for (int o = 0; o < 2; ++o) {
      float f[32];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        f[2 * i] = __uint_as_float(pw[o][i] << 16);
        f[2 * i + 1] = __uint_as_float(pw[o][i] & 0xFFFF0000u);
      }
      uint32_t w[8];
      const uint8_t sc = mx_quant32(f, w);
      const int col = (o ? a.I : 0) + ti.n0 + cc0;
      uint4* dst = reinterpret_cast<uint4*>(a.q_row + grow * (2LL * a.I) + col);
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      a.sf_row[mx_sf_offset(grow >> 7, (int)(grow & 127), col >> 5, a.sf_row_ngr)] = sc;
    }
    // dA gate, dA up and hs along the rows: the warp's 32 x 32 blocks
#pragma unroll
    for (int o = 0; o < 3; ++o) {
      uint4* vr = reinterpret_cast<uint4*>(vals + lane * kD2ValLd);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        vr[j] = make_uint4(pw[o][4 * j], pw[o][4 * j + 1], pw[o][4 * j + 2], pw[o][4 * j + 3]);
      __syncwarp();
      float f[32];
#pragma unroll
      for (int i = 0; i < 32; ++i)
        f[i] = __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(vals + i * kD2ValLd)[lane]
                               << 16);
      uint32_t w[8];
      const uint8_t sc = mx_quant32(f, w);
      __syncwarp();                     // every lane has read the block
      uint4* cr = reinterpret_cast<uint4*>(codes + lane * kD2CodeLd);
      cr[0] = make_uint4(w[0], w[1], w[2], w[3]);
      cr[1] = make_uint4(w[4], w[5], w[6], w[7]);
      __syncwarp();
      const long long colbase = (o == 1 ? a.I : 0) + ti.n0 + cc0;
      uint8_t* qt = o < 2 ? a.qt_a : a.qt_h;
      uint8_t* sft = o < 2 ? a.sft_a : a.sft_h;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int p = lane + 32 * t, col = p >> 1, hf = p & 1;
        *reinterpret_cast<uint4*>(qt + (colbase + col) * a.qt_ld + r32 + 16 * hf) =
            *reinterpret_cast<const uint4*>(codes + col * kD2CodeLd + 16 * hf);
      }
      const long long cl = colbase + lane;
      sft[mx_sf_offset(cl >> 7, (int)(cl & 127), (int)(r32 >> 5), (int)(a.qt_ld / 128))] = sc;
      __syncwarp();                     // the staging is rewritten next round
    }
  }
  // one partial per (n tile, column half)
  a.pdscore[grow * (2 * a.n_tiles) + 2 * ti.nt + half] = part;
}

// WGRAD epilogue: read-modify-write of the fp32 gradient, 32 columns (16 KB:
// 128 rows x 32 fp32, 128-byte swizzle, the layout of the fp32 tensor map) at a
// time.  Each such chunk is loaded by TMA into one of NB shared-memory
// buffers ahead of use (NB - 1 chunks ahead, across tile boundaries),
// every thread adds its row's accumulator values to it in place, and TMA stores
// it back.  (A TMA reduce-add in L2 does the same sum but moves fp32 data
// measurably slower than a load and a store.)  The chunk sequence is this CTA's
// tiles (cta_tile) times BN/32 chunks each; each output tile is visited once per
// launch, so no load can see a pending store.
// fp32 chunk buffers of 16 KB: 4 (three loads ahead) for the 256-wide bf16
// tiles, 5 for the 128-wide block-scaled ones (measured best for each)
template <bool MX>
__host__ __device__ constexpr int wgrad_bufs() { return MX ? 5 : 4; }

template <int BN, int NACC>
struct WgradPipe {
  uint32_t buf0;     // first chunk buffer
  uint32_t bar0;     // first of the NB chunk-load barriers
  int next;          // chunks consumed (all epilogue threads)
  int issued;        // chunks whose load has been issued (thread et == 0)
  // thread et == 0: the tiles in epilogue order, for the loads ahead
  SegIter<BN, NACC> order;
  int have;          // tiles taken from `order`
  TileInfo cur;      // the last of them
  // every epilogue thread; `issuer`: the thread that issues the loads
  __device__ __forceinline__ void init(const GemmArgs& a, int num_tiles, uint32_t b0,
                                       uint32_t bar, bool issuer) {
    buf0 = b0;
    bar0 = bar;
    next = 0;
    issued = 0;
    have = 0;
    if (issuer) order.init(a, num_tiles);
  }
};

template <int BN, int NACC, int NB>
__device__ __forceinline__ void wgrad_issue(const GemmArgs& a, const CUtensorMap* tmC,
                                            WgradPipe<BN, NACC>& p, int upto) {
  constexpr int CH = BN / 32;
  while (p.issued < upto) {
    const int n = p.issued;
    while (p.have <= n / CH) {   // the epilogue's next tile
      Seg sg;
      bool got = false;
      while (p.order.next(a, sg))
        if (sg.last) {
          got = true;
          break;
        }
      if (!got) return;
      p.cur = sg.ti;
      ++p.have;
    }
    const TileInfo& t = p.cur;
    const int b = n % NB;
    const uint32_t bar = p.bar0 + 8u * (uint32_t)b;
    mbar_arrive_expect_tx(bar, 16384u);
    tma_load_2d(p.buf0 + (uint32_t)b * 16384u, tmC, t.n0 + (n % CH) * 32,
                t.e * a.m_tiles * kBM + t.m0, bar);
    ++p.issued;
  }
}

// Returns false when a wait gave up (every epilogue thread returns the same).
template <int BN, int NACC, int NB>
__device__ __forceinline__ bool epilogue_wgrad(const GemmArgs& a, const CUtensorMap* tmC,
                                               const TileInfo& ti, int row, uint32_t tbase, int et,
                                               int half, WgradPipe<BN, NACC>& p,
                                               volatile int* abort_flag, uint64_t wlim) {
  const int ybase = ti.e * a.m_tiles * kBM + ti.m0;
  const uint32_t sw = (uint32_t)(row & 7);
  uint32_t r0[16];
#pragma unroll 1
  for (int c = 0; c < BN; c += 32) {
    const int n = p.next;
    const int b = n % NB;
    const uint32_t buf = p.buf0 + (uint32_t)b * 16384u;
    // this thread's half: 16 of the chunk's 32 columns (16-byte chunks 4h..4h+3)
    tmem_ld16(tbase + c + 16 * half, r0);
    const int w = mbar_wait(p.bar0 + 8u * (uint32_t)b, (uint32_t)((n / NB) & 1),
                            abort_flag, a.err, 6, wlim)
                      ? 1 : 0;
    tmem_ld_wait();
    if (w) {
      const uint32_t rbase = buf + (uint32_t)row * 128u;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t addr = rbase + (((uint32_t)(q + 4 * half) ^ sw) << 4);
        float v0, v1, v2, v3;
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(v0), "=f"(v1), "=f"(v2), "=f"(v3) : "r"(addr));
        st_shared_v4(addr, v0 + __uint_as_float(r0[4 * q]), v1 + __uint_as_float(r0[4 * q + 1]),
                     v2 + __uint_as_float(r0[4 * q + 2]), v3 + __uint_as_float(r0[4 * q + 3]));
      }
    }
    fence_proxy_async_smem();
    if (epi_bar_and(w) == 0) return false;
    p.next = n + 1;
    if (et == 0) {
      tma_store_2d(tmC, buf, ti.n0 + c, ybase);
      bulk_commit();
      // chunk n-1's buffer is free once its store has read it: load chunk
      // n + NB - 1 there
      bulk_wait_read<1>();
      wgrad_issue<BN, NACC, NB>(a, tmC, p, n + NB);
    }
  }
  return true;
}

}  // namespace gemm
}  // namespace moe
