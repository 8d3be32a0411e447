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
//   warp 10     NVFP4 only: copies each stage's scale factors into TMEM
//               (tcgen05.cp), so the MMA issuer only issues MMAs
// The accumulator is double buffered in TMEM (2 x BN fp32 columns) so the
// epilogue of tile i overlaps the main loop of tile i+1.  Every role walks the
// same sequence of K-stage segments (gemm::SegIter): whole tiles with the two
// accumulators alternating, or, for weight gradients of heavy experts, long
// tiles in pieces interleaved with short ones.
//
// Every mbarrier wait is bounded (moe::mbar_wait); a wait that gives up records
// MOE_ERR_TIMEOUT, all roles leave their loops, outstanding copies and MMAs are
// drained with bounded waits, and TMEM is freed before the CTA exits.

#include "moe_gemm_common.cuh"

namespace moe {

using namespace gemm;

namespace {

template <int BN, int EPI, bool MX, bool NV = false>
struct GemmShape {
  // A stage holds 128 rows (A) and BN rows (B) of 128 bytes of K: 64 bf16, 128
  // E4M3 or 256 E2M1 elements; MXFP8 stages also carry the 512-byte scale chunks
  // of A (one) and of B (one per 128 rows) for those 128 K-elements, NVFP4 stages
  // four chunks per 128 rows (one per 64-element K group), padded to keep stages
  // 1024-aligned.
  static_assert(!NV || MX, "NVFP4 is a block-scaled format");
  static constexpr int A_BYTES = kBM * 128;                    // 16 KB
  static constexpr int B_BYTES = BN * 128;
  static constexpr int SF_LOAD_BYTES = MX ? (NV ? 2048 : 512) * (1 + BN / 128) : 0;
  static constexpr int SF_STAGE_BYTES = (SF_LOAD_BYTES + 1023) / 1024 * 1024;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SF_STAGE_BYTES;
  static constexpr int TX_BYTES = A_BYTES + B_BYTES + SF_LOAD_BYTES;   // bytes a stage receives
  // Output staging: WGRAD's fp32 buffers (it needs few stages: its K loop is one
  // expert's rows and it is bound by the gradient traffic), else bf16 sub-tile
  // buffers for the TMA-store epilogues (the MXFP8 DGRAD-W2 epilogue uses the
  // same 32 KB as 4 KB of staging per epilogue warp).
  // (the NVFP4 W13 epilogue writes h from registers and never saves a: no staging)
  static constexpr int OUT_BYTES =
      (NV && EPI == EPI_SWIGLU ? 0 : EPI == EPI_WGRAD ? wgrad_bufs<MX>()
                        : (MX && BN == 256 ? wide_bufs<NV>()
                                           : (EPI == EPI_SCORE || EPI == EPI_STORE
                                                  ? kEpiStageBufs
                                                  : tri_bufs<EPI>()))) * 16384;
  static constexpr int STAGE_BUDGET = 226 * 1024 - OUT_BYTES;
  // at most 8 stages; block-scaled kernels at most 4: a fifth made the SwiGLU
  // backward slower (its epilogue's row loads gain from the L1 a smaller ring
  // leaves), and the 256-wide ones fit no more than four
  static constexpr int MAX_STAGES = MX ? 4 : 8;
  static constexpr int STAGES =
      STAGE_BUDGET / STAGE_BYTES > MAX_STAGES ? MAX_STAGES : STAGE_BUDGET / STAGE_BYTES;
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + OUT_BYTES + BAR_BYTES + 1024;
  // TMEM: the accumulators, then (MXFP8) SF_COLS scale columns per stage, A's
  // at +0 and B's at +SF_COLS/2 (four per 128 rows).  Two BN-column accumulators
  // alternate, except for 256-wide MXFP8 tiles, whose scale columns leave room
  // for one: their epilogue releases it as soon as it has read it.
  static constexpr int NACC = (MX && BN == 256) ? 1 : 2;
  static constexpr uint32_t SF_COL0 = NACC * BN;
  // per stage: MXFP8 A 4 + B 4 per 128 rows; NVFP4 four times that (one set per
  // 64-element K group), B's at +16, rounded up to 64 columns
  static constexpr uint32_t SF_COLS = MX ? (NV ? 64 : (BN == 256 ? 16 : 8)) : 0;
  static constexpr uint32_t TMEM_COLS = MX ? 512 : 2 * BN;
  static_assert(!MX || SF_COL0 + SF_COLS * STAGES <= 512, "TMEM budget");
  static_assert(STAGES >= 3, "operand ring");
};

// NVFP4 kernels add a warp that copies the scale factors into tensor memory: a
// stage's twelve copies cost as much tensor-core issue time as its MMAs when the
// MMA thread issues them itself (a diagnostic build without them ran W13 36 %
// faster).
template <bool NV>
constexpr int gemm_threads() { return NV ? kThreads + 32 : kThreads; }

template <int BN, bool A_MN, bool B_MN, int EPI, bool MX, bool NV = false>
__global__ void __launch_bounds__(gemm_threads<NV>(), 1)
    k_grouped_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmO0,
                   const __grid_constant__ CUtensorMap tmO1, const GemmArgs args) {
  using S = GemmShape<BN, EPI, MX, NV>;
  constexpr int STAGES = S::STAGES;
  constexpr uint32_t IDESC =
      NV ? idesc_nvf4(kBM, BN) : (MX ? idesc_mxf8(kBM, BN) : idesc_bf16(kBM, BN, A_MN, B_MN));
  static_assert(!NV || (BN == 256 && (EPI == EPI_SWIGLU || EPI == EPI_SCORE)),
                "NVFP4: 256-wide row GEMMs (W13 + SwiGLU, W2 x score)");
  constexpr int KE = MX ? 128 : kBK;     // K elements per stage (128 bytes per row)
  constexpr int WB = wgrad_bufs<MX>();   // WGRAD: fp32 gradient chunk buffers
  static_assert(!MX || (!A_MN && !B_MN && (BN == 128 || BN == 256)),
                "MXFP8: K-major operands, BN = 128 or 256");
  static_assert(S::SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN");
  pdl_wait();   // the previous kernel of the stream has completed

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t tmem_holder;
  __shared__ int num_tiles_s;
  __shared__ volatile int abort_s;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * S::STAGE_BYTES + S::OUT_BYTES);
  // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], drain, then WGRAD chunk
  // loads, or (NVFP4) sf_full[STAGES] (a stage's scales are in TMEM) and sf_drain
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
  const uint32_t wg_bar0 = bar0 + 8u * (2 * STAGES + 5);
  auto sf_full_bar = [&](int s) { return wg_bar0 + 8u * s; };
  const uint32_t sf_drain_bar = wg_bar0 + 8u * STAGES;
  static_assert(8 * (3 * STAGES + 6) <= S::BAR_BYTES, "barrier space");

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
    if (EPI == EPI_WGRAD)
      for (int b = 0; b < WB; ++b) mbar_init(wg_bar0 + 8u * b, 1);
    if (NV) {
      for (int s = 0; s < STAGES; ++s) mbar_init(sf_full_bar(s), 1);
      mbar_init(sf_drain_bar, 1);
    }
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
    if (EPI != EPI_WGRAD) {
      tma_prefetch_desc(&tmO0);
      tma_prefetch_desc(&tmO1);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_holder;
  const uint32_t stage0 = smem_u32(smem);


  if (warp == 0) {
    // ---------------- TMA producer ----------------
    // (lane 0 alone, like the MMA issuer: no warp-wide step per stage)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued_parity[STAGES];
#pragma unroll
      for (int s = 0; s < STAGES; ++s) issued_parity[s] = -1;
      bool ok = true;
      SegIter<BN, S::NACC> seq;
      seq.init(args, num_tiles);
      Seg sg;
      while (ok && seq.next(args, sg)) {
        const TileInfo& ti = sg.ti;
        // k_rotate (row GEMMs): the tiles that share an A tile (same m tile) or a
        // B tile (same expert and n tile) run at the same time; each starts its K
        // loop at its own offset (wrapping around), so each K chunk is read from
        // DRAM by one of them and from L2 by the others, instead of all of them
        // waiting on DRAM for the same chunk.
        const int kb0 = args.k_rotate ? (int)(((unsigned)(ti.m0 >> 7) * 7u + (unsigned)ti.nt * 5u) %
                                              (unsigned)ti.kb)
                                      : 0;
        for (int kb = sg.k0; kb < sg.k1; ++kb) {
          const int kc = kb + kb0 < ti.kb ? kb + kb0 : kb + kb0 - ti.kb;   // K chunk loaded
          ok = mbar_wait(empty_bar(stage), phase ^ 1u, &abort_s, args.err, 1, wlim);
          if (!ok) break;
          {
            const uint32_t fb = full_bar(stage);
            const uint32_t sa = stage0 + stage * S::STAGE_BYTES;
            const uint32_t sb = sa + S::A_BYTES;
            mbar_arrive_expect_tx(fb, S::TX_BYTES);
            if constexpr (NV) {
              // the four 512-byte scale chunks of this stage's 64-element K groups
              // (contiguous in the tiled layout): A's row block, then B's BN/128 row
              // blocks, 2 KB each (row GEMMs only)
              const uint32_t ssf = sb + S::B_BYTES;
              const long long kg = 4LL * kc;
              const long long gbr =
                  (long long)ti.e * args.b_blocks_per_expert + (long long)ti.nt * (BN / 128);
              bulk_g2s(ssf, args.sfa + ((long long)(ti.m0 >> 7) * args.sf_ngr + kg) * 512, 2048u, fb);
#pragma unroll
              for (int rb = 0; rb < BN / 128; ++rb)
                bulk_g2s(ssf + 2048u * (uint32_t)(1 + rb),
                         args.sfb + ((gbr + rb) * args.sf_ngr + kg) * 512, 2048u, fb);
            } else if constexpr (MX) {
              // the 512-byte scale chunks of this K group: A's row block, then B's
              // BN/128 row blocks
              const uint32_t ssf = sb + S::B_BYTES;
              // row GEMMs: K groups from 0, B row blocks of (expert, n tile); wgrad
              // mode: K groups from the expert's first row, B row blocks from n0/128
              const long long kg = (long long)(ti.krow0 >> 7) + kc;
              const long long ga = ((long long)(ti.m0 >> 7) * args.sf_ngr + kg) * 512;
              const long long gbr =
                  args.wgrad ? (long long)(ti.n0 >> 7)
                             : (long long)ti.e * args.b_blocks_per_expert + (long long)ti.nt * (BN / 128);
              bulk_g2s(ssf, args.sfa + ga, 512u, fb);
#pragma unroll
              for (int rb = 0; rb < BN / 128; ++rb)
                bulk_g2s(ssf + 512u * (uint32_t)(1 + rb),
                         args.sfb + ((gbr + rb) * args.sf_ngr + kg) * 512, 512u, fb);
            }
            // One TMA per operand tile (large boxes: the TMA cost is per box).
            // A: 128 rows x 128 bytes of K.  K-major: a 128-row box of [rows, K];
            // MN-major: two 64-wide atoms of the [K rows, M] tensor (3-D map).
            if (A_MN)
              tma_load_3d(sa, &tmA, 0, ti.krow0 + kc * kBK, ti.m0 >> 6, fb);
            else
              tma_load_2d(sa, &tmA, ti.krow0 + kc * KE, ti.m0, fb);
            // B: BN rows (N) x 128 bytes of K
            if (args.wgrad && B_MN) {
              tma_load_3d(sb, &tmB, 0, ti.krow0 + kc * kBK, ti.n0 >> 6, fb);
            } else if (args.wgrad) {
              // K-major transposed operand [N, rows]: this expert's K range
              tma_load_2d(sb, &tmB, ti.krow0 + kc * KE, ti.n0, fb);
            } else if (B_MN) {
              // [E*K, N]: BN/64 atoms of expert e's K rows
              tma_load_3d(sb, &tmB, 0, ti.e * args.b_expert_rows + kc * kBK, ti.n0 >> 6, fb);
            } else if (EPI == EPI_SWIGLU && MX && BN == 256) {
              // (K, 64, 2, I/64, E) view of W13: two 64-row blocks, each its gate
              // rows then the same up rows (the row order of the scale chunks)
              tma_load_5d(sb, &tmB, kc * KE, 0, 0, 2 * ti.nt, ti.e, fb);
            } else if (EPI == EPI_SWIGLU) {
              // (K, I, 2E) view of W13: this tile's BN/2 gate rows, then the same up
              // rows, in one box
              tma_load_3d(sb, &tmB, kc * KE, ti.nt * (BN / 2), 2 * ti.e, fb);
            } else {
              // [E*N, K]: a BN-row box
              tma_load_2d(sb, &tmB, kc * KE, ti.e * args.b_expert_rows + ti.n0, fb);
            }
            issued_parity[stage] = (int)phase;
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
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
    // Lane 0 runs the whole loop alone: a stage costs a barrier test and the
    // MMAs, whose shared-memory descriptors are a fixed base plus the stage and
    // K-step offsets (the address field counts 16-byte units, and no operand
    // address leaves its 14 bits), so the tensor pipe is not left idle between
    // stages while the next ones are prepared.
    if (lane == 0) {
      // K-major: rows of 128 B, 8-row groups 1024 B apart; K step = 32 B.
      // MN-major: 64-wide MN atoms 8 KB apart (LBO), 8-row K groups 1024 B apart
      // (SBO); K step of 16 rows = 2048 B.
      const uint64_t a_desc0 = A_MN ? smem_desc_sw128(stage0, 8192, 1024)
                                    : smem_desc_sw128(stage0, 16, 1024);
      const uint64_t b_desc0 = B_MN ? smem_desc_sw128(stage0 + S::A_BYTES, 8192, 1024)
                                    : smem_desc_sw128(stage0 + S::A_BYTES, 16, 1024);
      // (block-scaled: K-major, 32 bytes of K per MMA step as well)
      constexpr uint32_t A_KSTEP = (A_MN ? 2048u : 32u) >> 4;
      constexpr uint32_t B_KSTEP = (B_MN ? 2048u : 32u) >> 4;
      // MXFP8 scale chunks of a stage: A's 512 bytes after B, then B's per 128 rows
      const uint64_t sf_desc0 = smem_desc_noswz(stage0 + S::A_BYTES + S::B_BYTES, 512u, 128u);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_phase = 0u;   // bit a: uses of accumulator a so far, mod 2
      bool ok = true;
      SegIter<BN, S::NACC> seq;
      seq.init(args, num_tiles);
      Seg sg;
      while (ok && seq.next(args, sg)) {
        const int acc = sg.acc;
        if (sg.k0 == 0) {
          // a tile starts: its accumulator's previous tile has been read out
          ok = mbar_wait(tempty_bar(acc), ((acc_phase >> acc) & 1u) ^ 1u, &abort_s, args.err, 3,
                         wlim);
          // failure-path test: wait on the drain barrier, which nothing has arrived at
          if (args.stall_mma && ok) ok = mbar_wait(drain_bar, 0, &abort_s, args.err, 9, wlim);
          if (!ok) break;
          tc_fence_after();
        }
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = sg.k0; kb < sg.k1; ++kb) {
          ok = mbar_wait(full_bar(stage), phase, &abort_s, args.err, 4, wlim);
          // NVFP4: also wait until the scale warp's copies of this stage are in TMEM
          if (NV && ok) ok = mbar_wait(sf_full_bar(stage), phase, &abort_s, args.err, 10, wlim);
          if (!ok) break;
          tc_fence_after();
          const uint64_t soff = (uint64_t)((uint32_t)(stage * S::STAGE_BYTES) >> 4);
          if constexpr (NV) {
            // four K = 64 steps, step j reading the scale columns of 64-element K
            // group j: A's four at sfa_t + 4j, B's (four per 128 rows) at sfb_t + (BN/32)j
            const uint32_t sfa_t = tmem_base + S::SF_COL0 + S::SF_COLS * (uint32_t)stage;
            const uint32_t sfb_t = sfa_t + 16u;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              umma_nvf4(d_tmem, a_desc0 + soff + (uint64_t)(j * A_KSTEP),
                        b_desc0 + soff + (uint64_t)(j * B_KSTEP), IDESC, sfa_t + 4u * (uint32_t)j,
                        sfb_t + (uint32_t)(BN / 32) * (uint32_t)j, (kb | j) != 0 ? 1u : 0u);
          } else if constexpr (MX) {
            // this stage's scales -> its own TMEM columns (reused only after the
            // stage is released, i.e. after these MMAs have completed); then four
            // 32-element K steps, step j reading scale byte j
            const uint32_t sfa_t = tmem_base + S::SF_COL0 + S::SF_COLS * (uint32_t)stage;
            const uint32_t sfb_t = sfa_t + S::SF_COLS / 2;
            tmem_cp_32x128b_x4(sfa_t, sf_desc0 + soff);
#pragma unroll
            for (int rb = 0; rb < BN / 128; ++rb)
              tmem_cp_32x128b_x4(sfb_t + 4u * (uint32_t)rb,
                                 sf_desc0 + soff + (uint64_t)(32u * (uint32_t)(1 + rb)));
#pragma unroll
            for (int j = 0; j < 4; ++j)
              umma_mxf8(d_tmem, a_desc0 + soff + (uint64_t)(j * A_KSTEP),
                        b_desc0 + soff + (uint64_t)(j * B_KSTEP),
                        idesc_sf_ids(IDESC, (uint32_t)j, (uint32_t)j), sfa_t, sfb_t,
                        (kb | j) != 0 ? 1u : 0u);
          } else {
#pragma unroll
            for (int k16 = 0; k16 < kBK / 16; ++k16)
              umma_f16(d_tmem, a_desc0 + soff + (uint64_t)(k16 * A_KSTEP),
                       b_desc0 + soff + (uint64_t)(k16 * B_KSTEP), IDESC,
                       (kb | k16) != 0 ? 1u : 0u);
          }
          umma_commit(empty_bar(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (sg.last) {
          umma_commit(tfull_bar(acc));
          acc_phase ^= 1u << acc;
        }
      }
      if (abort_s) {
        // drain: wait for every MMA issued so far before TMEM is freed
        umma_commit(drain_bar);
        mbar_wait_drain(drain_bar, 0);
      }
    }
    __syncwarp();
  } else if (NV && warp == kThreads / 32) {
    // ---------------- scale-factor copies (NVFP4) ----------------
    // For each stage the MMA issuer consumes: wait for its bytes, copy the scales
    // of its four 64-element K groups into the stage's own TMEM columns (reused
    // only after the stage was released, i.e. after the MMAs that read them have
    // completed), and signal sf_full when the copies are done.  Lane 0 alone.
    if (lane == 0) {
      const uint64_t sf_desc0 = smem_desc_noswz(stage0 + S::A_BYTES + S::B_BYTES, 512u, 128u);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      SegIter<BN, S::NACC> seq;
      seq.init(args, num_tiles);
      Seg sg;
      while (ok && seq.next(args, sg)) {
        for (int kb = sg.k0; kb < sg.k1; ++kb) {
          ok = mbar_wait(full_bar(stage), phase, &abort_s, args.err, 11, wlim);
          if (!ok) break;
          tc_fence_after();
          // chunk j of A at +512 j bytes; of B's row block rb at +2048 (1 + rb) + 512 j
          const uint64_t sdesc = sf_desc0 + (uint64_t)((uint32_t)(stage * S::STAGE_BYTES) >> 4);
          const uint32_t sfa_t = tmem_base + S::SF_COL0 + S::SF_COLS * (uint32_t)stage;
          const uint32_t sfb_t = sfa_t + 16u;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            tmem_cp_32x128b_x4(sfa_t + 4u * (uint32_t)j, sdesc + (uint64_t)(32u * (uint32_t)j));
#pragma unroll
            for (int rb = 0; rb < BN / 128; ++rb)
              tmem_cp_32x128b_x4(sfb_t + (uint32_t)(BN / 32) * (uint32_t)j + 4u * (uint32_t)rb,
                                 sdesc + (uint64_t)(128u * (uint32_t)(1 + rb) + 32u * (uint32_t)j));
          }
          umma_commit(sf_full_bar(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (abort_s) {
        // drain: every copy issued so far lands before TMEM is freed
        umma_commit(sf_drain_bar);
        mbar_wait_drain(sf_drain_bar, 0);
      }
    }
    __syncwarp();
  } else if (warp < kThreads / 32) {
    // ---------------- epilogue (warps 2..5) ----------------
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int et = threadIdx.x - 64;          // 0..255 over the epilogue warps
    const int half = (warp - 2) >> 2;         // warps 2..5: columns' first half, 6..9: second
    uint32_t acc_phase = 0u;                  // bit a: uses of accumulator a so far, mod 2
    int sub = 0;                              // output staging-buffer sequence number
    WgradPipe<BN, S::NACC> wp;
    if (EPI == EPI_WGRAD) {
      wp.init(args, num_tiles, stage0 + STAGES * S::STAGE_BYTES, wg_bar0, et == 0);
      if (et == 0) wgrad_issue<BN, S::NACC, WB>(args, &tmC, wp, WB - 1);
    }
    // tiles in the order their last segments reach the MMA issuer
    SegIter<BN, S::NACC> seq;
    seq.init(args, num_tiles);
    Seg sg;
    while (seq.next(args, sg)) {
      if (!sg.last) continue;
      const TileInfo& ti = sg.ti;
      const int acc = sg.acc;
      int w = 1;
      if (lane == 0) w = mbar_wait(tfull_bar(acc), (acc_phase >> acc) & 1u, &abort_s, args.err, 5, wlim);
      // all eight epilogue warps leave together, so their named barriers stay matched
      const int ok_warp = __shfl_sync(0xffffffffu, w, 0);
      if (epi_bar_and(ok_warp) == 0) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
      if constexpr (S::NACC == 1) {
        // one accumulator: read it, release it, then compute the outputs
        epilogue_mx_wide<EPI, NV>(args, ti, row, tbase, half, &tmO0, &tmO1,
                                  stage0 + STAGES * S::STAGE_BYTES, et, tempty_bar(0));
        acc_phase ^= 1u;
        continue;
      } else if constexpr (EPI == EPI_WGRAD) {
        if (!epilogue_wgrad<BN, S::NACC, WB>(args, &tmC, ti, row, tbase, et, half, wp, &abort_s,
                                             wlim))
          break;
      } else if constexpr (MX && EPI == EPI_DGRAD2) {
        static_assert(S::OUT_BYTES >= 8 * kD2WarpBytes, "per-warp staging");
        epilogue_dgrad2_mx<BN>(args, ti, row, tbase, half, smem + STAGES * S::STAGE_BYTES, et);
      } else {
        epilogue<BN, EPI>(args, ti, row, tbase, half, &tmO0, &tmO1,
                          stage0 + STAGES * S::STAGE_BYTES, et, sub);
      }
      tc_fence_before();
      mbar_arrive(tempty_bar(acc));
      acc_phase ^= 1u << acc;
    }
    if (EPI == EPI_WGRAD && et == 0) {
      // after an abort: let every gradient chunk load still in flight land
      for (int n = wp.next; n < wp.issued; ++n)
        mbar_wait_drain(wg_bar0 + 8u * (uint32_t)(n % WB), (uint32_t)((n / WB) & 1));
    }
    if (et == 0) bulk_wait_all();   // every output store has completed
  }

  pdl_trigger();   // this CTA's tiles are done: the next kernel may be scheduled
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, S::TMEM_COLS);
  }
}

template <int BN, bool A_MN, bool B_MN, int EPI, bool MX, bool NV = false>
cudaError_t launch_one(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                       const CUtensorMap& to0, const CUtensorMap& to1, const GemmArgs& args,
                       int grid, cudaStream_t stream) {
  auto kern = k_grouped_gemm<BN, A_MN, B_MN, EPI, MX, NV>;
  const int smem = GemmShape<BN, EPI, MX, NV>::SMEM_BYTES;
  constexpr int threads = gemm_threads<NV>();
  static std::atomic<unsigned long long> configured{0};   // devices this kernel is set up on
  const cudaError_t e = smem_optin_once(kern, smem, configured);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(threads), smem, stream, ta, tb, tc, to0, to1, args);
}

}  // namespace

cudaError_t launch_gemm_nvfp4(int epi, const CUtensorMap& ta, const CUtensorMap& tb,
                              const CUtensorMap& to0, const GemmArgs& args, int grid,
                              cudaStream_t stream) {
  if (epi == EPI_SWIGLU)
    return launch_one<256, false, false, EPI_SWIGLU, true, true>(ta, tb, ta, to0, to0, args, grid,
                                                                 stream);
  if (epi == EPI_SCORE)
    return launch_one<256, false, false, EPI_SCORE, true, true>(ta, tb, ta, to0, to0, args, grid,
                                                                stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemm(int epi, int bn, bool a_mn, bool b_mn, const CUtensorMap& ta,
                        const CUtensorMap& tb, const CUtensorMap& tc, const CUtensorMap& to0,
                        const CUtensorMap& to1, const GemmArgs& args, int grid,
                        cudaStream_t stream, bool mx) {
  if (mx) {
    if (epi == EPI_SWIGLU && bn == 256 && !a_mn && !b_mn)
      return launch_one<256, false, false, EPI_SWIGLU, true>(ta, tb, tc, to0, to1, args, grid, stream);
    if (epi == EPI_SCORE && bn == 256 && !a_mn && !b_mn)
      return launch_one<256, false, false, EPI_SCORE, true>(ta, tb, tc, to0, to1, args, grid, stream);
    if (epi == EPI_SCORE && bn == 128 && !a_mn && !b_mn)
      return launch_one<128, false, false, EPI_SCORE, true>(ta, tb, tc, to0, to1, args, grid, stream);
    if (epi == EPI_STORE && bn == 256 && !a_mn && !b_mn)
      return launch_one<256, false, false, EPI_STORE, true>(ta, tb, tc, to0, to1, args, grid, stream);
    if (epi == EPI_DGRAD2 && bn == 128 && !a_mn && !b_mn)
      return launch_one<128, false, false, EPI_DGRAD2, true>(ta, tb, tc, to0, to1, args, grid, stream);
    if (epi == EPI_STORE && bn == 128 && !a_mn && !b_mn)
      return launch_one<128, false, false, EPI_STORE, true>(ta, tb, tc, to0, to1, args, grid, stream);
    if (epi == EPI_WGRAD && bn == 128 && !a_mn && !b_mn)
      return launch_one<128, false, false, EPI_WGRAD, true>(ta, tb, tc, to0, to1, args, grid, stream);
    return cudaErrorInvalidValue;
  }
#define MOE_CASE(EPI_, BN_, AMN_, BMN_)                                     \
  if (epi == EPI_ && bn == BN_ && a_mn == AMN_ && b_mn == BMN_)             \
    return launch_one<BN_, AMN_, BMN_, EPI_, false>(ta, tb, tc, to0, to1, args, grid, stream);
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
