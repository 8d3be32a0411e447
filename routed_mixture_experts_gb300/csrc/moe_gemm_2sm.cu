// moe_gemm_2sm.cu -- the grouped GEMM over routed rows on CTA pairs: two CTAs
// of a thread-block cluster compute one 256-row x 256-column tile with
// tcgen05.mma.cta_group::2 (M = 256).  Each CTA keeps its own 128 rows of A and
// one half of B (128 of the 256 columns) in shared memory, and its own 128
// accumulator rows in tensor memory, so a pipeline stage is 32 KB per CTA
// (6 stages) and each CTA reads a third less from L2 than a one-CTA tile of
// the same shape.  Used for W13 + SwiGLU, W2 x score, DGRAD-W2 + SwiGLU backward
// and DGRAD-W13 ("Dist-MoE" note, "What it is selling"; nvfp4moe README, "MoE
// layer" and "Training") when expert segments are padded to 256 rows.
//
// Roles (10 warps per CTA, both CTAs):
//   warp 0   TMA producer: loads this CTA's A rows and B half; completion is
//            counted on the leader CTA's (cluster rank 0) stage barrier
//   warp 1   TMEM allocation (cta_group::2, both CTAs); in the leader only, the
//            MMA issuer; its commits are multicast to both CTAs' barriers
//   warps 2..9  epilogue on this CTA's accumulator rows (same code as the
//            one-CTA kernel); each warp reports "accumulator drained" to the
//            leader
// Every mbarrier wait is bounded; a CTA whose wait gives up records
// MOE_ERR_TIMEOUT and stops.  Both CTAs always reach the closing cluster
// barrier, after which tensor memory is freed.

#include "moe_gemm_common.cuh"

namespace moe {

using namespace gemm;

namespace {

constexpr int kPairBN = 256;                 // N of the pair tile
constexpr int kPairStageBytes = 2 * 16384;   // A 128 x 64 + B half 128 x 64 (bf16)
constexpr uint32_t kPairTmemCols = 512;      // two 256-column accumulators

// bf16 output staging (one-output epilogues) and the pipeline depth it leaves
template <int EPI>
struct PairShape {
  static constexpr int OUT_BYTES = ((EPI == EPI_SCORE || EPI == EPI_STORE) ? kEpiStageBufs : tri_bufs<EPI>()) * 16384;
  // at most 6 stages (192 KB): the rest of the on-chip memory stays L1 for the
  // epilogues' row loads (SwiGLU backward reads h and a per row)
  static constexpr int STAGES_FIT = (226 * 1024 - OUT_BYTES) / kPairStageBytes;
  static constexpr int STAGES = STAGES_FIT > 6 ? 6 : STAGES_FIT;
  static constexpr int SMEM = STAGES * kPairStageBytes + OUT_BYTES + 256 + 1024;
};

template <bool B_MN, int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    k_grouped_gemm_2sm(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmO0,
                       const __grid_constant__ CUtensorMap tmO1, const GemmArgs args) {
  constexpr int BN = kPairBN;
  using PS = PairShape<EPI>;
  constexpr int STAGES = PS::STAGES;
  static_assert(PS::SMEM <= 232448, "shared memory budget");
  constexpr uint32_t IDESC = idesc_bf16(256, BN, false, B_MN);
  static_assert(EPI != EPI_WGRAD, "rows mode only");
  pdl_wait();   // the previous kernel of the stream has completed

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t tmem_holder;
  __shared__ int num_tiles_s;
  __shared__ volatile int abort_s;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * kPairStageBytes + PS::OUT_BYTES);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const uint64_t wlim = args.wait_limit_ns ? args.wait_limit_ns : kWaitLimitNs;

  if (threadIdx.x == 0) {
    num_tiles_s = (args.mtile_list ? *args.list_count : (*args.num_mtiles >> 1)) * args.n_tiles;
    abort_s = 0;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);        // leader: one arrive (with both CTAs' bytes)
      mbar_init(empty_bar(s), 1);       // one multicast commit per use
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 16);     // leader: 8 epilogue warps of each CTA
    }
    mbar_init(drain_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int num_tiles = num_tiles_s;
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;
  if (pair >= num_tiles) return;   // both CTAs of the cluster leave together

  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&tmem_holder), kPairTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmO0);
    tma_prefetch_desc(&tmO1);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();                  // both CTAs' barriers initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = tmem_holder;
  const uint32_t stage0 = smem_u32(smem);

  auto decode = [&](int tile, TileInfo& ti) {
    const int mp = tile / args.n_tiles;
    ti.nt = tile - mp * args.n_tiles;
    const int mt = args.mtile_list ? args.mtile_list[mp] : 2 * mp;   // the pair's first m tile
    ti.e = args.tile_expert ? args.tile_expert[mt] : 0;
    ti.m0 = mt * 128 + 128 * (int)rank;        // this CTA's rows
    ti.n0 = ti.nt * BN;
    ti.kb = args.k_blocks;
    ti.krow0 = 0;
  };

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs; lane 0 alone) ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued_parity[STAGES];
#pragma unroll
      for (int s = 0; s < STAGES; ++s) issued_parity[s] = -1;
      bool ok = true;
      for (int tile = pair; tile < num_tiles && ok; tile += npairs) {
        TileInfo ti;
        decode(tile, ti);
        for (int kb = 0; kb < ti.kb; ++kb) {
          ok = mbar_wait_cluster(empty_bar(stage), phase ^ 1u, &abort_s, args.err, 1, wlim);
          if (!ok) break;
          const uint32_t fb = mapa_shared(full_bar(stage), 0);    // the leader's barrier
          const uint32_t sa = stage0 + stage * kPairStageBytes;
          const uint32_t sb = sa + 16384;
          if (leader) mbar_arrive_expect_tx(full_bar(stage), 2 * kPairStageBytes);
          // one TMA per operand tile: this CTA's 128 A rows and its 128-column B half
          tma_load_2d_pair(sa, &tmA, kb * kBK, ti.m0, fb);
          if (B_MN) {
            // [E*K, N]: two 64-wide atoms of this CTA's half of the columns
            tma_load_3d_pair(sb, &tmB, 0, ti.e * args.b_expert_rows + kb * kBK,
                             (ti.n0 + 128 * (int)rank) >> 6, fb);
          } else if (EPI == EPI_SWIGLU) {
            // CTA 0: 128 gate rows, CTA 1: the 128 up rows of the same columns
            tma_load_2d_pair(sb, &tmB, kb * kBK,
                             ti.e * args.b_expert_rows + (int)rank * args.b_half_rows +
                                 ti.nt * (BN / 2),
                             fb);
          } else {
            tma_load_2d_pair(sb, &tmB, kb * kBK,
                             ti.e * args.b_expert_rows + ti.n0 + 128 * (int)rank, fb);
          }
          issued_parity[stage] = (int)phase;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!abort_s) {
        // every stage this CTA filled has been released by the leader's MMAs
        for (int s = 0; s < STAGES; ++s) {
          if (!mbar_wait_cluster(empty_bar(stage), phase ^ 1u, &abort_s, args.err, 2, wlim)) break;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (abort_s && leader) {
        // the leader's stage barriers count both CTAs' copies: let them land
        for (int s = 0; s < STAGES; ++s)
          if (issued_parity[s] >= 0) mbar_wait_drain(full_bar(s), (uint32_t)issued_parity[s]);
      }
      if (abort_s) {
        // a copy the peer issued for a stage this CTA never armed is not counted
        // anywhere: give every copy in flight time to land before the CTAs leave
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer (leader CTA, lane 0 alone) ----------------
    // shared-memory descriptors: a fixed base plus the stage and K-step offsets
    // in 16-byte units (K-major K step 32 B; MN-major B: 16 K rows = 2048 B)
    if (leader && lane == 0) {
      const uint64_t a_desc0 = smem_desc_sw128(stage0, 16, 1024);
      const uint64_t b_desc0 = B_MN ? smem_desc_sw128(stage0 + 16384, 8192, 1024)
                                    : smem_desc_sw128(stage0 + 16384, 16, 1024);
      constexpr uint32_t B_KSTEP = (B_MN ? 2048u : 32u) >> 4;
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = pair; tile < num_tiles && ok; tile += npairs) {
        TileInfo ti;
        decode(tile, ti);
        ok = mbar_wait_cluster(tempty_bar(acc), acc_phase ^ 1u, &abort_s, args.err, 3, wlim);
        if (args.stall_mma && ok)
          ok = mbar_wait(drain_bar, 0, &abort_s, args.err, 9, wlim);   // failure-path test
        if (!ok) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < ti.kb; ++kb) {
          ok = mbar_wait_cluster(full_bar(stage), phase, &abort_s, args.err, 4, wlim);
          if (!ok) break;
          tc_fence_after();
          const uint64_t soff = (uint64_t)((uint32_t)(stage * kPairStageBytes) >> 4);
#pragma unroll
          for (int k16 = 0; k16 < kBK / 16; ++k16)
            umma_f16_pair(d_tmem, a_desc0 + soff + (uint64_t)(k16 * 2),
                          b_desc0 + soff + (uint64_t)(k16 * B_KSTEP), IDESC,
                          (kb | k16) != 0 ? 1u : 0u);
          umma_commit_pair_mc(empty_bar(stage), 0x3);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair_mc(tfull_bar(acc), 0x3);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (abort_s) {
        umma_commit_pair_mc(drain_bar, 0x1);   // every MMA issued so far has completed
        mbar_wait_drain(drain_bar, 0);
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue (warps 2..9, both CTAs) ----------------
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int half = (warp - 2) >> 2;
    const uint32_t tempty0 = mapa_shared(tempty_bar(0), 0);
    const uint32_t tempty1 = mapa_shared(tempty_bar(1), 0);
    const int et = threadIdx.x - 64;
    const uint32_t out0 = stage0 + STAGES * kPairStageBytes;
    int seq = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = pair; tile < num_tiles; tile += npairs) {
      TileInfo ti;
      decode(tile, ti);
      int w = 1;
      if (lane == 0) w = mbar_wait_cluster(tfull_bar(acc), acc_phase, &abort_s, args.err, 5, wlim);
      // epilogues that share named barriers leave together; the others per warp
      const int ok_warp = __shfl_sync(0xffffffffu, w, 0);
      if (epi_bar_and(ok_warp) == 0) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
      epilogue<BN, EPI>(args, ti, row, tbase, half, &tmO0, &tmO1, out0, et, seq);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc ? tempty1 : tempty0);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (et == 0) bulk_wait_all();   // every output store has completed
  }

  pdl_trigger();   // this CTA's tiles are done: the next kernel may be scheduled
  tc_fence_before();
  __syncthreads();
  cluster_sync();                  // no CTA leaves while its peer may still signal it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kPairTmemCols);
  }
}

template <bool B_MN, int EPI>
cudaError_t launch_pair(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& to0,
                        const CUtensorMap& to1, const GemmArgs& args, int grid,
                        cudaStream_t stream) {
  auto kern = k_grouped_gemm_2sm<B_MN, EPI>;
  constexpr int smem = PairShape<EPI>::SMEM;
  static std::atomic<unsigned long long> configured{0};   // devices this kernel is set up on
  const cudaError_t e = smem_optin_once(kern, smem, configured);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid & ~1), dim3(kThreads), smem, stream, ta, tb, to0, to1, args);
}

}  // namespace

cudaError_t launch_gemm_pair(int epi, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb,
                             const CUtensorMap& to0, const CUtensorMap& to1, const GemmArgs& args,
                             int grid, cudaStream_t stream) {
  if (epi == EPI_SWIGLU && !b_mn) return launch_pair<false, EPI_SWIGLU>(ta, tb, to0, to1, args, grid, stream);
  if (epi == EPI_SCORE && !b_mn) return launch_pair<false, EPI_SCORE>(ta, tb, to0, to1, args, grid, stream);
  if (epi == EPI_STORE && !b_mn) return launch_pair<false, EPI_STORE>(ta, tb, to0, to1, args, grid, stream);
  if (epi == EPI_STORE && b_mn) return launch_pair<true, EPI_STORE>(ta, tb, to0, to1, args, grid, stream);
  if (epi == EPI_DGRAD2 && b_mn) return launch_pair<true, EPI_DGRAD2>(ta, tb, to0, to1, args, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace moe
