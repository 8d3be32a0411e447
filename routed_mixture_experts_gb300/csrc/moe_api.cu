// moe_api.cu -- the C ABI declared in include/moe.h: plan, workspace layout,
// tensor-map encoding and the launch sequence of forward and backward.
//
// Forward  ("Dist-MoE" note, "What it is selling": route on GPU -> W13 -> SwiGLU
//           -> W2 -> combine; nvfp4moe README, "MoE layer"):
//   route (3 small launches) -> gather x rows -> W13 GEMM + SwiGLU -> W2 GEMM x
//   score -> combine
// Backward ("What it is selling": DGRAD / WGRAD, in-place WGRAD accumulation;
//           nvfp4moe README, "Training": router gradients):
//   gather dY rows -> DGRAD-W2 + SwiGLU backward + score-grad partials ->
//   DGRAD-W13 -> combine dX and dscores -> WGRAD-W2 -> WGRAD-W13
// Everything is enqueued on the caller's stream; nothing allocates, nothing
// synchronises (moe_plan_check and moe_plan_set_workspace excepted).

#include <climits>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>

#include <cudaTypedefs.h>

#include "../../include/moe.h"
#include "moe_device.cuh"
#include "moe_internal.h"

using namespace moe;

struct moe_plan {
  int T, d, I, E, k, precision;
  float clamp;
  int num_sms;
  int R;        // T*k
  int RP;       // worst-case padded rows
  int nblk;     // dispatch chunks
  int bn13, bn2, bnd2, bnw2, bnw13;
  int bnmx_d;   // MXFP8 GEMMs whose N is d (W2, DGRAD-W13): 256-wide tiles when d allows
  int pair;     // W13, W2 and DGRAD-W13 on CTA pairs (256-row tiles over pairs of an
                // expert's 128-row m tiles; an odd last m tile runs on one CTA)
  int gran;     // padding granule of expert segments (128)
  // workspace
  char* ws;
  size_t ws_bytes;
  int ws_flags;
  // pointers into the workspace
  DevError* err;
  int32_t *counts, *m_indptr, *off_pad, *num_mtiles, *num_nonempty, *expert_order, *tile_expert,
      *blockcounts, *row_of, *token_of;
  float *score_of, *pdscore;
  uint16_t *xe, *h, *ys, *a, *dye, *dA, *hs, *dxe;
  // host staging
  uint16_t *st_x, *st_dy, *st_y, *st_dx;
  int32_t* st_ids;
  float *st_scores, *st_dscores;
  // tensor maps over workspace tensors
  // K-major maps load 128-row boxes (the A tiles); MN-major maps (suffix _mn) are
  // 3-D views loading a tile's 64-wide atoms in one box
  CUtensorMap tm_xe, tm_h, tm_dye, tm_dA;
  CUtensorMap tm_dye_mn, tm_dA_mn, tm_hs_mn, tm_xe_mn;
  // bf16 outputs stored by the TMA-store epilogues (128-row boxes)
  CUtensorMap tm_ys, tm_a, tm_hs, tm_dxe;
  // tensor maps over the caller's weights (re-encoded when the pointers change)
  CUtensorMap tm_w13, tm_w2, tm_w13_mn, tm_w2_mn;
  CUtensorMap tm_w13_p, tm_w2_p, tm_w13_mn_p;   // the CTA-pair kernel's (128-row halves)
  const void *w13_cached, *w2_cached;
  // CTA-pair tile lists (dispatch output): pairs of m tiles, odd last m tiles
  int32_t *pair_list, *left_list, *num_pairs, *num_left;
  // moe_forward_routed: the m tiles of the caller's layout and their count;
  // tensor maps over the caller's expert-major rows and outputs
  int32_t *routed_list, *routed_count;
  CUtensorMap tm_rx, tm_rys;
  const void *rx_cached, *rys_cached;
  long long rx_rows, rys_rows;
  // MXFP8: quantised expert-major activations and h, with tiled scales (NVFP4:
  // the same buffers hold packed E2M1 codes and E4M3 scales)
  uint8_t *xq, *xsf, *hq, *hsf;
  // NVFP4: static activation dequantisation scales (0: not set) and the weight maps
  float nv_x_scale, nv_h_scale;
  CUtensorMap tm_w13nv, tm_w2nv;
  const void *w13nv_cached, *w2nv_cached;
  int ngr_d, ngr_I;                 // 128-element scale groups along d and along I
  CUtensorMap tm_xq, tm_hq, tm_w13q, tm_w2q;
  const void *w13q_cached, *w2q_cached;
  // MXFP8 training: DGRAD operands quantised along their K (dY along d, dA along
  // 2I) and the WGRAD operands quantised along the rows, stored transposed
  // ([columns, Rpad], K-major over the rows), each with tiled scales
  uint8_t *dyq, *dysf, *dAq, *dAsf, *dyqT, *dyqTsf, *dAqT, *dAqTsf, *hsqT, *hsqTsf, *xqT, *xqTsf;
  CUtensorMap tm_dyq, tm_dAq, tm_dyqT, tm_dAqT, tm_hsqT, tm_xqT;
  CUtensorMap tm_w13t, tm_w2t;      // weights prepared for the backward (moe_prepare_weights_mxfp8_backward)
  const void *w13t_cached, *w2t_cached;
  // tensor maps over the caller's fp32 weight gradients (WGRAD outputs)
  CUtensorMap tm_dw13, tm_dw2;
  const void *dw13_cached, *dw2_cached;
  int saved;
  // failure-path testing knobs (moe_plan_set_debug)
  long long dbg_wait_limit_ns;
  int dbg_stall_w13;
  // optional stage events and the launch counter
  void* const* ev[2];
  int nev[2];
  long long launches;
  // moe_step_host: a side stream and events that overlap the dY upload with the
  // forward and the y download with the backward (created with a host-staging
  // workspace)
  cudaStream_t side;
  cudaEvent_t ev_fork, ev_dy, ev_y, ev_ydone, ev_x, ev_comb, ev_dxdone;
  // set by moe_step_host only: the forward waits on wait_before_gather before
  // its gather, the backward records record_after_combine after its combine
  cudaEvent_t wait_before_gather, record_after_combine;
  int prev_step_train;   // the last moe_step_host call on this plan was a complete training step
  // concurrent backward (moe_plan_set_backward_split): the weight-gradient GEMMs
  // run on wgrad_sms SMs on a plan-owned stream, beside DGRAD-W13 and the dX
  // combine on the rest (0: one stream, every GEMM on every SM)
  int wgrad_sms;
  cudaStream_t wstream;
  cudaEvent_t ev_wfork, ev_wjoin;
  // moe_plan_set_wgrad_interleave: weight-gradient tiles of experts with more
  // routed rows than this run interleaved with the shorter ones (0: plain order)
  long long wgrad_long_rows;
};

namespace moe {

namespace tmap_detail {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  // looked up once per process (thread-safe static initialisation)
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

int encode_2d(CUtensorMap* map, CUtensorMapDataType dt, int esize, const void* base,
              long long rows, long long cols, cuuint32_t box_cols, cuuint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return MOE_ERR_CUDA;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * esize};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace tmap_detail

using tmap_detail::encode_2d;

int encode_tmap_bf16(CUtensorMap* map, const void* base, long long rows, long long cols,
                     int box_rows) {
  return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, rows, cols, 64,
                   (cuuint32_t)box_rows);
}

int encode_tmap_bf16_mn(CUtensorMap* map, const void* base, long long krows, long long ncols,
                        int atoms) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = tmap_detail::encode_fn();
  if (!fn) return MOE_ERR_CUDA;
  // [K rows, N] viewed as dims (64 within an atom, K rows, N/64 atoms)
  const cuuint64_t dims[3] = {64, (cuuint64_t)krows, (cuuint64_t)(ncols / 64)};
  const cuuint64_t strides[2] = {(cuuint64_t)ncols * 2, 128};
  const cuuint32_t box[3] = {64, 64, (cuuint32_t)atoms};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

int encode_tmap_f32_out(CUtensorMap* map, const void* base, long long rows, long long cols) {
  return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, rows, cols, 32, 128);
}

int encode_tmap_u8(CUtensorMap* map, const void* base, long long rows, long long cols,
                   int box_rows) {
  return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base, rows, cols, 128,
                   (cuuint32_t)box_rows);
}

int encode_tmap_gate_up(CUtensorMap* map, bool fp8, const void* base, long long E, long long I,
                        long long cols, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = tmap_detail::encode_fn();
  if (!fn) return MOE_ERR_CUDA;
  const int esize = fp8 ? 1 : 2;
  // [E, 2, I, cols] viewed as dims (cols, I, 2E): one box takes box_rows gate rows
  // and the same rows of the up half
  const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)I, (cuuint64_t)(2 * E)};
  const cuuint64_t strides[2] = {(cuuint64_t)(cols * esize), (cuuint64_t)(I * cols * esize)};
  const cuuint32_t box[3] = {(cuuint32_t)(128 / esize), (cuuint32_t)box_rows, 2};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

// MXFP8 W13 [E, 2I, cols] (E4M3) viewed as (cols, 64, 2, I/64, E): one box takes
// two consecutive 64-row blocks of intermediate columns, each block its 64 gate
// rows followed by the same 64 up rows, which is the row order of the tiled
// scales of W13 (blocks of 64 gate + 64 up rows).
int encode_tmap_gate_up_blocks(CUtensorMap* map, const void* base, long long E, long long I,
                               long long cols) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = tmap_detail::encode_fn();
  if (!fn) return MOE_ERR_CUDA;
  const cuuint64_t dims[5] = {(cuuint64_t)cols, 64, 2, (cuuint64_t)(I / 64), (cuuint64_t)E};
  const cuuint64_t strides[4] = {(cuuint64_t)cols, (cuuint64_t)(I * cols),
                                 (cuuint64_t)(64 * cols), (cuuint64_t)(2 * I * cols)};
  const cuuint32_t box[5] = {128, 64, 2, 2, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

int pick_bn_n(int n) { return n % 256 == 0 ? 256 : (n % 128 == 0 ? 128 : 64); }

// Lays the workspace out (bases relative to `base`; base may be nullptr to size it).
size_t layout(moe_plan* p, char* base, int flags) {
  size_t off = 0;
  auto take = [&](size_t bytes) -> char* {
    char* r = base ? base + off : nullptr;
    off = align_up(off + bytes);
    return r;
  };
  const size_t RP = p->RP, d = p->d, I = p->I, E = p->E, T = p->T, k = p->k;
  p->err = reinterpret_cast<DevError*>(take(sizeof(DevError)));
  p->counts = reinterpret_cast<int32_t*>(take(4 * E));
  p->m_indptr = reinterpret_cast<int32_t*>(take(4 * (E + 1)));
  p->off_pad = reinterpret_cast<int32_t*>(take(4 * (E + 1)));
  p->num_mtiles = reinterpret_cast<int32_t*>(take(4));
  p->num_nonempty = reinterpret_cast<int32_t*>(take(4));
  p->expert_order = reinterpret_cast<int32_t*>(take(4 * E));
  p->tile_expert = reinterpret_cast<int32_t*>(take(4 * (RP / kBM)));
  p->routed_list = reinterpret_cast<int32_t*>(take(4 * (RP / kBM)));
  p->routed_count = reinterpret_cast<int32_t*>(take(4));
  p->pair_list = p->left_list = p->num_pairs = p->num_left = nullptr;
  if (p->pair) {
    p->pair_list = reinterpret_cast<int32_t*>(take(4 * (RP / kBM / 2 + 1)));
    p->left_list = reinterpret_cast<int32_t*>(take(4 * E));
    p->num_pairs = reinterpret_cast<int32_t*>(take(4));
    p->num_left = reinterpret_cast<int32_t*>(take(4));
  }
  p->blockcounts = reinterpret_cast<int32_t*>(take(4 * (size_t)p->nblk * E));
  p->row_of = reinterpret_cast<int32_t*>(take(4 * (size_t)p->R));
  p->token_of = reinterpret_cast<int32_t*>(take(4 * RP));
  p->score_of = reinterpret_cast<float*>(take(4 * RP));
  const bool mx = p->precision == MOE_PREC_MXFP8;
  const bool nv = p->precision == MOE_PREC_NVFP4;
  p->xe = (mx || nv) ? nullptr : reinterpret_cast<uint16_t*>(take(2 * RP * d));
  p->xq = p->xsf = p->hq = p->hsf = nullptr;
  if (nv) {
    // packed E2M1 codes, E4M3 scales per 16 elements (tiled, 64-element K groups)
    p->xq = reinterpret_cast<uint8_t*>(take(RP * d / 2));
    p->xsf = reinterpret_cast<uint8_t*>(take((size_t)nv_sf_bytes(RP, (int)d)));
    p->hq = reinterpret_cast<uint8_t*>(take(RP * I / 2));
    p->hsf = reinterpret_cast<uint8_t*>(take((size_t)nv_sf_bytes(RP, (int)I)));
  }
  if (mx) {
    p->xq = reinterpret_cast<uint8_t*>(take(RP * d));
    p->xsf = reinterpret_cast<uint8_t*>(take((size_t)mx_sf_bytes(RP, (int)d)));
    p->hq = reinterpret_cast<uint8_t*>(take(RP * I));
    p->hsf = reinterpret_cast<uint8_t*>(take((size_t)mx_sf_bytes(RP, (int)I)));
  }
  // bf16 h: the W2 operand of bf16 plans (MXFP8 plans keep only its E4M3 codes)
  p->h = (mx || nv) ? nullptr : reinterpret_cast<uint16_t*>(take(2 * RP * I));
  p->ys = reinterpret_cast<uint16_t*>(take(2 * RP * d));
  p->a = p->dye = p->dA = p->hs = p->dxe = nullptr;
  p->pdscore = nullptr;
  p->dyq = p->dysf = p->dAq = p->dAsf = p->dyqT = p->dyqTsf = nullptr;
  p->dAqT = p->dAqTsf = p->hsqT = p->hsqTsf = p->xqT = p->xqTsf = nullptr;
  if ((flags & MOE_WS_TRAINING) && mx) {
    // dA and hs only as E4M3 codes (written by the DGRAD-W2 epilogue)
    p->a = reinterpret_cast<uint16_t*>(take(2 * RP * 2 * I));
    p->dxe = reinterpret_cast<uint16_t*>(take(2 * RP * d));
    p->pdscore = reinterpret_cast<float*>(take(4 * RP * 2 * (I / p->bnd2)));
    auto q = [&](size_t rows, size_t cols, uint8_t** codes, uint8_t** sf) {
      *codes = reinterpret_cast<uint8_t*>(take(rows * cols));
      *sf = reinterpret_cast<uint8_t*>(take((size_t)mx_sf_bytes((long long)rows, (int)cols)));
    };
    q(RP, d, &p->dyq, &p->dysf);
    q(RP, 2 * I, &p->dAq, &p->dAsf);
    q(d, RP, &p->dyqT, &p->dyqTsf);
    q(2 * I, RP, &p->dAqT, &p->dAqTsf);
    q(I, RP, &p->hsqT, &p->hsqTsf);
    q(d, RP, &p->xqT, &p->xqTsf);
  }
  if ((flags & MOE_WS_TRAINING) && !mx) {
    p->a = reinterpret_cast<uint16_t*>(take(2 * RP * 2 * I));
    p->dye = reinterpret_cast<uint16_t*>(take(2 * RP * d));
    p->dA = reinterpret_cast<uint16_t*>(take(2 * RP * 2 * I));
    p->hs = reinterpret_cast<uint16_t*>(take(2 * RP * I));
    p->dxe = reinterpret_cast<uint16_t*>(take(2 * RP * d));
    p->pdscore = reinterpret_cast<float*>(take(4 * RP * 2 * (I / p->bnd2)));
  }
  p->st_x = p->st_dy = p->st_y = p->st_dx = nullptr;
  p->st_ids = nullptr;
  p->st_scores = p->st_dscores = nullptr;
  if (flags & MOE_WS_HOST_STAGING) {
    p->st_x = reinterpret_cast<uint16_t*>(take(2 * T * d));
    p->st_ids = reinterpret_cast<int32_t*>(take(4 * T * k));
    p->st_scores = reinterpret_cast<float*>(take(4 * T * k));
    p->st_y = reinterpret_cast<uint16_t*>(take(2 * T * d));
    if (flags & MOE_WS_TRAINING) {
      p->st_dy = reinterpret_cast<uint16_t*>(take(2 * T * d));
      p->st_dx = reinterpret_cast<uint16_t*>(take(2 * T * d));
      p->st_dscores = reinterpret_cast<float*>(take(4 * T * k));
    }
  }
  return off;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int cuda_status_at(cudaError_t e, int line) {
  if (e == cudaSuccess) return MOE_OK;
  fprintf(stderr, "moe_gb300: CUDA error %s (moe_api.cu:%d)\n", cudaGetErrorString(e), line);
  return MOE_ERR_CUDA;
}
#define cuda_status(e) cuda_status_at((e), __LINE__)

int reset_error_word(DevError* err) {
  DevError h;
  h.code = 0;
  h.first_bad = INT_MAX;
  h.where = 0;
  h.pad = 0;
  return cuda_status(cudaMemcpy(err, &h, sizeof(h), cudaMemcpyHostToDevice));
}

int refresh_weight_maps(moe_plan* p, const void* w13, const void* w2) {
  // B boxes of the one-CTA kernel: W13 gate and up rows of a tile in one 3-D box,
  // W2 rows of one N tile; the CTA-pair kernel loads 128-row halves (2-D boxes,
  // two 64-wide atoms MN-major)
  if (w13 != p->w13_cached) {
    const long long r13 = (long long)p->E * 2 * p->I;
    if (encode_tmap_gate_up(&p->tm_w13, false, w13, p->E, p->I, p->d, p->bn13 / 2) != MOE_OK ||
        encode_tmap_bf16_mn(&p->tm_w13_mn, w13, r13, p->d, p->bn2 / 64) != MOE_OK)
      return MOE_ERR_CUDA;
    if (p->pair && (encode_tmap_bf16(&p->tm_w13_p, w13, r13, p->d, 128) != MOE_OK ||
                    encode_tmap_bf16_mn(&p->tm_w13_mn_p, w13, r13, p->d, 2) != MOE_OK))
      return MOE_ERR_CUDA;
    p->w13_cached = w13;
  }
  if (w2 != p->w2_cached) {
    const long long r2 = (long long)p->E * p->d;
    if (encode_tmap_bf16(&p->tm_w2, w2, r2, p->I, p->bn2) != MOE_OK ||
        encode_tmap_bf16_mn(&p->tm_w2_mn, w2, r2, p->I, p->bnd2 / 64) != MOE_OK)
      return MOE_ERR_CUDA;
    if (p->pair && encode_tmap_bf16(&p->tm_w2_p, w2, r2, p->I, 128) != MOE_OK) return MOE_ERR_CUDA;
    p->w2_cached = w2;
  }
  return MOE_OK;
}

// Weight-gradient tiles of experts with more routed rows than this are
// interleaved with the shorter tiles (gemm::SegIter).  On the skewed workload
// (heaviest expert 15.7K rows, median 350) WGRAD-W2 / WGRAD-W13 took 0.465 /
// 0.840 ms in plain order, 0.442 / 0.828 with 2560 rows, 0.444 / 0.830 with
// 1280 and 0.460 / 0.848 with 5000.
constexpr long long kWgradLongRows = 2560;

GemmArgs rows_args(const moe_plan* p) {
  GemmArgs g;
  memset(&g, 0, sizeof(g));
  g.wait_limit_ns = (unsigned long long)p->dbg_wait_limit_ns;
  g.wgrad = 0;
  g.num_mtiles = p->num_mtiles;
  g.tile_expert = p->tile_expert;
  g.err = p->err;
  g.clamp = p->clamp;
  g.I = p->I;
  return g;
}

// rows per K stage: 64 (bf16) or 128 (block-scaled)
GemmArgs wgrad_args(const moe_plan* p, int kstep) {
  GemmArgs g;
  memset(&g, 0, sizeof(g));
  g.wait_limit_ns = (unsigned long long)p->dbg_wait_limit_ns;
  g.wgrad = 1;
  g.wgrad_kstep = kstep == 64 ? 0 : kstep;
  g.wgrad_long_kb = (int)(p->wgrad_long_rows / kstep);
  g.off_pad = p->off_pad;
  g.expert_order = p->expert_order;
  g.num_nonempty = p->num_nonempty;
  g.err = p->err;
  return g;
}

// gathers and combines: 16 CTAs of 256 threads per SM, of which the registers let
// two run at a time (the rest queue; more CTAs measured 5 % faster gathers than 8)
int gather_grid(const moe_plan* p) { return p->num_sms * 16; }

void mark(const moe_plan* p, int which, int i, cudaStream_t st);
cudaError_t launch_wgrad_bf16(moe_plan* p, cudaStream_t st, float* dw13, float* dw2, int grid);
cudaError_t launch_wgrad_mx(moe_plan* p, cudaStream_t st, float* dw13, float* dw2, int grid);

// MXFP8 forward after dispatch ("What it is selling": MXFP8 E4M3 quantises
// activations after routing and takes prepared weights; staged W13 and W2):
// gather + quantise x rows -> block-scaled W13 GEMM + SwiGLU + quantise h ->
// block-scaled W2 GEMM x score -> combine.
int forward_mxfp8(moe_plan* p, const void* x, const uint8_t* w13_sf, const uint8_t* w2_sf,
                  void* y, int save, cudaStream_t st) {
  // gather + quantise x rows along d; a saving forward also quantises them along
  // the rows, transposed (the WGRAD-W13 operand), in the same pass
  cudaError_t e =
      save ? launch_quant_two_way(x, p->token_of, p->off_pad + p->E, p->RP, p->d, p->xq, p->xsf,
                                  p->xqT, p->xqTsf, p->num_sms, st)
           : launch_gather_quant_rows(x, p->token_of, p->off_pad + p->E, p->d, p->xq, p->xsf,
                                      gather_grid(p), st);
  if (e != cudaSuccess) return cuda_status(e);
  p->launches += 1;
  mark(p, 0, 2, st);
  {
    // 256-wide tiles: 128 intermediate columns (two 64-row blocks of gate and up
    // rows) per tile; outputs hq/hsf, and a when saving
    GemmArgs g = rows_args(p);
    g.k_blocks = p->d / 128;
    g.b_expert_rows = 2 * p->I;
    g.b_half_rows = p->I;
    g.n_tiles = p->I / 128;
    g.ld0 = p->I;                        // row stride of hq
    g.sfa = p->xsf; g.sfb = w13_sf; g.sf_ngr = p->ngr_d; g.b_blocks_per_expert = p->I / 64;
    g.hq = p->hq; g.hsf = p->hsf; g.hsf_ngr = p->ngr_I;
    g.k_rotate = 1;
    g.save = save ? 1 : 0;
    g.stall_mma = p->dbg_stall_w13;
    const CUtensorMap& to = save ? p->tm_a : p->tm_ys;   // tm_ys: not written here
    e = launch_gemm(EPI_SWIGLU, 256, false, false, p->tm_xq, p->tm_w13q, p->tm_xq, to, to, g,
                    p->num_sms, st, true);
    if (e != cudaSuccess) return cuda_status(e);
    p->launches += 1;
    mark(p, 0, 3, st);
  }
  {
    GemmArgs g = rows_args(p);
    g.k_blocks = p->I / 128;
    g.b_expert_rows = p->d;
    g.n_tiles = p->d / p->bnmx_d;
    g.out0 = p->ys; g.ld0 = p->d;
    g.row_scale = p->score_of;
    g.sfa = p->hsf; g.sfb = w2_sf; g.sf_ngr = p->ngr_I; g.b_blocks_per_expert = p->d / 128;
    g.k_rotate = 1;
    e = launch_gemm(EPI_SCORE, p->bnmx_d, false, false, p->tm_hq, p->tm_w2q, p->tm_hq, p->tm_ys,
                    p->tm_ys, g, p->num_sms, st, true);
    if (e != cudaSuccess) return cuda_status(e);
    p->launches += 1;
    mark(p, 0, 4, st);
  }
  e = launch_combine(p->ys, p->row_of, p->T, p->k, p->d, y, nullptr, 0, nullptr, gather_grid(p), st);
  if (e != cudaSuccess) return cuda_status(e);
  p->launches += 1;
  mark(p, 0, 5, st);
  p->saved = 0;
  return MOE_OK;
}

// b5, b6 of the bf16 backward: dW2[e] += dY_e^T . hs_e, then dW13[e] += dA_e^T .
// x_e, on `grid` CTAs of stream st (stage marks 5 and 6 recorded there).
cudaError_t launch_wgrad_bf16(moe_plan* p, cudaStream_t st, float* dw13, float* dw2, int grid) {
  const int I = p->I, d = p->d;
  {
    GemmArgs g = wgrad_args(p, 64);
    g.m_tiles = d / kBM;
    g.n_tiles = I / p->bnw2;
    g.out0 = dw2; g.ld0 = I;
    g.out_expert_stride = (long long)d * I;
    cudaError_t e = launch_gemm(EPI_WGRAD, p->bnw2, true, true, p->tm_dye_mn, p->tm_hs_mn,
                                p->tm_dw2, p->tm_dw2, p->tm_dw2, g, grid, st);
    if (e != cudaSuccess) return e;
    p->launches += 1;
    mark(p, 1, 5, st);
  }
  {
    GemmArgs g = wgrad_args(p, 64);
    g.m_tiles = 2 * I / kBM;
    g.n_tiles = d / p->bnw13;
    g.out0 = dw13; g.ld0 = d;
    g.out_expert_stride = 2LL * I * d;
    cudaError_t e = launch_gemm(EPI_WGRAD, p->bnw13, true, true, p->tm_dA_mn, p->tm_xe_mn,
                                p->tm_dw13, p->tm_dw13, p->tm_dw13, g, grid, st);
    if (e != cudaSuccess) return e;
    p->launches += 1;
    mark(p, 1, 6, st);
  }
  return cudaSuccess;
}

// b5, b6 of the MXFP8 backward (block-scaled WGRAD over each expert's rows), on
// `grid` CTAs of stream st.
cudaError_t launch_wgrad_mx(moe_plan* p, cudaStream_t st, float* dw13, float* dw2, int grid) {
  const int I = p->I, d = p->d;
  const long long RP = p->RP;
  {
    GemmArgs g = wgrad_args(p, 128);
    g.m_tiles = d / kBM;
    g.n_tiles = I / 128;
    g.out0 = dw2; g.ld0 = I;
    g.out_expert_stride = (long long)d * I;
    g.sfa = p->dyqTsf; g.sfb = p->hsqTsf; g.sf_ngr = (int)(RP / 128);
    cudaError_t e = launch_gemm(EPI_WGRAD, 128, false, false, p->tm_dyqT, p->tm_hsqT, p->tm_dw2,
                                p->tm_dw2, p->tm_dw2, g, grid, st, true);
    if (e != cudaSuccess) return e;
    p->launches += 1;
    mark(p, 1, 5, st);
  }
  {
    GemmArgs g = wgrad_args(p, 128);
    g.m_tiles = 2 * I / kBM;
    g.n_tiles = d / 128;
    g.out0 = dw13; g.ld0 = d;
    g.out_expert_stride = 2LL * I * d;
    g.sfa = p->dAqTsf; g.sfb = p->xqTsf; g.sf_ngr = (int)(RP / 128);
    cudaError_t e = launch_gemm(EPI_WGRAD, 128, false, false, p->tm_dAqT, p->tm_xqT, p->tm_dw13,
                                p->tm_dw13, p->tm_dw13, g, grid, st, true);
    if (e != cudaSuccess) return e;
    p->launches += 1;
    mark(p, 1, 6, st);
  }
  return cudaSuccess;
}

void mark(const moe_plan* p, int which, int i, cudaStream_t st) {
  if (!(p->ev[which] && i < p->nev[which] && p->ev[which][i])) return;
  cudaEvent_t ev = static_cast<cudaEvent_t>(p->ev[which][i]);
  // while a stream is being captured into a CUDA graph the record must be an
  // "external" one to stay a real (timed) event record in the graph
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  const bool capturing =
      cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive;
  const cudaError_t e = capturing ? cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal)
                                  : cudaEventRecord(ev, st);
  if (e != cudaSuccess) (void)cudaGetLastError();   // optional timing: never fail the step
}

}  // namespace

extern "C" {

const char* moe_status_string(int s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_STATE: return "MOE_ERR_STATE";
    case MOE_ERR_BAD_IDS: return "MOE_ERR_BAD_IDS";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    default: return "MOE_ERR_UNKNOWN";
  }
}

int moe_tile_rows(void) { return kBM; }

int moe_plan_row_granule(const moe_plan* p) { return p ? p->gran : 0; }

moe_plan* moe_plan_create(int T, int d, int I, int E, int k, int precision) {
  if (T < 1 || d < 128 || I < 64 || d % 128 || I % 64 || k < 1 || E < k || E > 256) return nullptr;
  if ((long long)T * k >= (1LL << 31) - (long long)E * kBM) return nullptr;
  if (precision != MOE_PREC_BF16 && precision != MOE_PREC_MXFP8 && precision != MOE_PREC_NVFP4)
    return nullptr;
  // MXFP8: K loops in 128-element stages (scales travel with each stage); NVFP4:
  // 256-element stages along d (W13) and I (W2)
  if (precision == MOE_PREC_MXFP8 && I % 128) return nullptr;
  if (precision == MOE_PREC_NVFP4 && (I % 256 || d % 256)) return nullptr;
  moe_plan* p = new (std::nothrow) moe_plan;
  if (!p) return nullptr;
  memset(p, 0, sizeof(*p));
  p->T = T; p->d = d; p->I = I; p->E = E; p->k = k; p->precision = precision;
  p->R = T * k;
  // one-CTA row GEMMs with 128-row expert segments unless CTA pairs are chosen
  // (moe_plan_set_cta_pairs) before the workspace is sized
  p->pair = 0;
  p->gran = kBM;
  p->RP = (int)(((long long)p->R + (long long)E * (p->gran - 1)) / p->gran * p->gran);
  p->nblk = (p->R + 1023) / 1024;
  p->bn13 = I % 128 == 0 ? 256 : 128;
  p->bn2 = pick_bn_n(d) == 64 ? 128 : pick_bn_n(d);
  p->bnd2 = precision == MOE_PREC_MXFP8 ? 128 : pick_bn_n(I);   // block-scaled DGRAD-W2: 128 wide
  p->bnmx_d = d % 256 == 0 ? 256 : 128;
  p->bnw2 = pick_bn_n(I);
  p->bnw13 = p->bn2;
  p->ngr_d = d / 128;
  p->ngr_I = I / 128;
  p->wgrad_long_rows = kWgradLongRows;
  int dev = 0;
  p->num_sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
      p->num_sms = n;
  }
  return p;
}

void moe_plan_destroy(moe_plan* p) {
  if (!p) return;
  if (p->wstream) {
    cudaStreamDestroy(p->wstream);
    cudaEventDestroy(p->ev_wfork);
    cudaEventDestroy(p->ev_wjoin);
  }
  if (p->side) {
    cudaStreamDestroy(p->side);
    cudaEventDestroy(p->ev_fork);
    cudaEventDestroy(p->ev_dy);
    cudaEventDestroy(p->ev_y);
    cudaEventDestroy(p->ev_ydone);
    cudaEventDestroy(p->ev_x);
    cudaEventDestroy(p->ev_comb);
    cudaEventDestroy(p->ev_dxdone);
  }
  delete p;
}

int moe_plan_set_cta_pairs(moe_plan* p, int on) {
  if (!p) return MOE_ERR_INVALID_ARG;
  if (p->ws) return MOE_ERR_STATE;               // the granule sizes the workspace
  if (on && (p->precision != MOE_PREC_BF16 || p->I % 256 || p->d % 256)) return MOE_ERR_UNSUPPORTED;
  p->pair = on ? 1 : 0;
  return MOE_OK;
}

int moe_plan_set_swiglu_clamp(moe_plan* p, float limit) {
  if (!p || !(limit >= 0.f)) return MOE_ERR_INVALID_ARG;
  p->clamp = limit;
  return MOE_OK;
}

size_t moe_plan_workspace_bytes(const moe_plan* p, int flags) {
  if (!p) return 0;
  moe_plan tmp = *p;
  return layout(&tmp, nullptr, flags);
}

int moe_plan_set_workspace(moe_plan* p, void* ws, size_t bytes, int flags) {
  if (!p || !ws || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1))) return MOE_ERR_INVALID_ARG;
  // NVFP4 is inference-only: it refuses a training workspace
  if (p->precision == MOE_PREC_NVFP4 && (flags & MOE_WS_TRAINING)) return MOE_ERR_UNSUPPORTED;
  if (bytes < moe_plan_workspace_bytes(p, flags)) return MOE_ERR_WORKSPACE;
  if ((flags & MOE_WS_HOST_STAGING) && !p->side) {
    const unsigned ef = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&p->side, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&p->ev_fork, ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&p->ev_dy, ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&p->ev_y, ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&p->ev_ydone, ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&p->ev_x, ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&p->ev_comb, ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&p->ev_dxdone, ef) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  p->ws = static_cast<char*>(ws);
  p->ws_bytes = bytes;
  p->ws_flags = flags;
  layout(p, p->ws, flags);
  p->saved = 0;
  p->prev_step_train = 0;
  p->w13_cached = p->w2_cached = nullptr;
  p->dw13_cached = p->dw2_cached = nullptr;
  p->w13q_cached = p->w2q_cached = nullptr;
  p->rx_cached = p->rys_cached = nullptr;
  p->w13nv_cached = p->w2nv_cached = nullptr;
  const long long RP = p->RP;
  if (p->precision == MOE_PREC_NVFP4) {
    if (encode_tmap_u8(&p->tm_xq, p->xq, RP, p->d / 2, 128) ||
        encode_tmap_u8(&p->tm_hq, p->hq, RP, p->I / 2, 128) ||
        encode_tmap_bf16(&p->tm_ys, p->ys, RP, p->d, 128))
      return MOE_ERR_CUDA;
    if (flags & MOE_WS_HOST_STAGING) return MOE_ERR_UNSUPPORTED;
    return reset_error_word(p->err);
  }
  p->w13t_cached = p->w2t_cached = nullptr;
  if (p->precision == MOE_PREC_MXFP8) {
    if (encode_tmap_u8(&p->tm_xq, p->xq, RP, p->d, 128) ||
        encode_tmap_u8(&p->tm_hq, p->hq, RP, p->I, 128) ||
        encode_tmap_bf16(&p->tm_ys, p->ys, RP, p->d, 128))
      return MOE_ERR_CUDA;
    if ((flags & MOE_WS_TRAINING) &&
        encode_tmap_bf16(&p->tm_a, p->a, RP, 2LL * p->I, 128))
      return MOE_ERR_CUDA;
    if ((flags & MOE_WS_TRAINING) &&
        (encode_tmap_u8(&p->tm_dyq, p->dyq, RP, p->d, 128) ||
         encode_tmap_u8(&p->tm_dAq, p->dAq, RP, 2LL * p->I, 128) ||
         encode_tmap_u8(&p->tm_dyqT, p->dyqT, p->d, RP, 128) ||
         encode_tmap_u8(&p->tm_dAqT, p->dAqT, 2LL * p->I, RP, 128) ||
         encode_tmap_u8(&p->tm_hsqT, p->hsqT, p->I, RP, 128) ||
         encode_tmap_u8(&p->tm_xqT, p->xqT, p->d, RP, 128) ||
         encode_tmap_bf16(&p->tm_dxe, p->dxe, RP, p->d, 128)))
      return MOE_ERR_CUDA;
    return reset_error_word(p->err);
  }
  if (encode_tmap_bf16(&p->tm_xe, p->xe, RP, p->d, 128) ||
      encode_tmap_bf16(&p->tm_h, p->h, RP, p->I, 128) ||
      encode_tmap_bf16(&p->tm_ys, p->ys, RP, p->d, 128))
    return MOE_ERR_CUDA;
  if (flags & MOE_WS_TRAINING) {
    if (encode_tmap_bf16(&p->tm_dye, p->dye, RP, p->d, 128) ||
        encode_tmap_bf16(&p->tm_dA, p->dA, RP, 2LL * p->I, 128) ||
        encode_tmap_bf16_mn(&p->tm_dye_mn, p->dye, RP, p->d, 2) ||
        encode_tmap_bf16_mn(&p->tm_dA_mn, p->dA, RP, 2LL * p->I, 2) ||
        encode_tmap_bf16_mn(&p->tm_hs_mn, p->hs, RP, p->I, p->bnw2 / 64) ||
        encode_tmap_bf16_mn(&p->tm_xe_mn, p->xe, RP, p->d, p->bnw13 / 64) ||
        encode_tmap_bf16(&p->tm_a, p->a, RP, 2LL * p->I, 128) ||
        encode_tmap_bf16(&p->tm_hs, p->hs, RP, p->I, 128) ||
        encode_tmap_bf16(&p->tm_dxe, p->dxe, RP, p->d, 128))
      return MOE_ERR_CUDA;
  }
  return reset_error_word(p->err);
}

int moe_forward(moe_plan* p, const void* x, const int32_t* ids, const float* scores,
                const void* w13, const void* w2, const uint8_t* w13_sf, const uint8_t* w2_sf,
                void* y, int save_for_backward, void* stream_v) {
  if (!p || !x || !ids || !scores || !w13 || !w2 || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w13) || !aligned16(w2) || !aligned16(y))
    return MOE_ERR_INVALID_ARG;
  if (!p->ws) return MOE_ERR_WORKSPACE;
  if (p->precision == MOE_PREC_NVFP4) return MOE_ERR_UNSUPPORTED;   // moe_forward_nvfp4
  const bool mx = p->precision == MOE_PREC_MXFP8;
  if (save_for_backward && !(p->ws_flags & MOE_WS_TRAINING)) return MOE_ERR_WORKSPACE;
  if (mx && (!w13_sf || !w2_sf || !aligned16(w13_sf) || !aligned16(w2_sf)))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream_v);
  if (mx) {
    if (w13 != p->w13q_cached) {
      if (encode_tmap_gate_up_blocks(&p->tm_w13q, w13, p->E, p->I, p->d)) return MOE_ERR_CUDA;
      p->w13q_cached = w13;
    }
    if (w2 != p->w2q_cached) {
      if (encode_tmap_u8(&p->tm_w2q, w2, (long long)p->E * p->d, p->I, p->bnmx_d))
        return MOE_ERR_CUDA;
      p->w2q_cached = w2;
    }
  } else if (refresh_weight_maps(p, w13, w2) != MOE_OK) {
    return MOE_ERR_CUDA;
  }

  mark(p, 0, 0, st);
  // a1-a3: dispatch
  RouteArgs ra{};                 // every pointer not set below stays NULL
  ra.ids = ids; ra.scores = scores;
  ra.T = p->T; ra.k = p->k; ra.E = p->E; ra.BM = p->gran; ra.nblk = p->nblk;
  ra.blockcounts = p->blockcounts; ra.counts = p->counts; ra.m_indptr = p->m_indptr;
  ra.off_pad = p->off_pad; ra.num_mtiles = p->num_mtiles; ra.tile_expert = p->tile_expert;
  ra.expert_order = p->expert_order; ra.num_nonempty = p->num_nonempty;
  ra.row_of = p->row_of; ra.token_of = p->token_of; ra.score_of = p->score_of; ra.err = p->err;
  ra.pair_list = p->pair_list; ra.left_list = p->left_list;
  ra.num_pairs = p->num_pairs; ra.num_left = p->num_left;
  cudaError_t e = launch_route(ra, st);
  if (e != cudaSuccess) return cuda_status(e);
  p->launches += 3;
  mark(p, 0, 1, st);
  if (mx) {
    if (p->wait_before_gather &&
        (e = cudaStreamWaitEvent(st, p->wait_before_gather, 0)) != cudaSuccess)
      return cuda_status(e);
    const int rc = forward_mxfp8(p, x, w13_sf, w2_sf, y, save_for_backward, st);
    p->saved = (rc == MOE_OK && save_for_backward) ? 1 : 0;
    return rc;
  }
  // a4: gather x rows into expert-major order
  if (p->wait_before_gather && (e = cudaStreamWaitEvent(st, p->wait_before_gather, 0)) != cudaSuccess)
    return cuda_status(e);
  e = launch_gather_rows(x, p->token_of, p->off_pad + p->E, p->d, p->xe, gather_grid(p), st);
  if (e != cudaSuccess) return cuda_status(e);
  p->launches += 1;
  mark(p, 0, 2, st);
  // a5: W13 GEMM + SwiGLU
  {
    GemmArgs g = rows_args(p);
    g.k_blocks = p->d / kBK;
    g.b_expert_rows = 2 * p->I;
    g.b_half_rows = p->I;
    g.n_tiles = p->I / (p->bn13 / 2);
    g.out0 = p->h; g.ld0 = p->I;
    g.out1 = p->a; g.ld1 = 2LL * p->I;
    g.save = save_for_backward ? 1 : 0;
    g.stall_mma = p->dbg_stall_w13;
    if (p->pair) {
      GemmArgs gp = g;
      gp.n_tiles = p->I / 128;
      gp.mtile_list = p->pair_list; gp.list_count = p->num_pairs;
      e = launch_gemm_pair(EPI_SWIGLU, false, p->tm_xe, p->tm_w13_p, p->tm_h, p->tm_a, gp,
                           p->num_sms, st);
      if (e != cudaSuccess) return cuda_status(e);
      p->launches += 1;
      g.mtile_list = p->left_list; g.list_count = p->num_left;   // odd last m tiles
    }
    e = launch_gemm(EPI_SWIGLU, p->bn13, false, false, p->tm_xe, p->tm_w13, p->tm_xe, p->tm_h,
                    p->tm_a, g, p->num_sms, st);
    if (e != cudaSuccess) return cuda_status(e);
    p->launches += 1;
    mark(p, 0, 3, st);
  }
  // a6: W2 GEMM x score
  {
    GemmArgs g = rows_args(p);
    g.k_blocks = p->I / kBK;
    g.b_expert_rows = p->d;
    g.n_tiles = p->d / p->bn2;
    g.out0 = p->ys; g.ld0 = p->d;
    g.row_scale = p->score_of;
    g.k_rotate = 1;   // measured faster here; slower on W13 and DGRAD-W2 (bf16)
    if (p->pair) {
      GemmArgs gp = g;
      gp.n_tiles = p->d / 256;
      gp.mtile_list = p->pair_list; gp.list_count = p->num_pairs;
      e = launch_gemm_pair(EPI_SCORE, false, p->tm_h, p->tm_w2_p, p->tm_ys, p->tm_ys, gp,
                           p->num_sms, st);
      if (e != cudaSuccess) return cuda_status(e);
      p->launches += 1;
      g.mtile_list = p->left_list; g.list_count = p->num_left;
    }
    e = launch_gemm(EPI_SCORE, p->bn2, false, false, p->tm_h, p->tm_w2, p->tm_h, p->tm_ys,
                    p->tm_ys, g, p->num_sms, st);
    if (e != cudaSuccess) return cuda_status(e);
    p->launches += 1;
    mark(p, 0, 4, st);
  }
  // a7: combine
  e = launch_combine(p->ys, p->row_of, p->T, p->k, p->d, y, nullptr, 0, nullptr, gather_grid(p), st);
  if (e != cudaSuccess) return cuda_status(e);
  p->launches += 1;
  mark(p, 0, 5, st);
  p->saved = save_for_backward ? 1 : 0;
  return MOE_OK;
}

int moe_backward(moe_plan* p, const void* dy, const void* w13, const void* w2, void* dx,
                 float* dw13, float* dw2, float* dscores, void* stream_v) {
  if (!p || !dy || !w13 || !w2 || !dx || !dw13 || !dw2 || !dscores) return MOE_ERR_INVALID_ARG;
  if (!aligned16(dy) || !aligned16(w13) || !aligned16(w2) || !aligned16(dx) || !aligned16(dw13) ||
      !aligned16(dw2))
    return MOE_ERR_INVALID_ARG;
  if (p->precision != MOE_PREC_BF16) return MOE_ERR_UNSUPPORTED;
  if (!p->ws || !(p->ws_flags & MOE_WS_TRAINING)) return MOE_ERR_WORKSPACE;
  if (!p->saved) return MOE_ERR_STATE;
  cudaStream_t st = static_cast<cudaStream_t>(stream_v);
  if (refresh_weight_maps(p, w13, w2) != MOE_OK) return MOE_ERR_CUDA;
  if (dw13 != p->dw13_cached) {
    if (encode_tmap_f32_out(&p->tm_dw13, dw13, (long long)p->E * 2 * p->I, p->d)) return MOE_ERR_CUDA;
    p->dw13_cached = dw13;
  }
  if (dw2 != p->dw2_cached) {
    if (encode_tmap_f32_out(&p->tm_dw2, dw2, (long long)p->E * p->d, p->I)) return MOE_ERR_CUDA;
    p->dw2_cached = dw2;
  }
  const int I = p->I, d = p->d;
  mark(p, 1, 0, st);
  // b1: gather dY rows
  cudaError_t e = launch_gather_rows(dy, p->token_of, p->off_pad + p->E, d, p->dye, gather_grid(p), st);
  if (e != cudaSuccess) return cuda_status(e);
  p->launches += 1;
  mark(p, 1, 1, st);
  // b2: g = dY_e . W2_e, SwiGLU backward, hs, score-grad partials
  {
    GemmArgs g = rows_args(p);
    g.k_blocks = d / kBK;
    g.b_expert_rows = d;
    g.n_tiles = I / p->bnd2;
    g.in1 = p->a; g.ldi1 = 2LL * I;
    g.out0 = p->dA; g.ld0 = 2LL * I;
    g.out1 = p->hs; g.ld1 = I;
    g.row_scale = p->score_of;
    g.pdscore = p->pdscore;
    // one CTA per tile (also with CTA pairs: this epilogue-bound GEMM measured no faster on pairs)
    e = launch_gemm(EPI_DGRAD2, p->bnd2, false, true, p->tm_dye, p->tm_w2_mn, p->tm_dye, p->tm_dA,
                    p->tm_hs, g, p->num_sms, st);
    if (e != cudaSuccess) return cuda_status(e);
    p->launches += 1;
    mark(p, 1, 2, st);
  }
  // With a split, the weight gradients (b5, b6) run on their own stream and
  // SMs from here on, beside b3 and b4.
  const bool split = p->wgrad_sms > 0 && p->wstream;
  const int rows_grid = split ? p->num_sms - p->wgrad_sms : p->num_sms;
  cudaStream_t wst = split ? p->wstream : st;
  if (split && ((e = cudaEventRecord(p->ev_wfork, st)) != cudaSuccess ||
                (e = cudaStreamWaitEvent(wst, p->ev_wfork, 0)) != cudaSuccess))
    return cuda_status(e);
  if (split) {
    e = launch_wgrad_bf16(p, wst, dw13, dw2, p->wgrad_sms);
    if (e != cudaSuccess) return cuda_status(e);
  }
  // b3: dX_e = dA . W13_e
  {
    GemmArgs g = rows_args(p);
    g.k_blocks = 2 * I / kBK;
    g.b_expert_rows = 2 * I;
    g.n_tiles = d / p->bn2;
    g.out0 = p->dxe; g.ld0 = d;
    if (p->pair) {
      GemmArgs gp = g;
      gp.n_tiles = d / 256;
      gp.mtile_list = p->pair_list; gp.list_count = p->num_pairs;
      e = launch_gemm_pair(EPI_STORE, true, p->tm_dA, p->tm_w13_mn_p, p->tm_dxe, p->tm_dxe, gp,
                           p->num_sms, st);
      if (e != cudaSuccess) return cuda_status(e);
      p->launches += 1;
      g.mtile_list = p->left_list; g.list_count = p->num_left;
    }
    e = launch_gemm(EPI_STORE, p->bn2, false, true, p->tm_dA, p->tm_w13_mn, p->tm_dA, p->tm_dxe,
                    p->tm_dxe, g, rows_grid, st);
    if (e != cudaSuccess) return cuda_status(e);
    p->launches += 1;
    mark(p, 1, 3, st);
  }
  // b4: combine dX and dscores
  e = launch_combine(p->dxe, p->row_of, p->T, p->k, d, dx, p->pdscore, 2 * (I / p->bnd2), dscores,
                     gather_grid(p), st);
  if (e != cudaSuccess) return cuda_status(e);
  p->launches += 1;
  mark(p, 1, 4, st);
  if (p->record_after_combine &&
      (e = cudaEventRecord(p->record_after_combine, st)) != cudaSuccess)
    return cuda_status(e);
  if (split) {
    // join: the caller's stream continues once the weight gradients are done
    if ((e = cudaEventRecord(p->ev_wjoin, wst)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(st, p->ev_wjoin, 0)) != cudaSuccess)
      return cuda_status(e);
    return MOE_OK;
  }
  e = launch_wgrad_bf16(p, st, dw13, dw2, p->num_sms);
  return e == cudaSuccess ? MOE_OK : cuda_status(e);
}

// MXFP8 backward ("What it is selling": MXFP8 E4M3 for DGRAD and WGRAD; the
// block-scaled GEMM takes both operands quantised along its K):
//   b1  gather dY rows and quantise them along d and along the rows (transposed), one pass
//   b2  DGRAD-W2 (block-scaled, W2^T prepared along d) + SwiGLU bwd -> dA, hs, dscore partials
//   b2' dA quantised along 2I and along the rows (one pass); hs along the rows
//   b3  DGRAD-W13 (block-scaled, W13^T prepared along 2I) -> dX_e
//   b4  combine dX and dscores
//   b5  WGRAD-W2  += (dY^T)_q . (hs^T)_q over each expert's rows
//   b6  WGRAD-W13 += (dA^T)_q . (x^T)_q  (x^T quantised by the saving forward)
int moe_backward_mxfp8(moe_plan* p, const void* dy, const uint8_t* w13t, const uint8_t* w13t_sf,
                       const uint8_t* w2t, const uint8_t* w2t_sf, void* dx, float* dw13,
                       float* dw2, float* dscores, void* stream_v) {
  if (!p || !dy || !w13t || !w13t_sf || !w2t || !w2t_sf || !dx || !dw13 || !dw2 || !dscores)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(dy) || !aligned16(w13t) || !aligned16(w2t) || !aligned16(w13t_sf) ||
      !aligned16(w2t_sf) || !aligned16(dx) || !aligned16(dw13) || !aligned16(dw2))
    return MOE_ERR_INVALID_ARG;
  if (p->precision != MOE_PREC_MXFP8) return MOE_ERR_UNSUPPORTED;
  if (!p->ws || !(p->ws_flags & MOE_WS_TRAINING)) return MOE_ERR_WORKSPACE;
  if (!p->saved) return MOE_ERR_STATE;
  cudaStream_t st = static_cast<cudaStream_t>(stream_v);
  const int I = p->I, d = p->d, E = p->E;
  const long long RP = p->RP;
  if (w13t != p->w13t_cached) {
    if (encode_tmap_u8(&p->tm_w13t, w13t, (long long)E * d, 2 * I, p->bnmx_d)) return MOE_ERR_CUDA;
    p->w13t_cached = w13t;
  }
  if (w2t != p->w2t_cached) {
    if (encode_tmap_u8(&p->tm_w2t, w2t, (long long)E * I, d, 128)) return MOE_ERR_CUDA;
    p->w2t_cached = w2t;
  }
  if (dw13 != p->dw13_cached) {
    if (encode_tmap_f32_out(&p->tm_dw13, dw13, (long long)E * 2 * I, d)) return MOE_ERR_CUDA;
    p->dw13_cached = dw13;
  }
  if (dw2 != p->dw2_cached) {
    if (encode_tmap_f32_out(&p->tm_dw2, dw2, (long long)E * d, I)) return MOE_ERR_CUDA;
    p->dw2_cached = dw2;
  }
  const int32_t* nrows = p->off_pad + E;
  mark(p, 1, 0, st);
  // b1
  cudaError_t e = launch_quant_two_way(dy, p->token_of, nrows, (int)RP, d, p->dyq, p->dysf,
                                       p->dyqT, p->dyqTsf, p->num_sms, st);
  if (e != cudaSuccess) return cuda_status(e);
  p->launches += 1;
  mark(p, 1, 1, st);
  // b2
  {
    GemmArgs g = rows_args(p);
    g.k_blocks = d / 128;
    g.b_expert_rows = I;
    g.n_tiles = I / 128;
    g.in1 = p->a; g.ldi1 = 2LL * I;
    g.row_scale = p->score_of;
    g.pdscore = p->pdscore;
    g.sfa = p->dysf; g.sfb = w2t_sf; g.sf_ngr = d / 128; g.b_blocks_per_expert = I / 128;
    // dA and hs leave quantised: dA along 2I (the DGRAD-W13 operand), dA and hs
    // along the rows (the WGRAD operands)
    g.q_row = p->dAq; g.sf_row = p->dAsf; g.sf_row_ngr = 2 * I / 128;
    g.qt_a = p->dAqT; g.sft_a = p->dAqTsf;
    g.qt_h = p->hsqT; g.sft_h = p->hsqTsf;
    g.qt_ld = RP;
    // (the output maps are unused: this epilogue stores without TMA)
    e = launch_gemm(EPI_DGRAD2, 128, false, false, p->tm_dyq, p->tm_w2t, p->tm_dyq, p->tm_dyq,
                    p->tm_dyq, g, p->num_sms, st, true);
    if (e != cudaSuccess) return cuda_status(e);
    p->launches += 1;
  }
  mark(p, 1, 2, st);
  // With a split, the weight gradients (b5, b6) run on their own stream and
  // SMs from here on, beside b3 and b4.
  const bool split = p->wgrad_sms > 0 && p->wstream;
  const int rows_grid = split ? p->num_sms - p->wgrad_sms : p->num_sms;
  cudaStream_t wst = split ? p->wstream : st;
  if (split && ((e = cudaEventRecord(p->ev_wfork, st)) != cudaSuccess ||
                (e = cudaStreamWaitEvent(wst, p->ev_wfork, 0)) != cudaSuccess))
    return cuda_status(e);
  if (split && (e = launch_wgrad_mx(p, wst, dw13, dw2, p->wgrad_sms)) != cudaSuccess)
    return cuda_status(e);
  // b3
  {
    GemmArgs g = rows_args(p);
    g.k_blocks = 2 * I / 128;
    g.b_expert_rows = d;
    g.n_tiles = d / p->bnmx_d;
    g.out0 = p->dxe; g.ld0 = d;
    g.sfa = p->dAsf; g.sfb = w13t_sf; g.sf_ngr = 2 * I / 128; g.b_blocks_per_expert = d / 128;
    g.k_rotate = 1;
    e = launch_gemm(EPI_STORE, p->bnmx_d, false, false, p->tm_dAq, p->tm_w13t, p->tm_dAq,
                    p->tm_dxe, p->tm_dxe, g, rows_grid, st, true);
    if (e != cudaSuccess) return cuda_status(e);
    p->launches += 1;
    mark(p, 1, 3, st);
  }
  // b4
  e = launch_combine(p->dxe, p->row_of, p->T, p->k, d, dx, p->pdscore, 2 * (I / p->bnd2), dscores,
                     gather_grid(p), st);
  if (e != cudaSuccess) return cuda_status(e);
  p->launches += 1;
  mark(p, 1, 4, st);
  if (split) {
    if ((e = cudaEventRecord(p->ev_wjoin, wst)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(st, p->ev_wjoin, 0)) != cudaSuccess)
      return cuda_status(e);
    return MOE_OK;
  }
  e = launch_wgrad_mx(p, st, dw13, dw2, p->num_sms);
  return e == cudaSuccess ? MOE_OK : cuda_status(e);
}

// Forward over a caller-provided expert-major layout (nvfp4moe README, "MoE
// layer": the run_routed entry for callers that route on their own): check the layout
// and list its m tiles -> W13 GEMM + SwiGLU -> W2 GEMM (x score_of) into the
// caller's ys -> optionally combine into y.  Dispatch and gather are skipped.
int moe_forward_routed(moe_plan* p, const void* x_e, long long rows, const int32_t* m_indptr,
                       const int32_t* off_pad, const float* score_of, const void* w13,
                       const void* w2, void* ys, const int32_t* row_of, void* y, void* stream_v) {
  if (!p || !x_e || !m_indptr || !off_pad || !w13 || !w2 || !ys) return MOE_ERR_INVALID_ARG;
  if ((row_of == nullptr) != (y == nullptr)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x_e) || !aligned16(w13) || !aligned16(w2) || !aligned16(ys) ||
      (y && !aligned16(y)))
    return MOE_ERR_INVALID_ARG;
  if (rows < 0 || rows > p->RP) return MOE_ERR_INVALID_ARG;
  if (p->precision != MOE_PREC_BF16) return MOE_ERR_UNSUPPORTED;
  if (!p->ws) return MOE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream_v);
  if (rows == 0) {
    // no routed rows: y is all zeros
    if (y) return cuda_status(cudaMemsetAsync(y, 0, 2ull * p->T * p->d, st));
    return MOE_OK;
  }
  if (refresh_weight_maps(p, w13, w2) != MOE_OK) return MOE_ERR_CUDA;
  if (x_e != p->rx_cached || rows != p->rx_rows) {
    if (encode_tmap_bf16(&p->tm_rx, x_e, rows, p->d, 128)) return MOE_ERR_CUDA;
    p->rx_cached = x_e;
    p->rx_rows = rows;
  }
  if (ys != p->rys_cached || rows != p->rys_rows) {
    if (encode_tmap_bf16(&p->tm_rys, ys, rows, p->d, 128)) return MOE_ERR_CUDA;
    p->rys_cached = ys;
    p->rys_rows = rows;
  }
  RoutedArgs ra{};
  ra.m_indptr = m_indptr;
  ra.off_pad = off_pad;
  ra.E = p->E;
  ra.rows = rows;
  ra.row_of_in = row_of;
  ra.Tk = row_of ? p->R : 0;
  ra.row_of_out = p->row_of;
  ra.tile_expert = p->tile_expert;
  ra.mtile_list = p->routed_list;
  ra.list_count = p->routed_count;
  ra.err = p->err;
  const int pgrid = row_of ? (p->R + 4095) / 4096 : 1;
  cudaError_t e = launch_routed_prepare(ra, pgrid < 1 ? 1 : pgrid, st);
  if (e != cudaSuccess) return cuda_status(e);
  p->launches += 1;
  {
    GemmArgs g = rows_args(p);
    g.mtile_list = p->routed_list;
    g.list_count = p->routed_count;
    g.k_blocks = p->d / kBK;
    g.b_expert_rows = 2 * p->I;
    g.b_half_rows = p->I;
    g.n_tiles = p->I / (p->bn13 / 2);
    g.out0 = p->h; g.ld0 = p->I;
    g.ld1 = 2LL * p->I;
    g.save = 0;
    e = launch_gemm(EPI_SWIGLU, p->bn13, false, false, p->tm_rx, p->tm_w13, p->tm_rx, p->tm_h,
                    p->tm_h, g, p->num_sms, st);
    if (e != cudaSuccess) return cuda_status(e);
    p->launches += 1;
  }
  {
    GemmArgs g = rows_args(p);
    g.mtile_list = p->routed_list;
    g.list_count = p->routed_count;
    g.k_blocks = p->I / kBK;
    g.b_expert_rows = p->d;
    g.n_tiles = p->d / p->bn2;
    g.out0 = ys; g.ld0 = p->d;
    g.row_scale = score_of;           // NULL: no routing score
    g.k_rotate = 1;
    e = launch_gemm(EPI_SCORE, p->bn2, false, false, p->tm_h, p->tm_w2, p->tm_h, p->tm_rys,
                    p->tm_rys, g, p->num_sms, st);
    if (e != cudaSuccess) return cuda_status(e);
    p->launches += 1;
  }
  if (y) {
    e = launch_combine(ys, p->row_of, p->T, p->k, p->d, y, nullptr, 0, nullptr, gather_grid(p), st);
    if (e != cudaSuccess) return cuda_status(e);
    p->launches += 1;
  }
  p->saved = 0;
  return MOE_OK;
}

int moe_plan_set_activation_scales(moe_plan* p, float x_scale, float h_scale) {
  if (!p || !(x_scale > 0.f) || !(h_scale > 0.f) || !std::isfinite(x_scale) ||
      !std::isfinite(h_scale))
    return MOE_ERR_INVALID_ARG;
  if (p->precision != MOE_PREC_NVFP4) return MOE_ERR_UNSUPPORTED;
  p->nv_x_scale = x_scale;
  p->nv_h_scale = h_scale;
  return MOE_OK;
}

// NVFP4 inference forward ("Dist-MoE" note, "What it is selling": NVFP4 is
// inference-only with prepared weights; nvfp4moe README, "MoE layer": dispatch,
// BF16 activation quantisation, FC1 + gated activation + NVFP4 requantisation,
// FC2, probability weighting, deterministic combine):
//   route -> gather x rows + quantise (static input scale) -> NVFP4 W13 GEMM +
//   SwiGLU + h quantisation (static hidden scale) -> NVFP4 W2 GEMM x score ->
//   combine
int moe_forward_nvfp4(moe_plan* p, const void* x, const int32_t* ids, const float* scores,
                      const uint8_t* w13q, const uint8_t* w13_sf, const float* w13_scale,
                      const uint8_t* w2q, const uint8_t* w2_sf, const float* w2_scale, void* y,
                      void* stream_v) {
  if (!p || !x || !ids || !scores || !w13q || !w13_sf || !w13_scale || !w2q || !w2_sf ||
      !w2_scale || !y)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w13q) || !aligned16(w2q) || !aligned16(w13_sf) ||
      !aligned16(w2_sf) || !aligned16(y))
    return MOE_ERR_INVALID_ARG;
  if (p->precision != MOE_PREC_NVFP4) return MOE_ERR_UNSUPPORTED;
  if (!p->ws) return MOE_ERR_WORKSPACE;
  if (!(p->nv_x_scale > 0.f) || !(p->nv_h_scale > 0.f)) return MOE_ERR_STATE;
  cudaStream_t st = static_cast<cudaStream_t>(stream_v);
  const int d = p->d, I = p->I, E = p->E;
  if (w13q != p->w13nv_cached) {
    // (K bytes, 64, gate/up, I/64, E): two 64-row blocks of gate then up rows
    if (encode_tmap_gate_up_blocks(&p->tm_w13nv, w13q, E, I, d / 2)) return MOE_ERR_CUDA;
    p->w13nv_cached = w13q;
  }
  if (w2q != p->w2nv_cached) {
    if (encode_tmap_u8(&p->tm_w2nv, w2q, (long long)E * d, I / 2, 256)) return MOE_ERR_CUDA;
    p->w2nv_cached = w2q;
  }
  mark(p, 0, 0, st);
  RouteArgs ra{};
  ra.ids = ids; ra.scores = scores;
  ra.T = p->T; ra.k = p->k; ra.E = E; ra.BM = p->gran; ra.nblk = p->nblk;
  ra.blockcounts = p->blockcounts; ra.counts = p->counts; ra.m_indptr = p->m_indptr;
  ra.off_pad = p->off_pad; ra.num_mtiles = p->num_mtiles; ra.tile_expert = p->tile_expert;
  ra.expert_order = p->expert_order; ra.num_nonempty = p->num_nonempty;
  ra.row_of = p->row_of; ra.token_of = p->token_of; ra.score_of = p->score_of; ra.err = p->err;
  cudaError_t e = launch_route(ra, st);
  if (e != cudaSuccess) return cuda_status(e);
  p->launches += 3;
  mark(p, 0, 1, st);
  // gather + quantise along d with the static input scale (encode scale 1/x_scale)
  e = launch_gather_quant_nvfp4(x, p->token_of, p->off_pad + E, d, 1.0f / p->nv_x_scale, p->xq,
                                p->xsf, gather_grid(p), st);
  if (e != cudaSuccess) return cuda_status(e);
  p->launches += 1;
  mark(p, 0, 2, st);
  {
    GemmArgs g = rows_args(p);
    g.k_blocks = d / 256;
    g.b_expert_rows = 2 * I;
    g.b_half_rows = I;
    g.n_tiles = I / 128;
    g.ld0 = I / 2;                       // row stride of hq (bytes)
    g.sfa = p->xsf; g.sfb = w13_sf; g.sf_ngr = d / 64; g.b_blocks_per_expert = I / 64;
    g.hq = p->hq; g.hsf = p->hsf; g.hsf_ngr = I / 64;
    g.w_scale = w13_scale; g.act_scale = p->nv_x_scale; g.h_enc = 1.0f / p->nv_h_scale;
    g.k_rotate = 1;
    g.stall_mma = p->dbg_stall_w13;
    e = launch_gemm_nvfp4(EPI_SWIGLU, p->tm_xq, p->tm_w13nv, p->tm_ys, g, p->num_sms, st);
    if (e != cudaSuccess) return cuda_status(e);
    p->launches += 1;
    mark(p, 0, 3, st);
  }
  {
    GemmArgs g = rows_args(p);
    g.k_blocks = I / 256;
    g.b_expert_rows = d;
    g.n_tiles = d / 256;
    g.out0 = p->ys; g.ld0 = d;
    g.row_scale = p->score_of;
    g.sfa = p->hsf; g.sfb = w2_sf; g.sf_ngr = I / 64; g.b_blocks_per_expert = d / 128;
    g.w_scale = w2_scale; g.act_scale = p->nv_h_scale;
    g.k_rotate = 1;
    e = launch_gemm_nvfp4(EPI_SCORE, p->tm_hq, p->tm_w2nv, p->tm_ys, g, p->num_sms, st);
    if (e != cudaSuccess) return cuda_status(e);
    p->launches += 1;
    mark(p, 0, 4, st);
  }
  e = launch_combine(p->ys, p->row_of, p->T, p->k, d, y, nullptr, 0, nullptr, gather_grid(p), st);
  if (e != cudaSuccess) return cuda_status(e);
  p->launches += 1;
  mark(p, 0, 5, st);
  p->saved = 0;
  return MOE_OK;
}

int moe_step_host(moe_plan* p, const void* x_host, const int32_t* ids_host,
                  const float* scores_host, const void* dy_host, const void* w13, const void* w2,
                  float* dw13, float* dw2, void* y_host, void* dx_host, float* dscores_host,
                  void* stream_v) {
  if (!p || !x_host || !ids_host || !scores_host || !y_host) return MOE_ERR_INVALID_ARG;
  if (!p->ws || !(p->ws_flags & MOE_WS_HOST_STAGING)) return MOE_ERR_WORKSPACE;
  const bool train = dy_host != nullptr;
  if (train && (!(p->ws_flags & MOE_WS_TRAINING) || !dx_host || !dscores_host))
    return train && !(p->ws_flags & MOE_WS_TRAINING) ? MOE_ERR_WORKSPACE : MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream_v);
  cudaStream_t sd = p->side;
  const size_t xb = 2ull * p->T * p->d, sb = 4ull * p->T * p->k;
  cudaError_t e;
  // Copies overlap compute on a plan-owned side stream that joins `stream` at
  // the end of the step: x uploads during dispatch, dY during the forward; y
  // downloads during the backward, dx and dscores during the weight gradients.
  // The side stream forks from `stream` unless the previous step on this plan
  // was a training step: that step's last side-stream copies (dx, dscores)
  // waited for its dX combine, which came after every read of the staged x and
  // dY, so this step's uploads may start while its weight gradients still run.
  p->prev_step_train = p->prev_step_train && train;
  if (!p->prev_step_train && ((e = cudaEventRecord(p->ev_fork, st)) != cudaSuccess ||
                              (e = cudaStreamWaitEvent(sd, p->ev_fork, 0)) != cudaSuccess))
    return cuda_status(e);
  p->prev_step_train = 0;            // set again only when this step is fully enqueued
  if ((e = cudaMemcpyAsync(p->st_x, x_host, xb, cudaMemcpyHostToDevice, sd)) != cudaSuccess ||
      (e = cudaEventRecord(p->ev_x, sd)) != cudaSuccess)
    return cuda_status(e);
  if (train && ((e = cudaMemcpyAsync(p->st_dy, dy_host, xb, cudaMemcpyHostToDevice, sd)) !=
                    cudaSuccess ||
                (e = cudaEventRecord(p->ev_dy, sd)) != cudaSuccess))
    return cuda_status(e);
  if ((e = cudaMemcpyAsync(p->st_ids, ids_host, sb, cudaMemcpyHostToDevice, st)) != cudaSuccess ||
      (e = cudaMemcpyAsync(p->st_scores, scores_host, sb, cudaMemcpyHostToDevice, st)) != cudaSuccess)
    return cuda_status(e);
  p->wait_before_gather = p->ev_x;
  int rc = moe_forward(p, p->st_x, p->st_ids, p->st_scores, w13, w2, nullptr, nullptr, p->st_y,
                       train ? 1 : 0, stream_v);
  p->wait_before_gather = nullptr;
  if (rc != MOE_OK) return rc;
  if (!train) {
    if ((e = cudaMemcpyAsync(y_host, p->st_y, xb, cudaMemcpyDeviceToHost, st)) != cudaSuccess)
      return cuda_status(e);
    return MOE_OK;
  }
  if ((e = cudaEventRecord(p->ev_y, st)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(sd, p->ev_y, 0)) != cudaSuccess ||
      (e = cudaMemcpyAsync(y_host, p->st_y, xb, cudaMemcpyDeviceToHost, sd)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(st, p->ev_dy, 0)) != cudaSuccess)
    return cuda_status(e);
  p->record_after_combine = p->ev_comb;
  rc = moe_backward(p, p->st_dy, w13, w2, p->st_dx, dw13, dw2, p->st_dscores, stream_v);
  p->record_after_combine = nullptr;
  if (rc != MOE_OK) return rc;
  if ((e = cudaStreamWaitEvent(sd, p->ev_comb, 0)) != cudaSuccess ||
      (e = cudaMemcpyAsync(dx_host, p->st_dx, xb, cudaMemcpyDeviceToHost, sd)) != cudaSuccess ||
      (e = cudaMemcpyAsync(dscores_host, p->st_dscores, sb, cudaMemcpyDeviceToHost, sd)) !=
          cudaSuccess ||
      (e = cudaEventRecord(p->ev_dxdone, sd)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(st, p->ev_dxdone, 0)) != cudaSuccess)
    return cuda_status(e);
  p->prev_step_train = 1;
  return MOE_OK;
}

int moe_quantize_mxfp8(const void* in, long rows, int K, uint8_t* codes, uint8_t* scales,
                       void* stream) {
  if (!in || !codes || !scales || rows < 0 || K <= 0 || K % 32 || !aligned16(in) ||
      !aligned16(codes))
    return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  return cuda_status(launch_quant_mxfp8(in, rows, K, codes, scales, static_cast<cudaStream_t>(stream)));
}

int moe_plan_set_backward_split(moe_plan* p, int wgrad_sms) {
  if (!p || wgrad_sms < 0 || wgrad_sms >= p->num_sms) return MOE_ERR_INVALID_ARG;
  if (wgrad_sms > 0 && !p->wstream) {
    if (cudaStreamCreateWithFlags(&p->wstream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&p->ev_wfork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&p->ev_wjoin, cudaEventDisableTiming) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  p->wgrad_sms = wgrad_sms;
  return MOE_OK;
}

int moe_plan_set_wgrad_interleave(moe_plan* p, long long min_rows) {
  if (!p || min_rows < 0 || min_rows > (1LL << 30)) return MOE_ERR_INVALID_ARG;
  p->wgrad_long_rows = min_rows;
  return MOE_OK;
}

int moe_plan_num_sms(const moe_plan* p) { return p ? p->num_sms : 0; }

int moe_plan_set_debug(moe_plan* p, long long wait_limit_ns, int stall_w13) {
  if (!p || wait_limit_ns < 0) return MOE_ERR_INVALID_ARG;
  p->dbg_wait_limit_ns = wait_limit_ns;
  p->dbg_stall_w13 = stall_w13 ? 1 : 0;
  return MOE_OK;
}

size_t moe_nvfp4_weight_bytes(int d, int I, int E, int which) {
  if (d <= 0 || I <= 0 || E <= 0 || d % 256 || I % 256) return 0;
  if (which == 0) return (size_t)E * 2 * I * d / 2;                                  // W13 codes
  if (which == 1) return (size_t)nv_sf_bytes((long long)E * (I / 64) * 128, d);      // W13 scales
  if (which == 2) return (size_t)E * d * I / 2;                                      // W2 codes
  if (which == 3) return (size_t)nv_sf_bytes((long long)E * d, I);                   // W2 scales
  return 0;
}

int moe_prepare_weights_nvfp4(const void* w13, const void* w2, int d, int I, int E,
                              uint8_t* w13_codes, uint8_t* w13_sf, float* w13_scale,
                              uint8_t* w2_codes, uint8_t* w2_sf, float* w2_scale, void* stream) {
  if (!w13 || !w2 || !w13_codes || !w13_sf || !w13_scale || !w2_codes || !w2_sf || !w2_scale)
    return MOE_ERR_INVALID_ARG;
  if (d <= 0 || I <= 0 || E <= 0 || d % 256 || I % 256) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w13) || !aligned16(w2) || !aligned16(w13_codes) || !aligned16(w2_codes) ||
      (reinterpret_cast<uintptr_t>(w13_sf) & 3) || (reinterpret_cast<uintptr_t>(w2_sf) & 3))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_prepare_nvfp4(w13, E, 2LL * I, d, I, w13_codes, w13_sf, w13_scale, st);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(launch_prepare_nvfp4(w2, E, (long long)d, I, 0, w2_codes, w2_sf, w2_scale, st));
}

int moe_amax_bf16(const void* in, long long n, float* amax, void* stream) {
  if (!in || !amax || n < 0 || !aligned16(in)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_amax_bf16(in, 1, n, reinterpret_cast<unsigned int*>(amax),
                                      static_cast<cudaStream_t>(stream)));
}

size_t moe_mxfp8_weight_scale_bytes(int d, int I, int E, int which) {
  if (d <= 0 || I <= 0 || E <= 0 || d % 128 || I % 128) return 0;
  if (which == 0) return (size_t)mx_sf_bytes((long long)E * (I / 64) * 128, d);   // W13
  if (which == 1) return (size_t)mx_sf_bytes((long long)E * d, I);                // W2
  if (which == 2) return (size_t)mx_sf_bytes((long long)E * d, 2 * I);            // W13^T
  if (which == 3) return (size_t)mx_sf_bytes((long long)E * I, d);                // W2^T
  return 0;
}

int moe_prepare_weights_mxfp8_backward(const void* w13, const void* w2, int d, int I, int E,
                                       uint8_t* w13t_codes, uint8_t* w13t_scales,
                                       uint8_t* w2t_codes, uint8_t* w2t_scales, void* stream) {
  if (!w13 || !w2 || !w13t_codes || !w13t_scales || !w2t_codes || !w2t_scales)
    return MOE_ERR_INVALID_ARG;
  if (d <= 0 || I <= 0 || E <= 0 || d % 128 || I % 128) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w13) || !aligned16(w2) || !aligned16(w13t_codes) || !aligned16(w2t_codes))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // W13[e] [2I, d] -> [d, 2I] along 2I;  W2[e] [d, I] -> [I, d] along d
  cudaError_t e = launch_quant_rows_t(w13, nullptr, nullptr, E, 2 * I, d, w13t_codes, w13t_scales,
                                      st);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(launch_quant_rows_t(w2, nullptr, nullptr, E, d, I, w2t_codes, w2t_scales, st));
}

int moe_prepare_weights_mxfp8(const void* w13, const void* w2, int d, int I, int E,
                              uint8_t* w13_codes, uint8_t* w13_scales, uint8_t* w2_codes,
                              uint8_t* w2_scales, void* stream) {
  if (!w13 || !w2 || !w13_codes || !w13_scales || !w2_codes || !w2_scales) return MOE_ERR_INVALID_ARG;
  if (d <= 0 || I <= 0 || E <= 0 || d % 128 || I % 128) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w13) || !aligned16(w2) || !aligned16(w13_codes) || !aligned16(w2_codes))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_quant_tiled(w13, (long long)E * 2 * I, d, I, w13_codes, w13_scales, st);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(launch_quant_tiled(w2, (long long)E * d, I, 0, w2_codes, w2_scales, st));
}

int moe_plan_set_timing_events(moe_plan* p, int which, void* const* events, int n) {
  if (!p || which < 0 || which > 1 || n < 0) return MOE_ERR_INVALID_ARG;
  if (n > 0 && events && n < (which == 0 ? 6 : 7)) return MOE_ERR_INVALID_ARG;
  p->ev[which] = n > 0 ? events : nullptr;
  p->nev[which] = events ? n : 0;
  return MOE_OK;
}

long long moe_plan_launch_count(const moe_plan* p) { return p ? p->launches : 0; }

int moe_plan_check(moe_plan* p, long long* detail) {
  if (!p || !p->ws) return MOE_ERR_INVALID_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_status(e);
  DevError h;
  e = cudaMemcpy(&h, p->err, sizeof(h), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_status(e);
  int rc = reset_error_word(p->err);
  if (rc != MOE_OK) return rc;
  if (detail)
    *detail = (h.code == MOE_ERR_BAD_IDS || h.code == MOE_ERR_INVALID_ARG) ? (long long)h.first_bad
                                                                           : (long long)h.where;
  return h.code;
}

int moe_plan_buffer(const moe_plan* p, int which, void** ptr, size_t* bytes) {
  if (!p || !p->ws || !ptr) return MOE_ERR_INVALID_ARG;
  const size_t RP = p->RP, d = p->d, I = p->I, E = p->E;
  const bool nvp = p->precision == MOE_PREC_NVFP4;
  void* q = nullptr;
  size_t b = 0;
  switch (which) {
    case MOE_BUF_M_INDPTR: q = p->m_indptr; b = 4 * (E + 1); break;
    case MOE_BUF_OFF_PAD: q = p->off_pad; b = 4 * (E + 1); break;
    case MOE_BUF_ROW_OF: q = p->row_of; b = 4 * (size_t)p->R; break;
    case MOE_BUF_TOKEN_OF: q = p->token_of; b = 4 * RP; break;
    case MOE_BUF_SCORE_OF: q = p->score_of; b = 4 * RP; break;
    case MOE_BUF_XE: q = p->xe; b = 2 * RP * d; break;
    case MOE_BUF_A: q = p->a; b = 2 * RP * 2 * I; break;
    case MOE_BUF_H: q = p->h; b = 2 * RP * I; break;
    case MOE_BUF_YS: q = p->ys; b = 2 * RP * d; break;
    case MOE_BUF_DYE: q = p->dye; b = 2 * RP * d; break;
    case MOE_BUF_DA: q = p->dA; b = 2 * RP * 2 * I; break;
    case MOE_BUF_HS: q = p->hs; b = 2 * RP * I; break;
    case MOE_BUF_DXE: q = p->dxe; b = 2 * RP * d; break;
    case MOE_BUF_XQ: q = p->xq; b = nvp ? RP * d / 2 : RP * d; break;
    case MOE_BUF_XSF:
      q = p->xsf;
      b = (size_t)(nvp ? nv_sf_bytes((long long)RP, (int)d) : mx_sf_bytes((long long)RP, (int)d));
      break;
    case MOE_BUF_HQ: q = p->hq; b = nvp ? RP * I / 2 : RP * I; break;
    case MOE_BUF_HSF:
      q = p->hsf;
      b = (size_t)(nvp ? nv_sf_bytes((long long)RP, (int)I) : mx_sf_bytes((long long)RP, (int)I));
      break;
    case MOE_BUF_XQT: q = p->xqT; b = (size_t)d * RP; break;
    case MOE_BUF_XQTSF: q = p->xqTsf; b = (size_t)mx_sf_bytes((long long)d, (int)RP); break;
    case MOE_BUF_DAQ: q = p->dAq; b = RP * 2 * I; break;
    case MOE_BUF_DASF: q = p->dAsf; b = (size_t)mx_sf_bytes((long long)RP, (int)(2 * I)); break;
    case MOE_BUF_DAQT: q = p->dAqT; b = 2 * I * RP; break;
    case MOE_BUF_DAQTSF: q = p->dAqTsf; b = (size_t)mx_sf_bytes((long long)(2 * I), (int)RP); break;
    case MOE_BUF_HSQT: q = p->hsqT; b = I * RP; break;
    case MOE_BUF_HSQTSF: q = p->hsqTsf; b = (size_t)mx_sf_bytes((long long)I, (int)RP); break;
    default: return MOE_ERR_INVALID_ARG;
  }
  if (!q) return MOE_ERR_WORKSPACE;
  *ptr = q;
  if (bytes) *bytes = b;
  return MOE_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// dense GEMM entry point (tests): runs the grouped kernels with one "expert"

namespace {

__global__ void k_dense_meta(int* s, int mtiles, int K) {
  // s[0] num_mtiles, s[1] num_nonempty, s[2..3] off_pad, s[4] expert_order
  s[0] = mtiles;
  s[1] = 1;
  s[2] = 0;
  s[3] = K;
  s[4] = 0;
}

}  // namespace

extern "C" size_t moe_gemm_scratch_bytes(int M, int K) {
  (void)M;
  (void)K;
  return 256;
}

extern "C" int moe_gemm_bf16(int mode, const void* A, const void* B, void* C, int M, int N, int K,
                             void* scratch, void* stream_v) {
  if (!A || !B || !C || !scratch || M <= 0 || N <= 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (M % 128 || N % 64 || K % 64 || (mode == 2 && K % 128)) return MOE_ERR_INVALID_ARG;
  if ((mode == 3 || mode == 4) && (M % 256 || N % 256)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream_v);
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int* s = static_cast<int*>(scratch);
  k_dense_meta<<<1, 1, 0, st>>>(s, M / 128, K);
  CUtensorMap ta, tb, tc;
  GemmArgs g;
  memset(&g, 0, sizeof(g));
  const int bn = pick_bn_n(N);
  g.n_tiles = N / bn;
  g.out0 = C;
  g.ld0 = N;
  cudaError_t e;
  if (mode == 0 || mode == 1) {
    if (encode_tmap_bf16(&ta, A, M, K, 128)) return MOE_ERR_CUDA;
    if (mode == 0 ? encode_tmap_bf16(&tb, B, N, K, bn) : encode_tmap_bf16_mn(&tb, B, K, N, bn / 64))
      return MOE_ERR_CUDA;
    g.wgrad = 0;
    g.num_mtiles = s;
    g.tile_expert = nullptr;
    g.k_blocks = K / kBK;
    g.b_expert_rows = mode == 0 ? N : K;
    if (encode_tmap_bf16(&tc, C, M, N, 128)) return MOE_ERR_CUDA;
    e = launch_gemm(EPI_STORE, bn, false, mode == 1, ta, tb, ta, tc, tc, g, sms, st);
  } else if (mode == 3 || mode == 4) {
    // the same products on CTA pairs (256 x 256 tiles)
    if (encode_tmap_bf16(&ta, A, M, K, 128)) return MOE_ERR_CUDA;
    if (mode == 3 ? encode_tmap_bf16(&tb, B, N, K, 128) : encode_tmap_bf16_mn(&tb, B, K, N, 2))
      return MOE_ERR_CUDA;
    g.wgrad = 0;
    g.num_mtiles = s;
    g.tile_expert = nullptr;          // a single "expert"
    g.k_blocks = K / kBK;
    g.b_expert_rows = mode == 3 ? N : K;
    g.n_tiles = N / 256;
    if (encode_tmap_bf16(&tc, C, M, N, 128)) return MOE_ERR_CUDA;
    e = launch_gemm_pair(EPI_STORE, mode == 4, ta, tb, tc, tc, g, sms, st);
  } else if (mode == 2) {
    if (encode_tmap_bf16_mn(&ta, A, K, M, 2) || encode_tmap_bf16_mn(&tb, B, K, N, bn / 64) ||
        encode_tmap_f32_out(&tc, C, M, N))
      return MOE_ERR_CUDA;
    g.wgrad = 1;
    g.num_nonempty = s + 1;
    g.off_pad = s + 2;
    g.expert_order = s + 4;
    g.m_tiles = M / kBM;
    g.out_expert_stride = 0;
    e = launch_gemm(EPI_WGRAD, bn, true, true, ta, tb, tc, tc, tc, g, sms, st);
  } else {
    return MOE_ERR_INVALID_ARG;
  }
  return cuda_status(e);
}
