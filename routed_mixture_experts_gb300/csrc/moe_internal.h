// moe_internal.h -- host-side declarations shared by the library's translation
// units (kernel launchers and their argument blocks).  Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <atomic>
#include <utility>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

// Launch with programmatic stream serialization (see pdl_wait / pdl_trigger in
// moe_device.cuh): the kernel may be scheduled while the previous kernel of the
// stream finishes, and waits for it in pdl_wait().
// Opt `kernel` in to `bytes` of dynamic shared memory on the current device.
// The attribute belongs to the kernel on one device, so it is set once per
// device: `done` holds one bit per device (devices 64 and up set it every time).
template <typename... KArgs>
inline cudaError_t smem_optin_once(void (*kernel)(KArgs...), int bytes,
                                   std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev >= 0 && dev < 64 ? 1ull << dev : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct DevError;

constexpr int kBM = 128;  // rows per GEMM tile = padding granule of an expert segment
constexpr int kBK = 64;   // K per pipeline stage (one 128-byte swizzle atom of bf16)

// Epilogue kinds of the grouped GEMM.
enum Epi : int {
  EPI_SWIGLU = 0,  // W13 FPROP: a = bf16(acc) (saved when training), h = bf16(swiglu(a))
  EPI_SCORE = 1,   // W2 FPROP: ys = bf16(score * acc)
  EPI_DGRAD2 = 2,  // g = dY_e . W2_e: dscore partials, SwiGLU backward -> dA, hs = bf16(s*h)
  EPI_STORE = 3,   // plain bf16 store (DGRAD through W13)
  EPI_WGRAD = 4,   // fp32 read-modify-write accumulate (weight gradients)
};

// Arguments of one grouped-GEMM launch.  Two tile spaces:
//  rows mode  (wgrad == 0): output rows are routed rows; m tile mt covers padded rows
//             [mt*128, mt*128+128) of expert tile_expert[mt]; K loop over k_blocks.
//  wgrad mode (wgrad == 1): output is a per-expert weight gradient [M, N]; the K
//             loop runs over the expert's padded row segment [off_pad[e], off_pad[e+1]).
struct GemmArgs {
  int wgrad;
  // rows mode
  const int* num_mtiles;     // device scalar
  const int* tile_expert;    // device [max m tiles]; nullptr: every tile is expert 0
  int k_blocks;
  int b_expert_rows;         // rows of B's 2-D tensor map per expert
  int b_half_rows;           // EPI_SWIGLU: row offset of the up half (I)
  // wgrad mode
  const int* mtile_list;     // row mode: the m tiles to run (NULL: all, 0..num_mtiles-1);
                             // pair kernel: first m tile of each pair (NULL: 2q)
  const int* list_count;     // device count of mtile_list entries
  const int* off_pad;        // device [E+1]
  const int* expert_order;   // device [E]: experts with rows first, longest first
  const int* num_nonempty;   // device scalar
  int m_tiles;               // M / 128
  long long out_expert_stride;
  // both
  int n_tiles;               // N / BN
  // epilogue operands
  void* out0;  long long ld0;
  void* out1;  long long ld1;
  const void* in1; long long ldi1;   // EPI_DGRAD2: a
  const float* row_scale;    // score of each padded row
  float* pdscore;            // EPI_DGRAD2: [rows, 2*n_tiles] (n tile, column half)
  float clamp;               // SwiGLU limit (0 = plain)
  int I;                     // column offset of the up half in a / dA
  int save;                  // EPI_SWIGLU: store a
  int k_rotate;              // rows mode: start each tile's K loop at an offset of its own
                             // (m and n tile), so tiles sharing an operand tile read
                             // different K chunks at a time (changes the summation order)
  int wgrad_kstep;           // wgrad mode: rows per K stage (0: 64; MXFP8: 128)
  int wgrad_long_kb;         // wgrad mode: tiles of more K stages are interleaved with
                             // the shorter ones (gemm::SegIter); 0: plain order
  // MXFP8 (block-scaled) operands: tiled E8M0 scales (see mx_sf_offset)
  const uint8_t* sfa;        // scales of A, row blocks of 128 padded rows
  const uint8_t* sfb;        // scales of B, row block = e * b_blocks_per_expert + n tile
  int sf_ngr;                // 128-element K groups (512-byte scale chunks) per row block
  int b_blocks_per_expert;
  uint8_t* hq;               // EPI_SWIGLU (MXFP8): h quantised along I, codes [rows, I]
                             // (NVFP4: packed E2M1 codes [rows, I/2])
  uint8_t* hsf;              // ... and its tiled scales
  int hsf_ngr;
  // NVFP4: the accumulator is multiplied by alpha = act_scale * w_scale[e] (the
  // per-tensor dequantisation scales of the activation and of expert e's weights)
  // before its rounding point; EPI_SWIGLU quantises h with encode scale h_enc
  const float* w_scale;
  float act_scale;
  float h_enc;
  // EPI_DGRAD2 (MXFP8): dA and hs leave only as E4M3 codes with tiled scales: dA
  // along 2I (q_row [rows, 2I], sf_row with sf_row_ngr K groups), dA and hs along
  // the rows, transposed (qt_a [2I, qt_ld], qt_h [I, qt_ld]; scales sft_a, sft_h
  // with qt_ld/128 K groups)
  uint8_t* q_row;
  uint8_t* sf_row;
  int sf_row_ngr;
  uint8_t* qt_a;
  uint8_t* sft_a;
  uint8_t* qt_h;
  uint8_t* sft_h;
  long long qt_ld;
  // failure-path testing: every bounded wait gives up after wait_limit_ns (0 =
  // default); stall_mma = 1 makes the MMA role first wait on a barrier that
  // nothing arrives at, so the timeout path runs
  unsigned long long wait_limit_ns;
  int stall_mma;
  DevError* err;
};

// Encode a 2-D bf16 tensor map (row-major [rows, cols]) with a 64-column x
// box_rows box and 128-byte swizzle: K-major GEMM operand tiles (the TMA cost is
// per box, so a tile is loaded with one box).
int encode_tmap_bf16(CUtensorMap* map, const void* base, long long rows, long long cols,
                     int box_rows);

// Encode an MN-major operand view of a bf16 [krows, ncols] tensor: 3-D (64, krows,
// ncols/64) with box (64, 64, atoms), so one load lands `atoms` 64-wide atoms of
// 64 K rows each, 8 KB apart, in the 128-byte-swizzled MN-major tile layout.
int encode_tmap_bf16_mn(CUtensorMap* map, const void* base, long long krows, long long ncols,
                        int atoms);

// Encode a 2-D fp32 tensor map (row-major [rows, cols]) with a 32 x 128 box
// (128 bytes x 128 rows) and 128-byte swizzle: the weight-gradient tiles that the
// WGRAD epilogue adds into global memory.
int encode_tmap_f32_out(CUtensorMap* map, const void* base, long long rows, long long cols);

// Launch the grouped GEMM.  a_mn / b_mn select MN-major operands; tc is only
// read by EPI_WGRAD (the fp32 gradient [E*M, N]); to0 / to1 are the bf16 output
// tensors of the TMA-store epilogues (128-row boxes):
//   EPI_SWIGLU: h, a    EPI_SCORE: ys    EPI_STORE: out    EPI_DGRAD2: dA, hs
cudaError_t launch_gemm(int epi, int bn, bool a_mn, bool b_mn, const CUtensorMap& ta,
                        const CUtensorMap& tb, const CUtensorMap& tc, const CUtensorMap& to0,
                        const CUtensorMap& to1, const GemmArgs& args, int grid,
                        cudaStream_t stream, bool mx = false);

// The NVFP4 grouped GEMM (kind::mxf4nvf4, E4M3 scales per 16 elements): 128 x 256
// tiles over routed rows, K-major packed E2M1 operands (uint8 tensor maps over
// [rows, K/2]), scales in the tiled layout with 64-element K groups (sf_ngr =
// K/64).  EPI_SWIGLU (W13 through the gate/up block view; h quantised to NVFP4)
// or EPI_SCORE (W2, bf16 ys through tmO0).
cudaError_t launch_gemm_nvfp4(int epi, const CUtensorMap& ta, const CUtensorMap& tb,
                              const CUtensorMap& to0, const GemmArgs& args, int grid,
                              cudaStream_t stream);

// NVFP4 quantisers (moe_nvfp4.cu).  Scale bytes of the tiled layout for
// rows_padded128 rows and K columns: rows/128 x K/64 chunks of 512 bytes.
long long nv_sf_bytes(long long rows_padded128, int K);
// padded rows r < *nrows: quantise x[token_of[r]] (zero for padding) along d
cudaError_t launch_gather_quant_nvfp4(const void* x, const int32_t* token_of, const int32_t* nrows,
                                      int d, float g, uint8_t* codes, uint8_t* sf, int grid,
                                      cudaStream_t stream);
// amax[m] (float bits) of nmat consecutive bf16 matrices of `per` elements
cudaError_t launch_amax_bf16(const void* in, int nmat, long long per, unsigned int* amax,
                             cudaStream_t stream);
// prepared weights: per-expert scales scale[E], codes [E*rows, K/2], tiled scales
// (gu_I > 0: the W13 row blocking)
cudaError_t launch_prepare_nvfp4(const void* w, int E, long long rows_per_expert, int K, int gu_I,
                                 uint8_t* codes, uint8_t* sf, float* scale, cudaStream_t stream);

// Launch the CTA-pair grouped GEMM over routed rows (256 x 256 tiles, A K-major;
// requires expert segments padded to 256 rows and N % 256 == 0).
cudaError_t launch_gemm_pair(int epi, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb,
                             const CUtensorMap& to0, const CUtensorMap& to1, const GemmArgs& args,
                             int grid, cudaStream_t stream);

// 2-D uint8 tensor map (row-major [rows, cols]) with a 128-byte x box_rows box and
// 128-byte swizzle: the E4M3 operand tiles of the MXFP8 GEMMs.
int encode_tmap_u8(CUtensorMap* map, const void* base, long long rows, long long cols,
                   int box_rows);
// W13 [E, 2I, cols] (bf16, or E4M3 bytes) as (cols, I, 2E): a box of box_rows gate
// rows of expert e followed by the same rows of its up half (coordinates
// (k, row within the half, 2e)), one 128-byte swizzled K chunk wide
int encode_tmap_gate_up(CUtensorMap* map, bool fp8, const void* base, long long E, long long I,
                        long long cols, int box_rows);
// MXFP8 W13 [E, 2I, cols] as (cols, 64, 2, I/64, E): a box of two 64-row blocks,
// each its gate rows then the same up rows (coordinates (k, 0, 0, block, e))
int encode_tmap_gate_up_blocks(CUtensorMap* map, const void* base, long long E, long long I,
                               long long cols);

// Dispatch kernels.
struct RouteArgs {
  const int32_t* ids;
  const float* scores;
  int T, k, E, BM;             // BM: padding granule of expert segments (multiple of 128)
  int nblk;                  // ceil(T*k / 1024)
  int32_t* blockcounts;      // [nblk, E]
  int32_t* counts;           // [E]
  int32_t* m_indptr;         // [E+1]
  int32_t* off_pad;          // [E+1]
  int32_t* num_mtiles;       // scalar
  int32_t* tile_expert;      // [max m tiles]
  int32_t* expert_order;     // [E]
  int32_t* num_nonempty;     // scalar
  int32_t* row_of;           // [T*k]
  int32_t* token_of;         // [Rpad max]
  float* score_of;           // [Rpad max]
  DevError* err;
  // CTA-pair row GEMMs (NULL otherwise): each expert's m tiles two at a time
  // (first m tile of each pair) and its odd last m tile, with their counts
  int32_t* pair_list;        // [max m tiles / 2]
  int32_t* left_list;        // [E]
  int32_t* num_pairs;        // scalar
  int32_t* num_left;         // scalar
};
cudaError_t launch_route(const RouteArgs& a, cudaStream_t stream);

// Caller-provided expert-major layout (moe_forward_routed).
constexpr int kRoutedGranule = 128;   // off_pad entries are multiples of the GEMM tile rows
struct RoutedArgs {
  const int32_t* m_indptr;   // [E+1] caller's
  const int32_t* off_pad;    // [E+1] caller's
  int E;
  long long rows;            // rows of the caller's expert-major buffers
  const int32_t* row_of_in;  // [Tk] caller's (NULL: Tk = 0)
  int Tk;
  int32_t* row_of_out;       // [Tk] checked copy
  int32_t* tile_expert;      // [max m tiles]
  int32_t* mtile_list;       // [max m tiles]
  int32_t* list_count;       // scalar
  DevError* err;
};
cudaError_t launch_routed_prepare(const RoutedArgs& a, int grid, cudaStream_t stream);

// rows r < *nrows of dst[r] = src[token_of[r]] (zero where token_of[r] < 0).
cudaError_t launch_gather_rows(const void* src, const int32_t* token_of, const int32_t* nrows,
                               int d, void* dst, int grid, cudaStream_t stream);

// y[t] = bf16(sum_j rows[row_of[t,j]]) in j order; optionally dscores[t,j] =
// sum_nt pdscore[row_of[t,j], nt] in nt order (0 where row_of < 0).
cudaError_t launch_combine(const void* rows, const int32_t* row_of, int T, int k, int d,
                           void* y, const float* pdscore, int n_pd, float* dscores, int grid,
                           cudaStream_t stream);

cudaError_t launch_quant_mxfp8(const void* in, long long rows, int K, uint8_t* codes,
                               uint8_t* scales, cudaStream_t stream);

// Bytes of the tiled MXFP8 scale layout for `rows_padded128` rows (a multiple of
// 128) and K columns (a multiple of 128): rows/128 x K/128 chunks of 512 bytes.
long long mx_sf_bytes(long long rows_padded128, int K);

// Quantise [rows, K] bf16 to E4M3 codes plus tiled E8M0 scales; gu_I > 0 blocks
// the rows of W13 [E*2I, K] by (expert, 64-column gate/up n-tile).
cudaError_t launch_quant_tiled(const void* in, long long rows, int K, int gu_I, uint8_t* codes,
                               uint8_t* sf, cudaStream_t stream);

// Padded rows r < *nrows: quantise x[token_of[r]] (zero for padding) along d.
cudaError_t launch_gather_quant_rows(const void* x, const int32_t* token_of, const int32_t* nrows,
                                     int d, uint8_t* codes, uint8_t* sf, int grid,
                                     cudaStream_t stream);
// Quantise along rows, transposed: `batch` bf16 matrices [R, C] (batch stride
// R*C; with src_row the single matrix's row r is row src_row[r] of `in`, zero
// where negative) -> E4M3 codes [batch][C][R] and tiled E8M0 scales with row
// blocks of 128 over C (block batch*(C/128) + c/128) and K groups of 128 over R.
// Rows r >= *nrows (when nrows != NULL) are skipped.  R % 128 == 0, C % 128 == 0.
cudaError_t launch_quant_rows_t(const void* in, const int32_t* src_row, const int32_t* nrows,
                                int batch, int R, int C, uint8_t* codes, uint8_t* sf,
                                cudaStream_t stream);
// Both quantisations of one [R, C] bf16 operand (rows via src_row as above) in
// one pass: along C into codes_row [R, C] + tiled scales (128-row blocks, K
// groups over C), and along the rows into codes_t [C, R] + tiled scales
// (persistent: a few CTAs on each of num_sms SMs).
cudaError_t launch_quant_two_way(const void* in, const int32_t* src_row, const int32_t* nrows,
                                 int R, int C, uint8_t* codes_row, uint8_t* sf_row,
                                 uint8_t* codes_t, uint8_t* sf_t, int num_sms,
                                 cudaStream_t stream);

}  // namespace moe
