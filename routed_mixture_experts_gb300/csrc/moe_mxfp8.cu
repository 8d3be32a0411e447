// moe_mxfp8.cu -- MXFP8 (E4M3 elements, E8M0 block scales) quantiser.
//
// "Dist-MoE" note, "What it is selling": MXFP8 E4M3 quantises activations after
// routing and accepts prepared weights.  Block rule (OCP microscaling): blocks of
// 32 consecutive elements along K share the scale 2^X with
//   X = floor(log2(max |v|)) - 8        (8 = exponent of E4M3's largest normal)
// clamped to [-127, 127]; the scale byte is X + 127 (0 for an all-zero block);
// each element becomes E4M3(v * 2^-X), rounded to nearest even and saturated to
// +-448 by the hardware conversion cvt.rn.satfinite.e4m3x2.f32.

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

// One thread per 32-element block.
__global__ void __launch_bounds__(256) k_quant_mxfp8(const uint4* __restrict__ in, long long nblocks,
                                                     uint4* __restrict__ codes,
                                                     uint8_t* __restrict__ scales) {
  for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < nblocks;
       b += (long long)gridDim.x * blockDim.x) {
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = in[b * 4 + i];
    float f[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        f[i * 8 + 2 * q] = __uint_as_float(w[q] << 16);
        f[i * 8 + 2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
      }
    }
    uint32_t w[8];
    const uint8_t sc = mx_quant32(f, w);
    codes[b * 2] = make_uint4(w[0], w[1], w[2], w[3]);
    codes[b * 2 + 1] = make_uint4(w[4], w[5], w[6], w[7]);
    scales[b] = sc;
  }
}

__device__ __forceinline__ void unpack_bf16x32(const uint4 (&v)[4], float (&f)[32]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      f[i * 8 + 2 * q] = __uint_as_float(w[q] << 16);
      f[i * 8 + 2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
    }
  }
}

// Quantise [rows, K] bf16 into codes [rows, K] and scales in the tiled layout
// (moe::mx_sf_offset).  gu_I > 0 selects the W13 row blocking: within each
// expert's 2I rows, gate rows [64t, 64t+64) and up rows [I+64t, I+64t+64) form
// row block e*(I/64)+t (the B tile of one 64-column W13 n-tile); gu_I == 0 uses
// plain 128-row blocks.
__global__ void __launch_bounds__(256) k_quant_tiled(const uint4* __restrict__ in, long long rows,
                                                     int K, int gu_I, uint4* __restrict__ codes,
                                                     uint8_t* __restrict__ sf) {
  pdl_wait();   // the previous kernel of the stream has completed
  const int kbs = K / 32;
  const int ngr = K / 128;
  const long long nblocks = rows * kbs;
  for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < nblocks;
       b += (long long)gridDim.x * blockDim.x) {
    const long long row = b / kbs;
    const int kb = (int)(b - row * kbs);
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = in[b * 4 + i];
    float f[32];
    unpack_bf16x32(v, f);
    uint32_t w[8];
    const uint8_t sc = mx_quant32(f, w);
    codes[b * 2] = make_uint4(w[0], w[1], w[2], w[3]);
    codes[b * 2 + 1] = make_uint4(w[4], w[5], w[6], w[7]);
    long long rblock;
    int rin;
    if (gu_I > 0) {
      const long long e = row / (2 * gu_I);
      const int i = (int)(row - e * 2 * gu_I);
      const int up = i >= gu_I;
      const int ii = up ? i - gu_I : i;
      rblock = e * (gu_I / 64) + ii / 64;
      rin = up * 64 + (ii & 63);
    } else {
      rblock = row >> 7;
      rin = (int)(row & 127);
    }
    sf[mx_sf_offset(rblock, rin, kb, ngr)] = sc;
  }
  pdl_trigger();
}

// Gather + quantise: padded row r of the expert-major activations is token
// token_of[r] of x (zero where token_of[r] < 0), quantised along d.  One warp
// per row, one 32-element block per lane per pass.
__global__ void __launch_bounds__(256) k_gather_quant_rows(const uint4* __restrict__ x,
                                                           const int32_t* __restrict__ token_of,
                                                           const int32_t* __restrict__ nrows_p,
                                                           int d, uint4* __restrict__ codes,
                                                           uint8_t* __restrict__ sf) {
  pdl_wait();   // the previous kernel of the stream has completed
  const int nrows = *nrows_p;
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int kbs = d / 32;
  const int ngr = d / 128;
  for (int r = gw; r < nrows; r += nw) {
    const int t = token_of[r];
    for (int kb = lane; kb < kbs; kb += 32) {
      float f[32];
      if (t >= 0) {
        uint4 v[4];
        const uint4* src = x + ((long long)t * d + kb * 32) / 8;
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = src[i];
        unpack_bf16x32(v, f);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) f[i] = 0.f;
      }
      uint32_t w[8];
      const uint8_t sc = mx_quant32(f, w);
      uint4* dst = codes + ((long long)r * d + kb * 32) / 16;
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      sf[mx_sf_offset(r >> 7, r & 127, kb, ngr)] = sc;
    }
  }
  pdl_trigger();
}

// Quantise along rows, transposed: for each of `batch` matrices in [R, C] bf16
// (batch stride R*C; with src_row, row r of the single matrix is row
// src_row[r] of `in`, zero where src_row[r] < 0), write codes [C, R] (each
// column becomes a K-major row, K = R) and scales in the tiled layout with row
// blocks of 128 over the batch's C rows (block batch*(C/128) + c/128) and K
// groups of 128 over R.  The blocks of 32 run along r.  Rows r >= *nrows_p (when
// given) are not written.  A CTA takes 32 rows x 256 columns: it stages them in
// shared memory and each thread quantises one column's 32 values.
constexpr int kQtRows = 32, kQtCols = 256;

__global__ void __launch_bounds__(kQtCols) k_quant_rows_t(const uint16_t* __restrict__ in,
                                                          const int32_t* __restrict__ src_row,
                                                          const int32_t* __restrict__ nrows_p,
                                                          int R, int C,
                                                          uint8_t* __restrict__ codes,
                                                          uint8_t* __restrict__ sf) {
  pdl_wait();   // the previous kernel of the stream has completed
  __shared__ __align__(16) uint16_t tile[kQtRows][kQtCols];
  const int r0 = blockIdx.x * kQtRows;
  const int c0 = blockIdx.y * kQtCols;
  const long long b = blockIdx.z;
  const int nrows = nrows_p ? *nrows_p : R;
  if (r0 >= nrows) return;
  const uint16_t* mat = in + b * (long long)R * C;
  // coalesced loads: 32 rows x 256 columns, 8 bf16 (16 bytes) per access
  for (int q = threadIdx.x; q < kQtRows * kQtCols / 8; q += kQtCols) {
    const int rr = q / (kQtCols / 8), cc = (q % (kQtCols / 8)) * 8;
    const int r = r0 + rr;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    const long long srow = r >= nrows ? -1 : (src_row ? (long long)src_row[r] : (long long)r);
    if (srow >= 0 && c0 + cc < C) v = *reinterpret_cast<const uint4*>(mat + srow * C + c0 + cc);
    *reinterpret_cast<uint4*>(&tile[rr][cc]) = v;
  }
  __syncthreads();
  const int c = c0 + threadIdx.x;
  if (c >= C) return;
  float f[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(((uint32_t)tile[i][threadIdx.x]) << 16);
  uint32_t w[8];
  const uint8_t scv = mx_quant32(f, w);
  uint4* dst = reinterpret_cast<uint4*>(codes + (b * (long long)C + c) * R + r0);
  dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
  dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
  sf[mx_sf_offset(b * (C / 128) + (c >> 7), c & 127, r0 / 32, R / 128)] = scv;
  pdl_trigger();
}

// Both quantisations of one [R, C] bf16 operand in one pass (R = padded rows;
// with src_row, row r is row src_row[r] of `in`, zero where negative; rows
// r >= *nrows_p are skipped): along C into codes_row [R, C] with tiled scales
// (128-row blocks, K groups over C), and along the rows, transposed, into
// codes_t [C, R] with tiled scales as k_quant_rows_t.  The work is cut into
// tiles of kTwRows rows x 256 columns, staged in shared memory (rows padded by
// 16 bytes so the column pass is free of bank conflicts): each thread
// quantises kTwRows/32 32-column blocks of rows, then the kTwRows/32 32-row
// blocks of one column, whose scales (consecutive bytes) it writes whole and
// whose codes go back through shared memory so that the stores are coalesced.
// The kernel is persistent and double-buffered: while a CTA
// quantises one tile, the 16-byte asynchronous copies of its next tile are in
// flight.
constexpr int kTwRows = 64;
constexpr int kTwLd = kQtCols + 8;                 // staged row stride in elements (528 bytes)
constexpr int kTwBuf = kTwRows * kTwLd;            // elements per staging buffer
// transposed codes staged per column (bytes): kTwRows plus 16, so the 16-byte
// stores of a quarter warp fall in distinct banks
constexpr int kTwTLd = kTwRows + 16;
static_assert(kQtCols * kTwTLd <= kTwBuf * 2, "transposed codes fit the tile's buffer");
constexpr int kTwSmem = 2 * kTwBuf * 2;            // two buffers, bytes
constexpr int kTwCtasPerSm = 3;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  // bytes past src_bytes (0 or 16) are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_1() {
  asm volatile("cp.async.wait_group 1;" ::: "memory");
}

__global__ void __launch_bounds__(kQtCols, kTwCtasPerSm)
    k_quant_two_way(const uint16_t* __restrict__ in, const int32_t* __restrict__ src_row,
                    const int32_t* __restrict__ nrows_p, int R, int C,
                    uint8_t* __restrict__ codes_row, uint8_t* __restrict__ sf_row,
                    uint8_t* __restrict__ codes_t, uint8_t* __restrict__ sf_t) {
  pdl_wait();   // the previous kernel of the stream has completed
  extern __shared__ __align__(16) uint16_t tw_tile[];    // [2][kTwRows][kTwLd]
  const int nrows = nrows_p ? *nrows_p : R;
  const int ncb = (C + kQtCols - 1) / kQtCols;
  const int ntiles = (nrows + kTwRows - 1) / kTwRows * ncb;
  // A warp copies 512 contiguous bytes of one row.  The source rows of a tile's
  // copies are looked up one tile ahead (lookup), so no copy waits for them.
  constexpr int kPer = kTwRows * kQtCols / 8 / kQtCols;   // copies per thread and tile
  int srow[kPer];
  auto lookup = [&](int tile) {
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int r = tile / ncb * kTwRows + (threadIdx.x + j * kQtCols) / (kQtCols / 8);
      srow[j] = tile >= ntiles || r >= nrows ? -1 : (src_row ? src_row[r] : r);
    }
  };
  auto issue = [&](int tile, int buf) {
    const int c0 = tile % ncb * kQtCols;
    const uint32_t base = smem_u32(tw_tile + buf * kTwBuf);
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int q = threadIdx.x + j * kQtCols;
      const int rr = q / (kQtCols / 8), cc = (q % (kQtCols / 8)) * 8;
      const bool ok = srow[j] >= 0 && c0 + cc < C;
      cp_async16(base + (uint32_t)(rr * kTwLd + cc) * 2u,
                 ok ? in + (long long)srow[j] * C + c0 + cc : in, ok ? 16u : 0u);
    }
  };
  int tile = blockIdx.x;
  lookup(tile);
  if (tile < ntiles) issue(tile, 0);
  cp_async_commit();
  lookup(tile + gridDim.x);
#pragma unroll 1
  for (int it = 0; tile < ntiles; ++it, tile += gridDim.x) {
    const int buf = it & 1;
    if (tile + (int)gridDim.x < ntiles) issue(tile + gridDim.x, buf ^ 1);
    cp_async_commit();               // (possibly empty) group of the next tile
    lookup(tile + 2 * gridDim.x);    // in flight while this tile is quantised
    cp_async_wait_1();               // this tile's copies have landed
    __syncthreads();
    const uint16_t* t = tw_tile + buf * kTwBuf;
    const int r0 = tile / ncb * kTwRows, c0 = tile % ncb * kQtCols;
    // along C: rows rr = threadIdx/8 + 32*i, 32-column block jb (eight threads
    // write a row's 256 codes contiguously)
#pragma unroll 1
    for (int i = 0; i < kTwRows / 32; ++i) {
      const int rr = (threadIdx.x >> 3) + 32 * i, jb = threadIdx.x & 7;
      const int c = c0 + jb * 32;
      if (c < C) {
        float f[32];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 v = *reinterpret_cast<const uint4*>(&t[rr * kTwLd + jb * 32 + q * 8]);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            f[q * 8 + 2 * u] = __uint_as_float(w[u] << 16);
            f[q * 8 + 2 * u + 1] = __uint_as_float(w[u] & 0xFFFF0000u);
          }
        }
        uint32_t w[8];
        const uint8_t scv = mx_quant32(f, w);
        const long long r = r0 + rr;
        uint4* dst = reinterpret_cast<uint4*>(codes_row + r * C + c);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        sf_row[mx_sf_offset(r >> 7, (int)(r & 127), c >> 5, C / 128)] = scv;
      }
    }
    // along the rows: column c, its kTwRows/32 32-row blocks
    const int c = c0 + threadIdx.x;
    static_assert(kTwRows == 64, "rows per tile");
    uint4 tq[kTwRows / 16];          // column c's codes, 16 rows per vector
    if (c < C) {
      uint32_t sc4 = 0;
#pragma unroll
      for (int b = 0; b < kTwRows / 32; ++b) {
        float f[32];
#pragma unroll
        for (int i = 0; i < 32; ++i)
          f[i] = __uint_as_float(((uint32_t)t[(32 * b + i) * kTwLd + threadIdx.x]) << 16);
        uint32_t w[8];
        sc4 |= (uint32_t)mx_quant32(f, w) << (8 * b);
        tq[2 * b] = make_uint4(w[0], w[1], w[2], w[3]);
        tq[2 * b + 1] = make_uint4(w[4], w[5], w[6], w[7]);
      }
      // the blocks of one K group sit in consecutive bytes of the tiled layout
      *reinterpret_cast<uint16_t*>(sf_t + mx_sf_offset(c >> 7, c & 127, r0 / 32, R / 128)) =
          (uint16_t)sc4;
    }
    // Each column's codes are one kTwRows-byte piece of a different output row.
    // Stored from registers, a warp's 16-byte stores would land in 32 rows; the
    // tile's buffer (read completely by now) stages them instead, and
    // consecutive threads then write consecutive 16-byte pieces of a row.
    __syncthreads();
    uint8_t* stg = reinterpret_cast<uint8_t*>(tw_tile + buf * kTwBuf);
    if (c < C) {
#pragma unroll
      for (int j = 0; j < kTwRows / 16; ++j)
        *reinterpret_cast<uint4*>(stg + threadIdx.x * kTwTLd + j * 16) = tq[j];
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kTwRows / 16; ++j) {
      const int idx = threadIdx.x + j * kQtCols;
      const int cc = idx / (kTwRows / 16), pc = idx % (kTwRows / 16);
      if (c0 + cc < C)
        *reinterpret_cast<uint4*>(codes_t + (long long)(c0 + cc) * R + r0 + pc * 16) =
            *reinterpret_cast<const uint4*>(stg + cc * kTwTLd + pc * 16);
    }
    __syncthreads();                 // buffer `buf` is refilled next iteration
  }
  pdl_trigger();
}

}  // namespace

cudaError_t launch_quant_two_way(const void* in, const int32_t* src_row, const int32_t* nrows,
                                 int R, int C, uint8_t* codes_row, uint8_t* sf_row,
                                 uint8_t* codes_t, uint8_t* sf_t, int num_sms,
                                 cudaStream_t stream) {
  if (R % 128 || C % 128 || num_sms < 1) return cudaErrorInvalidValue;
  static std::atomic<unsigned long long> configured{0};   // devices the kernel is set up on
  const cudaError_t e = smem_optin_once(k_quant_two_way, kTwSmem, configured);
  if (e != cudaSuccess) return e;
  // persistent: a few CTAs per SM, at most one per tile
  const long long tiles = (long long)(R / kTwRows) * ((C + kQtCols - 1) / kQtCols);
  const int grid = (int)(tiles < (long long)num_sms * kTwCtasPerSm ? tiles
                                                                   : (long long)num_sms * kTwCtasPerSm);
  return launch_pdl(k_quant_two_way, dim3(grid), dim3(kQtCols), kTwSmem, stream,
                    static_cast<const uint16_t*>(in), src_row, nrows, R, C, codes_row, sf_row,
                    codes_t, sf_t);
}

cudaError_t launch_quant_rows_t(const void* in, const int32_t* src_row, const int32_t* nrows,
                                int batch, int R, int C, uint8_t* codes, uint8_t* sf,
                                cudaStream_t stream) {
  if (R % 128 || C % 128 || batch < 1) return cudaErrorInvalidValue;
  const dim3 grid(R / kQtRows, (C + kQtCols - 1) / kQtCols, batch);
  return launch_pdl(k_quant_rows_t, grid, dim3(kQtCols), 0, stream,
                    static_cast<const uint16_t*>(in), src_row, nrows, R, C, codes, sf);
}

long long mx_sf_bytes(long long rows_padded128, int K) {
  return rows_padded128 / 128 * (long long)(K / 128) * 512;
}

cudaError_t launch_quant_tiled(const void* in, long long rows, int K, int gu_I, uint8_t* codes,
                               uint8_t* sf, cudaStream_t stream) {
  const long long nblocks = rows * (K / 32);
  long long grid = (nblocks + 255) / 256;
  if (grid > 65535LL * 8) grid = 65535LL * 8;
  if (grid < 1) grid = 1;
  return launch_pdl(k_quant_tiled, dim3((unsigned)grid), dim3(256), 0, stream,
                    static_cast<const uint4*>(in), rows, K, gu_I,
                    reinterpret_cast<uint4*>(codes), sf);
}

cudaError_t launch_gather_quant_rows(const void* x, const int32_t* token_of, const int32_t* nrows,
                                     int d, uint8_t* codes, uint8_t* sf, int grid,
                                     cudaStream_t stream) {
  return launch_pdl(k_gather_quant_rows, dim3(grid), dim3(256), 0, stream,
                    static_cast<const uint4*>(x), token_of, nrows, d,
                    reinterpret_cast<uint4*>(codes), sf);
}

cudaError_t launch_quant_mxfp8(const void* in, long long rows, int K, uint8_t* codes,
                               uint8_t* scales, cudaStream_t stream) {
  const long long nblocks = rows * (K / 32);
  long long grid = (nblocks + 255) / 256;
  if (grid > 65535LL * 8) grid = 65535LL * 8;
  k_quant_mxfp8<<<(unsigned)grid, 256, 0, stream>>>(static_cast<const uint4*>(in), nblocks,
                                                   reinterpret_cast<uint4*>(codes), scales);
  return cudaGetLastError();
}

}  // namespace moe
