// moe_nvfp4.cu -- NVFP4 quantisers: E2M1 elements (two per byte, element 2i in
// the low nibble), one E4M3 scale per 16 consecutive elements along K, and a
// per-tensor scale.
//
// "Dist-MoE" note, "What it is selling": the FP4 mode serves inference only,
// with weights prepared ahead of the call; nvfp4moe README, "Dense GEMM" /
// "Grouped GEMM": E2M1 codes two to a byte, one E4M3 scale per block, one
// dequantisation scale per tensor, the GEMM scaled by the product of its
// operands' tensor scales; "MoE layer": fixed activation scales, the bf16
// activations quantised after dispatch.
//
// Block rule (two-level scaling; see nv_quant16): with the tensor's encode scale
// g = 1 / (its dequantisation scale), a 16-element block with amax A gets the
// E4M3 scale code E4M3((A / 6) * g) and its elements E2M1(v * (g / S)), S the
// scale's value, both rounded to nearest even and saturated.  Weights: per
// expert, dequantisation scale amax(W[e]) / (6 * 448) (1 for an all-zero
// expert).  Scales are stored in the tiled layout of the block-scaled GEMMs
// (mx_sf_offset with 16-element blocks and 64-element K groups).

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

__device__ __forceinline__ void unpack_bf16x16(const uint4 (&v)[2], float (&f)[16]) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      f[i * 8 + 2 * q] = __uint_as_float(w[q] << 16);
      f[i * 8 + 2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
    }
  }
}

// Quantise one 64-element group (four 16-element blocks) of bf16 values at
// `src` (NULL: zeros): 32 code bytes to `dst`, the four scale bytes as one word
// (block b in byte b), which is their order in the tiled layout.
__device__ __forceinline__ uint32_t nv_quant64(const uint4* src, float g, uint4* dst) {
  uint32_t sc = 0;
  uint32_t w[8];
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    float f[16];
    if (src) {
      const uint4 v[2] = {src[2 * b], src[2 * b + 1]};
      unpack_bf16x16(v, f);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) f[i] = 0.f;
    }
    uint32_t q[2];
    sc |= (uint32_t)nv_quant16(f, g, q) << (8 * b);
    w[2 * b] = q[0];
    w[2 * b + 1] = q[1];
  }
  dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
  dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
  return sc;
}

// Gather + quantise: padded row r of the expert-major activations is token
// token_of[r] of x (zero where token_of[r] < 0), quantised along d with the
// static encode scale g.  One warp per row; the row is read in coalesced 16-byte
// pieces (piece p = 8 elements, lane p % 32), so a 16-element block spans two
// neighbouring lanes: its amax is combined with one shuffle, each lane
// quantises its 8 elements (4 code bytes, stored coalesced) and the even lane
// writes the block's scale.
__global__ void __launch_bounds__(256) k_gather_quant_nvfp4(const uint4* __restrict__ x,
                                                            const int32_t* __restrict__ token_of,
                                                            const int32_t* __restrict__ nrows_p,
                                                            int d, float g,
                                                            uint8_t* __restrict__ codes,
                                                            uint8_t* __restrict__ sf) {
  pdl_wait();   // the previous kernel of the stream has completed
  const int nrows = *nrows_p;
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int npc = d / 8;                     // 16-byte pieces per row (a multiple of 2)
  const int ngr = d / 64;
  for (int r = gw; r < nrows; r += nw) {
    const int t = token_of[r];
    const uint4* src = x + (long long)(t < 0 ? 0 : t) * npc;
    uint32_t* dst = reinterpret_cast<uint32_t*>(codes + (long long)r * (d / 2));
    // every lane runs every pass (the shuffles need the whole warp); a lane past
    // the row's end holds zeros and stores nothing (blocks never straddle it)
#pragma unroll 4
    for (int p0 = 0; p0 < npc; p0 += 32) {
      const int pc = p0 + lane;
      const bool in = pc < npc;
      const uint4 v = (t >= 0 && in) ? src[pc] : make_uint4(0u, 0u, 0u, 0u);
      float f[8];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        f[2 * q] = __uint_as_float(w[q] << 16);
        f[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
      }
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));   // the block's other half
      const float tt = __fmul_rn(__fdiv_rn(amax, 6.0f), g);
      const uint8_t sc = (uint8_t)(cvt_e4m3x2(tt, 0.f) & 0xFFu);
      const float S = e4m3_to_f32(sc);
      uint32_t q8 = 0u;
      if (S > 0.f) {
        const float rr = __fdiv_rn(g, S);
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = __fmul_rn(f[i], rr);
        q8 = cvt_e2m1x8(f);
      }
      if (in) {
        dst[pc] = q8;
        if (!(lane & 1)) sf[mx_sf_offset(r >> 7, r & 127, pc >> 1, ngr)] = sc;
      }
    }
  }
  pdl_trigger();
}

// Per-matrix amax of `nmat` consecutive bf16 matrices of `per` elements each
// (bits of the non-negative float, combined with atomicMax: order-independent).
__global__ void __launch_bounds__(256) k_amax_bf16(const uint16_t* __restrict__ in, int nmat,
                                                   long long per, unsigned int* __restrict__ amax) {
  const long long n = (long long)nmat * per;
  for (long long i0 = (blockIdx.x * (long long)blockDim.x + threadIdx.x) * 8; i0 < n;
       i0 += (long long)gridDim.x * blockDim.x * 8) {
    const int m = (int)(i0 / per);
    const long long end = (m + 1) * per < n ? (m + 1) * per : n;
    float a = 0.f;
    if (i0 + 8 <= end && (i0 & 7) == 0) {
      const uint4 v = *reinterpret_cast<const uint4*>(in + i0);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        a = fmaxf(a, fmaxf(fabsf(__uint_as_float(w[q] << 16)),
                           fabsf(__uint_as_float(w[q] & 0xFFFF0000u))));
      atomicMax(amax + m, __float_as_uint(a));
    } else {
      for (long long i = i0; i < i0 + 8 && i < n; ++i) {
        const int mi = (int)(i / per);
        atomicMax(amax + mi, __float_as_uint(fabsf(__uint_as_float((uint32_t)in[i] << 16))));
      }
    }
  }
}

__global__ void k_fill_u32(unsigned int* p, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) p[i] = 0u;
}

// Per-expert weight scales, in place: the amax bits become the dequantisation
// scale amax / (6 * 448) (1 for zero).
__global__ void k_nv_weight_scales(float* __restrict__ scale, int E) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  const float a = scale[e];
  scale[e] = a > 0.f ? __fdiv_rn(a, 2688.0f) : 1.0f;
}

// Quantise [rows, K] bf16 weights (rows_per_expert rows per expert, encode scale
// enc[e]) into packed codes [rows, K/2] and tiled scales.  gu_I > 0 selects the
// W13 row blocking (within each expert's 2I rows, gate rows [64t, 64t+64) and up
// rows [I+64t, I+64t+64) form row block e*(I/64)+t); gu_I == 0 plain 128-row
// blocks.  One thread per 64-element group.
__global__ void __launch_bounds__(256) k_quant_nvfp4_tiled(const uint4* __restrict__ in,
                                                           long long rows, int K, int gu_I,
                                                           long long rows_per_expert,
                                                           const float* __restrict__ scale,
                                                           uint8_t* __restrict__ codes,
                                                           uint8_t* __restrict__ sf) {
  const int ngr = K / 64;
  const long long ngroups = rows * ngr;
  for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < ngroups;
       b += (long long)gridDim.x * blockDim.x) {
    const long long row = b / ngr;
    const int kg = (int)(b - row * ngr);
    const long long e = row / rows_per_expert;
    uint4* dst = reinterpret_cast<uint4*>(codes + row * (K / 2) + kg * 32);
    const uint32_t sc = nv_quant64(in + (row * K + kg * 64) / 8, __fdiv_rn(1.0f, scale[e]), dst);
    long long rblock;
    int rin;
    if (gu_I > 0) {
      const int i = (int)(row - e * 2 * gu_I);
      const int up = i >= gu_I;
      const int ii = up ? i - gu_I : i;
      rblock = e * (gu_I / 64) + ii / 64;
      rin = up * 64 + (ii & 63);
    } else {
      rblock = row >> 7;
      rin = (int)(row & 127);
    }
    *reinterpret_cast<uint32_t*>(sf + mx_sf_offset(rblock, rin, kg * 4, ngr)) = sc;
  }
}

int grid_for(long long n, int per_thread) {
  long long g = (n / per_thread + 255) / 256;
  if (g > 65535LL * 8) g = 65535LL * 8;
  return g < 1 ? 1 : (int)g;
}

}  // namespace

long long nv_sf_bytes(long long rows_padded128, int K) {
  return rows_padded128 / 128 * (long long)(K / 64) * 512;
}

cudaError_t launch_gather_quant_nvfp4(const void* x, const int32_t* token_of, const int32_t* nrows,
                                      int d, float g, uint8_t* codes, uint8_t* sf, int grid,
                                      cudaStream_t stream) {
  return launch_pdl(k_gather_quant_nvfp4, dim3(grid), dim3(256), 0, stream,
                    static_cast<const uint4*>(x), token_of, nrows, d, g, codes, sf);
}

cudaError_t launch_amax_bf16(const void* in, int nmat, long long per, unsigned int* amax,
                             cudaStream_t stream) {
  k_fill_u32<<<1, 256, 0, stream>>>(amax, nmat);
  cudaError_t e = cudaPeekAtLastError();
  if (e != cudaSuccess) return e;
  k_amax_bf16<<<grid_for((long long)nmat * per, 8), 256, 0, stream>>>(
      static_cast<const uint16_t*>(in), nmat, per, amax);
  return cudaPeekAtLastError();
}

cudaError_t launch_prepare_nvfp4(const void* w, int E, long long rows_per_expert, int K, int gu_I,
                                 uint8_t* codes, uint8_t* sf, float* scale, cudaStream_t stream) {
  // scale[] holds the amax bits first, then the scales
  cudaError_t e = launch_amax_bf16(w, E, rows_per_expert * K,
                                   reinterpret_cast<unsigned int*>(scale), stream);
  if (e != cudaSuccess) return e;
  k_nv_weight_scales<<<(E + 255) / 256, 256, 0, stream>>>(scale, E);
  if ((e = cudaPeekAtLastError()) != cudaSuccess) return e;
  const long long rows = (long long)E * rows_per_expert;
  k_quant_nvfp4_tiled<<<grid_for(rows * (K / 64), 1), 256, 0, stream>>>(
      static_cast<const uint4*>(w), rows, K, gu_I, rows_per_expert, scale, codes, sf);
  return cudaPeekAtLastError();
}

}  // namespace moe
