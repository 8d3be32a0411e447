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

// Two floats -> two E4M3 bytes (lo in bits 0-7), RNE, saturating.
__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// E8M0 exponent X of a block from its (non-negative) bf16-exact amax.
__device__ __forceinline__ int block_exponent(float amax) {
  const int ef = (int)((__float_as_uint(amax) >> 23) & 0xFF);   // biased exponent
  if (ef == 0) return -127;                                    // zero or subnormal
  const int X = ef - 127 - 8;
  return X < -127 ? -127 : (X > 127 ? 127 : X);
}

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
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(f[i]));
    uint4 out0 = make_uint4(0, 0, 0, 0), out1 = make_uint4(0, 0, 0, 0);
    int X = -127;
    if (amax > 0.f) {
      X = block_exponent(amax);
      const float inv = __uint_as_float((uint32_t)(127 - X) << 23);   // 2^-X, exact
      uint32_t w[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint16_t p0 = cvt_e4m3x2(f[4 * q] * inv, f[4 * q + 1] * inv);
        const uint16_t p1 = cvt_e4m3x2(f[4 * q + 2] * inv, f[4 * q + 3] * inv);
        w[q] = (uint32_t)p0 | ((uint32_t)p1 << 16);
      }
      out0 = make_uint4(w[0], w[1], w[2], w[3]);
      out1 = make_uint4(w[4], w[5], w[6], w[7]);
    }
    codes[b * 2] = out0;
    codes[b * 2 + 1] = out1;
    scales[b] = (uint8_t)(X + 127);
  }
}

}  // namespace

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
