// q4_0 block quantizer shared by the cache builder (fa_quant.cu) and the prefill that appends
// its own chunk to the cache (fa_prefill.cu).
//
// Format (the pages name the q4_0 cache type -- "FlashAttention on gfx90a: Why It's Broken and
// How to Fix It", Impact of the V Dequant Patch, -ctk q4_0 -ctv q4_0 -- but do not fix its bits;
// this is the block format the library defines): m = the signed element of largest magnitude
// (first one on ties), d = m / -8, codes q = min(15, trunc(x * (1/d) + 8.5)) computed as one
// rounded f32 multiply and one rounded f32 add, stored two per byte (element j low nibble,
// element j+16 high nibble), and d stored as fp16 (round to nearest even).  Every step uses the
// correctly rounded intrinsics so the result is bit-identical on any IEEE implementation.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace fa {

template <bool BF16>
__device__ __forceinline__ float q4_to_f32(uint16_t bits) {
  if (BF16) return __uint_as_float(static_cast<uint32_t>(bits) << 16);
  return __half2float(__ushort_as_half(bits));
}

// Quantize one block of 32 consecutive 16-bit values (four 16-byte words w[0..3], elements in
// order): the 16 bytes of nibbles and the fp16 scale.
template <bool BF16>
__device__ __forceinline__ void q4_quantize_block(const uint4 (&w)[4], uint4& nib, __half& scale) {
  float v[32];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t u[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[8 * i + 2 * k] = q4_to_f32<BF16>(static_cast<uint16_t>(u[k] & 0xFFFFu));
      v[8 * i + 2 * k + 1] = q4_to_f32<BF16>(static_cast<uint16_t>(u[k] >> 16));
    }
  }
  float amax = 0.f, m = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float a = fabsf(v[j]);
    if (a > amax) {
      amax = a;
      m = v[j];
    }
  }
  const float d = __fdiv_rn(m, -8.0f);
  const float id = (d != 0.f) ? __fdiv_rn(1.0f, d) : 0.f;
  uint32_t q[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float t = __fadd_rn(__fmul_rn(v[j], id), 8.5f);
    int qi = __float2int_rz(t);
    qi = min(15, max(0, qi));
    q[j] = static_cast<uint32_t>(qi);
  }
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t wd = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int j = 4 * i + k;
      wd |= (q[j] | (q[j + 16] << 4)) << (8 * k);
    }
    out[i] = wd;
  }
  nib = make_uint4(out[0], out[1], out[2], out[3]);
  scale = __float2half_rn(d);
}

}  // namespace fa
