// q4_0 cache builder: one thread per 32-element block along the head dimension.
//
// Format (the pages name the q4_0 cache type -- "FlashAttention on gfx90a: Why It's Broken and
// How to Fix It", Impact of the V Dequant Patch, -ctk q4_0 -ctv q4_0 -- but do not fix its bits;
// this is the block format the library defines): m = the signed element of largest magnitude
// (first one on ties), d = m / -8, codes q = min(15, trunc(x * (1/d) + 8.5)) computed as one
// rounded f32 multiply and one rounded f32 add, stored two per byte (element j low nibble,
// element j+16 high nibble), and d stored as fp16 (round to nearest even).  Every step uses the
// correctly rounded intrinsics so the result is bit-identical on any IEEE implementation.
#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

template <bool BF16>
__device__ __forceinline__ float to_f32(uint16_t bits) {
  if (BF16) return __uint_as_float(static_cast<uint32_t>(bits) << 16);
  return __half2float(__ushort_as_half(bits));
}

// blockIdx.y selects the job (K, then V when appending both); source block blk of row
// (bh, s) is written to destination row bh * Scap + pos0 + s
template <bool BF16>
__global__ void __launch_bounds__(256) quantize_kernel(QuantJob j0, QuantJob j1, int64_t nblocks,
                                                       int nb_row, int S_src, int Scap,
                                                       int pos0) {
  const int64_t blk = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (blk >= nblocks) return;
  // fields selected by value (a reference to the parameter would turn them into loads)
  const bool second = blockIdx.y != 0;
  const uint16_t* __restrict__ x = static_cast<const uint16_t*>(second ? j1.x : j0.x);
  uint8_t* __restrict__ nib = static_cast<uint8_t*>(second ? j1.nib : j0.nib);
  __half* __restrict__ scale = static_cast<__half*>(second ? j1.scale : j0.scale);
  // destination block: the same index when the whole tensor is written (uniform branch);
  // otherwise one 32-bit (or, for very large tensors, 64-bit) division per index
  int64_t dblk = blk;
  if (S_src != Scap || pos0 != 0) {
    int64_t row, bh;
    if (blk < 0x7fffffffLL) {
      const uint32_t r32 = static_cast<uint32_t>(blk) / static_cast<uint32_t>(nb_row);
      row = r32;
      bh = r32 / static_cast<uint32_t>(S_src);
    } else {
      row = blk / nb_row;
      bh = row / S_src;
    }
    dblk = ((bh * Scap + pos0) + (row - bh * S_src)) * nb_row + (blk - row * nb_row);
  }
  const uint4* src = reinterpret_cast<const uint4*>(x + blk * 32);
  float v[32];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 w = __ldg(src + i);
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[8 * i + 2 * k] = to_f32<BF16>(static_cast<uint16_t>(u[k] & 0xFFFFu));
      v[8 * i + 2 * k + 1] = to_f32<BF16>(static_cast<uint16_t>(u[k] >> 16));
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
    uint32_t w = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int j = 4 * i + k;
      w |= (q[j] | (q[j + 16] << 4)) << (8 * k);
    }
    out[i] = w;
  }
  reinterpret_cast<uint4*>(nib)[dblk] = make_uint4(out[0], out[1], out[2], out[3]);
  scale[dblk] = __float2half_rn(d);
}

}  // namespace

cudaError_t quantize_launch(QuantJob j0, QuantJob j1, int64_t BH, int S_src, int Scap, int pos0,
                            int D, bool bf16, cudaStream_t stream) {
  const int nb_row = D / 32;
  const int64_t nblocks = BH * S_src * nb_row;
  if (nblocks == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t grid = (nblocks + threads - 1) / threads;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  const dim3 g(static_cast<unsigned>(grid), j1.x ? 2u : 1u);
  if (bf16)
    quantize_kernel<true><<<g, threads, 0, stream>>>(j0, j1, nblocks, nb_row, S_src, Scap, pos0);
  else
    quantize_kernel<false><<<g, threads, 0, stream>>>(j0, j1, nblocks, nb_row, S_src, Scap, pos0);
  return cudaGetLastError();
}

}  // namespace fa
