// q4_0 cache builder: one thread per 32-element block along the head dimension, each block
// quantized by q4_quantize_block (fa_quant.cuh, which states the format).
#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa_quant.cuh"

namespace fa {
namespace {

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
  const uint4 w[4] = {__ldg(src), __ldg(src + 1), __ldg(src + 2), __ldg(src + 3)};
  uint4 nb;
  __half sc;
  q4_quantize_block<BF16>(w, nb, sc);
  reinterpret_cast<uint4*>(nib)[dblk] = nb;
  scale[dblk] = sc;
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
