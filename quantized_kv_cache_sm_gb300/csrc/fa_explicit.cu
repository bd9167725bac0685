// The explicit (non-flash) attention path, for comparison with the fused kernels: K and V are
// expanded to dense f16/bf16 when they are q4_0, S = scale * Q K^T is written out in f32 by a
// batched GEMM, a softmax kernel turns each row of S into P (causal mask, max, exp, normalise,
// rounded to the input dtype), and O = P V is a second batched GEMM.  This is Approach C of
// "FlashAttention on gfx90a: Why It's Broken and How to Fix It" (Approach C: dequantize K and V
// to f16, then two GEMMs and a softmax) and the "explicit f32 matmul + softmax + matmul"
// reference of "perf(rocm): defer SDPA accumulator rescale, stage Q once per block (#2306)" (Test
// plan).  The two GEMMs are plain library GEMMs (cuBLAS); the dequant and softmax are kernels
// of this file.
//
// Grouped-query heads: the G = Hq / Hkv query heads of a kv head are consecutive rows of Q, so
// one GEMM per (batch, kv head) computes their scores against that kv head's keys at once:
// S_g [G*Sq, Sk] = Q_g [G*Sq, D] K^T [D, Sk]; O_g [G*Sq, D] = P_g [G*Sq, Sk] V [Sk, D].
#include <cublas_v2.h>

#include <mutex>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

template <bool BF16>
__device__ __forceinline__ uint16_t to_bits(float v) {
  return BF16 ? __bfloat16_as_ushort(__float2bfloat16_rn(v))
              : __half_as_ushort(__float2half_rn(v));
}

// q4_0 -> dense: element = (q - 8) * d, the product formed in f32 (exact) and rounded once to
// the dtype -- the values the fused kernels feed their MMAs.  One thread per 32-element block.
template <bool BF16>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t* __restrict__ nib,
                                                      const __half* __restrict__ scale,
                                                      uint16_t* __restrict__ out,
                                                      int64_t nblocks) {
  const int64_t blk = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (blk >= nblocks) return;
  const uint4 w = reinterpret_cast<const uint4*>(nib)[blk];
  const float d = __half2float(scale[blk]);
  const uint32_t b4[4] = {w.x, w.y, w.z, w.w};
  uint32_t o[16];
#pragma unroll
  for (int j = 0; j < 16; j += 2) {
    // bytes j, j+1 hold elements j, j+1 (low nibbles) and j+16, j+17 (high nibbles)
    const uint32_t b0 = (b4[j >> 2] >> (8 * (j & 3))) & 0xFFu;
    const uint32_t b1 = (b4[(j + 1) >> 2] >> (8 * ((j + 1) & 3))) & 0xFFu;
    const float lo0 = static_cast<float>(static_cast<int>(b0 & 15u) - 8) * d;
    const float lo1 = static_cast<float>(static_cast<int>(b1 & 15u) - 8) * d;
    const float hi0 = static_cast<float>(static_cast<int>(b0 >> 4) - 8) * d;
    const float hi1 = static_cast<float>(static_cast<int>(b1 >> 4) - 8) * d;
    o[j >> 1] = to_bits<BF16>(lo0) | (static_cast<uint32_t>(to_bits<BF16>(lo1)) << 16);
    o[8 + (j >> 1)] = to_bits<BF16>(hi0) | (static_cast<uint32_t>(to_bits<BF16>(hi1)) << 16);
  }
  uint4* dst = reinterpret_cast<uint4*>(out + blk * 32);
#pragma unroll
  for (int i = 0; i < 4; ++i) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
}

// One CTA per row of S (row r of group (b, hkv): query head hkv*G + r / Sq, query i = r % Sq):
// keys j > q_pos_offset + i are masked when causal; P = e^(s - max) / sum, rounded to the dtype.
template <bool BF16>
__global__ void __launch_bounds__(256) softmax_kernel(const float* __restrict__ S,
                                                      uint16_t* __restrict__ P, int Sq, int Sk,
                                                      int q_pos_offset, int causal) {
  const int64_t row = blockIdx.x;
  const int i = static_cast<int>(row % Sq);
  const int lim = causal ? min(Sk, q_pos_offset + i + 1) : Sk;  // visible keys [0, lim)
  const float* s = S + row * Sk;
  uint16_t* p = P + row * Sk;
  __shared__ float red[8];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float m = -INFINITY;
  for (int j = tid; j < lim; j += 256) m = fmaxf(m, s[j]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  m = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) m = fmaxf(m, red[w]);
  __syncthreads();
  float l = 0.f;
  for (int j = tid; j < lim; j += 256) l += __expf(s[j] - m);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
  if (lane == 0) red[warp] = l;
  __syncthreads();
  l = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) l += red[w];
  const float inv = 1.f / l;
  for (int j = tid; j < Sk; j += 256) p[j] = to_bits<BF16>(j < lim ? __expf(s[j] - m) * inv : 0.f);
}

// one cuBLAS handle per device, created on first use (the library never destroys it)
cublasHandle_t handle_for_current_device() {
  static std::mutex mu;
  static cublasHandle_t handles[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> g(mu);
  if (!handles[dev] && cublasCreate(&handles[dev]) != CUBLAS_STATUS_SUCCESS) handles[dev] = nullptr;
  return handles[dev];
}

}  // namespace

size_t explicit_workspace(int B, int Hq, int Hkv, int Sq, int Sk, int D, bool kq4, bool vq4) {
  auto al = [](size_t n) { return (n + 255) / 256 * 256; };
  const size_t rows = static_cast<size_t>(B) * Hq * Sq;
  size_t n = al(rows * Sk * sizeof(float)) + al(rows * Sk * 2);  // S (f32), P (dtype)
  const size_t kv = static_cast<size_t>(B) * Hkv * Sk * D * 2;
  if (kq4) n += al(kv);
  if (vq4) n += al(kv);
  return n;
}

cudaError_t explicit_launch(const ExplicitLaunch& L, cudaStream_t stream, int* cublas_status) {
  *cublas_status = 0;
  auto al = [](size_t n) { return (n + 255) / 256 * 256; };
  const int G = L.Hq / L.Hkv;
  const size_t rows = static_cast<size_t>(L.B) * L.Hq * L.Sq;
  uint8_t* ws = static_cast<uint8_t*>(L.workspace);
  float* S = reinterpret_cast<float*>(ws);
  ws += al(rows * L.Sk * sizeof(float));
  uint16_t* P = reinterpret_cast<uint16_t*>(ws);
  ws += al(rows * L.Sk * 2);
  const size_t kv = static_cast<size_t>(L.B) * L.Hkv * L.Sk * L.D;
  const int64_t nblocks = static_cast<int64_t>(kv / 32);
  const unsigned dq_grid = static_cast<unsigned>((nblocks + 255) / 256);
  const void* K = L.k;
  const void* V = L.v;
  auto dequant = [&](const void* q4, uint16_t* out) {
    const uint8_t* nib = static_cast<const uint8_t*>(q4);
    const __half* sc = reinterpret_cast<const __half*>(nib + L.scale_offset);
    if (L.bf16)
      dequant_kernel<true><<<dq_grid, 256, 0, stream>>>(nib, sc, out, nblocks);
    else
      dequant_kernel<false><<<dq_grid, 256, 0, stream>>>(nib, sc, out, nblocks);
  };
  if (L.kq4) {
    uint16_t* kd = reinterpret_cast<uint16_t*>(ws);
    ws += al(kv * 2);
    dequant(L.k, kd);
    K = kd;
  }
  if (L.vq4) {
    uint16_t* vd = reinterpret_cast<uint16_t*>(ws);
    ws += al(kv * 2);
    dequant(L.v, vd);
    V = vd;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cublasHandle_t h = handle_for_current_device();
  if (!h) {
    *cublas_status = 1;
    return cudaSuccess;
  }
  const cudaDataType_t dt = L.bf16 ? CUDA_R_16BF : CUDA_R_16F;
  const int M = G * L.Sq;  // rows of a (batch, kv head) group
  const int batch = L.B * L.Hkv;
  cublasStatus_t st = cublasSetStream(h, stream);
  // S^T (col-major Sk x M) = K (Sk x D, from row-major K: op T) * Q_g^T (D x M)
  const float alpha = L.scale, beta = 0.f;
  if (st == CUBLAS_STATUS_SUCCESS)
    st = cublasGemmStridedBatchedEx(
        h, CUBLAS_OP_T, CUBLAS_OP_N, L.Sk, M, L.D, &alpha, K, dt, L.D,
        static_cast<long long>(L.Sk) * L.D, L.q, dt, L.D, static_cast<long long>(M) * L.D, &beta,
        S, CUDA_R_32F, L.Sk, static_cast<long long>(M) * L.Sk, batch, CUBLAS_COMPUTE_32F,
        CUBLAS_GEMM_DEFAULT);
  if (st != CUBLAS_STATUS_SUCCESS) {
    *cublas_status = static_cast<int>(st);
    return cudaSuccess;
  }
  if (L.bf16)
    softmax_kernel<true><<<static_cast<unsigned>(rows), 256, 0, stream>>>(
        S, P, L.Sq, L.Sk, L.q_pos_offset, L.causal);
  else
    softmax_kernel<false><<<static_cast<unsigned>(rows), 256, 0, stream>>>(
        S, P, L.Sq, L.Sk, L.q_pos_offset, L.causal);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // O^T (col-major D x M) = V^T (D x Sk, row-major V read as is) * P_g^T (Sk x M)
  const float one = 1.f;
  st = cublasGemmStridedBatchedEx(
      h, CUBLAS_OP_N, CUBLAS_OP_N, L.D, M, L.Sk, &one, V, dt, L.D,
      static_cast<long long>(L.Sk) * L.D, P, dt, L.Sk, static_cast<long long>(M) * L.Sk, &beta,
      L.o, dt, L.D, static_cast<long long>(M) * L.D, batch, CUBLAS_COMPUTE_32F,
      CUBLAS_GEMM_DEFAULT);
  if (st != CUBLAS_STATUS_SUCCESS) *cublas_status = static_cast<int>(st);
  return cudaSuccess;
}

}  // namespace fa
