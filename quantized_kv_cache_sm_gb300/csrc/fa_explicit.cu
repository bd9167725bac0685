// The explicit (non-flash) attention path, for comparison with the fused kernels: K and V are
// expanded to dense f16/bf16 when they are q4_0, S = scale * Q K^T is written out in f32 by a
// batched GEMM, a softmax kernel turns each row of S into P (causal mask, max, exp, normalise,
// rounded to the input dtype), and O = P V is a second batched GEMM.  This is Approach C of
// "FlashAttention on gfx90a: Why It's Broken and How to Fix It" (Approach C: dequantize K and V
// to f16, then two GEMMs and a softmax) and the "explicit f32 matmul + softmax + matmul"
// reference of "perf(rocm): defer SDPA accumulator rescale, stage Q once per block (#2306)" (Test
// plan).  Every step runs in kernels of this file; both GEMMs are one tcgen05 kernel.
//
// Grouped-query heads: the G = Hq / Hkv query heads of a kv head are consecutive rows of Q, so
// one GEMM per (batch, kv head) computes their scores against that kv head's keys at once:
// S_g [G*Sq, Sk] = Q_g [G*Sq, D] K^T [D, Sk]; O_g [G*Sq, D] = P_g [G*Sq, Sk] V [Sk, D].
// S and P rows are padded to Skp = Sk rounded up to 64 (the GEMM's K step), so that every row of
// P starts on a 16-byte boundary for the tensor-memory-access loads; the padding of P is zero.
//
// The GEMM (gemm_kernel): one CTA computes a 128 x BN tile of C = alpha * A B for one group.
// A [M, K] is K-major (Q, or P); B is K-major (K: [N = keys, K = D]) or MN-major (V: [K = keys,
// N = D]).  Warp 0 streams 64-wide K slices of A and B into a ring of shared-memory stages by TMA
// (128-byte swizzle), warp 1 issues tcgen05.mma (M 128, N = BN, K 16; f32 accumulator in tensor
// memory), then all four warps read the accumulator back (one row per thread) and store it.
// Causal masking is exact in the softmax kernel; the GEMMs only skip work that the mask makes
// irrelevant: S tiles whose keys lie past every row's last visible key are not computed (the
// softmax never reads them), and the P V GEMM stops its K loop at the tile's last visible key
// (P is zero beyond it).
#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

__device__ uint32_t g_explicit_error;

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
// keys j > q_pos_offset + i are masked when causal; P = e^(s - max) / sum, rounded to the dtype;
// P is zero at masked keys and in the row padding [Sk, Skp).
template <bool BF16>
__global__ void __launch_bounds__(256) softmax_kernel(const float* __restrict__ S,
                                                      uint16_t* __restrict__ P, int Sq, int Sk,
                                                      int Skp, int q_pos_offset, int causal) {
  const int64_t row = blockIdx.x;
  const int i = static_cast<int>(row % Sq);
  const int lim = causal ? min(Sk, q_pos_offset + i + 1) : Sk;  // visible keys [0, lim)
  const float* s = S + row * Skp;
  uint16_t* p = P + row * Skp;
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
  for (int j = tid; j < Skp; j += 256) p[j] = to_bits<BF16>(j < lim ? __expf(s[j] - m) * inv : 0.f);
}

// The same row softmax with the row held in registers: one read of S and one write of P per
// element (the kernel above reads S three times).  kVpt values per thread, thread j holding
// columns j, j + threads, ...; used when Skp <= kVpt * 1024.
constexpr int kVpt = 32;
template <bool BF16>
__global__ void __launch_bounds__(1024) softmax_regs_kernel(const float* __restrict__ S,
                                                            uint16_t* __restrict__ P, int Sq,
                                                            int Sk, int Skp, int q_pos_offset,
                                                            int causal) {
  const int64_t row = blockIdx.x;
  const int i = static_cast<int>(row % Sq);
  const int lim = causal ? min(Sk, q_pos_offset + i + 1) : Sk;  // visible keys [0, lim)
  const float* s = S + row * Skp;
  uint16_t* p = P + row * Skp;
  __shared__ float red[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nt = blockDim.x;
  const int nwarps = nt >> 5;
  float v[kVpt];
  float m = -INFINITY;
#pragma unroll
  for (int k = 0; k < kVpt; ++k) {
    const int j = tid + k * nt;
    v[k] = (j < lim) ? __ldcs(s + j) : -INFINITY;  // S is read once: streaming loads
    m = fmaxf(m, v[k]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  m = red[0];
  for (int w = 1; w < nwarps; ++w) m = fmaxf(m, red[w]);
  __syncthreads();
  float l = 0.f;
#pragma unroll
  for (int k = 0; k < kVpt; ++k) {
    v[k] = __expf(v[k] - m);  // 0 at masked keys
    l += v[k];
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
  if (lane == 0) red[warp] = l;
  __syncthreads();
  l = 0.f;
  for (int w = 0; w < nwarps; ++w) l += red[w];
  const float inv = 1.f / l;
#pragma unroll
  for (int k = 0; k < kVpt; ++k) {
    const int j = tid + k * nt;
    if (j < Skp) p[j] = to_bits<BF16>(v[k] * inv);
  }
}

// ------------------------------------------------------------------------------------------
// tcgen05 GEMM
// ------------------------------------------------------------------------------------------
constexpr int kGM = 128;      // rows of a C tile (the MMA's M)
constexpr int kGK = 64;       // K slice per stage: one 128-byte swizzle atom of 16-bit values
constexpr int kGStages = 3;   // 3 x 32 KB: two CTAs fit on an SM
constexpr int kGThreads = 128;

template <int BN>
struct GCfg {
  static constexpr int kABytes = kGM * kGK * 2;       // 16 KB
  static constexpr int kBBytes = BN * kGK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kOffBar = kGStages * kStageBytes;
  static constexpr int kSmemBytes = kOffBar + 256 + 1024;  // barriers, slots, alignment slack
  static constexpr uint32_t kTmemCols = BN < 32 ? 32 : BN;
};

struct GemmArgs {
  void* c;              // C [groups][M][ldc]: f32 (S) or 16-bit (O)
  int64_t ldc;          // elements per row of C
  int64_t c_group;      // elements per group of C
  int M, N, K;          // per group; N: columns of C written (S: Skp; O: D)
  float alpha;
  // causal skipping: C row r of a group is query i = r % Sq, whose last visible key is
  // q_pos_offset + i (non-causal: all keys)
  int Sq, q_pos_offset, causal;
  int k_is_keys;        // 1: the K dimension runs over keys (P V), 0: the N dimension does (Q K^T)
};

// largest query index among C rows [m0, m0 + 128) of a group
__device__ __forceinline__ int tile_i_max(const GemmArgs& a, int m0) {
  const int m_last = min(m0 + kGM, a.M) - 1;
  // the tile lies within one head's rows unless it crosses a multiple of Sq
  if (m0 / a.Sq == m_last / a.Sq) return m_last % a.Sq;
  return a.Sq - 1;
}

template <int BN, bool BF16, bool B_MN, bool OUT_F32>
__global__ void __launch_bounds__(kGThreads) gemm_kernel(const __grid_constant__ CUtensorMap tm_a,
                                                         const __grid_constant__ CUtensorMap tm_b,
                                                         const __grid_constant__ CUtensorMap tm_c,
                                                         const GemmArgs args) {
  using C = GCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - smem_u32(smem_raw));
  const uint32_t bar0 = sbase + C::kOffBar;
  auto full = [&](int s) -> uint32_t { return bar0 + 8u * s; };
  auto empty = [&](int s) -> uint32_t { return bar0 + 8u * (kGStages + s); };
  const uint32_t acc_full = bar0 + 8u * (2 * kGStages);
  const uint32_t drain = bar0 + 8u * (2 * kGStages + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sgen + C::kOffBar + 128);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + C::kOffBar + 136);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = static_cast<int>(blockIdx.x) * BN;
  const int m0 = static_cast<int>(blockIdx.y) * kGM;
  const int grp = static_cast<int>(blockIdx.z);

  // the work the causal mask leaves for this tile (uniform over the CTA: decided before any
  // barrier or tensor-memory allocation)
  int k_end = args.K;
  if (args.causal) {
    const int last_key = args.q_pos_offset + tile_i_max(args, m0);
    if (args.k_is_keys)
      k_end = min(args.K, last_key + 1);
    else if (n0 > last_key)
      return;  // every score of this tile is masked: the softmax never reads it
  }
  const int nk = (k_end + kGK - 1) / kGK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  bool ok = true;
  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_b);
    int issued = 0;
    for (int kb = 0; kb < nk && ok; ++kb) {
      const int s = kb % kGStages;
      if (kb >= kGStages)
        ok = mbar_wait(empty(s), ((kb / kGStages) - 1) & 1, abort_flag, &g_explicit_error);
      if (!ok) break;
      ++issued;
      const uint32_t a_dst = sbase + s * C::kStageBytes;
      const uint32_t b_dst = a_dst + C::kABytes;
      mbar_arrive_expect_tx(full(s), C::kStageBytes);
      tma_load_3d(a_dst, &tm_a, full(s), kb * kGK, m0, grp);
      if (B_MN) {
        // [K rows = keys][N = BN columns] as BN/64 boxes of 64 columns x 64 keys
#pragma unroll
        for (int c = 0; c < BN / 64; ++c)
          tma_load_3d(b_dst + c * (kGK * 128), &tm_b, full(s), n0 + c * 64, kb * kGK, grp);
      } else {
        tma_load_3d(b_dst, &tm_b, full(s), kb * kGK, n0, grp);
      }
    }
    if (!ok) {
      // let the copies already issued land before shared memory goes away
      volatile int never = 0;
      for (int kb = max(0, issued - kGStages); kb < issued; ++kb)
        mbar_wait(full(kb % kGStages), (kb / kGStages) & 1, &never, nullptr, kWaitLimitNs);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = make_idesc_f16(kGM, BN, BF16, B_MN);
    for (int kb = 0; kb < nk && ok; ++kb) {
      const int s = kb % kGStages;
      ok = mbar_wait(full(s), (kb / kGStages) & 1, abort_flag, &g_explicit_error);
      if (!ok) break;
      tc_fence_after();
      const uint32_t a_s = sbase + s * C::kStageBytes;
      const uint32_t b_s = a_s + C::kABytes;
#pragma unroll
      for (int kk = 0; kk < kGK / 16; ++kk) {
        const uint64_t ad = make_sdesc_sw128(a_s + kk * 32, 16, 1024);
        const uint64_t bd = B_MN ? make_sdesc_sw128(b_s + kk * (16 * 128), kGK * 128, 1024)
                                 : make_sdesc_sw128(b_s + kk * 32, 16, 1024);
        mma_ss(tmem, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
      }
      mma_commit(empty(s));
    }
    if (ok) {
      mma_commit(acc_full);
    } else {
      volatile int never = 0;
      mma_commit(drain);
      mbar_wait(drain, 0, &never, nullptr, kWaitLimitNs);
    }
  }
  __syncwarp();

  // ---------------------------------------------------------------- epilogue, all four warps
  ok = !*abort_flag && mbar_wait(acc_full, 0, abort_flag, &g_explicit_error);
  ok = __syncthreads_and(ok) != 0;  // the epilogue's barriers need every thread, or none
  if (ok) {
    tc_fence_after();
    const int row = m0 + 32 * warp + lane;
    const bool store = row < args.M;
    const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * warp) << 16);
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(taddr + c0, r);
      tmem_wait_ld();
      reg_fence32(r);
      if (OUT_F32) {
        // f32 tile: 32 columns of the 128 rows go to shared memory (128-byte swizzle: a row's
        // 16-byte chunk c sits at chunk c ^ (row % 8), conflict-free for one row per thread)
        // and leave by one tensor store, two buffers alternating; the ring is idle by now
        const int buf = (c0 / 32) & 1;
        const uint32_t sbuf = sbase + buf * (kGM * 128);
        if (c0 >= 64) {
          // the store issued from this buffer two chunks ago has read it
          if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
          asm volatile("bar.sync 1, %0;" ::"n"(kGThreads) : "memory");
        }
        const int rl = 32 * warp + lane;  // row within the tile
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t a = sbuf + rl * 128 + ((i ^ (rl & 7)) << 4);
          asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a),
                       "f"(__uint_as_float(r[4 * i]) * args.alpha),
                       "f"(__uint_as_float(r[4 * i + 1]) * args.alpha),
                       "f"(__uint_as_float(r[4 * i + 2]) * args.alpha),
                       "f"(__uint_as_float(r[4 * i + 3]) * args.alpha)
                       : "memory");
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("bar.sync 1, %0;" ::"n"(kGThreads) : "memory");
        if (threadIdx.x == 0 && n0 + c0 < args.N) {
          // rows past M and columns past N are clipped by the tensor store
          asm volatile(
              "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];"
              ::"l"(reinterpret_cast<uint64_t>(&tm_c)), "r"(n0 + c0), "r"(m0), "r"(grp),
              "r"(sbuf)
              : "memory");
          asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
        continue;
      }
      if (!store || n0 + c0 >= args.N) continue;
      {
        uint16_t* dst =
            static_cast<uint16_t*>(args.c) + grp * args.c_group + row * args.ldc + n0 + c0;
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack2<BF16>(__uint_as_float(r[2 * i]) * args.alpha,
                              __uint_as_float(r[2 * i + 1]) * args.alpha);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          reinterpret_cast<uint4*>(dst)[i] =
              make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
      }
    }
  }
  if (OUT_F32 && threadIdx.x == 0)
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");  // the tile's stores are done
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int BN, bool BF16, bool B_MN, bool OUT_F32>
cudaError_t gemm_launch(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                        const GemmArgs& a, int groups, cudaStream_t stream) {
  using C = GCfg<BN>;
  auto kern = gemm_kernel<BN, BF16, B_MN, OUT_F32>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const dim3 grid((a.N + BN - 1) / BN, (a.M + kGM - 1) / kGM, groups);
  kern<<<grid, kGThreads, C::kSmemBytes, stream>>>(ta, tb, tc, a);
  return cudaGetLastError();
}

size_t align256(size_t n) { return (n + 255) / 256 * 256; }
int padded_keys(int Sk) { return (Sk + kGK - 1) / kGK * kGK; }

}  // namespace

size_t explicit_workspace(int B, int Hq, int Hkv, int Sq, int Sk, int D, bool kq4, bool vq4) {
  const size_t rows = static_cast<size_t>(B) * Hq * Sq;
  const size_t skp = static_cast<size_t>(padded_keys(Sk));
  size_t n = align256(rows * skp * sizeof(float)) + align256(rows * skp * 2);  // S (f32), P
  const size_t kv = static_cast<size_t>(B) * Hkv * Sk * D * 2;
  if (kq4) n += align256(kv);
  if (vq4) n += align256(kv);
  return n;
}

cudaError_t explicit_launch(const ExplicitLaunch& L, cudaStream_t stream, int* map_status) {
  *map_status = 0;
  const int G = L.Hq / L.Hkv;
  const int Skp = padded_keys(L.Sk);
  const size_t rows = static_cast<size_t>(L.B) * L.Hq * L.Sq;
  uint8_t* ws = static_cast<uint8_t*>(L.workspace);
  float* S = reinterpret_cast<float*>(ws);
  ws += align256(rows * Skp * sizeof(float));
  uint16_t* P = reinterpret_cast<uint16_t*>(ws);
  ws += align256(rows * Skp * 2);
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
    ws += align256(kv * 2);
    dequant(L.k, kd);
    K = kd;
  }
  if (L.vq4) {
    uint16_t* vd = reinterpret_cast<uint16_t*>(ws);
    ws += align256(kv * 2);
    dequant(L.v, vd);
    V = vd;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  const int M = G * L.Sq;  // rows of a (batch, kv head) group
  const int groups = L.B * L.Hkv;
  const CUtensorMapDataType tdt =
      L.bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
  // S = scale Q_g K^T: A = Q_g [M][D], B = K [Sk][D] (K-major), C = S [M][Skp] f32; tiles of
  // 128 keys, the last one covering the padding
  CUtensorMap tq, tk, tp, tv, ts;
  if (!encode_map_3d(&ts, S, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, Skp, M, groups, 32, kGM, sw) ||
      !encode_map_3d(&tq, L.q, tdt, 2, L.D, M, groups, kGK, kGM, sw) ||
      !encode_map_3d(&tk, K, tdt, 2, L.D, L.Sk, groups, kGK, 128, sw) ||
      !encode_map_3d(&tp, P, tdt, 2, Skp, M, groups, kGK, kGM, sw) ||
      !encode_map_3d(&tv, V, tdt, 2, L.D, L.Sk, groups, 64, kGK, sw)) {
    *map_status = 1;
    return cudaSuccess;
  }
  GemmArgs ga;
  ga.c = S;
  ga.ldc = Skp;
  ga.c_group = static_cast<int64_t>(M) * Skp;
  ga.M = M;
  ga.N = Skp;
  ga.K = L.D;
  ga.alpha = L.scale;
  ga.Sq = L.Sq;
  ga.q_pos_offset = L.q_pos_offset;
  ga.causal = L.causal;
  ga.k_is_keys = 0;
  e = L.bf16 ? gemm_launch<128, true, false, true>(tq, tk, ts, ga, groups, stream)
             : gemm_launch<128, false, false, true>(tq, tk, ts, ga, groups, stream);
  if (e != cudaSuccess) return e;
  if (Skp <= kVpt * 1024) {
    // one warp per 32 x kVpt columns (Skp is a multiple of 64)
    const int nt = (Skp + kVpt * 32 - 1) / (kVpt * 32) * 32;
    if (L.bf16)
      softmax_regs_kernel<true><<<static_cast<unsigned>(rows), nt, 0, stream>>>(
          S, P, L.Sq, L.Sk, Skp, L.q_pos_offset, L.causal);
    else
      softmax_regs_kernel<false><<<static_cast<unsigned>(rows), nt, 0, stream>>>(
          S, P, L.Sq, L.Sk, Skp, L.q_pos_offset, L.causal);
  } else if (L.bf16) {
    softmax_kernel<true><<<static_cast<unsigned>(rows), 256, 0, stream>>>(
        S, P, L.Sq, L.Sk, Skp, L.q_pos_offset, L.causal);
  } else {
    softmax_kernel<false><<<static_cast<unsigned>(rows), 256, 0, stream>>>(
        S, P, L.Sq, L.Sk, Skp, L.q_pos_offset, L.causal);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // O_g = P_g V: A = P_g [M][Skp], B = V [Sk][D] (MN-major; keys past Sk read as zeros, where
  // P is zero too), C = O_g [M][D] in the dtype
  GemmArgs go = ga;
  go.c = L.o;
  go.ldc = L.D;
  go.c_group = static_cast<int64_t>(M) * L.D;
  go.N = L.D;
  go.K = Skp;
  go.alpha = 1.f;
  go.k_is_keys = 1;
  // (the O GEMM writes with plain stores: its tensor-store map is unused)
  if (L.D == 128)
    return L.bf16 ? gemm_launch<128, true, true, false>(tp, tv, ts, go, groups, stream)
                  : gemm_launch<128, false, true, false>(tp, tv, ts, go, groups, stream);
  return L.bf16 ? gemm_launch<64, true, true, false>(tp, tv, ts, go, groups, stream)
                : gemm_launch<64, false, true, false>(tp, tv, ts, go, groups, stream);
}

uint32_t explicit_take_error() {
  uint32_t v = 0;
  if (cudaMemcpyFromSymbol(&v, g_explicit_error, sizeof(v)) != cudaSuccess) return 0xffffffffu;
  const uint32_t z = 0;
  cudaMemcpyToSymbol(g_explicit_error, &z, sizeof(z));
  return v;
}

}  // namespace fa
