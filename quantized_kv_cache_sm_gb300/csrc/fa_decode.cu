// Split-K decode (one query token per sequence) for sm_103a, dense or q4_0 K/V cache.
//
// Decode reads the whole K/V cache once per token, so it is bound by HBM bandwidth, not by the
// tensor cores (the pages' decode figures, "FlashAttention on gfx90a: Why It's Broken and How to
// Fix It", The Problem table, are where flash attention lost most).  The design follows that:
//
//  * grid = (split, kv head, batch); every CTA streams one contiguous key range of one kv head
//    through a ring of shared-memory stages (TMA for nibble / dense tiles, cp.async for the fp16
//    scale rows), and all query heads of the GQA group are served from that single read;
//  * the two contractions are tiny (N = group size <= 8), so they run on mma.sync m16n8k16 with
//    the *keys* as the M dimension: S^T = K Q^T and O^T += V^T P^T.  The q4_0 nibbles go straight
//    from shared memory into MMA fragment registers (ldmatrix, LOP3 + HSUB2 to exact (q - 8));
//    the per-block fp16 scales are applied in f32 on the accumulator for K and folded into P for
//    V, so no dequantized tile is ever written back;
//  * each consumer warp keeps its own online softmax state; the warps of a CTA merge through
//    shared memory and write one partial (m, l, unnormalised O) per query head and split;
//  * a combine kernel merges the splits: M = max m_s, O = sum e^(m_s - M) O_s / sum e^(m_s - M) l_s.
#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

__device__ uint32_t g_decode_error;

namespace {

constexpr int kTileKeys = 64;      // keys per stage
constexpr int kConsumers = 4;      // consumer warps, 16 keys of every tile each
constexpr float kLog2e = 1.4426950408889634f;

template <int D, bool Q4>
struct DCfg {
  static constexpr int kNibBytes = kTileKeys * D / 2;            // q4_0 nibble tile
  static constexpr int kScaleBytes = kTileKeys * (D / 32) * 2;   // q4_0 scale rows
  static constexpr int kDenseBytes = kTileKeys * D * 2;          // f16/bf16 tile
  static constexpr int kKBytes = Q4 ? kNibBytes : kDenseBytes;
  // stage: K tile | V tile | K scales | V scales, each region 1024-byte aligned
  static constexpr int kOffV = (kKBytes + 1023) / 1024 * 1024;
  static constexpr int kOffKs = kOffV + (kKBytes + 1023) / 1024 * 1024;
  static constexpr int kOffVs = kOffKs + (Q4 ? kScaleBytes : 0);
  static constexpr int kStageBytes = ((kOffVs + (Q4 ? kScaleBytes : 0)) + 1023) / 1024 * 1024;
  static constexpr int kStages = Q4 ? (D == 128 ? 5 : 8) : (D == 128 ? 3 : 5);
  static constexpr int kCtasPerSm = Q4 ? 4 : 2;
  static constexpr int kOffBar = kStages * kStageBytes;
  static constexpr int kSmemBytes = kOffBar + 256 + 1024;
  static constexpr int kThreads = 32 * (1 + kConsumers);
  static constexpr int kPartStride = D + 4;  // m, l, pad, pad, O[D]
  // cross-warp merge buffer (reuses the stages): per warp 8 heads x (D + 2) floats
  static_assert(kConsumers * 8 * (D + 2) * 4 <= kStages * kStageBytes, "merge buffer");
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
template <bool BF16>
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  if (BF16)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// nibble pairs -> exact (q - 8) pairs, in the input dtype
template <bool BF16>
__device__ __forceinline__ uint32_t nib_lo(uint32_t w) {
  uint32_t x = (w & 0x000F000Fu) | (BF16 ? 0x43004300u : 0x64006400u);
  if (BF16) {
    const uint32_t c = 0x43084308u;
    __nv_bfloat162 r = __hsub2(*reinterpret_cast<__nv_bfloat162*>(&x),
                               *reinterpret_cast<const __nv_bfloat162*>(&c));
    return *reinterpret_cast<uint32_t*>(&r);
  } else {
    const uint32_t c = 0x64086408u;
    __half2 r = __hsub2(*reinterpret_cast<__half2*>(&x), *reinterpret_cast<const __half2*>(&c));
    return *reinterpret_cast<uint32_t*>(&r);
  }
}
template <bool BF16>
__device__ __forceinline__ uint32_t nib_hi(uint32_t w) {
  if (BF16) {
    // bf16 has 7 mantissa bits: a high nibble at bits 4-7 would reach the exponent
    return nib_lo<true>(w >> 4);
  } else {
    uint32_t x = (w & 0x00F000F0u) | 0x64006400u;     // 1024 + 16 n
    const uint32_t s = 0x2C002C00u, c = 0xD480D480u;  // 1/16, -72
    __half2 r = __hfma2(*reinterpret_cast<__half2*>(&x), *reinterpret_cast<const __half2*>(&s),
                        *reinterpret_cast<const __half2*>(&c));
    return *reinterpret_cast<uint32_t*>(&r);
  }
}

struct DecodeArgs {
  const uint16_t* q;
  const uint8_t* k_scale;
  const uint8_t* v_scale;
  float* partial;
  int Hq, Hkv, Sk, Sk_eff, nsplit, chunk;
  float scale_log2;
};

template <int D, bool BF16, bool Q4>
__global__ void __launch_bounds__(DCfg<D, Q4>::kThreads, DCfg<D, Q4>::kCtasPerSm)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const DecodeArgs args) {
  using C = DCfg<D, Q4>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - smem_u32(smem_raw));
  const uint32_t bar_full = sbase + C::kOffBar;
  const uint32_t bar_empty = bar_full + 8 * C::kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + C::kOffBar + 16 * C::kStages);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  const int hkv = blockIdx.y;
  const int b = blockIdx.z;
  const int G = args.Hq / args.Hkv;
  const int kb0 = split * args.chunk;
  const int kb1 = min(args.Sk_eff, kb0 + args.chunk);
  const int ntiles = (kb1 - kb0 + kTileKeys - 1) / kTileKeys;
  const int64_t bh = static_cast<int64_t>(b) * args.Hkv + hkv;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar_full + 8 * s, Q4 ? 1 + 32 : 1);
      mbar_init(bar_empty + 8 * s, kConsumers);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
    }
    bool ok = true;
    int n = 0;
    for (; n < ntiles; ++n) {
      const int s = n % C::kStages;
      if (n >= C::kStages) {
        if (lane == 0)
          ok = mbar_wait(bar_empty + 8 * s, ((n / C::kStages) - 1) & 1, abort_flag,
                         &g_decode_error);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
      }
      const int key0 = kb0 + n * kTileKeys;
      const uint32_t st = sbase + s * C::kStageBytes;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar_full + 8 * s, 2 * C::kKBytes);
        if (Q4) {
          tma_load_3d(st, &tm_k, bar_full + 8 * s, 0, key0, static_cast<int>(bh));
          tma_load_3d(st + C::kOffV, &tm_v, bar_full + 8 * s, 0, key0, static_cast<int>(bh));
        } else {
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            tma_load_3d(st + c * (kTileKeys * 128), &tm_k, bar_full + 8 * s, 64 * c, key0,
                        static_cast<int>(bh));
            tma_load_3d(st + C::kOffV + c * (kTileKeys * 128), &tm_v, bar_full + 8 * s, 64 * c,
                        key0, static_cast<int>(bh));
          }
        }
      }
      if (Q4) {
        constexpr int kRow = (D / 32) * 2;  // scale bytes per key
        for (int i = lane; i < 2 * kTileKeys; i += 32) {
          const bool is_v = i >= kTileKeys;
          const int r = is_v ? i - kTileKeys : i;
          const int key = key0 + r;
          const bool in = key < args.Sk;
          const uint8_t* src =
              (is_v ? args.v_scale : args.k_scale) + (bh * args.Sk + (in ? key : 0)) * kRow;
          const uint32_t dst = st + (is_v ? C::kOffVs : C::kOffKs) + r * kRow;
          if (kRow == 8)
            cp_async_8(dst, src, in ? 8u : 0u);
          else
            cp_async_4(dst, src, in ? 4u : 0u);
        }
        cp_async_mbar_arrive_noinc(bar_full + 8 * s);
      }
    }
    if (!ok && lane == 0) {
      volatile int never = 0;
      for (int i = max(0, n - C::kStages); i < n; ++i)
        mbar_wait(bar_full + 8 * (i % C::kStages), (i / C::kStages) & 1, &never, nullptr);
    }
    return;  // the producer takes no part in the merge
  }

  // -------------------------------------------------------------- consumers
  const int cw = warp - 1;  // 0..3
  const int g8 = lane >> 2;  // fragment row group
  const int t4 = lane & 3;   // fragment column pair
  const float sl2 = args.scale_log2;

  // Q^T as mma B fragments (k = head dim, n = query head of the group), loaded once.
  // q4_0 uses a permutation of the head dimension that matches the nibble layout (see below).
  uint32_t qf[D / 16][2];
  {
    const int hq = hkv * G + g8;
    const uint16_t* qrow = args.q + (static_cast<int64_t>(b) * args.Hq + hq) * D;
    const bool valid = g8 < G;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      int d0, d1, d2, d3;
      if (Q4) {
        // k-step kk = (block kk/2, nibble half kk%2): fragment column 2t+e <-> element
        // 16*kk + 4t + 2e, column 2t+8+e <-> element 16*kk + 4t + 1 + 2e
        d0 = 16 * kk + 4 * t4;
        d1 = d0 + 2;
        d2 = d0 + 1;
        d3 = d0 + 3;
      } else {
        d0 = 16 * kk + 2 * t4;
        d1 = d0 + 1;
        d2 = d0 + 8;
        d3 = d0 + 9;
      }
      const uint32_t e0 = valid ? qrow[d0] : 0u, e1 = valid ? qrow[d1] : 0u;
      const uint32_t e2 = valid ? qrow[d2] : 0u, e3 = valid ? qrow[d3] : 0u;
      qf[kk][0] = e0 | (e1 << 16);
      qf[kk][1] = e2 | (e3 << 16);
    }
  }

  // O^T accumulators: m-tile i covers 16 head-dim rows, columns = query heads 2t, 2t+1
  float o[D / 16][4];
#pragma unroll
  for (int i = 0; i < D / 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY;  // running max (base-2 scaled) for heads 2t, 2t+1
  float l0 = 0.f, l1 = 0.f;              // this thread's share of the row sums

  bool ok = true;
  for (int n = 0; n < ntiles; ++n) {
    const int s = n % C::kStages;
    if (lane == 0)
      ok = mbar_wait(bar_full + 8 * s, (n / C::kStages) & 1, abort_flag, &g_decode_error);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (!ok) break;
    const uint32_t st = sbase + s * C::kStageBytes;
    const int kl = 16 * cw;                        // this warp's first key in the tile
    const int keyg = kb0 + n * kTileKeys + kl + g8; // absolute key of fragment row g
    // ---------------- S^T = K Q^T (16 keys x 8 heads)
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
    if (Q4) {
      const __half* ks = reinterpret_cast<const __half*>(sgen + (st - sbase) + C::kOffKs);
      const int mi = lane >> 3, r = lane & 7;
#pragma unroll
      for (int bb = 0; bb < D / 32; bb += 2) {
        const int key = kl + (mi & 1) * 8 + r;
        const int blk = bb + (mi >> 1);
        const int chunk = (D == 128) ? (blk ^ ((key >> 1) & 3)) : (blk ^ ((key >> 2) & 1));
        uint32_t w[4];
        ldsm_x4(st + key * (D / 2) + chunk * 16, w[0], w[1], w[2], w[3]);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int blkk = bb + e;
          const uint32_t wg = w[2 * e], wg8 = w[2 * e + 1];
          float cb[4] = {0.f, 0.f, 0.f, 0.f};
          mma16816<BF16>(cb, nib_lo<BF16>(wg), nib_lo<BF16>(wg8), nib_lo<BF16>(wg >> 8),
                         nib_lo<BF16>(wg8 >> 8), qf[2 * blkk][0], qf[2 * blkk][1]);
          mma16816<BF16>(cb, nib_hi<BF16>(wg), nib_hi<BF16>(wg8), nib_hi<BF16>(wg >> 8),
                         nib_hi<BF16>(wg8 >> 8), qf[2 * blkk + 1][0], qf[2 * blkk + 1][1]);
          const float dg = __half2float(ks[(kl + g8) * (D / 32) + blkk]);
          const float dg8 = __half2float(ks[(kl + g8 + 8) * (D / 32) + blkk]);
          sc[0] = fmaf(cb[0], dg, sc[0]);
          sc[1] = fmaf(cb[1], dg, sc[1]);
          sc[2] = fmaf(cb[2], dg8, sc[2]);
          sc[3] = fmaf(cb[3], dg8, sc[3]);
        }
      }
    } else {
      const int mi = lane >> 3, r = lane & 7;
      const int key = kl + (mi & 1) * 8 + r;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int d0 = 16 * kk + (mi >> 1) * 8;
        const uint32_t addr =
            st + (d0 >> 6) * (kTileKeys * 128) + key * 128 + ((((d0 & 63) >> 3) ^ (key & 7)) << 4);
        uint32_t a0, a1, a2, a3;
        ldsm_x4(addr, a0, a1, a2, a3);
        mma16816<BF16>(sc, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
      }
    }
    // ---------------- online softmax over this warp's 16 keys
    const bool vg = keyg < kb1, vg8 = keyg + 8 < kb1;
    const float t0 = vg ? sc[0] * sl2 : -INFINITY;
    const float t1 = vg ? sc[1] * sl2 : -INFINITY;
    const float t2 = vg8 ? sc[2] * sl2 : -INFINITY;
    const float t3 = vg8 ? sc[3] * sl2 : -INFINITY;
    float mx0 = fmaxf(t0, t2), mx1 = fmaxf(t1, t3);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float nm0 = fmaxf(m0, mx0), nm1 = fmaxf(m1, mx1);
    const bool grow = (nm0 > m0) || (nm1 > m1);
    if (__any_sync(0xffffffffu, grow)) {
      const float a0 = (nm0 == -INFINITY) ? 1.f : ex2(m0 - nm0);
      const float a1 = (nm1 == -INFINITY) ? 1.f : ex2(m1 - nm1);
      l0 *= a0;
      l1 *= a1;
#pragma unroll
      for (int i = 0; i < D / 16; ++i) {
        o[i][0] *= a0;
        o[i][1] *= a1;
        o[i][2] *= a0;
        o[i][3] *= a1;
      }
      m0 = nm0;
      m1 = nm1;
    }
    const float b0 = (m0 == -INFINITY) ? 0.f : m0, b1 = (m1 == -INFINITY) ? 0.f : m1;
    const float p0 = ex2(t0 - b0), p1 = ex2(t1 - b1), p2 = ex2(t2 - b0), p3 = ex2(t3 - b1);
    l0 += p0 + p2;
    l1 += p1 + p3;
    // ---------------- O^T += V^T P^T
    if (Q4) {
      const __half* vs = reinterpret_cast<const __half*>(sgen + (st - sbase) + C::kOffVs);
      const int mi = lane >> 3, r = lane & 7;
      const uint32_t vbase = st + C::kOffV;
#pragma unroll
      for (int bb = 0; bb < D / 32; bb += 2) {
        const int key = kl + (mi & 1) * 8 + r;
        const int blk = bb + (mi >> 1);
        const int chunk = (D == 128) ? (blk ^ ((key >> 1) & 3)) : (blk ^ ((key >> 2) & 1));
        uint32_t w[4];
        ldsm_x4_t(vbase + key * (D / 2) + chunk * 16, w[0], w[1], w[2], w[3]);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int blkk = bb + e;
          const float dg = __half2float(vs[(kl + g8) * (D / 32) + blkk]);
          const float dg8 = __half2float(vs[(kl + g8 + 8) * (D / 32) + blkk]);
          // P scaled by this block's V scale, transposed into the B fragment (keys x heads)
          const uint32_t pb0 = movtrans(pack2<BF16>(p0 * dg, p1 * dg));
          const uint32_t pb1 = movtrans(pack2<BF16>(p2 * dg8, p3 * dg8));
          const uint32_t w1 = w[2 * e], w2 = w[2 * e + 1];
          // m-tile (block, low nibbles): rows g <-> element 2g, g+8 <-> element 2g+1
          mma16816<BF16>(o[2 * blkk], nib_lo<BF16>(w1), nib_lo<BF16>(w1 >> 8), nib_lo<BF16>(w2),
                         nib_lo<BF16>(w2 >> 8), pb0, pb1);
          // m-tile (block, high nibbles): rows g <-> element 16+2g, g+8 <-> element 17+2g
          mma16816<BF16>(o[2 * blkk + 1], nib_hi<BF16>(w1), nib_hi<BF16>(w1 >> 8),
                         nib_hi<BF16>(w2), nib_hi<BF16>(w2 >> 8), pb0, pb1);
        }
      }
    } else {
      const uint32_t pb0 = movtrans(pack2<BF16>(p0, p1));
      const uint32_t pb1 = movtrans(pack2<BF16>(p2, p3));
      const int mi = lane >> 3, r = lane & 7;
      const int key = kl + (mi >> 1) * 8 + r;
      const uint32_t vbase = st + C::kOffV;
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        const int d0 = 16 * mt + (mi & 1) * 8;
        const uint32_t addr = vbase + (d0 >> 6) * (kTileKeys * 128) + key * 128 +
                              ((((d0 & 63) >> 3) ^ (key & 7)) << 4);
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(addr, a0, a1, a2, a3);
        mma16816<BF16>(o[mt], a0, a1, a2, a3, pb0, pb1);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * s);
  }

  // ------------------------------------------------------------------ merge the 4 warps
  // full row sums of this warp's keys
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumers) : "memory");  // all tiles consumed
  if (*abort_flag) return;
  float* mb = reinterpret_cast<float*>(sgen);  // [warp][head][D + 2]: m, l, O[D]
  constexpr int kW = D + 2;
  {
    float* wbase = mb + cw * 8 * kW;
    if (g8 == 0) {
      wbase[(2 * t4) * kW + 0] = m0;
      wbase[(2 * t4) * kW + 1] = l0;
      wbase[(2 * t4 + 1) * kW + 0] = m1;
      wbase[(2 * t4 + 1) * kW + 1] = l1;
    }
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      int dr0, dr1;  // head-dim rows of accumulator rows g and g+8 of m-tile i
      if (Q4) {
        dr0 = 32 * (i >> 1) + 16 * (i & 1) + 2 * g8;
        dr1 = dr0 + 1;
      } else {
        dr0 = 16 * i + g8;
        dr1 = dr0 + 8;
      }
      wbase[(2 * t4) * kW + 2 + dr0] = o[i][0];
      wbase[(2 * t4 + 1) * kW + 2 + dr0] = o[i][1];
      wbase[(2 * t4) * kW + 2 + dr1] = o[i][2];
      wbase[(2 * t4 + 1) * kW + 2 + dr1] = o[i][3];
    }
  }
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumers) : "memory");
  const int tid = threadIdx.x - 32;  // 0..127
  for (int idx = tid; idx < G * (D + 2); idx += 32 * kConsumers) {
    const int hh = idx / (D + 2);
    const int c = idx % (D + 2);
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, mb[(w * 8 + hh) * kW]);
    float out;
    if (c == 0) {
      out = M;
    } else {
      float acc = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumers; ++w) {
        const float mw = mb[(w * 8 + hh) * kW];
        const float f = (mw == -INFINITY) ? 0.f : ex2(mw - M);
        acc += f * mb[(w * 8 + hh) * kW + c];
      }
      out = acc;
    }
    const int hq = hkv * G + hh;
    float* dst = args.partial +
                 ((static_cast<int64_t>(b) * args.Hq + hq) * args.nsplit + split) * C::kPartStride;
    dst[c == 0 ? 0 : (c == 1 ? 1 : c + 2)] = out;
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(128) decode_combine_kernel(const float* __restrict__ partial,
                                                             uint16_t* __restrict__ o, int nsplit) {
  constexpr int kStride = D + 4;
  const int64_t row = blockIdx.x;  // b * Hq + hq
  const float* p = partial + row * nsplit * kStride;
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, p[s * kStride]);
  float L = 0.f;
  for (int s = 0; s < nsplit; ++s) {
    const float ms = p[s * kStride];
    if (ms != -INFINITY) L += ex2(ms - M) * p[s * kStride + 1];
  }
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float acc = 0.f;
    for (int s = 0; s < nsplit; ++s) {
      const float ms = p[s * kStride];
      if (ms != -INFINITY) acc += ex2(ms - M) * p[s * kStride + 4 + d];
    }
    const float v = acc / L;
    o[row * D + d] = BF16 ? __bfloat16_as_ushort(__float2bfloat16_rn(v))
                          : __half_as_ushort(__float2half_rn(v));
  }
}

}  // namespace

void decode_plan(int B, int Hkv, int Sk_eff, int num_sms, int* nsplit, int* chunk) {
  // one wave of CTAs at the resident count of the q4_0 configuration, equal key chunks
  const int units = B * Hkv;
  const int slots = num_sms * 4;
  int ns = (slots + units / 2) / units;
  if (ns < 1) ns = 1;
  const int max_tiles = (Sk_eff + kTileKeys - 1) / kTileKeys;
  if (ns > max_tiles) ns = max_tiles;
  if (ns < 1) ns = 1;
  int ck = (Sk_eff + ns - 1) / ns;
  ck = (ck + kTileKeys - 1) / kTileKeys * kTileKeys;
  if (ck < kTileKeys) ck = kTileKeys;
  *chunk = ck;
  *nsplit = (Sk_eff + ck - 1) / ck;
}

template <int D, bool BF16, bool Q4>
static cudaError_t launch_t(const DecodeLaunch& L, cudaStream_t stream) {
  using C = DCfg<D, Q4>;
  auto kern = decode_split_kernel<D, BF16, Q4>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  DecodeArgs a;
  a.q = static_cast<const uint16_t*>(L.q);
  a.k_scale = static_cast<const uint8_t*>(L.k_scale);
  a.v_scale = static_cast<const uint8_t*>(L.v_scale);
  a.partial = L.partial;
  a.Hq = L.Hq;
  a.Hkv = L.Hkv;
  a.Sk = L.Sk;
  a.Sk_eff = L.Sk_eff;
  a.nsplit = L.nsplit;
  a.chunk = L.chunk;
  a.scale_log2 = L.scale * kLog2e;
  dim3 grid(L.nsplit, L.Hkv, L.B);
  kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(L.tm_k, L.tm_v, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_combine_kernel<D, BF16><<<L.B * L.Hq, 128, 0, stream>>>(
      L.partial, static_cast<uint16_t*>(L.o), L.nsplit);
  return cudaGetLastError();
}

cudaError_t decode_launch(const DecodeLaunch& L, cudaStream_t stream) {
  if (L.D == 128) {
    if (L.q4) return L.bf16 ? launch_t<128, true, true>(L, stream) : launch_t<128, false, true>(L, stream);
    return L.bf16 ? launch_t<128, true, false>(L, stream) : launch_t<128, false, false>(L, stream);
  }
  if (L.q4) return L.bf16 ? launch_t<64, true, true>(L, stream) : launch_t<64, false, true>(L, stream);
  return L.bf16 ? launch_t<64, true, false>(L, stream) : launch_t<64, false, false>(L, stream);
}

uint32_t decode_take_error() {
  uint32_t v = 0;
  if (cudaMemcpyFromSymbol(&v, g_decode_error, sizeof(v)) != cudaSuccess) return 0xffffffffu;
  const uint32_t z = 0;
  cudaMemcpyToSymbol(g_decode_error, &z, sizeof(z));
  return v;
}

}  // namespace fa
