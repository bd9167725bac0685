// Split-K decode (one query token per sequence) for sm_103a; K and V each dense or q4_0.
//
// Decode reads the whole K/V cache once per token, so it is bound by HBM bandwidth, not by the
// tensor cores (the pages' decode figures, "FlashAttention on gfx90a: Why It's Broken and How to
// Fix It", The Problem table, are where flash attention lost most).  The design follows that:
//
//  * grid = (split, kv head, batch); every CTA streams one contiguous key range of one kv head
//    through a ring of shared-memory stages (TMA for nibble / dense tiles, bulk copies or
//    cp.async for the fp16 scale rows), and all query heads of the GQA group are served from that
//    single read;
//  * the two contractions are tiny (N = group size <= 8), so they run on mma.sync m16n8k16 with
//    the *keys* as the M dimension: S^T = K Q^T and O^T += V^T P^T.  The q4_0 nibbles go straight
//    from shared memory into MMA fragment registers (ldmatrix + one LOP3 per pair), so no
//    dequantized tile is ever written back;
//  * K side: the MMA consumes the raw "magic number" values (1024 + q) and (1024 + 16 q) (f16) or
//    (128 + q) (bf16); the constant offsets are removed by starting each block's accumulator at
//    -(offset * sum of the matching Q elements), and the block's fp16 scale is applied in f32 on
//    the accumulator;
//  * V side: exact (q - 8) values in the A fragments; the V scales are folded into P, which the
//    B fragment takes from the S accumulator through movmatrix.trans;
//  * each consumer warp keeps its own online softmax state over 16 or 32 keys per step; the warps
//    of a CTA merge through shared memory and write one partial (m, l, unnormalised O) per query
//    head and split;
//  * the splits of one (batch, kv head) merge inside the same launch: each CTA publishes its
//    partials and an arrival flag, reads the flags of its sibling splits, and a CTA that finds
//    them all set computes M = max m_s, O = sum e^(m_s - M) O_s / sum e^(m_s - M) l_s from L2.
//    No second kernel, and no gap between two launches, sits on the decode step.
#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

__device__ uint32_t g_decode_error;

namespace {

constexpr int kConsumers = 4;  // consumer warps per CTA
constexpr float kLog2e = 1.4426950408889634f;

template <int D, bool KQ4, bool VQ4>
struct DCfg {
  static constexpr bool kAnyQ4 = KQ4 || VQ4;
  static constexpr int kSub = kAnyQ4 ? 2 : 1;                  // 16-key sub-tiles per warp step
  static constexpr int kTileKeys = 16 * kSub * kConsumers;     // keys per stage
  static constexpr int kNB = D / 32;                           // q4_0 blocks per key row
  static constexpr int kRow = kNB * 2;                         // scale bytes per key row
  static_assert(kRow > 0, "scale row");
  static constexpr int kNibBytes = kTileKeys * D / 2;
  // scales as the producer leaves them: K as f32 [key][block] (times the softmax scale in base
  // 2); V as f32 [key][block] (bf16) or as fp16 key pairs [16-key group][t][half][block] (f16)
  static constexpr int kScaleBytes = kTileKeys * kNB * 4;
  static constexpr int kDenseBytes = kTileKeys * D * 2;
  static constexpr int kKBytes = KQ4 ? kNibBytes : kDenseBytes;
  static constexpr int kVBytes = VQ4 ? kNibBytes : kDenseBytes;
  // stage: K tile | V tile | K scales (q4_0 K) | V scales (q4_0 V)
  static constexpr int kOffV = (kKBytes + 1023) / 1024 * 1024;
  static constexpr int kOffKs = kOffV + (kVBytes + 1023) / 1024 * 1024;
  static constexpr int kOffVs = kOffKs + (KQ4 ? kScaleBytes : 0);
  static constexpr int kStageBytes = ((kOffVs + (VQ4 ? kScaleBytes : 0)) + 1023) / 1024 * 1024;
  // one dense side of 128 keys makes a stage ~42 KB (D = 128): two stages and two CTAs per SM
  static constexpr int kStages = (KQ4 == VQ4) ? (D == 128 ? 3 : 6) : (D == 128 ? 2 : 4);
  static constexpr int kCtasPerSm = (KQ4 && VQ4) ? 3 : 2;
  static constexpr int kOffBar = kStages * kStageBytes;
  static constexpr int kOffQ = kOffBar + 256;  // the group's query rows, [8][D] 16-bit
  static constexpr int kSmemBytes = kOffQ + 8 * D * 2 + 1024;
  static constexpr int kThreads = 32 * (1 + kConsumers);
  static constexpr int kPartStride = D + 4;  // m, l, pad, pad, O[D]
  // cross-warp merge buffer (reuses the stages): per warp 8 heads x (D + 2) floats
  static_assert(kConsumers * 8 * (D + 2) * 4 <= kStages * kStageBytes, "merge buffer");
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
// d = A B + c with separate accumulator input and output registers
template <bool BF16>
__device__ __forceinline__ void mma16816_c(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                           uint32_t a3, uint32_t b0, uint32_t b1, float c0,
                                           float c1, float c2, float c3) {
  if (BF16)
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2),
          "f"(c3));
  else
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2),
          "f"(c3));
}
template <bool BF16>
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  if (BF16)
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  else
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------------------------------------
// nibble pairs -> f16/bf16 pairs.  Low nibbles sit at bits 0-3 / 16-19 of the word, high
// nibbles at bits 4-7 / 20-23.
// ---------------------------------------------------------------------------------------------
// raw values (one LOP3 with the exponent pattern `mg` in a register): f16 (1024 + q) from low
// nibbles, (1024 + 16 q) from high nibbles; bf16 (128 + q) from low nibbles only (bf16 has 7
// mantissa bits).  mg = 0x64006400 (f16) or 0x43004300 (bf16).
__device__ __forceinline__ uint32_t raw_lo(uint32_t w, uint32_t mg) {
  return and_or<0x000F000Fu>(w, mg);
}
__device__ __forceinline__ uint32_t raw_hi_f16(uint32_t w, uint32_t mg) {
  return and_or<0x00F000F0u>(w, mg);
}
// exact (q - 8) pairs
template <bool BF16>
__device__ __forceinline__ uint32_t nib_lo(uint32_t w, uint32_t mg) {
  uint32_t x = raw_lo(w, mg);
  if (BF16) {
    const uint32_t c = 0x43084308u;  // 136
    __nv_bfloat162 r = __hsub2(*reinterpret_cast<__nv_bfloat162*>(&x),
                               *reinterpret_cast<const __nv_bfloat162*>(&c));
    return *reinterpret_cast<uint32_t*>(&r);
  } else {
    const uint32_t c = 0x64086408u;  // 1032
    __half2 r = __hsub2(*reinterpret_cast<__half2*>(&x), *reinterpret_cast<const __half2*>(&c));
    return *reinterpret_cast<uint32_t*>(&r);
  }
}
template <bool BF16>
__device__ __forceinline__ uint32_t nib_hi(uint32_t w, uint32_t mg) {
  if (BF16) {
    return nib_lo<true>(w >> 4, mg);
  } else {
    uint32_t x = raw_hi_f16(w, mg);                   // 1024 + 16 q
    const uint32_t s = 0x2C002C00u, c = 0xD480D480u;  // 1/16, -72
    __half2 r = __hfma2(*reinterpret_cast<__half2*>(&x), *reinterpret_cast<const __half2*>(&s),
                        *reinterpret_cast<const __half2*>(&c));
    return *reinterpret_cast<uint32_t*>(&r);
  }
}

template <bool BF16>
__device__ __forceinline__ float h2f(uint16_t bits) {
  return BF16 ? __uint_as_float(static_cast<uint32_t>(bits) << 16)
              : __half2float(__ushort_as_half(bits));
}
template <bool BF16>
__device__ __forceinline__ uint16_t f2h(float v) {
  return BF16 ? __bfloat16_as_ushort(__float2bfloat16_rn(v))
              : __half_as_ushort(__float2half_rn(v));
}

struct DecodeArgs {
  const uint16_t* q;
  uint16_t* o;
  const uint8_t* k_scale;
  const uint8_t* v_scale;
  float* partial;
  int Scap;  // tokens per (batch, kv head) in the K/V tensors (row stride); Sk <= Scap
  // arrival flags [B, Hkv, nsplit]: a split that has published its partials stores this call's
  // tag in its flag.  A flag holding anything else counts as not arrived, so the workspace needs
  // no clearing; a merging CTA sets its flags back to 0, so a replay of the same launch (same
  // tag) starts from cleared flags too.
  uint32_t* flags;
  uint32_t tag;
  int Hq, Hkv, Sk, Sk_eff, nsplit, chunk;
  float scale_log2;
  // paged cache (PAGED kernels): K/V pages [num_pages][Hkv][page_size][D], logical page p of
  // sequence b at block_table[b * pages_per_seq + p], seq_lens[b] tokens in sequence b
  const int32_t* block_table;
  const int32_t* seq_lens;
  int page_size, pages_per_seq, num_pages;
  int B;
};

// Paged batch: the `nsplit` CTAs of a kv head are shared out over the B sequences in proportion
// to their lengths in tiles of `tile_keys` keys, at least one CTA each; every CTA computes the
// same plan from the lengths.  A sequence's length is clamped to [1, cap] here (an out-of-range
// length is reported by the kernel).  For CTA `cta`: its sequence b, its split within the
// sequence, the sequence's split count and the index of its first CTA; false when the CTA lies
// past the plan.  Runs on the host too (seq_lens then in host memory).
struct PagedSlot {
  int b, split, nsplit_b, first;
};
__host__ __device__ __forceinline__ int paged_len(const int32_t* seq_lens, int b, int cap) {
  const int n = seq_lens[b];
  return max(1, min(n, cap));
}
__host__ __device__ __forceinline__ bool paged_slot(const int32_t* seq_lens, int B, int cap,
                                                    int nsplit, int tile_keys, int cta,
                                                    PagedSlot& ps) {
  int64_t total = 0;  // tiles of the whole batch
  for (int bb = 0; bb < B; ++bb) total += (paged_len(seq_lens, bb, cap) + tile_keys - 1) / tile_keys;
  const int spare = nsplit - B;  // CTAs beyond one per sequence
  int s = cta;
  for (int bb = 0; bb < B; ++bb) {
    const int t = (paged_len(seq_lens, bb, cap) + tile_keys - 1) / tile_keys;
    const int ns = 1 + static_cast<int>(static_cast<int64_t>(spare) * t / total);
    if (s < ns) {
      ps.b = bb;
      ps.split = s;
      ps.nsplit_b = ns;
      ps.first = cta - s;
      return true;
    }
    s -= ns;
  }
  return false;
}
// Uniform batch: split s of ns over `len` keys in tiles of `tile` keys.  The tiles are shared out
// as evenly as whole tiles allow, the longer splits first: every CTA of the launch then does the
// same work to within one tile, and with the grid's split index slowest the CTAs dispatched
// last onto each SM (the highest splits) get the shorter ranges (measured: 64.1 -> 62.3 us at 4 x
// 65 536 keys, against equal chunks with a short last one and the split index fastest).
__host__ __device__ __forceinline__ void uniform_split(int s, int ns, int len, int tile, int& kb0,
                                                       int& kb1) {
  const int tiles = (len + tile - 1) / tile;
  const int base = tiles / ns, extra = tiles % ns;
  const int t0 = s * base + min(s, extra);
  const int t1 = t0 + base + (s < extra ? 1 : 0);
  kb0 = min(len, t0 * tile);
  kb1 = min(len, t1 * tile);
}

template <int D, bool BF16, bool KQ4, bool VQ4, bool PAGED>
__global__ void __launch_bounds__(DCfg<D, KQ4, VQ4>::kThreads, DCfg<D, KQ4, VQ4>::kCtasPerSm)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const DecodeArgs args) {
  using C = DCfg<D, KQ4, VQ4>;
  constexpr bool Q4 = C::kAnyQ4;  // some side streams q4_0 (scale rows through the producer)
  constexpr int kSub = C::kSub;
  constexpr int kTileKeys = C::kTileKeys;
  constexpr int kNB = C::kNB;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - smem_u32(smem_raw));
  const uint32_t bar_full = sbase + C::kOffBar;
  const uint32_t bar_empty = bar_full + 8 * C::kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + C::kOffBar + 16 * C::kStages);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int hkv = blockIdx.x;
  const int G = args.Hq / args.Hkv;
  // (sequence, split) of this CTA, this sequence's visible keys, split length and split count.
  // Uniform batch: grid (kv head, batch, split).  Paged batch: grid (kv head, CTA); the CTAs of
  // a kv head are shared out over the sequences in proportion to their lengths (in tiles), every
  // CTA computing the same plan from seq_lens; CTAs past the plan have nothing to do.
  int b = PAGED ? 0 : static_cast<int>(blockIdx.y);
  int split = PAGED ? static_cast<int>(blockIdx.y) : static_cast<int>(blockIdx.z);
  int sk_b = args.Sk_eff, nsplit_b = args.nsplit;
  int first = 0;  // paged: the plan index of this sequence's first CTA
  if constexpr (PAGED) {
    const int cap = args.pages_per_seq * args.page_size;
    PagedSlot ps;
    if (!paged_slot(args.seq_lens, args.B, cap, args.nsplit, kTileKeys,
                    static_cast<int>(blockIdx.y), ps))
      return;  // nothing planned for this CTA (no barrier or memory touched yet)
    b = ps.b;
    split = ps.split;
    nsplit_b = ps.nsplit_b;
    first = ps.first;
    sk_b = args.seq_lens[b];
    if (sk_b < 1 || sk_b > cap) {
      if (threadIdx.x == 0 && split == 0 && hkv == 0)
        atomicCAS(&g_decode_error, kErrNone, kErrBadIndex);
      sk_b = max(1, min(sk_b, cap));
    }
  }
  // slots of the partials and flags.  Uniform batch: [B, Hq, nsplit] partial rows, [B, Hkv,
  // nsplit] flags.  Paged batch: one slot per (kv head, plan CTA): [Hkv, nsplit, G] partial rows,
  // [Hkv, nsplit] flags, a sequence's slots being consecutive -- independent of the batch size.
  const int64_t row0 = static_cast<int64_t>(b) * args.Hq + static_cast<int64_t>(hkv) * G;
  const int64_t part_base = PAGED ? (static_cast<int64_t>(hkv) * args.nsplit + first) * G
                                  : row0 * args.nsplit;
  const int64_t head_stride = PAGED ? 1 : args.nsplit;
  const int64_t slot_stride = PAGED ? G : 1;
  const int64_t flag_base = PAGED ? static_cast<int64_t>(hkv) * args.nsplit + first
                                  : (static_cast<int64_t>(b) * args.Hkv + hkv) * args.nsplit;
  const int sk_lim = PAGED ? sk_b : args.Sk;  // keys stored (scale rows past it are not read)
  int kb0, kb1;
  uniform_split(split, nsplit_b, sk_b, kTileKeys, kb0, kb1);
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
    constexpr int kKeysPerLane = kTileKeys / 32;
    for (; n < ntiles; ++n) {
      const int s = n % C::kStages;
      const int key0 = kb0 + n * kTileKeys;
      // where the tile lives: row tma_row of (page or (batch, kv head)) block tma_bh; a tile
      // never straddles pages (page_size is a multiple of the tile)
      int tma_row = key0;
      int64_t tma_bh = bh;
      int64_t rows_per_bh = args.Scap;
      if constexpr (PAGED) {
        const int lp = key0 / args.page_size;
        int page = args.block_table[static_cast<int64_t>(b) * args.pages_per_seq + lp];
        if (page < 0 || page >= args.num_pages) {
          if (lane == 0) atomicCAS(&g_decode_error, kErrNone, kErrBadIndex);
          page = -1;  // TMA rows out of the map read as zeros; scale loads are skipped
        }
        tma_row = key0 - lp * args.page_size;
        tma_bh = static_cast<int64_t>(page) * args.Hkv + hkv;
        rows_per_bh = args.page_size;
      }
      // q4_0: this lane's scale rows (keys 4*lane .. 4*lane+3 of the tile), zero past Sk; the
      // loads are issued before waiting for the slot so their latency overlaps the wait
      uint32_t kr[kKeysPerLane][2], vr[kKeysPerLane][2];
      if constexpr (Q4) {
#pragma unroll
        for (int j = 0; j < kKeysPerLane; ++j) {
          const int key = key0 + kKeysPerLane * lane + j;
          kr[j][0] = kr[j][1] = vr[j][0] = vr[j][1] = 0u;
          if (key < sk_lim && tma_bh >= 0) {
            const int64_t off = (tma_bh * rows_per_bh + (tma_row + (key - key0))) * C::kRow;
            if (kNB == 4) {
              if (KQ4) {
                const uint2 a = __ldg(reinterpret_cast<const uint2*>(args.k_scale + off));
                kr[j][0] = a.x; kr[j][1] = a.y;
              }
              if (VQ4) {
                const uint2 c = __ldg(reinterpret_cast<const uint2*>(args.v_scale + off));
                vr[j][0] = c.x; vr[j][1] = c.y;
              }
            } else {
              if (KQ4) kr[j][0] = __ldg(reinterpret_cast<const uint32_t*>(args.k_scale + off));
              if (VQ4) vr[j][0] = __ldg(reinterpret_cast<const uint32_t*>(args.v_scale + off));
            }
          }
        }
      }
      if (n >= C::kStages) {
        if (lane == 0)
          ok = mbar_wait(bar_empty + 8 * s, ((n / C::kStages) - 1) & 1, abort_flag,
                         &g_decode_error);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
      }
      const uint32_t st = sbase + s * C::kStageBytes;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar_full + 8 * s, C::kKBytes + C::kVBytes);
        if constexpr (KQ4) {
          tma_load_3d(st, &tm_k, bar_full + 8 * s, 0, tma_row, static_cast<int>(tma_bh));
        } else {
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(st + c * (kTileKeys * 128), &tm_k, bar_full + 8 * s, 64 * c, tma_row,
                        static_cast<int>(tma_bh));
        }
        if constexpr (VQ4) {
          tma_load_3d(st + C::kOffV, &tm_v, bar_full + 8 * s, 0, tma_row, static_cast<int>(tma_bh));
        } else {
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(st + C::kOffV + c * (kTileKeys * 128), &tm_v, bar_full + 8 * s, 64 * c,
                        tma_row, static_cast<int>(tma_bh));
        }
      }
      if constexpr (Q4) {
        uint8_t* stg = sgen + (st - sbase);
#pragma unroll
        for (int j = 0; j < kKeysPerLane; ++j) {
          const int kt = kKeysPerLane * lane + j;  // key within the tile
          if (KQ4) {
            float kf[kNB];
#pragma unroll
            for (int blk = 0; blk < kNB; ++blk)
              kf[blk] = __half2float(__ushort_as_half(
                            static_cast<uint16_t>(kr[j][blk >> 1] >> (16 * (blk & 1))))) *
                        args.scale_log2;
            float* kdst = reinterpret_cast<float*>(stg + C::kOffKs) + kt * kNB;
            if (kNB == 4)
              *reinterpret_cast<float4*>(kdst) = make_float4(kf[0], kf[1], kf[2], kf[3]);
            else
              *reinterpret_cast<float2*>(kdst) = make_float2(kf[0], kf[1]);
          }
          if (BF16 && VQ4) {
            float vf[kNB];
#pragma unroll
            for (int blk = 0; blk < kNB; ++blk)
              vf[blk] = __half2float(__ushort_as_half(
                  static_cast<uint16_t>(vr[j][blk >> 1] >> (16 * (blk & 1)))));
            float* vdst = reinterpret_cast<float*>(stg + C::kOffVs) + kt * kNB;
            if (kNB == 4)
              *reinterpret_cast<float4*>(vdst) = make_float4(vf[0], vf[1], vf[2], vf[3]);
            else
              *reinterpret_cast<float2*>(vdst) = make_float2(vf[0], vf[1]);
          }
        }
        if (!BF16 && VQ4) {
          // key pairs (4*lane, 4*lane+1) and (4*lane+2, 4*lane+3): fp16 pairs per block at
          // [16-key group][t][half][block], t and half from the pair's position in its group
#pragma unroll
          for (int pr = 0; pr < kKeysPerLane / 2; ++pr) {
            const int ka = kKeysPerLane * lane + 2 * pr;  // even key of the pair
            const int grp = ka >> 4, w16 = ka & 15;
            const int h8 = w16 >> 3, t = (w16 & 7) >> 1;
            uint32_t pv[kNB];
#pragma unroll
            for (int blk = 0; blk < kNB; ++blk)
              pv[blk] = __byte_perm(vr[2 * pr][blk >> 1], vr[2 * pr + 1][blk >> 1],
                                    (blk & 1) ? 0x7632u : 0x5410u);
            uint32_t* vdst = reinterpret_cast<uint32_t*>(stg + C::kOffVs) +
                             ((grp * 4 + t) * 2 + h8) * kNB;
            if (kNB == 4)
              *reinterpret_cast<uint4*>(vdst) = make_uint4(pv[0], pv[1], pv[2], pv[3]);
            else
              *reinterpret_cast<uint2*>(vdst) = make_uint2(pv[0], pv[1]);
          }
        }
        mbar_arrive(bar_full + 8 * s);  // release: the scale stores above are visible
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
  const int cw = warp - 1;   // 0..3
  const int g8 = lane >> 2;  // fragment row group
  const int t4 = lane & 3;   // fragment column pair
  const float sl2 = args.scale_log2;

  // Q^T as mma B fragments (k = head dim, n = query head of the group), loaded once.  For q4_0
  // the head dimension is permuted to match the nibble layout: k-step (block, half) uses
  // fragment column 2t+e <-> element 32 block + 16 half + 4t + 2e and column 2t+8+e <->
  // 32 block + 16 half + 4t + 1 + 2e; the high-nibble k-steps of f16 take Q / 16 (exact) to
  // cancel the factor 16 of the raw (1024 + 16 q) values.
  uint32_t qf[D / 16][2];
  // q4_0: -(offset * sum of Q) per block and head, the accumulator start that removes the raw
  // values' constant offsets (f16: 1032 on low halves, 72 on high halves; bf16: 136)
  float corr[kNB][2];
  {
    // the G query rows of this group are contiguous: stage them in shared memory with one
    // 16-byte load per thread, then build the fragments from there
    const uint16_t* qsrc = args.q + (static_cast<int64_t>(b) * args.Hq + hkv * G) * D;
    uint16_t* qs = reinterpret_cast<uint16_t*>(sgen + C::kOffQ);
    for (int idx = threadIdx.x - 32; idx < G * D / 8; idx += 32 * kConsumers)
      reinterpret_cast<uint4*>(qs)[idx] = __ldg(reinterpret_cast<const uint4*>(qsrc) + idx);
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumers) : "memory");
    const uint16_t* qrow = qs + g8 * D;
    const bool valid = g8 < G;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      int d[4];
      if (KQ4) {
        d[0] = 16 * kk + 4 * t4;
        d[1] = d[0] + 2;
        d[2] = d[0] + 1;
        d[3] = d[0] + 3;
      } else {
        d[0] = 16 * kk + 2 * t4;
        d[1] = d[0] + 1;
        d[2] = d[0] + 8;
        d[3] = d[0] + 9;
      }
      uint32_t e[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint16_t v = valid ? qrow[d[i]] : static_cast<uint16_t>(0);
        if (KQ4 && !BF16 && (kk & 1)) v = f2h<false>(h2f<false>(v) * 0.0625f);
        e[i] = v;
      }
      qf[kk][0] = e[0] | (e[1] << 16);
      qf[kk][1] = e[2] | (e[3] << 16);
    }
    if constexpr (KQ4) {
#pragma unroll
      for (int blk = 0; blk < kNB; ++blk) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float lo = 0.f, hi = 0.f;
          if (2 * t4 + hh < G) {
            const uint16_t* qr = qs + (2 * t4 + hh) * D + 32 * blk;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              lo += h2f<BF16>(qr[i]);
              hi += h2f<BF16>(qr[16 + i]);
            }
          }
          corr[blk][hh] = BF16 ? -136.f * (lo + hi) : -(1032.f * lo + 72.f * hi);
        }
      }
    }
  }

  // O^T accumulators: m-tile i covers 16 head-dim rows, columns = query heads 2t, 2t+1
  float o[D / 16][4];
#pragma unroll
  for (int i = 0; i < D / 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY;  // running max (base-2 scaled) for heads 2t, 2t+1
  float l0 = 0.f, l1 = 0.f;              // this thread's share of the row sums
  const int mi = lane >> 3, r8 = lane & 7;  // ldmatrix: matrix index and row of this lane
  const uint32_t mg = opaque_u32(BF16 ? 0x43004300u : 0x64006400u);

  bool ok = true;
  for (int n = 0; n < ntiles; ++n) {
    const int s = n % C::kStages;
    ok = mbar_wait(bar_full + 8 * s, (n / C::kStages) & 1, abort_flag, &g_decode_error);
    if (!__all_sync(0xffffffffu, ok)) break;
    const uint32_t st = sbase + s * C::kStageBytes;
    const int tile_key0 = kb0 + n * kTileKeys;

    // ---------------- S^T = K Q^T, kSub sub-tiles of 16 keys x 8 heads
    float sc[kSub][4];
#pragma unroll
    for (int u = 0; u < kSub; ++u) {
      const int kl = (kSub * 16) * cw + 16 * u;  // first key of the sub-tile in the stage
      sc[u][0] = sc[u][1] = sc[u][2] = sc[u][3] = 0.f;
      if constexpr (KQ4) {
        float kf_g[4], kf_g8[4];  // f32 scales (times the base-2 softmax scale), keys g, g+8
        if (kNB == 4) {
          const uint4 x = lds128(st + C::kOffKs + (kl + g8) * 16);
          const uint4 y = lds128(st + C::kOffKs + (kl + g8 + 8) * 16);
          kf_g[0] = __uint_as_float(x.x); kf_g[1] = __uint_as_float(x.y);
          kf_g[2] = __uint_as_float(x.z); kf_g[3] = __uint_as_float(x.w);
          kf_g8[0] = __uint_as_float(y.x); kf_g8[1] = __uint_as_float(y.y);
          kf_g8[2] = __uint_as_float(y.z); kf_g8[3] = __uint_as_float(y.w);
        } else {
          const uint2 x = lds64(st + C::kOffKs + (kl + g8) * 8);
          const uint2 y = lds64(st + C::kOffKs + (kl + g8 + 8) * 8);
          kf_g[0] = __uint_as_float(x.x); kf_g[1] = __uint_as_float(x.y);
          kf_g8[0] = __uint_as_float(y.x); kf_g8[1] = __uint_as_float(y.y);
          kf_g[2] = kf_g[3] = kf_g8[2] = kf_g8[3] = 0.f;
        }
#pragma unroll
        for (int bb = 0; bb < kNB; bb += 2) {
          const int key = kl + (mi & 1) * 8 + r8;
          const int blk = bb + (mi >> 1);
          const int chunk = (D == 128) ? (blk ^ ((key >> 1) & 3)) : (blk ^ ((key >> 2) & 1));
          uint32_t w[4];
          ldsm_x4(st + key * (D / 2) + chunk * 16, w[0], w[1], w[2], w[3]);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int blkk = bb + e;
            const uint32_t wg = w[2 * e], wg8 = w[2 * e + 1];
            const uint32_t wgs = wg >> 8, wg8s = wg8 >> 8;
            float cb[4];
            mma16816_c<BF16>(cb, raw_lo(wg, mg), raw_lo(wg8, mg), raw_lo(wgs, mg),
                             raw_lo(wg8s, mg), qf[2 * blkk][0], qf[2 * blkk][1], corr[blkk][0],
                             corr[blkk][1], corr[blkk][0], corr[blkk][1]);
            if (BF16)
              mma16816<BF16>(cb, raw_lo(wg >> 4, mg), raw_lo(wg8 >> 4, mg),
                             raw_lo(wgs >> 4, mg), raw_lo(wg8s >> 4, mg),
                             qf[2 * blkk + 1][0], qf[2 * blkk + 1][1]);
            else
              mma16816<BF16>(cb, raw_hi_f16(wg, mg), raw_hi_f16(wg8, mg), raw_hi_f16(wgs, mg),
                             raw_hi_f16(wg8s, mg), qf[2 * blkk + 1][0], qf[2 * blkk + 1][1]);
            const float dg = kf_g[blkk], dg8 = kf_g8[blkk];
            sc[u][0] = fmaf(cb[0], dg, sc[u][0]);
            sc[u][1] = fmaf(cb[1], dg, sc[u][1]);
            sc[u][2] = fmaf(cb[2], dg8, sc[u][2]);
            sc[u][3] = fmaf(cb[3], dg8, sc[u][3]);
          }
        }
      } else {
        const int key = kl + (mi & 1) * 8 + r8;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int d0 = 16 * kk + (mi >> 1) * 8;
          const uint32_t addr = st + (d0 >> 6) * (kTileKeys * 128) + key * 128 +
                                ((((d0 & 63) >> 3) ^ (key & 7)) << 4);
          uint32_t a0, a1, a2, a3;
          ldsm_x4(addr, a0, a1, a2, a3);
          mma16816<BF16>(sc[u], a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
        }
      }
    }

    // ---------------- online softmax over this warp's kSub * 16 keys
    // scores in base-2 units (the q4_0 K scales already carry the softmax scale); keys past
    // the split's end are masked, which only the last tile of a split can contain
    float t[kSub][4];
    float mx0 = -INFINITY, mx1 = -INFINITY;
    const bool full_tile = tile_key0 + kTileKeys <= kb1;
#pragma unroll
    for (int u = 0; u < kSub; ++u) {
#pragma unroll
      for (int i = 0; i < 4; ++i) t[u][i] = KQ4 ? sc[u][i] : sc[u][i] * sl2;
      if (!full_tile) {
        const int keyg = tile_key0 + (kSub * 16) * cw + 16 * u + g8;
        if (keyg >= kb1) t[u][0] = t[u][1] = -INFINITY;
        if (keyg + 8 >= kb1) t[u][2] = t[u][3] = -INFINITY;
      }
      mx0 = fmaxf(mx0, fmaxf(t[u][0], t[u][2]));
      mx1 = fmaxf(mx1, fmaxf(t[u][1], t[u][3]));
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float nm0 = fmaxf(m0, mx0), nm1 = fmaxf(m1, mx1);
    if (__any_sync(0xffffffffu, (nm0 > m0) || (nm1 > m1))) {
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
    float p[kSub][4];
#pragma unroll
    for (int u = 0; u < kSub; ++u) {
      p[u][0] = ex2(t[u][0] - b0);
      p[u][1] = ex2(t[u][1] - b1);
      p[u][2] = ex2(t[u][2] - b0);
      p[u][3] = ex2(t[u][3] - b1);
      l0 += p[u][0] + p[u][2];
      l1 += p[u][1] + p[u][3];
    }

    // ---------------- O^T += V^T P^T
#pragma unroll
    for (int u = 0; u < kSub; ++u) {
      const int kl = (kSub * 16) * cw + 16 * u;
      if constexpr (VQ4) {
        const uint32_t vbase = st + C::kOffV;
        // P of keys (2t, 2t+1) and (2t+8, 2t+9) for head g (f16: transposed once, then scaled
        // per block with the V scales of those key pairs)
        uint32_t pt0 = 0, pt1 = 0;
        uint32_t sp01[4] = {0u, 0u, 0u, 0u};  // fp16 V-scale pairs of keys (2t, 2t+1), per block
        uint32_t sp89[4] = {0u, 0u, 0u, 0u};  // and of keys (2t+8, 2t+9)
        float vf_g[4] = {0.f, 0.f, 0.f, 0.f}, vf_g8[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (!BF16) {
          pt0 = movtrans(pack2<false>(p[u][0], p[u][1]));
          pt1 = movtrans(pack2<false>(p[u][2], p[u][3]));
          const uint32_t pa = st + C::kOffVs + ((kl >> 4) * 4 + t4) * 2 * kNB * 4;
          if (kNB == 4) {
            const uint4 x = lds128(pa), y = lds128(pa + 16);
            sp01[0] = x.x; sp01[1] = x.y; sp01[2] = x.z; sp01[3] = x.w;
            sp89[0] = y.x; sp89[1] = y.y; sp89[2] = y.z; sp89[3] = y.w;
          } else {
            const uint2 x = lds64(pa), y = lds64(pa + 8);
            sp01[0] = x.x; sp01[1] = x.y; sp89[0] = y.x; sp89[1] = y.y;
          }
        } else {
          if (kNB == 4) {
            const uint4 x = lds128(st + C::kOffVs + (kl + g8) * 16);
            const uint4 y = lds128(st + C::kOffVs + (kl + g8 + 8) * 16);
            vf_g[0] = __uint_as_float(x.x); vf_g[1] = __uint_as_float(x.y);
            vf_g[2] = __uint_as_float(x.z); vf_g[3] = __uint_as_float(x.w);
            vf_g8[0] = __uint_as_float(y.x); vf_g8[1] = __uint_as_float(y.y);
            vf_g8[2] = __uint_as_float(y.z); vf_g8[3] = __uint_as_float(y.w);
          } else {
            const uint2 x = lds64(st + C::kOffVs + (kl + g8) * 8);
            const uint2 y = lds64(st + C::kOffVs + (kl + g8 + 8) * 8);
            vf_g[0] = __uint_as_float(x.x); vf_g[1] = __uint_as_float(x.y);
            vf_g8[0] = __uint_as_float(y.x); vf_g8[1] = __uint_as_float(y.y);
          }
        }
#pragma unroll
        for (int bb = 0; bb < kNB; bb += 2) {
          const int key = kl + (mi & 1) * 8 + r8;
          const int blk = bb + (mi >> 1);
          const int chunk = (D == 128) ? (blk ^ ((key >> 1) & 3)) : (blk ^ ((key >> 2) & 1));
          uint32_t w[4];
          ldsm_x4_t(vbase + key * (D / 2) + chunk * 16, w[0], w[1], w[2], w[3]);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int blkk = bb + e;
            uint32_t pb0, pb1;
            if constexpr (!BF16) {
              __half2 r0 = __hmul2(*reinterpret_cast<const __half2*>(&pt0),
                                   *reinterpret_cast<const __half2*>(&sp01[blkk]));
              __half2 r1 = __hmul2(*reinterpret_cast<const __half2*>(&pt1),
                                   *reinterpret_cast<const __half2*>(&sp89[blkk]));
              pb0 = *reinterpret_cast<uint32_t*>(&r0);
              pb1 = *reinterpret_cast<uint32_t*>(&r1);
            } else {
              // bf16: scale P in f32 (the fp16 scale is exact there), then round once
              const float dg = vf_g[blkk], dg8 = vf_g8[blkk];
              pb0 = movtrans(pack2<true>(p[u][0] * dg, p[u][1] * dg));
              pb1 = movtrans(pack2<true>(p[u][2] * dg8, p[u][3] * dg8));
            }
            const uint32_t w1 = w[2 * e], w2 = w[2 * e + 1];
            // m-tile (block, low nibbles): rows g <-> element 2g, g+8 <-> element 2g+1
            const uint32_t w1s = w1 >> 8, w2s = w2 >> 8;
            mma16816<BF16>(o[2 * blkk], nib_lo<BF16>(w1, mg), nib_lo<BF16>(w1s, mg),
                           nib_lo<BF16>(w2, mg), nib_lo<BF16>(w2s, mg), pb0, pb1);
            // m-tile (block, high nibbles): rows g <-> element 16+2g, g+8 <-> element 17+2g
            mma16816<BF16>(o[2 * blkk + 1], nib_hi<BF16>(w1, mg), nib_hi<BF16>(w1s, mg),
                           nib_hi<BF16>(w2, mg), nib_hi<BF16>(w2s, mg), pb0, pb1);
          }
        }
      } else {
        const uint32_t pb0 = movtrans(pack2<BF16>(p[u][0], p[u][1]));
        const uint32_t pb1 = movtrans(pack2<BF16>(p[u][2], p[u][3]));
        const int key = kl + (mi >> 1) * 8 + r8;
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
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * s);
  }

  // ------------------------------------------------------------------ merge the 4 warps
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
      if (VQ4) {
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
    float* dst =
        args.partial + (part_base + hh * head_stride + split * slot_stride) * C::kPartStride;
    dst[c == 0 ? 0 : (c == 1 ? 1 : c + 2)] = out;
  }

  // ------------------------------------------------------------------ merge the splits
  // After a barrier over the consumer threads one thread publishes this split's flag with a
  // gpu-scope release store (cumulative: it covers the partial stores of every thread that
  // reached the barrier), orders that store before its loads with a sequentially consistent
  // fence, and one warp loads the flags of every split of this (batch, kv head).  Of two splits
  // that publish at the same time at least one sees the other's flag (the fence forbids both
  // missing), so at least one CTA finds all flags set; every CTA that does merges, and they all
  // write the same bytes.  No CTA waits for another and no atomic read-modify-write is contended.
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumers) : "memory");
  volatile uint32_t* is_last =
      reinterpret_cast<volatile uint32_t*>(sgen + C::kOffBar + 16 * C::kStages + 8);
  uint32_t* flags = args.flags + flag_base;
  if (cw == 0) {
    if (lane == 0) st_release_gpu(flags + split, args.tag);
    __syncwarp();
    fence_sc_gpu();  // the whole warp: its flag loads below come after the store above
    bool all = true;
    for (int s = lane; s < nsplit_b; s += 32) all = all && ld_relaxed_gpu(flags + s) == args.tag;
    all = __all_sync(0xffffffffu, all);
    if (all) fence_acq_rel_gpu();  // the partials behind the flags are read after this
    if (lane == 0) *is_last = all ? 1u : 0u;
  }
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumers) : "memory");
  if (*is_last == 0u) return;
  if (cw == 0)
    for (int s = lane; s < nsplit_b; s += 32) st_relaxed_gpu(flags + s, 0u);
  constexpr int kPer = D / 32;  // head-dim elements per lane
  constexpr int kStride = C::kPartStride;
  for (int hh = cw; hh < G; hh += kConsumers) {
    const float* p = args.partial + (part_base + hh * head_stride) * kStride;
    const int64_t ss = slot_stride * kStride;  // floats from one split's row to the next
    // (m_s, l_s) with the splits across the lanes, 32 at a time; the first 32 stay in registers
    float2 ml0 = make_float2(-INFINITY, 0.f);
    if (lane < nsplit_b) ml0 = __ldcg(reinterpret_cast<const float2*>(p + lane * ss));
    // paged batch, up to kFast splits: their O rows are loaded in the same round trip as (m, l)
    // (a merge sits at the end of the launch, where each round trip to L2 is exposed; measured
    // -3 % on the paged workloads; the uniform kernel keeps the loop below, where the extra
    // registers cost more than they gain)
    constexpr int kFast = PAGED ? 16 : 1;
    const bool fast = PAGED && nsplit_b <= kFast;
    float xf[kFast][kPer];
    if (fast) {
#pragma unroll
      for (int j = 0; j < kFast; ++j) {
        const float* row = p + j * ss + 4;
        if (j < nsplit_b) {
          if constexpr (kPer == 4) {
            const float4 v = __ldcg(reinterpret_cast<const float4*>(row) + lane);
            xf[j][0] = v.x; xf[j][1] = v.y; xf[j][2] = v.z; xf[j][3] = v.w;
          } else {
            const float2 v = __ldcg(reinterpret_cast<const float2*>(row) + lane);
            xf[j][0] = v.x; xf[j][1] = v.y;
          }
        } else {
#pragma unroll
          for (int e = 0; e < kPer; ++e) xf[j][e] = 0.f;
        }
      }
    }
    float M = ml0.x;
    for (int s = lane + 32; s < nsplit_b; s += 32) M = fmaxf(M, __ldcg(p + s * ss));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float L = 0.f;
    float acc[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
    if (fast) {
      const float wl = (ml0.x == -INFINITY) ? 0.f : ex2(ml0.x - M);  // e^(m_s - M), lane s
      L = wl * ml0.y;
#pragma unroll
      for (int j = 0; j < kFast; ++j) {
        const float wj = __shfl_sync(0xffffffffu, wl, j);
#pragma unroll
        for (int e = 0; e < kPer; ++e) acc[e] = fmaf(wj, xf[j][e], acc[e]);
      }
    }
    for (int s0 = 0; s0 < (fast ? 0 : nsplit_b); s0 += 32) {
      float2 ml = ml0;
      if (s0 > 0) {
        ml = make_float2(-INFINITY, 0.f);
        if (s0 + lane < nsplit_b)
          ml = __ldcg(reinterpret_cast<const float2*>(p + (s0 + lane) * ss));
      }
      const float wl = (ml.x == -INFINITY) ? 0.f : ex2(ml.x - M);  // e^(m_s - M), lane s
      L = fmaf(wl, ml.y, L);
      const int n = min(32, nsplit_b - s0);
      // O_s rows, eight splits' loads in flight before their multiply-adds (in split order)
      for (int j0 = 0; j0 < n; j0 += 8) {
        float x[8][kPer];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float* row = p + (s0 + j0 + j) * ss + 4;
          if (j0 + j < n) {
            if constexpr (kPer == 4) {
              const float4 v = __ldcg(reinterpret_cast<const float4*>(row) + lane);
              x[j][0] = v.x; x[j][1] = v.y; x[j][2] = v.z; x[j][3] = v.w;
            } else {
              const float2 v = __ldcg(reinterpret_cast<const float2*>(row) + lane);
              x[j][0] = v.x; x[j][1] = v.y;
            }
          } else {
#pragma unroll
            for (int e = 0; e < kPer; ++e) x[j][e] = 0.f;
          }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float wj = __shfl_sync(0xffffffffu, wl, (j0 + j) & 31);
#pragma unroll
          for (int e = 0; e < kPer; ++e) acc[e] = fmaf(wj, x[j][e], acc[e]);
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    const float inv = 1.f / L;
    uint16_t* dst = args.o + (row0 + hh) * D + lane * kPer;
    const uint32_t w0 = static_cast<uint32_t>(f2h<BF16>(acc[0] * inv)) |
                        (static_cast<uint32_t>(f2h<BF16>(acc[1] * inv)) << 16);
    if constexpr (kPer == 4) {
      const uint32_t w1 = static_cast<uint32_t>(f2h<BF16>(acc[2] * inv)) |
                          (static_cast<uint32_t>(f2h<BF16>(acc[3] * inv)) << 16);
      *reinterpret_cast<uint2*>(dst) = make_uint2(w0, w1);
    } else {
      *reinterpret_cast<uint32_t*>(dst) = w0;
    }
  }
}

constexpr int kMaxSplits = 1024;  // splits per (batch, kv head)

}  // namespace

size_t decode_flag_bytes(int B, int Hkv, int nsplit) {
  return (static_cast<size_t>(B) * Hkv * nsplit * sizeof(uint32_t) + 255) / 256 * 256;
}

int decode_tile_keys(bool kq4, bool vq4) {
  return (kq4 || vq4) ? DCfg<128, true, true>::kTileKeys : DCfg<128, false, false>::kTileKeys;
}

static int decode_ctas_per_sm(bool kq4, bool vq4) {
  if (kq4 && vq4) return DCfg<128, true, true>::kCtasPerSm;
  if (kq4 || vq4) return DCfg<128, true, false>::kCtasPerSm;
  return DCfg<128, false, false>::kCtasPerSm;
}

int decode_paged_ctas(int B, int Hkv, int num_sms, bool kq4, bool vq4) {
  // one wave of CTAs at the kernel's resident count, at least one per sequence
  const int slots = (num_sms < 1 ? 1 : num_sms) * decode_ctas_per_sm(kq4, vq4);
  const int per_head = slots / (Hkv < 1 ? 1 : Hkv);
  return per_head > B ? per_head : B;
}

void decode_plan(int B, int Hkv, int Sk_eff, int num_sms, bool kq4, bool vq4, int* nsplit,
                 int* chunk) {
  // one wave of CTAs at the kernel's resident count; the keys shared out in whole tiles as
  // evenly as possible (uniform_split), chunk = the longer splits' length
  const int tile = decode_tile_keys(kq4, vq4);
  const int units = B * Hkv;
  const int slots = num_sms * decode_ctas_per_sm(kq4, vq4);
  int ns = slots / units;
  if (ns < 1) ns = 1;
  const int max_tiles = (Sk_eff + tile - 1) / tile;
  if (ns > max_tiles) ns = max_tiles;
  if (ns > kMaxSplits) ns = kMaxSplits;
  if (ns < 1) ns = 1;
  *chunk = (max_tiles + ns - 1) / ns * tile;
  *nsplit = ns;
}

template <int D, bool BF16, bool KQ4, bool VQ4>
static cudaError_t launch_t(const DecodeLaunch& L, cudaStream_t stream) {
  using C = DCfg<D, KQ4, VQ4>;
  auto kern = L.block_table ? decode_split_kernel<D, BF16, KQ4, VQ4, true>
                            : decode_split_kernel<D, BF16, KQ4, VQ4, false>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  DecodeArgs a;
  a.q = static_cast<const uint16_t*>(L.q);
  a.k_scale = static_cast<const uint8_t*>(L.k_scale);
  a.v_scale = static_cast<const uint8_t*>(L.v_scale);
  a.o = static_cast<uint16_t*>(L.o);
  a.partial = L.partial;
  a.Scap = L.Scap;
  a.block_table = L.block_table;
  a.seq_lens = L.seq_lens;
  a.page_size = L.page_size;
  a.pages_per_seq = L.pages_per_seq;
  a.num_pages = L.num_pages;
  a.B = L.B;
  a.flags = L.flags;
  a.tag = L.tag;
  a.Hq = L.Hq;
  a.Hkv = L.Hkv;
  a.Sk = L.Sk;
  a.Sk_eff = L.Sk_eff;
  a.nsplit = L.nsplit;
  a.chunk = L.chunk;
  a.scale_log2 = L.scale * kLog2e;
  // paged: nsplit CTAs per kv head shared over the batch (the plan is made on the device)
  const dim3 grid = L.block_table ? dim3(L.Hkv, L.nsplit, 1) : dim3(L.Hkv, L.B, L.nsplit);
  kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(L.tm_k, L.tm_v, a);
  return cudaGetLastError();
}

template <int D, bool BF16>
static cudaError_t launch_fmt(const DecodeLaunch& L, cudaStream_t stream) {
  if (L.kq4) return L.vq4 ? launch_t<D, BF16, true, true>(L, stream)
                          : launch_t<D, BF16, true, false>(L, stream);
  return L.vq4 ? launch_t<D, BF16, false, true>(L, stream)
               : launch_t<D, BF16, false, false>(L, stream);
}

cudaError_t decode_launch(const DecodeLaunch& L, cudaStream_t stream) {
  if (L.D == 128)
    return L.bf16 ? launch_fmt<128, true>(L, stream) : launch_fmt<128, false>(L, stream);
  return L.bf16 ? launch_fmt<64, true>(L, stream) : launch_fmt<64, false>(L, stream);
}

int64_t decode_debug_schedule(const int32_t* seq_lens, int B, int Hkv, int Sk, int cap,
                              bool kq4, bool vq4, int num_sms, int32_t* rows,
                              int64_t max_rows) {
  const int tile = decode_tile_keys(kq4, vq4);
  int64_t n = 0;
  auto put = [&](int b, int split, int nsplit_b, int kb0, int kb1) {
    if (rows != nullptr && n < max_rows) {
      int32_t* r = rows + n * kDecodeScheduleRowWidth;
      r[0] = b;
      r[1] = split;
      r[2] = nsplit_b;
      r[3] = kb0;
      r[4] = kb1;
    }
    ++n;
  };
  if (seq_lens == nullptr) {  // uniform batch: grid (kv head, batch, split)
    int ns = 1, ck = Sk;
    decode_plan(B, Hkv, Sk, num_sms, kq4, vq4, &ns, &ck);
    for (int b = 0; b < B; ++b)
      for (int sp = 0; sp < ns; ++sp) {
        int kb0, kb1;
        uniform_split(sp, ns, Sk, tile, kb0, kb1);
        put(b, sp, ns, kb0, kb1);
      }
    return n;
  }
  const int nt = decode_paged_ctas(B, Hkv, num_sms, kq4, vq4);  // CTAs per kv head
  for (int c = 0; c < nt; ++c) {
    PagedSlot ps;
    if (!paged_slot(seq_lens, B, cap, nt, tile, c, ps)) {
      put(-1, 0, 0, 0, 0);
      continue;
    }
    const int len = paged_len(seq_lens, ps.b, cap);
    int kb0, kb1;
    uniform_split(ps.split, ps.nsplit_b, len, tile, kb0, kb1);
    put(ps.b, ps.split, ps.nsplit_b, kb0, kb1);
  }
  return n;
}

uint32_t decode_take_error() {
  uint32_t v = 0;
  if (cudaMemcpyFromSymbol(&v, g_decode_error, sizeof(v)) != cudaSuccess) return 0xffffffffu;
  const uint32_t z = 0;
  cudaMemcpyToSymbol(g_decode_error, &z, sizeof(z));
  return v;
}

}  // namespace fa
