// Fused causal GQA flash-attention forward (chunked prefill) for sm_103a.
//
// What it computes: O = softmax(scale * Q K^T + causal mask) V per query head, with query head h
// reading key/value head h / (Hq / Hkv), and the query chunk placed at absolute positions
// q_pos_offset .. q_pos_offset + Sq - 1 (a key is visible when its position is <= the row's).
// This is the fused kernel of "perf(rocm): defer SDPA accumulator rescale, stage Q once per
// block (#2306)" (Conversation; What changed), rebuilt for tcgen05:
//
//  * one CTA owns two 128-row query tiles (A, B) of one query head; both Q tiles are brought
//    into shared memory once by TMA and stay there for the CTA's whole key range ("Q is staged
//    once per block");
//  * K and V tiles of 128 keys stream through a ring of shared-memory stages, each side either
//    by TMA (dense f16/bf16 cache) or as q4_0 nibble/scale tiles that dequant warps expand into
//    the same f16/bf16 swizzled layout; K and V formats are independent template parameters.
//    This is the fused K and V dequant of "FlashAttention on gfx90a: Why It's Broken and How to
//    Fix It" (Why FA-off Can't Do V Quantization, point 5); every K/V tile serves both query
//    tiles;
//  * S = Q K^T and O += P V are tcgen05.mma into tensor memory; the single MMA thread
//    interleaves the tiles (PV_A(j), QK_A(j+1), PV_B(j), QK_B(j+1)) so the tensor core works on
//    one tile while the softmax warps of the other run.  When even one query tile per CTA
//    leaves SMs idle (2 x pair units <= SMs), each CTA takes one tile instead, and with dense
//    K/V that tile's key blocks alternate between the two S buffers (QK(j+2) is issued right
//    after PV(j)), so the softmax finds the next block's scores ready;
//  * the softmax warps own one row each: block max, the deferred rescale, P = 2^(t - f) written
//    back over S as f16/bf16 for the PV MMA, running row sum l;
//  * deferred rescale ("perf(rocm): defer SDPA accumulator rescale, stage Q once per block
//    (#2306)", Summary; What changed): a row keeps its frame f until a block max exceeds f by
//    more than 10 natural-log units; only then are O and l multiplied by e^(f_old - f_new).
//    P stays below e^10 = 22026 in every frame.
//
// Warp roles (12 warps with dense K/V, 16 with a q4_0 side):
//   warp 0        TMA producer (one lane)
//   warp 1        TMEM allocator + MMA issuer (one lane)
//   warps 2, 3    q4_0 dequant with warps 12..15 (six warps sharing each raw tile's items);
//                 idle with dense K/V
//   warps 4..7    softmax / rescale / epilogue of query tile A, one row per thread
//   warps 8..11   the same for query tile B
#include <algorithm>

#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa_quant.cuh"

namespace fa {

__device__ uint32_t g_prefill_error;

namespace {

constexpr int kBM = 128;                      // query rows per tile
constexpr int kBN = 128;                      // keys per tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kMarginLog2 = 10.0f * kLog2e; // the 10-point margin, in base-2 units
constexpr uint32_t kTmemCols = 512;
// TMEM column of the S block of query tile t (0: A, 1: B); P overwrites its first half
__host__ __device__ constexpr uint32_t col_s(int t) { return t ? 128u : 0u; }

// WIDE: the sixteen-warp layout with q4_0 K or V (both prefill kernels use it)
template <int D, bool KQ4, bool VQ4, bool WIDE = false>
struct Cfg {
  static constexpr bool kAnyQ4 = KQ4 || VQ4;
  static constexpr int kTileBytes = kBN * D * 2;          // one f16/bf16 K or V tile
  static constexpr int kQBytes = kBM * D * 2;             // one Q tile
  // ring of K/V tiles in MMA order K0 V0 K1 V1 ...; with one q4_0 side the stage count is even,
  // so K tiles always land on even stages and V tiles on odd ones (fixed arrival counts)
  static constexpr int kStages = (KQ4 && VQ4) ? 3 : (D == 128 ? 4 : 6);
  static constexpr int kRawStages = (KQ4 && VQ4) ? 3 : (kAnyQ4 ? 2 : 0);
  static_assert(KQ4 == VQ4 || kStages % 2 == 0, "mixed formats need an even ring");
  // dense K and V: the ring is used as kStages / 2 slots of two stages, slot g holding the V
  // tile of block j and the K tile of block j + 1 (the first slot of a unit or segment: K of
  // its first block alone), so that the MMA issuer waits for one slot and commits one release
  // per block step.  Each wait or commit costs the single issuing thread 120-350 clk of its
  // block period (measured), during which the tensor pipe drains.  A slot whose K tile tile B
  // multiplies is released by tile B's softmax on seeing that QK complete (the issuer's commit
  // covers every MMA it issued before, so also the earlier reads of the slot); the issuer
  // commits the release only of the others.
  static constexpr bool kPaired = !kAnyQ4;
  static constexpr int kSlots = kStages / 2;
  static_assert(!kPaired || kStages % 2 == 0, "paired ring");
  static constexpr int kNibRow = D / 2;                   // bytes of nibbles per key
  static constexpr int kScaleRow = D / 32 * 2;            // bytes of scales per key
  static constexpr int kRawNib = kBN * kNibRow;
  static constexpr int kRawBytes = ((kRawNib + kBN * kScaleRow) + 1023) / 1024 * 1024;
  static constexpr int kOffQ = 0;                         // Q_A, Q_B
  static constexpr int kOffRing = kOffQ + 2 * kQBytes;
  static constexpr int kOffRaw = kOffRing + kStages * kTileBytes;
  static constexpr int kOffBar = kOffRaw + kRawStages * kRawBytes;
  static constexpr int kBarBytes = 512 + 1024;  // barriers, flags, then the segment table
  static constexpr int kSmemBytes = kOffBar + kBarBytes + 1024;  // + alignment slack
  // warps: 0 producer, 1 MMA issuer, 4-11 softmax (one thread per query row), 2-3 dequant
  // with q4_0 K or V; WIDE adds dequant warps 12-15 (sixteen warps, 128 registers a thread at
  // launch; the kernels then move registers from warpgroups 0 and 3 to the two softmax
  // warpgroups, 88 and 168 a thread).  Measured at 16K keys, q4_0 K and V: with two dequant
  // warps the step waits for dequantized tiles; six of them took the cut kernel from 0.477 to
  // 0.410 ms and the one-unit kernel from 0.484 to 0.443 ms.
  static constexpr bool kWide = WIDE && kAnyQ4;
  static constexpr int kDqWarps = kAnyQ4 ? (kWide ? 6 : 2) : 0;
  static constexpr int kDqThreads = kDqWarps * 32;
  static constexpr int kWarps = kWide ? 16 : 12;
  static __device__ __forceinline__ bool is_dq_warp(int w) {
    return w == 2 || w == 3 || (kWide && w >= 12);
  }
  static __device__ __forceinline__ int dq_index(int w, int lane) {
    return (w < 4 ? w - 2 : w - 10) * 32 + lane;
  }
  static constexpr int kThreads = kWarps * 32;
  static constexpr uint32_t kColO0 = 256, kColO1 = 256 + D;     // O of tile A / B
};

// barrier slots (8 bytes each) inside the barrier area
enum {
  kBarQFull = 0,
  kBarSFull = 1,       // + tile (2)
  kBarPReady = 3,      // + tile (2)
  kBarODone = 5,       // + tile (2): completes once, after the tile's last PV MMA
  kBarDrain = 7,
  kBarRingFull = 8,    // + stage (up to 8)
  kBarRingEmpty = 16,  // + stage
  kBarRawFull = 24,    // + raw stage
  kBarRawEmpty = 32,   // + raw stage
  kBarQEmpty = 40,     // the segment's last QK MMA has read the Q tiles (commit)
  kBarOFree = 41,      // + tile (2): the segment's epilogue has read O out of TMEM (128 threads)
  kBarPiece = 43,      // all 256 softmax threads have stored their rows of a piece
  kBarMergeDecided = 44,  // the piece's flag is published and the merge decision made
  kBarCount = 45
};
constexpr int kOffTmemSlot = kBarCount * 8;
constexpr int kOffAbort = kOffTmemSlot + 8;
constexpr int kOffMergeFlag = kOffAbort + 8;
constexpr int kOffSegCount = 512;        // within the barrier area: this CTA's segment count,
constexpr int kOffSegs = kOffSegCount + 16;  // then its segments (SegS)
constexpr int kMaxSegs = 16;

struct PrefillArgs {
  void* o;
  const uint8_t* k_scale;  // q4_0 only: fp16 scale planes [B, Hkv, Sk, D/32]
  const uint8_t* v_scale;
  int32_t* rescale_count;  // optional [B, Hq, Sq]
  float* p_max;            // optional [B, Hq, Sq]: a bound on the largest P the row's softmax
                           // wrote (see softmax_block)
  int B, Hq, Hkv, Sq, Sk, q_pos_offset, causal, n_qtiles, n_pairs;
  // prefill_kernel: query rows per work unit, 256 (a pair of consecutive tiles) or 128 (one
  // tile per CTA, tile B absent; n_pairs then counts query tiles)
  int unit_rows;
  int Scap;  // tokens per (batch, kv head) in the K/V tensors (row stride); Sk <= Scap
  float scale_log2;
  // cut schedule (prefill_seg_kernel): W key-block steps in all, CTA c runs steps
  // [range_start(c), range_start(c + 1))
  int64_t W;
  int n_ctas;
  float* part;           // partial rows of units cut between CTAs (workspace), 2 slots per CTA
  uint32_t* pflags;      // [n_ctas][2] publication flags (workspace), tagged per call
  uint32_t tag;
  // a chunk appended to q4_0 K and V caches in the same launch (prefill_seg_kernel with q4_0
  // on both sides, cooperative launch): phase 1 quantizes tokens [app_pos0, app_pos0 + app_len)
  // of every (batch, kv head) from k_new / v_new into the caches, one item per (batch, kv head,
  // 128-key cache block), and sets the item's flag in app_flags (zeroed before the launch);
  // the producer waits for an item's flag before it reads that block from the caches
  const uint16_t* k_new;  // [B, Hkv, app_len, D]
  const uint16_t* v_new;
  uint8_t* k_nib;         // the caches' nibble planes [B, Hkv, Scap, D/2]
  uint8_t* v_nib;
  __half* k_scw;          // the caches' scale planes [B, Hkv, Scap, D/32]
  __half* v_scw;
  uint32_t* app_flags;    // [B * Hkv * app_nb]; null: no append
  int app_pos0, app_len, app_j_lo, app_nb;
};

// ------------------------------------------------------------------------------------------
// q4_0 nibble pair -> f16/bf16 pair
// ------------------------------------------------------------------------------------------
template <bool BF16>
struct Dq;
template <>
struct Dq<false> {
  // low nibbles at bits 0-3 / 16-19 -> (n - 8) exactly; mg = 0x64006400 in a register
  static __device__ __forceinline__ __half2 lo(uint32_t w, uint32_t mg) {
    uint32_t x = and_or<0x000F000Fu>(w, mg);  // 1024 + n
    return __hsub2(*reinterpret_cast<__half2*>(&x), __halves2half2(__ushort_as_half(0x6408),
                                                                    __ushort_as_half(0x6408)));
  }
  // high nibbles at bits 4-7 / 20-23 -> (n - 8) exactly
  static __device__ __forceinline__ __half2 hi(uint32_t w, uint32_t mg) {
    uint32_t x = and_or<0x00F000F0u>(w, mg);  // 1024 + 16 n
    const __half2 s = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));  // 1/16
    const __half2 c = __halves2half2(__ushort_as_half(0xD480), __ushort_as_half(0xD480));  // -72
    return __hfma2(*reinterpret_cast<__half2*>(&x), s, c);
  }
  static __device__ __forceinline__ uint32_t scale(__half2 v, __half d) {
    __half2 r = __hmul2(v, __halves2half2(d, d));
    return *reinterpret_cast<uint32_t*>(&r);
  }
};
template <>
struct Dq<true> {
  static __device__ __forceinline__ __nv_bfloat162 lo(uint32_t w, uint32_t mg) {
    uint32_t x = and_or<0x000F000Fu>(w, mg);  // 128 + n (mg = 0x43004300)
    const uint32_t c = 0x43084308u;           // 136
    return __hsub2(*reinterpret_cast<__nv_bfloat162*>(&x),
                   *reinterpret_cast<const __nv_bfloat162*>(&c));
  }
  // bf16 has 7 mantissa bits, so a high nibble at bits 4-7 would reach the exponent: shift it
  // down to bits 0-3 first
  static __device__ __forceinline__ __nv_bfloat162 hi(uint32_t w, uint32_t mg) {
    return lo(w >> 4, mg);
  }
  static __device__ __forceinline__ uint32_t scale(__nv_bfloat162 v, float d) {
    // (n - 8) * d rounded once to bf16: the product of a 4-bit integer and an fp16 value is
    // exact in f32, so round only after the f32 multiply.
    const float2 f = __bfloat1622float2(v);
    __nv_bfloat162 r = __floats2bfloat162_rn(f.x * d, f.y * d);
    return *reinterpret_cast<uint32_t*>(&r);
  }
};


template <bool BF16>
__device__ __forceinline__ float block_row_exp_regs(uint32_t scol, const float (&s)[kBN],
                                                    float sl2, float nf) {
  // the scale-and-shift and the row sum run two keys per instruction (packed f32 pairs)
  const uint64_t sl2x2 = f2_pack(sl2, sl2), nfx2 = f2_pack(nf, nf);
  uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = acc0;
#pragma unroll
  for (int c = 0; c < kBN / 32; ++c) {
    uint32_t pr[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 t =
          f2_unpack(f2_fma(f2_pack(s[32 * c + 2 * i], s[32 * c + 2 * i + 1]), sl2x2, nfx2));
      const float p0 = ex2(t.x), p1 = ex2(t.y);
      const uint64_t pp = f2_pack(p0, p1);
      if (i & 1) acc1 = f2_add(acc1, pp); else acc0 = f2_add(acc0, pp);
      pr[i] = pack2<BF16>(p0, p1);
    }
    tmem_st16(scol + 16 * c, pr);
  }
  const float2 a = f2_unpack(f2_add(acc0, acc1));
  return a.x + a.y;
}

// the scores of S(j) for this row with one TMEM wait, keys past rel_lim set to -inf (MASK)
template <bool MASK>
__device__ __forceinline__ void block_row_scores(uint32_t scol, int rel_lim, float (&s)[kBN]) {
  uint32_t r0[32], r1[32], r2[32], r3[32];
  tmem_ld32(scol, r0);
  tmem_ld32(scol + 32, r1);
  tmem_ld32(scol + 64, r2);
  tmem_ld32(scol + 96, r3);
  tmem_wait_ld();
  reg_fence32(r0);
  reg_fence32(r1);
  reg_fence32(r2);
  reg_fence32(r3);
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    s[i] = __uint_as_float(r0[i]);
    s[32 + i] = __uint_as_float(r1[i]);
    s[64 + i] = __uint_as_float(r2[i]);
    s[96 + i] = __uint_as_float(r3[i]);
    if (MASK) {
      if (i > rel_lim) s[i] = -INFINITY;
      if (32 + i > rel_lim) s[32 + i] = -INFINITY;
      if (64 + i > rel_lim) s[64 + i] = -INFINITY;
      if (96 + i > rel_lim) s[96 + i] = -INFINITY;
    }
  }
}
__device__ __forceinline__ float row_max_regs(const float (&s)[kBN]) {
  float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    m0 = fmax3(m0, s[i], s[i + 1]);
    m1 = fmax3(m1, s[32 + i], s[33 + i]);
    m2 = fmax3(m2, s[64 + i], s[65 + i]);
    m3 = fmax3(m3, s[96 + i], s[97 + i]);
  }
  return fmax3(fmaxf(m0, m1), m2, m3);
}

// Single-read form: a block's P is first formed in the row's current frame f.  Its row sum can exceed
// kSumTrigger only when some P does, and every P stays below 2^margin = e^10 unless the block
// max outgrows the frame by more than the margin; so a warp in which no row's sum exceeds it
// keeps those P without ever forming the block max.  Otherwise (or on a row's first block,
// f = -inf) the frame test proper runs: the block max, the frame move when it exceeds f by
// more than the margin, and P formed again in the new frame.  The frame decisions are exactly
// those of testing every block's max.  kSumTrigger sits just below e^10, so that the rounding
// of the exponential cannot hide a P at the bound.
constexpr float kSumTrigger = 21800.f;


// One key block of the online softmax for this thread's query row: read S(j), move the frame f
// to the block max when that exceeds f by more than the margin (l and, when it already holds
// earlier blocks (o_live), O are scaled by 2^(f_old - f)), write P = 2^(s - f) over S and add
// its row sum to l.  O may be rescaled in place: S(j) being ready means PV(j-1) has completed
// (QK(j) was issued after it).  The caller waits for the TMEM stores.
//
// One TMEM wait per block: the 128 scores stay in registers (168 a thread in every layout;
// with q4_0 sides by a register split between warpgroups) and P is formed in the current frame
// first.
//
// pmx tracks a bound on the largest P written (before its rounding to the dtype), each in the
// frame in force for its block: the exact largest P of a block that ran the frame test (P is
// monotonic in the score), the block's sum of P otherwise (at least its largest P, and below
// kSumTrigger).  Either way pmx <= e^10 whenever the frame rule holds.
struct NoWait {
  __device__ void operator()() const {}
};
// wait_o runs before O is rescaled in tensor memory (a PV MMA may still be adding to it when the
// S buffers alternate within one query tile)
template <int D, bool BF16, class WaitO = NoWait>
__device__ __forceinline__ void softmax_block(uint32_t scol, uint32_t ocol, bool need_mask,
                                              int rel_lim, float sl2, bool o_live, float& f,
                                              float& l, int& nres, float& pmx,
                                              const WaitO& wait_o = WaitO()) {
  auto rescale_o = [&](float alpha) {
    wait_o();
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(ocol + 32 * c, r);
      tmem_wait_ld();
      reg_fence32(r);
#pragma unroll
      for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
      tmem_st32(ocol + 32 * c, r);
    }
  };
  // the frame test proper: block max mx (scaled to m2), frame move, O rescale; true if any row
  // of the warp moved its frame
  auto frame_test = [&](float mx, float& alpha) -> bool {
    const float m2 = mx * sl2;
    const bool need = m2 > f + kMarginLog2;
    alpha = 1.f;
    if (need) {
      alpha = ex2(f - m2);
      l *= alpha;
      f = m2;
      ++nres;
    }
    return __any_sync(0xffffffffu, need);
  };
  const bool first = __any_sync(0xffffffffu, f == -INFINITY);
  float s[kBN];
  if (need_mask)
    block_row_scores<true>(scol, rel_lim, s);
  else
    block_row_scores<false>(scol, rel_lim, s);
  float sum = 0.f;
  bool done = false;
  if (!first) {
    sum = block_row_exp_regs<BF16>(scol, s, sl2, -f);
    done = !__any_sync(0xffffffffu, sum > kSumTrigger);
  }
  if (done) {
    pmx = fmaxf(pmx, sum);
  } else {
    const float mx = row_max_regs(s);
    float alpha;
    const bool any = frame_test(mx, alpha);
    if (any || first) {
      sum = block_row_exp_regs<BF16>(scol, s, sl2, -f);
      if (any && o_live) rescale_o(alpha);
    }
    pmx = fmaxf(pmx, ex2(fmaf(mx, sl2, -f)));  // -inf keys (a masked row) give 0
  }
  l += sum;
}

// One q4_0 dequant item: the 32 elements of block blk of key row t of a raw tile (nibble rows of
// NIB bytes, 64B-swizzled at D = 128 and 32B-swizzled at D = 64, then the fp16 scale rows of SROW
// bytes from byte RAWNIB), expanded to (q - 8) * d in f16/bf16 into the 128B-swizzled ring stage.
template <int D, bool BF16, int NIB, int SROW, int RAWNIB>
__device__ __forceinline__ void dequant_item(const uint8_t* raw, uint8_t* dst, int t, int blk,
                                             uint32_t mg) {
  const uint8_t* nrow = raw + t * NIB;
  const __half* srow = reinterpret_cast<const __half*>(raw + RAWNIB + t * SROW);
    // 16 bytes of nibbles of this key, 64B-swizzled (D=128) or 32B-swizzled (D=64)
    const int chunk = (D == 128) ? (blk ^ ((t >> 1) & 3)) : (blk ^ ((t >> 2) & 1));
    const uint4 wv = *reinterpret_cast<const uint4*>(nrow + 16 * chunk);
    const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
    const __half dh = srow[blk];
    uint32_t outv[16];  // 32 dequantized elements, packed in pairs, natural order
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      // bytes 4q..4q+3 -> elements 4q..4q+3 (low) and 4q+16..4q+19 (high)
      const uint32_t a = __byte_perm(w[q], 0u, 0x5150);   // byte0 at b0, byte1 at b2
      const uint32_t c2 = __byte_perm(w[q], 0u, 0x5352);  // byte2 at b0, byte3 at b2
      if (BF16) {
        const float d = __half2float(dh);
        outv[2 * q + 0] = Dq<true>::scale(Dq<true>::lo(a, mg), d);
        outv[2 * q + 1] = Dq<true>::scale(Dq<true>::lo(c2, mg), d);
        outv[8 + 2 * q + 0] = Dq<true>::scale(Dq<true>::hi(a, mg), d);
        outv[8 + 2 * q + 1] = Dq<true>::scale(Dq<true>::hi(c2, mg), d);
      } else {
        outv[2 * q + 0] = Dq<false>::scale(Dq<false>::lo(a, mg), dh);
        outv[2 * q + 1] = Dq<false>::scale(Dq<false>::lo(c2, mg), dh);
        outv[8 + 2 * q + 0] = Dq<false>::scale(Dq<false>::hi(a, mg), dh);
        outv[8 + 2 * q + 1] = Dq<false>::scale(Dq<false>::hi(c2, mg), dh);
      }
    }
    // elements 32 blk + 8 cc .. +7 form 16-byte chunk (4 blk + cc) of the row
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      const int col16 = 4 * blk + cc;        // 16-byte chunk index along D
      const int atom = col16 >> 3;           // 64-element swizzle atom
      const int ch = (col16 & 7) ^ (t & 7);  // 128B swizzle
      *reinterpret_cast<uint4*>(dst + atom * (kBN * 128) + t * 128 + ch * 16) =
          make_uint4(outv[4 * cc], outv[4 * cc + 1], outv[4 * cc + 2], outv[4 * cc + 3]);
    }
}

// number of 128-key blocks a query tile starting at row q0 must visit
__host__ __device__ __forceinline__ int tile_blocks(const PrefillArgs& a, int q0) {
  if (q0 >= a.Sq) return 0;
  const int last_row = min(q0 + kBM - 1, a.Sq - 1);
  const int kend = a.causal ? min(a.Sk, a.q_pos_offset + last_row + 1) : a.Sk;
  return (kend + kBN - 1) / kBN;
}

// ALT: one query tile per CTA (dense K/V) whose key blocks alternate between the two S buffers
template <int D, bool BF16, bool KQ4, bool VQ4, bool ALT>
__global__ void __launch_bounds__(Cfg<D, KQ4, VQ4, true>::kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefillArgs args) {
  using C = Cfg<D, KQ4, VQ4, true>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - smem_u32(smem_raw));
  const uint32_t bar0 = sbase + C::kOffBar;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + C::kOffBar + kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sgen + C::kOffBar + kOffTmemSlot);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // work unit: a pair of consecutive query tiles of one head, longest pairs first (the slowest
  // grid dimension enumerates units); tile B may lie past Sq (odd tile count).  With
  // unit_rows = 128 each unit is one query tile and tile B is absent.
  const int h = blockIdx.x;
  const int b = blockIdx.y;
  const int unit = args.n_pairs - 1 - static_cast<int>(blockIdx.z);
  const int q0A = unit * args.unit_rows;
  const int q0B = q0A + kBM;
  const int g = h / (args.Hq / args.Hkv);
  const int nbA = tile_blocks(args, q0A);
  const int nbB = args.unit_rows == kBM ? 0 : tile_blocks(args, q0B);
  const int nbmax = max(nbA, nbB);  // causal rows further down see at least as many keys
  const bool hasB = nbB > 0;

  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQFull), 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(kBarSFull + t), 1);
      mbar_init(bar(kBarPReady + t), 128);
      mbar_init(bar(kBarODone + t), 1);
    }
    mbar_init(bar(kBarDrain), 1);
    for (int s = 0; s < C::kStages; ++s) {
      // a q4_0 stage is filled by the dequant threads, a dense one by the TMA lane
      const bool q4s = (C::kStages % 2 == 0) ? ((s & 1) ? VQ4 : KQ4) : (KQ4 && VQ4);
      mbar_init(bar(kBarRingFull + s), q4s ? C::kDqThreads : 1);
      mbar_init(bar(kBarRingEmpty + s), 1);
    }
    for (int s = 0; s < C::kRawStages; ++s) {
      mbar_init(bar(kBarRawFull + s), 1 + 32);  // TMA lane + 32 cp.async arrivals
      mbar_init(bar(kBarRawEmpty + s), C::kDqThreads);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Roles by warpgroup first.  With a q4_0 side (sixteen warps) the two softmax warpgroups
  // raise their registers to 168 a thread and the other two lower theirs to 88 (setmaxnreg is
  // executed by whole warpgroups, so warps 0-3 take it together before splitting into producer,
  // issuer and dequant), and the softmax keeps a block's 128 scores in registers as with dense
  // K/V; 2 x 128 x 168 + 2 x 128 x 88 is exactly the 65 536 registers the launch reserved.
  if (warp < 4 || warp >= 12) {
    if constexpr (C::kWide) asm volatile("setmaxnreg.dec.sync.aligned.u32 88;" ::: "memory");
    if (warp == 0) {
      // ---------------------------------------------------------------- producer
      if (lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
      }
      bool ok = true;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(kBarQFull), (hasB ? 2 : 1) * C::kQBytes);
        for (int t = 0; t < (hasB ? 2 : 1); ++t)
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(sbase + C::kOffQ + t * C::kQBytes + c * (kBM * 128), &tm_q,
                        bar(kBarQFull), c * 64, t ? q0B : q0A, b * args.Hq + h);
      }
      // tiles in the order the MMA first uses them: K0, V0, K1, V1, ...; dense tiles go by TMA
      // straight into the ring, q4_0 tiles (nibbles + scales) into the raw stages
      int n = 0;  // ring tiles
      int r = 0;  // raw q4_0 tiles
      auto produce = [&](bool is_v, int j) {
        if (!ok) return;
        if (!(is_v ? VQ4 : KQ4)) {
          const int s = n % C::kStages;
          if (lane == 0) {
            if (n >= C::kStages)
              ok = mbar_wait(bar(kBarRingEmpty + s), ((n / C::kStages) - 1) & 1, abort_flag,
                             &g_prefill_error);
            if (ok) {
              mbar_arrive_expect_tx(bar(kBarRingFull + s), C::kTileBytes);
              const uint32_t dst = sbase + C::kOffRing + s * C::kTileBytes;
              for (int c = 0; c < D / 64; ++c)
                tma_load_3d(dst + c * (kBN * 128), is_v ? &tm_v : &tm_k, bar(kBarRingFull + s),
                            c * 64, j * kBN, b * args.Hkv + g);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        } else if constexpr (C::kAnyQ4) {  // a q4_0 side: raw stages exist
          const int s = r % C::kRawStages;
          if (r >= C::kRawStages) {
            if (lane == 0)
              ok = mbar_wait(bar(kBarRawEmpty + s), ((r / C::kRawStages) - 1) & 1, abort_flag,
                             &g_prefill_error);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) return;
          }
          const uint32_t dst = sbase + C::kOffRaw + s * C::kRawBytes;
          if (lane == 0) {
            mbar_arrive_expect_tx(bar(kBarRawFull + s), C::kRawNib);
            tma_load_3d(dst, is_v ? &tm_v : &tm_k, bar(kBarRawFull + s), 0, j * kBN,
                        b * args.Hkv + g);
          }
          // scales: one 4- or 8-byte row per key, zero-filled past Sk
          const uint8_t* sp = is_v ? args.v_scale : args.k_scale;
          for (int row = lane; row < kBN; row += 32) {
            const int key = j * kBN + row;
            const bool in = key < args.Sk;
            const uint8_t* src =
                sp + (static_cast<int64_t>(b * args.Hkv + g) * args.Scap + (in ? key : 0)) *
                         C::kScaleRow;
            const uint32_t d = dst + C::kRawNib + row * C::kScaleRow;
            if (C::kScaleRow == 8)
              cp_async_8(d, src, in ? 8u : 0u);
            else
              cp_async_4(d, src, in ? 4u : 0u);
          }
          cp_async_mbar_arrive_noinc(bar(kBarRawFull + s));
          ++r;
        }
        ++n;
      };
      // dense K/V: one slot per block step, K tile in its first stage, V tile in its second
      int pg = 0;  // slots filled
      auto produce_pair = [&](int kj, int vj) {
        if (!ok) return;
        const int p = pg % C::kSlots;
        if (lane == 0) {
          if (pg >= C::kSlots)
            ok = mbar_wait(bar(kBarRingEmpty + p), ((pg / C::kSlots) - 1) & 1, abort_flag,
                           &g_prefill_error);
          if (ok) {
            mbar_arrive_expect_tx(bar(kBarRingFull + p),
                                  ((kj >= 0 ? 1 : 0) + (vj >= 0 ? 1 : 0)) * C::kTileBytes);
            const uint32_t dst = sbase + C::kOffRing + 2 * p * C::kTileBytes;
            for (int c = 0; c < D / 64; ++c) {
              if (kj >= 0)
                tma_load_3d(dst + c * (kBN * 128), &tm_k, bar(kBarRingFull + p), c * 64, kj * kBN,
                            b * args.Hkv + g);
              if (vj >= 0)
                tma_load_3d(dst + C::kTileBytes + c * (kBN * 128), &tm_v, bar(kBarRingFull + p),
                            c * 64, vj * kBN, b * args.Hkv + g);
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (ok) ++pg;
      };
      if constexpr (C::kPaired) {
        produce_pair(0, -1);
        for (int j = 0; j < nbmax; ++j) produce_pair(j + 1 < nbmax ? j + 1 : -1, j);
      } else {
        for (int j = 0; j < nbmax; ++j) {
          produce(false, j);
          produce(true, j);
        }
      }
      if (!ok && lane == 0) {
        // let copies already issued land before the CTA's shared memory goes away: the last
        // dense tiles sent into the ring and the last raw q4_0 tiles
        volatile int never = 0;
        if constexpr (C::kPaired) {
          for (int i = max(0, pg - C::kSlots); i < pg; ++i)
            mbar_wait(bar(kBarRingFull + i % C::kSlots), (i / C::kSlots) & 1, &never, nullptr,
                      kWaitLimitNs);
        }
        for (int i = max(0, n - C::kStages); i < n; ++i)
          if (!((i & 1) ? VQ4 : KQ4))
            mbar_wait(bar(kBarRingFull + i % C::kStages), (i / C::kStages) & 1, &never, nullptr,
                      kWaitLimitNs);
        if constexpr (C::kAnyQ4) {
          for (int i = max(0, r - C::kRawStages); i < r; ++i)
            mbar_wait(bar(kBarRawFull + i % C::kRawStages), (i / C::kRawStages) & 1, &never,
                      nullptr, kWaitLimitNs);
        }
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------------- MMA issuer
      if (lane == 0) {
        constexpr uint32_t idesc_qk = make_idesc_f16(kBM, kBN, BF16, false);
        constexpr uint32_t idesc_pv = make_idesc_f16(kBM, D, BF16, true);
        bool ok = mbar_wait(bar(kBarQFull), 0, abort_flag, &g_prefill_error);
        tc_fence_after();
        int n = 0;
        auto acquire = [&]() -> int {
          const int s = n % C::kStages;
          if (ok) ok = mbar_wait(bar(kBarRingFull + s), (n / C::kStages) & 1, abort_flag,
                                 &g_prefill_error);
          tc_fence_after();
          ++n;
          return s;
        };
        auto release = [&](int s) { mma_commit(bar(kBarRingEmpty + s)); };
        // QK of query tile t into S buffer sb (tile t's own, except in the alternating mode)
        auto issue_qk = [&](int t, int s, int sb) {
          const uint32_t qaddr = sbase + C::kOffQ + t * C::kQBytes;
          const uint32_t kaddr = sbase + C::kOffRing + s * C::kTileBytes;
  #pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * (kBM * 128) + (kk & 3) * 32;
            mma_ss(tmem + col_s(sb), make_sdesc_sw128(qaddr + off, 16, 1024),
                   make_sdesc_sw128(kaddr + off, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(kBarSFull + sb));
        };
        auto issue_pv = [&](int t, int j, int s, int nb_t) {
          ok = ok && mbar_wait(bar(kBarPReady + t), j & 1, abort_flag, &g_prefill_error);
          if (!ok) return;
          tc_fence_after();
          const uint32_t vaddr = sbase + C::kOffRing + s * C::kTileBytes;
          const uint32_t ocol = t ? C::kColO1 : C::kColO0;
  #pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            mma_ts(tmem + ocol, tmem + col_s(t) + kk * 8,
                   make_sdesc_sw128(vaddr + kk * (16 * 128), kBN * 128, 1024), idesc_pv,
                   (j > 0 || kk > 0) ? 1u : 0u);
          if (j == nb_t - 1) mma_commit(bar(kBarODone + t));
        };
        // PV of block j of a lone query tile whose blocks alternate between the S buffers; tile
        // B's O-done barrier, unused then, completes after every PV (the softmax waits for it
        // before it rescales O)
        auto issue_pv_alt = [&](int j, int s, int nb_t) {
          const int sb = j & 1;
          ok = ok && mbar_wait(bar(kBarPReady + sb), (j >> 1) & 1, abort_flag, &g_prefill_error);
          if (!ok) return;
          tc_fence_after();
          const uint32_t vaddr = sbase + C::kOffRing + s * C::kTileBytes;
  #pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            mma_ts(tmem + C::kColO0, tmem + col_s(sb) + kk * 8,
                   make_sdesc_sw128(vaddr + kk * (16 * 128), kBN * 128, 1024), idesc_pv,
                   (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(bar(kBarODone + 1));
          if (j == nb_t - 1) mma_commit(bar(kBarODone));
        };
        // order: QK_A(0) QK_B(0) | PV_A(j) QK_A(j+1) PV_B(j) QK_B(j+1) | ...  A K/V stage is
        // acquired at the start of the step that first uses it and released after its last use
        // (all in ring order).
        if constexpr (C::kPaired) {
          // one slot per step: V(j) in stage 2p + 1, K(j + 1) in stage 2p
          int gn = 0;
          auto acquire_g = [&]() -> int {
            const int p = gn % C::kSlots;
            if (ok) ok = mbar_wait(bar(kBarRingFull + p), (gn / C::kSlots) & 1, abort_flag,
                                   &g_prefill_error);
            tc_fence_after();
            ++gn;
            return p;
          };
          if constexpr (ALT) {
            // one query tile whose key blocks alternate between the two S buffers: QK(j + 2) goes
            // into block j's buffer right after PV(j) has read P from it, so the softmax finds
            // block j + 1's scores ready when it finishes block j.  Slot 0 holds K(0), slot g
            // holds V(g - 1) and K(g).
            int pvs = 0;  // the slot holding the V of the next PV
            if (nbA > 0 && ok) {
              const int p = acquire_g();
              if (ok) {
                issue_qk(0, 2 * p, 0);
                release(p);
                pvs = acquire_g();
                if (ok && nbA > 1) issue_qk(0, 2 * pvs, 1);
              }
            }
            for (int j = 0; j < nbA && ok; ++j) {
              issue_pv_alt(j, 2 * pvs + 1, nbA);
              if (!ok) break;
              release(pvs);
              if (j + 1 < nbA) {
                pvs = acquire_g();
                if (ok && j + 2 < nbA) issue_qk(0, 2 * pvs, j & 1);
              }
            }
          } else {
          if (nbmax > 0 && ok) {
            const int p = acquire_g();
            if (ok) {
              if (nbA > 0) issue_qk(0, 2 * p, 0);
              if (nbB > 0)
                issue_qk(1, 2 * p, 1);  // tile B's softmax releases the slot
              else
                release(p);
            }
          }
          for (int j = 0; j < nbmax && ok; ++j) {
            const int p = acquire_g();
            const bool next = j + 1 < nbmax;
            if (!ok) break;
            if (j < nbA) issue_pv(0, j, 2 * p + 1, nbA);
            if (!ok) break;
            if (next && j + 1 < nbA) issue_qk(0, 2 * p, 0);
            if (j < nbB) issue_pv(1, j, 2 * p + 1, nbB);
            if (!ok) break;
            if (next && j + 1 < nbB)
              issue_qk(1, 2 * p, 1);
            else
              release(p);
          }
          }
        } else {
        if (nbmax > 0 && ok) {
          const int sK = acquire();
          if (ok) {
            if (nbA > 0) issue_qk(0, sK, 0);
            if (nbB > 0) issue_qk(1, sK, 1);
            release(sK);
          }
        }
        for (int j = 0; j < nbmax && ok; ++j) {
          // both ring waits of the step sit next to the P_A wait: an mbarrier wait issued while
          // the MMA queue is short stalls the issue of the next MMAs, so the waits are grouped
          // where they cost one stall instead of one per wait
          const int sV = acquire();
          const bool next = j + 1 < nbmax;
          const int sK = next ? acquire() : 0;
          if (!ok) break;
          if (j < nbA) issue_pv(0, j, sV, nbA);
          if (!ok) break;
          if (next && j + 1 < nbA) issue_qk(0, sK, 0);
          if (j < nbB) issue_pv(1, j, sV, nbB);
          if (!ok) break;
          release(sV);
          if (next) {
            if (j + 1 < nbB) issue_qk(1, sK, 1);
            release(sK);
          }
        }
        }
        if (!ok) {
          // wait until every MMA issued so far has finished before TMEM is released
          volatile int never = 0;
          mma_commit(bar(kBarDrain));
          mbar_wait(bar(kBarDrain), 0, &never, nullptr, kWaitLimitNs);
        }
      }
    } else if constexpr (C::kAnyQ4) {
      if (C::is_dq_warp(warp)) {
        // -------------------------------------------------------------- q4_0 dequant
        // the dequant threads share out each raw tile's (key row, block) items and expand them
        // into the 128B-swizzled f16/bf16 ring stage
        const int u = C::dq_index(warp, lane);
        const uint32_t mg = opaque_u32(BF16 ? 0x43004300u : 0x64006400u);
        bool ok = true;
        const int ntiles = 2 * nbmax;
        int r = 0;  // raw q4_0 tiles consumed
        for (int n = 0; n < ntiles; ++n) {
          if (!((n & 1) ? VQ4 : KQ4)) continue;  // a dense tile: the producer's TMA fills it
          const int rs = r % C::kRawStages;
          const int s = n % C::kStages;
          ok = mbar_wait(bar(kBarRawFull + rs), (r / C::kRawStages) & 1, abort_flag,
                         &g_prefill_error);
          if (ok && n >= C::kStages)
            ok = mbar_wait(bar(kBarRingEmpty + s), ((n / C::kStages) - 1) & 1, abort_flag,
                           &g_prefill_error);
          if (!ok) break;
          const uint8_t* raw = sgen + C::kOffRaw + rs * C::kRawBytes;
          uint8_t* dst = sgen + C::kOffRing + s * C::kTileBytes;
          // items (key row t, 32-element block blk) of the tile, rows fastest; unrolled so that
          // the items' shared-memory loads overlap
          constexpr int kItems = kBN * (D / 32);
  #pragma unroll
          for (int k = 0; k < (kItems + C::kDqThreads - 1) / C::kDqThreads; ++k) {
            const int it = u + k * C::kDqThreads;
            if (kItems % C::kDqThreads == 0 || it < kItems)
              dequant_item<D, BF16, C::kNibRow, C::kScaleRow, C::kRawNib>(raw, dst, it % kBN,
                                                                          it / kBN, mg);
          }
          // generic-proxy writes must be visible to the tensor core's async proxy
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          mbar_arrive(bar(kBarRingFull + s));
          mbar_arrive(bar(kBarRawEmpty + rs));
          ++r;
        }
      }
  
    }
  } else {
    if constexpr (C::kWide) asm volatile("setmaxnreg.inc.sync.aligned.u32 168;" ::: "memory");
    // ---------------------------------------------------------------- softmax rows
    const int t = (warp >= 8) ? 1 : 0;  // query tile
    const int nb = t ? nbB : nbA;
    const int q0 = t ? q0B : q0A;
    const int row = 32 * (warp & 3) + lane;
    const int qrow = q0 + row;
    const int pos = args.q_pos_offset + qrow;
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t scol_t = tmem + lane_off + col_s(t);
    const uint32_t ocol = tmem + lane_off + (t ? C::kColO1 : C::kColO0);
    const float sl2 = args.scale_log2;
    // a lone query tile (dense K/V) alternates its key blocks between the two S buffers
    constexpr bool alt = ALT;
    static_assert(!ALT || C::kPaired, "alternating S buffers need the paired dense ring");
    float f = -INFINITY;  // frame, base-2 units of the scaled score
    float l = 0.f;
    int nres = 0;
    float pmx = -INFINITY;  // bound on the largest P written
    bool ok = true;
    for (int j = 0; j < nb; ++j) {
      const int sb = alt ? (j & 1) : t;  // S buffer of this block
      const uint32_t scol = alt ? tmem + lane_off + col_s(sb) : scol_t;
      ok = mbar_wait(bar(kBarSFull + sb), alt ? ((j >> 1) & 1) : (j & 1), abort_flag,
                     &g_prefill_error);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if constexpr (C::kPaired) {
        // QK_B of block j done: release the ring slot holding K(j) (slot j of the unit)
        if (t == 1 && warp == 8 && lane == 0) mbar_arrive(bar(kBarRingEmpty + j % C::kSlots));
      }
      const int kb = j * kBN;
      const bool need_mask =
          (kb + kBN > args.Sk) || (args.causal && kb + kBN - 1 > args.q_pos_offset + q0);
      // last visible key of this row, relative to the block
      const int rel_lim = (args.causal ? min(args.Sk - 1, pos) : args.Sk - 1) - kb;
      if constexpr (alt) {
        // PV(j - 1) may still be adding to O when this block moves the frame; PV(j) cannot
        // have started, so the PV-done barrier has completed j - 1 or j times
        auto wait_pv = [&]() {
          mbar_wait(bar(kBarODone + 1), (j - 1) & 1, abort_flag, &g_prefill_error);
          tc_fence_after();
        };
        softmax_block<D, BF16>(scol, ocol, need_mask, rel_lim, sl2, j > 0,
                                                    f, l, nres, pmx, wait_pv);
      } else {
        softmax_block<D, BF16>(scol, ocol, need_mask, rel_lim, sl2, j > 0,
                                                    f, l, nres, pmx);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(kBarPReady + sb));
    }
    if (ok && nb > 0) {
      // the tile's last PV MMA completing implies all of its MMAs have
      ok = mbar_wait(bar(kBarODone + t), 0, abort_flag, &g_prefill_error);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok && nb > 0) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      const bool store = qrow < args.Sq;
      uint8_t* orow = static_cast<uint8_t*>(args.o) +
                      ((static_cast<int64_t>(b * args.Hq + h) * args.Sq + qrow) * D) * 2;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(ocol + 32 * c, r);
        tmem_wait_ld();
        reg_fence32(r);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack2<BF16>(__uint_as_float(r[2 * i]) * inv_l,
                              __uint_as_float(r[2 * i + 1]) * inv_l);
        if (store) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 64);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      if (store && args.rescale_count)
        args.rescale_count[static_cast<int64_t>(b * args.Hq + h) * args.Sq + qrow] = nres;
      if (store && args.p_max)
        args.p_max[static_cast<int64_t>(b * args.Hq + h) * args.Sq + qrow] = pmx;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------------------------------
// Cut schedule.  A work unit is a pair of consecutive 128-row query tiles (A, B) of one query
// head; it takes nbmax steps, step j being key block j for both tiles.  Units are ordered by
// pair (longest first), then batch, then head, and their steps concatenated; the sequence is cut
// into equal contiguous ranges, one per resident CTA.  A CTA's range is a run of segments -- the
// tail of one unit, whole units, the head of another -- so every SM does the same number of
// steps and none idles through a last partial wave.  A unit cut between CTAs is finished by
// whichever of its CTAs finds all its pieces published.
// ------------------------------------------------------------------------------------------
__host__ __device__ __forceinline__ int pair_steps(const PrefillArgs& a, int z) {
  const int q0A = 2 * (a.n_pairs - 1 - z) * kBM;
  return max(tile_blocks(a, q0A), tile_blocks(a, q0A + kBM));
}

struct Seg {
  int b, h, g, q0A, q0B, nbA, nbB, nbmax, j0, j1;
  bool hasB;
  int64_t unit_start;  // global step of the unit's block 0
};
// a segment as stored in shared memory (computed once per CTA by one thread, read by every role)
struct SegS {
  int b, h, q0A, nbA, nbB, nbmax, j0, j1;
  int64_t unit_start;
};

// the segment that starts at global step t of a range ending at t_end; false if t lies past
// the last unit, which a consistent schedule never asks for
__host__ __device__ __forceinline__ bool locate(const PrefillArgs& a, int64_t t, int64_t t_end,
                                                Seg& sg) {
  const int64_t per_class = static_cast<int64_t>(a.B) * a.Hq;
  int64_t acc = 0;
  int z = 0;
  int nbm = pair_steps(a, 0);
  while (t >= acc + per_class * nbm) {
    acc += per_class * nbm;
    if (++z >= a.n_pairs || t < 0 || nbm <= 0) return false;
    nbm = pair_steps(a, z);
  }
  if (nbm <= 0) return false;
  const int64_t within = t - acc;
  const int64_t idx = within / nbm;
  sg.j0 = static_cast<int>(within - idx * nbm);
  sg.b = static_cast<int>(idx / a.Hq);
  sg.h = static_cast<int>(idx % a.Hq);
  sg.g = sg.h / (a.Hq / a.Hkv);
  sg.q0A = 2 * (a.n_pairs - 1 - z) * kBM;
  sg.q0B = sg.q0A + kBM;
  sg.nbA = tile_blocks(a, sg.q0A);
  sg.nbB = tile_blocks(a, sg.q0B);
  sg.nbmax = nbm;
  sg.hasB = sg.q0B < a.Sq;
  sg.unit_start = t - sg.j0;
  sg.j1 = static_cast<int>(min(static_cast<int64_t>(nbm), sg.j0 + (t_end - t)));
  return sg.j1 > sg.j0;
}
// first global step of CTA c's range (equal cuts)
__host__ __device__ __forceinline__ int64_t range_start(const PrefillArgs& a, int c) {
  return c >= a.n_ctas ? a.W : static_cast<int64_t>(c) * a.W / a.n_ctas;
}
// the CTA whose range holds global step t
__host__ __device__ __forceinline__ int cta_of(const PrefillArgs& a, int64_t t) {
  return static_cast<int>(((t + 1) * a.n_ctas - 1) / a.W);
}
// the same, and a piece's partial slot, on plain scalars (W steps over n CTAs): slot 0 when the
// unit is where CTA c's range begins, 1 when the CTA reached it after other segments
__host__ __device__ __forceinline__ int64_t cut_start(int c, int64_t W, int n) {
  return c >= n ? W : static_cast<int64_t>(c) * W / n;
}
__host__ __device__ __forceinline__ int cut_cta_of(int64_t t, int64_t W, int n) {
  return static_cast<int>(((t + 1) * n - 1) / W);
}
__host__ __device__ __forceinline__ int cut_slot(int c, int64_t unit_start, int64_t W, int n) {
  return cut_start(c, W, n) >= unit_start ? 0 : 1;
}
// CTA c's segments in order (at most kMaxSegs); -1 if its range does not fit the table or
// runs past the last unit, which a consistent plan never produces
__host__ __device__ __forceinline__ int build_segments(const PrefillArgs& a, int c, SegS* segs) {
  const int64_t t_end = range_start(a, c + 1);
  int ns = 0;
  for (int64_t tt = range_start(a, c); tt < t_end;) {
    Seg sg;
    if (ns >= kMaxSegs || !locate(a, tt, t_end, sg)) return -1;
    segs[ns] = SegS{sg.b, sg.h, sg.q0A, sg.nbA, sg.nbB, sg.nbmax, sg.j0, sg.j1, sg.unit_start};
    ++ns;
    tt += sg.j1 - sg.j0;
  }
  return ns;
}
// one tile of a piece, column-major so that a warp's 32 rows of one column are 128 contiguous
// bytes: [D + 4 columns][128 rows] f32, columns O[0..D), frame, row sum, frame moves, the
// bound on the largest P
template <int D>
__device__ __forceinline__ float* part_tile(float* part, int c, int slot, int t) {
  return part + ((static_cast<int64_t>(c) * 2 + slot) * 2 + t) * (D + 4) * kBM;
}

// record a schedule fault and stop the CTA's roles
__device__ __forceinline__ void schedule_fault(volatile int* abort_flag) {
  *abort_flag = 1;
  atomicCAS(&g_prefill_error, kErrNone, kErrSchedule);
}

// Bounded wait (all lanes of the warp) for an appended block's flag, with acquire semantics;
// then a proxy fence, so that the tensor copies this warp issues next read the stored block.
// Gives up when the CTA aborts or after the wait limit (then records a timeout).
__device__ __forceinline__ bool app_wait(const uint32_t* flag, volatile int* abort_flag) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
  if (v == 0u) {
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
      __nanosleep(64);
      asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
      if (v != 0u) break;
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        atomicCAS(&g_prefill_error, kErrNone, kErrTimeout);
        return false;
      }
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}

// Epilogue of one piece of a unit cut between CTAs, run by both tiles' softmax warps: store
// this row's (O, frame, row sum, frame moves), release O, publish the piece's flag, and merge
// all pieces if this CTA finds them all published.  Of two pieces published at the same time at
// least one sees the other's flag (release store, then a sequentially consistent fence before
// the flag loads), so at least one CTA merges; every CTA that does writes the same bytes.  Both
// CTA-wide waits are bounded mbarriers.  Kept out of line: it runs a few times per CTA and would
// otherwise take registers from the softmax loop.  Returns false if a bounded wait gave up.
template <int D, bool BF16>
__device__ __noinline__ bool piece_epilogue(int64_t W, int n_ctas, float* part,
                                            uint32_t* pflags, uint32_t tag,
                                            int32_t* rescale_count, float* p_max, void* o,
                                            int Hq, int Sq, const SegS* sgp, uint32_t ocol,
                                            bool active, float f, float l, int nres, float pmx,
                                            uint32_t bar0, int pseg,
                                            volatile int* abort_flag,
                                            volatile uint32_t* merge_flag) {
  // everything else follows from the thread and the segment (kept out of the caller's registers)
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int t = (warp >= 8) ? 1 : 0;
  const int row = 32 * (warp & 3) + lane;
  const int cta = static_cast<int>(blockIdx.x);
  const int64_t unit_start = sgp->unit_start;
  const int nbmax = sgp->nbmax;
  const int qrow = sgp->q0A + t * kBM + row;
  const bool exists = sgp->q0A + t * kBM < Sq;
  const bool store = exists && qrow < Sq;
  const int64_t orow_idx = static_cast<int64_t>(sgp->b * Hq + sgp->h) * Sq + qrow;
  uint8_t* orow = static_cast<uint8_t*>(o) + orow_idx * D * 2;
  const int slot = cut_slot(cta, unit_start, W, n_ctas);
  if (exists) {
    float* pt = part_tile<D>(part, cta, slot, t) + row;
    if (active) {
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(ocol + 32 * c, r);
        tmem_wait_ld();
        reg_fence32(r);
#pragma unroll
        for (int i = 0; i < 32; ++i) pt[(32 * c + i) * kBM] = __uint_as_float(r[i]);
      }
    }
    pt[D * kBM] = active ? f : -INFINITY;
    pt[(D + 1) * kBM] = active ? l : 0.f;
    pt[(D + 2) * kBM] = __int_as_float(active ? nres : 0);
    pt[(D + 3) * kBM] = active ? pmx : -INFINITY;
  }
  if (active) {
    // O has been read out of tensor memory: the next segment's PV may overwrite it
    tc_fence_before();
    mbar_arrive(bar0 + 8u * (kBarOFree + t));
  }
  const int c_first = cut_cta_of(unit_start, W, n_ctas);
  const int c_last = cut_cta_of(unit_start + nbmax - 1, W, n_ctas);
  mbar_arrive(bar0 + 8u * kBarPiece);
  if (warp == 4) {
    bool okw = mbar_wait(bar0 + 8u * kBarPiece, pseg & 1, abort_flag, &g_prefill_error);
    okw = __all_sync(0xffffffffu, okw);
    bool all = false;
    if (okw) {
      if (lane == 0) st_release_gpu(pflags + 2 * cta + slot, tag);
      __syncwarp();
      fence_sc_gpu();
      all = true;
      for (int c = c_first + lane; c <= c_last; c += 32)
        all = all && ld_relaxed_gpu(pflags + 2 * c + cut_slot(c, unit_start, W, n_ctas)) == tag;
      all = __all_sync(0xffffffffu, all);
      if (all) fence_acq_rel_gpu();
    }
    if (lane == 0) {
      *merge_flag = all ? 1u : 0u;
      mbar_arrive(bar0 + 8u * kBarMergeDecided);
    }
  }
  const bool ok = mbar_wait(bar0 + 8u * kBarMergeDecided, pseg & 1, abort_flag, &g_prefill_error);
  if (!__all_sync(0xffffffffu, ok)) return false;
  const bool merge = *merge_flag != 0u;
  if (merge && exists) {
    // frame F = max over the pieces, weights 2^(f_p - F), pieces in CTA order
    auto tile_of = [&](int c) -> const float* {
      return part_tile<D>(part, c, cut_slot(c, unit_start, W, n_ctas), t) + row;
    };
    float F = -INFINITY;
    for (int c = c_first; c <= c_last; ++c) F = fmaxf(F, __ldcg(tile_of(c) + D * kBM));
    // frame moves: each piece counts its own first frame; the row as a whole counts one
    float L = 0.f;
    int moves = 1;
    float T = -INFINITY;  // the pieces' bounds on their largest P (each in its own frame)
    for (int c = c_first; c <= c_last; ++c) {
      const float* pc = tile_of(c);
      const float fp = __ldcg(pc + D * kBM);
      if (fp == -INFINITY) continue;
      L = fmaf(ex2(fp - F), __ldcg(pc + (D + 1) * kBM), L);
      moves += __float_as_int(__ldcg(pc + (D + 2) * kBM)) - 1;
      T = fmaxf(T, __ldcg(pc + (D + 3) * kBM));
    }
    const float inv_l = 1.f / L;
    // half a row (D/2 columns) of every piece in turn, all of a piece's loads issued together:
    // one L2 round trip per piece and half row, not one per piece and 16 columns
    constexpr int kH = D / 2;
#pragma unroll 1
    for (int h2 = 0; h2 < 2; ++h2) {
      float acc[kH];
#pragma unroll
      for (int i = 0; i < kH; ++i) acc[i] = 0.f;
      for (int c = c_first; c <= c_last; ++c) {
        const float* pc = tile_of(c);
        const float fp = __ldcg(pc + D * kBM);
        float v[kH];
#pragma unroll
        for (int i = 0; i < kH; ++i) v[i] = __ldcg(pc + (kH * h2 + i) * kBM);
        if (fp == -INFINITY) continue;
        const float w = ex2(fp - F);
#pragma unroll
        for (int i = 0; i < kH; ++i) acc[i] = fmaf(w, v[i], acc[i]);
      }
      if (store) {
#pragma unroll
        for (int cc = 0; cc < kH / 8; ++cc) {
          uint32_t pk[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            pk[i] = pack2<BF16>(acc[8 * cc + 2 * i] * inv_l, acc[8 * cc + 2 * i + 1] * inv_l);
          reinterpret_cast<uint4*>(orow + kH * 2 * h2)[cc] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
    }
    if (store && rescale_count) rescale_count[orow_idx] = moves;
    if (store && p_max) p_max[orow_idx] = T;
  }
  if (merge && warp == 4) {
    // clear the unit's flags for the next call (or graph replay) with this tag
    for (int c = c_first + lane; c <= c_last; c += 32)
      st_relaxed_gpu(pflags + 2 * c + cut_slot(c, unit_start, W, n_ctas), 0u);
  }
  return true;
}

// ------------------------------------------------------------------------------------------
// The same kernel run over segments of work units (the equal-cuts schedule below): every role
// walks this CTA's segments, a unit cut between CTAs is published as partial rows and merged by
// its last piece.  Used at D = 128 where cutting beats one unit per CTA (more units than SMs,
// long units).
// ------------------------------------------------------------------------------------------
template <int D, bool BF16, bool KQ4, bool VQ4>
__global__ void __launch_bounds__(Cfg<D, KQ4, VQ4, true>::kThreads, 1)
    prefill_seg_kernel(const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefillArgs args) {
  using C = Cfg<D, KQ4, VQ4, true>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - smem_u32(smem_raw));
  const uint32_t bar0 = sbase + C::kOffBar;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + C::kOffBar + kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sgen + C::kOffBar + kOffTmemSlot);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // this CTA's run of key-block steps, an equal cut of all units' steps; each role walks the
  // same segments (see the cut schedule above).  Tile B of a unit may lie past
  // Sq (odd tile count); causal rows further down see at least as many keys, so nbmax = nbB
  // whenever tile B exists.
  const int cta = static_cast<int>(blockIdx.x);
  const int64_t t_begin = range_start(args, cta);
  const int64_t t_end = range_start(args, cta + 1);
  volatile int* seg_count = reinterpret_cast<volatile int*>(sgen + C::kOffBar + kOffSegCount);
  SegS* segs = reinterpret_cast<SegS*>(sgen + C::kOffBar + kOffSegs);

  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQFull), 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(kBarSFull + t), 1);
      mbar_init(bar(kBarPReady + t), 128);
      mbar_init(bar(kBarODone + t), 1);
    }
    mbar_init(bar(kBarDrain), 1);
    mbar_init(bar(kBarQEmpty), 1);
    mbar_init(bar(kBarOFree + 0), 128);
    mbar_init(bar(kBarOFree + 1), 128);
    mbar_init(bar(kBarPiece), 256);
    mbar_init(bar(kBarMergeDecided), 1);
    for (int s = 0; s < C::kStages; ++s) {
      // a q4_0 stage is filled by the dequant threads, a dense one by the TMA lane
      const bool q4s = (C::kStages % 2 == 0) ? ((s & 1) ? VQ4 : KQ4) : (KQ4 && VQ4);
      mbar_init(bar(kBarRingFull + s), q4s ? C::kDqThreads : 1);
      mbar_init(bar(kBarRingEmpty + s), 1);
    }
    for (int s = 0; s < C::kRawStages; ++s) {
      mbar_init(bar(kBarRawFull + s), 1 + 32);  // TMA lane + 32 cp.async arrivals
      mbar_init(bar(kBarRawEmpty + s), C::kDqThreads);
    }
    *abort_flag = 0;
    fence_mbar_init();
    // this CTA's segments, once: the roles read them back instead of each locating them
    int ns = build_segments(args, cta, segs);
    if (ns < 0) {
      schedule_fault(abort_flag);
      ns = 0;
    }
    *seg_count = ns;
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int nseg = *seg_count;

  // Roles by warpgroup first.  With a q4_0 side (sixteen warps) the two softmax warpgroups
  // raise their registers to 168 a thread and the other two lower theirs to 88 (setmaxnreg is
  // executed by whole warpgroups, so warps 0-3 take it together before splitting into producer,
  // issuer and dequant), and the softmax keeps a block's 128 scores in registers as with dense
  // K/V; 2 x 128 x 168 + 2 x 128 x 88 is exactly the 65 536 registers the launch reserved.
  if (warp < 4 || warp >= 12) {
    if constexpr (C::kWide) asm volatile("setmaxnreg.dec.sync.aligned.u32 88;" ::: "memory");
    if (warp == 0) {
      // ---------------------------------------------------------------- producer
      if (lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
      }
      bool ok = true;
      // tiles in the order the MMA first uses them: K0, V0, K1, V1, ... of each segment; dense
      // tiles go by TMA straight into the ring, q4_0 tiles (nibbles + scales) into the raw stages
      int n = 0;   // ring tiles
      int r = 0;   // raw q4_0 tiles
      int qn = 0;  // Q loads issued
      int b = 0, g = 0;  // the segment's batch and kv head
      auto produce = [&](bool is_v, int j) {
        if (!ok) return;
        if (!(is_v ? VQ4 : KQ4)) {
          const int s = n % C::kStages;
          if (lane == 0) {
            if (n >= C::kStages)
              ok = mbar_wait(bar(kBarRingEmpty + s), ((n / C::kStages) - 1) & 1, abort_flag,
                             &g_prefill_error);
            if (ok) {
              mbar_arrive_expect_tx(bar(kBarRingFull + s), C::kTileBytes);
              const uint32_t dst = sbase + C::kOffRing + s * C::kTileBytes;
              for (int c = 0; c < D / 64; ++c)
                tma_load_3d(dst + c * (kBN * 128), is_v ? &tm_v : &tm_k, bar(kBarRingFull + s),
                            c * 64, j * kBN, b * args.Hkv + g);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        } else if constexpr (C::kAnyQ4) {  // a q4_0 side: raw stages exist
          const int s = r % C::kRawStages;
          if (r >= C::kRawStages) {
            if (lane == 0)
              ok = mbar_wait(bar(kBarRawEmpty + s), ((r / C::kRawStages) - 1) & 1, abort_flag,
                             &g_prefill_error);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) return;
          }
          const uint32_t dst = sbase + C::kOffRaw + s * C::kRawBytes;
          if (lane == 0) {
            mbar_arrive_expect_tx(bar(kBarRawFull + s), C::kRawNib);
            tma_load_3d(dst, is_v ? &tm_v : &tm_k, bar(kBarRawFull + s), 0, j * kBN,
                        b * args.Hkv + g);
          }
          // scales: one 4- or 8-byte row per key, zero-filled past Sk
          const uint8_t* sp = is_v ? args.v_scale : args.k_scale;
          for (int row = lane; row < kBN; row += 32) {
            const int key = j * kBN + row;
            const bool in = key < args.Sk;
            const uint8_t* src =
                sp + (static_cast<int64_t>(b * args.Hkv + g) * args.Scap + (in ? key : 0)) *
                         C::kScaleRow;
            const uint32_t d = dst + C::kRawNib + row * C::kScaleRow;
            if (C::kScaleRow == 8)
              cp_async_8(d, src, in ? 8u : 0u);
            else
              cp_async_4(d, src, in ? 4u : 0u);
          }
          cp_async_mbar_arrive_noinc(bar(kBarRawFull + s));
          ++r;
        }
        ++n;
      };
      // dense K/V: one slot per block step, K tile in its first stage, V tile in its second
      int pg = 0;  // slots filled
      auto produce_pair = [&](int kj, int vj) {
        if (!ok) return;
        const int p = pg % C::kSlots;
        if (lane == 0) {
          if (pg >= C::kSlots)
            ok = mbar_wait(bar(kBarRingEmpty + p), ((pg / C::kSlots) - 1) & 1, abort_flag,
                           &g_prefill_error);
          if (ok) {
            mbar_arrive_expect_tx(bar(kBarRingFull + p),
                                  ((kj >= 0 ? 1 : 0) + (vj >= 0 ? 1 : 0)) * C::kTileBytes);
            const uint32_t dst = sbase + C::kOffRing + 2 * p * C::kTileBytes;
            for (int c = 0; c < D / 64; ++c) {
              if (kj >= 0)
                tma_load_3d(dst + c * (kBN * 128), &tm_k, bar(kBarRingFull + p), c * 64, kj * kBN,
                            b * args.Hkv + g);
              if (vj >= 0)
                tma_load_3d(dst + C::kTileBytes + c * (kBN * 128), &tm_v, bar(kBarRingFull + p),
                            c * 64, vj * kBN, b * args.Hkv + g);
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (ok) ++pg;
      };
      for (int sidx = 0; sidx < nseg && ok; ++sidx) {
        const SegS sg = segs[sidx];
        const bool hasB = sg.q0A + kBM < args.Sq;
        b = sg.b;
        g = sg.h / (args.Hq / args.Hkv);
        // the segment's Q tiles, once the previous segment's last QK MMA has read the previous ones
        if (lane == 0) {
          if (sidx > 0)
            ok = mbar_wait(bar(kBarQEmpty), (sidx - 1) & 1, abort_flag, &g_prefill_error);
          if (ok) {
            mbar_arrive_expect_tx(bar(kBarQFull), (hasB ? 2 : 1) * C::kQBytes);
            for (int t = 0; t < (hasB ? 2 : 1); ++t)
              for (int c = 0; c < D / 64; ++c)
                tma_load_3d(sbase + C::kOffQ + t * C::kQBytes + c * (kBM * 128), &tm_q,
                            bar(kBarQFull), c * 64, sg.q0A + t * kBM, sg.b * args.Hq + sg.h);
            ++qn;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if constexpr (C::kPaired) {
          produce_pair(sg.j0, -1);
          for (int j = sg.j0; j < sg.j1; ++j) produce_pair(j + 1 < sg.j1 ? j + 1 : -1, j);
        } else {
        for (int j = sg.j0; j < sg.j1; ++j) {
          if constexpr (KQ4 && VQ4) {
            if (args.app_flags != nullptr && ok && j >= args.app_j_lo &&
                j < args.app_j_lo + args.app_nb) {
              // the block holds appended tokens: wait until phase 1 has stored them
              ok = app_wait(args.app_flags + (b * args.Hkv + g) * args.app_nb + (j - args.app_j_lo),
                            abort_flag);
              ok = __all_sync(0xffffffffu, ok);
            }
          }
          produce(false, j);
          produce(true, j);
        }
        }
      }
      if (!ok && lane == 0) {
        // let copies already issued land before the CTA's shared memory goes away: the last
        // Q tiles, the last dense tiles sent into the ring and the last raw q4_0 tiles
        volatile int never = 0;
        if (qn > 0)
          mbar_wait(bar(kBarQFull), (qn - 1) & 1, &never, nullptr, kWaitLimitNs);
        if constexpr (C::kPaired) {
          for (int i = max(0, pg - C::kSlots); i < pg; ++i)
            mbar_wait(bar(kBarRingFull + i % C::kSlots), (i / C::kSlots) & 1, &never, nullptr,
                      kWaitLimitNs);
        }
        for (int i = max(0, n - C::kStages); i < n; ++i)
          if (!((i & 1) ? VQ4 : KQ4))
            mbar_wait(bar(kBarRingFull + i % C::kStages), (i / C::kStages) & 1, &never, nullptr,
                      kWaitLimitNs);
        if constexpr (C::kAnyQ4) {
          for (int i = max(0, r - C::kRawStages); i < r; ++i)
            mbar_wait(bar(kBarRawFull + i % C::kRawStages), (i / C::kRawStages) & 1, &never,
                      nullptr, kWaitLimitNs);
        }
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------------- MMA issuer
      if (lane == 0) {
        constexpr uint32_t idesc_qk = make_idesc_f16(kBM, kBN, BF16, false);
        constexpr uint32_t idesc_pv = make_idesc_f16(kBM, D, BF16, true);
        bool ok = true;
        int n = 0;
        int prA = 0, prB = 0;    // P-ready waits per tile before this segment (barrier phases)
        int actA = 0, actB = 0;  // earlier segments in which the tile had blocks
        int gn = 0;              // paired ring: slots taken
        auto acquire_g = [&]() -> int {
          const int p = gn % C::kSlots;
          if (ok) ok = mbar_wait(bar(kBarRingFull + p), (gn / C::kSlots) & 1, abort_flag,
                                 &g_prefill_error);
          tc_fence_after();
          ++gn;
          return p;
        };
        auto acquire = [&]() -> int {
          const int s = n % C::kStages;
          if (ok) ok = mbar_wait(bar(kBarRingFull + s), (n / C::kStages) & 1, abort_flag,
                                 &g_prefill_error);
          tc_fence_after();
          ++n;
          return s;
        };
        auto release = [&](int s) { mma_commit(bar(kBarRingEmpty + s)); };
        auto issue_qk = [&](int t, int s) {
          const uint32_t qaddr = sbase + C::kOffQ + t * C::kQBytes;
          const uint32_t kaddr = sbase + C::kOffRing + s * C::kTileBytes;
  #pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * (kBM * 128) + (kk & 3) * 32;
            mma_ss(tmem + col_s(t), make_sdesc_sw128(qaddr + off, 16, 1024),
                   make_sdesc_sw128(kaddr + off, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(kBarSFull + t));
        };
        // PV of tile t for block j of a segment whose blocks for t are [j0, e_t); the P-ready
        // phase of block j is (pb + j) & 1, pb = the tile's earlier P-ready waits - j0
        auto issue_pv = [&](int t, int j, int s, int j0, int e_t, int pb) {
          ok = ok && mbar_wait(bar(kBarPReady + t), (pb + j) & 1, abort_flag, &g_prefill_error);
          if (!ok) return;
          tc_fence_after();
          const uint32_t vaddr = sbase + C::kOffRing + s * C::kTileBytes;
          const uint32_t ocol = t ? C::kColO1 : C::kColO0;
  #pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            mma_ts(tmem + ocol, tmem + col_s(t) + kk * 8,
                   make_sdesc_sw128(vaddr + kk * (16 * 128), kBN * 128, 1024), idesc_pv,
                   (j > j0 || kk > 0) ? 1u : 0u);
          if (j == e_t - 1) mma_commit(bar(kBarODone + t));
        };
        // per segment: QK_A(j0) QK_B(j0) | PV_A(j) QK_A(j+1) PV_B(j) QK_B(j+1) | ...  A K/V stage
        // is acquired at the start of the step that first uses it and released after its last use
        // (all in ring order).  Both ring waits of a step sit next to the P_A wait: an mbarrier
        // wait issued while the MMA queue is short stalls the issue of the next MMAs, so the waits
        // are grouped where they cost one stall instead of one per wait.
        for (int sidx = 0; sidx < nseg && ok; ++sidx) {
          const int j0 = segs[sidx].j0, j1 = segs[sidx].j1;
          const int eA = min(j1, segs[sidx].nbA);
          const int eB = segs[sidx].q0A + kBM < args.Sq ? min(j1, segs[sidx].nbB) : 0;
          ok = mbar_wait(bar(kBarQFull), sidx & 1, abort_flag, &g_prefill_error);
          tc_fence_after();
          if (!ok) break;
          const int pbA = prA - j0, pbB = prB - j0;
          if constexpr (C::kPaired) {
            // one slot per step: V(j) in stage 2p + 1, K(j + 1) in stage 2p
            {
              const int p = acquire_g();
              if (!ok) break;
              if (j0 < eA) issue_qk(0, 2 * p);
              if (j0 < eB)
                issue_qk(1, 2 * p);  // tile B's softmax releases the slot
              else
                release(p);
              if (j0 + 1 == j1) mma_commit(bar(kBarQEmpty));
            }
            if (j0 < eA && actA > 0)
              ok = ok && mbar_wait(bar(kBarOFree + 0), (actA - 1) & 1, abort_flag,
                                   &g_prefill_error);
            if (j0 < eB && actB > 0)
              ok = ok && mbar_wait(bar(kBarOFree + 1), (actB - 1) & 1, abort_flag,
                                   &g_prefill_error);
            for (int j = j0; j < j1 && ok; ++j) {
              const int p = acquire_g();
              const bool next = j + 1 < j1;
              if (!ok) break;
              if (j < eA) issue_pv(0, j, 2 * p + 1, j0, eA, pbA);
              if (!ok) break;
              if (next && j + 1 < eA) issue_qk(0, 2 * p);
              if (j < eB) issue_pv(1, j, 2 * p + 1, j0, eB, pbB);
              if (!ok) break;
              if (next && j + 1 < eB)
                issue_qk(1, 2 * p);
              else
                release(p);
              if (next && j + 2 == j1) mma_commit(bar(kBarQEmpty));
            }
          } else {
          {
            const int sK = acquire();
            if (!ok) break;
            if (j0 < eA) issue_qk(0, sK);
            if (j0 < eB) issue_qk(1, sK);
            release(sK);
            if (j0 + 1 == j1) mma_commit(bar(kBarQEmpty));  // no further QK reads these Q tiles
          }
          // a tile's first PV of the segment overwrites O: wait until the previous segment's
          // epilogue has read it (after this segment's first QKs are on their way)
          if (j0 < eA && actA > 0)
            ok = ok && mbar_wait(bar(kBarOFree + 0), (actA - 1) & 1, abort_flag, &g_prefill_error);
          if (j0 < eB && actB > 0)
            ok = ok && mbar_wait(bar(kBarOFree + 1), (actB - 1) & 1, abort_flag, &g_prefill_error);
          for (int j = j0; j < j1 && ok; ++j) {
            const int sV = acquire();
            const bool next = j + 1 < j1;
            const int sK = next ? acquire() : 0;
            if (!ok) break;
            if (j < eA) issue_pv(0, j, sV, j0, eA, pbA);
            if (!ok) break;
            if (next && j + 1 < eA) issue_qk(0, sK);
            if (j < eB) issue_pv(1, j, sV, j0, eB, pbB);
            if (!ok) break;
            release(sV);
            if (next) {
              if (j + 1 < eB) issue_qk(1, sK);
              release(sK);
              if (j + 2 == j1) mma_commit(bar(kBarQEmpty));
            }
          }
          }
          if (j0 < eA) {
            ++actA;
            prA += eA - j0;
          }
          if (j0 < eB) {
            ++actB;
            prB += eB - j0;
          }
        }
        if (!ok) {
          // wait until every MMA issued so far has finished before TMEM is released
          volatile int never = 0;
          mma_commit(bar(kBarDrain));
          mbar_wait(bar(kBarDrain), 0, &never, nullptr, kWaitLimitNs);
        }
      }
    } else if constexpr (C::kAnyQ4) {
      if (C::is_dq_warp(warp)) {
        // -------------------------------------------------------------- q4_0 dequant
        // the dequant threads share out each raw tile's (key row, block) items and expand them
        // into the 128B-swizzled f16/bf16 ring stage
        const int u = C::dq_index(warp, lane);
        const uint32_t mg = opaque_u32(BF16 ? 0x43004300u : 0x64006400u);
        bool ok = true;
        const int ntiles = static_cast<int>(2 * (t_end - t_begin));  // K and V of every step
        int r = 0;  // raw q4_0 tiles consumed
        for (int n = 0; n < ntiles; ++n) {
          if (!((n & 1) ? VQ4 : KQ4)) continue;  // a dense tile: the producer's TMA fills it
          const int rs = r % C::kRawStages;
          const int s = n % C::kStages;
          ok = mbar_wait(bar(kBarRawFull + rs), (r / C::kRawStages) & 1, abort_flag,
                         &g_prefill_error);
          if (ok && n >= C::kStages)
            ok = mbar_wait(bar(kBarRingEmpty + s), ((n / C::kStages) - 1) & 1, abort_flag,
                           &g_prefill_error);
          if (!ok) break;
          const uint8_t* raw = sgen + C::kOffRaw + rs * C::kRawBytes;
          uint8_t* dst = sgen + C::kOffRing + s * C::kTileBytes;
          // items (key row t, 32-element block blk) of the tile, rows fastest; unrolled so that
          // the items' shared-memory loads overlap
          constexpr int kItems = kBN * (D / 32);
  #pragma unroll
          for (int k = 0; k < (kItems + C::kDqThreads - 1) / C::kDqThreads; ++k) {
            const int it = u + k * C::kDqThreads;
            if (kItems % C::kDqThreads == 0 || it < kItems)
              dequant_item<D, BF16, C::kNibRow, C::kScaleRow, C::kRawNib>(raw, dst, it % kBN,
                                                                          it / kBN, mg);
          }
          // generic-proxy writes must be visible to the tensor core's async proxy
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          mbar_arrive(bar(kBarRingFull + s));
          mbar_arrive(bar(kBarRawEmpty + rs));
          ++r;
        }
      }
  
    }
  } else {
    if constexpr (C::kWide) asm volatile("setmaxnreg.inc.sync.aligned.u32 168;" ::: "memory");
    // ---------------------------------------------------------------- softmax rows
    if constexpr (KQ4 && VQ4) {
      if (args.app_flags != nullptr) {
        // -------------------------------------------------------- phase 1: append the chunk
        // done by the 256 softmax threads while the producer and the MMA issuer fill the
        // pipeline: items c, c + n_ctas, ...: every thread quantizes 32-element blocks of the
        // item's rows (K, then V) with the cache builder's exact sequence; the item's flag is
        // set once all of them are stored
        constexpr int kNb = D / 32;
        const int st = threadIdx.x - 4 * 32;  // 0..255
        const int n_items = args.B * args.Hkv * args.app_nb;
        for (int it = cta; it < n_items; it += args.n_ctas) {
          const int bh = it / args.app_nb;  // b * Hkv + g
          const int jb = args.app_j_lo + it % args.app_nb;
          const int r0 = max(jb * kBN, args.app_pos0);
          const int r1 = min((jb + 1) * kBN, args.app_pos0 + args.app_len);
          const int per_side = (r1 - r0) * kNb;
          for (int t = st; t < 2 * per_side; t += 256) {
            const bool vside = t >= per_side;
            const int tt = vside ? t - per_side : t;
            const int row = r0 + tt / kNb;  // cache token
            const int blk = tt % kNb;
            const uint4* src = reinterpret_cast<const uint4*>(
                (vside ? args.v_new : args.k_new) +
                (static_cast<int64_t>(bh) * args.app_len + (row - args.app_pos0)) * D +
                blk * 32);
            const uint4 w[4] = {__ldg(src), __ldg(src + 1), __ldg(src + 2), __ldg(src + 3)};
            uint4 nb;
            __half sc;
            q4_quantize_block<BF16>(w, nb, sc);
            const int64_t crow = static_cast<int64_t>(bh) * args.Scap + row;
            reinterpret_cast<uint4*>((vside ? args.v_nib : args.k_nib) + crow * (D / 2))[blk] =
                nb;
            (vside ? args.v_scw : args.k_scw)[crow * kNb + blk] = sc;
          }
          asm volatile("bar.sync 2, 256;" ::: "memory");  // the 256 softmax threads
          if (st == 0) {
            // their stores (observed through the barrier) before the flag, for the tensor
            // copies and cp.async loads that other CTAs issue after reading it
            __threadfence();
            asm volatile("fence.proxy.async.global;" ::: "memory");
            st_release_gpu(args.app_flags + it, 1u);
          }
        }
      }
    }
    const int t = (warp >= 8) ? 1 : 0;  // query tile
    const int row = 32 * (warp & 3) + lane;
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t scol = tmem + lane_off + col_s(t);
    const uint32_t ocol = tmem + lane_off + (t ? C::kColO1 : C::kColO0);
    const float sl2 = args.scale_log2;
    volatile uint32_t* merge_flag =
        reinterpret_cast<volatile uint32_t*>(sgen + C::kOffBar + kOffMergeFlag);
    bool ok = true;
    int sf = 0;    // S-full waits so far (barrier phase)
    int od = 0;    // segments in which this tile had blocks (O-done phase)
    int pseg = 0;  // pieces published so far
    int gn = 0;    // paired ring: slots of the segments before this one
    for (int sidx = 0; sidx < nseg && ok; ++sidx) {
      // only what the block loop needs is read before it; the rest after it
      const int j0 = segs[sidx].j0;
      const int g0 = gn - j0;  // ring slot of the one holding K(j): g0 + j
      gn += segs[sidx].j1 - j0 + 1;
      const int q0 = segs[sidx].q0A + t * kBM;
      const int e_t = q0 < args.Sq ? min(segs[sidx].j1, t ? segs[sidx].nbB : segs[sidx].nbA) : 0;
      const int pos = args.q_pos_offset + q0 + row;
      float f = -INFINITY;  // frame, base-2 units of the scaled score
      float l = 0.f;
      int nres = 0;
      float pmx = -INFINITY;  // bound on the largest P written
      for (int j = j0; j < e_t; ++j) {
        ok = mbar_wait(bar(kBarSFull + t), sf & 1, abort_flag, &g_prefill_error);
        ++sf;
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if constexpr (C::kPaired) {
          // QK_B of block j done: release the ring slot holding K(j)
          if (t == 1 && warp == 8 && lane == 0)
            mbar_arrive(bar(kBarRingEmpty + (g0 + j) % C::kSlots));
        }
        const int kb = j * kBN;
        const bool need_mask =
            (kb + kBN > args.Sk) || (args.causal && kb + kBN - 1 > args.q_pos_offset + q0);
        // last visible key of this row, relative to the block
        const int rel_lim = (args.causal ? min(args.Sk - 1, pos) : args.Sk - 1) - kb;
        // O holds this segment's earlier blocks when j > j0
        softmax_block<D, BF16>(scol, ocol, need_mask, rel_lim, sl2, j > j0, f,
                                              l, nres, pmx);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(kBarPReady + t));
      }
      if (!ok) break;
      const SegS sg = segs[sidx];
      const bool exists = q0 < args.Sq;
      const bool active = e_t > j0;  // the tile had key blocks in this segment
      const int qrow = q0 + row;
      if (active) {
        // the tile's last PV MMA of the segment completing implies all of its MMAs have
        ok = mbar_wait(bar(kBarODone + t), od & 1, abort_flag, &g_prefill_error);
        ++od;
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      const bool store = exists && qrow < args.Sq;
      const int64_t orow_idx = static_cast<int64_t>(sg.b * args.Hq + sg.h) * args.Sq + qrow;
      uint8_t* orow = static_cast<uint8_t*>(args.o) + orow_idx * D * 2;
      const bool split = cta_of(args, sg.unit_start) != cta_of(args, sg.unit_start + sg.nbmax - 1);
      if (!split) {
        if (active) {
          const float inv_l = 1.f / l;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(ocol + 32 * c, r);
            tmem_wait_ld();
            reg_fence32(r);
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack2<BF16>(__uint_as_float(r[2 * i]) * inv_l,
                                  __uint_as_float(r[2 * i + 1]) * inv_l);
            if (store) {
              uint4* dst = reinterpret_cast<uint4*>(orow + c * 64);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
            }
          }
          if (store && args.rescale_count) args.rescale_count[orow_idx] = nres;
          if (store && args.p_max) args.p_max[orow_idx] = pmx;
          // O has been read out of tensor memory: the next segment's PV may overwrite it
          tc_fence_before();
          mbar_arrive(bar(kBarOFree + t));
        }
      } else {
        ok = piece_epilogue<D, BF16>(args.W, args.n_ctas, args.part, args.pflags, args.tag,
                                     args.rescale_count, args.p_max, args.o, args.Hq, args.Sq,
                                     segs + sidx, ocol, active, f, l, nres, pmx, bar0, pseg,
                                     abort_flag, merge_flag);
        ++pseg;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

// ------------------------------------------------------------------------------------------
// host launch
// ------------------------------------------------------------------------------------------
// The schedule of a launch: W key-block steps over `units` work units; equal cuts over n_ctas
// resident CTAs (one per SM) when that is estimated to finish sooner than one unit per CTA,
// else one unit per CTA.  Estimates in steps: one unit per CTA takes ceil(units / SMs) waves of
// an average unit; equal cuts take W / SMs steps plus ~8 steps per segment boundary (the Q
// reload, the epilogue, the partial write and merge, measured at 16K keys).
struct Plan {
  int64_t W, units;
  int n_ctas;
  bool whole;
  size_t flag_bytes, bytes;
};
// the fields of PrefillArgs that the cut schedule reads, for a call of this shape
static PrefillArgs schedule_args(int B, int Hq, int Hkv, int Sq, int Sk, int q_pos_offset,
                                 int causal) {
  PrefillArgs a{};
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Sq = Sq;
  a.Sk = Sk;
  a.Scap = Sk;
  a.q_pos_offset = causal ? q_pos_offset : 0;
  a.causal = causal;
  a.n_qtiles = (Sq + kBM - 1) / kBM;
  a.n_pairs = (a.n_qtiles + 1) / 2;
  return a;
}

static Plan make_plan(int B, int Hq, int Sq, int Sk, int q_pos_offset, int causal, int D,
                      int num_sms, bool force_cut = false) {
  const PrefillArgs a = schedule_args(B, Hq, Hq, Sq, Sk, q_pos_offset, causal);
  const int64_t per_class = static_cast<int64_t>(B) * Hq;
  Plan p;
  p.units = per_class * a.n_pairs;
  p.W = 0;
  int64_t nb_min = 0;  // the shortest unit
  for (int z = 0; z < a.n_pairs; ++z) {
    const int64_t nb = pair_steps(a, z);
    p.W += per_class * nb;
    if (z == 0 || nb < nb_min) nb_min = nb;
  }
  // a CTA's range spans at most ceil(steps / nb_min) + 2 segments, which must fit its table
  const int64_t per_cta = num_sms > 0 ? (p.W + num_sms - 1) / num_sms : 0;
  const bool fits = nb_min > 0 && (per_cta + nb_min - 1) / nb_min + 2 <= kMaxSegs;
  bool cuts = D == 128 && num_sms > 0 && p.units > num_sms && fits;
  if (force_cut) {
    cuts = D == 128 && num_sms > 0 && fits;
  } else if (cuts) {
    const double avg = static_cast<double>(p.W) / static_cast<double>(p.units);
    const double whole_est = static_cast<double>((p.units + num_sms - 1) / num_sms) * avg;
    const double cut_est = static_cast<double>(per_cta) + 8.0 * (per_cta / avg + 1.0);
    cuts = cut_est < 0.97 * whole_est;
  }
  p.whole = !cuts;
  // one CTA per SM, but never more CTAs than steps: every CTA's range must hold at least one
  // step, since a unit's merge waits for every CTA between its first and its last piece
  p.n_ctas = p.whole ? 0 : static_cast<int>(std::min<int64_t>(num_sms, p.W));
  p.flag_bytes = p.whole ? 0 : (static_cast<size_t>(p.n_ctas) * 2 * sizeof(uint32_t) + 255) /
                                   256 * 256;
  p.bytes = p.whole ? 0
                    : p.flag_bytes + static_cast<size_t>(p.n_ctas) * 2 * 2 * (D + 4) * kBM *
                                         sizeof(float);
  return p;
}

size_t prefill_workspace_bytes(int B, int Hq, int Sq, int Sk, int q_pos_offset, int causal,
                               int D, int num_sms) {
  return make_plan(B, Hq, Sq, Sk, causal ? q_pos_offset : 0, causal, D, num_sms).bytes;
}

int64_t prefill_debug_schedule(int B, int Hq, int Hkv, int Sq, int Sk, int q_pos_offset,
                               int causal, int D, int num_sms, bool force_cut, int64_t* plan,
                               int64_t* rows, int64_t max_rows) {
  const Plan p = make_plan(B, Hq, Sq, Sk, q_pos_offset, causal, D, num_sms);
  PrefillArgs a = schedule_args(B, Hq, Hkv, Sq, Sk, q_pos_offset, causal);
  const bool cut = !p.whole || (force_cut && num_sms > 0 && p.W > 0);
  a.W = p.W;
  // as in the launch: one CTA per SM, never more CTAs than steps
  a.n_ctas = cut ? static_cast<int>(std::min<int64_t>(num_sms, p.W)) : 0;
  if (plan != nullptr) {
    plan[0] = p.whole ? 0 : 1;
    plan[1] = a.n_ctas;
    plan[2] = p.W;
    plan[3] = p.units;
    plan[4] = static_cast<int64_t>(p.bytes);
  }
  if (!cut) return 0;
  int64_t n = 0;
  SegS segs[kMaxSegs];
  for (int c = 0; c < a.n_ctas; ++c) {
    const int ns = build_segments(a, c, segs);
    if (ns < 0) return -1;
    for (int i = 0; i < ns; ++i, ++n) {
      if (rows == nullptr || n >= max_rows) continue;
      const SegS& g = segs[i];
      const bool split = cta_of(a, g.unit_start) != cta_of(a, g.unit_start + g.nbmax - 1);
      int64_t* r = rows + n * kScheduleRowWidth;
      r[0] = c;
      r[1] = g.b;
      r[2] = g.h;
      r[3] = g.q0A;
      r[4] = g.nbA;
      r[5] = g.nbB;
      r[6] = g.nbmax;
      r[7] = g.j0;
      r[8] = g.j1;
      r[9] = g.unit_start;
      r[10] = split ? cut_slot(c, g.unit_start, a.W, a.n_ctas) : -1;
    }
  }
  return n;
}

template <int D, bool BF16, bool KQ4, bool VQ4>
static cudaError_t launch_t(const PrefillLaunch& L, cudaStream_t stream) {
  using C = Cfg<D, KQ4, VQ4, true>;
  static_assert(C::kSmemBytes <= 227 * 1024, "shared memory budget");
  PrefillArgs a{};
  a.o = L.o;
  a.k_scale = static_cast<const uint8_t*>(L.k_scale);
  a.v_scale = static_cast<const uint8_t*>(L.v_scale);
  a.rescale_count = L.rescale_count;
  a.p_max = L.p_max;
  a.B = L.B;
  a.Hq = L.Hq;
  a.Hkv = L.Hkv;
  a.Sq = L.Sq;
  a.Sk = L.Sk;
  a.Scap = L.Scap;
  a.q_pos_offset = L.q_pos_offset;
  a.causal = L.causal;
  a.n_qtiles = (L.Sq + kBM - 1) / kBM;
  // one query tile per CTA when even that many CTAs fit on the SMs at once: the two tiles of a
  // pair share the SM sub-partitions for their softmax, so a lone tile steps faster, and
  // with idle SMs the pair's longer chain is what the launch waits for
  const int pairs = (a.n_qtiles + 1) / 2;
  const bool single = a.n_qtiles > 1 && L.num_sms > 0 &&
                      2LL * L.B * L.Hq * pairs <= static_cast<int64_t>(L.num_sms);
  a.n_pairs = single ? a.n_qtiles : pairs;
  a.unit_rows = single ? kBM : 2 * kBM;
  a.scale_log2 = L.scale * kLog2e;
  a.W = 0;  // one unit per CTA from the grid coordinates; the cut-schedule fields are unused
  a.n_ctas = 0;
  a.part = nullptr;
  a.pflags = nullptr;
  a.tag = 0;
  // a lone query tile with dense K/V also alternates its key blocks between the two S buffers;
  // that form is its own instantiation, so the pair form's code is untouched by it
  constexpr bool kAlt = !KQ4 && !VQ4;
  auto kern = (single && kAlt) ? prefill_kernel<D, BF16, KQ4, VQ4, kAlt>
                               : prefill_kernel<D, BF16, KQ4, VQ4, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(L.Hq, L.B, a.n_pairs);
  kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(L.tm_q, L.tm_k, L.tm_v, a);
  return cudaGetLastError();
}

template <int D, bool BF16>
static cudaError_t launch_fmt(const PrefillLaunch& L, cudaStream_t stream) {
  if (L.kq4) return L.vq4 ? launch_t<D, BF16, true, true>(L, stream)
                          : launch_t<D, BF16, true, false>(L, stream);
  return L.vq4 ? launch_t<D, BF16, false, true>(L, stream)
               : launch_t<D, BF16, false, false>(L, stream);
}

// equal cuts of the step sequence over one CTA per SM (D = 128, any pair of K/V formats)
template <bool BF16, bool KQ4, bool VQ4>
static cudaError_t launch_seg(const PrefillLaunch& L, const Plan& p, cudaStream_t stream) {
  using C = Cfg<128, KQ4, VQ4, true>;
  static_assert(C::kSmemBytes <= 227 * 1024, "shared memory budget");
  auto kern = prefill_seg_kernel<128, BF16, KQ4, VQ4>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e != cudaSuccess) return e;
  PrefillArgs a{};
  a.o = L.o;
  a.k_scale = static_cast<const uint8_t*>(L.k_scale);
  a.v_scale = static_cast<const uint8_t*>(L.v_scale);
  a.rescale_count = L.rescale_count;
  a.p_max = L.p_max;
  a.B = L.B;
  a.Hq = L.Hq;
  a.Hkv = L.Hkv;
  a.Sq = L.Sq;
  a.Sk = L.Sk;
  a.Scap = L.Scap;
  a.q_pos_offset = L.q_pos_offset;
  a.causal = L.causal;
  a.n_qtiles = (L.Sq + kBM - 1) / kBM;
  a.n_pairs = (a.n_qtiles + 1) / 2;
  a.scale_log2 = L.scale * kLog2e;
  a.W = p.W;
  a.n_ctas = p.n_ctas;
  a.pflags = static_cast<uint32_t*>(L.workspace);
  a.part = reinterpret_cast<float*>(static_cast<uint8_t*>(L.workspace) + p.flag_bytes);
  a.tag = L.tag;
  kern<<<dim3(a.n_ctas), C::kThreads, C::kSmemBytes, stream>>>(L.tm_q, L.tm_k, L.tm_v, a);
  return cudaGetLastError();
}

template <bool BF16>
static cudaError_t launch_seg_fmt(const PrefillLaunch& L, const Plan& p, cudaStream_t stream) {
  if (L.kq4) return L.vq4 ? launch_seg<BF16, true, true>(L, p, stream)
                          : launch_seg<BF16, true, false>(L, p, stream);
  return L.vq4 ? launch_seg<BF16, false, true>(L, p, stream)
               : launch_seg<BF16, false, false>(L, p, stream);
}

// The append fused into the cut schedule: the cut is forced (every CTA takes part in phase 1)
// and the launch is cooperative, so that all CTAs are resident together and a producer that
// waits for another CTA's phase-1 item cannot wait on a CTA that has not started.
static int app_blocks(int pos0, int len) { return (pos0 + len - 1) / kBN - pos0 / kBN + 1; }
static size_t app_flag_bytes(int B, int Hkv, int pos0, int len) {
  return (static_cast<size_t>(B) * Hkv * app_blocks(pos0, len) * sizeof(uint32_t) + 255) / 256 *
         256;
}

size_t prefill_append_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Sk, int q_pos_offset,
                                      int D, int num_sms) {
  const Plan p = make_plan(B, Hq, Sq, Sk, q_pos_offset, 1, D, num_sms, true);
  if (p.whole) return 0;
  return p.bytes + app_flag_bytes(B, Hkv, q_pos_offset, Sq);
}

template <bool BF16>
static cudaError_t launch_seg_append(const PrefillLaunch& L, const PrefillAppend& A,
                                     const Plan& p, cudaStream_t stream) {
  using C = Cfg<128, true, true, true>;
  auto kern = prefill_seg_kernel<128, BF16, true, true>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e != cudaSuccess) return e;
  PrefillArgs a{};
  a.o = L.o;
  a.k_scale = static_cast<const uint8_t*>(L.k_scale);
  a.v_scale = static_cast<const uint8_t*>(L.v_scale);
  a.rescale_count = L.rescale_count;
  a.p_max = L.p_max;
  a.B = L.B;
  a.Hq = L.Hq;
  a.Hkv = L.Hkv;
  a.Sq = L.Sq;
  a.Sk = L.Sk;
  a.Scap = L.Scap;
  a.q_pos_offset = L.q_pos_offset;
  a.causal = 1;
  a.n_qtiles = (L.Sq + kBM - 1) / kBM;
  a.n_pairs = (a.n_qtiles + 1) / 2;
  a.scale_log2 = L.scale * kLog2e;
  a.W = p.W;
  a.n_ctas = p.n_ctas;
  uint8_t* ws = static_cast<uint8_t*>(L.workspace);
  a.pflags = reinterpret_cast<uint32_t*>(ws);
  a.part = reinterpret_cast<float*>(ws + p.flag_bytes);
  a.tag = L.tag;
  a.k_new = static_cast<const uint16_t*>(A.k_new);
  a.v_new = static_cast<const uint16_t*>(A.v_new);
  a.k_nib = static_cast<uint8_t*>(A.k_nib);
  a.v_nib = static_cast<uint8_t*>(A.v_nib);
  a.k_scw = static_cast<__half*>(A.k_sc);
  a.v_scw = static_cast<__half*>(A.v_sc);
  a.app_flags = reinterpret_cast<uint32_t*>(ws + p.bytes);
  a.app_pos0 = A.pos0;
  a.app_len = A.len;
  a.app_j_lo = A.pos0 / kBN;
  a.app_nb = app_blocks(A.pos0, A.len);
  e = cudaMemsetAsync(a.app_flags, 0, app_flag_bytes(L.B, L.Hkv, A.pos0, A.len), stream);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_ctas);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, L.tm_q, L.tm_k, L.tm_v, a);
}

cudaError_t prefill_append_launch(const PrefillLaunch& L, const PrefillAppend& A,
                                  cudaStream_t stream) {
  if (L.D != 128 || !L.kq4 || !L.vq4) return cudaErrorNotSupported;
  const Plan p = make_plan(L.B, L.Hq, L.Sq, L.Sk, L.q_pos_offset, 1, L.D, L.num_sms, true);
  if (p.whole) return cudaErrorNotSupported;
  if (L.workspace == nullptr ||
      L.workspace_bytes < p.bytes + app_flag_bytes(L.B, L.Hkv, A.pos0, A.len))
    return cudaErrorInvalidValue;
  return L.bf16 ? launch_seg_append<true>(L, A, p, stream)
                : launch_seg_append<false>(L, A, p, stream);
}

cudaError_t prefill_launch(const PrefillLaunch& L, cudaStream_t stream) {
  if (L.D == 128) {
    const Plan p = make_plan(L.B, L.Hq, L.Sq, L.Sk, L.q_pos_offset, L.causal, L.D, L.num_sms);
    if (!p.whole && L.workspace != nullptr && L.workspace_bytes >= p.bytes)
      return L.bf16 ? launch_seg_fmt<true>(L, p, stream) : launch_seg_fmt<false>(L, p, stream);
  }
  if (L.D == 128)
    return L.bf16 ? launch_fmt<128, true>(L, stream) : launch_fmt<128, false>(L, stream);
  return L.bf16 ? launch_fmt<64, true>(L, stream) : launch_fmt<64, false>(L, stream);
}

uint32_t prefill_take_error() {
  uint32_t v = 0;
  if (cudaMemcpyFromSymbol(&v, g_prefill_error, sizeof(v)) != cudaSuccess) return 0xffffffffu;
  const uint32_t z = 0;
  cudaMemcpyToSymbol(g_prefill_error, &z, sizeof(z));
  return v;
}

}  // namespace fa
