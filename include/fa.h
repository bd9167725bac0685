/*
 * fa.h -- C ABI of the GB300 (sm_103a) fused causal GQA flash-attention forward with an optional
 * q4_0 K/V cache.
 *
 * Operation (fa_fwd): for every batch b, query head h and query row i
 *
 *     O[b,h,i,:] = sum_j softmax_j( scale * <Q[b,h,i,:], K[b,g,j,:]> + mask(i,j) ) * V[b,g,j,:]
 *
 * with g = h / (Hq / Hkv) (grouped-query heads in contiguous groups) and, when causal, key j
 * hidden from row i iff j > q_pos_offset + i.  This is the fused prefill call of
 * "perf(rocm): defer SDPA accumulator rescale, stage Q once per block (#2306)" (Conversation:
 * chunked-prefill query chunks against 2K-16K keys, GQA 32/8, head dim 128; What changed: the
 * deferred O/l rescale with its 10-point margin and Q staged once per block) and the
 * flash_attn_func / scaled_dot_product_attention(is_causal=True) call of "Build FlashAttention
 * (CK backend) on gfx90a" (Verification).  With kv_format = FA_KV_Q4_0 the K and V caches are
 * q4_0 and are dequantized inside the kernel, the fused V dequant that "FlashAttention on gfx90a:
 * Why It's Broken and How to Fix It" (Why FA-off Can't Do V Quantization; The V Dequantization
 * Gap) describes as what the flash-attention path provides.
 *
 * Conventions shared by every entry point
 *  - All tensors are device memory of the current device (the kernels launch there), owned by
 *    the caller, contiguous, head-major:
 *      Q, O : [B, Hq, Sq, D]        K, V (dense) : [B, Hkv, Sk, D]   (dtype of Q)
 *    Every pointer must be 16-byte aligned.  The entry points check alignment and sizes but
 *    cannot tell host memory or another device's memory from the current device's: such a
 *    pointer is undefined behaviour (the Python binding refuses those tensors before calling).
 *  - q4_0 tensor (one buffer per K or V, built by fa_quantize_q4_0), for a [B, H, S, D] source:
 *      nibble plane [B, H, S, D/2] uint8 at offset 0: byte j of each 32-element block holds
 *        element j in its low nibble and element j+16 in its high nibble;
 *      scale plane  [B, H, S, D/32] fp16 at offset fa_q4_0_scale_offset(B,H,S,D) (256-aligned).
 *    Element value = (nibble - 8) * scale.  The pages name q4_0 (-ctk q4_0 -ctv q4_0) without
 *    fixing its bits; this planar layout carries exactly the bits of the usual 18-byte
 *    {fp16 d, 16 bytes of nibbles} block and converts to it losslessly.
 *  - Every call is asynchronous on `stream` (0 = legacy default stream).  The return value
 *    reports host-side argument checks and launch errors only; faults detected on the device
 *    (a bounded wait that ran out) are reported by fa_get_status.
 *  - Calls are thread-safe; concurrent calls on different streams are independent.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fa_stream_t; /* a cudaStream_t */

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad shape, bad causal offset, scale */
  FA_ERR_UNSUPPORTED = 2,   /* valid but not implemented: D not in {64, 128}, group size > 8 */
  FA_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed */
  FA_ERR_TIMEOUT = 4        /* a device-side bounded wait ran out (see fa_get_status) */
} fa_status;

typedef enum { FA_F16 = 0, FA_BF16 = 1 } fa_dtype;

typedef enum {
  FA_KV_DENSE = 0, /* K, V in the dtype of Q */
  FA_KV_Q4_0 = 1   /* K, V are q4_0 tensors (see above) */
} fa_kv_format;

/* Attention forward.
 *  q, o      : [B, Hq, Sq, D] in `dtype`
 *  k, v      : [B, Hkv, Sk, D] in `dtype` (FA_KV_DENSE) or q4_0 tensors of that shape
 *  B, Hq, Hkv, Sq, Sk >= 1, Hq % Hkv == 0, Hq / Hkv <= 8 when Sq == 1; D in {64, 128}
 *  q_pos_offset : absolute position of query row 0 (used when causal); requires
 *                 0 <= q_pos_offset and q_pos_offset + Sq <= Sk, so that no row is fully masked
 *                 (Sk - Sq gives the bottom-right aligned chunked-prefill mask)
 *  causal    : nonzero for the causal mask
 *  scale     : softmax scale, finite and > 0 (typically 1/sqrt(D))
 * Sq == 1 runs the split-K decode kernels and needs a scratch buffer of fa_workspace_bytes().
 * Sq >= 2 runs the prefill kernel; where there are more work units than SMs and cutting them
 * evenly over one CTA per SM is estimated to finish sooner (D = 128), it uses
 * fa_workspace_bytes() of scratch for the partial rows of units cut between CTAs; with less
 * scratch (or none) it runs one unit per CTA.  fa_fwd takes the scratch from the stream-ordered
 * allocator (cudaMallocAsync/cudaFreeAsync on `stream`); if that fails, decode returns
 * FA_ERR_CUDA and prefill runs one unit per CTA.  Use fa_fwd_ex to pass the scratch instead. */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv,
                 int Sq, int Sk, int D, int q_pos_offset, int causal, float scale,
                 fa_dtype dtype, fa_kv_format kv_format, fa_stream_t stream);

/* fa_fwd with caller-provided scratch and an optional rescale counter.
 *  workspace, workspace_bytes : device buffer of at least fa_workspace_bytes(...) bytes (may be
 *                 NULL when that is 0; for Sq >= 2 a smaller or NULL buffer selects one work
 *                 unit per CTA); owned by the caller, must not be used by another call in
 *                 flight at the same time.  Its contents on entry do not matter: it holds one
 *                 32-bit arrival flag per split of each (batch, kv head) -- prefill: per piece
 *                 slot of each CTA -- which is set to a tag drawn afresh for every call once the
 *                 partial result behind it is stored, then the partial results, which the piece
 *                 that finds all its siblings' flags set merges (it also clears those flags).  A
 *                 call reads only what it wrote itself, apart from the flags; a stale flag is
 *                 mistaken for this call's only if it holds exactly the call's 32-bit tag.
 *  rescale_count : optional device int32 [B, Hq, Sq] (NULL to skip).  The prefill kernel writes
 *                 for every query row how many times its softmax frame was moved (the first
 *                 key block always sets it, so every value is >= 1); the deferred rescale
 *                 ("perf(rocm): defer SDPA accumulator rescale, stage Q once per block
 *                 (#2306)", Summary) fires only on the moves after the first.  Not written
 *                 when Sq == 1. */
fa_status fa_fwd_ex(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv,
                    int Sq, int Sk, int D, int q_pos_offset, int causal, float scale,
                    fa_dtype dtype, fa_kv_format kv_format, void* workspace,
                    size_t workspace_bytes, int32_t* rescale_count, fa_stream_t stream);

/* fa_fwd_ex over K/V caches with independent formats and a token capacity.
 * The cache configuration "FlashAttention on gfx90a: Why It's Broken and How to Fix It" (The V
 * Dequantization Gap; Impact of the V Dequant Patch) describes users being pushed into -- f16 K
 * with a q4_0 V, set separately with -ctk / -ctv -- and the chunked-prefill flow where a chunk
 * attends to a cache that is larger than the tokens filled so far.
 *  k, v       : [B, Hkv, kv_capacity, D] each, in its own format: k_format / v_format (dense in
 *               the dtype of Q, or a q4_0 tensor built for [B, Hkv, kv_capacity, D]);
 *               only tokens 0 .. Sk - 1 of each (batch, kv head) are read
 *  kv_capacity: >= Sk (the cache's allocated length; Sk = tokens filled)
 *  Other arguments, scratch, errors: as fa_fwd_ex (fa_workspace_bytes covers every pair of
 *  formats).  fa_fwd_ex(…) is fa_fwd_kv with k_format = v_format and kv_capacity = Sk. */
fa_status fa_fwd_kv(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv,
                    int Sq, int Sk, int kv_capacity, int D, int q_pos_offset, int causal,
                    float scale, fa_dtype dtype, fa_kv_format k_format, fa_kv_format v_format,
                    void* workspace, size_t workspace_bytes, int32_t* rescale_count,
                    fa_stream_t stream);

/* fa_fwd_kv that also reports, per query row, a bound on the largest softmax numerator P it
 * produced.  The deferred rescale of "perf(rocm): defer SDPA accumulator rescale, stage Q once
 * per block (#2306)" (What changed) keeps a row's frame f until a key block's maximum score
 * exceeds it by more than 10 natural-log units, so every P = e^(s - f) the kernel writes stays
 * at or below e^10 = 22026.47 (up to the rounding of the f32 exponent argument).  This call
 * exposes that bound for testing.
 *  p_max : optional device float [B, Hq, Sq] (NULL to skip): for every query row the largest,
 *          over its key blocks, of a per-block value that is at least the block's largest P
 *          (before its rounding to the dtype, in the frame in force for that block): the
 *          block's largest P where the kernel tested the block's max against the frame, its
 *          sum of P where the sum already showed that no P can reach the bound (the kernels
 *          form P in the current frame first and run the frame test only when a block's sum
 *          exceeds 21 800, just below e^10).  Where the cut schedule splits a row between CTAs,
 *          the largest over the pieces.  So p_max <= e^10 holds exactly when no written P
 *          exceeds e^10 by more than the rounding above.  Not written when Sq == 1.
 *  Other arguments, scratch, errors: as fa_fwd_kv (which is this call with p_max = NULL). */
fa_status fa_fwd_kv_stats(const void* q, const void* k, const void* v, void* o, int B, int Hq,
                          int Hkv, int Sq, int Sk, int kv_capacity, int D, int q_pos_offset,
                          int causal, float scale, fa_dtype dtype, fa_kv_format k_format,
                          fa_kv_format v_format, void* workspace, size_t workspace_bytes,
                          int32_t* rescale_count, float* p_max, fa_stream_t stream);

/* Scratch bytes fa_fwd_ex needs for this shape on the current device (decode: the split
 * partials; prefill: the partial rows of work units cut between CTAs, 0 when the launch runs
 * one unit per CTA). */
size_t fa_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Sk, int D, int q_pos_offset,
                          int causal);

/* Size of the fixed scratch area behind fa_fwd_decode_noalloc (4 MiB). */
#define FA_NOALLOC_SCRATCH_BYTES (4u << 20)

/* Decode (one query token per sequence, Sq = 1) that allocates no device memory.
 * The pages have no counterpart of this entry point: it exists for callers that cannot allocate
 * on the call path -- runtimes that reserve all device memory at start-up and manage it
 * themselves, or hosts that forbid allocation once serving has started because an allocation
 * may block on the device.  fa_fwd takes decode scratch from the stream-ordered allocator and
 * fa_fwd_ex needs a caller-provided buffer; this call instead uses a fixed device array of
 * FA_NOALLOC_SCRATCH_BYTES that the library itself holds on every GPU that loads it, until the
 * process exits.  It calls no cudaMalloc, cudaFree or other allocating routine.
 *  Arguments: as fa_fwd with Sq = 1 (q, o: [B, Hq, 1, D]; k, v: [B, Hkv, Sk, D] dense or q4_0).
 *  Limit: a shape is accepted exactly when
 *      fa_workspace_bytes(B, Hq, Hkv, 1, Sk, D, q_pos_offset, causal) <= FA_NOALLOC_SCRATCH_BYTES
 *    -- that query is the largest need over every pair of cache formats, so the answer does not
 *    depend on kv_format -- and rejected with FA_ERR_UNSUPPORTED otherwise.  The need grows
 *    with B * Hq times the split count the decode plan picks for the device (about
 *    3 * SM count / (B * Hkv), at least 1, at most the key tiles), so call fa_workspace_bytes
 *    to know whether a shape fits.  Invalid shapes give FA_ERR_INVALID_ARG.
 *  First call per device: it looks up the array's device address (cudaGetSymbolAddress) with
 *    that device current, so make the first call on each device before any stream capture.  The
 *    address is kept per device together with the context it was looked up in, and looked up
 *    again when a call finds another context current (after cudaDeviceReset, say): that call
 *    too should not be captured.
 *  Sharing: every call on a device uses the same array and leaves its contents behind.  Nothing
 *    in it needs clearing (see the workspace of fa_fwd_ex), but calls whose
 *    execution overlaps on the GPU -- on different streams, or from different host threads --
 *    race on the array and produce wrong results; order them on one stream or with events. */
fa_status fa_fwd_decode_noalloc(const void* q, const void* k, const void* v, void* o, int B,
                                int Hq, int Hkv, int Sk, int D, int q_pos_offset, int causal,
                                float scale, fa_dtype dtype, fa_kv_format kv_format,
                                fa_stream_t stream);

/* Decode for a batch of sequences of different lengths over a paged K/V cache: the batch-4
 * server session named in "perf(rocm): defer SDPA accumulator rescale, stage Q once per block
 * (#2306)", Conversation (benchmark session page), with the cache of "FlashAttention on gfx90a:
 * Why It's Broken and How to Fix It", Impact of the V Dequant Patch, kept in q4_0.
 *  q, o        : [B, Hq, 1, D] in `dtype`; sequence b's query is its last token and sees all of
 *                its seq_lens[b] keys
 *  k_pages,
 *  v_pages     : page pools [num_pages, Hkv, page_size, D], each dense (dtype of Q) or a q4_0
 *                tensor built for that shape (fa_q4_0_bytes(num_pages, Hkv, page_size, D))
 *  block_table : device int32 [B, pages_per_seq]: physical page of logical page p of sequence b
 *                (entries past a sequence's last page are not read)
 *  seq_lens    : device int32 [B], 1 <= seq_lens[b] <= pages_per_seq * page_size
 *  page_size   : a multiple of 128 tokens when either side is q4_0, of 64 otherwise
 *  workspace   : >= fa_decode_paged_workspace_bytes(...) bytes, contents on entry irrelevant
 *                (see fa_fwd_ex); the split plan is sized for the longest possible sequence.
 * Host-side checks return FA_ERR_INVALID_ARG / FA_ERR_UNSUPPORTED; a page number or length out of
 * range found on the device is recorded (that tile reads zeros) and fa_get_status then returns
 * FA_ERR_INVALID_ARG. */
size_t fa_decode_paged_workspace_bytes(int B, int Hq, int Hkv, int D, int page_size,
                                       int pages_per_seq);
fa_status fa_decode_paged(const void* q, const void* k_pages, const void* v_pages, void* o,
                          const int32_t* block_table, const int32_t* seq_lens, int B, int Hq,
                          int Hkv, int D, int num_pages, int page_size, int pages_per_seq,
                          float scale, fa_dtype dtype, fa_kv_format k_format,
                          fa_kv_format v_format, void* workspace, size_t workspace_bytes,
                          fa_stream_t stream);

/* The explicit (non-flash) attention path, for comparison with fa_fwd_kv: q4_0 sides are first
 * expanded to dense f16/bf16, S = scale * Q K^T is written out in f32 by a batched GEMM, a
 * softmax kernel makes P (causal mask, rounded to the dtype), and O = P V is a second batched
 * GEMM -- Approach C of "FlashAttention on gfx90a: Why It's Broken and How to Fix It" (dequantize
 * K and V, two GEMMs and a softmax), the path that page measures against flash attention.  Both
 * GEMMs are this library's own tcgen05 kernel; S tiles that the causal mask hides from every row
 * are not computed and the P V GEMM stops at each row tile's last visible key.
 *  Arguments: as fa_fwd_kv without a capacity (K, V: [B, Hkv, Sk, D] each, dense or q4_0).
 *  workspace: >= fa_explicit_workspace_bytes(...) bytes: S (4 bytes per score), P (2 bytes per
 *             score), rows padded to a multiple of 64 keys, and per q4_0 side its dense copy --
 *             about B*Hq*Sq*Sk*6 bytes, so this path is for moderate shapes (Hq = 32,
 *             Sq = 2048, Sk = 16384 needs 6.4 GB).
 *  Errors: as fa_fwd_ex; a tensor map the driver cannot encode gives FA_ERR_CUDA. */
size_t fa_explicit_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Sk, int D,
                                   fa_kv_format k_format, fa_kv_format v_format);
fa_status fa_fwd_explicit(const void* q, const void* k, const void* v, void* o, int B, int Hq,
                          int Hkv, int Sq, int Sk, int D, int q_pos_offset, int causal,
                          float scale, fa_dtype dtype, fa_kv_format k_format,
                          fa_kv_format v_format, void* workspace, size_t workspace_bytes,
                          fa_stream_t stream);

/* Size in bytes of a q4_0 tensor for a [B, H, S, D] source, and the offset of its scale plane. */
size_t fa_q4_0_bytes(int B, int H, int S, int D);
size_t fa_q4_0_scale_offset(int B, int H, int S, int D);

/* Build a q4_0 tensor from x [B, H, S, D] (`dtype`).  out_q4 has fa_q4_0_bytes(B,H,S,D) bytes.
 * The result is bit-identical to the block definition (f32 multiply and add, each rounded to
 * nearest even; fp16 scale rounded to nearest even).  x must be finite.  D % 32 == 0. */
fa_status fa_quantize_q4_0(const void* x, void* out_q4, int B, int H, int S, int D,
                           fa_dtype dtype, fa_stream_t stream);

/* Append a chunk of new tokens to q4_0 caches: quantizes k_new (and v_new, in the same launch)
 * straight into tokens pos0 .. pos0 + S_new - 1 of each (batch, head) of k_cache (v_cache), with
 * the bits fa_quantize_q4_0 would produce.  This is the step before a chunked prefill over a
 * q4_0 cache ("FlashAttention on gfx90a: Why It's Broken and How to Fix It", Impact of the V
 * Dequant Patch: the cache is stored quantized).
 *  k_new, v_new     : [B, H, S_new, D] in `dtype`, device memory; v_new may be NULL (then
 *                     v_cache must be NULL too)
 *  k_cache, v_cache : q4_0 tensors of fa_q4_0_bytes(B, H, kv_capacity, D) bytes
 *  Requires 0 <= pos0, pos0 + S_new <= kv_capacity, D % 32 == 0; tokens outside the range are
 *  left untouched.  Inputs must be finite. */
fa_status fa_append_q4_0(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                         int B, int H, int S_new, int kv_capacity, int pos0, int D,
                         fa_dtype dtype, fa_stream_t stream);

/* Chunked prefill over q4_0 caches that appends the chunk to the caches in the same launch.
 * The step before the fused path of "FlashAttention on gfx90a: Why It's Broken and How to Fix
 * It" (Impact of the V Dequant Patch: the K/V cache is stored quantized, -ctk q4_0 -ctv q4_0):
 * the chunk's own K and V are quantized into the caches and the chunk's queries attend to the
 * whole cache, its own tokens included, as stored.
 *  q, o           : [B, Hq, S_new, D] in `dtype`; query row i sits at position pos0 + i
 *  k_new, v_new   : [B, Hkv, S_new, D] in `dtype`, the chunk's keys and values (finite)
 *  k_cache,
 *  v_cache        : q4_0 tensors built for [B, Hkv, kv_capacity, D]; tokens 0 .. pos0 - 1 hold
 *                   the earlier chunks; tokens pos0 .. pos0 + S_new - 1 are overwritten with the
 *                   bits fa_append_q4_0 writes; tokens past pos0 + S_new are untouched
 *  Result: exactly fa_append_q4_0(k_new, v_new, ...) followed by fa_fwd_kv(q, k_cache,
 *  v_cache, o, ..., Sk = pos0 + S_new, q_pos_offset = pos0, causal = 1, both formats q4_0).
 *  Requires 0 <= pos0, pos0 + S_new <= kv_capacity, D in {64, 128}, and the shape checks of
 *  fa_fwd.  workspace: >= fa_prefill_append_workspace_bytes(...) bytes, contents on entry
 *  irrelevant (see fa_fwd_ex); the call also clears a small region of it with
 *  cudaMemsetAsync on `stream`.
 *  How it runs: at D = 128 one cooperative launch of the cut-schedule prefill, one CTA per SM:
 *  every CTA first quantizes its share of the chunk (per (batch, kv head, 128-token cache
 *  block)) and publishes it with a flag; a CTA's loads of a cache block holding chunk tokens
 *  wait for that block's flag.  Other shapes (D = 64, or work too large for one CTA per SM's
 *  segment table) run the append and the prefill as two launches on `stream`, with the same
 *  result. */
size_t fa_prefill_append_workspace_bytes(int B, int Hq, int Hkv, int S_new, int kv_capacity,
                                         int D, int pos0);
fa_status fa_prefill_append_q4_0(const void* q, const void* k_new, const void* v_new,
                                 void* k_cache, void* v_cache, void* o, int B, int Hq, int Hkv,
                                 int S_new, int kv_capacity, int D, int pos0, float scale,
                                 fa_dtype dtype, void* workspace, size_t workspace_bytes,
                                 fa_stream_t stream);

/* Synchronize `stream`, then report (and clear) any device-side error recorded by this
 * library's kernels since the last call: FA_ERR_TIMEOUT when a bounded wait inside a kernel ran
 * out (the kernel then abandoned its work and returned), FA_ERR_INVALID_ARG when a device-side
 * index input was out of range (fa_decode_paged), FA_ERR_UNSUPPORTED when a prefill CTA's
 * share of the work did not fit its segment table (see fa_prefill_schedule; the launch plans
 * never produce one), FA_ERR_CUDA when the stream reports a CUDA error, FA_OK otherwise. */
fa_status fa_get_status(fa_stream_t stream);

/* Human-readable name of a status code (static storage). */
const char* fa_status_string(fa_status s);

/* Self-test of the bounded-wait machinery: launches one tiny kernel that waits on a barrier
 * nothing will complete, with a limit of `limit_ns` nanoseconds (clamped to [1e3, 1e9]).  The
 * kernel records FA_ERR_TIMEOUT and returns; fa_get_status then reports it.  No GPU fault, trap
 * or hang is involved. */
fa_status fa_debug_wait_timeout(int64_t limit_ns, fa_stream_t stream);

/* The prefill's work schedule for a call of this shape on a device with `num_sms` SMs, computed
 * on the host by the same code the kernel runs (no device is needed or touched).  The schedule
 * is this library's own arrangement of the sums that fa_fwd computes (attention forward, the
 * sections cited at fa_fwd): it changes which CTA adds which key blocks, not the result's
 * definition.
 *
 * A work unit is a pair of consecutive 128-row query tiles (A at q0A, B at q0A + 128) of one
 * query head and batch; it takes nbmax = max(nbA, nbB) key-block steps, where nbA and nbB are the
 * 128-key blocks holding any key visible to tile A or B.  Units are ordered by pair index from
 * the last query tiles to the first, then batch, then head, and their steps concatenated into W
 * steps.  When the plan cuts (D = 128, more units than SMs, and an estimate favours it), CTA c
 * of num_sms runs the steps [floor(c W / num_sms), floor((c + 1) W / num_sms)).  When it keeps
 * one unit per CTA and twice the units fit on the SMs at once (2 x units <= num_sms, more than
 * one query tile), that launch gives each query tile a CTA of its own instead of a pair (tile B
 * absent), so that no two tiles share an SM; the result is the same.
 *
 * plan (5 values, may be NULL): {cut (1) or one unit per CTA (0), CTAs of the cut launch (0 when
 * not cut), W, units, workspace bytes the cut needs}.  force_cut != 0 lays the cuts out over
 * num_sms CTAs even where the plan keeps whole units (plan[0] still reports the plan's choice).
 * rows (max_rows x 11 int64, row-major, caller-owned, may be NULL when max_rows is 0): one row
 * per segment, CTA by CTA in order: {cta, batch, query head, q0A, nbA, nbB, nbmax, j0, j1,
 * unit_start, slot} -- steps [j0, j1) of the unit whose step 0 is global step unit_start; slot is
 * the partial-result slot (0 or 1) of a unit cut between CTAs, else -1.
 * Returns the number of segments (rows beyond max_rows are counted, not written), 0 when the
 * launch runs one unit per CTA, -1 when a CTA's range needs more segments than the kernel's
 * segment table holds (only under force_cut: the plan keeps whole units for such shapes; a
 * kernel that met it would stop and fa_get_status would report FA_ERR_UNSUPPORTED), -2 for
 * invalid arguments (the checks of fa_fwd; Sq >= 2; num_sms >= 1). */
int64_t fa_prefill_schedule(int B, int Hq, int Hkv, int Sq, int Sk, int D, int q_pos_offset,
                            int causal, int num_sms, int force_cut, int64_t* plan,
                            int64_t* rows, int64_t max_rows);

/* The decode kernels' work split, computed on the host by the kernels' own plan code (no device
 * is needed or touched).  Like fa_prefill_schedule this is this library's arrangement of the
 * decode sums (fa_fwd with Sq == 1, and fa_decode_paged): which CTA adds which keys, and the
 * splits that the launch merges.
 *  seq_lens == NULL: a uniform batch of B sequences of Sk keys each (fa_fwd decode at position
 *    Sk - 1): every (sequence, kv head) is cut into the same number of splits, the key tiles
 *    shared out as evenly as whole tiles allow (the first tiles-mod-splits splits take one tile
 *    more); one row per (sequence, split), B x splits rows.
 *  seq_lens != NULL (host array of B lengths): a paged batch (fa_decode_paged) whose pages hold
 *    page_size tokens, pages_per_seq per sequence; the CTAs of a kv head (the row count) are
 *    shared out over the sequences in proportion to their lengths, at least one each, every
 *    length clamped to [1, page_size * pages_per_seq] as the kernel does (which also reports
 *    the out-of-range length), each sequence's key tiles shared out over its CTAs as evenly as
 *    whole tiles allow (a sequence with fewer tiles than CTAs leaves the last ones empty); one
 *    row per CTA.  Sk is ignored.
 * rows (max_rows x 5 int32, row-major, caller-owned; may be NULL when max_rows is 0):
 * {sequence (-1: the CTA has no work), split, splits of that sequence, first key, end key}.
 * Returns the number of rows (rows beyond max_rows are counted, not written), or -2 for
 * invalid arguments (B, Hkv, num_sms >= 1; formats; Sk >= 1 when uniform; page_size >= 1 and
 * a multiple of the kernel's tile, pages_per_seq >= 1, when paged). */
int64_t fa_decode_schedule(const int32_t* seq_lens, int B, int Hkv, int Sk, int page_size,
                           int pages_per_seq, fa_kv_format k_format, fa_kv_format v_format,
                           int num_sms, int32_t* rows, int64_t max_rows);

/* Library ABI version (major * 100 + minor): 101 adds fa_fwd_kv and fa_append_q4_0, 102
 * fa_decode_paged, 103 fa_fwd_explicit, 104 fa_prefill_schedule, 105 fa_decode_schedule, 106 fa_fwd_kv_stats, 107 fa_prefill_append_q4_0. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
