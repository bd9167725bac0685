// Internal host-side interfaces between the C-ABI front end (fa_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

// 3-D tiled TMA map over a contiguous [d2][d1][d0] tensor of esize-byte elements; box =
// {box0, box1, 1}; false if the driver entry point is missing or rejects the arguments
bool encode_map_3d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize,
                   uint64_t d0, uint64_t d1, uint64_t d2, uint32_t box0, uint32_t box1,
                   CUtensorMapSwizzle sw);

struct PrefillLaunch {
  CUtensorMap tm_q, tm_k, tm_v;  // Q tiles; K and V: dense tiles or q4_0 nibble tiles
  void* o;
  const void* k_scale;           // scale plane of a q4_0 K (else null)
  const void* v_scale;           // scale plane of a q4_0 V (else null)
  int32_t* rescale_count;
  float* p_max;                  // optional per-row bound on the largest P (fa_fwd_kv_stats)
  int B, Hq, Hkv, Sq, Sk, Scap, D, q_pos_offset, causal;  // Scap: K/V tokens per (b, kv head)
  float scale;
  bool bf16, kq4, vq4;
  // scratch for the equal-cuts schedule (flags + partial rows; see prefill_workspace_bytes);
  // with less than that the launch runs one work unit per CTA
  void* workspace;
  size_t workspace_bytes;
  uint32_t tag;  // nonzero, different for every call
  int num_sms;
};
cudaError_t prefill_launch(const PrefillLaunch& L, cudaStream_t stream);
// A chunk appended to q4_0 K and V caches by the prefill launch itself: k_new / v_new
// [B, Hkv, len, D] in the dtype, quantized into tokens [pos0, pos0 + len) of the caches (nibble
// and scale planes writable here) before the attention reads those tokens back.
struct PrefillAppend {
  const void* k_new;
  const void* v_new;
  void* k_nib;
  void* v_nib;
  void* k_sc;
  void* v_sc;
  int pos0, len;
};
// the fused append-and-prefill (L: q4_0 K and V, D = 128, causal, Sq = A.len, q_pos_offset =
// A.pos0); cudaErrorNotSupported when the shape cannot run fused (the caller appends and then
// runs the prefill), cudaErrorInvalidValue when the workspace is short
cudaError_t prefill_append_launch(const PrefillLaunch& L, const PrefillAppend& A,
                                  cudaStream_t stream);
// its scratch (0: the shape cannot run fused)
size_t prefill_append_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Sk, int q_pos_offset,
                                      int D, int num_sms);
// scratch the prefill launch needs to cut work units between CTAs (0: it runs whole units)
size_t prefill_workspace_bytes(int B, int Hq, int Sq, int Sk, int q_pos_offset, int causal,
                               int D, int num_sms);
uint32_t prefill_take_error();
// the cut schedule of a prefill call of this shape on num_sms SMs, computed on the host by the
// kernel's own segment code: the plan {cut, CTAs, steps W, units, workspace bytes} and one row
// of kScheduleRowWidth values per segment; returns the segment count, -1 if a CTA's range does
// not fit its segment table.  force_cut lays out the cuts even where the plan keeps whole units.
constexpr int kScheduleRowWidth = 11;
int64_t prefill_debug_schedule(int B, int Hq, int Hkv, int Sq, int Sk, int q_pos_offset,
                               int causal, int D, int num_sms, bool force_cut, int64_t* plan,
                               int64_t* rows, int64_t max_rows);

struct DecodeLaunch {
  CUtensorMap tm_k, tm_v;        // K/V tiles (dense) or nibble tiles (q4_0)
  const void* q;
  void* o;
  const void* k_scale;           // q4_0 only
  const void* v_scale;
  uint32_t* flags;               // [B, Hkv, nsplit] arrival flags (workspace, offset 0)
  float* partial;                // [B, Hq, nsplit, D + 4] f32: m, l, pad, pad, O (workspace)
  uint32_t tag;                  // nonzero, different for every call
  int B, Hq, Hkv, Sk_eff, Sk, Scap, D, nsplit, chunk;
  float scale;
  bool bf16, kq4, vq4;
  // paged cache (block_table != nullptr): pages [num_pages][Hkv][page_size][D]; per-sequence
  // lengths on the device; Sk_eff then bounds every sequence's length
  const int32_t* block_table = nullptr;
  const int32_t* seq_lens = nullptr;
  int page_size = 0, pages_per_seq = 0, num_pages = 0;
};
cudaError_t decode_launch(const DecodeLaunch& L, cudaStream_t stream);
uint32_t decode_take_error();
// decode scratch: the arrival flags, padded to 256 bytes, then the partials
size_t decode_flag_bytes(int B, int Hkv, int nsplit);
// decode work split for a given shape and cache format (shared by the workspace query and the
// launch), and the keys per pipeline stage (the TMA box height)
void decode_plan(int B, int Hkv, int Sk_eff, int num_sms, bool kq4, bool vq4, int* nsplit,
                 int* chunk);
int decode_tile_keys(bool kq4, bool vq4);
// CTAs per kv head of a paged decode launch (shared over the batch on the device)
int decode_paged_ctas(int B, int Hkv, int num_sms, bool kq4, bool vq4);
// the decode kernels' work split computed on the host by the kernels' own plan code: one row of
// kDecodeScheduleRowWidth values {sequence, split, splits of the sequence, first key, end key}
// per CTA of one kv head (uniform batch, seq_lens == nullptr: B x nsplit rows; paged batch:
// seq_lens in host memory, lengths clamped to [1, cap], sequence -1 past the plan); returns
// the row count
constexpr int kDecodeScheduleRowWidth = 5;
int64_t decode_debug_schedule(const int32_t* seq_lens, int B, int Hkv, int Sk, int cap,
                              bool kq4, bool vq4, int num_sms, int32_t* rows, int64_t max_rows);

// q4_0 quantization of up to two tensors in one launch (job 1 may be absent: x1 == nullptr).
// Source rows [B*H][S_src][D]; row (bh, s) goes to destination row bh * Scap + pos0 + s.
struct QuantJob {
  const void* x;
  void* nib;
  void* scale;
};
cudaError_t quantize_launch(QuantJob j0, QuantJob j1, int64_t BH, int S_src, int Scap, int pos0,
                            int D, bool bf16, cudaStream_t stream);

// the explicit (non-flash) path: dequant (q4_0 sides), S = scale Q K^T (f32), softmax -> P,
// O = P V; workspace = S, P and the dequantized K / V
struct ExplicitLaunch {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  void* workspace;
  size_t scale_offset;  // of the q4_0 scale plane within a K or V tensor
  int B, Hq, Hkv, Sq, Sk, D, q_pos_offset, causal;
  float scale;
  bool bf16, kq4, vq4;
};
size_t explicit_workspace(int B, int Hq, int Hkv, int Sq, int Sk, int D, bool kq4, bool vq4);
// returns the CUDA launch status; *map_status is non-zero when a TMA map could not be encoded
cudaError_t explicit_launch(const ExplicitLaunch& L, cudaStream_t stream, int* map_status);
uint32_t explicit_take_error();

cudaError_t debug_timeout_launch(uint64_t limit_ns, cudaStream_t stream);
uint32_t debug_take_error();

}  // namespace fa
