// C-ABI front end: argument checks, TMA descriptors, kernel dispatch, device status.
#include <math.h>
#include <atomic>
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

__device__ uint32_t g_debug_error;

namespace {

__global__ void debug_wait_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // nothing arrives on this barrier: the bounded wait must give up and record the timeout
    mbar_wait(smem_u32(&bar), 0, &abort_flag, &g_debug_error, limit_ns);
    mbar_arrive(smem_u32(&bar));  // leave the barrier completed
  }
  __syncthreads();
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D tiled map over a contiguous [d2][d1][d0] tensor; box = {box0, box1, 1}.
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t d0,
              uint64_t d1, uint64_t d2, uint32_t box0, uint32_t box1, CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * esize, d0 * d1 * esize};
  const cuuint32_t box[3] = {box0, box1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// map of a K or V tensor [BHkv][Scap][D]: q4_0 nibble tiles (D/2 bytes x `tile` keys, 64-B or
// 32-B swizzle) or dense tiles (64 elements x `tile` keys, 128-B swizzle)
bool kv_map(CUtensorMap* m, const void* base, bool q4, CUtensorMapDataType tdt, int D, int Scap,
            uint64_t BHkv, uint32_t tile, CUtensorMapSwizzle nib_sw) {
  if (q4)
    return make_map(m, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, D / 2, Scap, BHkv, D / 2, tile,
                    nib_sw);
  return make_map(m, base, tdt, 2, D, Scap, BHkv, 64, tile, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

size_t q4_scale_offset(int64_t rows, int D) {
  const size_t nib = static_cast<size_t>(rows) * (D / 2);
  return (nib + 255) / 256 * 256;
}

fa_status check_common(int B, int Hq, int Hkv, int Sq, int Sk, int D, int q_pos_offset,
                       int causal, float scale, int dtype, int kv_format) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Sq < 1 || Sk < 1) return FA_ERR_INVALID_ARG;
  if (B > 65535 || Hkv > 65535 || Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_INVALID_ARG;
  if (kv_format != FA_KV_DENSE && kv_format != FA_KV_Q4_0) return FA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (causal && (q_pos_offset < 0 || static_cast<int64_t>(q_pos_offset) + Sq > Sk))
    return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  if ((Sq + 127) / 128 > 65535) return FA_ERR_UNSUPPORTED;
  if (Sq == 1 && Hq / Hkv > 8) return FA_ERR_UNSUPPORTED;
  // offsets are 64-bit; keep every tensor far below the address-space limits
  if (static_cast<int64_t>(B) * Hq * Sq * D >= (1LL << 40)) return FA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(B) * Hkv * Sk * D >= (1LL << 40)) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// scratch of one call: the decode splits' flags and partials for one pair of cache formats, or
// (Sq >= 2) the prefill cut schedule's flags and partial rows (0 when it runs whole units)
size_t workspace_for(int B, int Hq, int Hkv, int Sq, int Sk, int D, int q_pos_offset,
                     int causal, bool kq4, bool vq4, int* nsplit_out, int* chunk_out) {
  if (Sq != 1)  // the prefill's cut schedule runs at D = 128
    return D != 128 ? 0
                    : prefill_workspace_bytes(B, Hq, Sq, Sk, q_pos_offset, causal, D, num_sms());
  const int sk_eff = causal ? q_pos_offset + 1 : Sk;
  int ns = 1, ck = sk_eff;
  decode_plan(B, Hkv, sk_eff, num_sms(), kq4, vq4, &ns, &ck);
  if (nsplit_out) *nsplit_out = ns;
  if (chunk_out) *chunk_out = ck;
  return decode_flag_bytes(B, Hkv, ns) +
         static_cast<size_t>(B) * Hq * ns * (D + 4) * sizeof(float);
}

// a call tag for the decode arrival flags: nonzero and unlike any nearby call's, and unlike
// small integers or common float bit patterns that a reused buffer may still hold
uint32_t next_call_tag() {
  static std::atomic<uint64_t> calls{0};
  uint64_t z = calls.fetch_add(1, std::memory_order_relaxed) + 0x9e3779b97f4a7c15ull;
  // 64-bit finalizer of SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
  // generators", OOPSLA 2014)
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  z ^= z >> 31;
  const uint32_t t = static_cast<uint32_t>(z >> 32);
  return t ? t : 1u;
}

// enough decode scratch for any pair of cache formats
size_t workspace_any(int B, int Hq, int Hkv, int Sq, int Sk, int D, int q_pos_offset,
                     int causal) {
  size_t m = 0;
  for (int f = 0; f < 3; ++f) {  // both q4_0, both dense, one of each (one plan for either)
    const size_t w = workspace_for(B, Hq, Hkv, Sq, Sk, D, q_pos_offset, causal, f != 1, f == 0,
                                   nullptr, nullptr);
    if (w > m) m = w;
  }
  return m;
}

}  // namespace

bool encode_map_3d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize,
                   uint64_t d0, uint64_t d1, uint64_t d2, uint32_t box0, uint32_t box1,
                   CUtensorMapSwizzle sw) {
  return make_map(m, base, dt, esize, d0, d1, d2, box0, box1, sw);
}

}  // namespace fa

using namespace fa;

extern "C" {

size_t fa_q4_0_scale_offset(int B, int H, int S, int D) {
  if (B < 1 || H < 1 || S < 1 || D < 32 || D % 32) return 0;
  return q4_scale_offset(static_cast<int64_t>(B) * H * S, D);
}

size_t fa_q4_0_bytes(int B, int H, int S, int D) {
  if (B < 1 || H < 1 || S < 1 || D < 32 || D % 32) return 0;
  const int64_t rows = static_cast<int64_t>(B) * H * S;
  return q4_scale_offset(rows, D) + static_cast<size_t>(rows) * (D / 32) * 2;
}

size_t fa_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Sk, int D, int q_pos_offset,
                          int causal) {
  if (check_common(B, Hq, Hkv, Sq, Sk, D, q_pos_offset, causal, 1.f, FA_F16, FA_KV_DENSE) !=
      FA_OK)
    return 0;
  return workspace_any(B, Hq, Hkv, Sq, Sk, D, q_pos_offset, causal);
}

fa_status fa_quantize_q4_0(const void* x, void* out_q4, int B, int H, int S, int D,
                           fa_dtype dtype, fa_stream_t stream) {
  if (!aligned16(x) || !aligned16(out_q4)) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || S < 1 || D < 32 || D % 32) return FA_ERR_INVALID_ARG;
  if (dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_INVALID_ARG;
  const int64_t rows = static_cast<int64_t>(B) * H * S;
  uint8_t* base = static_cast<uint8_t*>(out_q4);
  const QuantJob j0 = {x, base, base + q4_scale_offset(rows, D)};
  const QuantJob none = {nullptr, nullptr, nullptr};
  const cudaError_t e = quantize_launch(j0, none, static_cast<int64_t>(B) * H, S, S, 0, D,
                                        dtype == FA_BF16, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_append_q4_0(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                         int B, int H, int S_new, int kv_capacity, int pos0, int D,
                         fa_dtype dtype, fa_stream_t stream) {
  if (!aligned16(k_new) || !aligned16(k_cache)) return FA_ERR_INVALID_ARG;
  if ((v_new == nullptr) != (v_cache == nullptr)) return FA_ERR_INVALID_ARG;
  if (v_new && (!aligned16(v_new) || !aligned16(v_cache))) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || S_new < 1 || kv_capacity < 1 || D < 32 || D % 32)
    return FA_ERR_INVALID_ARG;
  if (pos0 < 0 || static_cast<int64_t>(pos0) + S_new > kv_capacity) return FA_ERR_INVALID_ARG;
  if (dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_INVALID_ARG;
  const int64_t BH = static_cast<int64_t>(B) * H;
  const size_t soff = q4_scale_offset(BH * kv_capacity, D);
  uint8_t* kc = static_cast<uint8_t*>(k_cache);
  uint8_t* vc = static_cast<uint8_t*>(v_cache);
  const QuantJob jk = {k_new, kc, kc + soff};
  const QuantJob jv = {v_new, vc, vc ? vc + soff : nullptr};
  const cudaError_t e = quantize_launch(jk, jv, BH, S_new, kv_capacity, pos0, D,
                                        dtype == FA_BF16, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_fwd_kv_stats(const void* q, const void* k, const void* v, void* o, int B, int Hq,
                          int Hkv, int Sq, int Sk, int kv_capacity, int D, int q_pos_offset,
                          int causal, float scale, fa_dtype dtype, fa_kv_format k_format,
                          fa_kv_format v_format, void* workspace, size_t workspace_bytes,
                          int32_t* rescale_count, float* p_max, fa_stream_t stream) {
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FA_ERR_INVALID_ARG;
  fa_status st = check_common(B, Hq, Hkv, Sq, Sk, D, q_pos_offset, causal, scale, dtype, k_format);
  if (st != FA_OK) return st;
  if (v_format != FA_KV_DENSE && v_format != FA_KV_Q4_0) return FA_ERR_INVALID_ARG;
  if (kv_capacity < Sk) return FA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(B) * Hkv * kv_capacity * D >= (1LL << 40)) return FA_ERR_UNSUPPORTED;
  const int Scap = kv_capacity;
  const bool bf16 = dtype == FA_BF16;
  const bool kq4 = k_format == FA_KV_Q4_0;
  const bool vq4 = v_format == FA_KV_Q4_0;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const CUtensorMapDataType tdt =
      bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const uint64_t BHkv = static_cast<uint64_t>(B) * Hkv;
  const size_t kv_scale_off = q4_scale_offset(static_cast<int64_t>(BHkv) * Scap, D);
  const CUtensorMapSwizzle nib_sw =
      D == 128 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;

  if (Sq == 1) {
    int nsplit = 1, chunk = 1;
    const size_t need =
        workspace_for(B, Hq, Hkv, Sq, Sk, D, q_pos_offset, causal, kq4, vq4, &nsplit, &chunk);
    const uint32_t tile = static_cast<uint32_t>(decode_tile_keys(kq4, vq4));
    if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)))
      return FA_ERR_INVALID_ARG;
    DecodeLaunch L;
    if (!kv_map(&L.tm_k, k, kq4, tdt, D, Scap, BHkv, tile, nib_sw) ||
        !kv_map(&L.tm_v, v, vq4, tdt, D, Scap, BHkv, tile, nib_sw))
      return FA_ERR_CUDA;
    L.k_scale = kq4 ? static_cast<const uint8_t*>(k) + kv_scale_off : nullptr;
    L.v_scale = vq4 ? static_cast<const uint8_t*>(v) + kv_scale_off : nullptr;
    L.q = q;
    L.o = o;
    L.flags = static_cast<uint32_t*>(workspace);
    L.partial = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                         decode_flag_bytes(B, Hkv, nsplit));
    L.tag = next_call_tag();
    L.B = B;
    L.Hq = Hq;
    L.Hkv = Hkv;
    L.Sk = Sk;
    L.Scap = Scap;
    L.Sk_eff = causal ? q_pos_offset + 1 : Sk;
    L.D = D;
    L.nsplit = nsplit;
    L.chunk = chunk;
    L.scale = scale;
    L.bf16 = bf16;
    L.kq4 = kq4;
    L.vq4 = vq4;
    return decode_launch(L, s) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
  }

  PrefillLaunch L;
  if (!make_map(&L.tm_q, q, tdt, 2, D, Sq, static_cast<uint64_t>(B) * Hq, 64, 128,
                CU_TENSOR_MAP_SWIZZLE_128B) ||
      !kv_map(&L.tm_k, k, kq4, tdt, D, Scap, BHkv, 128, nib_sw) ||
      !kv_map(&L.tm_v, v, vq4, tdt, D, Scap, BHkv, 128, nib_sw))
    return FA_ERR_CUDA;
  L.k_scale = kq4 ? static_cast<const uint8_t*>(k) + kv_scale_off : nullptr;
  L.v_scale = vq4 ? static_cast<const uint8_t*>(v) + kv_scale_off : nullptr;
  L.o = o;
  L.rescale_count = rescale_count;
  L.p_max = p_max;
  L.B = B;
  L.Hq = Hq;
  L.Hkv = Hkv;
  L.Sq = Sq;
  L.Sk = Sk;
  L.Scap = Scap;
  L.D = D;
  L.q_pos_offset = causal ? q_pos_offset : 0;
  L.causal = causal ? 1 : 0;
  L.scale = scale;
  L.bf16 = bf16;
  L.kq4 = kq4;
  L.vq4 = vq4;
  L.workspace = aligned16(workspace) ? workspace : nullptr;
  L.workspace_bytes = L.workspace ? workspace_bytes : 0;
  L.tag = next_call_tag();
  L.num_sms = num_sms();
  return prefill_launch(L, s) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_fwd_kv(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv,
                    int Sq, int Sk, int kv_capacity, int D, int q_pos_offset, int causal,
                    float scale, fa_dtype dtype, fa_kv_format k_format, fa_kv_format v_format,
                    void* workspace, size_t workspace_bytes, int32_t* rescale_count,
                    fa_stream_t stream) {
  return fa_fwd_kv_stats(q, k, v, o, B, Hq, Hkv, Sq, Sk, kv_capacity, D, q_pos_offset, causal,
                         scale, dtype, k_format, v_format, workspace, workspace_bytes,
                         rescale_count, nullptr, stream);
}

// the fused append's argument checks (0: fine), shared by the call and its scratch query
static fa_status append_checks(int B, int Hq, int Hkv, int S_new, int kv_capacity, int D,
                               int pos0) {
  if (pos0 < 0 || S_new < 1 || static_cast<int64_t>(pos0) + S_new > kv_capacity)
    return FA_ERR_INVALID_ARG;
  const fa_status st = check_common(B, Hq, Hkv, S_new, pos0 + S_new, D, pos0, 1, 1.f, FA_F16,
                                    FA_KV_Q4_0);
  if (st != FA_OK) return st;
  if (static_cast<int64_t>(B) * Hkv * kv_capacity * D >= (1LL << 40)) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

size_t fa_prefill_append_workspace_bytes(int B, int Hq, int Hkv, int S_new, int kv_capacity,
                                         int D, int pos0) {
  if (append_checks(B, Hq, Hkv, S_new, kv_capacity, D, pos0) != FA_OK) return 0;
  const size_t fused = prefill_append_workspace_bytes(B, Hq, Hkv, S_new, pos0 + S_new, pos0, D,
                                                      num_sms());
  if (fused > 0) return fused;
  // shapes that run as an append followed by the prefill: the prefill's own scratch
  return workspace_for(B, Hq, Hkv, S_new, pos0 + S_new, D, pos0, 1, true, true, nullptr,
                       nullptr);
}

fa_status fa_prefill_append_q4_0(const void* q, const void* k_new, const void* v_new,
                                 void* k_cache, void* v_cache, void* o, int B, int Hq, int Hkv,
                                 int S_new, int kv_capacity, int D, int pos0, float scale,
                                 fa_dtype dtype, void* workspace, size_t workspace_bytes,
                                 fa_stream_t stream) {
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) ||
      !aligned16(v_cache) || !aligned16(o))
    return FA_ERR_INVALID_ARG;
  fa_status st = append_checks(B, Hq, Hkv, S_new, kv_capacity, D, pos0);
  if (st != FA_OK) return st;
  if (dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return FA_ERR_INVALID_ARG;
  const int Sk = pos0 + S_new;
  const size_t need = fa_prefill_append_workspace_bytes(B, Hq, Hkv, S_new, kv_capacity, D, pos0);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)))
    return FA_ERR_INVALID_ARG;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool bf16 = dtype == FA_BF16;
  const size_t soff = q4_scale_offset(static_cast<int64_t>(B) * Hkv * kv_capacity, D);
  const int nsm = num_sms();
  if (prefill_append_workspace_bytes(B, Hq, Hkv, S_new, Sk, pos0, D, nsm) > 0) {
    const CUtensorMapDataType tdt =
        bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const uint64_t BHkv = static_cast<uint64_t>(B) * Hkv;
    PrefillLaunch L{};
    if (!make_map(&L.tm_q, q, tdt, 2, D, S_new, static_cast<uint64_t>(B) * Hq, 64, 128,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !kv_map(&L.tm_k, k_cache, true, tdt, D, kv_capacity, BHkv, 128,
                CU_TENSOR_MAP_SWIZZLE_64B) ||
        !kv_map(&L.tm_v, v_cache, true, tdt, D, kv_capacity, BHkv, 128,
                CU_TENSOR_MAP_SWIZZLE_64B))
      return FA_ERR_CUDA;
    uint8_t* kc = static_cast<uint8_t*>(k_cache);
    uint8_t* vc = static_cast<uint8_t*>(v_cache);
    L.k_scale = kc + soff;
    L.v_scale = vc + soff;
    L.o = o;
    L.B = B;
    L.Hq = Hq;
    L.Hkv = Hkv;
    L.Sq = S_new;
    L.Sk = Sk;
    L.Scap = kv_capacity;
    L.D = D;
    L.q_pos_offset = pos0;
    L.causal = 1;
    L.scale = scale;
    L.bf16 = bf16;
    L.kq4 = L.vq4 = true;
    L.workspace = workspace;
    L.workspace_bytes = workspace_bytes;
    L.tag = next_call_tag();
    L.num_sms = nsm;
    const PrefillAppend A = {k_new, v_new, kc, vc, kc + soff, vc + soff, pos0, S_new};
    const cudaError_t e = prefill_append_launch(L, A, s);
    if (e == cudaSuccess) return FA_OK;
    if (e != cudaErrorNotSupported) return FA_ERR_CUDA;
    (void)cudaGetLastError();
  }
  // not fusable (D = 64, or a cut that does not fit): append, then the prefill over the cache
  st = fa_append_q4_0(k_new, v_new, k_cache, v_cache, B, Hkv, S_new, kv_capacity, pos0, D, dtype,
                      stream);
  if (st != FA_OK) return st;
  return fa_fwd_kv(q, k_cache, v_cache, o, B, Hq, Hkv, S_new, Sk, kv_capacity, D, pos0, 1, scale,
                   dtype, FA_KV_Q4_0, FA_KV_Q4_0, workspace, workspace_bytes, nullptr, stream);
}

fa_status fa_fwd_ex(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv,
                    int Sq, int Sk, int D, int q_pos_offset, int causal, float scale,
                    fa_dtype dtype, fa_kv_format kv_format, void* workspace,
                    size_t workspace_bytes, int32_t* rescale_count, fa_stream_t stream) {
  return fa_fwd_kv(q, k, v, o, B, Hq, Hkv, Sq, Sk, Sk, D, q_pos_offset, causal, scale, dtype,
                   kv_format, kv_format, workspace, workspace_bytes, rescale_count, stream);
}

// paged decode scratch: flags [Hkv, NT] u32 (256-B padded) then partials [Hkv, NT, G, D + 4]
// f32, NT = CTAs per kv head
static size_t paged_workspace(int B, int Hq, int Hkv, int D, bool kq4, bool vq4, int* nt_out) {
  const int nt = decode_paged_ctas(B, Hkv, num_sms(), kq4, vq4);
  if (nt_out) *nt_out = nt;
  return decode_flag_bytes(1, Hkv, nt) + static_cast<size_t>(Hq) * nt * (D + 4) * sizeof(float);
}

size_t fa_decode_paged_workspace_bytes(int B, int Hq, int Hkv, int D, int page_size,
                                       int pages_per_seq) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || page_size < 1 || pages_per_seq < 1) return 0;
  if (D != 64 && D != 128) return 0;
  size_t m = 0;
  for (int f = 0; f < 3; ++f) {  // both q4_0, both dense, one of each
    const size_t w = paged_workspace(B, Hq, Hkv, D, f != 1, f == 0, nullptr);
    if (w > m) m = w;
  }
  return m;
}

fa_status fa_decode_paged(const void* q, const void* k_pages, const void* v_pages, void* o,
                          const int32_t* block_table, const int32_t* seq_lens, int B, int Hq,
                          int Hkv, int D, int num_pages, int page_size, int pages_per_seq,
                          float scale, fa_dtype dtype, fa_kv_format k_format,
                          fa_kv_format v_format, void* workspace, size_t workspace_bytes,
                          fa_stream_t stream) {
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(o))
    return FA_ERR_INVALID_ARG;
  if (!block_table || !seq_lens || (reinterpret_cast<uintptr_t>(block_table) & 3u) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return FA_ERR_INVALID_ARG;
  if (num_pages < 1 || page_size < 1 || pages_per_seq < 1) return FA_ERR_INVALID_ARG;
  const int64_t max_len = static_cast<int64_t>(page_size) * pages_per_seq;
  if (max_len > (1 << 30)) return FA_ERR_UNSUPPORTED;
  // the shape checks of a decode over max_len keys (the longest sequence the table can hold)
  fa_status st = check_common(B, Hq, Hkv, 1, static_cast<int>(max_len), D,
                              static_cast<int>(max_len) - 1, 1, scale, dtype, k_format);
  if (st != FA_OK) return st;
  if (v_format != FA_KV_DENSE && v_format != FA_KV_Q4_0) return FA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(num_pages) * Hkv * page_size * D >= (1LL << 40))
    return FA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(num_pages) * Hkv >= (1LL << 31)) return FA_ERR_UNSUPPORTED;
  const bool bf16 = dtype == FA_BF16;
  const bool kq4 = k_format == FA_KV_Q4_0;
  const bool vq4 = v_format == FA_KV_Q4_0;
  const uint32_t tile = static_cast<uint32_t>(decode_tile_keys(kq4, vq4));
  if (page_size % static_cast<int>(tile) != 0) return FA_ERR_UNSUPPORTED;
  int nt = 1;
  const size_t need = paged_workspace(B, Hq, Hkv, D, kq4, vq4, &nt);
  if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace))
    return FA_ERR_INVALID_ARG;
  const CUtensorMapDataType tdt =
      bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUtensorMapSwizzle nib_sw =
      D == 128 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
  const uint64_t rows = static_cast<uint64_t>(num_pages) * Hkv;  // (page, kv head) blocks
  const size_t scale_off = q4_scale_offset(static_cast<int64_t>(rows) * page_size, D);
  DecodeLaunch L;
  if (!kv_map(&L.tm_k, k_pages, kq4, tdt, D, page_size, rows, tile, nib_sw) ||
      !kv_map(&L.tm_v, v_pages, vq4, tdt, D, page_size, rows, tile, nib_sw))
    return FA_ERR_CUDA;
  L.k_scale = kq4 ? static_cast<const uint8_t*>(k_pages) + scale_off : nullptr;
  L.v_scale = vq4 ? static_cast<const uint8_t*>(v_pages) + scale_off : nullptr;
  L.q = q;
  L.o = o;
  L.flags = static_cast<uint32_t*>(workspace);
  L.partial = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                       decode_flag_bytes(1, Hkv, nt));
  L.tag = next_call_tag();
  L.B = B;
  L.Hq = Hq;
  L.Hkv = Hkv;
  L.Sk = static_cast<int>(max_len);
  L.Scap = page_size;
  L.Sk_eff = static_cast<int>(max_len);
  L.D = D;
  L.nsplit = nt;
  L.chunk = 0;
  L.scale = scale;
  L.bf16 = bf16;
  L.kq4 = kq4;
  L.vq4 = vq4;
  L.block_table = block_table;
  L.seq_lens = seq_lens;
  L.page_size = page_size;
  L.pages_per_seq = pages_per_seq;
  L.num_pages = num_pages;
  return decode_launch(L, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK
                                                                                 : FA_ERR_CUDA;
}

size_t fa_explicit_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Sk, int D,
                                   fa_kv_format k_format, fa_kv_format v_format) {
  if (check_common(B, Hq, Hkv, Sq, Sk, D, 0, 0, 1.f, FA_F16, k_format) != FA_OK) return 0;
  if (v_format != FA_KV_DENSE && v_format != FA_KV_Q4_0) return 0;
  return explicit_workspace(B, Hq, Hkv, Sq, Sk, D, k_format == FA_KV_Q4_0,
                            v_format == FA_KV_Q4_0);
}

fa_status fa_fwd_explicit(const void* q, const void* k, const void* v, void* o, int B, int Hq,
                          int Hkv, int Sq, int Sk, int D, int q_pos_offset, int causal,
                          float scale, fa_dtype dtype, fa_kv_format k_format,
                          fa_kv_format v_format, void* workspace, size_t workspace_bytes,
                          fa_stream_t stream) {
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FA_ERR_INVALID_ARG;
  const fa_status st =
      check_common(B, Hq, Hkv, Sq, Sk, D, q_pos_offset, causal, scale, dtype, k_format);
  if (st != FA_OK) return st;
  if (v_format != FA_KV_DENSE && v_format != FA_KV_Q4_0) return FA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(B) * Hq * Sq > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(Hq / Hkv) * Sq > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  const bool kq4 = k_format == FA_KV_Q4_0, vq4 = v_format == FA_KV_Q4_0;
  const size_t need = explicit_workspace(B, Hq, Hkv, Sq, Sk, D, kq4, vq4);
  if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace))
    return FA_ERR_INVALID_ARG;
  ExplicitLaunch L;
  L.q = q;
  L.k = k;
  L.v = v;
  L.o = o;
  L.workspace = workspace;
  L.scale_offset = q4_scale_offset(static_cast<int64_t>(B) * Hkv * Sk, D);
  L.B = B;
  L.Hq = Hq;
  L.Hkv = Hkv;
  L.Sq = Sq;
  L.Sk = Sk;
  L.D = D;
  L.q_pos_offset = causal ? q_pos_offset : 0;
  L.causal = causal ? 1 : 0;
  L.scale = scale;
  L.bf16 = dtype == FA_BF16;
  L.kq4 = kq4;
  L.vq4 = vq4;
  int map_status = 0;
  if (explicit_launch(L, reinterpret_cast<cudaStream_t>(stream), &map_status) != cudaSuccess)
    return FA_ERR_CUDA;
  return map_status ? FA_ERR_CUDA : FA_OK;
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv,
                 int Sq, int Sk, int D, int q_pos_offset, int causal, float scale,
                 fa_dtype dtype, fa_kv_format kv_format, fa_stream_t stream) {
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FA_ERR_INVALID_ARG;
  const fa_status st =
      check_common(B, Hq, Hkv, Sq, Sk, D, q_pos_offset, causal, scale, dtype, kv_format);
  if (st != FA_OK) return st;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool q4 = kv_format == FA_KV_Q4_0;
  const size_t need =
      workspace_for(B, Hq, Hkv, Sq, Sk, D, q_pos_offset, causal, q4, q4, nullptr, nullptr);
  void* ws = nullptr;
  if (need > 0 && cudaMallocAsync(&ws, need, s) != cudaSuccess) {
    // decode cannot run without its split scratch; prefill runs one unit per CTA instead (the
    // failed allocation's error is cleared so that the launch check does not report it)
    ws = nullptr;
    if (Sq == 1) return FA_ERR_CUDA;
    (void)cudaGetLastError();
  }
  const fa_status r = fa_fwd_ex(q, k, v, o, B, Hq, Hkv, Sq, Sk, D, q_pos_offset, causal, scale,
                                dtype, kv_format, ws, need, nullptr, stream);
  if (ws && cudaFreeAsync(ws, s) != cudaSuccess && r == FA_OK) return FA_ERR_CUDA;
  return r;
}

fa_status fa_get_status(fa_stream_t stream) {
  const cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return FA_ERR_CUDA;
  const uint32_t a = prefill_take_error();
  const uint32_t b = decode_take_error();
  const uint32_t x = explicit_take_error();
  uint32_t c = 0;
  if (cudaMemcpyFromSymbol(&c, g_debug_error, sizeof(c)) != cudaSuccess) return FA_ERR_CUDA;
  const uint32_t z = 0;
  if (c != 0 && cudaMemcpyToSymbol(g_debug_error, &z, sizeof(z)) != cudaSuccess)
    return FA_ERR_CUDA;
  if (a == 0xffffffffu || b == 0xffffffffu || x == 0xffffffffu) return FA_ERR_CUDA;
  if (b == kErrBadIndex) return FA_ERR_INVALID_ARG;
  if (a == kErrSchedule) return FA_ERR_UNSUPPORTED;
  if (a || b || c || x) return FA_ERR_TIMEOUT;
  return FA_OK;
}

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
  }
  return "FA_ERR_UNKNOWN";
}

fa_status fa_debug_wait_timeout(int64_t limit_ns, fa_stream_t stream) {
  if (limit_ns < 1000) limit_ns = 1000;
  if (limit_ns > 1000000000) limit_ns = 1000000000;
  debug_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<uint64_t>(limit_ns));
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int64_t fa_prefill_schedule(int B, int Hq, int Hkv, int Sq, int Sk, int D, int q_pos_offset,
                            int causal, int num_sms, int force_cut, int64_t* plan, int64_t* rows,
                            int64_t max_rows) {
  if (Sq < 2 || num_sms < 1 || max_rows < 0 || (max_rows > 0 && rows == nullptr) ||
      check_common(B, Hq, Hkv, Sq, Sk, D, q_pos_offset, causal, 1.f, FA_F16, FA_KV_DENSE) !=
          FA_OK)
    return -2;
  return prefill_debug_schedule(B, Hq, Hkv, Sq, Sk, q_pos_offset, causal, D, num_sms,
                                force_cut != 0, plan, rows, max_rows);
}

int64_t fa_decode_schedule(const int32_t* seq_lens, int B, int Hkv, int Sk, int page_size,
                           int pages_per_seq, fa_kv_format k_format, fa_kv_format v_format,
                           int num_sms, int32_t* rows, int64_t max_rows) {
  if (B < 1 || Hkv < 1 || num_sms < 1 || max_rows < 0 || (max_rows > 0 && rows == nullptr))
    return -2;
  if ((k_format != FA_KV_DENSE && k_format != FA_KV_Q4_0) ||
      (v_format != FA_KV_DENSE && v_format != FA_KV_Q4_0))
    return -2;
  const bool kq4 = k_format == FA_KV_Q4_0, vq4 = v_format == FA_KV_Q4_0;
  int cap = 0;
  if (seq_lens == nullptr) {
    if (Sk < 1) return -2;
  } else {
    if (page_size < 1 || pages_per_seq < 1 || page_size % decode_tile_keys(kq4, vq4) != 0)
      return -2;
    const int64_t c = static_cast<int64_t>(page_size) * pages_per_seq;
    if (c > (1 << 30)) return -2;
    cap = static_cast<int>(c);
  }
  return decode_debug_schedule(seq_lens, B, Hkv, Sk, cap, kq4, vq4, num_sms, rows, max_rows);
}

int fa_version(void) { return 107; }

}  // extern "C"
