// Decode entry point that allocates nothing.
//
// Some callers cannot allocate device memory on the call path: inference runtimes that reserve
// the whole HBM pool at start-up and hand out slices themselves (a cudaMalloc or cudaMallocAsync
// from a library would either fail or fragment their pool), and hosts that forbid any allocation
// once serving has started because an allocation can block on the device.  fa_fwd needs a few MB
// of split-K scratch for decode and takes it from the stream-ordered allocator; fa_fwd_ex needs
// the caller to find that memory.  fa_fwd_decode_noalloc instead uses a fixed scratch area that
// lives in this file as a `static __device__` array: every GPU that loads the library holds it
// (FA_NOALLOC_SCRATCH_BYTES) until the process exits.
#include <cuda.h>

#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr size_t kNoallocScratchBytes = FA_NOALLOC_SCRATCH_BYTES;
static_assert(kNoallocScratchBytes % 256 == 0, "scratch size");

// The decode split partials of every fa_fwd_decode_noalloc call.  In host code this name is only
// a stand-in for the device array, never a device address: the address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) float g_noalloc_scratch[kNoallocScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
// device address of g_noalloc_scratch, per device, and the context it was looked up in: a
// context that is destroyed and created again (cudaDeviceReset) loads the module afresh, so the
// address is looked up again whenever the current context differs from the recorded one
void* g_scratch_addr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn ctx_get_current_fn() {
  static std::once_flag once;
  static CtxGetCurrentFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

}  // namespace
}  // namespace fa

extern "C" fa_status fa_fwd_decode_noalloc(const void* q, const void* k, const void* v, void* o,
                                           int B, int Hq, int Hkv, int Sk, int D,
                                           int q_pos_offset, int causal, float scale,
                                           fa_dtype dtype, fa_kv_format kv_format,
                                           fa_stream_t stream) {
  using namespace fa;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  {
    // one-time set-up per device (and context), with that device current: look up where the
    // array lives.  If no context is bound to this thread yet, cudaSetDevice binds the device's
    // primary context (it initialises it, allocating nothing), so that the context read here is
    // the one the lookup and the launch use.
    CtxGetCurrentFn get_ctx = ctx_get_current_fn();
    if (get_ctx == nullptr) return FA_ERR_CUDA;
    CUcontext ctx = nullptr;
    if (get_ctx(&ctx) != CUDA_SUCCESS) return FA_ERR_CUDA;
    if (ctx == nullptr) {
      if (cudaSetDevice(dev) != cudaSuccess || get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr)
        return FA_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_addr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
        return FA_ERR_CUDA;
      g_scratch_addr[dev] = p;
      g_scratch_ctx[dev] = ctx;
    }
    scratch = g_scratch_addr[dev];
  }
  // the scratch this shape needs (0 means the shape itself is invalid)
  const size_t need = fa_workspace_bytes(B, Hq, Hkv, 1, Sk, D, q_pos_offset, causal);
  if (need == 0) return FA_ERR_INVALID_ARG;
  if (need > kNoallocScratchBytes) return FA_ERR_UNSUPPORTED;
  // Every partial the merging CTA reads is written earlier in the same call, and the arrival
  // flags are tagged per call (and start as zeros here), so the area needs no clearing.
  return fa_fwd_ex(q, k, v, o, B, Hq, Hkv, 1, Sk, D, q_pos_offset, causal, scale, dtype,
                   kv_format, scratch, kNoallocScratchBytes, nullptr, stream);
}
