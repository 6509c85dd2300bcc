// fa_bwd_noalloc: the backward pass for callers that cannot allocate device
// memory.
//
// fa_bwd needs a caller-provided workspace (the fp32 dQ accumulator and the
// per-row D and LSE*log2(e) vectors). Some callers have no way to provide one:
// host code running inside a framework or plugin callback that owns every
// device allocation and forbids cudaMalloc there, or latency-critical code that
// must not call cudaMalloc/cudaFree because those calls can synchronize the
// whole device. This entry point takes the same inputs and outputs as fa_bwd
// but draws its scratch from a fixed array in the library's own device memory,
// so it performs no allocation of any kind.
//
// The array lives for as long as the library is loaded, on every GPU that
// loads it. All calls share it and it keeps the previous call's contents; the
// backward's first kernel rewrites every part of it that the later kernels
// read (the dQ accumulator is zeroed, D and LSE rows are written), so stale
// contents never leak into a result. Two calls whose kernels overlap on the
// GPU (different streams without ordering, or different host threads) race on
// the array and give wrong results; the caller must order them.
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr size_t kScratchBytes = FA_NOALLOC_SCRATCH_BYTES;

// Device scratch. In host code `g_scratch` is only a host-side stand-in for the
// symbol, never a device address: its device address comes from
// cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device, looked up on the first
// call made with that device current. Returns nullptr on failure.
void* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace fa

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* out,
                              const void* dout, const float* lse, void* dq, void* dk, void* dv,
                              int B, int Hq, int Hkv, int S, int d, int causal, float scale,
                              int dtype, fa_stream_t stream) {
  // the argument errors of fa_bwd first, then the scratch limit; neither
  // failure looks up or touches the scratch array
  const int rc = fa::check_bwd_args(q, k, v, out, dout, lse, dq, dk, dv, B, Hq, Hkv, S, S, d,
                                    causal, scale, dtype);
  if (rc != FA_OK) return rc;
  if (fa_bwd_workspace_bytes(B, Hq, Hkv, S, d) > fa::kScratchBytes) return FA_ERR_NOALLOC_LIMIT;
  void* scratch = fa::scratch_on_current_device();
  if (!scratch) return FA_ERR_CUDA;
  return fa_bwd(q, k, v, out, dout, lse, dq, dk, dv, B, Hq, Hkv, S, d, causal, scale, dtype,
                scratch, fa::kScratchBytes, stream);
}
