// sss_conv_state_bwd_noalloc: the conv backward with its scratch in a static
// device array, for callers that cannot allocate device memory.
//
// The conv backward needs one row of per-CTA partial sums of dw and dbias per
// (sequence, 64-token group) before the fixed-order reduction.  Here those
// rows live in a file-scope device array of fixed size instead of a workspace
// the caller allocates.  Everything else is the regular conv backward entry
// point, unchanged.
#include <mutex>

#include "common.cuh"

namespace sss {
extern thread_local cudaError_t g_last_cuda_error;
size_t conv_state_bwd_workspace(int64_t Bz, int64_t L, int64_t D, int K);
}  // namespace sss

namespace {

// The scratch.  Every GPU that loads the library holds it until the process
// exits.  In host code this name is only a stand-in for the symbol, never a
// usable device address: the address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_conv_bwd_scratch[SSS_CONV_BWD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices];
void* g_scratch_ctx[kMaxDevices];  // the context the cached address belongs to

// The calling thread's current context (driver entry point, fetched through
// the runtime once); null when the entry point is unavailable.
void* current_context() {
  using Fn = int (*)(void**);
  static Fn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<Fn>(f);
  });
  void* ctx = nullptr;
  if (!fn || fn(&ctx) != 0) return nullptr;
  return ctx;
}

// The scratch's device address on the current device, looked up with that
// device current and cached per (device, context): a device reset or any new
// primary context loads the module again, possibly at another address, so a
// changed context (or an unknown one) means a fresh lookup.
cudaError_t scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  const void* ctx = current_context();
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev] || !ctx || g_scratch_ctx[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_conv_bwd_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
    // the lookup makes the device's primary context current if it was not
    g_scratch_ctx[dev] = current_context();
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" sss_status sss_conv_state_bwd_noalloc(
    const void* x, sss_dtype x_dtype, const float* w, const float* bias, const void* state_in,
    const void* dy, sss_dtype dy_dtype, const void* dstate_out, void* dx, sss_dtype dx_dtype,
    void* dstate_in, float* dw, float* dbias, int64_t Bz, int64_t L, int64_t D, int K,
    int apply_silu, sss_stream_t stream) {
  if (Bz < 0 || L < 0 || D < 0 || K < 1) return SSS_ERR_INVALID_ARG;
  // The partial-sum rows this call needs must fit the static scratch.  Every
  // row the reduction reads is written earlier in the same call, so nothing
  // has to be cleared from the previous call's contents.
  const size_t need = sss::conv_state_bwd_workspace(Bz, L, D, K);
  if (need > size_t(SSS_CONV_BWD_NOALLOC_SCRATCH_BYTES)) return SSS_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if (need > 0) {
    const cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
      sss::g_last_cuda_error = e;
      return SSS_ERR_CUDA;
    }
  }
  return sss_conv_state_bwd(x, x_dtype, w, bias, state_in, dy, dy_dtype, dstate_out, dx,
                            dx_dtype, dstate_in, dw, dbias, Bz, L, D, K, apply_silu, scratch,
                            need > 0 ? size_t(SSS_CONV_BWD_NOALLOC_SCRATCH_BYTES) : 0, stream);
}

extern "C" size_t sss_conv_state_bwd_noalloc_scratch_bytes(void) {
  return size_t(SSS_CONV_BWD_NOALLOC_SCRATCH_BYTES);
}
