// C ABI of libsss: argument validation, path selection and launch.  All
// arithmetic runs in the kernels of the other files.
#include <mutex>

#include "common.cuh"

namespace sss {

__device__ int g_status_word;

cudaError_t mamba2_scan_launch(const float* u, const void* z, const void* dt_raw, sss_dtype at,
                               const float* dt_bias, const float* A, const float* D_skip,
                               const float* h0, float* hT, void* y, sss_dtype yt, int64_t Bz,
                               int64_t L, int H, int P, int N, int G, cudaStream_t st);
bool ssm_scan_simt_supports(int P, int N);
cudaError_t conv_state_fwd_launch(const void* x, sss_dtype xt, const float* w,
                                  const float* bias, const void* s_in, void* s_out,
                                  void* u, sss_dtype ut, int64_t Bz, int64_t L,
                                  int64_t D, int K, int silu_on, cudaStream_t st);
bool ssm_scan_simt_supports(int P, int N);
cudaError_t ssm_scan_simt_launch(const void* x, sss_dtype xt, const void* dt, const float* A,
                                 const void* B, const void* C, sss_dtype at,
                                 const float* h0, float* hT, void* y, sss_dtype yt,
                                 int64_t Bz, int64_t L, int H, int P, int N, int G,
                                 const int32_t* seq_idx, cudaStream_t st);
bool ssm_scan_tc_supports(sss_dtype xt, sss_dtype at, sss_dtype yt, int64_t L, int H, int P,
                          int N, int G);
cudaError_t ssm_scan_tc_launch(const void* x, sss_dtype xt, const void* dt, const float* A,
                               const void* B, const void* C, const float* h0, float* hT,
                               void* y, sss_dtype yt, int64_t Bz, int64_t L, int H, int P,
                               int N, int G, int* status, const int32_t* seq_idx,
                               cudaStream_t st);
bool mixer_fwd_tc_supports(sss_dtype xt, sss_dtype at, int K, int64_t L, int H, int P, int N,
                           int G);
cudaError_t mixer_fwd_tc_launch(const void* x, const float* w, const float* bias,
                                const void* s_in, void* s_out, const void* dt, const float* A,
                                const void* B, const void* C, const float* h0, float* hT,
                                void* y, sss_dtype yt, int64_t Bz, int64_t L, int H, int G, int K,
                                int* status, const int32_t* seq_idx, cudaStream_t st);
bool ssm_scan_pair_supports(sss_dtype at, int64_t L, int H, int P, int N, int G);
cudaError_t ssm_scan_pair_launch(const void* x, sss_dtype xt, const void* dt, const float* A,
                                 const void* B, const void* C, const float* h0, float* hT,
                                 void* y, sss_dtype yt, int64_t Bz, int64_t L, int H, int G,
                                 int* status, const int32_t* seq_idx, cudaStream_t st,
                                 bool dependent = false);
cudaError_t mixer_fwd_pair_launch(const void* x, const float* w, const float* bias,
                                  const void* s_in, void* s_out, const void* dt, const float* A,
                                  const void* B, const void* C, const float* h0, float* hT,
                                  void* y, sss_dtype yt, int64_t Bz, int64_t L, int H, int G,
                                  int K, int* status, const int32_t* seq_idx, cudaStream_t st,
                                  bool dependent = false);
cudaError_t conv_state_bwd_launch(const void* x, sss_dtype xt, const float* w, const float* bias,
                                  const void* s_in, const void* dy, sss_dtype dyt, const void* q,
                                  void* dx, sss_dtype dxt, void* dS, float* dw, float* dbias,
                                  int64_t Bz, int64_t L, int64_t D, int K, int silu_on,
                                  void* ws, cudaStream_t st);
size_t conv_state_bwd_workspace(int64_t Bz, int64_t L, int64_t D, int K);
cudaError_t conv_packed_launch(const void* x, sss_dtype xt, const float* w, const float* bias,
                               const void* s_in, void* s_out, const int32_t* seq_idx, void* u,
                               sss_dtype ut, int64_t Bz, int64_t L, int64_t D, int K, int silu_on,
                               cudaStream_t st);
bool conv_state_bwd_supports(int K);
size_t ssm_scan_bwd_workspace(int64_t Bz, int64_t L, int H, int P, int N);
cudaError_t state_reset_launch(const float* u, float p, float* h, int64_t Bz, int64_t h_elems,
                               void* conv, sss_dtype conv_t, int64_t conv_elems, cudaStream_t st);
cudaError_t span_prepare_launch(const void* x, const void* s_in, void* s_out, void* s_span,
                                const void* dt, const float* A, float* part, int64_t Bz,
                                int64_t L, int64_t D, int H, int K, int ns, cudaStream_t st);
cudaError_t span_combine_launch(const float* part, const float* hloc, const float* h0,
                                float* h0_span, float* hT, int64_t Bz, int64_t L, int H,
                                int64_t PN, int ns, cudaStream_t st);
size_t span_part_floats(int64_t Bz, int64_t L, int H, int ns);
cudaError_t ssm_scan_pair_state_launch(const void* x, sss_dtype xt, const void* dt,
                                       const float* A, const void* B, float* hT, int64_t Bz,
                                       int64_t L, int H, int G, int* status, cudaStream_t st);
cudaError_t mixer_fwd_pair_state_launch(const void* x, const float* w, const float* bias,
                                        const void* s_in, const void* dt, const float* A,
                                        const void* B, float* hT, int64_t Bz, int64_t L, int H,
                                        int G, int K, int* status, cudaStream_t st);
bool span_sizes_ok(int64_t Bz, int64_t L, int64_t D, int H, int P, int N, int K, int ns);

cudaError_t fitted_noise_update_launch(const float* hT, int64_t Bz, int H, int64_t PN, float beta,
                                       int has_history, float* mu, float* var, cudaStream_t st);
cudaError_t fitted_noise_sample_launch(const float* mu, const float* var, const float* eps,
                                       float* h0, int64_t Bz, int H, int64_t PN, cudaStream_t st);
int state_trace_max_stride();
cudaError_t prefill_to_pool_launch(const void* x, sss_dtype dt, const void* state_in, int K,
                                   const float* hT, void* conv_pool, int64_t pool, int S_len,
                                   float* ssm_pool, const int32_t* seqlens, const int32_t* idx,
                                   int64_t Bz, int64_t L, int64_t D, int64_t ssm_row_elems,
                                   int* status, cudaStream_t st);
cudaError_t state_std_trace_launch(const void* x, sss_dtype x_t, const void* dt, const float* A,
                                   const void* B, sss_dtype act_t, const float* h0, float* out,
                                   int64_t Bz, int64_t L, int H, int P, int N, int G, int stride,
                                   cudaStream_t st);
bool ssm_scan_bwd_supports(int P, int N);
cudaError_t ssm_scan_bwd_launch(const void* x, sss_dtype x_t, const void* dt, const float* A,
                                const void* B, const void* C, sss_dtype act_t, const float* h0,
                                const float* dy, const float* dhT, float* dx, float* ddt,
                                float* dA, float* dB, float* dC, float* dh0, int64_t Bz, int64_t L,
                                int H, int P, int N, int G, void* ws, cudaStream_t st);
bool mixer_update_supports(int P, int N, int K, int L_new);
int mixer_update_path(sss_dtype at, int S_len, int L_new, int P, int N, int K);
cudaError_t mixer_update_launch(const void* x, sss_dtype at, const float* w, const float* bias,
                                void* cp, int64_t pool, int S_len, const int32_t* sl,
                                const int32_t* ix, const void* dt, const float* A,
                                const void* B, const void* C, float* sp, void* y, int64_t Bz,
                                int L_new, int H, int P, int N, int G, int K, int* status,
                                cudaStream_t st);

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_sms[kMaxDevices];
int* g_status_ptr[kMaxDevices];

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}
}  // namespace

int sm_count() {
  const int dev = current_device();
  if (dev < 0) return 1;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sms[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    g_sms[dev] = v > 0 ? v : 1;
  }
  return g_sms[dev];
}

int* status_word() {
  const int dev = current_device();
  if (dev < 0) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  return g_status_ptr[dev];
}

static bool aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

thread_local cudaError_t g_last_cuda_error = cudaSuccess;

static sss_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return SSS_OK;
  g_last_cuda_error = e;
  if (e == cudaErrorNotSupported) {
    cudaGetLastError();
    return SSS_ERR_UNSUPPORTED;
  }
  return SSS_ERR_CUDA;
}

}  // namespace sss

using namespace sss;

extern "C" {

int sss_version(void) { return 100; }

const char* sss_last_cuda_error(void) { return cudaGetErrorString(sss::g_last_cuda_error); }

const char* sss_status_string(int s) {
  switch (s) {
    case SSS_OK: return "ok";
    case SSS_ERR_INVALID_ARG: return "invalid argument";
    case SSS_ERR_UNSUPPORTED: return "unsupported configuration";
    case SSS_ERR_INDEX: return "pool index or length out of range (device)";
    case SSS_ERR_TIMEOUT: return "bounded device wait ran out";
    case SSS_ERR_CUDA: return "CUDA runtime error";
    default: return "several errors (bitwise OR of sss_status values)";
  }
}

sss_status sss_conv_state_fwd(const void* x, sss_dtype x_dtype, const float* w,
                              const float* bias, const void* state_in, void* state_out,
                              void* u, sss_dtype u_dtype, int64_t Bz, int64_t L, int64_t D,
                              int K, int apply_silu, sss_stream_t stream) {
  if (!dtype_ok(x_dtype) || !dtype_ok(u_dtype)) return SSS_ERR_INVALID_ARG;
  if (Bz < 0 || L < 0 || D < 0 || K < 1) return SSS_ERR_INVALID_ARG;
  if (K > 8) return SSS_ERR_UNSUPPORTED;
  if (Bz == 0 || D == 0) return SSS_OK;
  const size_t xs = dtype_size(x_dtype), us = dtype_size(u_dtype);
  if (!w || !aligned(w, 4) || (bias && !aligned(bias, 4))) return SSS_ERR_INVALID_ARG;
  if (L > 0 && (!x || !u || !aligned(x, xs) || !aligned(u, us))) return SSS_ERR_INVALID_ARG;
  if ((state_in && !aligned(state_in, xs)) || (state_out && !aligned(state_out, xs)))
    return SSS_ERR_INVALID_ARG;
  if (L == 0 && !state_out) return SSS_OK;
  return from_cuda(conv_state_fwd_launch(x, x_dtype, w, bias, state_in, state_out, u, u_dtype,
                                         Bz, L, D, K, apply_silu != 0,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

sss_status sss_conv_state_fwd_packed(const void* x, sss_dtype x_dtype, const float* w,
                                     const float* bias, const void* state_in, void* state_out,
                                     const int32_t* seq_idx, void* u, sss_dtype u_dtype,
                                     int64_t Bz, int64_t L, int64_t D, int K, int apply_silu,
                                     sss_stream_t stream) {
  if (!dtype_ok(x_dtype) || !dtype_ok(u_dtype)) return SSS_ERR_INVALID_ARG;
  if (Bz < 0 || L < 0 || D < 0 || K < 1) return SSS_ERR_INVALID_ARG;
  if (K > 8) return SSS_ERR_UNSUPPORTED;
  if (Bz == 0 || D == 0) return SSS_OK;
  if (Bz > 65535 || (L + 15) / 16 > 65535) return SSS_ERR_UNSUPPORTED;
  const size_t xs = dtype_size(x_dtype), us = dtype_size(u_dtype);
  if (!w || !aligned(w, 4) || (bias && !aligned(bias, 4))) return SSS_ERR_INVALID_ARG;
  if (L > 0 && (!x || !u || !seq_idx || !aligned(x, xs) || !aligned(u, us) ||
                !aligned(seq_idx, 4)))
    return SSS_ERR_INVALID_ARG;
  if ((state_in && !aligned(state_in, xs)) || (state_out && !aligned(state_out, xs)))
    return SSS_ERR_INVALID_ARG;
  if (L == 0 && !state_out) return SSS_OK;
  return from_cuda(conv_packed_launch(x, x_dtype, w, bias, state_in, state_out, seq_idx, u,
                                      u_dtype, Bz, L, D, K, apply_silu != 0,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

size_t sss_ssm_scan_workspace_size(int64_t Bz, int64_t L, int H, int P, int N, int G,
                                   sss_dtype x_dtype, sss_dtype act_dtype) {
  (void)Bz; (void)L; (void)H; (void)P; (void)N; (void)G; (void)x_dtype; (void)act_dtype;
  return 0;
}

int sss_ssm_scan_path(int64_t Bz, int64_t L, int H, int P, int N, int G, sss_dtype x_dtype,
                      sss_dtype act_dtype, sss_dtype y_dtype) {
  (void)Bz;
  if (ssm_scan_tc_supports(x_dtype, act_dtype, y_dtype, L, H, P, N, G))
    return ssm_scan_pair_supports(act_dtype, L, H, P, N, G) ? 2 : 1;
  if (ssm_scan_simt_supports(P, N)) return 0;
  return -1;
}

size_t sss_conv_state_bwd_workspace_size(int64_t Bz, int64_t L, int64_t D, int K) {
  return sss::conv_state_bwd_workspace(Bz, L, D, K);
}

static bool ranges_overlap(const void* a, const void* b, size_t bytes) {
  if (!a || !b || bytes == 0) return false;
  const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
  return pa < pb + bytes && pb < pa + bytes;
}

sss_status sss_conv_state_bwd(const void* x, sss_dtype x_dtype, const float* w,
                              const float* bias, const void* state_in, const void* dy,
                              sss_dtype dy_dtype, const void* dstate_out, void* dx,
                              sss_dtype dx_dtype, void* dstate_in, float* dw, float* dbias,
                              int64_t Bz, int64_t L, int64_t D, int K, int apply_silu,
                              void* workspace, size_t workspace_bytes, sss_stream_t stream) {
  if (!dtype_ok(x_dtype) || !dtype_ok(dy_dtype) || !dtype_ok(dx_dtype))
    return SSS_ERR_INVALID_ARG;
  if (Bz < 0 || L < 0 || D < 0 || K < 1) return SSS_ERR_INVALID_ARG;
  if (!sss::conv_state_bwd_supports(K)) return SSS_ERR_UNSUPPORTED;
  if (Bz == 0 || D == 0) return SSS_OK;
  const size_t xs = dtype_size(x_dtype), ys = dtype_size(dy_dtype), os = dtype_size(dx_dtype);
  if (!w || !dw || !aligned(w, 4) || !aligned(dw, 4) || (bias && !aligned(bias, 4)) ||
      (dbias && !aligned(dbias, 4)))
    return SSS_ERR_INVALID_ARG;
  if (K > 1 && (!dstate_in || !aligned(dstate_in, os))) return SSS_ERR_INVALID_ARG;
  if ((state_in && !aligned(state_in, xs)) || (dstate_out && !aligned(dstate_out, ys)))
    return SSS_ERR_INVALID_ARG;
  if (L > 0 && (!x || !dy || !dx || !aligned(x, xs) || !aligned(dy, ys) || !aligned(dx, os)))
    return SSS_ERR_INVALID_ARG;
  const size_t state_bytes = size_t(Bz) * size_t(D) * size_t(K - 1);
  if (ranges_overlap(dstate_in, dstate_out, state_bytes * (os > ys ? os : ys)))
    return SSS_ERR_INVALID_ARG;
  const size_t need = sss::conv_state_bwd_workspace(Bz, L, D, K);
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 16)))
    return SSS_ERR_INVALID_ARG;
  return from_cuda(sss::conv_state_bwd_launch(
      x, x_dtype, w, bias, state_in, dy, dy_dtype, dstate_out, dx, dx_dtype, dstate_in, dw,
      dbias, Bz, L, D, K, apply_silu != 0, workspace, reinterpret_cast<cudaStream_t>(stream)));
}

static sss_status scan_fwd_impl(const void* x, sss_dtype x_dtype, const void* dt, const float* A,
                                const void* B, const void* C, sss_dtype act_dtype,
                                const float* h0_in, float* hT_out, void* y, sss_dtype y_dtype,
                                int64_t Bz, int64_t L, int H, int P, int N, int G,
                                const int32_t* seq_idx, sss_stream_t stream) {
  if (!dtype_ok(x_dtype) || !dtype_ok(act_dtype) || !dtype_ok(y_dtype)) return SSS_ERR_INVALID_ARG;
  if (Bz < 0 || L < 0 || H < 1 || P < 1 || N < 1 || G < 1 || H % G) return SSS_ERR_INVALID_ARG;
  if (Bz == 0) return SSS_OK;
  const size_t xs = dtype_size(x_dtype), as = dtype_size(act_dtype), ys = dtype_size(y_dtype);
  if (!A || !aligned(A, 4)) return SSS_ERR_INVALID_ARG;
  if (L > 0 && (!x || !dt || !B || !C || !y)) return SSS_ERR_INVALID_ARG;
  if (L > 0 && (!aligned(x, xs) || !aligned(dt, as) || !aligned(B, as) || !aligned(C, as) ||
                !aligned(y, ys)))
    return SSS_ERR_INVALID_ARG;
  if ((h0_in && !aligned(h0_in, 4)) || (hT_out && !aligned(hT_out, 4))) return SSS_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (L > 0 && ssm_scan_tc_supports(x_dtype, act_dtype, y_dtype, L, H, P, N, G) &&
      aligned(x, 16) && aligned(B, 16) && aligned(C, 16) && aligned(y, 16) &&
      (!h0_in || aligned(h0_in, 16)) && (!hT_out || aligned(hT_out, 16))) {
    if (ssm_scan_pair_supports(act_dtype, L, H, P, N, G))
      return from_cuda(ssm_scan_pair_launch(x, x_dtype, dt, A, B, C, h0_in, hT_out, y, y_dtype,
                                            Bz, L, H, G, status_word(), seq_idx, st));
    return from_cuda(ssm_scan_tc_launch(x, x_dtype, dt, A, B, C, h0_in, hT_out, y, y_dtype, Bz,
                                        L, H, P, N, G, status_word(), seq_idx, st));
  }
  if (!ssm_scan_simt_supports(P, N)) return SSS_ERR_UNSUPPORTED;
  return from_cuda(ssm_scan_simt_launch(x, x_dtype, dt, A, B, C, act_dtype, h0_in, hT_out, y,
                                        y_dtype, Bz, L, H, P, N, G, seq_idx, st));
}

sss_status sss_ssm_scan_fwd(const void* x, sss_dtype x_dtype, const void* dt, const float* A,
                            const void* B, const void* C, sss_dtype act_dtype,
                            const float* h0_in, float* hT_out, void* y, sss_dtype y_dtype,
                            int64_t Bz, int64_t L, int H, int P, int N, int G, void* workspace,
                            size_t workspace_bytes, sss_stream_t stream) {
  (void)workspace; (void)workspace_bytes;
  return scan_fwd_impl(x, x_dtype, dt, A, B, C, act_dtype, h0_in, hT_out, y, y_dtype, Bz, L, H,
                       P, N, G, nullptr, stream);
}

sss_status sss_ssm_scan_fwd_packed(const void* x, sss_dtype x_dtype, const void* dt,
                                   const float* A, const void* B, const void* C,
                                   sss_dtype act_dtype, const float* h0_in, float* hT_out,
                                   const int32_t* seq_idx, void* y, sss_dtype y_dtype, int64_t Bz,
                                   int64_t L, int H, int P, int N, int G, sss_stream_t stream) {
  if (Bz > 0 && L > 0 && (!seq_idx || !aligned(seq_idx, 4))) return SSS_ERR_INVALID_ARG;
  return scan_fwd_impl(x, x_dtype, dt, A, B, C, act_dtype, h0_in, hT_out, y, y_dtype, Bz, L, H,
                       P, N, G, seq_idx, stream);
}

size_t sss_ssm_scan_bwd_workspace_size(int64_t Bz, int64_t L, int H, int P, int N, int G) {
  (void)G;
  if (Bz < 0 || L < 0 || H < 1 || P < 1 || N < 1) return 0;
  return sss::ssm_scan_bwd_workspace(Bz, L, H, P, N);
}

sss_status sss_ssm_scan_bwd(const void* x, sss_dtype x_dtype, const void* dt, const float* A,
                            const void* B, const void* C, sss_dtype act_dtype, const float* h0_in,
                            const float* dy, const float* dhT, float* dx, float* ddt, float* dA,
                            float* dB, float* dC, float* dh0, int64_t Bz, int64_t L, int H, int P,
                            int N, int G, void* workspace, size_t workspace_bytes,
                            sss_stream_t stream) {
  if (!dtype_ok(x_dtype) || !dtype_ok(act_dtype)) return SSS_ERR_INVALID_ARG;
  if (Bz < 0 || L < 0 || H < 1 || P < 1 || N < 1 || G < 1 || H % G) return SSS_ERR_INVALID_ARG;
  if (!sss::ssm_scan_bwd_supports(P, N)) return SSS_ERR_UNSUPPORTED;
  const size_t xs = dtype_size(x_dtype), as = dtype_size(act_dtype);
  if (!A || !dA || !aligned(A, 4) || !aligned(dA, 4)) return SSS_ERR_INVALID_ARG;
  if (Bz > 0 && L > 0 &&
      (!x || !dt || !B || !C || !dy || !dx || !ddt || !dB || !dC || !aligned(x, xs) ||
       !aligned(dt, as) || !aligned(B, as) || !aligned(C, as) || !aligned(dy, 4) ||
       !aligned(dx, 4) || !aligned(ddt, 4) || !aligned(dB, 4) || !aligned(dC, 4)))
    return SSS_ERR_INVALID_ARG;
  if ((h0_in && !aligned(h0_in, 4)) || (dhT && !aligned(dhT, 4)) || (dh0 && !aligned(dh0, 4)))
    return SSS_ERR_INVALID_ARG;
  const size_t state_bytes = size_t(Bz) * size_t(H) * size_t(P) * size_t(N) * 4;
  if (dh0 != dhT && ranges_overlap(dh0, dhT, state_bytes)) return SSS_ERR_INVALID_ARG;
  const size_t need = sss::ssm_scan_bwd_workspace(Bz, L, H, P, N);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return SSS_ERR_INVALID_ARG;
  return from_cuda(sss::ssm_scan_bwd_launch(x, x_dtype, dt, A, B, C, act_dtype, h0_in, dy, dhT, dx,
                                            ddt, dA, dB, dC, dh0, Bz, L, H, P, N, G, workspace,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

sss_status sss_prefill_to_pool(const void* x, sss_dtype x_dtype, const void* conv_state_in, int K,
                               const float* hT, void* conv_pool, int64_t pool, int S_len,
                               float* ssm_pool, const int32_t* cache_seqlens,
                               const int32_t* conv_state_indices, int64_t Bz, int64_t L,
                               int64_t D, int H, int P, int N, sss_stream_t stream) {
  if (!dtype_ok(x_dtype) || Bz < 0 || L < 0 || D < 1 || K < 1 || S_len < 1 || S_len < K - 1 ||
      pool < 0 || H < 1 || P < 1 || N < 1 || int64_t(H) * P != D)
    return SSS_ERR_INVALID_ARG;
  if (Bz == 0) return SSS_OK;
  const size_t xs = dtype_size(x_dtype);
  if (!conv_pool || !aligned(conv_pool, xs) || (L > 0 && (!x || !aligned(x, xs))) ||
      (conv_state_in && !aligned(conv_state_in, xs)) ||
      (cache_seqlens && !aligned(cache_seqlens, 4)) ||
      (conv_state_indices && !aligned(conv_state_indices, 4)))
    return SSS_ERR_INVALID_ARG;
  if ((hT != nullptr) != (ssm_pool != nullptr)) return SSS_ERR_INVALID_ARG;
  if (hT && (!aligned(hT, 16) || !aligned(ssm_pool, 16) || (int64_t(P) * N) % 4))
    return SSS_ERR_INVALID_ARG;
  return from_cuda(sss::prefill_to_pool_launch(
      x, x_dtype, conv_state_in, K, hT, conv_pool, pool, S_len, ssm_pool, cache_seqlens,
      conv_state_indices, Bz, L, D, int64_t(H) * P * N, status_word(),
      reinterpret_cast<cudaStream_t>(stream)));
}

sss_status sss_state_reset(const float* u, float p_reset, float* h, int64_t Bz,
                           int64_t h_row_elems, void* conv_state, sss_dtype conv_dtype,
                           int64_t conv_row_elems, sss_stream_t stream) {
  if (Bz < 0 || h_row_elems < 0 || conv_row_elems < 0 || !dtype_ok(conv_dtype))
    return SSS_ERR_INVALID_ARG;
  if (Bz == 0) return SSS_OK;
  if (!u || !aligned(u, 4) || (h && !aligned(h, 4)) ||
      (conv_state && !aligned(conv_state, dtype_size(conv_dtype))))
    return SSS_ERR_INVALID_ARG;
  if (!h && !conv_state) return SSS_ERR_INVALID_ARG;
  return from_cuda(sss::state_reset_launch(u, p_reset, h, Bz, h ? h_row_elems : 0, conv_state,
                                           conv_dtype, conv_state ? conv_row_elems : 0,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

sss_status sss_fitted_noise_update(const float* hT, int64_t Bz, int H, int P, int N, float beta,
                                   int has_history, float* mu, float* var, sss_stream_t stream) {
  if (Bz < 1 || H < 1 || P < 1 || N < 1 || !(beta >= 0.0f && beta <= 1.0f))
    return SSS_ERR_INVALID_ARG;
  if (!hT || !mu || !var || !aligned(hT, 4) || !aligned(mu, 4) || !aligned(var, 4))
    return SSS_ERR_INVALID_ARG;
  return from_cuda(sss::fitted_noise_update_launch(hT, Bz, H, int64_t(P) * N, beta, has_history,
                                                   mu, var, reinterpret_cast<cudaStream_t>(stream)));
}

sss_status sss_fitted_noise_sample(const float* mu, const float* var, const float* eps,
                                   float* h0, int64_t Bz, int H, int P, int N,
                                   sss_stream_t stream) {
  if (Bz < 0 || H < 1 || P < 1 || N < 1) return SSS_ERR_INVALID_ARG;
  if (Bz == 0) return SSS_OK;
  if (!mu || !var || !eps || !h0 || !aligned(mu, 4) || !aligned(var, 4) || !aligned(eps, 4) ||
      !aligned(h0, 4))
    return SSS_ERR_INVALID_ARG;
  return from_cuda(sss::fitted_noise_sample_launch(mu, var, eps, h0, Bz, H, int64_t(P) * N,
                                                   reinterpret_cast<cudaStream_t>(stream)));
}

sss_status sss_state_std_trace(const void* x, sss_dtype x_dtype, const void* dt, const float* A,
                               const void* B, sss_dtype act_dtype, const float* h0, float* out,
                               int64_t Bz, int64_t L, int H, int P, int N, int G, int stride,
                               sss_stream_t stream) {
  if (!dtype_ok(x_dtype) || !dtype_ok(act_dtype)) return SSS_ERR_INVALID_ARG;
  if (Bz < 0 || L < 0 || H < 1 || P < 1 || N < 1 || G < 1 || H % G || stride < 1)
    return SSS_ERR_INVALID_ARG;
  if (!sss::ssm_scan_bwd_supports(P, N) || stride > sss::state_trace_max_stride())
    return SSS_ERR_UNSUPPORTED;
  if (Bz == 0 || L == 0) return SSS_OK;
  if (!x || !dt || !A || !B || !out || !aligned(x, dtype_size(x_dtype)) ||
      !aligned(dt, dtype_size(act_dtype)) || !aligned(B, dtype_size(act_dtype)) ||
      !aligned(A, 4) || !aligned(out, 4) || (h0 && !aligned(h0, 4)))
    return SSS_ERR_INVALID_ARG;
  return from_cuda(sss::state_std_trace_launch(x, x_dtype, dt, A, B, act_dtype, h0, out, Bz, L, H,
                                               P, N, G, stride,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

int sss_mixer_fwd_supported(int64_t Bz, int64_t L, int H, int P, int N, int G, int K,
                            sss_dtype x_dtype, sss_dtype y_dtype) {
  (void)Bz; (void)y_dtype;
  return (L == 0 || mixer_fwd_tc_supports(x_dtype, x_dtype, K, L > 0 ? L : 1, H, P, N, G)) ? 1 : 0;
}

static sss_status mixer_fwd_impl(const void* x, sss_dtype x_dtype, const float* w, const float* bias,
                         const void* conv_state_in, void* conv_state_out, const void* dt,
                         const float* A, const void* B, const void* C, const float* h0_in,
                         float* hT_out, void* y, sss_dtype y_dtype, int64_t Bz, int64_t L, int H,
                         int P, int N, int G, int K, const int32_t* seq_idx, sss_stream_t stream) {
  if (!dtype_ok(x_dtype) || !dtype_ok(y_dtype)) return SSS_ERR_INVALID_ARG;
  if (Bz < 0 || L < 0 || H < 1 || P < 1 || N < 1 || G < 1 || H % G || K < 1)
    return SSS_ERR_INVALID_ARG;
  if (!sss_mixer_fwd_supported(Bz, L, H, P, N, G, K, x_dtype, y_dtype)) return SSS_ERR_UNSUPPORTED;
  if (Bz == 0) return SSS_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (!w || !A || !aligned(w, 4) || !aligned(A, 4) || (bias && !aligned(bias, 4)))
    return SSS_ERR_INVALID_ARG;
  if ((conv_state_in && !aligned(conv_state_in, 2)) || (conv_state_out && !aligned(conv_state_out, 2)) ||
      (h0_in && !aligned(h0_in, 4)) || (hT_out && !aligned(hT_out, 4)))
    return SSS_ERR_INVALID_ARG;
  if (L == 0) {  // no tokens: F = S and hT = h0, through the general kernels
    sss_status r = sss_conv_state_fwd(nullptr, x_dtype, w, bias, conv_state_in, conv_state_out,
                                      nullptr, SSS_F32, Bz, 0, int64_t(H) * P, K, 1, stream);
    if (r != SSS_OK) return r;
    return from_cuda(ssm_scan_simt_launch(nullptr, SSS_F32, nullptr, A, nullptr, nullptr,
                                          x_dtype, h0_in, hT_out, nullptr, y_dtype, Bz, 0, H, P,
                                          N, G, nullptr, st));
  }
  if (!x || !dt || !B || !C || !y || !aligned(x, 16) || !aligned(dt, 2) || !aligned(B, 16) ||
      !aligned(C, 16) || !aligned(y, 16))
    return SSS_ERR_INVALID_ARG;
  if (ssm_scan_pair_supports(x_dtype, L, H, P, N, G))
    return from_cuda(mixer_fwd_pair_launch(x, w, bias, conv_state_in, conv_state_out, dt, A, B,
                                           C, h0_in, hT_out, y, y_dtype, Bz, L, H, G, K,
                                           status_word(), seq_idx, st));
  // packed rows need the pair kernel's per-piece halo mask
  if (seq_idx) return SSS_ERR_UNSUPPORTED;
  return from_cuda(mixer_fwd_tc_launch(x, w, bias, conv_state_in, conv_state_out, dt, A, B, C,
                                       h0_in, hT_out, y, y_dtype, Bz, L, H, G, K, status_word(),
                                       nullptr, st));
}

sss_status sss_mixer_fwd(const void* x, sss_dtype x_dtype, const float* w, const float* bias,
                         const void* conv_state_in, void* conv_state_out, const void* dt,
                         const float* A, const void* B, const void* C, const float* h0_in,
                         float* hT_out, void* y, sss_dtype y_dtype, int64_t Bz, int64_t L, int H,
                         int P, int N, int G, int K, sss_stream_t stream) {
  return mixer_fwd_impl(x, x_dtype, w, bias, conv_state_in, conv_state_out, dt, A, B, C, h0_in,
                        hT_out, y, y_dtype, Bz, L, H, P, N, G, K, nullptr, stream);
}

sss_status sss_mixer_fwd_packed(const void* x, sss_dtype x_dtype, const float* w,
                                const float* bias, const void* conv_state_in,
                                void* conv_state_out, const void* dt, const float* A,
                                const void* B, const void* C, const float* h0_in, float* hT_out,
                                const int32_t* seq_idx, void* y, sss_dtype y_dtype, int64_t Bz,
                                int64_t L, int H, int P, int N, int G, int K,
                                sss_stream_t stream) {
  if (Bz > 0 && L > 0 && (!seq_idx || !aligned(seq_idx, 4))) return SSS_ERR_INVALID_ARG;
  return mixer_fwd_impl(x, x_dtype, w, bias, conv_state_in, conv_state_out, dt, A, B, C, h0_in,
                        hT_out, y, y_dtype, Bz, L, H, P, N, G, K, seq_idx, stream);
}

// ---- span-parallel forward --------------------------------------------------

// Scratch of the span path, in order, each 256-byte aligned: partial sums of
// the log-decay over 64-token pieces of every span [Bz*ns][ceil(Ls/64)][H],
// the spans' zero-start final states and their initial states
// [Bz*ns][H][P][N] fp32, and (conv only) their conv states [Bz*ns][H*P][K-1]
// bf16.
struct SpanWs {
  float* part;
  float* hloc;
  float* h0s;
  void* s_span;
  size_t bytes;
};

static size_t round256(size_t v) { return (v + 255) & ~size_t(255); }

static SpanWs span_ws(void* base, int64_t Bz, int64_t L, int H, int P, int N, int K, int ns) {
  const size_t rows = size_t(Bz) * size_t(ns);
  const size_t lam = round256(span_part_floats(Bz, L, H, ns) * sizeof(float));
  const size_t st = round256(rows * H * P * N * sizeof(float));
  const size_t cs = K > 1 ? round256(rows * H * P * (K - 1) * 2) : 0;
  char* b = static_cast<char*>(base);
  if (!b) return {nullptr, nullptr, nullptr, nullptr, lam + 2 * st + cs};
  return {reinterpret_cast<float*>(b), reinterpret_cast<float*>(b + lam),
          reinterpret_cast<float*>(b + lam + st), K > 1 ? b + lam + 2 * st : nullptr,
          lam + 2 * st + cs};
}

// The split that minimises the estimated time: CTAs of the head-pair kernel
// (one per SM) run in waves; a launch of it costs about its span length plus
// a fixed pipeline fill and drain worth ~450 tokens (measured: 81 us for
// 2048 tokens and 275 us for 8192 at 24 CTAs, 32 us for 512 at 96 CTAs); the
// span path adds two passes and its two small kernels (~150 tokens).  A split
// is taken when it is estimated to save a tenth of the one-pass time.
static int span_count_for(int64_t Bz, int64_t L, int H, int K) {
  constexpr int64_t kMinSpan = 256, kStartup = 450, kSmall = 150;
  const int64_t ctas = Bz * (H / 2);
  if (ctas < 1 || L < 2 * kMinSpan) return 1;
  const int64_t sms = sm_count();
  const double one = double((ctas + sms - 1) / sms) * double(L + kStartup);
  int best = 1;
  double best_t = 0.9 * one;
  for (int ns = 2; ns <= 32; ++ns) {
    if (L % ns) continue;
    const int64_t Ls = L / ns;
    if (Ls < kMinSpan || Ls < K - 1) continue;
    const double t =
        double((ctas * ns + sms - 1) / sms) * 2.0 * double(Ls + kStartup) + double(kSmall);
    if (t < best_t) {
      best = ns;
      best_t = t;
    }
  }
  return best;
}

static bool spans_supported(bool fused, sss_dtype x_dtype, sss_dtype act_dtype, sss_dtype y_dtype,
                            int64_t Bz, int64_t Ls, int H, int P, int N, int G, int K,
                            int ns) {
  if (!span_sizes_ok(Bz, Ls * ns, int64_t(H) * P, H, P, N, K, ns)) return false;
  if (!ssm_scan_pair_supports(act_dtype, Ls, H, P, N, G)) return false;
  if (fused)
    return x_dtype == SSS_BF16 && sss_mixer_fwd_supported(Bz, Ls, H, P, N, G, K, x_dtype, y_dtype);
  return ssm_scan_tc_supports(x_dtype, act_dtype, y_dtype, Ls, H, P, N, G);
}

static sss_status fwd_spans_impl(bool fused, const void* x, sss_dtype x_dtype, const float* w,
                                 const float* bias, const void* s_in, void* s_out, const void* dt,
                                 const float* A, const void* B, const void* C, sss_dtype act_dtype,
                                 const float* h0_in, float* hT_out, void* y, sss_dtype y_dtype,
                                 int64_t Bz, int64_t L, int H, int P, int N, int G, int K, int ns,
                                 void* workspace, size_t workspace_bytes, sss_stream_t stream) {
  if (!dtype_ok(x_dtype) || !dtype_ok(act_dtype) || !dtype_ok(y_dtype)) return SSS_ERR_INVALID_ARG;
  if (ns < 1 || ns > 32 || Bz < 0 || L < 0 || H < 1 || P < 1 || N < 1 || G < 1 || H % G || K < 1)
    return SSS_ERR_INVALID_ARG;
  if (ns == 1 || Bz == 0 || L == 0) {
    if (fused)
      return mixer_fwd_impl(x, x_dtype, w, bias, s_in, s_out, dt, A, B, C, h0_in, hT_out, y,
                            y_dtype, Bz, L, H, P, N, G, K, nullptr, stream);
    return scan_fwd_impl(x, x_dtype, dt, A, B, C, act_dtype, h0_in, hT_out, y, y_dtype, Bz, L, H,
                         P, N, G, nullptr, stream);
  }
  if (L % ns || L / ns < K - 1) return SSS_ERR_INVALID_ARG;
  const int64_t Ls = L / ns;
  if (!fused) K = 1;
  if (!spans_supported(fused, x_dtype, act_dtype, y_dtype, Bz, Ls, H, P, N, G, K, ns))
    return SSS_ERR_UNSUPPORTED;
  // the span kernels (gather of the conv state and per-span decay sums) read
  // dt, B, C and, fused, x and the conv state as bf16
  if (act_dtype != SSS_BF16 || (fused && x_dtype != SSS_BF16)) return SSS_ERR_UNSUPPORTED;
  if (!x || !dt || !A || !B || !C || !y || !aligned(x, 16) || !aligned(dt, 2) || !aligned(A, 4) ||
      !aligned(B, 16) || !aligned(C, 16) || !aligned(y, 16))
    return SSS_ERR_INVALID_ARG;
  if ((h0_in && !aligned(h0_in, 16)) || (hT_out && !aligned(hT_out, 16)))
    return SSS_ERR_INVALID_ARG;
  if (fused && (!w || !aligned(w, 4) || (bias && !aligned(bias, 4)) ||
                (s_in && !aligned(s_in, 2)) || (s_out && !aligned(s_out, 2))))
    return SSS_ERR_INVALID_ARG;
  const SpanWs need = span_ws(nullptr, Bz, L, H, P, N, K, ns);
  if (!workspace || workspace_bytes < need.bytes || !aligned(workspace, 256))
    return SSS_ERR_INVALID_ARG;
  const SpanWs ws = span_ws(workspace, Bz, L, H, P, N, K, ns);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int64_t rows = Bz * ns;
  int* status = status_word();
  cudaError_t e = span_prepare_launch(x, fused ? s_in : nullptr, fused ? s_out : nullptr,
                                      ws.s_span, dt, A, ws.part, Bz, L, int64_t(H) * P, H, K,
                                      ns, st);
  // pass 1: every span from a zero state, only its final state kept (the
  // state-only kernel: no y)
  if (e == cudaSuccess)
    e = fused ? mixer_fwd_pair_state_launch(x, w, bias, ws.s_span, dt, A, B, ws.hloc, rows, Ls, H,
                                            G, K, status, st)
              : ssm_scan_pair_state_launch(x, x_dtype, dt, A, B, ws.hloc, rows, Ls, H, G, status,
                                           st);
  // the carry over the spans, then pass 2: every span from its true initial
  // state, writing y.  The three launches after the first are programmatic
  // dependents: each starts while the one before drains and waits
  // (griddepcontrol.wait) for its results before it reads them.
  if (e == cudaSuccess)
    e = span_combine_launch(ws.part, ws.hloc, h0_in, ws.h0s, hT_out, Bz, L, H, int64_t(P) * N, ns,
                            st);
  if (e == cudaSuccess)
    e = fused ? mixer_fwd_pair_launch(x, w, bias, ws.s_span, nullptr, dt, A, B, C, ws.h0s,
                                      nullptr, y, y_dtype, rows, Ls, H, G, K, status, nullptr, st,
                                      true)
              : ssm_scan_pair_launch(x, x_dtype, dt, A, B, C, ws.h0s, nullptr, y, y_dtype, rows,
                                     Ls, H, G, status, nullptr, st, true);
  return from_cuda(e);
}

int sss_mixer_fwd_span_count(int64_t Bz, int64_t L, int H, int P, int N, int G, int K,
                             sss_dtype x_dtype, sss_dtype y_dtype) {
  if (!dtype_ok(x_dtype) || !dtype_ok(y_dtype)) return 1;
  if (Bz < 1 || L < 1 || H < 1 || P < 1 || N < 1 || G < 1 || H % G || K < 1) return 1;
  const int ns = span_count_for(Bz, L, H, K);
  if (ns > 1 && !spans_supported(true, x_dtype, x_dtype, y_dtype, Bz, L / ns, H, P, N, G, K, ns))
    return 1;
  return ns;
}

int sss_ssm_scan_fwd_span_count(int64_t Bz, int64_t L, int H, int P, int N, int G,
                                sss_dtype x_dtype, sss_dtype act_dtype, sss_dtype y_dtype) {
  if (!dtype_ok(x_dtype) || !dtype_ok(act_dtype) || !dtype_ok(y_dtype)) return 1;
  if (Bz < 1 || L < 1 || H < 1 || P < 1 || N < 1 || G < 1 || H % G) return 1;
  const int ns = span_count_for(Bz, L, H, 1);
  if (ns > 1 && !spans_supported(false, x_dtype, act_dtype, y_dtype, Bz, L / ns, H, P, N, G, 1, ns))
    return 1;
  return ns;
}

size_t sss_fwd_spans_workspace_size(int64_t Bz, int64_t L, int H, int P, int N, int K, int ns) {
  if (Bz < 1 || L < 1 || H < 1 || P < 1 || N < 1 || K < 1 || ns < 2 || ns > 32) return 0;
  return span_ws(nullptr, Bz, L, H, P, N, K, ns).bytes;
}

sss_status sss_mixer_fwd_spans(const void* x, sss_dtype x_dtype, const float* w,
                               const float* bias, const void* conv_state_in,
                               void* conv_state_out, const void* dt, const float* A,
                               const void* B, const void* C, const float* h0_in, float* hT_out,
                               void* y, sss_dtype y_dtype, int64_t Bz, int64_t L, int H, int P,
                               int N, int G, int K, int ns, void* workspace,
                               size_t workspace_bytes, sss_stream_t stream) {
  return fwd_spans_impl(true, x, x_dtype, w, bias, conv_state_in, conv_state_out, dt, A, B, C,
                        x_dtype, h0_in, hT_out, y, y_dtype, Bz, L, H, P, N, G, K, ns, workspace,
                        workspace_bytes, stream);
}

sss_status sss_ssm_scan_fwd_spans(const void* x, sss_dtype x_dtype, const void* dt,
                                  const float* A, const void* B, const void* C,
                                  sss_dtype act_dtype, const float* h0_in, float* hT_out, void* y,
                                  sss_dtype y_dtype, int64_t Bz, int64_t L, int H, int P, int N,
                                  int G, int ns, void* workspace, size_t workspace_bytes,
                                  sss_stream_t stream) {
  return fwd_spans_impl(false, x, x_dtype, nullptr, nullptr, nullptr, nullptr, dt, A, B, C,
                        act_dtype, h0_in, hT_out, y, y_dtype, Bz, L, H, P, N, G, 1, ns, workspace,
                        workspace_bytes, stream);
}

int sss_mixer_update_path(int L_new, int P, int N, int K, int S_len, sss_dtype act_dtype) {
  if (!dtype_ok(act_dtype) || L_new < 0 || P < 1 || N < 1 || K < 1 || S_len < 1 ||
      S_len < K - 1)
    return -1;
  return sss::mixer_update_path(act_dtype, S_len, L_new, P, N, K);
}

sss_status sss_mixer_update(const void* x_new, sss_dtype act_dtype, const float* w,
                            const float* bias, void* conv_pool, int64_t pool, int S_len,
                            const int32_t* cache_seqlens, const int32_t* conv_state_indices,
                            const void* dt, const float* A, const void* B, const void* C,
                            float* ssm_pool, void* y, int64_t Bz, int L_new, int H, int P,
                            int N, int G, int K, sss_stream_t stream) {
  if (!dtype_ok(act_dtype)) return SSS_ERR_INVALID_ARG;
  if (Bz < 0 || pool < 0 || L_new < 0 || H < 1 || P < 1 || N < 1 || G < 1 || H % G || K < 1 ||
      S_len < 1 || S_len < K - 1)
    return SSS_ERR_INVALID_ARG;
  if (!mixer_update_supports(P, N, K, L_new)) return SSS_ERR_UNSUPPORTED;
  if (Bz == 0 || L_new == 0) return SSS_OK;
  const size_t as = dtype_size(act_dtype);
  if (!x_new || !w || !conv_pool || !dt || !A || !B || !C || !ssm_pool || !y)
    return SSS_ERR_INVALID_ARG;
  if (!aligned(x_new, as) || !aligned(conv_pool, as) || !aligned(dt, as) || !aligned(B, as) ||
      !aligned(C, as) || !aligned(y, as) || !aligned(w, 4) || (bias && !aligned(bias, 4)) ||
      !aligned(A, 4) || !aligned(ssm_pool, 16) ||
      (cache_seqlens && !aligned(cache_seqlens, 4)) ||
      (conv_state_indices && !aligned(conv_state_indices, 4)))
    return SSS_ERR_INVALID_ARG;
  return from_cuda(mixer_update_launch(x_new, act_dtype, w, bias, conv_pool, pool, S_len,
                                       cache_seqlens, conv_state_indices, dt, A, B, C,
                                       ssm_pool, y, Bz, L_new, H, P, N, G, K, status_word(),
                                       reinterpret_cast<cudaStream_t>(stream)));
}

sss_status sss_device_status(int* status_out, int clear, sss_stream_t stream) {
  if (!status_out) return SSS_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int* p = status_word();
  if (!p) return SSS_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyAsync(&v, p, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return SSS_ERR_CUDA;
  if (clear && cudaMemsetAsync(p, 0, sizeof(int), st) != cudaSuccess) return SSS_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SSS_ERR_CUDA;
  *status_out = v;
  return SSS_OK;
}

// ---- the full Mamba-2 mixer wiring ------------------------------------------
size_t sss_mamba2_mixer_fwd_workspace_size(int64_t Bz, int64_t L, int H, int P, int N, int G) {
  if (Bz < 0 || L < 0 || H < 1 || P < 1 || N < 1 || G < 1) return 0;
  return size_t(Bz) * size_t(L) * size_t(int64_t(H) * P + 2 * int64_t(G) * N) * sizeof(float);
}

sss_status sss_mamba2_mixer_fwd(const void* xBC, const void* z, sss_dtype act_dtype,
                                const void* dt_raw, const float* dt_bias, const float* A,
                                const float* D_skip, const float* conv_w, const float* conv_b,
                                const void* conv_state_in, void* conv_state_out,
                                const float* h0_in, float* hT_out, void* y, sss_dtype y_dtype,
                                int64_t Bz, int64_t L, int H, int P, int N, int G, int K,
                                void* workspace, size_t workspace_bytes, sss_stream_t stream) {
  if (!dtype_ok(act_dtype) || !dtype_ok(y_dtype)) return SSS_ERR_INVALID_ARG;
  if (Bz < 0 || L < 0 || H < 1 || P < 1 || N < 1 || G < 1 || H % G || K < 1)
    return SSS_ERR_INVALID_ARG;
  if (K > 8 || !ssm_scan_simt_supports(P, N)) return SSS_ERR_UNSUPPORTED;
  if (Bz == 0) return SSS_OK;
  const size_t as = dtype_size(act_dtype), ys = dtype_size(y_dtype);
  const int64_t Dt = int64_t(H) * P + 2 * int64_t(G) * N;
  if (!A || !conv_w || !aligned(A, 4) || !aligned(conv_w, 4) || (conv_b && !aligned(conv_b, 4)) ||
      (dt_bias && !aligned(dt_bias, 4)) || (D_skip && !aligned(D_skip, 4)))
    return SSS_ERR_INVALID_ARG;
  if ((conv_state_in && !aligned(conv_state_in, as)) ||
      (conv_state_out && !aligned(conv_state_out, as)) || (h0_in && !aligned(h0_in, 4)) ||
      (hT_out && !aligned(hT_out, 4)))
    return SSS_ERR_INVALID_ARG;
  if (L > 0) {
    if (!xBC || !dt_raw || !y || !aligned(xBC, as) || !aligned(dt_raw, as) || !aligned(y, ys) ||
        (z && !aligned(z, as)))
      return SSS_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 16) ||
        workspace_bytes < sss_mamba2_mixer_fwd_workspace_size(Bz, L, H, P, N, G))
      return SSS_ERR_INVALID_ARG;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the conv + SiLU of every xBC channel into the workspace, in fp32 (the
  // scan reads B and C from it unrounded), and the final conv state
  if (L > 0 || conv_state_out) {
    cudaError_t e = conv_state_fwd_launch(xBC, act_dtype, conv_w, conv_b, conv_state_in,
                                          conv_state_out, L > 0 ? workspace : nullptr, SSS_F32,
                                          Bz, L, Dt, K, 1, st);
    if (e != cudaSuccess) return from_cuda(e);
  }
  if (L == 0) {
    // no tokens: the state passes through unchanged
    if (hT_out && hT_out != h0_in) {
      const size_t bytes = size_t(Bz) * H * P * N * sizeof(float);
      const cudaError_t e = h0_in ? cudaMemcpyAsync(hT_out, h0_in, bytes, cudaMemcpyDeviceToDevice, st)
                                  : cudaMemsetAsync(hT_out, 0, bytes, st);
      if (e != cudaSuccess) return from_cuda(e);
    }
    return SSS_OK;
  }
  return from_cuda(mamba2_scan_launch(static_cast<const float*>(workspace), z, dt_raw, act_dtype,
                                      dt_bias, A, D_skip, h0_in, hT_out, y, y_dtype, Bz, L, H, P,
                                      N, G, st));
}

}  // extern "C"
