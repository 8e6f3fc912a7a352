// State-passing training utilities of "Understanding and Improving Length
// Generalization in Recurrent Models":
//  * state_reset (section 4.4, state passing): a batch row restarts from zero
//    when its uniform draw is below p (the pages use p = 0.1); the conv state
//    row is reset with it.  Only the reset rows are written.
//  * fitted_noise_update (section 4.2, Eqs. (5)-(6)): per head, the mean and
//    the (population) variance of the final states over batch x P x N, mixed
//    into the running values with weight 1 - beta on the new statistic and
//    beta on the history (beta = 0.1: the new statistic weighs 0.9).
//  * fitted_noise_sample: h0 = mu_h + sqrt(var_h) eps, eps ~ N(0, 1) given.
// The random draws are inputs, so results are reproducible from the caller's
// generator.  The per-head state-std trace (section 3.5) lives with the
// chunk walk in ssm_scan_bwd.cu.
#include "common.cuh"

namespace sss {

namespace {
constexpr int kResetThreads = 256;
constexpr int kStatThreads = 512;

// grid (row chunks, Bz): rows whose draw is below p are zeroed, 16 bytes a
// thread where the row is aligned
template <typename T>
__global__ void __launch_bounds__(kResetThreads)
state_reset_kernel(const float* __restrict__ u, float p, T* __restrict__ rows, int64_t elems) {
  const int64_t b = blockIdx.y;
  if (!(u[b] < p)) return;
  T* row = rows + b * elems;
  constexpr int kVec = 16 / sizeof(T);
  const bool vec = (reinterpret_cast<uintptr_t>(row) & 15) == 0;
  const int64_t nv = vec ? elems / kVec : 0;
  for (int64_t i = blockIdx.x * int64_t(kResetThreads) + threadIdx.x; i < nv;
       i += int64_t(gridDim.x) * kResetThreads)
    reinterpret_cast<uint4*>(row)[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int64_t i = nv * kVec + blockIdx.x * int64_t(kResetThreads) + threadIdx.x; i < elems;
       i += int64_t(gridDim.x) * kResetThreads)
    row[i] = from_f32<T>(0.0f);
}

// fixed-order block sum (deterministic)
__device__ double block_sum(double v, double* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  double s = 0.0;
  for (int i = 0; i < kStatThreads / 32; ++i) s += red[i];
  return s;
}

// one CTA per head: mean, then the centred sum of squares, then the EMA
__global__ void __launch_bounds__(kStatThreads)
fitted_noise_update_kernel(const float* __restrict__ hT, int64_t Bz, int H, int64_t PN, float beta,
                           int has_history, float* __restrict__ mu, float* __restrict__ var) {
  __shared__ double red[kStatThreads / 32];
  const int h = blockIdx.x;
  const int64_t n = Bz * PN;
  double s = 0.0;
  for (int64_t i = threadIdx.x; i < n; i += kStatThreads) {
    const int64_t b = i / PN, e = i % PN;
    s += double(hT[(b * H + h) * PN + e]);
  }
  const double mean = n > 0 ? block_sum(s, red) / double(n) : 0.0;
  double q = 0.0;
  for (int64_t i = threadIdx.x; i < n; i += kStatThreads) {
    const int64_t b = i / PN, e = i % PN;
    const double d = double(hT[(b * H + h) * PN + e]) - mean;
    q += d * d;
  }
  const double v = n > 0 ? block_sum(q, red) / double(n) : 0.0;
  if (threadIdx.x == 0) {
    if (has_history) {
      mu[h] = float((1.0 - double(beta)) * mean + double(beta) * double(mu[h]));
      var[h] = float((1.0 - double(beta)) * v + double(beta) * double(var[h]));
    } else {
      mu[h] = float(mean);
      var[h] = float(v);
    }
  }
}

__global__ void __launch_bounds__(kResetThreads)
fitted_noise_sample_kernel(const float* __restrict__ mu, const float* __restrict__ var,
                           const float* __restrict__ eps, float* __restrict__ h0, int64_t total,
                           int H, int64_t PN) {
  for (int64_t i = blockIdx.x * int64_t(kResetThreads) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * kResetThreads) {
    const int h = int((i / PN) % H);
    h0[i] = fmaf(sqrtf(var[h]), eps[i], mu[h]);
  }
}

inline int grid_for(int64_t work, int64_t per_block, int cap) {
  const int64_t g = (work + per_block - 1) / per_block;
  return int(g < 1 ? 1 : (g > cap ? cap : g));
}
}  // namespace

cudaError_t state_reset_launch(const float* u, float p, float* h, int64_t Bz, int64_t h_elems,
                               void* conv, sss_dtype conv_t, int64_t conv_elems, cudaStream_t st) {
  if (Bz == 0) return cudaSuccess;
  if (h && h_elems > 0) {
    const dim3 g(grid_for(h_elems / 4, kResetThreads, 64), unsigned(Bz));
    state_reset_kernel<float><<<g, kResetThreads, 0, st>>>(u, p, h, h_elems);
  }
  if (conv && conv_elems > 0) {
    const dim3 g(grid_for(conv_elems / 8, kResetThreads, 64), unsigned(Bz));
    if (conv_t == SSS_BF16)
      state_reset_kernel<__nv_bfloat16><<<g, kResetThreads, 0, st>>>(
          u, p, static_cast<__nv_bfloat16*>(conv), conv_elems);
    else
      state_reset_kernel<float><<<g, kResetThreads, 0, st>>>(u, p, static_cast<float*>(conv),
                                                              conv_elems);
  }
  return cudaGetLastError();
}

cudaError_t fitted_noise_update_launch(const float* hT, int64_t Bz, int H, int64_t PN, float beta,
                                       int has_history, float* mu, float* var, cudaStream_t st) {
  fitted_noise_update_kernel<<<H, kStatThreads, 0, st>>>(hT, Bz, H, PN, beta, has_history, mu, var);
  return cudaGetLastError();
}

cudaError_t fitted_noise_sample_launch(const float* mu, const float* var, const float* eps,
                                       float* h0, int64_t Bz, int H, int64_t PN, cudaStream_t st) {
  const int64_t total = Bz * H * PN;
  if (total == 0) return cudaSuccess;
  fitted_noise_sample_kernel<<<grid_for(total, kResetThreads, 4096), kResetThreads, 0, st>>>(
      mu, var, eps, h0, total, H, PN);
  return cudaGetLastError();
}

}  // namespace sss
