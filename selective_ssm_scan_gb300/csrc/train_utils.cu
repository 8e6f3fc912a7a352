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
#include <cooperative_groups.h>

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

// Fixed-order sum over the CTAs of a cluster of kStatCtas (deterministic):
// warp shuffles, the CTA's warps in order, then every CTA reads the partials
// of all cluster ranks in rank order through distributed shared memory.
constexpr int kStatCtas = 8;
__device__ double cluster_sum(double v, double* red, double* part) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    double s = 0.0;
    for (int i = 0; i < kStatThreads / 32; ++i) s += red[i];
    *part = s;
  }
  cl.sync();  // every rank's partial is written
  double t = 0.0;
  for (int r = 0; r < kStatCtas; ++r) t += *cl.map_shared_rank(part, r);
  cl.sync();  // no rank rewrites its partial while another still reads it
  return t;
}

// a cluster of kStatCtas CTAs per head: each sums a contiguous share of the
// head's Bz x P x N values (fp32 over four interleaved float4 streams, fp64
// across threads and CTAs), the mean, then the centred squares, then the EMA
__global__ void __launch_bounds__(kStatThreads)
fitted_noise_update_kernel(const float* __restrict__ hT, int64_t Bz, int H, int64_t PN, float beta,
                           int has_history, float* __restrict__ mu, float* __restrict__ var) {
  __shared__ double red[kStatThreads / 32];
  __shared__ double part;
  const int h = blockIdx.x / kStatCtas, rank = blockIdx.x % kStatCtas;
  const int64_t n = Bz * PN;
  const bool vec = (PN & 3) == 0 && (reinterpret_cast<uintptr_t>(hT) & 15) == 0;
  // this CTA's rows: batch rows b with b % kStatCtas == rank, each a
  // contiguous block of PN values of head h
  // first pass: the sum
  double s1 = 0.0, s2 = 0.0;
  for (int64_t b = rank; b < Bz; b += kStatCtas) {
    const float* row = hT + (b * H + h) * PN;
    float a4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (vec) {
      const float4* r4 = reinterpret_cast<const float4*>(row);
      for (int64_t i = threadIdx.x; i < PN / 4; i += kStatThreads) {
        const float4 q = r4[i];
        a4[0] += q.x;
        a4[1] += q.y;
        a4[2] += q.z;
        a4[3] += q.w;
      }
    } else {
      for (int64_t i = threadIdx.x; i < PN; i += kStatThreads) a4[i & 3] += row[i];
    }
    s1 += double(a4[0]) + double(a4[1]) + double(a4[2]) + double(a4[3]);
  }
  const double mean = n > 0 ? cluster_sum(s1, red, &part) / double(n) : 0.0;
  const float mf = float(mean);
  for (int64_t b = rank; b < Bz; b += kStatCtas) {
    const float* row = hT + (b * H + h) * PN;
    float a4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (vec) {
      const float4* r4 = reinterpret_cast<const float4*>(row);
      for (int64_t i = threadIdx.x; i < PN / 4; i += kStatThreads) {
        const float4 q = r4[i];
        const float d0 = q.x - mf, d1 = q.y - mf, d2 = q.z - mf, d3 = q.w - mf;
        a4[0] = fmaf(d0, d0, a4[0]);
        a4[1] = fmaf(d1, d1, a4[1]);
        a4[2] = fmaf(d2, d2, a4[2]);
        a4[3] = fmaf(d3, d3, a4[3]);
      }
    } else {
      for (int64_t i = threadIdx.x; i < PN; i += kStatThreads) {
        const float d = row[i] - mf;
        a4[i & 3] = fmaf(d, d, a4[i & 3]);
      }
    }
    s2 += double(a4[0]) + double(a4[1]) + double(a4[2]) + double(a4[3]);
  }
  // centred on the fp32-rounded mean: sum (x - m)^2 = sum (x - mf)^2 - n (m - mf)^2
  const double dm = mean - double(mf);
  const double v = n > 0 ? cluster_sum(s2, red, &part) / double(n) - dm * dm : 0.0;
  if (rank == 0 && threadIdx.x == 0) {
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(H) * kStatCtas);
  cfg.blockDim = dim3(kStatThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kStatCtas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fitted_noise_update_kernel, hT, Bz, H, PN, beta, has_history, mu,
                            var);
}

cudaError_t fitted_noise_sample_launch(const float* mu, const float* var, const float* eps,
                                       float* h0, int64_t Bz, int H, int64_t PN, cudaStream_t st) {
  const int64_t total = Bz * H * PN;
  if (total == 0) return cudaSuccess;
  fitted_noise_sample_kernel<<<grid_for(total, kResetThreads, 4096), kResetThreads, 0, st>>>(
      mu, var, eps, h0, total, H, PN);
  return cudaGetLastError();
}


// ---- prefill into the pool ---------------------------------------------------
// A prompt's state written into the pool rows the decode update reads ("Chapter
// 7: state, chunking and incremental inference", sections "continuous
// batching" and "circular mode"): row r = idx[b] of the conv pool gets the
// newest S_len entries of u = [state_in, x] (zeros where u has none) - at slot
// q mod S_len for logical position q in circular mode (the prompt at positions
// p - L .. p - 1, p = seqlens[b]), oldest first without lengths - and row r of
// the SSM pool gets hT[b].  Bad rows are skipped and reported.
namespace {
template <typename T>
__global__ void __launch_bounds__(kResetThreads)
prefill_conv_kernel(const T* __restrict__ x, const T* __restrict__ state_in, int K,
                    T* __restrict__ conv_pool, int64_t pool, int S_len,
                    const int32_t* __restrict__ seqlens, const int32_t* __restrict__ idx,
                    int64_t L, int64_t D, int* status) {
  const int64_t b = blockIdx.y;
  const int64_t r = idx ? int64_t(idx[b]) : b;
  const int64_t p = seqlens ? int64_t(seqlens[b]) : L;
  if (r < 0 || r >= pool || p < 0) {
    if (blockIdx.x == 0 && threadIdx.x == 0) raise_status(status, SSS_ERR_INDEX);
    return;
  }
  const int64_t first = p - L - (K - 1);  // logical position of u[0]
  for (int64_t d = blockIdx.x * int64_t(kResetThreads) + threadIdx.x; d < D;
       d += int64_t(gridDim.x) * kResetThreads) {
    T* row = conv_pool + (r * D + d) * S_len;
    for (int j = 0; j < S_len; ++j) {
      const int64_t q = p - S_len + j;
      const int64_t i = q - first;
      T v = from_f32<T>(0.0f);
      if (i >= 0 && i < K - 1) {
        if (state_in) v = state_in[(b * D + d) * (K - 1) + i];
      } else if (i >= K - 1 && i < K - 1 + L) {
        v = x[(b * L + (i - (K - 1))) * D + d];
      }
      const int64_t slot = seqlens ? ((q % S_len) + S_len) % S_len : j;
      row[slot] = v;
    }
  }
}

__global__ void __launch_bounds__(kResetThreads)
prefill_ssm_kernel(const float* __restrict__ hT, float* __restrict__ ssm_pool, int64_t pool,
                   const int32_t* __restrict__ seqlens, const int32_t* __restrict__ idx,
                   int64_t row_elems) {
  const int64_t b = blockIdx.y;
  const int64_t r = idx ? int64_t(idx[b]) : b;
  if (r < 0 || r >= pool || (seqlens && seqlens[b] < 0)) return;  // reported by the conv kernel
  const float4* src = reinterpret_cast<const float4*>(hT + b * row_elems);
  float4* dst = reinterpret_cast<float4*>(ssm_pool + r * row_elems);
  for (int64_t i = blockIdx.x * int64_t(kResetThreads) + threadIdx.x; i < row_elems / 4;
       i += int64_t(gridDim.x) * kResetThreads)
    dst[i] = src[i];
}
}  // namespace

cudaError_t prefill_to_pool_launch(const void* x, sss_dtype dt, const void* state_in, int K,
                                   const float* hT, void* conv_pool, int64_t pool, int S_len,
                                   float* ssm_pool, const int32_t* seqlens, const int32_t* idx,
                                   int64_t Bz, int64_t L, int64_t D, int64_t ssm_row_elems,
                                   int* status, cudaStream_t st) {
  if (Bz == 0) return cudaSuccess;
  const dim3 gc(grid_for(D, kResetThreads, 64), unsigned(Bz));
  if (dt == SSS_BF16)
    prefill_conv_kernel<__nv_bfloat16><<<gc, kResetThreads, 0, st>>>(
        static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(state_in), K,
        static_cast<__nv_bfloat16*>(conv_pool), pool, S_len, seqlens, idx, L, D, status);
  else
    prefill_conv_kernel<float><<<gc, kResetThreads, 0, st>>>(
        static_cast<const float*>(x), static_cast<const float*>(state_in), K,
        static_cast<float*>(conv_pool), pool, S_len, seqlens, idx, L, D, status);
  if (hT && ssm_pool && ssm_row_elems > 0) {
    const dim3 gs(grid_for(ssm_row_elems / 4, kResetThreads, 64), unsigned(Bz));
    prefill_ssm_kernel<<<gs, kResetThreads, 0, st>>>(hT, ssm_pool, pool, seqlens, idx,
                                                     ssm_row_elems);
  }
  return cudaGetLastError();
}

}  // namespace sss
