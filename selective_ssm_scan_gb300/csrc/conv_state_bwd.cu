// Gradient of the causal depthwise conv with an explicit (K-1)-sample state.
//
// Follows "Chapter 7: state, chunking and incremental inference" (causal-conv1d
// tutorial), section "unified derivation of the backward pass with state":
// with u = [S, x], z_t = bias + sum_k w_k u_{t+k}, out_t = SiLU(z_t) and
// F = u[L : L+K-1], the upstream gradients dy = dL/dout and q = dL/dF give
//   delta_t = dy_t SiLU'(z_t),
//   dL/du_j = sum_{t,k: t+k=j} delta_t w_k + [L <= j < L+K-1] q_{j-L},
//   dS = du[0 : K-1],  dx = du[K-1 : K-1+L],
//   dw_k = sum_t delta_t u_{t+k},  dbias = sum_t delta_t   (and over the batch).
//
// GB300 mapping (HBM-bound: read x and dy once, write dx once):
//  * a CTA is 8 warps; warp w takes the token tile tg * 8 + w of kTile tokens,
//    lane l the channel vector d0 = (blockIdx.x * 32 + l) * VEC, so each load
//    of a token row is one contiguous line per warp;
//  * a thread recomputes z for the tokens [t0, t0 + kTile + K - 1) from the
//    x window [t0 - (K-1), t0 + kTile + K - 1) (the conv state in front of
//    token 0), turns dy into delta there, and forms dx_t for its kTile
//    tokens from delta_{t..t+K-1} (the correlation runs forward in time);
//  * the tile holding token 0 writes dS, the tiles holding the last K-1
//    tokens add q;
//  * dw and dbias: each thread sums its tile, the CTA sums its 8 tiles in
//    shared memory and writes one row of partials to the workspace; a second
//    kernel adds the rows in a fixed order, so the result is deterministic.
#include "common.cuh"

namespace sss {

namespace {
constexpr int kBwdWarps = 8;
constexpr int kBwdTile = 8;         // tokens per warp
constexpr int kBwdMaxK = 8;
constexpr int kBwdCtaTokens = kBwdWarps * kBwdTile;

__device__ __forceinline__ float dsilu(float z) {
  // d/dz [z s(z)] = s (1 + z (1 - s)), s = 1 / (1 + exp(-z))
  const float s = __fdividef(1.0f, 1.0f + __expf(fminf(-z, 80.0f)));
  return s * fmaf(z, 1.0f - s, 1.0f);
}
}  // namespace

template <typename TX, typename TD, typename TO, int VEC, int KT, bool SILU>
__global__ void __launch_bounds__(kBwdWarps * 32)
conv_state_bwd_kernel(const TX* __restrict__ x, const float* __restrict__ w,
                      const float* __restrict__ bias, const TX* __restrict__ s_in,
                      const TD* __restrict__ dy, const TD* __restrict__ q, TO* __restrict__ dx,
                      TO* __restrict__ dS, float* __restrict__ part, int L, int D, int K_rt,
                      int n_dvec, int n_groups) {
  constexpr int MK = KT > 0 ? KT : kBwdMaxK;
  constexpr int NW = kBwdTile + 2 * (MK - 1);  // x window: u indices
  constexpr int NZ = kBwdTile + MK - 1;        // tokens whose z (delta) is needed
  const int K = KT > 0 ? KT : K_rt;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int dvec = blockIdx.x * 32 + lane;
  const int tg = blockIdx.y;
  const int64_t b = blockIdx.z;
  const int t0 = (tg * kBwdWarps + warp) * kBwdTile;
  const bool live = dvec < n_dvec && t0 < L;
  const int d0 = dvec * VEC;

  float dwp[MK][VEC], dbp[VEC];
#pragma unroll
  for (int v = 0; v < VEC; ++v) {
    dbp[v] = 0.0f;
#pragma unroll
    for (int k = 0; k < MK; ++k) dwp[k][v] = 0.0f;
  }

  if (live) {
    float wk[MK][VEC], bs[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
      bs[v] = bias ? bias[d0 + v] : 0.0f;
#pragma unroll
      for (int k = 0; k < MK; ++k) wk[k][v] = k < K ? w[(d0 + v) * K + k] : 0.0f;
    }
    // ext[i] = u_{t0 + i} = x_{t0 + i - (K-1)}, i in [0, NW); S in front of
    // token 0, zero past the end
    float ext[NW][VEC];
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      const int tx = t0 + i - (K - 1);
#pragma unroll
      for (int v = 0; v < VEC; ++v) {
        float val = 0.0f;
        if (i < kBwdTile + 2 * (K - 1)) {
          if (tx >= 0 && tx < L)
            val = to_f32(x[(b * L + tx) * D + d0 + v]);
          else if (tx < 0 && s_in)
            val = to_f32(s_in[(b * D + d0 + v) * (K - 1) + (K - 1) + tx]);
        }
        ext[i][v] = val;
      }
    }
    // delta_t for t = t0 + i, i in [0, NZ), zero for t >= L
    float dl[NZ][VEC];
#pragma unroll
    for (int i = 0; i < NZ; ++i) {
      const int t = t0 + i;
#pragma unroll
      for (int v = 0; v < VEC; ++v) {
        float dv = 0.0f;
        if (i < kBwdTile + K - 1 && t < L) {
          float z = bs[v];
#pragma unroll
          for (int k = 0; k < MK; ++k)
            if (k < K) z = fmaf(wk[k][v], ext[i + k][v], z);
          const float g = to_f32(dy[(b * L + t) * D + d0 + v]);
          dv = SILU ? g * dsilu(z) : g;
        }
        dl[i][v] = dv;
      }
    }
    // dx_t = sum_k w_k delta_{t+K-1-k} (+ q for the last K-1 tokens)
#pragma unroll
    for (int i = 0; i < kBwdTile; ++i) {
      const int t = t0 + i;
      if (t < L) {
        float o[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
          float acc = 0.0f;
#pragma unroll
          for (int k = 0; k < MK; ++k)
            if (k < K) acc = fmaf(wk[k][v], dl[i + K - 1 - k][v], acc);
          const int r = t + K - 1 - L;  // tail slot of F this input became
          if (r >= 0 && q) acc += to_f32(q[(b * D + d0 + v) * (K - 1) + r]);
          o[v] = acc;
        }
#pragma unroll
        for (int v = 0; v < VEC; ++v) dx[(b * L + t) * D + d0 + v] = from_f32<TO>(o[v]);
      }
    }
    // dS_j = du_j = sum_k w_k delta_{j-k} (+ q_{j-L} when j >= L), j < K-1
    if (t0 == 0) {
      for (int j = 0; j < K - 1; ++j) {
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
          float acc = 0.0f;
#pragma unroll
          for (int k = 0; k < MK; ++k) {
            const int i = j - k;
            if (k < K && i >= 0) {
              // dl is indexed from t0 = 0; i < K-1 < NZ
#pragma unroll
              for (int ii = 0; ii < NZ; ++ii)
                if (ii == i) acc = fmaf(wk[k][v], dl[ii][v], acc);
            }
          }
          if (j >= L && q) acc += to_f32(q[(b * D + d0 + v) * (K - 1) + (j - L)]);
          dS[(b * D + d0 + v) * (K - 1) + j] = from_f32<TO>(acc);
        }
      }
    }
    // this tile's dw_k = sum_t delta_t u_{t+k}, dbias = sum_t delta_t
#pragma unroll
    for (int i = 0; i < kBwdTile; ++i) {
#pragma unroll
      for (int v = 0; v < VEC; ++v) {
        dbp[v] += dl[i][v];
#pragma unroll
        for (int k = 0; k < MK; ++k) dwp[k][v] = fmaf(dl[i][v], ext[i + k][v], dwp[k][v]);
      }
    }
  }

  // the CTA's 8 tiles summed in shared memory, in warp order
  __shared__ float red[kBwdWarps][MK + 1][32 * VEC];
#pragma unroll
  for (int v = 0; v < VEC; ++v) {
#pragma unroll
    for (int k = 0; k < MK; ++k) red[warp][k][lane * VEC + v] = dwp[k][v];
    red[warp][MK][lane * VEC + v] = dbp[v];
  }
  __syncthreads();
  // row (b, tg) of the partials: [D][K+1] floats
  float* row = part + (b * n_groups + tg) * int64_t(D) * (K + 1);
  for (int e = threadIdx.x; e < 32 * VEC * (K + 1); e += blockDim.x) {
    const int c = e / (K + 1), k = e % (K + 1);  // channel c of this CTA's 32*VEC
    const int d = blockIdx.x * 32 * VEC + c;
    if (d < n_dvec * VEC) {
      const int kk = k < K ? k : MK;
      float acc = 0.0f;
      for (int ww = 0; ww < kBwdWarps; ++ww) acc += red[ww][kk][c];
      row[int64_t(d) * (K + 1) + k] = acc;
    }
  }
}

// dw[d][k] = sum over rows of part[row][d][k] (k < K); dbias[d] = part[..][d][K]
__global__ void conv_bwd_reduce_kernel(const float* __restrict__ part, float* __restrict__ dw,
                                       float* __restrict__ dbias, int64_t rows, int D, int K) {
  const int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t n = int64_t(D) * (K + 1);
  if (e >= n) return;
  float acc = 0.0f;
  for (int64_t r = 0; r < rows; ++r) acc += part[r * n + e];
  const int d = int(e / (K + 1)), k = int(e % (K + 1));
  if (k < K)
    dw[int64_t(d) * K + k] = acc;
  else if (dbias)
    dbias[d] = acc;
}

// L = 0: F = S, so dS = q, and there is no weight or bias gradient
template <typename TD, typename TO>
__global__ void conv_bwd_empty_kernel(const TD* __restrict__ q, TO* __restrict__ dS,
                                      float* __restrict__ dw, float* __restrict__ dbias,
                                      int64_t n_state, int D, int K) {
  const int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e < n_state) dS[e] = from_f32<TO>(q ? to_f32(q[e]) : 0.0f);
  if (e < int64_t(D) * K) dw[e] = 0.0f;
  if (dbias && e < D) dbias[e] = 0.0f;
}

size_t conv_state_bwd_workspace(int64_t Bz, int64_t L, int64_t D, int K) {
  if (Bz <= 0 || L <= 0 || D <= 0 || K < 1) return 0;
  const int64_t groups = (L + kBwdCtaTokens - 1) / kBwdCtaTokens;
  return size_t(Bz * groups * D * (K + 1)) * sizeof(float);
}

bool conv_state_bwd_supports(int K) { return K >= 1 && K <= kBwdMaxK; }

template <typename TX, typename TD, typename TO, int VEC>
static cudaError_t launch_bwd(const void* x, const float* w, const float* bias, const void* s_in,
                              const void* dy, const void* q, void* dx, void* dS, float* dw,
                              float* dbias, int64_t Bz, int64_t L, int64_t D, int K, int silu_on,
                              void* ws, cudaStream_t st) {
  const int64_t n_dvec = D / VEC;
  const int64_t groups = (L + kBwdCtaTokens - 1) / kBwdCtaTokens;
  if (groups > 65535 || Bz > 65535) return cudaErrorInvalidValue;
  const dim3 grid(unsigned((n_dvec + 31) / 32), unsigned(groups), unsigned(Bz));
  float* part = static_cast<float*>(ws);
  auto args = [&](auto kern) -> cudaError_t {
    kern<<<grid, kBwdWarps * 32, 0, st>>>(
        static_cast<const TX*>(x), w, bias, static_cast<const TX*>(s_in),
        static_cast<const TD*>(dy), static_cast<const TD*>(q), static_cast<TO*>(dx),
        static_cast<TO*>(dS), part, int(L), int(D), K, int(n_dvec), int(groups));
    return cudaGetLastError();
  };
  cudaError_t e;
  if (K == 4)
    e = silu_on ? args(conv_state_bwd_kernel<TX, TD, TO, VEC, 4, true>)
                : args(conv_state_bwd_kernel<TX, TD, TO, VEC, 4, false>);
  else
    e = silu_on ? args(conv_state_bwd_kernel<TX, TD, TO, VEC, 0, true>)
                : args(conv_state_bwd_kernel<TX, TD, TO, VEC, 0, false>);
  if (e != cudaSuccess) return e;
  const int64_t n = D * (K + 1);
  conv_bwd_reduce_kernel<<<unsigned((n + 255) / 256), 256, 0, st>>>(part, dw, dbias,
                                                                     Bz * groups, int(D), K);
  return cudaGetLastError();
}

template <typename TX, typename TD, typename TO>
static cudaError_t bwd_vec(const void* x, const float* w, const float* bias, const void* s_in,
                           const void* dy, const void* q, void* dx, void* dS, float* dw,
                           float* dbias, int64_t Bz, int64_t L, int64_t D, int K, int silu_on,
                           void* ws, cudaStream_t st) {
  if (L == 0) {
    const int64_t n_state = Bz * D * (K - 1);
    const int64_t n = n_state > D * K ? n_state : D * K;
    if (n == 0) return cudaSuccess;
    conv_bwd_empty_kernel<TD, TO><<<unsigned((n + 255) / 256), 256, 0, st>>>(
        static_cast<const TD*>(q), static_cast<TO*>(dS), dw, dbias, n_state, int(D), K);
    return cudaGetLastError();
  }
  if (D % 2 == 0)
    return launch_bwd<TX, TD, TO, 2>(x, w, bias, s_in, dy, q, dx, dS, dw, dbias, Bz, L, D, K,
                                     silu_on, ws, st);
  return launch_bwd<TX, TD, TO, 1>(x, w, bias, s_in, dy, q, dx, dS, dw, dbias, Bz, L, D, K,
                                   silu_on, ws, st);
}

cudaError_t conv_state_bwd_launch(const void* x, sss_dtype xt, const float* w, const float* bias,
                                  const void* s_in, const void* dy, sss_dtype dyt, const void* q,
                                  void* dx, sss_dtype dxt, void* dS, float* dw, float* dbias,
                                  int64_t Bz, int64_t L, int64_t D, int K, int silu_on,
                                  void* ws, cudaStream_t st) {
#define SSS_BWD(TX, TD, TO)                                                                   \
  return bwd_vec<TX, TD, TO>(x, w, bias, s_in, dy, q, dx, dS, dw, dbias, Bz, L, D, K, silu_on, \
                             ws, st)
  using bf = __nv_bfloat16;
  if (xt == SSS_BF16) {
    if (dyt == SSS_F32) {
      if (dxt == SSS_BF16) SSS_BWD(bf, float, bf);
      SSS_BWD(bf, float, float);
    }
    if (dxt == SSS_BF16) SSS_BWD(bf, bf, bf);
    SSS_BWD(bf, bf, float);
  }
  if (dyt == SSS_F32) {
    if (dxt == SSS_BF16) SSS_BWD(float, float, bf);
    SSS_BWD(float, float, float);
  }
  if (dxt == SSS_BF16) SSS_BWD(float, bf, bf);
  SSS_BWD(float, bf, float);
#undef SSS_BWD
}

}  // namespace sss
