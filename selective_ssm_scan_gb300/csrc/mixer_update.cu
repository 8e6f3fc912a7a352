// Single/multi-token decode update over a circular conv-state pool, followed
// by the scalar-decay recurrence on the pool's SSM state.
//
// Follows "Chapter 7: state, chunking and incremental inference", sections
// "single-token update" (window of the K-1 previous inputs, store x not y),
// "the physical cache may be longer than the minimum history", "circular
// mode" (write slot p mod S_len, history j at slot (p - j) mod S_len, read
// before overwrite, cache_seqlens not advanced here) and "continuous
// batching" (conv_state_indices maps batch rows to pool rows); the state
// update is Eq. (1) of "Understanding and Improving Length Generalization in
// Recurrent Models" with A_t = exp(dt_t A_h).
//
// GB300 mapping (HBM-bound: the fp32 SSM state, P*N*4 bytes per head and
// request, is read and written once and dominates the traffic):
//  * one CTA per (request, head), 8 warps; warp w owns state rows
//    p = w + 8 r, lane l owns the float4 column groups n4 = l + 32 c, so the
//    state moves as fully coalesced 16-byte accesses and three CTAs share an
//    SM (the loads of the state are what keeps HBM busy);
//  * threads p < P first run the conv of channel d = h*P + p: they read every
//    history slot they need into registers, compute u for the L_new tokens
//    and only then store the new inputs into the slots, so the kernel is
//    correct for any L_new, including L_new >= S_len;
//  * the readout y[p] = sum_n h[p,n] C[n] is a warp reduce-scatter;
//  * a row whose pool index is outside [0, pool) or whose length is negative
//    is skipped (y rows zeroed, status bit SSS_ERR_INDEX raised).
#include "common.cuh"

namespace sss {

constexpr int kUpdWarps = 8;
constexpr int kUpdMaxLnew = 64;
constexpr int kUpdMaxK = 8;

template <int R>
__device__ __forceinline__ float upd_reduce_scatter(float* v, int lane, int* row) {
  int r = 0;
#pragma unroll
  for (int s = 0; s < 5; ++s) {
    const int off = 16 >> s;
    const int w = R >> s;
    if (w >= 2) {
      const int half = w / 2;
      const bool up = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < half; ++i) {
        const float send = up ? v[i] : v[i + half];
        const float keep = up ? v[i + half] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
      }
      if (up) r += half;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
    }
  }
  *row = r;
  return v[0];
}

__device__ __forceinline__ int64_t pos_mod(int64_t a, int64_t m) {
  int64_t r = a % m;
  return r < 0 ? r + m : r;
}

template <typename T, int RP, int CV, int KT>
__global__ void __launch_bounds__(kUpdWarps * 32, RP * CV <= 8 ? 3 : 1)
mixer_update_kernel(const T* __restrict__ x, const float* __restrict__ w,
                    const float* __restrict__ bias, T* conv_pool, int64_t pool, int S_len,
                    const int32_t* __restrict__ seqlens, const int32_t* __restrict__ idx,
                    const T* __restrict__ dt, const float* __restrict__ A,
                    const T* __restrict__ Bm, const T* __restrict__ Cm, float* ssm_pool,
                    T* __restrict__ y, int L_new, int H, int P, int N, int G, int K,
                    int* status) {
  extern __shared__ float sm[];
  float* us = sm;                             // [L_new][P]  conv outputs of this head
  float* bs = us + ((L_new * P + 3) & ~3);    // [L_new][N]  16-byte aligned
  float* cs = bs + L_new * N;            // [L_new][N]
  float* as = cs + L_new * N;            // [L_new]

  const int b = blockIdx.x / H, h = blockIdx.x % H;
  const int g = h / (H / G);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int D = H * P;
  const int64_t r = idx ? int64_t(idx[b]) : int64_t(b);
  const int64_t p0 = int64_t(seqlens[b]);

  if (r < 0 || r >= pool || p0 < 0) {
    for (int i = tid; i < L_new * P; i += blockDim.x) {
      const int tt = i / P, p = i % P;
      y[((int64_t(b) * L_new + tt) * H + h) * P + p] = from_f32<T>(0.0f);
    }
    if (tid == 0) raise_status(status, SSS_ERR_INDEX);
    return;
  }

  // ---- SSM state (loads issued first, consumed after the conv):
  //      rows p = warp + kUpdWarps rr, float4 groups n4 = lane + 32 c ----
  float* hs = ssm_pool + (r * H + h) * int64_t(P) * N;
  const int N4 = N / 4;
  float4 st[RP][CV];
#pragma unroll
  for (int rr = 0; rr < RP; ++rr)
#pragma unroll
    for (int c = 0; c < CV; ++c) {
      const int p = warp + kUpdWarps * rr, n4 = lane + 32 * c;
      st[rr][c] = (p < P && n4 < N4) ? reinterpret_cast<const float4*>(hs + int64_t(p) * N)[n4]
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }

  // ---- conv over the circular window, one thread per channel ------------
  for (int p = tid; p < P; p += blockDim.x) {
    const int64_t d = int64_t(h) * P + p;
    T* row = conv_pool + (r * D + d) * S_len;
    // every history value this call needs is read before any slot write:
    // logical position p0 - (K-1) + j sits in slot (p0 - (K-1) + j) mod S_len
    float win[KT - 1];
#pragma unroll
    for (int j = 0; j < KT - 1; ++j)
      win[j] = (j < K - 1) ? to_f32(row[pos_mod(p0 - (K - 1) + j, S_len)]) : 0.0f;
    float wk[KT];
#pragma unroll
    for (int k = 0; k < KT; ++k) wk[k] = k < K ? w[d * K + k] : 0.0f;
    const float bsd = bias ? bias[d] : 0.0f;
    for (int i = 0; i < L_new; ++i) {
      const float xv = to_f32(x[(int64_t(b) * L_new + i) * D + d]);
      float z = bsd;
#pragma unroll
      for (int k = 0; k < KT - 1; ++k)
        if (k < K - 1) z = fmaf(wk[k], win[k], z);
#pragma unroll
      for (int k = 0; k < KT; ++k)
        if (k == K - 1) z = fmaf(wk[k], xv, z);
      us[i * P + p] = silu(z);
#pragma unroll
      for (int k = 0; k < KT - 2; ++k)
        if (k < K - 2) win[k] = win[k + 1];
#pragma unroll
      for (int k = 0; k < KT - 1; ++k)
        if (k == K - 2) win[k] = xv;
    }
    // store the inputs (not the outputs) at the write pointer, in token
    // order, after all reads of this channel's row
    for (int i = 0; i < L_new; ++i)
      row[pos_mod(p0 + i, S_len)] = x[(int64_t(b) * L_new + i) * D + d];
  }
  for (int i = tid; i < L_new * N; i += blockDim.x) {
    const int tt = i / N, n = i % N;
    const int64_t o = ((int64_t(b) * L_new + tt) * G + g) * N + n;
    bs[tt * N + n] = to_f32(Bm[o]);
    cs[tt * N + n] = to_f32(Cm[o]);
  }
  for (int i = tid; i < L_new; i += blockDim.x)
    as[i] = expf(to_f32(dt[(int64_t(b) * L_new + i) * H + h]) * A[h]);
  __syncthreads();

  for (int i = 0; i < L_new; ++i) {
    const float a = as[i];
    float part[RP];
#pragma unroll
    for (int rr = 0; rr < RP; ++rr) {
      const int p = warp + kUpdWarps * rr;
      const float xv = p < P ? us[i * P + p] : 0.0f;
      float acc = 0.0f;
#pragma unroll
      for (int c = 0; c < CV; ++c) {
        const int n4 = lane + 32 * c;
        if (n4 < N4) {
          const float4 bv = reinterpret_cast<const float4*>(bs + i * N)[n4];
          const float4 cv = reinterpret_cast<const float4*>(cs + i * N)[n4];
          float4& s = st[rr][c];
          s.x = fmaf(a, s.x, xv * bv.x);
          s.y = fmaf(a, s.y, xv * bv.y);
          s.z = fmaf(a, s.z, xv * bv.z);
          s.w = fmaf(a, s.w, xv * bv.w);
          acc = fmaf(s.x, cv.x, acc);
          acc = fmaf(s.y, cv.y, acc);
          acc = fmaf(s.z, cv.z, acc);
          acc = fmaf(s.w, cv.w, acc);
        }
      }
      part[rr] = acc;
    }
    int row;
    const float yv = upd_reduce_scatter<RP>(part, lane, &row);
    const int p = warp + kUpdWarps * row;
    if ((lane & (32 / RP - 1)) == 0 && p < P)
      y[((int64_t(b) * L_new + i) * H + h) * P + p] = from_f32<T>(yv);
  }
#pragma unroll
  for (int rr = 0; rr < RP; ++rr)
#pragma unroll
    for (int c = 0; c < CV; ++c) {
      const int p = warp + kUpdWarps * rr, n4 = lane + 32 * c;
      if (p < P && n4 < N4) reinterpret_cast<float4*>(hs + int64_t(p) * N)[n4] = st[rr][c];
    }
}

template <typename T, int RP, int CV, int KT>
static cudaError_t launch_upd(const void* x, const float* w, const float* bias, void* cp,
                              int64_t pool, int S_len, const int32_t* sl, const int32_t* ix,
                              const void* dt, const float* A, const void* B, const void* C,
                              float* sp, void* y, int64_t Bz, int L_new, int H, int P, int N,
                              int G, int K, int* status, cudaStream_t st) {
  const size_t smem = size_t(((L_new * P + 3) & ~3) + 2 * L_new * N + L_new) * sizeof(float);
  auto kern = mixer_update_kernel<T, RP, CV, KT>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
    if (e != cudaSuccess) return e;
  }
  const int64_t grid = Bz * H;
  if (grid == 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<unsigned(grid), kUpdWarps * 32, smem, st>>>(
      static_cast<const T*>(x), w, bias, static_cast<T*>(cp), pool, S_len, sl, ix,
      static_cast<const T*>(dt), A, static_cast<const T*>(B), static_cast<const T*>(C), sp,
      static_cast<T*>(y), L_new, H, P, N, G, K, status);
  return cudaGetLastError();
}

template <typename T>
static cudaError_t upd_shape(const void* x, const float* w, const float* bias, void* cp,
                             int64_t pool, int S_len, const int32_t* sl, const int32_t* ix,
                             const void* dt, const float* A, const void* B, const void* C,
                             float* sp, void* y, int64_t Bz, int L_new, int H, int P, int N,
                             int G, int K, int* status, cudaStream_t st) {
#define SSS_UPD(RP, CV)                                                                     \
  if (P <= kUpdWarps * RP && N <= 128 * CV) {                                               \
    if (K <= 4)                                                                             \
      return launch_upd<T, RP, CV, 4>(x, w, bias, cp, pool, S_len, sl, ix, dt, A, B, C, sp, y, \
                                      Bz, L_new, H, P, N, G, K, status, st);                 \
    return launch_upd<T, RP, CV, 8>(x, w, bias, cp, pool, S_len, sl, ix, dt, A, B, C, sp, y,   \
                                    Bz, L_new, H, P, N, G, K, status, st);                   \
  }
  SSS_UPD(1, 1)
  SSS_UPD(8, 1)
  SSS_UPD(16, 2)
#undef SSS_UPD
  return cudaErrorNotSupported;
}

bool mixer_update_supports(int P, int N, int K, int L_new) {
  return P <= kUpdWarps * 16 && N <= 256 && N % 4 == 0 && K >= 1 && K <= kUpdMaxK &&
         L_new <= kUpdMaxLnew;
}

cudaError_t mixer_update_launch(const void* x, sss_dtype at, const float* w, const float* bias,
                                void* cp, int64_t pool, int S_len, const int32_t* sl,
                                const int32_t* ix, const void* dt, const float* A,
                                const void* B, const void* C, float* sp, void* y, int64_t Bz,
                                int L_new, int H, int P, int N, int G, int K, int* status,
                                cudaStream_t st) {
  if (at == SSS_BF16)
    return upd_shape<__nv_bfloat16>(x, w, bias, cp, pool, S_len, sl, ix, dt, A, B, C, sp, y,
                                    Bz, L_new, H, P, N, G, K, status, st);
  return upd_shape<float>(x, w, bias, cp, pool, S_len, sl, ix, dt, A, B, C, sp, y, Bz, L_new,
                          H, P, N, G, K, status, st);
}

}  // namespace sss
