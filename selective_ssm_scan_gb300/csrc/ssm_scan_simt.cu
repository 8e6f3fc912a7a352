// fp32 CUDA-core selective scan (one scalar decay per head) from an initial
// state, one token at a time.
//
// Follows "Understanding and Improving Length Generalization in Recurrent
// Models", section 2 Eq. (1), h_t = A_t h_{t-1} + B_t x_t, y_t = C_t^T h_t,
// with A_t = exp(dt_t A_h) and the non-zero initial state of Eq. (4).
//
// This is the path for fp32 activations (where the result must match to
// ~1e-5) and for head/state sizes the tensor-core chunked scan does not
// take.  One CTA owns one (batch, head) and keeps its P x N state in
// registers for the whole sequence: warp w holds rows p = w + 8 r, lane l
// holds columns n = l + 32 c.  Per token each thread updates its state
// elements and forms partial dot products with C_t; the readout
// y[p] = sum_n h[p,n] C[n] is a reduce-scatter over the warp's lanes:
// R - 1 + 5 - log2(R) shuffles for the warp's R rows instead of 5 R.
// Inputs of TCH tokens are staged in shared memory with the decay
// a_t = exp(dt_t A_h) computed once per token.
#include "common.cuh"

namespace sss {

constexpr int kSimtWarps = 8;

// Sum v[0..R) over the 32 lanes of a warp so that each lane ends with the
// full sum of one row; `row` says which.  R must be a power of two <= 32.
template <int R>
__device__ __forceinline__ float warp_reduce_scatter(float* v, int lane, int* row) {
  int r = 0;
#pragma unroll
  for (int s = 0; s < 5; ++s) {
    const int off = 16 >> s;
    const int w = R >> s;  // values still held before this step
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

template <typename TX, typename TA, typename TY, int RP, int CN>
__global__ void __launch_bounds__(kSimtWarps * 32)
ssm_scan_simt_kernel(const TX* __restrict__ x, const TA* __restrict__ dt,
                     const float* __restrict__ A, const TA* __restrict__ Bm,
                     const TA* __restrict__ Cm, const float* h0, float* hT,
                     TY* __restrict__ y, int64_t L, int H, int P, int N, int G, int TCH,
                     const int32_t* __restrict__ seq_idx) {
  extern __shared__ float smem[];
  float* xs = smem;               // [TCH][P]
  float* bs = xs + TCH * P;       // [TCH][N]
  float* cs = bs + TCH * N;       // [TCH][N]
  float* as = cs + TCH * N;       // [TCH]

  const int b = blockIdx.x / H, h = blockIdx.x % H;
  const int g = h / (H / G);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float Ah = A[h];

  float st[RP][CN];
#pragma unroll
  for (int r = 0; r < RP; ++r)
#pragma unroll
    for (int c = 0; c < CN; ++c) {
      const int p = warp + kSimtWarps * r, n = lane + 32 * c;
      st[r][c] = (h0 && p < P && n < N) ? h0[((int64_t(b) * H + h) * P + p) * N + n] : 0.0f;
    }

  for (int64_t t0 = 0; t0 < L; t0 += TCH) {
    const int nt = int((L - t0) < TCH ? (L - t0) : TCH);
    __syncthreads();
    for (int i = tid; i < nt * P; i += blockDim.x) {
      const int tt = i / P, p = i % P;
      xs[tt * P + p] = to_f32(x[((int64_t(b) * L + t0 + tt) * H + h) * P + p]);
    }
    for (int i = tid; i < nt * N; i += blockDim.x) {
      const int tt = i / N, n = i % N;
      const int64_t o = ((int64_t(b) * L + t0 + tt) * G + g) * N + n;
      bs[tt * N + n] = to_f32(Bm[o]);
      cs[tt * N + n] = to_f32(Cm[o]);
    }
    for (int i = tid; i < nt; i += blockDim.x)
      as[i] = expf(sample_start(seq_idx, b, L, t0 + i)
                       ? kSampleStartLog
                       : to_f32(dt[(int64_t(b) * L + t0 + i) * H + h]) * Ah);
    __syncthreads();

    for (int tt = 0; tt < nt; ++tt) {
      const float a = as[tt];
      float bv[CN], cv[CN];
#pragma unroll
      for (int c = 0; c < CN; ++c) {
        const int n = lane + 32 * c;
        bv[c] = n < N ? bs[tt * N + n] : 0.0f;
        cv[c] = n < N ? cs[tt * N + n] : 0.0f;
      }
      float part[RP];
#pragma unroll
      for (int r = 0; r < RP; ++r) {
        const int p = warp + kSimtWarps * r;
        const float xv = p < P ? xs[tt * P + p] : 0.0f;
        float acc = 0.0f;
#pragma unroll
        for (int c = 0; c < CN; ++c) {
          st[r][c] = fmaf(a, st[r][c], xv * bv[c]);
          acc = fmaf(st[r][c], cv[c], acc);
        }
        part[r] = acc;
      }
      int row;
      const float yv = warp_reduce_scatter<RP>(part, lane, &row);
      const int p = warp + kSimtWarps * row;
      if ((lane & (32 / RP - 1)) == 0 && p < P)
        y[((int64_t(b) * L + t0 + tt) * H + h) * P + p] = from_f32<TY>(yv);
    }
  }

  if (hT) {
#pragma unroll
    for (int r = 0; r < RP; ++r)
#pragma unroll
      for (int c = 0; c < CN; ++c) {
        const int p = warp + kSimtWarps * r, n = lane + 32 * c;
        if (p < P && n < N) hT[((int64_t(b) * H + h) * P + p) * N + n] = st[r][c];
      }
  }
}

template <typename TX, typename TA, typename TY, int RP, int CN>
static cudaError_t launch_simt(const void* x, const void* dt, const float* A,
                               const void* B, const void* C, const float* h0,
                               float* hT, void* y, int64_t Bz, int64_t L, int H,
                               int P, int N, int G, const int32_t* seq_idx, cudaStream_t st) {
  const int per_tok = (P + 2 * N + 1) * int(sizeof(float));
  int TCH = (40 * 1024) / per_tok;
  if (TCH > 32) TCH = 32;
  if (TCH < 1) TCH = 1;
  const size_t smem = size_t(TCH) * per_tok;
  auto kern = ssm_scan_simt_kernel<TX, TA, TY, RP, CN>;
  const int64_t grid = Bz * H;
  if (grid == 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<unsigned(grid), kSimtWarps * 32, smem, st>>>(
      static_cast<const TX*>(x), static_cast<const TA*>(dt), A, static_cast<const TA*>(B),
      static_cast<const TA*>(C), h0, hT, static_cast<TY*>(y), L, H, P, N, G, TCH, seq_idx);
  return cudaGetLastError();
}

template <typename TX, typename TA, typename TY>
static cudaError_t simt_shape(const void* x, const void* dt, const float* A, const void* B,
                              const void* C, const float* h0, float* hT, void* y, int64_t Bz,
                              int64_t L, int H, int P, int N, int G, const int32_t* seq_idx, cudaStream_t st) {
#define SSS_SIMT(RP, CN)                                                                  \
  if (P <= kSimtWarps * RP && N <= 32 * CN)                                               \
    return launch_simt<TX, TA, TY, RP, CN>(x, dt, A, B, C, h0, hT, y, Bz, L, H, P, N, G, seq_idx, st);
  SSS_SIMT(1, 1)
  SSS_SIMT(2, 2)
  SSS_SIMT(4, 4)
  SSS_SIMT(8, 4)
  SSS_SIMT(16, 8)
#undef SSS_SIMT
  return cudaErrorNotSupported;
}

template <typename TX>
static cudaError_t simt_act(const void* x, sss_dtype at, sss_dtype yt, const void* dt,
                            const float* A, const void* B, const void* C, const float* h0,
                            float* hT, void* y, int64_t Bz, int64_t L, int H, int P, int N,
                            int G, const int32_t* seq_idx, cudaStream_t st) {
  if (at == SSS_F32 && yt == SSS_F32)
    return simt_shape<TX, float, float>(x, dt, A, B, C, h0, hT, y, Bz, L, H, P, N, G, seq_idx, st);
  if (at == SSS_F32)
    return simt_shape<TX, float, __nv_bfloat16>(x, dt, A, B, C, h0, hT, y, Bz, L, H, P, N, G, seq_idx, st);
  if (yt == SSS_F32)
    return simt_shape<TX, __nv_bfloat16, float>(x, dt, A, B, C, h0, hT, y, Bz, L, H, P, N, G, seq_idx, st);
  return simt_shape<TX, __nv_bfloat16, __nv_bfloat16>(x, dt, A, B, C, h0, hT, y, Bz, L, H, P, N, G, seq_idx, st);
}

bool ssm_scan_simt_supports(int P, int N) { return P <= kSimtWarps * 16 && N <= 256; }

cudaError_t ssm_scan_simt_launch(const void* x, sss_dtype xt, const void* dt, const float* A,
                                 const void* B, const void* C, sss_dtype at,
                                 const float* h0, float* hT, void* y, sss_dtype yt,
                                 int64_t Bz, int64_t L, int H, int P, int N, int G,
                                 const int32_t* seq_idx, cudaStream_t st) {
  if (xt == SSS_F32)
    return simt_act<float>(x, at, yt, dt, A, B, C, h0, hT, y, Bz, L, H, P, N, G, seq_idx, st);
  return simt_act<__nv_bfloat16>(x, at, yt, dt, A, B, C, h0, hT, y, Bz, L, H, P, N, G, seq_idx, st);
}

// ---------------------------------------------------------------------------
// The scan of the full Mamba-2 wiring (the Mamba-2 layers of "Understanding
// and Improving Length Generalization in Recurrent Models", with the xBC conv
// of "Chapter 7: state, chunking and incremental inference"): u [Bz, L, D +
// 2 G N] is the fp32 conv + SiLU output of every xBC channel (x in [0, D),
// then B, then C).  Per token dt = softplus(dt_raw + dt_bias_h),
// a = exp(dt A_h), h = a h + dt x B^T, y = (h C + D_h x) SiLU(z).  Same CTA
// layout as the kernel above: the fp32 state stays in registers, B and C are
// fp32 (the conv output is not rounded before the scan).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float softplusf(float v) {
  return v > 20.0f ? v + log1pf(expf(-v)) : log1pf(expf(v));
}

template <typename TA, typename TY, int RP, int CN>
__global__ void __launch_bounds__(kSimtWarps * 32)
mamba2_scan_kernel(const float* __restrict__ u, const TA* __restrict__ z,
                   const TA* __restrict__ dt_raw, const float* __restrict__ dt_bias,
                   const float* __restrict__ A, const float* __restrict__ D_skip,
                   const float* h0, float* hT, TY* __restrict__ y, int64_t L, int H, int P,
                   int N, int G, int TCH) {
  extern __shared__ float smem[];
  float* xs = smem;               // [TCH][P]  x (not scaled by dt)
  float* bs = xs + TCH * P;       // [TCH][N]
  float* cs = bs + TCH * N;       // [TCH][N]
  float* as = cs + TCH * N;       // [TCH]     a_t
  float* ds = as + TCH;           // [TCH]     dt_t

  const int b = blockIdx.x / H, h = blockIdx.x % H;
  const int g = h / (H / G);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float Ah = A[h];
  const float bh = dt_bias ? dt_bias[h] : 0.0f;
  const float Dh = D_skip ? D_skip[h] : 0.0f;
  const int64_t Dx = int64_t(H) * P, Dt = Dx + 2 * int64_t(G) * N;

  float st[RP][CN];
#pragma unroll
  for (int r = 0; r < RP; ++r)
#pragma unroll
    for (int c = 0; c < CN; ++c) {
      const int p = warp + kSimtWarps * r, n = lane + 32 * c;
      st[r][c] = (h0 && p < P && n < N) ? h0[((int64_t(b) * H + h) * P + p) * N + n] : 0.0f;
    }

  for (int64_t t0 = 0; t0 < L; t0 += TCH) {
    const int nt = int((L - t0) < TCH ? (L - t0) : TCH);
    __syncthreads();
    for (int i = tid; i < nt * P; i += blockDim.x) {
      const int tt = i / P, p = i % P;
      xs[tt * P + p] = u[(int64_t(b) * L + t0 + tt) * Dt + int64_t(h) * P + p];
    }
    for (int i = tid; i < nt * N; i += blockDim.x) {
      const int tt = i / N, n = i % N;
      const float* ut = u + (int64_t(b) * L + t0 + tt) * Dt + Dx;
      bs[tt * N + n] = ut[int64_t(g) * N + n];
      cs[tt * N + n] = ut[int64_t(G) * N + int64_t(g) * N + n];
    }
    for (int i = tid; i < nt; i += blockDim.x) {
      const float dtv = softplusf(to_f32(dt_raw[(int64_t(b) * L + t0 + i) * H + h]) + bh);
      ds[i] = dtv;
      as[i] = expf(dtv * Ah);
    }
    __syncthreads();

    for (int tt = 0; tt < nt; ++tt) {
      const float a = as[tt], dtv = ds[tt];
      float bv[CN], cv[CN];
#pragma unroll
      for (int c = 0; c < CN; ++c) {
        const int n = lane + 32 * c;
        bv[c] = n < N ? bs[tt * N + n] : 0.0f;
        cv[c] = n < N ? cs[tt * N + n] : 0.0f;
      }
      float part[RP];
#pragma unroll
      for (int r = 0; r < RP; ++r) {
        const int p = warp + kSimtWarps * r;
        const float xd = p < P ? dtv * xs[tt * P + p] : 0.0f;
        float acc = 0.0f;
#pragma unroll
        for (int c = 0; c < CN; ++c) {
          st[r][c] = fmaf(a, st[r][c], xd * bv[c]);
          acc = fmaf(st[r][c], cv[c], acc);
        }
        part[r] = acc;
      }
      int row;
      const float yv = warp_reduce_scatter<RP>(part, lane, &row);
      const int p = warp + kSimtWarps * row;
      if ((lane & (32 / RP - 1)) == 0 && p < P) {
        const int64_t tok = int64_t(b) * L + t0 + tt;
        const float gate = z ? silu(to_f32(z[tok * Dx + int64_t(h) * P + p])) : 1.0f;
        y[(tok * H + h) * P + p] = from_f32<TY>((yv + Dh * xs[tt * P + p]) * gate);
      }
    }
  }

  if (hT) {
#pragma unroll
    for (int r = 0; r < RP; ++r)
#pragma unroll
      for (int c = 0; c < CN; ++c) {
        const int p = warp + kSimtWarps * r, n = lane + 32 * c;
        if (p < P && n < N) hT[((int64_t(b) * H + h) * P + p) * N + n] = st[r][c];
      }
  }
}

template <typename TA, typename TY, int RP, int CN>
static cudaError_t launch_mamba2(const float* u, const void* z, const void* dt_raw,
                                 const float* dt_bias, const float* A, const float* D_skip,
                                 const float* h0, float* hT, void* y, int64_t Bz, int64_t L,
                                 int H, int P, int N, int G, cudaStream_t st) {
  const int per_tok = (P + 2 * N + 2) * int(sizeof(float));
  int TCH = (40 * 1024) / per_tok;
  if (TCH > 32) TCH = 32;
  if (TCH < 1) TCH = 1;
  const size_t smem = size_t(TCH) * per_tok;
  const int64_t grid = Bz * H;
  if (grid == 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  mamba2_scan_kernel<TA, TY, RP, CN><<<unsigned(grid), kSimtWarps * 32, smem, st>>>(
      u, static_cast<const TA*>(z), static_cast<const TA*>(dt_raw), dt_bias, A, D_skip, h0, hT,
      static_cast<TY*>(y), L, H, P, N, G, TCH);
  return cudaGetLastError();
}

template <typename TA, typename TY>
static cudaError_t mamba2_shape(const float* u, const void* z, const void* dt_raw,
                                const float* dt_bias, const float* A, const float* D_skip,
                                const float* h0, float* hT, void* y, int64_t Bz, int64_t L,
                                int H, int P, int N, int G, cudaStream_t st) {
#define SSS_M2(RP, CN)                                                                        \
  if (P <= kSimtWarps * RP && N <= 32 * CN)                                                   \
    return launch_mamba2<TA, TY, RP, CN>(u, z, dt_raw, dt_bias, A, D_skip, h0, hT, y, Bz, L, H, \
                                         P, N, G, st);
  SSS_M2(1, 1)
  SSS_M2(2, 2)
  SSS_M2(4, 4)
  SSS_M2(8, 4)
  SSS_M2(16, 8)
#undef SSS_M2
  return cudaErrorNotSupported;
}

cudaError_t mamba2_scan_launch(const float* u, const void* z, const void* dt_raw, sss_dtype at,
                               const float* dt_bias, const float* A, const float* D_skip,
                               const float* h0, float* hT, void* y, sss_dtype yt, int64_t Bz,
                               int64_t L, int H, int P, int N, int G, cudaStream_t st) {
  if (at == SSS_F32 && yt == SSS_F32)
    return mamba2_shape<float, float>(u, z, dt_raw, dt_bias, A, D_skip, h0, hT, y, Bz, L, H, P, N, G, st);
  if (at == SSS_F32)
    return mamba2_shape<float, __nv_bfloat16>(u, z, dt_raw, dt_bias, A, D_skip, h0, hT, y, Bz, L, H, P, N, G, st);
  if (yt == SSS_F32)
    return mamba2_shape<__nv_bfloat16, float>(u, z, dt_raw, dt_bias, A, D_skip, h0, hT, y, Bz, L, H, P, N, G, st);
  return mamba2_shape<__nv_bfloat16, __nv_bfloat16>(u, z, dt_raw, dt_bias, A, D_skip, h0, hT, y, Bz, L, H, P, N, G, st);
}

}  // namespace sss
