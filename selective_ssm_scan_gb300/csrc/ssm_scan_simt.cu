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

// ---------------------------------------------------------------------------
// The same scan, register-tiled for P a multiple of 16 and N in {32, 64, 128}.
// Lanes form groups of Q; a group owns R rows p and all N state columns, lane
// q of the group holding n = 4 q + 4 Q k + e (k < N / (4 Q), e < 4) of each
// of its R rows, so each float4 read of a staged B or C row fetches Q
// consecutive 16-byte pieces (conflict-free).  NW warps per CTA cover
// (32 / Q) R NW rows of one (sequence, head).  Chunks of 32 tokens are
// staged in shared memory by cp.async, two chunks deep: B, C, the CTA's x
// rows of u and the z rows arrive while the previous chunk runs, and warp 0
// loads the next chunk's dt_raw the same way (one token per lane).  Per chunk
// warp 0 forms dt, the log decays and their prefix; the CTA forms the input
// coefficients cf_t = x_t dt_t / Lam_t; then every lane runs the chunk's
// tokens from registers.
//
// Scaled form: with Lam_t = exp(sum of dt A over the chunk up to t) and the
// chunk-start state as reference, hs = h / Lam obeys hs_t = hs_{t-1} +
// cf_t B_t^T and y_t = Lam_t (hs_t C_t) + D x_t: one FMA per state element
// for the update and one for the output.  At the chunk end h = Lam_end hs.
// A chunk whose log-decay range passes kM2Range (|sum| > 60, factors beyond
// e^60) runs the direct form h = a h + dt x B^T instead.  The lanes' partial
// outputs of the R rows are summed over the group by a transposing butterfly
// (each step hands half of the rows still held to the partner), and the
// chunk's sums go through shared memory, where the gate applies Lam_t, the D
// skip and SiLU(z) and writes whole y rows.
// ---------------------------------------------------------------------------
namespace {
constexpr int kM2Tch = 32;         // tokens per staged chunk (one per lane of warp 0)
constexpr float kM2Range = 60.0f;  // largest |log-decay| a chunk spans in the scaled form

template <typename TA, int NW, int N, int Q, int R>
struct M2Layout {
  static constexpr int M = N / Q;                // state columns per lane
  static constexpr int PB = (32 / Q) * R * NW;   // rows p of the CTA
  static_assert(M % 4 == 0 && R <= Q && R % 4 == 0, "lane tile");
  // per stage: B, C [chunk][N], x [chunk][PB] (fp32), z [chunk][PB] (TA)
  static constexpr size_t kB = 0;
  static constexpr size_t kC = kB + sizeof(float) * kM2Tch * N;
  static constexpr size_t kX = kC + sizeof(float) * kM2Tch * N;
  static constexpr size_t kZ = kX + sizeof(float) * kM2Tch * PB;
  static constexpr size_t kStage = kZ + ((sizeof(TA) * kM2Tch * PB + 15) / 16) * 16;
  static constexpr size_t kCf = 2 * kStage;                        // cf [chunk][PB]
  static constexpr size_t kY = kCf + sizeof(float) * kM2Tch * PB;  // sums [chunk][PB]
  static constexpr size_t kRl = kY + sizeof(float) * kM2Tch * PB;
  static constexpr size_t kLm = kRl + sizeof(float) * kM2Tch;
  static constexpr size_t kBytes = kLm + sizeof(float) * kM2Tch;
};

__device__ __forceinline__ void cp16(void* dst, const void* src, bool full) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src),
               "r"(full ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// The row a lane ends the butterfly with: the levels with offsets Q/2 .. 1
// first halve the R rows (log2 R levels), and bit `off` of the lane's group
// index picks the upper half at each of them.  Register slot s of a lane holds
// row s ^ m2rt_row(qi), so that at every level the half a lane keeps is in
// slots [0, cnt) and the half it hands over in [cnt, 2 cnt).
template <int Q, int R>
__device__ __forceinline__ int m2rt_row(int qi) {
  int row = 0, cnt = R;
#pragma unroll
  for (int off = Q / 2; off >= 1; off >>= 1)
    if (cnt > 1) {
      cnt >>= 1;
      if (qi & off) row += cnt;
    }
  return row;
}

template <bool DIRECT, int N, int Q, int R, int PB>
__device__ __forceinline__ void m2rt_tokens(float (&st)[R][N / Q], const float* bs,
                                            const float* cs, const float* cf, float* ys,
                                            const float* lm, int nt, int pl0, int qi) {
  constexpr int M = N / Q;
  const int row = m2rt_row<Q, R>(qi);
  int wmask = 0;  // the levels past the halving add; their lanes hold copies
  {
    int cnt = R;
#pragma unroll
    for (int off = Q / 2; off >= 1; off >>= 1) {
      if (cnt > 1)
        cnt >>= 1;
      else
        wmask |= off;
    }
  }
#pragma unroll 2
  for (int tt = 0; tt < nt; ++tt) {
    float cv8[R];
#pragma unroll
    for (int r = 0; r < R; ++r) cv8[r] = cf[tt * PB + pl0 + (r ^ row)];
    const float m = DIRECT ? lm[tt] : 1.0f;
    float a[R];
#pragma unroll
    for (int r = 0; r < R; ++r) a[r] = 0.0f;
#pragma unroll
    for (int k = 0; k < M / 4; ++k) {
      const float4 b4 = *reinterpret_cast<const float4*>(bs + tt * N + 4 * qi + 4 * Q * k);
      const float4 c4 = *reinterpret_cast<const float4*>(cs + tt * N + 4 * qi + 4 * Q * k);
      const float bv[4] = {b4.x, b4.y, b4.z, b4.w};
      const float cv[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int r = 0; r < R; ++r) {
          float& s = st[r][4 * k + e];
          s = DIRECT ? fmaf(cv8[r], bv[e], m * s) : fmaf(cv8[r], bv[e], s);
          a[r] = fmaf(cv[e], s, a[r]);
        }
    }
    int cnt = R;
#pragma unroll
    for (int off = Q / 2; off >= 1; off >>= 1) {
      if (cnt > 1) {
        cnt >>= 1;
#pragma unroll
        for (int i = 0; i < R / 2; ++i)
          if (i < cnt) a[i] += __shfl_xor_sync(0xffffffffu, a[cnt + i], off);
      } else {
        a[0] += __shfl_xor_sync(0xffffffffu, a[0], off);
      }
    }
    if ((qi & wmask) == 0) ys[tt * PB + pl0 + row] = a[0];
  }
}
}  // namespace

template <typename TA, typename TY, int NW, int N, int Q, int R>
__global__ void __launch_bounds__(NW * 32)
mamba2_scan_rt_kernel(const float* __restrict__ u, const TA* __restrict__ z,
                      const TA* __restrict__ dt_raw, const float* __restrict__ dt_bias,
                      const float* __restrict__ A, const float* __restrict__ D_skip,
                      const float* h0, float* hT, TY* __restrict__ y, int64_t L, int H, int P,
                      int G) {
  using Lay = M2Layout<TA, NW, N, Q, R>;
  constexpr int M = Lay::M, PB = Lay::PB;
  constexpr int ZV = int(16 / sizeof(TA));  // z elements per 16-byte copy
  extern __shared__ __align__(16) uint8_t m2s[];
  float* cf = reinterpret_cast<float*>(m2s + Lay::kCf);
  float* ys = reinterpret_cast<float*>(m2s + Lay::kY);
  float* rl = reinterpret_cast<float*>(m2s + Lay::kRl);  // dt / Lam (scaled) or dt (direct)
  float* lm = reinterpret_cast<float*>(m2s + Lay::kLm);  // Lam (scaled) or a (direct)
  __shared__ int direct_s;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qi = lane % Q;
  const int b = int(blockIdx.x / unsigned(H)), h = int(blockIdx.x % unsigned(H));
  const int g = h / (H / G);
  const int p0 = int(blockIdx.y) * PB;
  const int pl0 = (warp * (32 / Q) + lane / Q) * R;  // this group's first row, CTA-local
  const int prow = m2rt_row<Q, R>(qi);  // register slot r holds row pl0 + (r ^ prow)
  const float Ah = A[h];
  const float bias_h = dt_bias ? dt_bias[h] : 0.0f;
  const float Dh = D_skip ? D_skip[h] : 0.0f;
  const int64_t Dx = int64_t(H) * P, Dt = Dx + 2 * int64_t(G) * N;
  const int64_t nch = (L + kM2Tch - 1) / kM2Tch;

  // stage chunk c into buffer c & 1 (rows past the end are zero-filled)
  auto stage = [&](int64_t c) {
    uint8_t* sb = m2s + (c & 1) * Lay::kStage;
    const int64_t t0 = c * kM2Tch;
    const int nt = int((L - t0) < kM2Tch ? (L - t0) : kM2Tch);
    const float* ub = u + (int64_t(b) * L + t0) * Dt;
    for (int i = tid; i < kM2Tch * (N / 4); i += NW * 32) {
      const int tt = i / (N / 4), q = i % (N / 4);
      const float* row = ub + int64_t(tt < nt ? tt : 0) * Dt + Dx + int64_t(g) * N + 4 * q;
      cp16(sb + Lay::kB + 16 * i, row, tt < nt);
      cp16(sb + Lay::kC + 16 * i, row + int64_t(G) * N, tt < nt);
    }
    for (int i = tid; i < kM2Tch * (PB / 4); i += NW * 32) {
      const int tt = i / (PB / 4), q = i % (PB / 4);
      cp16(sb + Lay::kX + 16 * i, ub + int64_t(tt < nt ? tt : 0) * Dt + int64_t(h) * P + p0 + 4 * q,
           tt < nt);
    }
    if (z) {
      const TA* zb = z + (int64_t(b) * L + t0) * Dx + int64_t(h) * P + p0;
      for (int i = tid; i < kM2Tch * (PB / ZV); i += NW * 32) {
        const int tt = i / (PB / ZV), q = i % (PB / ZV);
        cp16(sb + Lay::kZ + 16 * i, zb + int64_t(tt < nt ? tt : 0) * Dx + ZV * q, tt < nt);
      }
    }
  };
  auto load_dt = [&](int64_t c) -> float {  // warp 0: dt_raw of token lane of chunk c
    const int64_t t = c * kM2Tch + lane;
    return (c < nch && t < L) ? to_f32(dt_raw[(int64_t(b) * L + t) * H + h]) : 0.0f;
  };

  float st[R][M];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int i = 0; i < M; ++i) {
      const int n = 4 * qi + 4 * Q * (i >> 2) + (i & 3);
      st[r][i] = h0 ? h0[((int64_t(b) * H + h) * P + p0 + pl0 + (r ^ prow)) * N + n] : 0.0f;
    }

  stage(0);
  cp_commit();
  float dt_cur = warp == 0 ? load_dt(0) : 0.0f;
  for (int64_t c = 0; c < nch; ++c) {
    const int64_t t0 = c * kM2Tch;
    const int nt = int((L - t0) < kM2Tch ? (L - t0) : kM2Tch);
    if (c + 1 < nch) stage(c + 1);
    cp_commit();  // possibly empty: one group per chunk keeps the count
    if (warp == 0) {
      const float dt_next = load_dt(c + 1);
      float dtv = 0.0f, lav = 0.0f;  // tokens past the end add no decay
      if (lane < nt) {
        dtv = softplusf(dt_cur + bias_h);
        lav = dtv * Ah;
      }
      float cum = lav;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float v = __shfl_up_sync(0xffffffffu, cum, o);
        if (lane >= o) cum += v;
      }
      // dt A has the sign of A_h in every token: the chunk's largest |prefix| is its total
      const float total = __shfl_sync(0xffffffffu, cum, 31);
      const bool direct = !(fabsf(total) <= kM2Range);
      rl[lane] = direct ? dtv : dtv * expf(-cum);
      lm[lane] = direct ? expf(lav) : expf(cum);
      if (lane == 0) direct_s = direct ? 1 : 0;
      dt_cur = dt_next;
    }
    cp_wait1();  // this thread's copies of chunk c have landed
    __syncthreads();
    const uint8_t* sb = m2s + (c & 1) * Lay::kStage;
    const float* xs = reinterpret_cast<const float*>(sb + Lay::kX);
    for (int i = tid; i < kM2Tch * PB; i += NW * 32) cf[i] = xs[i] * rl[i / PB];
    const bool direct = direct_s != 0;
    __syncthreads();
    const float* bs = reinterpret_cast<const float*>(sb + Lay::kB);
    const float* cs = reinterpret_cast<const float*>(sb + Lay::kC);
    if (direct) {
      m2rt_tokens<true, N, Q, R, PB>(st, bs, cs, cf, ys, lm, nt, pl0, qi);
    } else {
      m2rt_tokens<false, N, Q, R, PB>(st, bs, cs, cf, ys, lm, nt, pl0, qi);
      const float m = lm[nt - 1];
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int i = 0; i < M; ++i) st[r][i] *= m;
    }
    __syncthreads();
    // the gate over whole rows: y = (Lam hs C + D x) SiLU(z)
    const TA* zs = reinterpret_cast<const TA*>(sb + Lay::kZ);
    for (int i = tid; i < nt * (PB / 4); i += NW * 32) {
      const int tt = i / (PB / 4), q = i % (PB / 4);
      const float4 v4 = reinterpret_cast<const float4*>(ys)[i];
      const float4 x4 = reinterpret_cast<const float4*>(xs)[i];
      const float m = direct ? 1.0f : lm[tt];
      float v[4] = {fmaf(m, v4.x, Dh * x4.x), fmaf(m, v4.y, Dh * x4.y), fmaf(m, v4.z, Dh * x4.z),
                    fmaf(m, v4.w, Dh * x4.w)};
      if (z) {
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] *= silu(to_f32(zs[tt * PB + 4 * q + e]));
      }
      st_vec<TY, 4>(y + ((int64_t(b) * L + t0 + tt) * H + h) * P + p0 + 4 * q, v);
    }
    __syncthreads();  // buffer c & 1, cf and the sums are free for the next chunks
  }

  if (hT) {
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int i = 0; i < M; ++i) {
        const int n = 4 * qi + 4 * Q * (i >> 2) + (i & 3);
        hT[((int64_t(b) * H + h) * P + p0 + pl0 + (r ^ prow)) * N + n] = st[r][i];
      }
  }
}

template <typename TA, typename TY, int NW, int N, int Q, int R>
static cudaError_t launch_mamba2_rt(const float* u, const void* z, const void* dt_raw,
                                    const float* dt_bias, const float* A, const float* D_skip,
                                    const float* h0, float* hT, void* y, int64_t Bz, int64_t L,
                                    int H, int P, int G, cudaStream_t st) {
  using Lay = M2Layout<TA, NW, N, Q, R>;
  if (P % Lay::PB) return cudaErrorNotSupported;
  auto kern = mamba2_scan_rt_kernel<TA, TY, NW, N, Q, R>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(Lay::kBytes));
  if (e != cudaSuccess) return e;
  kern<<<dim3(unsigned(Bz * H), unsigned(P / Lay::PB)), NW * 32, Lay::kBytes, st>>>(
      u, static_cast<const TA*>(z), static_cast<const TA*>(dt_raw), dt_bias, A, D_skip, h0, hT,
      static_cast<TY*>(y), L, H, P, G);
  return cudaGetLastError();
}

// The register-tiled kernel when the shape and the pointers allow it: P a
// multiple of 16, N in {32, 64, 128}, u and z 16-byte aligned (the row
// strides H P + 2 G N floats and H P elements then keep every 16-byte copy
// aligned), y aligned for 4-element stores.  Returns cudaErrorNotSupported
// otherwise.
template <typename TA, typename TY>
static cudaError_t mamba2_rt(const float* u, const void* z, const void* dt_raw,
                             const float* dt_bias, const float* A, const float* D_skip,
                             const float* h0, float* hT, void* y, int64_t Bz, int64_t L, int H,
                             int P, int N, int G, cudaStream_t st) {
  if (P % 16 || (N != 32 && N != 64 && N != 128) || Bz * H > 0x7fffffffLL || P / 16 > 65535 ||
      reinterpret_cast<uintptr_t>(u) % 16 || reinterpret_cast<uintptr_t>(z) % 16 ||
      reinterpret_cast<uintptr_t>(y) % (4 * sizeof(TY)))
    return cudaErrorNotSupported;
#define SSS_M2RT(NW, NN, Q, R)                                                               \
  if (N == NN) {                                                                             \
    const cudaError_t e = launch_mamba2_rt<TA, TY, NW, NN, Q, R>(u, z, dt_raw, dt_bias, A,     \
                                                                D_skip, h0, hT, y, Bz, L, H, \
                                                                P, G, st);                   \
    if (e != cudaErrorNotSupported) return e;                                                \
  }
  // the widest CTA whose rows divide P
  SSS_M2RT(4, 128, 16, 8)
  SSS_M2RT(2, 128, 16, 8)
  SSS_M2RT(1, 128, 16, 8)
  SSS_M2RT(2, 64, 8, 8)
  SSS_M2RT(1, 64, 8, 8)
  SSS_M2RT(1, 64, 8, 4)
  SSS_M2RT(4, 32, 8, 4)
  SSS_M2RT(2, 32, 8, 4)
  SSS_M2RT(1, 32, 8, 4)
  return cudaErrorNotSupported;
#undef SSS_M2RT
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
  {
    const cudaError_t e = mamba2_rt<TA, TY>(u, z, dt_raw, dt_bias, A, D_skip, h0, hT, y, Bz, L, H,
                                            P, N, G, st);
    if (e != cudaErrorNotSupported) return e;
  }
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
