// Gradient of the scalar-decay selective scan with state (dx, ddt, dA, dB,
// dC and dh0 from dy and the final state's gradient dhT), for state-passing
// and truncated-backpropagation training: "Understanding and Improving
// Length Generalization in Recurrent Models" sections 4.4-4.5 (the final
// state of one segment starts the next; the gradient of that state is the
// next segment's dh0), with the recurrence of section 2 Eq. (1) and its
// initial-state form Eq. (4), and the causal-conv chapter's section on
// chunked training ("the state gradient of chunk B must flow into chunk A").
//
// Chunked form.  Cut the sequence into chunks of Q = 64 tokens; inside a
// chunk let Lam_t be the inclusive sum of l_s = dt_s A_h, M_ts = exp(Lam_t -
// Lam_s) [s <= t], G = C B^T and W = dY X^T (t x s), h_in the state entering
// the chunk and g_out = dL/dh at its end.  Then
//   y     = diag(e^Lam) C h_in^T + (G o M) X
//   h_out = e^{Lam_e} h_in + X^T diag(e^{Lam_e - Lam}) B
// and the chunk's gradients are
//   dX    = (G o M)^T dY + diag(e^{Lam_e - Lam}) B g_out^T
//   dB    = (W o M)^T C  + diag(e^{Lam_e - Lam}) X g_out
//   dC    = diag(e^Lam) dY h_in + (W o M) B
//   dh_in = e^{Lam_e} g_out + dY^T diag(e^Lam) C
//   dLam_t = dy_t . y_t - sum_t' (G o M o W)_{t' t}
//            - e^{Lam_e - Lam_t} x_t . (g_out B_t) + [t = e] <g_out, h_out>
//   dl_t  = sum_{t' >= t in the chunk} dLam_t',  ddt = dl A_h,  dA_h = sum dl dt.
// Every exponent above is <= 0, so no factor leaves the fp32 range.
//
// Kernels (fp32 CUDA-core arithmetic throughout):
//  1. chunk_states: per (batch, head) the states entering
//     every chunk, walking the chunks forward (workspace Hin, with the final
//     state after the last chunk);
//  2. chunk_grads:  the same rows walking backward, g_out of every chunk
//     (workspace Gout) and dh0;
//  3. chunk_bwd:    per (batch, head, chunk) everything else from the
//     formulas above, chunk tiles in shared memory; dB and dC per head to
//     the workspace;
//  4. reduce:       dB, dC summed over each group's heads, dA over batch and
//     chunks, in a fixed order (deterministic).
#include <algorithm>

#include "common.cuh"

namespace sss {

namespace {
constexpr int kQ = 64;          // chunk length
constexpr int kMaxP = 64;
constexpr int kMaxN = 128;
constexpr int kThreadsB = 256;
// padded leading dimensions of the shared tiles (odd: column walks spread
// over the banks)
constexpr int kLdP = kMaxP + 1;
constexpr int kLdN = kMaxN + 1;

template <typename T>
__device__ __forceinline__ float ldf(const T* p) {
  return to_f32<T>(*p);
}

// two fp32 FMAs in one instruction: d = a * b + c on packed pairs
__device__ __forceinline__ uint64_t pk2f(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk2f(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2f(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// for i < total: put(i, get(i)), eight independent loads in flight per
// thread before any store (a rolled loop of single loads waits one memory
// round trip per element)
template <typename Get, typename Put>
__device__ __forceinline__ void batched_copy(int total, Get get, Put put) {
  for (int base = threadIdx.x; base < total; base += kThreadsB * 8) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = base + u * kThreadsB;
      v[u] = i < total ? get(i) : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = base + u * kThreadsB;
      if (i < total) put(i, v[u]);
    }
  }
}

// inclusive prefix of l_s = dt_s A_h over the chunk's tokens (zeros past
// the chunk's end); warp 0, two tokens per lane
template <typename TA>
__device__ void chunk_lambda(const TA* __restrict__ dt, int64_t row0, int64_t stride, int Qc,
                             float Ah, float* lam, float* dts) {
  if (threadIdx.x < 32) {
    const int l = threadIdx.x;
    float v0 = 0.0f, v1 = 0.0f, d0 = 0.0f, d1 = 0.0f;
    if (2 * l < Qc) d0 = ldf(dt + (row0 + 2 * l) * stride);
    if (2 * l + 1 < Qc) d1 = ldf(dt + (row0 + 2 * l + 1) * stride);
    v0 = d0 * Ah;
    v1 = v0 + d1 * Ah;
    float s = v1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float u = __shfl_up_sync(0xffffffffu, s, o);
      if (l >= o) s += u;
    }
    const float before = s - v1;
    lam[2 * l] = before + v0;
    lam[2 * l + 1] = before + v1;
    dts[2 * l] = d0;
    dts[2 * l + 1] = d1;
  }
}

// ---- kernels 1 and 2: chunk-boundary states and state gradients -----------
// REV = false: h_in of every chunk (and h after the last) from h0, with
//   h <- e^{Lam_e} h + sum_s e^{Lam_e - Lam_s} x_s B_s^T.
// REV = true: g_out of every chunk from dhT, with
//   g <- e^{Lam_e} g + sum_t e^{Lam_t} dy_t C_t^T, and dh0 = g at the start.
// One CTA per (batch, head); thread (pq, nq) holds state rows 4 pq .. 4 pq + 3
// and columns nq + 16 j (j < 8), so one float4 of x and eight B values feed
// 32 FMAs per token.
// TRACE (forward only): chunks of Qlen <= kQ tokens, and instead of the
// states, the standard deviation over the head's P x N state elements after
// every chunk, to trace[b, c, h] (the state-scale diagnostic of "Understanding
// and Improving Length Generalization in Recurrent Models" section 3.5).
struct BoundSmem {
  float xs[kQ][kMaxP];
  float bs[kQ][kMaxN];
  float lam[kQ], dts[kQ], wgt[kQ];
  float red[kThreadsB / 32];
};

__device__ float block_sum_f(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.0f;
#pragma unroll
  for (int i = 0; i < kThreadsB / 32; ++i) t += red[i];
  return t;
}

template <bool REV, bool TRACE, typename TX, typename TA>
__global__ void __launch_bounds__(kThreadsB)
chunk_bound_kernel(const TX* __restrict__ x, const float* __restrict__ dy, const TA* __restrict__ dt,
                   const float* __restrict__ A, const TA* __restrict__ BC,
                   const float* __restrict__ init, float* __restrict__ bound,
                   float* __restrict__ final_out, int64_t L, int H, int P, int N, int G, int nC,
                   int Qlen) {
  extern __shared__ __align__(16) unsigned char smraw[];
  BoundSmem& sm = *reinterpret_cast<BoundSmem*>(smraw);
  const int tid = threadIdx.x;
  const int h = blockIdx.x, b = blockIdx.y;
  const int g = h / (H / G);
  const int pq = tid >> 4, nq = tid & 15;
  const float Ah = A[h];
  float st[4][kMaxN / 16];
  const int64_t soff = (int64_t(b) * H + h) * P * N;
  auto in = [&](int r, int j) { return 4 * pq + r < P && nq + 16 * j < N; };
  auto sidx = [&](int r, int j) { return int64_t(4 * pq + r) * N + nq + 16 * j; };
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int j = 0; j < kMaxN / 16; ++j) st[r][j] = (init && in(r, j)) ? init[soff + sidx(r, j)] : 0.0f;
  for (int k = 0; k < nC; ++k) {
    const int c = REV ? nC - 1 - k : k;
    const int64_t t0 = int64_t(c) * Qlen;
    const int Qc = L - t0 < Qlen ? int(L - t0) : Qlen;
    if (!TRACE) {  // the bound of chunk c before its update: h_in(c), or g_out(c)
      float* bc = bound + ((int64_t(b) * H + h) * (REV ? nC : nC + 1) + c) * P * N;
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int j = 0; j < kMaxN / 16; ++j)
          if (in(r, j)) bc[sidx(r, j)] = st[r][j];
    }
    __syncthreads();  // the previous chunk's tiles are no longer read
    chunk_lambda(dt + h, int64_t(b) * L + t0, H, Qc, Ah, sm.lam, sm.dts);
    batched_copy(
        kQ * kMaxP,
        [&](int i) {
          const int t = i / kMaxP, pp = i % kMaxP;
          if (t >= Qc || pp >= P) return 0.0f;
          const int64_t off = ((int64_t(b) * L + t0 + t) * H + h) * P + pp;
          return REV ? dy[off] : ldf(x + off);
        },
        [&](int i, float v) { sm.xs[i / kMaxP][i % kMaxP] = v; });
    batched_copy(
        kQ * kMaxN,
        [&](int i) {
          const int t = i / kMaxN, n = i % kMaxN;
          return (t < Qc && n < N) ? ldf(BC + ((int64_t(b) * L + t0 + t) * G + g) * N + n) : 0.0f;
        },
        [&](int i, float v) { sm.bs[i / kMaxN][i % kMaxN] = v; });
    __syncthreads();
    const float lam_e = sm.lam[Qc - 1];
    if (tid < kQ)
      sm.wgt[tid] = tid < Qc ? (REV ? expf(sm.lam[tid]) : expf(lam_e - sm.lam[tid])) : 0.0f;
    __syncthreads();
    const float dec = expf(lam_e);
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int j = 0; j < kMaxN / 16; ++j) st[r][j] *= dec;
    {
      // columns j and j + 1 of a row as one packed pair: two FMAs per instruction
      uint64_t st2[4][kMaxN / 32];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int j = 0; j < kMaxN / 32; ++j) st2[r][j] = pk2f(st[r][2 * j], st[r][2 * j + 1]);
      for (int t = 0; t < Qc; ++t) {
        const float w = sm.wgt[t];
        const float4 xv = *reinterpret_cast<const float4*>(&sm.xs[t][4 * pq]);
        const uint64_t wx[4] = {pk2f(w * xv.x, w * xv.x), pk2f(w * xv.y, w * xv.y),
                                pk2f(w * xv.z, w * xv.z), pk2f(w * xv.w, w * xv.w)};
#pragma unroll
        for (int j = 0; j < kMaxN / 32; ++j) {
          const uint64_t bv = pk2f(sm.bs[t][nq + 32 * j], sm.bs[t][nq + 32 * j + 16]);
#pragma unroll
          for (int r = 0; r < 4; ++r) st2[r][j] = fma2f(wx[r], bv, st2[r][j]);
        }
      }
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int j = 0; j < kMaxN / 32; ++j) upk2f(st2[r][j], st[r][2 * j], st[r][2 * j + 1]);
    }
    if (TRACE) {  // std of the state after this chunk: mean, then centred squares
      float s1 = 0.0f;
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int j = 0; j < kMaxN / 16; ++j) s1 += in(r, j) ? st[r][j] : 0.0f;
      const float mean = block_sum_f(s1, sm.red) / float(P * N);
      float s2 = 0.0f;
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int j = 0; j < kMaxN / 16; ++j) {
          const float d = in(r, j) ? st[r][j] - mean : 0.0f;
          s2 = fmaf(d, d, s2);
        }
      const float var = block_sum_f(s2, sm.red) / float(P * N);
      if (tid == 0) bound[(int64_t(b) * nC + c) * H + h] = sqrtf(var);
    }
  }
  if (TRACE) return;
  // the state after the last chunk, or dh0
  float* out = REV ? (final_out ? final_out + soff : nullptr)
                   : bound + ((int64_t(b) * H + h) * (nC + 1) + nC) * P * N;
  if (out) {
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int j = 0; j < kMaxN / 16; ++j)
        if (in(r, j)) out[sidx(r, j)] = st[r][j];
  }
}

// ---- kernel 3: the chunk's gradients ----------------------------------------
// out(i, j) = rs(i) * sum_k a1(i,k) b1(k,j) + sum_k a2(i,k) b2(k,j) for
// i < M, j < Nn, register tiles of 4 x TN per thread; epi(i, j, value).
struct Op {
  const float* a;
  int ai, ak;  // a(i,k) = a[i * ai + k * ak]
  const float* b;
  int bk, bj;  // b(k,j) = b[k * bk + j * bj]
  int K;
};
template <int TN, typename RS, typename Epi>
__device__ __forceinline__ void smem_mm(int M, int Nn, const Op& o1, RS rs, const Op& o2, Epi epi) {
  static_assert(TN % 2 == 0, "columns go in packed pairs");
  const int tn = (Nn + TN - 1) / TN, tm = (M + 3) / 4;
  for (int tile = threadIdx.x; tile < tm * tn; tile += kThreadsB) {
    const int i0 = 4 * (tile / tn), j0 = TN * (tile % tn);
    // columns q, q + 1 of a row as one packed pair: two FMAs per instruction
    uint64_t acc[4][TN / 2];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int q = 0; q < TN / 2; ++q) acc[r][q] = 0ull;
    auto run = [&](const Op& o) {
#pragma unroll 8
      for (int k = 0; k < o.K; ++k) {
        uint64_t av[4], bv[TN / 2];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float a = o.a[(i0 + r) * o.ai + k * o.ak];
          av[r] = pk2f(a, a);
        }
#pragma unroll
        for (int q = 0; q < TN / 2; ++q)
          bv[q] = pk2f(o.b[k * o.bk + (j0 + 2 * q) * o.bj], o.b[k * o.bk + (j0 + 2 * q + 1) * o.bj]);
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int q = 0; q < TN / 2; ++q) acc[r][q] = fma2f(av[r], bv[q], acc[r][q]);
      }
    };
    run(o1);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float sc = rs(i0 + r);
      const uint64_t s2 = pk2f(sc, sc);
#pragma unroll
      for (int q = 0; q < TN / 2; ++q) {
        uint64_t d;
        asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(acc[r][q]), "l"(s2));
        acc[r][q] = d;
      }
    }
    run(o2);
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int q = 0; q < TN / 2; ++q) {
        float lo, hi;
        upk2f(acc[r][q], lo, hi);
        if (i0 + r < M && j0 + 2 * q < Nn) epi(i0 + r, j0 + 2 * q, lo);
        if (i0 + r < M && j0 + 2 * q + 1 < Nn) epi(i0 + r, j0 + 2 * q + 1, hi);
      }
  }
}

struct ChunkSmem {
  float X[kQ][kLdP], DY[kQ][kLdP];
  float Bm[kQ][kLdN], Cm[kQ][kLdN];
  float Hin[kMaxP][kLdN], Go[kMaxP][kLdN];
  float Gm[kQ][kLdP], Wm[kQ][kLdP];  // [t][s]
  float S[kQ][kLdP];                  // scratch: y, then B g_out^T
  float lam[kQ], dts[kQ], el[kQ], ee[kQ];  // Lam, dt, e^Lam, e^{Lam_e - Lam}
  float At[kQ], Dt[kQ], Et[kQ], red[kThreadsB / 32];
};

template <typename TX, typename TA>
__global__ void __launch_bounds__(kThreadsB, 1)
chunk_bwd_kernel(const TX* __restrict__ x, const float* __restrict__ dy, const TA* __restrict__ dt,
                 const float* __restrict__ A, const TA* __restrict__ B, const TA* __restrict__ C,
                 const float* __restrict__ Hin_ws, const float* __restrict__ Gout_ws,
                 float* __restrict__ dx, float* __restrict__ ddt, float* __restrict__ dBp,
                 float* __restrict__ dCp, float* __restrict__ dAp, int64_t L, int H, int P,
                 int N, int G, int nC) {
  extern __shared__ __align__(16) unsigned char smraw[];
  ChunkSmem& s = *reinterpret_cast<ChunkSmem*>(smraw);
  const int tid = threadIdx.x;
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int g = h / (H / G);
  const int64_t t0 = int64_t(c) * kQ;
  const int Qc = L - t0 < kQ ? int(L - t0) : kQ;
  const float Ah = A[h];
  const int64_t hrow = (int64_t(b) * H + h);
  chunk_lambda(dt + h, int64_t(b) * L + t0, H, Qc, Ah, s.lam, s.dts);
  // chunk tiles (zero past the chunk's end and past P / N)
  auto xoff = [&](int i) { return ((int64_t(b) * L + t0 + i / kMaxP) * H + h) * P + i % kMaxP; };
  auto xin = [&](int i) { return i / kMaxP < Qc && i % kMaxP < P; };
  batched_copy(kQ * kMaxP, [&](int i) { return xin(i) ? ldf(x + xoff(i)) : 0.0f; },
               [&](int i, float v) { s.X[i / kMaxP][i % kMaxP] = v; });
  batched_copy(kQ * kMaxP, [&](int i) { return xin(i) ? dy[xoff(i)] : 0.0f; },
               [&](int i, float v) { s.DY[i / kMaxP][i % kMaxP] = v; });
  auto boff = [&](int i) { return ((int64_t(b) * L + t0 + i / kMaxN) * G + g) * N + i % kMaxN; };
  auto bin = [&](int i) { return i / kMaxN < Qc && i % kMaxN < N; };
  batched_copy(kQ * kMaxN, [&](int i) { return bin(i) ? ldf(B + boff(i)) : 0.0f; },
               [&](int i, float v) { s.Bm[i / kMaxN][i % kMaxN] = v; });
  batched_copy(kQ * kMaxN, [&](int i) { return bin(i) ? ldf(C + boff(i)) : 0.0f; },
               [&](int i, float v) { s.Cm[i / kMaxN][i % kMaxN] = v; });
  const float* hin = Hin_ws + (hrow * (nC + 1) + c) * P * N;
  const float* go = Gout_ws + (hrow * nC + c) * P * N;
  auto sin_ = [&](int i) { return i / kMaxN < P && i % kMaxN < N; };
  auto soff = [&](int i) { return int64_t(i / kMaxN) * N + i % kMaxN; };
  batched_copy(kMaxP * kMaxN, [&](int i) { return sin_(i) ? hin[soff(i)] : 0.0f; },
               [&](int i, float v) { s.Hin[i / kMaxN][i % kMaxN] = v; });
  batched_copy(kMaxP * kMaxN, [&](int i) { return sin_(i) ? go[soff(i)] : 0.0f; },
               [&](int i, float v) { s.Go[i / kMaxN][i % kMaxN] = v; });
  __syncthreads();
  const float lam_e = s.lam[Qc - 1];
  if (tid < kQ) {
    s.el[tid] = tid < Qc ? expf(s.lam[tid]) : 0.0f;
    s.ee[tid] = tid < Qc ? expf(lam_e - s.lam[tid]) : 0.0f;
  }
  __syncthreads();
  auto one = [](int) { return 1.0f; };
  const Op none{nullptr, 0, 0, nullptr, 0, 0, 0};
  // G o M and W (raw) ------------------------------------------------------
  smem_mm<4>(Qc, Qc, Op{&s.Cm[0][0], kLdN, 1, &s.Bm[0][0], 1, kLdN, N}, one, none,
             [&](int t, int sI, float v) {
               s.Gm[t][sI] = sI <= t ? v * expf(s.lam[t] - s.lam[sI]) : 0.0f;
             });
  smem_mm<4>(Qc, Qc, Op{&s.DY[0][0], kLdP, 1, &s.X[0][0], 1, kLdP, P}, one, none,
             [&](int t, int sI, float v) { s.Wm[t][sI] = v; });
  __syncthreads();
  // D_s = sum_t (G o M)_{ts} W_{ts}, then W <- W o M
  if (tid < Qc) {
    float d = 0.0f;
    for (int t = tid; t < Qc; ++t) d = fmaf(s.Gm[t][tid], s.Wm[t][tid], d);
    s.Dt[tid] = d;
  }
  __syncthreads();
  for (int i = tid; i < kQ * kQ; i += kThreadsB) {
    const int t = i / kQ, sI = i % kQ;
    s.Wm[t][sI] = (sI <= t && t < Qc) ? s.Wm[t][sI] * expf(s.lam[t] - s.lam[sI]) : 0.0f;
  }
  // y = diag(e^Lam) C h_in^T + (G o M) X, then A_t = dy_t . y_t
  smem_mm<4>(Qc, P, Op{&s.Cm[0][0], kLdN, 1, &s.Hin[0][0], 1, kLdN, N},
             [&](int t) { return s.el[t]; },
             Op{&s.Gm[0][0], kLdP, 1, &s.X[0][0], kLdP, 1, Qc},
             [&](int t, int p, float v) { s.S[t][p] = v; });
  __syncthreads();
  if (tid < Qc) {
    float a = 0.0f;
    for (int p = 0; p < P; ++p) a = fmaf(s.DY[tid][p], s.S[tid][p], a);
    s.At[tid] = a;
  }
  __syncthreads();
  // dC = diag(e^Lam) dY h_in + (W o M) B  (this head's share)
  float* dCrow = dCp + ((int64_t(b) * L + t0) * H + h) * N;
  smem_mm<8>(Qc, N, Op{&s.DY[0][0], kLdP, 1, &s.Hin[0][0], kLdN, 1, P},
             [&](int t) { return s.el[t]; },
             Op{&s.Wm[0][0], kLdP, 1, &s.Bm[0][0], kLdN, 1, Qc},
             [&](int t, int n, float v) { dCrow[int64_t(t) * H * N + n] = v; });
  // B g_out^T into the scratch, then E_s and dX
  smem_mm<4>(Qc, P, Op{&s.Bm[0][0], kLdN, 1, &s.Go[0][0], 1, kLdN, N}, one, none,
             [&](int sI, int p, float v) { s.S[sI][p] = v; });
  __syncthreads();
  if (tid < Qc) {
    float e = 0.0f;
    for (int p = 0; p < P; ++p) e = fmaf(s.X[tid][p], s.S[tid][p], e);
    s.Et[tid] = s.ee[tid] * e;
  }
  float* dxrow = dx + ((int64_t(b) * L + t0) * H + h) * P;
  smem_mm<4>(Qc, P, Op{&s.Gm[0][0], 1, kLdP, &s.DY[0][0], kLdP, 1, Qc}, one, none,
             [&](int sI, int p, float v) {
               dxrow[int64_t(sI) * H * P + p] = fmaf(s.ee[sI], s.S[sI][p], v);
             });
  // dB = diag(e^{Lam_e - Lam}) X g_out + (W o M)^T C  (this head's share)
  float* dBrow = dBp + ((int64_t(b) * L + t0) * H + h) * N;
  smem_mm<8>(Qc, N, Op{&s.X[0][0], kLdP, 1, &s.Go[0][0], kLdN, 1, P},
             [&](int sI) { return s.ee[sI]; },
             Op{&s.Wm[0][0], 1, kLdP, &s.Cm[0][0], kLdN, 1, Qc},
             [&](int sI, int n, float v) { dBrow[int64_t(sI) * H * N + n] = v; });
  // <g_out, h_out>, h_out = the next chunk's h_in (or the final state)
  const float* hout = Hin_ws + (hrow * (nC + 1) + c + 1) * P * N;
  float part = 0.0f;
  for (int i = tid; i < P * N; i += kThreadsB) part = fmaf(go[i], hout[i], part);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  if ((tid & 31) == 0) s.red[tid >> 5] = part;
  __syncthreads();
  // dLam, its reverse sum over the chunk (dl), ddt and the chunk's dA share
  if (tid < 32) {
    float gh = 0.0f;
#pragma unroll
    for (int w = 0; w < kThreadsB / 32; ++w) gh += s.red[w];
    const int l = tid;
    float v[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int t = kQ - 1 - (2 * l + e);  // lane 0 holds the chunk's last tokens
      float d = 0.0f;
      if (t < Qc) d = s.At[t] - s.Dt[t] - s.Et[t] + (t == Qc - 1 ? gh : 0.0f);
      v[e] = d;
    }
    // inclusive scan over the reversed order = sum over t' >= t
    const float pair = v[0] + v[1];
    float sc = pair;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float u = __shfl_up_sync(0xffffffffu, sc, o);
      if (l >= o) sc += u;
    }
    const float before = sc - pair;
    float dA_acc = 0.0f;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int t = kQ - 1 - (2 * l + e);
      const float dl = before + (e == 0 ? v[0] : v[0] + v[1]);
      if (t < Qc) {
        ddt[(int64_t(b) * L + t0 + t) * H + h] = dl * Ah;
        dA_acc = fmaf(dl, s.dts[t], dA_acc);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dA_acc += __shfl_xor_sync(0xffffffffu, dA_acc, o);
    if (l == 0) dAp[hrow * nC + c] = dA_acc;
  }
}

// ---- kernel 4: group sums of dB and dC, dA over batch and chunks -----------
__global__ void __launch_bounds__(kThreadsB)
scan_bwd_reduce_kernel(const float* __restrict__ dBp, const float* __restrict__ dCp,
                       const float* __restrict__ dAp, float* __restrict__ dB,
                       float* __restrict__ dC, float* __restrict__ dA, int64_t rows, int H,
                       int N, int G, int64_t Bz, int nC) {
  const int hpg = H / G;
  const int64_t total = rows * G * N;
  for (int64_t i = blockIdx.x * int64_t(kThreadsB) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * kThreadsB) {
    const int n = int(i % N);
    const int g = int((i / N) % G);
    const int64_t r = i / (int64_t(N) * G);
    float sb = 0.0f, sc = 0.0f;
    for (int k = 0; k < hpg; ++k) {
      const int64_t off = (r * H + g * hpg + k) * N + n;
      sb += dBp[off];
      sc += dCp[off];
    }
    dB[i] = sb;
    dC[i] = sc;
  }
  if (blockIdx.x == 0) {
    for (int h = threadIdx.x; h < H; h += kThreadsB) {
      float a = 0.0f;
      for (int64_t b = 0; b < Bz; ++b)
        for (int c = 0; c < nC; ++c) a += dAp[(b * H + h) * nC + c];
      dA[h] = a;
    }
  }
}

struct WsLayout {
  size_t hin, gout, dbp, dcp, dap, total;
};
WsLayout ws_layout(int64_t Bz, int64_t L, int H, int P, int N) {
  const int64_t nC = (L + kQ - 1) / kQ;
  auto al = [](size_t v) { return (v + 255) & ~size_t(255); };
  WsLayout w;
  w.hin = 0;
  w.gout = w.hin + al(sizeof(float) * size_t(Bz * H * (nC + 1) * P * N));
  w.dbp = w.gout + al(sizeof(float) * size_t(Bz * H * nC * P * N));
  w.dcp = w.dbp + al(sizeof(float) * size_t(Bz * L * H * N));
  w.dap = w.dcp + al(sizeof(float) * size_t(Bz * L * H * N));
  w.total = w.dap + al(sizeof(float) * size_t(Bz * H * (nC > 0 ? nC : 1)));
  return w;
}

template <typename TX, typename TA>
cudaError_t launch_bwd(const void* x, const void* dt, const float* A, const void* B, const void* C,
                       const float* h0, const float* dy, const float* dhT, float* dx, float* ddt,
                       float* dA, float* dB, float* dC, float* dh0, int64_t Bz, int64_t L, int H,
                       int P, int N, int G, void* ws, cudaStream_t st) {
  const int nC = int((L + kQ - 1) / kQ);
  const WsLayout w = ws_layout(Bz, L, H, P, N);
  unsigned char* base = static_cast<unsigned char*>(ws);
  float* hin = reinterpret_cast<float*>(base + w.hin);
  float* gout = reinterpret_cast<float*>(base + w.gout);
  float* dbp = reinterpret_cast<float*>(base + w.dbp);
  float* dcp = reinterpret_cast<float*>(base + w.dcp);
  float* dap = reinterpret_cast<float*>(base + w.dap);
  const TX* xx = static_cast<const TX*>(x);
  const TA* dtt = static_cast<const TA*>(dt);
  const TA* Bb = static_cast<const TA*>(B);
  const TA* Cc = static_cast<const TA*>(C);
  const dim3 gb(H, unsigned(Bz));
  if (Bz > 0) {
    const int bsm = int(sizeof(BoundSmem));
    auto k1 = chunk_bound_kernel<false, false, TX, TA>;
    auto k2 = chunk_bound_kernel<true, false, TX, TA>;
    cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, bsm);
    cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, bsm);
    k1<<<gb, kThreadsB, bsm, st>>>(xx, dy, dtt, A, Bb, h0, hin, nullptr, L, H, P, N, G, nC, kQ);
    k2<<<gb, kThreadsB, bsm, st>>>(xx, dy, dtt, A, Cc, dhT, gout, dh0, L, H, P, N, G, nC, kQ);
  }
  if (nC > 0 && Bz > 0) {
    auto k3 = chunk_bwd_kernel<TX, TA>;
    const int smem = int(sizeof(ChunkSmem));
    cudaFuncSetAttribute(k3, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    k3<<<dim3(nC, H, unsigned(Bz)), kThreadsB, smem, st>>>(xx, dy, dtt, A, Bb, Cc, hin, gout, dx,
                                                           ddt, dbp, dcp, dap, L, H, P, N, G, nC);
  }
  const int64_t rows = Bz * L;
  const int64_t total = rows * G * N;
  const int blocks = int(std::max<int64_t>(1, std::min<int64_t>((total + kThreadsB - 1) / kThreadsB, 4096)));
  scan_bwd_reduce_kernel<<<blocks, kThreadsB, 0, st>>>(dbp, dcp, dap, dB, dC, dA, rows, H, N, G,
                                                       Bz, nC);
  return cudaGetLastError();
}
}  // namespace

size_t ssm_scan_bwd_workspace(int64_t Bz, int64_t L, int H, int P, int N) {
  return ws_layout(Bz, L, H, P, N).total;
}

cudaError_t ssm_scan_bwd_launch(const void* x, sss_dtype x_t, const void* dt, const float* A,
                                const void* B, const void* C, sss_dtype act_t, const float* h0,
                                const float* dy, const float* dhT, float* dx, float* ddt,
                                float* dA, float* dB, float* dC, float* dh0, int64_t Bz, int64_t L,
                                int H, int P, int N, int G, void* ws, cudaStream_t st) {
  if (x_t == SSS_BF16 && act_t == SSS_BF16)
    return launch_bwd<__nv_bfloat16, __nv_bfloat16>(x, dt, A, B, C, h0, dy, dhT, dx, ddt, dA, dB,
                                                    dC, dh0, Bz, L, H, P, N, G, ws, st);
  if (x_t == SSS_F32 && act_t == SSS_BF16)
    return launch_bwd<float, __nv_bfloat16>(x, dt, A, B, C, h0, dy, dhT, dx, ddt, dA, dB, dC, dh0,
                                            Bz, L, H, P, N, G, ws, st);
  if (x_t == SSS_BF16 && act_t == SSS_F32)
    return launch_bwd<__nv_bfloat16, float>(x, dt, A, B, C, h0, dy, dhT, dx, ddt, dA, dB, dC, dh0,
                                            Bz, L, H, P, N, G, ws, st);
  return launch_bwd<float, float>(x, dt, A, B, C, h0, dy, dhT, dx, ddt, dA, dB, dC, dh0, Bz, L, H,
                                  P, N, G, ws, st);
}

bool ssm_scan_bwd_supports(int P, int N) { return P >= 1 && P <= kMaxP && N >= 1 && N <= kMaxN; }

namespace {
template <typename TX, typename TA>
cudaError_t launch_trace(const void* x, const void* dt, const float* A, const void* B,
                         const float* h0, float* out, int64_t Bz, int64_t L, int H, int P, int N,
                         int G, int stride, cudaStream_t st) {
  const int nC = int((L + stride - 1) / stride);
  if (Bz == 0 || nC == 0) return cudaSuccess;
  const int bsm = int(sizeof(BoundSmem));
  auto k = chunk_bound_kernel<false, true, TX, TA>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bsm);
  k<<<dim3(H, unsigned(Bz)), kThreadsB, bsm, st>>>(
      static_cast<const TX*>(x), nullptr, static_cast<const TA*>(dt), A, static_cast<const TA*>(B),
      h0, out, nullptr, L, H, P, N, G, nC, stride);
  return cudaGetLastError();
}
}  // namespace

int state_trace_max_stride() { return kQ; }

cudaError_t state_std_trace_launch(const void* x, sss_dtype x_t, const void* dt, const float* A,
                                   const void* B, sss_dtype act_t, const float* h0, float* out,
                                   int64_t Bz, int64_t L, int H, int P, int N, int G, int stride,
                                   cudaStream_t st) {
  if (x_t == SSS_BF16 && act_t == SSS_BF16)
    return launch_trace<__nv_bfloat16, __nv_bfloat16>(x, dt, A, B, h0, out, Bz, L, H, P, N, G,
                                                      stride, st);
  if (x_t == SSS_F32 && act_t == SSS_BF16)
    return launch_trace<float, __nv_bfloat16>(x, dt, A, B, h0, out, Bz, L, H, P, N, G, stride, st);
  if (x_t == SSS_BF16 && act_t == SSS_F32)
    return launch_trace<__nv_bfloat16, float>(x, dt, A, B, h0, out, Bz, L, H, P, N, G, stride, st);
  return launch_trace<float, float>(x, dt, A, B, h0, out, Bz, L, H, P, N, G, stride, st);
}

}  // namespace sss
