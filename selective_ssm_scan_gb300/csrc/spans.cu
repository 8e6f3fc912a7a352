// Span-parallel forward: a long sequence cut into ns equal spans that run as
// separate rows of the chunked forward, their states joined by an associative
// scan.  "Understanding and Improving Length Generalization in Recurrent
// Models", section 2.5 Eq. (4): the state at the end of a span is the state
// reached from a zero start plus the inherited state decayed by the span's
// total decay, h_end = exp(sum of its l_t) h_in + h_end(zero start).  So the
// spans' (total decay, zero-start final state) pairs compose associatively,
//   (a1, s1) o (a2, s2) = (a1 a2, a2 s1 + s2),
// and one scan over them gives every span the state it starts from.
// Kernels here:
//  * span_prepare_kernel, two kinds of blocks in one launch:
//    - the conv state each span starts from (the K-1 inputs before it; span
//      0 takes the call's state) and the call's final conv state
//      F = u[L : L+K-1], the last K-1 inputs;
//    - partial sums of l_t = dt_t A_h over 64-token pieces of each span;
//  * span_combine_kernel: per state element, a Kogge-Stone scan over the
//    spans with warp shuffles (ns <= 32, fp32), giving every span its initial
//    state and the call its final state.
// The two passes of the chunked forward run from the API layer.
#include "common.cuh"

namespace sss {

namespace {
constexpr int kSpanThreads = 256;
constexpr int kDecayPiece = 64;  // tokens per partial decay sum
constexpr int kMaxKm = 7;        // K - 1 for K <= 8

struct SpanGeom {
  int Bz, ns, Ls, L, D, H, km;
  int prep_bx;   // blocks per (b, k) of conv-state work
  int dec_c;     // partial sums per span
  int dec_hg;    // 32-head groups
  __host__ __device__ int prep_blocks() const { return km > 0 ? Bz * ns * prep_bx : 0; }
  __host__ __device__ int dec_blocks() const { return Bz * ns * dec_c * dec_hg; }
};

// Conv-state blocks: one thread per (b, k, d) loads its K-1 values before it
// stores any.  The k = 0 thread reads S_in[b][d][*] and then writes
// F[b][d][*], so F may overwrite S_in in place.  Rows of s_span are b*ns + k.
// Decay blocks: lane = head within a group of 32, warp w sums tokens
// w, w+8, ... of one 64-token piece; the 8 warp sums are added in a fixed
// order, so the partial sums are deterministic.
__global__ void __launch_bounds__(kSpanThreads)
span_prepare_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* s_in,
                    __nv_bfloat16* s_out, __nv_bfloat16* __restrict__ s_span,
                    const __nv_bfloat16* __restrict__ dt, const float* __restrict__ A,
                    float* __restrict__ part, SpanGeom g) {
  int blk = blockIdx.x;
  if (blk < g.prep_blocks()) {
    const int bx = blk % g.prep_bx;
    const int row = blk / g.prep_bx;  // b * ns + k
    const int k = row % g.ns, b = row / g.ns;
    const int d = bx * kSpanThreads + threadIdx.x;
    if (d >= g.D) return;
    __nv_bfloat16 v[kMaxKm];
    const int64_t xrow = int64_t(b) * g.L + int64_t(k) * g.Ls - g.km;  // first input row
#pragma unroll
    for (int j = 0; j < kMaxKm; ++j)
      if (j < g.km)
        v[j] = k > 0  ? x[(xrow + j) * g.D + d]
               : s_in ? s_in[(int64_t(b) * g.D + d) * g.km + j]
                      : __float2bfloat16_rn(0.0f);
#pragma unroll
    for (int j = 0; j < kMaxKm; ++j)
      if (j < g.km) s_span[(int64_t(row) * g.D + d) * g.km + j] = v[j];
    if (k == 0 && s_out) {
      const int64_t frow = int64_t(b) * g.L + g.L - g.km;
#pragma unroll
      for (int j = 0; j < kMaxKm; ++j)
        if (j < g.km) v[j] = x[(frow + j) * g.D + d];
#pragma unroll
      for (int j = 0; j < kMaxKm; ++j)
        if (j < g.km) s_out[(int64_t(b) * g.D + d) * g.km + j] = v[j];
    }
    return;
  }
  blk -= g.prep_blocks();
  __shared__ float red[kSpanThreads / 32][32];
  const int hg = blk % g.dec_hg;
  const int c = (blk / g.dec_hg) % g.dec_c;
  const int row = blk / (g.dec_hg * g.dec_c);  // b * ns + k
  const int k = row % g.ns, b = row / g.ns;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int h = hg * 32 + lane;
  const int t0 = c * kDecayPiece, t1 = min(g.Ls, t0 + kDecayPiece);
  float s = 0.0f;
  if (h < g.H) {
    const float a = A[h];
    const int64_t base = int64_t(b) * g.L + int64_t(k) * g.Ls;
    float v[kDecayPiece / 8];
#pragma unroll
    for (int i = 0; i < kDecayPiece / 8; ++i) {
      const int t = t0 + w + 8 * i;
      v[i] = t < t1 ? __bfloat162float(dt[(base + t) * g.H + h]) : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < kDecayPiece / 8; ++i) s = fmaf(v[i], a, s);
  }
  red[w][lane] = s;
  __syncthreads();
  if (w == 0 && h < g.H) {
    float t = 0.0f;
#pragma unroll
    for (int i = 0; i < kSpanThreads / 32; ++i) t += red[i][lane];
    part[(int64_t(row) * g.dec_c + c) * g.H + h] = t;
  }
}

// Block (x, b * H + h) carries 4 * kCombineVec4 consecutive elements of the
// [P][N] state of (b, h).  Lane l of a warp holds span k = l / E of float4
// element group warp * E + l % E, E = 32 / ns, so the lanes of one span read
// E consecutive float4 (16 E contiguous bytes).  The block first turns the
// partial decay sums of (b, h) into the spans' decay factors exp(sum l_t).
constexpr int kCombineVec4 = 256;  // float4 groups per block

__global__ void __launch_bounds__(kSpanThreads)
span_combine_kernel(const float* __restrict__ part, const float* __restrict__ hloc,
                    const float* h0, float* __restrict__ h0_span, float* hT, int H, int PN,
                    int ns, int dec_c) {
  __shared__ float dec[32];
  dep_wait();  // the first pass's final states are complete and visible
  const int bh = blockIdx.y, b = bh / H, h = bh % H;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int k = w; k < ns; k += kSpanThreads / 32) {
    const float* p = part + (int64_t(b) * ns + k) * dec_c * H + h;
    float s = 0.0f;
    for (int c = lane; c < dec_c; c += 32) s += p[int64_t(c) * H];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) dec[k] = expf(s);
  }
  __syncthreads();
  const int E = 32 / ns;
  const int k = lane / E, eo = lane % E;
  const int nvec = PN / 4;
  const int64_t row0 = int64_t(b) * H + h;  // (b, h) in [Bz][H]
  const float4* hl4 = reinterpret_cast<const float4*>(hloc);
  const float4* h04 = reinterpret_cast<const float4*>(h0);
  float4* hs4 = reinterpret_cast<float4*>(h0_span);
  float4* hT4 = reinterpret_cast<float4*>(hT);
  const int warps = kSpanThreads / 32;
  const int v_begin = blockIdx.x * kCombineVec4;
  const int v_end = min(nvec, v_begin + kCombineVec4);
  for (int v0 = v_begin + w * E; v0 < v_end; v0 += warps * E) {
    const int v = v0 + eo;
    const bool live = k < ns && v < v_end;
    // span k's state of (b, h) is row (b * ns + k) * H + h of [Bz*ns][H]
    const int64_t srow = (int64_t(b) * ns + k) * H + h;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f), init = s;
    float a = 1.0f;
    if (live) {
      s = hl4[srow * nvec + v];
      a = dec[k];
      if (h0) init = h04[row0 * nvec + v];
    }
    __syncwarp();  // every lane's read of h0 is ordered before the write of hT
    // inclusive Kogge-Stone scan: afterwards (a, s) composes spans 0 .. k
    for (int dd = 1; dd < ns; dd <<= 1) {
      const float ap = __shfl_up_sync(0xffffffffu, a, dd * E);
      const float sx = __shfl_up_sync(0xffffffffu, s.x, dd * E);
      const float sy = __shfl_up_sync(0xffffffffu, s.y, dd * E);
      const float sz = __shfl_up_sync(0xffffffffu, s.z, dd * E);
      const float sw = __shfl_up_sync(0xffffffffu, s.w, dd * E);
      if (k >= dd) {  // (ap, sp) o (a, s) = (ap a, a sp + s)
        s = make_float4(fmaf(a, sx, s.x), fmaf(a, sy, s.y), fmaf(a, sz, s.z), fmaf(a, sw, s.w));
        a = ap * a;
      }
    }
    // exclusive prefix: the composition of spans 0 .. k-1 (identity for k = 0)
    float ae = __shfl_up_sync(0xffffffffu, a, E);
    float4 se;
    se.x = __shfl_up_sync(0xffffffffu, s.x, E);
    se.y = __shfl_up_sync(0xffffffffu, s.y, E);
    se.z = __shfl_up_sync(0xffffffffu, s.z, E);
    se.w = __shfl_up_sync(0xffffffffu, s.w, E);
    if (k == 0) {
      ae = 1.0f;
      se = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (live) {
      hs4[srow * nvec + v] = make_float4(fmaf(ae, init.x, se.x), fmaf(ae, init.y, se.y),
                                         fmaf(ae, init.z, se.z), fmaf(ae, init.w, se.w));
      if (hT && k == ns - 1)
        hT4[row0 * nvec + v] = make_float4(fmaf(a, init.x, s.x), fmaf(a, init.y, s.y),
                                           fmaf(a, init.z, s.z), fmaf(a, init.w, s.w));
    }
  }
}

SpanGeom geom(int64_t Bz, int64_t L, int64_t D, int H, int K, int ns) {
  SpanGeom g;
  g.Bz = int(Bz);
  g.ns = ns;
  g.L = int(L);
  g.Ls = int(L / ns);
  g.D = int(D);
  g.H = H;
  g.km = K - 1;
  g.prep_bx = int((D + kSpanThreads - 1) / kSpanThreads);
  g.dec_c = (g.Ls + kDecayPiece - 1) / kDecayPiece;
  g.dec_hg = (H + 31) / 32;
  return g;
}
}  // namespace

// Partial decay sums: [Bz*ns][ceil(Ls/64)][H] floats.
size_t span_part_floats(int64_t Bz, int64_t L, int H, int ns) {
  return size_t(Bz) * ns * ((L / ns + kDecayPiece - 1) / kDecayPiece) * H;
}

bool span_sizes_ok(int64_t Bz, int64_t L, int64_t D, int H, int P, int N, int K, int ns) {
  const int64_t blocks = Bz * ns * ((D + kSpanThreads - 1) / kSpanThreads) +
                         Bz * ns * ((L / ns + kDecayPiece - 1) / kDecayPiece) * ((H + 31) / 32);
  return ns >= 1 && ns <= 32 && K - 1 <= kMaxKm && L < (int64_t(1) << 31) &&
         D < (int64_t(1) << 31) && (int64_t(P) * N) % 4 == 0 &&
         int64_t(P) * N < (int64_t(1) << 31) && Bz * H <= 65535 && blocks < (int64_t(1) << 31);
}

// x, s_in, s_out, s_span and dt are bf16 (the caller checks the dtypes).
cudaError_t span_prepare_launch(const void* x, const void* s_in, void* s_out, void* s_span,
                                const void* dt, const float* A, float* part, int64_t Bz,
                                int64_t L, int64_t D, int H, int K, int ns, cudaStream_t st) {
  if (Bz == 0) return cudaSuccess;
  const SpanGeom g = geom(Bz, L, D, H, K, ns);
  const int blocks = g.prep_blocks() + g.dec_blocks();
  span_prepare_kernel<<<blocks, kSpanThreads, 0, st>>>(
      static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(s_in),
      static_cast<__nv_bfloat16*>(s_out), static_cast<__nv_bfloat16*>(s_span),
      static_cast<const __nv_bfloat16*>(dt), A, part, g);
  return cudaGetLastError();
}

cudaError_t span_combine_launch(const float* part, const float* hloc, const float* h0,
                                float* h0_span, float* hT, int64_t Bz, int64_t L, int H,
                                int64_t PN, int ns, cudaStream_t st) {
  if (Bz == 0) return cudaSuccess;
  const int dec_c = int((L / ns + kDecayPiece - 1) / kDecayPiece);
  const int nvec = int(PN / 4);
  const dim3 grid(unsigned((nvec + kCombineVec4 - 1) / kCombineVec4), unsigned(Bz * H));
  return launch_dep(span_combine_kernel, grid, dim3(kSpanThreads), 0, st, true, part, hloc, h0,
                    h0_span, hT, H, int(PN), ns, dec_c);
}

}  // namespace sss
