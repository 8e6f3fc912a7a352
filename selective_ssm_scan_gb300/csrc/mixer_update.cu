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
#include "tc_ptx.cuh"

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
  // no lengths: the non-circular mode, whose newest S_len inputs sit in
  // slots 0 .. S_len-1 oldest first (the history reads as if p = S_len)
  const int64_t p0 = seqlens ? int64_t(seqlens[b]) : int64_t(S_len);

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
    // store the inputs (not the outputs), after all reads of this channel's
    // row: at the write pointer in token order, or (non-circular) by dropping
    // the oldest L_new entries and appending the new inputs (ascending j
    // reads slot j + L_new before it is written)
    if (seqlens) {
      for (int i = 0; i < L_new; ++i)
        row[pos_mod(p0 + i, S_len)] = x[(int64_t(b) * L_new + i) * D + d];
    } else {
      for (int j = 0; j < S_len; ++j)
        row[j] = j + L_new < S_len ? row[j + L_new]
                                   : x[(int64_t(b) * L_new + j + L_new - S_len) * D + d];
    }
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

// ---------------------------------------------------------------------------
// Pipelined variant (N = 128): the state of one (request, head) is a
// contiguous P*N*4-byte block of the pool, so it streams into shared memory
// as one bulk copy.
//
//  * persistent grid, one CTA per SM, each CTA owns a contiguous range of
//    (request, head) items;
//  * warp 8 is the producer: for item k it bulk-copies into ring stage
//    k mod S the state block, the head's conv-slot tile [P][S_len] (also
//    contiguous), the head's weights and bias, and per token the x row of the
//    head and the B and C rows of its group, and publishes the item's pool
//    row, length and decays exp(dt A_h) (gathered one group of 32 items
//    ahead, so the producer never waits on them).  When the compute warps
//    release stage k mod S it refills it with item k + S: S stages of ~34 KB
//    keep ~140 KB of loads per SM in flight;
//  * warps 0-7 compute: the conv of the head's P channels from the slot tile
//    (every read before the slot writes, as in the kernel above; the new
//    inputs go straight to the pool row), then the recurrence, warp w on
//    rows p = w + 8 r and lane l on the float4 column group l; the updated
//    state goes back to the pool from registers as coalesced 16-byte stores
//    and y is a warp reduce-scatter;
//  * every wait is bounded: on expiry SSS_ERR_TIMEOUT is raised, the compute
//    warps stop, and the producer waits (bounded) for its copies in flight
//    before the CTA exits.
constexpr int kPipeWarps = 8;
constexpr int kPipeThreads = (kPipeWarps + 1) * 32;
constexpr int kPipeMaxStages = 6;
constexpr int kPipeMaxLnew = 8;
constexpr int kPipeN = 128;
constexpr int kPipeMaxP = 128;
constexpr uint32_t kPipeRingBudget = 200u * 1024u;
constexpr uint64_t kPipeWaitNs = 2000000000ull;

struct PipeGeom {
  // byte offsets inside one stage, and the stage size
  uint32_t st, cv, xs, bs, cs, ws, bi, stage;
  // bytes of the state block, slot tile, one x row, one B/C row, weights, bias
  uint32_t n_st, n_cv, n_x, n_bc, n_ws, n_bi;
};

__host__ __device__ inline uint32_t pipe_up16(uint32_t v) { return (v + 15u) & ~15u; }

__host__ inline PipeGeom pipe_geom(int P, int S_len, int L_new, int K, int esz, bool has_bias) {
  PipeGeom g;
  g.n_st = uint32_t(P) * kPipeN * 4u;
  g.n_cv = uint32_t(P) * uint32_t(S_len) * uint32_t(esz);
  g.n_x = uint32_t(P) * uint32_t(esz);
  g.n_bc = uint32_t(kPipeN) * uint32_t(esz);
  g.n_ws = uint32_t(P) * uint32_t(K) * 4u;
  g.n_bi = has_bias ? uint32_t(P) * 4u : 0u;
  g.st = 0;
  g.cv = pipe_up16(g.st + g.n_st);
  g.xs = pipe_up16(g.cv + g.n_cv);
  g.bs = pipe_up16(g.xs + uint32_t(L_new) * g.n_x);
  g.cs = pipe_up16(g.bs + uint32_t(L_new) * g.n_bc);
  g.ws = pipe_up16(g.cs + uint32_t(L_new) * g.n_bc);
  g.bi = pipe_up16(g.ws + g.n_ws);
  g.stage = (g.bi + g.n_bi + 127u) & ~127u;
  return g;
}

// shared memory after the ring
constexpr int kPipeMaxGroups = 2;
struct PipeMisc {
  float us[kPipeMaxGroups][kPipeMaxLnew][kPipeMaxP];  // conv outputs of each group's item
  float a[kPipeMaxStages][kPipeMaxLnew];  // decays exp(dt A_h) of the stage's item
  uint64_t full[kPipeMaxStages];      // stage landed
  uint64_t done[kPipeMaxStages];      // compute finished with the stage
  int valid[kPipeMaxStages];
  int p0[kPipeMaxStages];
  int row[kPipeMaxStages];
  int go[kPipeMaxGroups];
  int abort;
};

template <typename T>
__device__ __forceinline__ float4 ld4_f32(const T* p);
template <>
__device__ __forceinline__ float4 ld4_f32<float>(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
template <>
__device__ __forceinline__ float4 ld4_f32<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 r = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xFFFF0000u),
                     __uint_as_float(r.y << 16), __uint_as_float(r.y & 0xFFFF0000u));
}

// bounded wait on an mbarrier phase; false on expiry or when the CTA aborts
__device__ __forceinline__ bool pipe_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          int* status) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = tc::globaltimer_ns();
  while (!tc::mbar_try_wait_sleep(bar, parity, 20000u)) {
    if (*abort) return false;
    if (tc::globaltimer_ns() - t0 > kPipeWaitNs) {
      *abort = 1;
      raise_status(status, SSS_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

template <typename T, int RP, int LT, int KT>
__global__ void __launch_bounds__(kPipeThreads, 1)
mixer_update_pipe_kernel(const T* __restrict__ x, const float* __restrict__ w,
                         const float* __restrict__ bias, T* conv_pool, int64_t pool, int S_len,
                         const int32_t* __restrict__ seqlens, const int32_t* __restrict__ idx,
                         const T* __restrict__ dt, const float* __restrict__ A,
                         const T* __restrict__ Bm, const T* __restrict__ Cm, float* ssm_pool,
                         T* __restrict__ y, int64_t n_items, int L_new, int H, int P, int G,
                         int K, int stages, PipeGeom geo, int* status) {
  extern __shared__ uint8_t pipe_smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(pipe_smem_raw) + 127) & ~uintptr_t(127));
  PipeMisc* ms = reinterpret_cast<PipeMisc*>(ring + size_t(stages) * geo.stage);
  const uint32_t ring_u32 = tc::smem_u32(ring);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int D = H * P;
  const int64_t i_begin = int64_t(blockIdx.x) * n_items / gridDim.x;
  const int64_t i_end = int64_t(blockIdx.x + 1) * n_items / gridDim.x;
  const int n = int(i_end - i_begin);
  // items are (b, h) pairs, h fastest; each role steps through its range
  // incrementally (no 64-bit division per item)
  const int64_t b_first = i_begin / H;
  const int h_first = int(i_begin - b_first * H);
  volatile int* abort_flag = &ms->abort;

  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      tc::mbar_init(tc::smem_u32(&ms->full[s]), 1);
      tc::mbar_init(tc::smem_u32(&ms->done[s]), 1);
    }
    ms->abort = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();

  if (warp == kPipeWarps) {
    // ------------------------------ producer ------------------------------
    // per lane, the (pool row, length, decays) of item g0 + lane of the
    // current group of 32 items, and the raw inputs of the next group
    // (loaded one group ahead, so nothing waits for them)
    int grp = -1, my_r = -1, my_p0 = -1;
    float my_a[LT];
    int nx_r = -1, nx_p0 = -1;
    float nx_A = 0.0f;
    T nx_dt[LT];
#pragma unroll
    for (int i = 0; i < LT; ++i) {
      my_a[i] = 0.0f;
      nx_dt[i] = from_f32<T>(0.0f);
    }
    auto fetch_group = [&](int g0) {
      const int kk = g0 + lane;
      if (kk < n) {
        const int lin = h_first + kk;
        const int64_t bl = b_first + lin / H;
        const int hl = lin % H;
        nx_r = idx ? idx[bl] : int(bl);
        nx_p0 = seqlens ? seqlens[bl] : S_len;  // no lengths: non-circular
        nx_A = A[hl];
#pragma unroll
        for (int i = 0; i < LT; ++i)
          if (i < L_new) nx_dt[i] = dt[(bl * L_new + i) * H + hl];
      }
    };
    fetch_group(0);
    int loaded = 0;
    int64_t lb = b_first;  // (b, h) of the next item to load
    int lh = h_first;
    // loads are issued for k = 0, 1, 2, ... in order
    auto issue_load = [&](int k) {
      const int s = k % stages;
      const int64_t b = lb;
      const int h = lh;
      if (++lh == H) {
        lh = 0;
        ++lb;
      }
      const int g = h / (H / G);
      const int g0 = k & ~31;
      if (g0 != grp) {  // move to the next group and prefetch the one after
        grp = g0;
        my_r = nx_r;
        my_p0 = nx_p0;
#pragma unroll
        for (int i = 0; i < LT; ++i) my_a[i] = expf(to_f32(nx_dt[i]) * nx_A);
        fetch_group(g0 + 32);
      }
      const int r = __shfl_sync(0xffffffffu, my_r, k & 31);
      const int p0 = __shfl_sync(0xffffffffu, my_p0, k & 31);
#pragma unroll
      for (int i = 0; i < LT; ++i) {
        const float ai = __shfl_sync(0xffffffffu, my_a[i], k & 31);
        if (lane == 0 && i < L_new) ms->a[s][i] = ai;
      }
      const bool valid = r >= 0 && int64_t(r) < pool && p0 >= 0;
      const uint32_t full = tc::smem_u32(&ms->full[s]);
      const uint32_t stg = ring_u32 + uint32_t(s) * geo.stage;
      if (lane == 0) {
        ms->valid[s] = valid ? 1 : 0;
        ms->p0[s] = p0;
        ms->row[s] = r;
      }
      if (!valid) {
        if (lane == 0) tc::mbar_arrive(full);
        return;
      }
      const uint32_t bytes = geo.n_st + geo.n_cv + geo.n_ws + geo.n_bi +
                             uint32_t(L_new) * (geo.n_x + 2u * geo.n_bc);
      if (lane == 0) tc::mbar_arrive_expect_tx(full, bytes);
      __syncwarp();
      const int n_copies = 4 + 3 * L_new;
      for (int j = lane; j < n_copies; j += 32) {
        if (j == 0) {
          tc::bulk_load(stg + geo.st, ssm_pool + (int64_t(r) * H + h) * int64_t(P) * kPipeN,
                        geo.n_st, full);
        } else if (j == 1) {
          tc::bulk_load(stg + geo.cv, conv_pool + (int64_t(r) * D + int64_t(h) * P) * S_len,
                        geo.n_cv, full);
        } else if (j == 2) {
          tc::bulk_load(stg + geo.ws, w + int64_t(h) * P * K, geo.n_ws, full);
        } else if (j == 3) {
          if (geo.n_bi) tc::bulk_load(stg + geo.bi, bias + int64_t(h) * P, geo.n_bi, full);
        } else {
          const int q = j - 4;
          const int i = q % L_new, kind = q / L_new;
          const int64_t tok = b * L_new + i;
          if (kind == 0)
            tc::bulk_load(stg + geo.xs + uint32_t(i) * geo.n_x, x + tok * D + int64_t(h) * P,
                          geo.n_x, full);
          else if (kind == 1)
            tc::bulk_load(stg + geo.bs + uint32_t(i) * geo.n_bc,
                          Bm + (tok * G + g) * int64_t(kPipeN), geo.n_bc, full);
          else
            tc::bulk_load(stg + geo.cs + uint32_t(i) * geo.n_bc,
                          Cm + (tok * G + g) * int64_t(kPipeN), geo.n_bc, full);
        }
      }
    };

    const int prime = n < stages ? n : stages;
    for (int k = 0; k < prime; ++k) issue_load(k);
    loaded = prime;
    int k = 0;
    bool ok = true;
    for (; k < n; ++k) {
      const int s = k % stages;
      int wok = 1;
      if (lane == 0)
        wok = pipe_wait(tc::smem_u32(&ms->done[s]), uint32_t((k / stages) & 1), abort_flag,
                        status) ? 1 : 0;
      wok = __shfl_sync(0xffffffffu, wok, 0);
      if (!wok) {
        ok = false;
        break;
      }
      // the compute warps have written the item's results from registers:
      // the stage is free again
      if (k + stages < n) {
        issue_load(k + stages);
        ++loaded;
      }
    }
    if (!ok && lane == 0) {
      // copies into stages that nobody will consume: wait for them to land
      for (int j = k; j < loaded; ++j)
        tc::mbar_wait(tc::smem_u32(&ms->full[j % stages]), uint32_t((j / stages) & 1),
                      kPipeWaitNs / 4);
    }
    return;
  }

  // ------------------------------ compute ------------------------------
  // With up to four new tokens the compute warps form two groups of four that
  // take alternate items, so one item's barriers and shuffle chains overlap
  // the other's arithmetic; group g syncs on named barrier 1 + g.
  constexpr int CG = LT <= 4 ? 2 : 1;
  constexpr int GW = kPipeWarps / CG;  // warps per group
  constexpr int RPG = RP * CG;         // state rows per warp of a group
  const int grp = warp / GW, gwarp = warp % GW, gtid = tid % (GW * 32);
  for (int k = grp; k < n; k += CG) {
    const int s = k % stages;
    const int64_t b = b_first + (h_first + k) / H;
    const int h = (h_first + k) % H;
    if (gtid == 0)
      ms->go[grp] = pipe_wait(tc::smem_u32(&ms->full[s]), uint32_t((k / stages) & 1), abort_flag,
                              status) ? 1 : 0;
    tc::role_sync(1 + grp, GW * 32);
    if (!ms->go[grp]) return;
    const int valid = ms->valid[s];
    const int p0 = ms->p0[s];
    uint8_t* stg = ring + size_t(s) * geo.stage;
    if (!valid) {
      for (int i = gtid; i < L_new * P; i += GW * 32) {
        const int tt = i / P, pp = i % P;
        y[((b * L_new + tt) * H + h) * P + pp] = from_f32<T>(0.0f);
      }
      if (gtid == 0) raise_status(status, SSS_ERR_INDEX);
    } else {
      // ---- conv over the slot tile: one (token i, channel c) per thread, so
      // the L_new tokens' convs run side by side.  Every read is of the
      // shared-memory copy of the pool row (the history) or of the new rows,
      // and every write goes to the pool in global memory: no read sees a write.
      {
        const T* xs = reinterpret_cast<const T*>(stg + geo.xs);
        const T* tile = reinterpret_cast<const T*>(stg + geo.cv);
        const int base = p0 % S_len;  // slot of logical position p0
        for (int e = gtid; e < L_new * P; e += GW * 32) {
          const int i = e / P, c = e - (e / P) * P;
          const T* row = tile + c * S_len;
          const float* wr = reinterpret_cast<const float*>(stg + geo.ws) + c * K;
          float z = geo.n_bi ? reinterpret_cast<const float*>(stg + geo.bi)[c] : 0.0f;
          // taps 0 .. K-2 read logical positions p0 + i - (K-1) + kk: a new
          // row when that is >= p0, else a history slot (one wrap at most)
#pragma unroll
          for (int kk = 0; kk < KT - 1; ++kk) {
            if (kk < K - 1) {
              const int rel = i - (K - 1) + kk;
              float v;
              if (rel >= 0) {
                v = to_f32(xs[rel * P + c]);
              } else {
                int sl = base + rel;
                sl += sl < 0 ? S_len : 0;
                v = to_f32(row[sl]);
              }
              z = fmaf(wr[kk], v, z);
            }
          }
          z = fmaf(wr[K - 1], to_f32(xs[i * P + c]), z);
          ms->us[grp][i][c] = silu(z);
          // the new input goes to the pool row: at the write pointer, or
          // (non-circular) the row shifted by L_new with the inputs appended
          T* grow = conv_pool + (int64_t(ms->row[s]) * D + int64_t(h) * P + c) * S_len;
          // (when L_new > S_len two tokens share a slot: the later one's
          // input is the one that stays, so only the last S_len tokens write)
          if (seqlens && i + S_len >= L_new) grow[(base + i) % S_len] = xs[i * P + c];
        }
        if (!seqlens) {
          for (int e = gtid; e < S_len * P; e += GW * 32) {
            const int j = e / P, c = e - (e / P) * P;
            const T* row = tile + c * S_len;
            T* grow = conv_pool + (int64_t(ms->row[s]) * D + int64_t(h) * P + c) * S_len;
            grow[j] = j + L_new < S_len ? row[j + L_new] : xs[(j + L_new - S_len) * P + c];
          }
        }
      }
      tc::role_sync(1 + grp, GW * 32);

      // ---- recurrence on the state block, in place
      const T* bsm = reinterpret_cast<const T*>(stg + geo.bs);
      const T* csm = reinterpret_cast<const T*>(stg + geo.cs);
      const float4* hst = reinterpret_cast<const float4*>(stg + geo.st);
      float4* gst = reinterpret_cast<float4*>(
          ssm_pool + (int64_t(ms->row[s]) * H + h) * int64_t(P) * kPipeN);
      // row-invariant operands, read once (the in-place state stores would
      // otherwise make the compiler re-read them for every row)
      // per token: the decay as a packed pair, this lane's four columns of B
      // and C as two packed pairs each (the state rows then take packed
      // f32x2 multiplies and FMAs: half the instructions)
      uint64_t av2[LT], b01[LT], b23[LT], c01[LT], c23[LT];
#pragma unroll
      for (int i = 0; i < LT; ++i) {
        const float a = i < L_new ? ms->a[s][i] : 0.0f;
        const float4 bv = i < L_new ? ld4_f32<T>(bsm + i * kPipeN + lane * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 cv = i < L_new ? ld4_f32<T>(csm + i * kPipeN + lane * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
        av2[i] = pk2(a, a);
        b01[i] = pk2(bv.x, bv.y);
        b23[i] = pk2(bv.z, bv.w);
        c01[i] = pk2(cv.x, cv.y);
        c23[i] = pk2(cv.z, cv.w);
      }
      float part[LT][RPG];
#pragma unroll
      for (int rr = 0; rr < RPG; ++rr) {
        const int p = gwarp + GW * rr;
#pragma unroll
        for (int i = 0; i < LT; ++i) part[i][rr] = 0.0f;
        if (p < P) {
          const float4 hv = hst[p * (kPipeN / 4) + lane];
          uint64_t h01 = pk2(hv.x, hv.y), h23 = pk2(hv.z, hv.w);
#pragma unroll
          for (int i = 0; i < LT; ++i) {
            if (i < L_new) {
              // h = a h + u B (columns in pairs), then this lane's part of h C
              const float u = ms->us[grp][i][p];
              const uint64_t u2 = pk2(u, u);
              h01 = fma2(av2[i], h01, mul2(u2, b01[i]));
              h23 = fma2(av2[i], h23, mul2(u2, b23[i]));
              float e, o;
              upk2(fma2(h23, c23[i], mul2(h01, c01[i])), e, o);
              part[i][rr] = e + o;
            }
          }
          float4 hn;
          upk2(h01, hn.x, hn.y);
          upk2(h23, hn.z, hn.w);
          gst[p * (kPipeN / 4) + lane] = hn;  // coalesced 16-byte stores
        }
      }
#pragma unroll
      for (int i = 0; i < LT; ++i) {
        if (i < L_new) {
          int rsel;
          const float yv = upd_reduce_scatter<RPG>(part[i], lane, &rsel);
          const int p = gwarp + GW * rsel;
          if ((lane & (32 / RPG - 1)) == 0 && p < P)
            y[((b * L_new + i) * H + h) * P + p] = from_f32<T>(yv);
        }
      }
    }
    tc::role_sync(1 + grp, GW * 32);
    if (gtid == 0) tc::mbar_arrive(tc::smem_u32(&ms->done[s]));
  }
}

template <typename T, int RP, int LT, int KT>
static cudaError_t launch_pipe(const void* x, const float* w, const float* bias, void* cp,
                               int64_t pool, int S_len, const int32_t* sl, const int32_t* ix,
                               const void* dt, const float* A, const void* B, const void* C,
                               float* sp, void* y, int64_t Bz, int L_new, int H, int P, int G,
                               int K, const PipeGeom& geo, int stages, int* status,
                               cudaStream_t st) {
  auto kern = mixer_update_pipe_kernel<T, RP, LT, KT>;
  const size_t smem = 128 + size_t(stages) * geo.stage + sizeof(PipeMisc);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(smem));
  if (e != cudaSuccess) return e;
  const int64_t n_items = Bz * H;
  const int64_t grid = n_items < sm_count() ? n_items : sm_count();
  kern<<<unsigned(grid), kPipeThreads, smem, st>>>(
      static_cast<const T*>(x), w, bias, static_cast<T*>(cp), pool, S_len, sl, ix,
      static_cast<const T*>(dt), A, static_cast<const T*>(B), static_cast<const T*>(C), sp,
      static_cast<T*>(y), n_items, L_new, H, P, G, K, stages, geo, status);
  return cudaGetLastError();
}

static bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Stages the pipelined kernel gets for this shape, or 0 when it does not
// take the call (then the per-(request, head) kernel above runs).
static int pipe_stages(const void* x, const float* w, const float* bias, const void* cp,
                       const void* B, const void* C, const float* sp, int esz, int S_len,
                       int L_new, int P, int N, int K, PipeGeom* geo) {
  if (N != kPipeN || P % 8 != 0 || P > kPipeMaxP || L_new < 1 || L_new > kPipeMaxLnew ||
      K > kUpdMaxK || (P * esz) % 16 != 0)
    return 0;
  if (!a16(x) || !a16(w) || (bias && !a16(bias)) || !a16(cp) || !a16(B) || !a16(C) || !a16(sp))
    return 0;
  *geo = pipe_geom(P, S_len, L_new, K, esz, bias != nullptr);
  int stages = int(kPipeRingBudget / geo->stage);
  if (stages > kPipeMaxStages) stages = kPipeMaxStages;
  return stages >= 2 ? stages : 0;
}

template <typename T>
static cudaError_t pipe_shape(const void* x, const float* w, const float* bias, void* cp,
                              int64_t pool, int S_len, const int32_t* sl, const int32_t* ix,
                              const void* dt, const float* A, const void* B, const void* C,
                              float* sp, void* y, int64_t Bz, int L_new, int H, int P, int G,
                              int K, const PipeGeom& geo, int stages, int* status,
                              cudaStream_t st) {
#define SSS_PIPE(RP, LT, KT)                                                                  \
  return launch_pipe<T, RP, LT, KT>(x, w, bias, cp, pool, S_len, sl, ix, dt, A, B, C, sp, y, \
                                    Bz, L_new, H, P, G, K, geo, stages, status, st)
  // the token count rounded up to 1, 2, 4 or 8: every loop over the tokens
  // unrolls and the operands of the new tokens stay in registers
  if (P <= 64) {
    if (L_new == 1) {
      if (K <= 4) SSS_PIPE(8, 1, 4);
      SSS_PIPE(8, 1, 8);
    }
    if (L_new == 2) {
      if (K <= 4) SSS_PIPE(8, 2, 4);
      SSS_PIPE(8, 2, 8);
    }
    if (L_new <= 4) {
      if (K <= 4) SSS_PIPE(8, 4, 4);
      SSS_PIPE(8, 4, 8);
    }
    if (K <= 4) SSS_PIPE(8, kPipeMaxLnew, 4);
    SSS_PIPE(8, kPipeMaxLnew, 8);
  }
  if (L_new == 1) {
    if (K <= 4) SSS_PIPE(16, 1, 4);
    SSS_PIPE(16, 1, 8);
  }
  if (K <= 4) SSS_PIPE(16, kPipeMaxLnew, 4);
  SSS_PIPE(16, kPipeMaxLnew, 8);
#undef SSS_PIPE
}

bool mixer_update_supports(int P, int N, int K, int L_new);

int mixer_update_path(sss_dtype at, int S_len, int L_new, int P, int N, int K) {
  if (!mixer_update_supports(P, N, K, L_new)) return -1;
  // any 16-byte aligned, non-null addresses: the choice depends on the
  // alignment only
  const void* a = reinterpret_cast<const void*>(uintptr_t(256));
  PipeGeom geo;
  return pipe_stages(a, static_cast<const float*>(a), static_cast<const float*>(a), a, a, a,
                     static_cast<const float*>(a), at == SSS_BF16 ? 2 : 4, S_len, L_new, P, N, K,
                     &geo) > 0
             ? 1
             : 0;
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
  PipeGeom geo;
  const int esz = at == SSS_BF16 ? 2 : 4;
  const int stages = pipe_stages(x, w, bias, cp, B, C, sp, esz, S_len, L_new, P, N, K, &geo);
  if (stages > 0) {
    if (at == SSS_BF16)
      return pipe_shape<__nv_bfloat16>(x, w, bias, cp, pool, S_len, sl, ix, dt, A, B, C, sp, y,
                                       Bz, L_new, H, P, G, K, geo, stages, status, st);
    return pipe_shape<float>(x, w, bias, cp, pool, S_len, sl, ix, dt, A, B, C, sp, y, Bz, L_new,
                             H, P, G, K, geo, stages, status, st);
  }
  if (at == SSS_BF16)
    return upd_shape<__nv_bfloat16>(x, w, bias, cp, pool, S_len, sl, ix, dt, A, B, C, sp, y,
                                    Bz, L_new, H, P, N, G, K, status, st);
  return upd_shape<float>(x, w, bias, cp, pool, S_len, sl, ix, dt, A, B, C, sp, y, Bz, L_new,
                          H, P, N, G, K, status, st);
}

}  // namespace sss
