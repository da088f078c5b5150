// Router: affinity s = Sigmoid(u . e_i), biased top-K selection, gate = s,
// per-expert load histogram.
// ("【推理llm論文精讀】DeepSeek V3技術論文", section 2.2: affinity equation,
// routing-weight equation, auxiliary-loss-free selection over s + b.)
#pragma once
#include "common.cuh"

namespace moe {

constexpr int kRouteTile = 128;   // tokens per CTA (both router variants)
constexpr int kTopKMax = 16;

// Running top-KT of (beta, index) pairs, best first, in registers (KT is a
// compile-time size >= K; the first K entries are the top-K).  A pair ranks
// above another when its beta is larger, or equal with a lower index -- so
// the lowest index wins a tie, whatever order candidates arrive in.
template <int KT>
struct TopK {
  float b[KT];
  float s[KT];
  int i[KT];

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int j = 0; j < KT; ++j) {
      b[j] = -INFINITY;
      s[j] = 0.f;
      i[j] = 0x7fffffff;
    }
  }
  // Candidates arrive in ascending index order, so a candidate whose beta
  // only equals the current last entry never enters (the earlier index
  // keeps its place).
  __device__ __forceinline__ void push(float beta, float sv, int idx) {
    if (!(beta > b[KT - 1])) return;
    float cb = beta, cs = sv;
    int ci = idx;
#pragma unroll
    for (int j = 0; j < KT; ++j) {
      const bool better = (cb > b[j]) || (cb == b[j] && ci < i[j]);
      const float tb = b[j], ts = s[j];
      const int ti = i[j];
      b[j] = better ? cb : tb;
      s[j] = better ? cs : ts;
      i[j] = better ? ci : ti;
      cb = better ? tb : cb;
      cs = better ? ts : cs;
      ci = better ? ti : ci;
    }
  }
  // Writes token t's first K entries and counts them in the CTA histogram.
  // A slot left empty (only possible with non-finite affinities) is written
  // as -1 and reported; it is never used as an index.
  __device__ __forceinline__ void store(int t, int K, int N, int* topk_idx,
                                        float* topk_gate, int* hist) const {
#pragma unroll
    for (int j = 0; j < KT; ++j) {
      if (j < K) {
        int e = i[j];
        if (e < 0 || e >= N) {
          report_error(ERR_CHECK, KID_ROUTE_TC, static_cast<unsigned>(t));
          e = -1;
        } else {
          atomicAdd(&hist[e], 1);
        }
        topk_idx[static_cast<size_t>(t) * K + j] = e;
        topk_gate[static_cast<size_t>(t) * K + j] = s[j];
      }
    }
  }
};

// Biased top-K of one token from its affinities s[e * stride] (e < N), fp32:
// beta = s + b, candidates in ascending expert order.
template <int KT>
__device__ __forceinline__ void select_token(const float* s, int stride,
                                             const float* bias, int N, int K,
                                             int t, int* topk_idx,
                                             float* topk_gate, int* hist) {
  TopK<KT> top;
  top.reset();
#pragma unroll 4
  for (int e = 0; e < N; ++e) {
    const float sv = s[e * stride];
    top.push(__fadd_rn(sv, bias[e]), sv, e);
  }
  top.store(t, K, N, topk_idx, topk_gate, hist);
}

constexpr int kMaxExpertGroups = 64;  // group mask is one 64-bit word
constexpr int kMaxTopGroups = 8;

// Group-limited variant.  The pages name node-limited routing
// ("解码DeepSeek创新之道：三代模型演进路线图", V3 part) and a limit of 4
// nodes per token (the cooktownmusic.com report commentary, training
// framework part) without a group-score rule; the reading taken here: the
// N experts form G groups of N/G consecutive indices; a group scores the
// largest beta among its experts; the token keeps its M best groups (lower
// group index first on ties) and takes its top-K experts among them only.
// Kept groups are visited in ascending order, so candidates still arrive in
// ascending expert order and TopK's tie rule holds.
template <int KT>
__device__ __forceinline__ void select_token_grouped(
    const float* s, int stride, const float* bias, int N, int K, int G, int M,
    int t, int* topk_idx, float* topk_gate, int* hist) {
  const int per = N / G;
  TopK<kMaxTopGroups> gtop;
  gtop.reset();
  for (int g = 0; g < G; ++g) {
    float gm = -INFINITY;
    for (int e = g * per; e < (g + 1) * per; ++e)
      gm = fmaxf(gm, __fadd_rn(s[e * stride], bias[e]));
    gtop.push(gm, 0.f, g);
  }
  unsigned long long keep = 0;
#pragma unroll
  for (int j = 0; j < kMaxTopGroups; ++j)
    if (j < M && gtop.i[j] < G) keep |= 1ull << gtop.i[j];
  TopK<KT> top;
  top.reset();
  while (keep) {
    const int g = __ffsll(static_cast<long long>(keep)) - 1;
    keep &= keep - 1;
    for (int e = g * per; e < (g + 1) * per; ++e) {
      const float sv = s[e * stride];
      top.push(__fadd_rn(sv, bias[e]), sv, e);
    }
  }
  top.store(t, K, N, topk_idx, topk_gate, hist);
}

// G == M keeps every group: plain selection.
__device__ __forceinline__ void select_token_any(const float* s, int stride,
                                                 const float* bias, int N,
                                                 int K, int G, int M, int t,
                                                 int* topk_idx,
                                                 float* topk_gate, int* hist) {
  if (M < G) {
    if (K <= 4)
      select_token_grouped<4>(s, stride, bias, N, K, G, M, t, topk_idx,
                              topk_gate, hist);
    else if (K <= 8)
      select_token_grouped<8>(s, stride, bias, N, K, G, M, t, topk_idx,
                              topk_gate, hist);
    else
      select_token_grouped<16>(s, stride, bias, N, K, G, M, t, topk_idx,
                               topk_gate, hist);
    return;
  }
  if (K <= 4)
    select_token<4>(s, stride, bias, N, K, t, topk_idx, topk_gate, hist);
  else if (K <= 8)
    select_token<8>(s, stride, bias, N, K, t, topk_idx, topk_gate, hist);
  else
    select_token<16>(s, stride, bias, N, K, t, topk_idx, topk_gate, hist);
}

// ------------------------------------------------------------------------
// bf16 router on the tensor cores.  One CTA = 128 tokens x all N experts:
// D[token lane, expert column] = u_tile . E^T accumulated in fp32 in TMEM,
// K-loop over d in 64-wide TMA stages.  Warp 0 lane 0 issues TMA, warp 1
// lane 0 issues tcgen05.mma; then all 4 warps read their 32 TMEM lanes (one
// token per thread) and run the sigmoid + biased top-K in fp32.
constexpr int kRtStages = 4;
constexpr int kRtBK = 64;

struct RouteTcSmemLayout {
  static constexpr int a_bytes = kRouteTile * kRtBK * 2;   // 16 KB / stage
  static constexpr int b_bytes_max = 256 * kRtBK * 2;      // 32 KB / stage
  static constexpr int a_off = 0;
  static constexpr int b_off = a_off + kRtStages * a_bytes;
  static constexpr int bar_off = b_off + kRtStages * b_bytes_max;
  static constexpr int misc_off = bar_off + (2 * kRtStages + 1) * 8;
  static constexpr int hist_off = misc_off + 16;
  static constexpr int bias_off = hist_off + 256 * 4;
  static constexpr int total = bias_off + 256 * 4;
  static constexpr int alloc = total + 1024;   // base re-aligned to 1024
};

__global__ void __launch_bounds__(128, 1)
route_tc_kernel(const __grid_constant__ CUtensorMap tm_u,
                const __grid_constant__ CUtensorMap tm_e,
                const float* __restrict__ bias, int T, int d, int N, int K,
                int G, int M, int* __restrict__ topk_idx,
                float* __restrict__ topk_gate,
                int* __restrict__ hist_partial) {
  using L = RouteTcSmemLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + L::bar_off;            // [stages]
  const uint32_t bar_empty = bar_full + 8 * kRtStages;     // [stages]
  const uint32_t bar_done = bar_empty + 8 * kRtStages;
  volatile uint32_t* tmem_slot =
      reinterpret_cast<volatile uint32_t*>(smem + L::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc_off + 4);
  int* hist = reinterpret_cast<int*>(smem + L::hist_off);
  float* bias_s = reinterpret_cast<float*>(smem + L::bias_off);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x;
  const int nk = d / kRtBK;
  const uint32_t b_bytes = static_cast<uint32_t>(N) * kRtBK * 2;
  // The K loop round-robins over n_acc TMEM accumulators (summed in fp32 in
  // the epilogue): each accumulator then sees 1/n_acc of the d/16 MMA
  // accumulation steps, which divides the rounding drift of the tensor
  // core's fp32 accumulation by n_acc.  All of TMEM is used when N = 256.
  uint32_t acc_cols = 32;
  while (acc_cols < static_cast<uint32_t>(N)) acc_cols <<= 1;
  const int n_acc = min(4, static_cast<int>(512u / acc_cols));
  const uint32_t ncols = acc_cols * n_acc;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRtStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_u);
    tma_prefetch_desc(&tm_e);
  }
  if (warp == 1) {
    tmem_alloc(sbase + L::misc_off, ncols);
    tmem_relinquish();
  }
  for (int e = threadIdx.x; e < N; e += blockDim.x) {
    hist[e] = 0;
    bias_s[e] = bias[e];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // TMA producer.  Each CTA walks d from its own starting block (rotated
    // order), so the CTAs do not all fetch the same centroid block from the
    // same L2 slices at the same moment.
    int issued = 0;
    const int kb0 = (tile * 5) % nk;
    for (int i = 0; i < nk; ++i) {
      const int s = i % kRtStages;
      const uint32_t ph = (i / kRtStages) & 1;
      const int kb = (kb0 + i) % nk;
      if (!mbar_wait(bar_empty + 8 * s, ph ^ 1, abort_flag, KID_ROUTE_TC, 1))
        break;
      ++issued;
      mbar_arrive_expect_tx(bar_full + 8 * s, L::a_bytes + b_bytes);
      tma_load_2d(sbase + L::a_off + s * L::a_bytes, &tm_u, kb * kRtBK,
                  tile * kRouteTile, bar_full + 8 * s);
      tma_load_2d(sbase + L::b_off + s * L::b_bytes_max, &tm_e, kb * kRtBK, 0,
                  bar_full + 8 * s);
    }
    if (*abort_flag)   // let loads still in flight land before exit
      for (int j = issued > kRtStages ? issued - kRtStages : 0; j < issued; ++j)
        mbar_drain(bar_full + 8 * (j % kRtStages), (j / kRtStages) & 1);
  } else if (warp == 1 && lane == 0) {
    // MMA issuer
    const uint32_t idesc = idesc_bf16_f32(128, N);
    for (int i = 0; i < nk; ++i) {
      const int s = i % kRtStages;
      const uint32_t ph = (i / kRtStages) & 1;
      if (!mbar_wait(bar_full + 8 * s, ph, abort_flag, KID_ROUTE_TC, 2))
        break;
      tc_fence_after();
      const uint32_t a0 = sbase + L::a_off + s * L::a_bytes;
      const uint32_t b0 = sbase + L::b_off + s * L::b_bytes_max;
      const uint32_t d_acc = tmem + (i % n_acc) * acc_cols;
#pragma unroll
      for (int kk = 0; kk < kRtBK / 16; ++kk)
        mma_bf16(d_acc, sdesc_k128(a0 + kk * 32), sdesc_k128(b0 + kk * 32),
                 idesc, (i >= n_acc || kk > 0) ? 1u : 0u);
      mma_commit(bar_empty + 8 * s);
    }
    mma_commit(bar_done);   // also fires when the loop stopped early
  }
  __syncwarp();

  // Epilogue: every thread owns one token (TMEM lane).  Its affinities go
  // to shared memory (the pipeline buffers are free by now), row-major with
  // a padded stride so a warp's accesses hit distinct banks, then a plain
  // loop selects the top-K.
  const bool done_ok = mbar_wait(bar_done, 0, abort_flag, KID_ROUTE_TC, 3);
  tc_fence_after();
  const bool go = __all_sync(0xffffffffu, done_ok && !*abort_flag);
  const int row = warp * 32 + lane;
  const int t = tile * kRouteTile + row;
  float* srow = reinterpret_cast<float*>(smem) + row * (N + 1);
  if (go) {
    const int used = min(n_acc, nk);
    for (int c0 = 0; c0 < N; c0 += 32) {
      float z[32];
      uint32_t r[32];
      const uint32_t ta = tmem + (static_cast<uint32_t>(warp * 32) << 16) + c0;
      tmem_ld32(ta, r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) z[j] = __uint_as_float(r[j]);
      for (int a = 1; a < used; ++a) {
        tmem_ld32(ta + a * acc_cols, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) z[j] += __uint_as_float(r[j]);
      }
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (c0 + j < N) srow[c0 + j] = sigmoid_f32(z[j]);
    }
    if (t < T)
      select_token_any(srow, 1, bias_s, N, K, G, M, t, topk_idx, topk_gate,
                       hist);
  }
  tc_fence_before();
  __syncthreads();
  for (int e = threadIdx.x; e < N; e += blockDim.x)
    hist_partial[static_cast<size_t>(blockIdx.x) * N + e] = hist[e];
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

// ------------------------------------------------------------------------
// fp32 router on the CUDA cores: one warp per token, lanes split d, a
// butterfly sum gives z = u . e_i for every expert; lane 0 selects.
__global__ void __launch_bounds__(128)
route_f32_kernel(const float* __restrict__ u, const float* __restrict__ E,
                 const float* __restrict__ bias, int T, int d, int N, int K,
                 int G, int M, int* __restrict__ topk_idx,
                 float* __restrict__ topk_gate,
                 int* __restrict__ hist_partial) {
  extern __shared__ float zbuf[];        // [4 warps][N]
  __shared__ int hist[1024];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < N; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  float* z = zbuf + warp * N;
  for (int r = warp; r < kRouteTile; r += 4) {
    const int t = blockIdx.x * kRouteTile + r;
    if (t >= T) break;
    const float* ut = u + static_cast<size_t>(t) * d;
    for (int e = 0; e < N; ++e) {
      const float* ee = E + static_cast<size_t>(e) * d;
      float acc = 0.f;
      for (int j = lane; j < d; j += 32) acc = fmaf(ut[j], ee[j], acc);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) z[e] = acc;
    }
    __syncwarp();
    for (int e = lane; e < N; e += 32) z[e] = sigmoid_f32(z[e]);
    __syncwarp();
    if (lane == 0)
      select_token_any(z, 1, bias, N, K, G, M, t, topk_idx, topk_gate, hist);
    __syncwarp();
  }
  __syncthreads();
  for (int e = threadIdx.x; e < N; e += blockDim.x)
    hist_partial[static_cast<size_t>(blockIdx.x) * N + e] = hist[e];
}

// counts[e] = sum over router CTAs of their histograms (fixed order).
__global__ void route_hist_reduce_kernel(const int* __restrict__ hist_partial,
                                         int nblk, int N,
                                         int* __restrict__ counts) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= N) return;
  int c = 0;
  for (int b = 0; b < nblk; ++b) c += hist_partial[static_cast<size_t>(b) * N + e];
  counts[e] = c;
}

}  // namespace moe
