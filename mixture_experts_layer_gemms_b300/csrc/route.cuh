// Router: affinity s = Sigmoid(u . e_i), biased top-K selection, gate = s,
// per-expert load histogram.
// ("【推理llm論文精讀】DeepSeek V3技術論文", section 2.2: affinity equation,
// routing-weight equation, auxiliary-loss-free selection over s + b.)
#pragma once
#include "common.cuh"

namespace moe {

constexpr int kRouteTile = 128;   // tokens per CTA (both router variants)
constexpr int kTopKMax = 16;

constexpr int kMaxExpertGroups = 64;  // group mask is one 64-bit word

// (beta, e) ranks above (ob, oe): larger beta, or equal beta and lower index.
__device__ __forceinline__ bool ranks_above(float b, int e, float ob, int oe) {
  return b > ob || (b == ob && e < oe);
}

// Mask of the M best of G contiguous expert groups for one token, computed
// by one warp (every lane gets the mask).  A group scores the largest beta
// among its N/G experts; ties go to the lower group index.
//
// Group-limited variant.  The pages name node-limited routing
// ("解码DeepSeek创新之道：三代模型演进路线图", V3 part) and a limit of 4
// nodes per token (the cooktownmusic.com report commentary, training
// framework part) without a group-score rule; the reading taken here: the
// N experts form G groups of N/G consecutive indices; a group scores the
// largest beta among its experts; the token keeps its M best groups and
// takes its top-K experts among them only.
__device__ __forceinline__ unsigned long long warp_group_mask(
    const float* s, const float* bias, int N, int G, int M, int lane) {
  const int per = N / G;
  float g0 = -INFINITY, g1 = -INFINITY;   // groups lane and lane + 32
  if (lane < G)
    for (int e = lane * per; e < (lane + 1) * per; ++e)
      g0 = fmaxf(g0, __fadd_rn(s[e], bias[e]));
  if (lane + 32 < G)
    for (int e = (lane + 32) * per; e < (lane + 33) * per; ++e)
      g1 = fmaxf(g1, __fadd_rn(s[e], bias[e]));
  int r0 = 0, r1 = 0;                     // groups ranked above each
  for (int h = 0; h < G; ++h) {
    const float a = __shfl_sync(0xffffffffu, g0, h & 31);
    const float c = __shfl_sync(0xffffffffu, g1, h & 31);
    const float gh = h < 32 ? a : c;
    r0 += ranks_above(gh, h, g0, lane) ? 1 : 0;
    r1 += ranks_above(gh, h, g1, lane + 32) ? 1 : 0;
  }
  const unsigned lo = __ballot_sync(0xffffffffu, lane < G && r0 < M);
  const unsigned hi = __ballot_sync(0xffffffffu, lane + 32 < G && r1 < M);
  return (static_cast<unsigned long long>(hi) << 32) | lo;
}

// Order-preserving map of a biased score to an unsigned key: a larger score
// gives a larger key, -0 is folded onto +0 (they compare equal as floats),
// and NaN maps to 0, below every real score, so it is never selected.
// Keys at or below kKeyNegInf (-inf) are not candidates.
constexpr uint32_t kKeyNegInf = 0x007FFFFFu;
__device__ __forceinline__ uint32_t score_key(float b) {
  uint32_t u = __float_as_uint(b);
  if (u == 0x80000000u) u = 0u;
  if (b != b) return 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Biased top-K of one token by one warp ("【推理llm論文精讀】DeepSeek V3
// 技術論文", section 2.2: selection over s + b, gate = s).  s[e] (e < N <=
// 32 PER) are the token's affinities in shared memory; lane j holds experts
// j, j + 32, ... (conflict-free reads) as score keys.  K rounds: every lane
// offers its best remaining candidate (highest key, lowest index among
// equal keys), a warp max-reduction (redux.sync) finds the highest key and a
// min-reduction the lowest expert index holding it, and the owner retires
// that expert -- so the result is sorted by (s + b desc, index asc) and the
// lowest index wins ties.  With M < G only experts of the token's M best
// groups compete.  Lanes 0..K-1 write the winners of rounds 0..K-1 and count
// them in the CTA histogram.  A round without a finite candidate (only with
// non-finite inputs) writes expert -1 and reports it.
template <int PER>
__device__ __forceinline__ void warp_select(const float* s, const float* bias,
                                            int N, int K, int G, int M, int t,
                                            int lane, int* topk_idx,
                                            float* topk_gate, int* hist) {
  uint32_t key[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane + 32 * i;
    key[i] = e < N ? score_key(__fadd_rn(s[e], bias[e])) : kKeyNegInf;
  }
  if (M < G) {
    const unsigned long long keep = warp_group_mask(s, bias, N, G, M, lane);
    const int per = N / G;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane + 32 * i;
      if (e < N && !((keep >> (e / per)) & 1ull)) key[i] = kKeyNegInf;
    }
  }
  int mine = -1;
  for (int k = 0; k < K; ++k) {
    uint32_t bk = 0u;
    int bi = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i)       // ascending index: '>' keeps the lowest
      if (key[i] > bk) {
        bk = key[i];
        bi = i;
      }
    const uint32_t top = __reduce_max_sync(0xffffffffu, bk);
    const uint32_t cand = (bk == top && top > kKeyNegInf)
                              ? static_cast<uint32_t>(lane + 32 * bi)
                              : 0xffffffffu;
    const int win = static_cast<int>(__reduce_min_sync(0xffffffffu, cand));
    if (lane == k) mine = win;          // -1 when no candidate was left
#pragma unroll
    for (int i = 0; i < PER; ++i)
      if (lane + 32 * i == win) key[i] = 0u;
  }
  if (lane < K) {
    int e = mine;
    float g = 0.f;
    if (e < 0 || e >= N) {
      report_error(ERR_CHECK, KID_ROUTE_TC, static_cast<unsigned>(t));
      e = -1;
    } else {
      g = s[e];
      atomicAdd(&hist[e], 1);
    }
    topk_idx[static_cast<size_t>(t) * K + lane] = e;
    topk_gate[static_cast<size_t>(t) * K + lane] = g;
  }
}

// ------------------------------------------------------------------------
// bf16 router on the tensor cores.  A 128-token tile x all N experts is
// computed by a cluster of S CTAs (S = 1, 2, 4 or 8) that split d:
// D[token lane, expert column] = u_tile . E^T over the CTA's share of d,
// accumulated in fp32 in TMEM, K-loop in 64-wide TMA stages.  Warp 0 lane 0
// issues TMA, warp 1 lane 0 issues tcgen05.mma.  With S = 1 all 4 warps then
// read their 32 TMEM lanes (one token per thread) and run the sigmoid +
// biased top-K in fp32.  With S > 1 every CTA dumps its partial z to its own
// shared memory; CTA r then sums the S partials (in rank order, through
// distributed shared memory) for tokens r*128/S .. (r+1)*128/S - 1 and
// selects for those tokens.  Splitting d keeps one wave of CTAs busy when
// there are fewer tiles than SMs.
constexpr int kRtStages = 4;
constexpr int kRtBK = 64;
constexpr int kRouteThreads = 512;   // 16 warps: 2 pipeline roles, all epilogue
constexpr int kRtMaxSplit = 8;

// CTAs per token tile: the largest of 1, 2, 4, 8 that keeps the grid within
// one wave of `sms` CTAs and gives each CTA at least 8 of the 64-wide
// K-blocks.
inline int route_split(long long T, int d, int sms) {
  const long long nblk = (T + kRouteTile - 1) / kRouteTile;
  int S = 1;
  while (S < kRtMaxSplit && nblk * S * 2 <= sms && d / kRtBK >= S * 2 * 8)
    S *= 2;
  return S;
}

struct RouteTcSmemLayout {
  static constexpr int a_bytes = kRouteTile * kRtBK * 2;   // 16 KB / stage
  static constexpr int b_bytes_max = 256 * kRtBK * 2;      // 32 KB / stage
  static constexpr int a_off = 0;
  static constexpr int b_off = a_off + kRtStages * a_bytes;
  static constexpr int ring_end = b_off + kRtStages * b_bytes_max;
  // epilogue, over the freed ring: z [128][P] fp32 (affinities when S = 1,
  // this CTA's partial when S > 1), then the affinities of this CTA's token
  // slice [128/S][P] (S >= 2); P = row_stride(N)
  static constexpr int kMaxP = 260;
  static constexpr int zpart_off = 0;
  static constexpr int zpart_bytes = kRouteTile * kMaxP * 4;
  static constexpr int slice_off = zpart_off + zpart_bytes;
  static constexpr int slice_end = slice_off + (kRouteTile / 2) * kMaxP * 4;
  // Row stride (floats) of the epilogue's score rows: a multiple of 4 above
  // N, so rows start on 16-byte boundaries (vector stores and loads) and the
  // 16-byte stores of 8 consecutive rows cover all 32 banks.
  __host__ __device__ static constexpr int row_stride(int n) {
    return (n + 4) & ~3;
  }
  static constexpr int bar_off =
      ((ring_end > slice_end ? ring_end : slice_end) + 15) & ~15;
  static constexpr int misc_off = bar_off + (2 * kRtStages + 1) * 8;
  static constexpr int hist_off = misc_off + 16;
  static constexpr int bias_off = hist_off + 256 * 4;
  static constexpr int total = bias_off + 256 * 4;
  static constexpr int alloc = total + 1024;   // base re-aligned to 1024
};

__global__ void __launch_bounds__(kRouteThreads, 1)
route_tc_kernel(const __grid_constant__ CUtensorMap tm_u,
                const __grid_constant__ CUtensorMap tm_e,
                const float* __restrict__ bias, int T, int d, int N, int K,
                int G, int M, int split, int* __restrict__ topk_idx,
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
  const int S = split;
  const int rank = S > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int tile = blockIdx.x / S;
  const int nk_all = d / kRtBK;
  const int kb_lo = rank * nk_all / S;
  const int nk = (rank + 1) * nk_all / S - kb_lo;   // this CTA's K-blocks
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
      const int kb = kb_lo + (kb0 + i) % nk;
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

  // Epilogue.  Warp w reads TMEM lane quarter w % 4 (32 token rows, one per
  // lane) and every fourth 32-column chunk from chunk w / 4, and stores z
  // summed over the accumulators to shared memory (the pipeline buffers are
  // free by now), row-major with stride P in 16-byte vectors: as affinities
  // s = sigmoid(z) when S = 1, as the raw partial when S > 1.  Then one warp
  // per token selects (warp_select).
  const bool done_ok = mbar_wait(bar_done, 0, abort_flag, KID_ROUTE_TC, 3);
  tc_fence_after();
  const bool go = __all_sync(0xffffffffu, done_ok && !*abort_flag);
  constexpr int kWarps = kRouteThreads / 32;
  const int P = L::row_stride(N);
  {
    const int q = warp & 3;
    const int row = q * 32 + lane;
    float* srow = reinterpret_cast<float*>(smem) + row * P;
    if (go) {
      const int used = min(n_acc, nk);
      for (int c0 = (warp >> 2) * 32; c0 < N; c0 += 32 * (kWarps / 4)) {
        float z[32];
        uint32_t r[32];
        const uint32_t ta = tmem + (static_cast<uint32_t>(q * 32) << 16) + c0;
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
        if (S == 1) {
#pragma unroll
          for (int j = 0; j < 32; ++j) z[j] = sigmoid_f32(z[j]);
        }
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          if (c0 + j < N)
            *reinterpret_cast<float4*>(srow + c0 + j) =
                make_float4(z[j], z[j + 1], z[j + 2], z[j + 3]);
      }
    }
  }
  __syncthreads();
  if (S == 1) {
    const float* sfull = reinterpret_cast<const float*>(smem);
    for (int r = warp; r < kRouteTile; r += kWarps) {
      const int t = tile * kRouteTile + r;
      if (go && t < T)
        warp_select<8>(sfull + r * P, bias_s, N, K, G, M, t, lane,
                       topk_idx, topk_gate, hist);
    }
  } else {
    // Every CTA of the cluster passes both cluster barriers, whatever its
    // own state (a CTA that skipped one would leave the others waiting).
    cluster_sync();                     // all partials are in place
    const int R = kRouteTile / S;       // tokens selected by this CTA
    const int r0 = rank * R;
    float* slice = reinterpret_cast<float*>(smem + L::slice_off);
    if (go) {
      // z = the S partials summed in rank order, four experts per 16-byte
      // vector: the own partial from local shared memory, the others
      // through distributed shared memory.  Each thread takes four vectors
      // at a time and issues all four loads of a rank before adding them.
      const uint32_t zbase = sbase + L::zpart_off;
      const float* zloc = reinterpret_cast<const float*>(smem + L::zpart_off);
      const int n4 = (N + 3) >> 2;
      const int items = R * n4;
      const int nthr = static_cast<int>(blockDim.x);
      for (int i0 = threadIdx.x; i0 < items; i0 += 4 * nthr) {
        float4 acc[4], x[4];
        int w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = min(i0 + u * nthr, items - 1);
          const int rl = i / n4;
          w[u] = (r0 + rl) * P + (i - rl * n4) * 4;
        }
        for (int q = 0; q < S; ++q) {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            x[u] = q == rank
                       ? *reinterpret_cast<const float4*>(zloc + w[u])
                       : ld_cluster_v4(mapa_shared(zbase + 4u * w[u], q));
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (q == 0) {
              acc[u] = x[u];
            } else {
              acc[u].x = __fadd_rn(acc[u].x, x[u].x);
              acc[u].y = __fadd_rn(acc[u].y, x[u].y);
              acc[u].z = __fadd_rn(acc[u].z, x[u].z);
              acc[u].w = __fadd_rn(acc[u].w, x[u].w);
            }
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + u * nthr;
          if (i < items) {
            const int rl = i / n4;
            *reinterpret_cast<float4*>(slice + rl * P + (i - rl * n4) * 4) =
                make_float4(sigmoid_f32(acc[u].x), sigmoid_f32(acc[u].y),
                            sigmoid_f32(acc[u].z), sigmoid_f32(acc[u].w));
          }
        }
      }
    }
    __syncthreads();
    for (int r = warp; r < R; r += kWarps) {
      const int t = tile * kRouteTile + r0 + r;
      if (go && t < T)
        warp_select<8>(slice + r * P, bias_s, N, K, G, M, t, lane, topk_idx,
                       topk_gate, hist);
    }
    cluster_sync();                     // no CTA leaves while read remotely
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
    if (N <= 256)
      warp_select<8>(z, bias, N, K, G, M, t, lane, topk_idx, topk_gate, hist);
    else
      warp_select<32>(z, bias, N, K, G, M, t, lane, topk_idx, topk_gate,
                      hist);
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
