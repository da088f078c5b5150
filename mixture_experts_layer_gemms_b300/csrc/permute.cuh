// Dispatch of the token rows to expert-contiguous slots.
// ("【推理llm論文精讀】DeepSeek V3技術論文", section 2.2: each token's routed
// FFNs are those of its top-K_r experts; the layout -- experts in index
// order, tokens in ascending order inside an expert -- is this library's.)
#pragma once
#include "common.cuh"

namespace moe {

constexpr int kPermChunk = 128;   // tokens per CTA in the slot kernels

// chunk_hist[c][e] = assignments of tokens [c*128, c*128+128) to expert e.
__global__ void __launch_bounds__(256)
permute_chunk_hist_kernel(const int* __restrict__ topk_idx, int T, int K,
                          int N, int* __restrict__ chunk_hist) {
  __shared__ int hist[1024];
  for (int e = threadIdx.x; e < N; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int t0 = blockIdx.x * kPermChunk;
  const int nt = min(kPermChunk, T - t0);
  const int na = nt * K;
  const int* idx = topk_idx + static_cast<size_t>(t0) * K;
  for (int a = threadIdx.x; a < na; a += blockDim.x) {
    const int e = idx[a];
    if (e >= 0 && e < N)
      atomicAdd(&hist[e], 1);
    else
      report_error(ERR_CHECK, 10, static_cast<unsigned>(t0 * K + a));
  }
  __syncthreads();
  for (int e = threadIdx.x; e < N; e += blockDim.x)
    chunk_hist[static_cast<size_t>(blockIdx.x) * N + e] = hist[e];
}

// Block-wide exclusive scan of v[0..n) in shared memory (n <= 1024,
// blockDim.x == 256): out[i] = sum_{j<i} v[j], out[n] = total.
static __device__ void block_exclusive_scan(const int* v, int* out, int n,
                                     int* warp_tot) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // each thread owns 4 consecutive entries
  int loc[4];
  int sum = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = tid * 4 + j;
    loc[j] = (i < n) ? v[i] : 0;
    sum += loc[j];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int wbase = 0;
  for (int w = 0; w < warp; ++w) wbase += warp_tot[w];
  int run = wbase + incl - sum;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = tid * 4 + j;
    if (i < n) out[i] = run;
    run += loc[j];
  }
  if (tid == blockDim.x - 1) out[n] = run;
  __syncthreads();
}

// Slots of chunk c.  offsets = exclusive scan of counts (every CTA computes
// it; CTA 0 writes it).  Expert e's slots for this chunk start at
// offsets[e] + sum_{c'<c} chunk_hist[c'][e].  Inside the chunk, warp 0 walks
// the assignments in (token, k) order 32 at a time: lanes holding the same
// expert find each other with __match_any_sync, take consecutive slots in
// lane order, and the first of them advances that expert's running slot --
// so slots follow token order and nothing depends on atomics.
__global__ void __launch_bounds__(256)
permute_slots_kernel(const int* __restrict__ topk_idx,
                     const int* __restrict__ counts,
                     const int* __restrict__ chunk_hist, int T, int K, int N,
                     int* __restrict__ offsets, int* __restrict__ perm,
                     int* __restrict__ inv) {
  __shared__ int cnt[1024];
  __shared__ int offs[1025];
  __shared__ int run[1024];
  __shared__ int idx_s[kPermChunk * 16];
  __shared__ int warp_tot[8];
  for (int e = threadIdx.x; e < N; e += blockDim.x) cnt[e] = counts[e];
  __syncthreads();
  block_exclusive_scan(cnt, offs, N, warp_tot);
  if (blockIdx.x == 0)
    for (int e = threadIdx.x; e <= N; e += blockDim.x) offsets[e] = offs[e];
  const int c = blockIdx.x;
  for (int e = threadIdx.x; e < N; e += blockDim.x) {
    int b = offs[e];
    for (int cc = 0; cc < c; ++cc) b += chunk_hist[static_cast<size_t>(cc) * N + e];
    run[e] = b;
  }
  const int t0 = c * kPermChunk;
  const int nt = min(kPermChunk, T - t0);
  const int na = nt * K;
  for (int a = threadIdx.x; a < na; a += blockDim.x)
    idx_s[a] = topk_idx[static_cast<size_t>(t0) * K + a];
  __syncthreads();
  // slots never exceed the T*K assignments, whatever counts say
  const int total = min(offs[N], T * K);
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  const unsigned lt = (1u << lane) - 1u;
  for (int a0 = 0; a0 < na; a0 += 32) {
    const int a = a0 + lane;
    const bool valid = a < na;
    const int e = valid ? idx_s[a] : -1;
    const bool good = valid && e >= 0 && e < N;
    const unsigned m = __match_any_sync(0xffffffffu, good ? e : N + lane);
    const int rank = __popc(m & lt);
    const int base = good ? run[e] : 0;
    __syncwarp();
    if (good && rank == 0) run[e] = base + __popc(m);
    __syncwarp();
    if (good) {
      const int slot = base + rank;
      if (slot < total) {
        inv[static_cast<size_t>(t0) * K + a] = slot;
        perm[slot] = t0 + a / K;
      } else {
        report_error(ERR_CHECK, 11, static_cast<unsigned>(slot));
      }
    } else if (valid) {
      report_error(ERR_CHECK, 13, static_cast<unsigned>(t0 * K + a));
    }
  }
}

// x_perm[inv[t,k]] = u[t] for every k: one warp per token, 16-byte vectors,
// each u row read once and written K times.
__global__ void __launch_bounds__(256)
permute_gather_kernel(const uint4* __restrict__ u, const int* __restrict__ inv,
                      int T, int K, int nvec, long long total_slots,
                      uint4* __restrict__ x_perm) {
  const int lane = threadIdx.x & 31;
  const int warps_per_block = blockDim.x >> 5;
  for (int t = blockIdx.x * warps_per_block + (threadIdx.x >> 5); t < T;
       t += gridDim.x * warps_per_block) {
    int slot[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      slot[k] = (k < K) ? inv[static_cast<size_t>(t) * K + k] : -1;
      if (k < K && (slot[k] < 0 || slot[k] >= total_slots)) {
        if (lane == 0) report_error(ERR_CHECK, 12, static_cast<unsigned>(t));
        slot[k] = -1;
      }
    }
    const uint4* src = u + static_cast<size_t>(t) * nvec;
    // four 16-byte loads in flight per lane before the stores
    for (int v0 = lane; v0 < nvec; v0 += 128) {
      uint4 val[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (v0 + 32 * j < nvec) val[j] = __ldg(src + v0 + 32 * j);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int v = v0 + 32 * j;
        if (v < nvec) {
#pragma unroll
          for (int k = 0; k < 16; ++k)
            if (k < K && slot[k] >= 0)
              x_perm[static_cast<size_t>(slot[k]) * nvec + v] = val[j];
        }
      }
    }
  }
}

}  // namespace moe
