// Bandwidth-bound kernels of the MoE layer: combine, bias update, weight
// repack.  ("【推理llm論文精讀】DeepSeek V3技術論文", section 2.2: FFN-output
// equation; auxiliary-loss-free bias adjustment.)
#pragma once
#include "common.cuh"

namespace moe {

// 8 bf16 or 4 fp32 per 16-byte vector.
template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int n = 8;
  __device__ static void load(const void* p, float* f) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x = __bfloat1622float2(h[i]);
      f[2 * i] = x.x;
      f[2 * i + 1] = x.y;
    }
  }
};
template <>
struct Vec<float> {
  static constexpr int n = 4;
  __device__ static void load(const void* p, float* f) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(p));
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
  }
};

// Loads V consecutive expert outputs (fp32 or fp16; V = 4 or 8) as fp32.
template <int V>
__device__ __forceinline__ void load_y(const float* p, float* f) {
#pragma unroll
  for (int i = 0; i < V; i += 4) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(p + i));
    f[i] = v.x; f[i + 1] = v.y; f[i + 2] = v.z; f[i + 3] = v.w;
  }
}
template <int V>
__device__ __forceinline__ void load_y(const __half* p, float* f) {
#pragma unroll
  for (int i = 0; i < V; i += 4) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(p + i));
    const __half2* h = reinterpret_cast<const __half2*>(&v);
    const float2 a = __half22float2(h[0]), b = __half22float2(h[1]);
    f[i] = a.x; f[i + 1] = a.y; f[i + 2] = b.x; f[i + 3] = b.y;
  }
}

// h[t] = u[t] + y_shared[t] + sum_k gate[t,k] * y_perm[inv[t,k]], fp32 in
// that order (y_perm, y_shared are TY: fp16 or fp32).  One CTA per token,
// 16-byte vectors of u along d.
template <typename TI, typename TY, typename TO>
__global__ void __launch_bounds__(128)
combine_kernel(const TI* __restrict__ u, const TY* __restrict__ y_perm,
               const TY* __restrict__ y_shared, const int* __restrict__ inv,
               const float* __restrict__ gate, int T, int d, int K,
               long long total_slots, TO* __restrict__ h) {
  constexpr int V = Vec<TI>::n;
  __shared__ int slot_s[16];
  __shared__ float gate_s[16];
  const int t = blockIdx.x;
  if (threadIdx.x < K) {
    int s = inv[static_cast<size_t>(t) * K + threadIdx.x];
    if (s < 0 || s >= total_slots) {
      report_error(ERR_CHECK, 20, static_cast<unsigned>(t));
      s = -1;
    }
    slot_s[threadIdx.x] = s;
    gate_s[threadIdx.x] = gate[static_cast<size_t>(t) * K + threadIdx.x];
  }
  __syncthreads();
  const int nvec = d / V;
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    float acc[V], tmp[V];
    Vec<TI>::load(u + static_cast<size_t>(t) * d + v * V, acc);
    if (y_shared != nullptr) {
      load_y<V>(y_shared + static_cast<size_t>(t) * d + v * V, tmp);
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] += tmp[i];
    }
    for (int k = 0; k < K; ++k) {
      const int s = slot_s[k];
      if (s < 0) continue;
      const float g = gate_s[k];
      load_y<V>(y_perm + static_cast<size_t>(s) * d + v * V, tmp);
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] = fmaf(g, tmp[i], acc[i]);
    }
    TO* dst = h + static_cast<size_t>(t) * d + v * V;
    if constexpr (sizeof(TO) == 4) {
#pragma unroll
      for (int i = 0; i < V; i += 4)
        *reinterpret_cast<float4*>(dst + i) =
            make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < V; i += 4) {
        uint2 o;
        o.x = pack_bf16x2(acc[i], acc[i + 1]);
        o.y = pack_bf16x2(acc[i + 2], acc[i + 3]);
        *reinterpret_cast<uint2*>(dst + i) = o;
      }
    }
  }
}

__global__ void zero_i32_kernel(int* __restrict__ p, int n) {
  for (int i = threadIdx.x; i < n; i += blockDim.x) p[i] = 0;
}

// b_i <- fl32(b_i - gamma) when counts[i]*N > total_assign, fl32(b_i + gamma)
// when counts[i]*N < total_assign, unchanged otherwise.
__global__ void update_bias_kernel(const int* __restrict__ counts, int N,
                                   long long total_assign, float gamma,
                                   float* __restrict__ bias) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= N) return;
  const long long load = static_cast<long long>(counts[i]) * N;
  const float b = bias[i];
  if (load > total_assign)
    bias[i] = __fsub_rn(b, gamma);
  else if (load < total_assign)
    bias[i] = __fadd_rn(b, gamma);
}

// Packed gate/up: row r of group g = [64 gate rows | 64 up rows] block r/128.
// Intermediate column c of the group maps to (expert c / I, row c % I) of
// the source, so concatenated shared experts pack the same way.
__global__ void pack_gate_up_kernel(const uint4* __restrict__ w_gate,
                                    const uint4* __restrict__ w_up,
                                    int groups, int experts_per_group, int I,
                                    int rvec, uint4* __restrict__ out) {
  const long long rows = static_cast<long long>(groups) * 2 * experts_per_group * I;
  for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
    const long long per_group = 2LL * experts_per_group * I;
    const int g = static_cast<int>(r / per_group);
    const int rr = static_cast<int>(r % per_group);
    const int blk = rr / 128, w = rr % 128;
    const int c = blk * 64 + (w & 63);
    const int ex = g * experts_per_group + c / I;
    const int row = c % I;
    const uint4* src = (w < 64 ? w_gate : w_up) +
                       (static_cast<size_t>(ex) * I + row) * rvec;
    uint4* dst = out + static_cast<size_t>(r) * rvec;
    for (int v = threadIdx.x; v < rvec; v += blockDim.x) dst[v] = __ldg(src + v);
  }
}

// Shared down projections side by side: out[r][s*I + c] = ws_down[s][r][c].
__global__ void pack_shared_down_kernel(const uint4* __restrict__ ws_down,
                                        int S, int d, int ivec,
                                        uint4* __restrict__ out) {
  const long long rows = static_cast<long long>(S) * d;
  for (long long q = blockIdx.x; q < rows; q += gridDim.x) {
    const int s = static_cast<int>(q / d), r = static_cast<int>(q % d);
    const uint4* src = ws_down + (static_cast<size_t>(s) * d + r) * ivec;
    uint4* dst = out + (static_cast<size_t>(r) * S + s) * ivec;
    for (int v = threadIdx.x; v < ivec; v += blockDim.x) dst[v] = __ldg(src + v);
  }
}

// ------------------------------------------------------------------------
// fp32 expert FFN on the CUDA cores (fp32 has no full-precision tensor-core
// kind).  Gate/up: H[row][c] = SiLU(x.Wg[c]) * (x.Wu[c]) with the packed
// gate/up layout; row -> expert through offsets (routed) or 0 (shared).
__device__ __forceinline__ int group_of_row(const int* offsets, int n, int row) {
  int lo = 0, hi = n;   // offsets[lo] <= row < offsets[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (offsets[mid] <= row) lo = mid; else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(256)
ffn_f32_gate_up_kernel(const float* __restrict__ x, int rows,
                       const int* __restrict__ offsets, int n_groups,
                       const float* __restrict__ w_gu, int I_seg, int d,
                       float* __restrict__ H) {
  const int c = blockIdx.x * 64 + (threadIdx.x & 63);
  const int row = blockIdx.y * 4 + (threadIdx.x >> 6);
  if (c >= I_seg || row >= rows) return;
  const int g = offsets ? group_of_row(offsets, n_groups, row) : 0;
  const size_t grow = static_cast<size_t>(g) * 2 * I_seg +
                      static_cast<size_t>(c / 64) * 128 + (c & 63);
  const float* wg = w_gu + grow * d;
  const float* wu = wg + static_cast<size_t>(64) * d;
  const float* xr = x + static_cast<size_t>(row) * d;
  float a = 0.f, b = 0.f;
  for (int j = 0; j < d; ++j) {
    a = fmaf(xr[j], wg[j], a);
    b = fmaf(xr[j], wu[j], b);
  }
  H[static_cast<size_t>(row) * I_seg + c] = silu_f32(a) * b;
}

// Down: Y[row][j] = sum_c H[row][c] * Wd[g][j][c].
__global__ void __launch_bounds__(256)
ffn_f32_down_kernel(const float* __restrict__ H, int rows,
                    const int* __restrict__ offsets, int n_groups,
                    const float* __restrict__ w_down, int I_seg, int d,
                    float* __restrict__ Y) {
  const int j = blockIdx.x * 64 + (threadIdx.x & 63);
  const int row = blockIdx.y * 4 + (threadIdx.x >> 6);
  if (j >= d || row >= rows) return;
  const int g = offsets ? group_of_row(offsets, n_groups, row) : 0;
  const float* w = w_down + (static_cast<size_t>(g) * d + j) * I_seg;
  const float* hr = H + static_cast<size_t>(row) * I_seg;
  float acc = 0.f;
  for (int c = 0; c < I_seg; ++c) acc = fmaf(hr[c], w[c], acc);
  Y[static_cast<size_t>(row) * d + j] = acc;
}

}  // namespace moe
