// Bandwidth-bound kernels of the layer backward pass: the padded layout,
// the gather of the per-assignment operands with the gate gradient, the
// centroid gradient and the final input gradient.  The layer is the
// FFN-output equation of "【推理llm論文精讀】DeepSeek V3技術論文", section 2.2
// (h = u + sum_s FFN_s(u) + sum_i g_i FFN_i(u), g_i = Sigmoid(u . e_i) at the
// selected experts); the gradients are its chain rule:
//   dY = g dh_t,  dz = (dh_t . y) g (1 - g),
//   du_t = dh_t + dX_shared + sum_k (dX_k + dz_k e_k),  dE_e = sum dz x.
#pragma once
#include "common.cuh"
#include "gemm_bwd.cuh"
#include "permute.cuh"

namespace moe {

// Checks the forward's offsets (offsets[0] = 0, non-decreasing,
// offsets[N] = T*K) and writes offs[e] (= offsets when they are valid; all
// zero, with the device error word set, when not: every later kernel then
// skips all work) and offpad[e] = sum_{e'<e} roundup(cnt[e'], 64),
// offpad[N] = total; zeroes the backward GEMMs' item counters.  One CTA of
// 256 threads, N <= 1024.
__global__ void __launch_bounds__(256)
bwd_offpad_kernel(const int* __restrict__ offsets, int N, long long A,
                  int* __restrict__ offs, int* __restrict__ offpad,
                  int* __restrict__ ctr, int n_ctr) {
  __shared__ int v[1024];
  __shared__ int out[1025];
  __shared__ int wt[8];
  __shared__ int bad;
  if (threadIdx.x == 0)
    bad = (offsets[0] != 0 || static_cast<long long>(offsets[N]) != A);
  for (int i = threadIdx.x; i < n_ctr; i += blockDim.x) ctr[i] = 0;
  __syncthreads();
  for (int e = threadIdx.x; e < N; e += blockDim.x)
    if (offsets[e + 1] < offsets[e]) bad = 1;
  __syncthreads();
  if (bad && threadIdx.x == 0) report_error(ERR_CHECK, KID_BWD, 1);
  for (int e = threadIdx.x; e < N; e += blockDim.x)
    v[e] = bad ? 0 : offsets[e + 1] - offsets[e];
  __syncthreads();
  block_exclusive_scan(v, out, N, wt);
  for (int e = threadIdx.x; e <= N; e += blockDim.x) offs[e] = out[e];
  __syncthreads();
  for (int e = threadIdx.x; e < N; e += blockDim.x)
    v[e] = (v[e] + kPadRows - 1) / kPadRows * kPadRows;
  __syncthreads();
  block_exclusive_scan(v, out, N, wt);
  for (int e = threadIdx.x; e <= N; e += blockDim.x) offpad[e] = out[e];
}

// One CTA (128 threads) per token t.  Assignment k of t has slot s_k =
// inv[t,k] in the forward's order (expert e_k = topk_idx[t,k]) and padded row
// p_k = s_k - offsets[e_k] + offpad[e_k].
//   pass 1: dg_k = dh_t . y_perm[s_k] (fp32), dz_k = dg_k g_k (1 - g_k) ->
//           dz[p_k];
//   pass 2: dY[p_k] = bf16(g_k dh_t), X[p_k] = u_t.
// Vectors of 8 elements (16 bytes of bf16 / fp16) along d.
__global__ void __launch_bounds__(128)
bwd_gather_kernel(const __nv_bfloat16* __restrict__ dh,
                  const __nv_bfloat16* __restrict__ u,
                  const int* __restrict__ topk_idx,
                  const float* __restrict__ gate, const int* __restrict__ inv,
                  const int* __restrict__ offsets,
                  const int* __restrict__ offpad,
                  const __half* __restrict__ y_perm, int d, int K, int N,
                  long long A, long long A_pad, __nv_bfloat16* __restrict__ dY,
                  __nv_bfloat16* __restrict__ X, float* __restrict__ dz) {
  __shared__ int slot_s[kTopKMax], pad_s[kTopKMax];
  __shared__ float g_s[kTopKMax];
  __shared__ float red[4][kTopKMax];
  const int t = blockIdx.x, tid = threadIdx.x;
  if (tid < K) {
    const size_t a = static_cast<size_t>(t) * K + tid;
    const int e = topk_idx[a];
    int s = inv[a];
    long long pr = -1;
    if (e >= 0 && e < N && s >= offsets[e] && s < offsets[e + 1] && s < A) {
      pr = static_cast<long long>(s) - offsets[e] + offpad[e];
      if (pr >= offpad[e + 1] || pr >= A_pad) pr = -1;
    }
    if (pr < 0) {
      report_error(ERR_CHECK, KID_BWD, 2);
      s = -1;
    }
    slot_s[tid] = s;
    pad_s[tid] = static_cast<int>(pr);
    g_s[tid] = gate[a];
  }
  __syncthreads();
  const int nvec = d / 8;
  float acc[kTopKMax];
#pragma unroll
  for (int k = 0; k < kTopKMax; ++k) acc[k] = 0.f;
  for (int v = tid; v < nvec; v += blockDim.x) {
    const uint4 hv = __ldg(reinterpret_cast<const uint4*>(
        dh + static_cast<size_t>(t) * d + v * 8));
    const __nv_bfloat162* hb = reinterpret_cast<const __nv_bfloat162*>(&hv);
    float f[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x = __bfloat1622float2(hb[i]);
      f[2 * i] = x.x;
      f[2 * i + 1] = x.y;
    }
#pragma unroll
    for (int k = 0; k < kTopKMax; ++k) {
      if (k >= K) break;
      const int s = slot_s[k];
      if (s < 0) continue;
      const uint4 yv = __ldg(reinterpret_cast<const uint4*>(
          y_perm + static_cast<size_t>(s) * d + v * 8));
      const __half2* yh = reinterpret_cast<const __half2*>(&yv);
      float a = acc[k];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 y = __half22float2(yh[i]);
        a = fmaf(f[2 * i], y.x, a);
        a = fmaf(f[2 * i + 1], y.y, a);
      }
      acc[k] = a;
    }
  }
  const int warp = tid >> 5, lane = tid & 31;
#pragma unroll
  for (int k = 0; k < kTopKMax; ++k) {
    if (k >= K) break;
    float a = acc[k];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    if (lane == 0) red[warp][k] = a;
  }
  __syncthreads();
  if (tid < K) {
    const float dg = (red[0][tid] + red[1][tid]) + (red[2][tid] + red[3][tid]);
    const float g = g_s[tid];
    if (pad_s[tid] >= 0) dz[pad_s[tid]] = dg * g * (1.0f - g);
  }
  for (int v = tid; v < nvec; v += blockDim.x) {
    const size_t src = static_cast<size_t>(t) * d + v * 8;
    const uint4 hv = __ldg(reinterpret_cast<const uint4*>(dh + src));
    const uint4 uv = __ldg(reinterpret_cast<const uint4*>(u + src));
    const __nv_bfloat162* hb = reinterpret_cast<const __nv_bfloat162*>(&hv);
    float f[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x = __bfloat1622float2(hb[i]);
      f[2 * i] = x.x;
      f[2 * i + 1] = x.y;
    }
    for (int k = 0; k < K; ++k) {
      const int pr = pad_s[k];
      if (pr < 0) continue;
      const float g = g_s[k];
      uint4 o;
      o.x = pack_bf16x2(g * f[0], g * f[1]);
      o.y = pack_bf16x2(g * f[2], g * f[3]);
      o.z = pack_bf16x2(g * f[4], g * f[5]);
      o.w = pack_bf16x2(g * f[6], g * f[7]);
      const size_t dst = static_cast<size_t>(pr) * d + v * 8;
      *reinterpret_cast<uint4*>(dY + dst) = o;
      *reinterpret_cast<uint4*>(X + dst) = uv;
    }
  }
}

// Zero rows offpad[e] + cnt[e] .. offpad[e+1] of the padded operands (X, dY
// [.., d], H [.., I], dA [.., 2I]) and of dz: the Wgrad GEMMs multiply
// whole 16-row steps.  One CTA per expert.
__global__ void __launch_bounds__(256)
bwd_zero_pad_kernel(const int* __restrict__ offsets,
                    const int* __restrict__ offpad, int d, int I,
                    __nv_bfloat16* __restrict__ X,
                    __nv_bfloat16* __restrict__ dY,
                    __nv_bfloat16* __restrict__ H,
                    __nv_bfloat16* __restrict__ dA, float* __restrict__ dz) {
  const int e = blockIdx.x;
  const long long r0 =
      static_cast<long long>(offpad[e]) + (offsets[e + 1] - offsets[e]);
  const long long r1 = offpad[e + 1];
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  const int vd = d / 8, vi = I / 8;
  const int per_row = 2 * vd + 3 * vi;      // 16-byte vectors per padded row
  for (long long i = threadIdx.x; i < (r1 - r0) * per_row; i += blockDim.x) {
    const long long r = r0 + i / per_row;
    int c = static_cast<int>(i % per_row);
    if (c < vd) {
      reinterpret_cast<uint4*>(X + r * d)[c] = z;
    } else if ((c -= vd) < vd) {
      reinterpret_cast<uint4*>(dY + r * d)[c] = z;
    } else if ((c -= vd) < vi) {
      reinterpret_cast<uint4*>(H + r * I)[c] = z;
    } else {
      c -= vi;
      reinterpret_cast<uint4*>(dA + r * 2 * I)[c] = z;
    }
  }
  for (long long r = r0 + threadIdx.x; r < r1; r += blockDim.x) dz[r] = 0.f;
}

// dE[e][j] = sum over the rows m of expert e of dz[m] * X[m][j] (fp32, rows
// in order).  Grid (N, ceil(d / 1024)), 128 threads x 8 columns.
__global__ void __launch_bounds__(128)
bwd_centroid_grad_kernel(const int* __restrict__ offsets,
                         const int* __restrict__ offpad,
                         const float* __restrict__ dz,
                         const __nv_bfloat16* __restrict__ X, int d,
                         float* __restrict__ dE) {
  const int e = blockIdx.x;
  const int j0 = (blockIdx.y * blockDim.x + threadIdx.x) * 8;
  if (j0 >= d) return;
  const long long r0 = offpad[e];
  const long long r1 = r0 + (offsets[e + 1] - offsets[e]);
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll 4
  for (long long r = r0; r < r1; ++r) {
    const float z = __ldg(dz + r);
    const uint4 xv = __ldg(reinterpret_cast<const uint4*>(X + r * d + j0));
    const __nv_bfloat162* xb = reinterpret_cast<const __nv_bfloat162*>(&xv);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x = __bfloat1622float2(xb[i]);
      acc[2 * i] = fmaf(z, x.x, acc[2 * i]);
      acc[2 * i + 1] = fmaf(z, x.y, acc[2 * i + 1]);
    }
  }
  float* dst = dE + static_cast<size_t>(e) * d + j0;
  *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
  *reinterpret_cast<float4*>(dst + 4) =
      make_float4(acc[4], acc[5], acc[6], acc[7]);
}

__device__ __forceinline__ void add_half8(const __half* p, float* f) {
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
  const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 x = __half22float2(h[i]);
    f[2 * i] += x.x;
    f[2 * i + 1] += x.y;
  }
}

// du[t] = dh[t] + dX_s[t] + sum_k (dX[p_k] + dz[p_k] E[e_k]), fp32, in that
// order.  One CTA (128 threads) per token, 8 columns per vector.
__global__ void __launch_bounds__(128)
bwd_input_grad_kernel(const __nv_bfloat16* __restrict__ dh,
                      const __half* __restrict__ dX_s,
                      const __half* __restrict__ dX,
                      const __nv_bfloat16* __restrict__ E,
                      const float* __restrict__ dz,
                      const int* __restrict__ topk_idx,
                      const int* __restrict__ inv,
                      const int* __restrict__ offsets,
                      const int* __restrict__ offpad, int d, int K, int N,
                      long long A, float* __restrict__ du) {
  __shared__ int pad_s[kTopKMax], e_s[kTopKMax];
  __shared__ float z_s[kTopKMax];
  const int t = blockIdx.x, tid = threadIdx.x;
  if (tid < K) {
    const size_t a = static_cast<size_t>(t) * K + tid;
    const int e = topk_idx[a];
    const int s = inv[a];
    int pr = -1;
    if (e >= 0 && e < N && s >= offsets[e] && s < offsets[e + 1] && s < A)
      pr = s - offsets[e] + offpad[e];
    pad_s[tid] = pr;
    e_s[tid] = pr >= 0 ? e : 0;
    z_s[tid] = pr >= 0 ? dz[pr] : 0.f;
  }
  __syncthreads();
  const int nvec = d / 8;
  for (int v = tid; v < nvec; v += blockDim.x) {
    const size_t off = static_cast<size_t>(t) * d + v * 8;
    float f[8];
    const uint4 hv = __ldg(reinterpret_cast<const uint4*>(dh + off));
    const __nv_bfloat162* hb = reinterpret_cast<const __nv_bfloat162*>(&hv);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x = __bfloat1622float2(hb[i]);
      f[2 * i] = x.x;
      f[2 * i + 1] = x.y;
    }
    if (dX_s != nullptr) add_half8(dX_s + off, f);
    for (int k = 0; k < K; ++k) {
      const int pr = pad_s[k];
      if (pr < 0) continue;
      add_half8(dX + static_cast<size_t>(pr) * d + v * 8, f);
      const float z = z_s[k];
      const uint4 ev = __ldg(reinterpret_cast<const uint4*>(
          E + static_cast<size_t>(e_s[k]) * d + v * 8));
      const __nv_bfloat162* eb = reinterpret_cast<const __nv_bfloat162*>(&ev);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 x = __bfloat1622float2(eb[i]);
        f[2 * i] = fmaf(z, x.x, f[2 * i]);
        f[2 * i + 1] = fmaf(z, x.y, f[2 * i + 1]);
      }
    }
    float* dst = du + off;
    *reinterpret_cast<float4*>(dst) = make_float4(f[0], f[1], f[2], f[3]);
    *reinterpret_cast<float4*>(dst + 4) = make_float4(f[4], f[5], f[6], f[7]);
  }
}

}  // namespace moe
