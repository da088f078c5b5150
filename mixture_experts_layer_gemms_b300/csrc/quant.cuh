// e4m3 block quantization of weights and activations.
// (DeepSeek-V3 report commentary, cooktownmusic.com, FP8 training-framework
// part, Fig. 7a: activations and weights are grouped into blocks and each
// block is scaled on its own.)
//
// Blocks: 1 x 128 for activations (one row, 128 consecutive channels of the
// reduction dimension), 128 x 128 for weights.  A block with largest
// magnitude a gets the scale 2^e, e the smallest integer with a <= 448 * 2^e
// (e = 0 for an all-zero block); its codes are e4m3(x * 2^-e), rounded to
// nearest even and saturated at +-448 (the conversion instruction's
// satfinite mode).  x * 2^-e is exact, so GPU and CPU codes agree bit for
// bit.  Scales are stored as fp32 powers of two and, for the block-scaled
// tensor-core kernels, once more as UE8M0 bytes (the biased exponent,
// 127 + e) in a row-major [R][P] table: R = rows for activations (one byte
// per row and 128-block of the reduction), R = row blocks for weights;
// P = the block count rounded up to 16, the padding bytes 127 (2^0), so a
// row of the table is a 16-byte multiple.  Exponents outside [-126, 126]
// (block maxima beyond the fp32 power-of-two range) are reported as a
// device check and the block is written as zeros.
#pragma once
#include <cuda_fp8.h>
#include "common.cuh"

namespace moe {

constexpr int kQBlock = 128;

__device__ __forceinline__ int e4m3_scale_exp(float amax) {
  if (!(amax > 0.f)) return 0;
  int ex;
  const float m = frexpf(amax, &ex);      // amax = m 2^ex, m in [0.5, 1)
  return m <= 0.875f ? ex - 9 : ex - 8;   // 448 = 0.875 * 2^9
}

__device__ __forceinline__ float pow2f(int e) {   // exact for |e| <= 126
  return __int_as_float((127 + e) << 23);
}

// Row stride (bytes) of a UE8M0 scale table for a reduction of k elements.
__host__ __device__ __forceinline__ int ue8_pitch(long long k) {
  return static_cast<int>(((k / kQBlock) + 15) / 16 * 16);
}
// UE8M0 byte of a stored fp32 power-of-two scale (0 for the zero written
// after a reported bad exponent).
__device__ __forceinline__ uint8_t ue8_of(float s) {
  return static_cast<uint8_t>((__float_as_uint(s) >> 23) & 0xFFu);
}

__device__ __forceinline__ uint32_t e4m3_code(float x, float inv_scale) {
  return static_cast<uint32_t>(
      __nv_cvt_float_to_fp8(x * inv_scale, __NV_SATFINITE, __NV_E4M3));
}

// Largest |v| of a warp's values (non-negative floats order like their bits).
__device__ __forceinline__ float warp_amax(float v) {
  return __uint_as_float(
      __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v))));
}

// Four bf16 values (8 bytes) -> four e4m3 codes (one 32-bit word), given the
// block's scale exponent.
__device__ __forceinline__ uint32_t quant4(const float* f, float inv) {
  return e4m3_code(f[0], inv) | (e4m3_code(f[1], inv) << 8) |
         (e4m3_code(f[2], inv) << 16) | (e4m3_code(f[3], inv) << 24);
}

__device__ __forceinline__ void load4_bf16(const __nv_bfloat16* p, float* f) {
  const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
  const float2 a = __bfloat1622float2(h[0]), b = __bfloat1622float2(h[1]);
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
}

// One warp quantizes one 1 x 128 block held as 4 values per lane; returns the
// lane's 4 codes and sets *scale (same on every lane).  A bad exponent is
// reported and gives zero codes.
__device__ __forceinline__ uint32_t warp_quant_block(const float* f,
                                                     float* scale) {
  float a = fmaxf(fmaxf(fabsf(f[0]), fabsf(f[1])), fmaxf(fabsf(f[2]), fabsf(f[3])));
  a = warp_amax(a);
  const int e = e4m3_scale_exp(a);
  if (e < -126 || e > 126) {
    if ((threadIdx.x & 31) == 0) report_error(ERR_CHECK, KID_QUANT, 1);
    *scale = 0.f;
    return 0u;
  }
  *scale = pow2f(e);
  return quant4(f, pow2f(-e));
}

__device__ __forceinline__ void load4_f32(const float* p, float* f) {
  const float4 v = __ldg(reinterpret_cast<const float4*>(p));
  f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* p, float* f) {
  load4_bf16(p, f);
}
__device__ __forceinline__ void load4(const float* p, float* f) {
  load4_f32(p, f);
}

// Activations: x (bf16 or fp32) [R, K] row-major -> codes [R, K] and scales
// [K/128][ld_s] (column index = row), one warp per (row, block).
// ue8 (optional): UE8M0 table [R][ue8_pitch(K)].
template <typename TX>
__global__ void __launch_bounds__(256)
quantize_rows_kernel(const TX* __restrict__ x, int R, int K,
                     uint8_t* __restrict__ q, float* __restrict__ scales,
                     long long ld_s, uint8_t* __restrict__ ue8 = nullptr) {
  const int nb = K / kQBlock;
  const long long w = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) +
                      (threadIdx.x >> 5);
  if (w >= static_cast<long long>(R) * nb) return;
  const int lane = threadIdx.x & 31;
  const long long r = w / nb;
  const int b = static_cast<int>(w % nb);
  const size_t off = static_cast<size_t>(r) * K + b * kQBlock + 4 * lane;
  float f[4];
  load4(x + off, f);
  float sc;
  const uint32_t c = warp_quant_block(f, &sc);
  *reinterpret_cast<uint32_t*>(q + off) = c;
  if (lane == 0) scales[static_cast<size_t>(b) * ld_s + r] = sc;
  if (ue8 != nullptr) {
    const int P = ue8_pitch(K);
    uint8_t* row = ue8 + static_cast<size_t>(r) * P;
    if (lane == 0) row[b] = ue8_of(sc);
    if (b == nb - 1)                       // padding of the row
      for (int j = nb + lane; j < P; j += 32) row[j] = 127;
  }
}

// Dispatch fused with quantization: x8[inv[t,k]] = codes of u[t] for every
// k, scales sx[b][inv[t,k]].  One warp per (token, 1 x 128 block): the block
// is quantized once and written K times.
__global__ void __launch_bounds__(256)
permute_gather_fp8_kernel(const __nv_bfloat16* __restrict__ u,
                          const int* __restrict__ inv, int T, int K, int d,
                          long long total_slots, uint8_t* __restrict__ x8,
                          float* __restrict__ sx,
                          uint8_t* __restrict__ ue8 = nullptr) {
  const int lane = threadIdx.x & 31;
  const int nb = d / kQBlock;
  const long long nwarps =
      static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long w = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) +
                     (threadIdx.x >> 5);
       w < static_cast<long long>(T) * nb; w += nwarps) {
    const int t = static_cast<int>(w / nb), b = static_cast<int>(w % nb);
    // lane k < K holds the slot of assignment (t, k)
    int myslot = lane < K ? inv[static_cast<size_t>(t) * K + lane] : -1;
    if (lane < K && (myslot < 0 || myslot >= total_slots)) {
      if (b == 0) report_error(ERR_CHECK, KID_QUANT, 2);
      myslot = -1;
    }
    float f[4];
    load4_bf16(u + static_cast<size_t>(t) * d + b * kQBlock + 4 * lane, f);
    float sc;
    const uint32_t c = warp_quant_block(f, &sc);
    for (int k = 0; k < K; ++k) {
      const int s = __shfl_sync(0xffffffffu, myslot, k);
      if (s >= 0)
        *reinterpret_cast<uint32_t*>(
            x8 + static_cast<size_t>(s) * d + b * kQBlock + 4 * lane) = c;
    }
    if (myslot >= 0) sx[static_cast<size_t>(b) * total_slots + myslot] = sc;
    if (ue8 != nullptr) {
      const int P = ue8_pitch(d);
      for (int k = 0; k < K; ++k) {
        const int s = __shfl_sync(0xffffffffu, myslot, k);
        if (s < 0) continue;
        uint8_t* row = ue8 + static_cast<size_t>(s) * P;
        if (lane == 0) row[b] = ue8_of(sc);
        if (b == nb - 1)
          for (int j = nb + lane; j < P; j += 32) row[j] = 127;
      }
    }
  }
}

// Weights: one CTA (256 threads) per 128 x 128 destination block.  The
// destination is a row-major code matrix [rows, K] (row stride K) with
// scales [rows/128][K/128]; the source rows of destination row block rb and
// column block cb depend on `mode`:
//   0 identity:       src rows rb*128.., cols cb*128.., row stride K;
//   1 gate/up:        destination row blocks alternate gate and up blocks of
//                     the same 128 intermediate rows (rb = 2 j + gu):
//                     src = (gu ? up : gate) rows (rb/2)*128.. of a matrix
//                     [I_total, K] whose rows are the intermediate index;
//   2 shared down:    the shared experts' down matrices [S][d][I] side by
//                     side along K: destination [d, S*I], cb -> expert
//                     cb*128 / I, column (cb*128) % I; src row stride I.
__global__ void __launch_bounds__(256)
quantize_weight_blocks_kernel(const __nv_bfloat16* __restrict__ src0,
                              const __nv_bfloat16* __restrict__ src1,
                              int mode, int K, int I, int d,
                              uint8_t* __restrict__ q,
                              float* __restrict__ scales,
                              uint8_t* __restrict__ ue8 = nullptr) {
  __shared__ float red[8];
  const int cb = blockIdx.x, rb = blockIdx.y;
  const int nkb = K / kQBlock;
  const __nv_bfloat16* src;
  long long ld;
  if (mode == 0) {
    src = src0 + (static_cast<size_t>(rb) * kQBlock) * K + cb * kQBlock;
    ld = K;
  } else if (mode == 1) {
    src = ((rb & 1) ? src1 : src0) +
          (static_cast<size_t>(rb >> 1) * kQBlock) * K + cb * kQBlock;
    ld = K;
  } else {
    const int s = (cb * kQBlock) / I, c0 = (cb * kQBlock) % I;
    src = src0 + static_cast<size_t>(s) * d * I +
          static_cast<size_t>(rb) * kQBlock * I + c0;
    ld = I;
  }
  // thread t: row t / 2, 64 columns from (t % 2) * 64
  const int r = threadIdx.x >> 1, c = (threadIdx.x & 1) * 64;
  const __nv_bfloat16* p = src + static_cast<size_t>(r) * ld + c;
  float f[64];
#pragma unroll
  for (int i = 0; i < 64; i += 4) load4_bf16(p + i, f + i);
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < 64; ++i) a = fmaxf(a, fabsf(f[i]));
  a = warp_amax(a);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
  __syncthreads();
  a = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) a = fmaxf(a, red[i]);
  const int e = e4m3_scale_exp(a);
  const bool ok = e >= -126 && e <= 126;
  if (!ok && threadIdx.x == 0) report_error(ERR_CHECK, KID_QUANT, 3);
  const float inv = ok ? pow2f(-e) : 0.f;
  uint8_t* dst = q + (static_cast<size_t>(rb) * kQBlock + r) * K +
                 cb * kQBlock + c;
#pragma unroll
  for (int i = 0; i < 64; i += 16) {
    uint4 w;
    w.x = quant4(f + i, inv);
    w.y = quant4(f + i + 4, inv);
    w.z = quant4(f + i + 8, inv);
    w.w = quant4(f + i + 12, inv);
    *reinterpret_cast<uint4*>(dst + i) = w;
  }
  if (threadIdx.x == 0)
    scales[static_cast<size_t>(rb) * nkb + cb] = ok ? pow2f(e) : 0.f;
  if (ue8 != nullptr) {
    const int P = ue8_pitch(K);
    uint8_t* row = ue8 + static_cast<size_t>(rb) * P;
    if (threadIdx.x == 0) row[cb] = ue8_of(ok ? pow2f(e) : 0.f);
    if (cb == nkb - 1)
      for (int j = nkb + static_cast<int>(threadIdx.x); j < P;
           j += static_cast<int>(blockDim.x))
        row[j] = 127;
  }
}

}  // namespace moe
