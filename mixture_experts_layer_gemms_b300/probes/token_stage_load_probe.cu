// Load-throughput probe (not part of the library): how fast can a CTA fill
// 32 KB token stages (128 rows x 2 K-atoms of bf16) when the rows are
// (0) contiguous: one tiled 3-D TMA box, (1) gathered: 64 tile::gather4 TMA
// loads from one thread, (2) the same 64 spread over the 32 lanes of a warp,
// (3) over 64 threads of two warps, (4) gathered by 128 threads with 16-byte
// cp.async (manual swizzle).  One CTA per SM, 4-stage ring, a consumer
// thread that releases each stage as soon as it lands (no MMA): pure load
// throughput.  Every wait is bounded (2 s of globaltimer); a timeout sets a
// flag and the kernel unwinds.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdio>
#include <cstdlib>
#include <cstdint>
#include <vector>
#include <algorithm>
#include <random>

#define CK(x) do { cudaError_t e = (x); if (e != cudaSuccess) { printf("CUDA %s at %d\n", cudaGetErrorString(e), __LINE__); exit(1);} } while (0)

constexpr int T = 8192, D = 7168;
constexpr int ROWS = 128, ATOMS = 2;
constexpr int STAGE = ROWS * ATOMS * 128;   // 32 KB
constexpr int NST = 4;
constexpr int STEPS = 2000;
constexpr int KSTAGES = D / 64 / ATOMS;     // 56 stages per row set
constexpr unsigned long long LIMIT = 2000000000ull;

__device__ int g_err = 0;

__device__ __forceinline__ unsigned long long gtime() {
  unsigned long long t; asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)); return t;
}
__device__ __forceinline__ uint32_t su32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void minit(uint32_t b, uint32_t c) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(b), "r"(c));
}
__device__ __forceinline__ void marrive(uint32_t b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(b) : "memory");
}
__device__ __forceinline__ void mexpect(uint32_t b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(b), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mtry(uint32_t b, uint32_t ph) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0,1,0,p;\n\t}"
               : "=r"(ok) : "r"(b), "r"(ph) : "memory");
  return ok;
}
__device__ __forceinline__ bool mwait(uint32_t b, uint32_t ph, volatile int* abort) {
  unsigned long long t0 = gtime();
  while (!mtry(b, ph)) {
    if (*abort) return false;
    if (gtime() - t0 > LIMIT) { *abort = 1; atomicExch(&g_err, 1); return false; }
  }
  return true;
}

__global__ void __launch_bounds__(160, 1)
probe_kernel(const __grid_constant__ CUtensorMap tm3, const __grid_constant__ CUtensorMap tm1,
             const __nv_bfloat16* __restrict__ u, const int* __restrict__ rows,
             int mode, unsigned long long* times) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t bars[2 * NST];
  __shared__ int abort_s;
  const uint32_t full = su32(&bars[0]), empty = su32(&bars[NST]);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // producers: mode 0/1: thread 0; mode 2: warp 0; mode 3: warps 0-1; mode 4: warps 0-3
  const int nprod = mode <= 1 ? 1 : (mode == 2 ? 32 : (mode == 3 ? 64 : 128));
  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      minit(full + 8 * s, mode == 4 ? 128 : 1);
      minit(empty + 8 * s, 1);
    }
    abort_s = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  volatile int* abort = &abort_s;
  const unsigned long long t0 = gtime();
  if (tid < nprod) {
    for (int i = 0; i < STEPS; ++i) {
      const int s = i % NST;
      const uint32_t ph = (i / NST) & 1;
      if (!mwait(empty + 8 * s, ph ^ 1, abort)) break;
      const int set = i / KSTAGES, ks = i % KSTAGES;
      const int* r = rows + (size_t)((blockIdx.x * 131 + set) % 512) * ROWS;   // a row set
      const uint32_t dst = su32(smem + s * STAGE);
      const int ka = ks * ATOMS;
      if (mode == 0) {
        mexpect(full + 8 * s, STAGE);
        asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                     " [%0], [%1, {%3, %4, %5}], [%2];"
                     :: "r"(dst), "l"((uint64_t)&tm3), "r"(full + 8 * s), "r"(0), "r"(r[0]), "r"(ka) : "memory");
      } else if (mode <= 3) {
        // the expect-tx arrival is the phase's only arrival, so bytes that
        // land before it cannot complete the phase early
        if (tid == 0) mexpect(full + 8 * s, STAGE);
        for (int j = tid; j < 64; j += nprod) {        // 64 gather4 = 256 rows x 1 atom
          const int a = j >> 5, g = j & 31;
          const int* rr = r + 4 * g;
          asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
                       " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];"
                       :: "r"(dst + a * (ROWS * 128) + g * 512), "l"((uint64_t)&tm1), "r"(full + 8 * s),
                          "r"((ka + a) * 64), "r"(rr[0]), "r"(rr[1]), "r"(rr[2]), "r"(rr[3]) : "memory");
        }
      } else {
        // 2048 16-byte pieces: row = c >> 4, piece p = c & 15 (atom p >> 3)
        for (int c = tid; c < ROWS * 16; c += 128) {
          const int row = c >> 4, p = c & 15, a = p >> 3, w = p & 7;
          const uint32_t d = dst + a * (ROWS * 128) + row * 128 + ((w ^ (row & 7)) << 4);
          const __nv_bfloat16* src = u + (size_t)r[row] * D + (ka + a) * 64 + w * 8;
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(d), "l"(src) : "memory");
        }
        asm volatile("cp.async.mbarrier.arrive.noinc.shared.b64 [%0];" :: "r"(full + 8 * s) : "memory");
      }
    }
  } else if (tid == 128) {     // consumer
    for (int i = 0; i < STEPS; ++i) {
      const int s = i % NST;
      if (!mwait(full + 8 * s, (i / NST) & 1, abort)) break;
      marrive(empty + 8 * s);
    }
  }
  if (mode == 4) asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  if (tid == 0) {
    times[blockIdx.x] = gtime() - t0;
    // error path only: give TMA loads still in flight time to land (bounded)
    if (*abort) {
      const unsigned long long ts = gtime();
      while (gtime() - ts < 100000000ull) {}
    }
  }
  __syncthreads();
}

typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                             const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                             CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int main() {
  int sms = 0;
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  CK(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q));
  EncodeFn enc = (EncodeFn)fn;
  __nv_bfloat16* u;
  CK(cudaMalloc(&u, (size_t)T * D * 2));
  CK(cudaMemset(u, 0, (size_t)T * D * 2));
  // 512 row sets of 128 sorted random rows (like an expert's tokens)
  std::mt19937 rng(7);
  std::vector<int> h(512 * ROWS);
  for (int s = 0; s < 512; ++s) {
    std::vector<int> v(ROWS);
    for (auto& x : v) x = rng() % T;
    std::sort(v.begin(), v.end());
    // the contiguous mode starts at the set's first row, clamped in range
    v[0] = std::min(v[0], T - ROWS);
    for (int i = 0; i < ROWS; ++i) h[s * ROWS + i] = v[i];
  }
  int* rows;
  CK(cudaMalloc(&rows, h.size() * 4));
  CK(cudaMemcpy(rows, h.data(), h.size() * 4, cudaMemcpyHostToDevice));
  CUtensorMap tm3, tm1;
  {
    cuuint64_t dims[3] = {64, (cuuint64_t)T, (cuuint64_t)(D / 64)};
    cuuint64_t str[2] = {(cuuint64_t)D * 2, 128};
    cuuint32_t box[3] = {64, ROWS, ATOMS}, es[3] = {1, 1, 1};
    if (enc(&tm3, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, u, dims, str, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE)) {
      printf("encode3 failed\n"); return 1; }
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)T};
    cuuint64_t str[1] = {(cuuint64_t)D * 2};
    cuuint32_t box[2] = {64, 1}, es[2] = {1, 1};
    // gather4 destinations are 512-byte aligned (4 rows of 128 B): no swizzle
    if (enc(&tm1, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, u, dims, str, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE)) {
      printf("encode1 failed\n"); return 1; }
  }
  const int smem = NST * STAGE + 1024;
  CK(cudaFuncSetAttribute(probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  unsigned long long* times;
  CK(cudaMalloc(&times, sms * 8));
  const char* names[5] = {"tiled 3-D box, 128 contiguous rows x 2 atoms, 1 thread",
                          "64 tile::gather4 (4 rows x 1 atom), 1 thread",
                          "64 tile::gather4 over the 32 lanes of one warp",
                          "64 tile::gather4 over 64 threads (2 warps)",
                          "cp.async 16 B x 2048 over 128 threads (4 warps)"};
  for (int mode = 0; mode < 5; ++mode) {
    for (int rep = 0; rep < 2; ++rep) {
      cudaEvent_t e0, e1;
      CK(cudaEventCreate(&e0)); CK(cudaEventCreate(&e1));
      CK(cudaEventRecord(e0));
      probe_kernel<<<sms, 160, smem>>>(tm3, tm1, u, rows, mode, times);
      CK(cudaEventRecord(e1));
      CK(cudaEventSynchronize(e1));
      CK(cudaGetLastError());
      float ms = 0; CK(cudaEventElapsedTime(&ms, e0, e1));
      int err = 0; CK(cudaMemcpyFromSymbol(&err, g_err, 4));
      if (rep == 1)
        printf("mode %d (%s): %.3f ms, %.3f us per stage per CTA, %.2f TB/s into shared memory%s\n", mode,
               names[mode], ms, ms * 1e3 / STEPS, (double)sms * STEPS * STAGE / (ms * 1e-3) / 1e12,
               err ? "  [TIMEOUT]" : "");
      if (err) return 2;
    }
  }
  return 0;
}
