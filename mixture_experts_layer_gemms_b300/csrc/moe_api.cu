// C ABI of the MoE layer forward (declared in include/moe_b300.h):
// argument validation, workspace layout, TMA descriptors and kernel
// launches on the caller's stream.  One translation unit holds every kernel.
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "common.cuh"
#include "elementwise.cuh"
#include "gemm.cuh"
#include "gemm2sm.cuh"
#include "permute.cuh"
#include "route.cuh"
#include "gemm_fp8.cuh"
#include "gemm_fp8_pair.cuh"
#include "bwd.cuh"
#include "gemm_bwd.cuh"
#include "gemm_bwd2sm.cuh"
#include "moe_b300.h"

using namespace moe;

namespace {

thread_local std::string g_detail;
thread_local int g_launches = 0;

moe_status fail(moe_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_detail = buf;
  return st;
}

#define MOE_CHECK_CUDA(call)                                                 \
  do {                                                                       \
    cudaError_t e_ = (call);                                                 \
    if (e_ != cudaSuccess)                                                   \
      return fail(MOE_ERR_CUDA, "%s: %s (%s:%d)", #call,                      \
                  cudaGetErrorString(e_), __FILE__, __LINE__);               \
  } while (0)

#define MOE_CHECK_LAUNCH()                                                   \
  do {                                                                       \
    cudaError_t e_ = cudaGetLastError();                                     \
    if (e_ != cudaSuccess)                                                   \
      return fail(MOE_ERR_CUDA, "launch: %s (%s:%d)", cudaGetErrorString(e_), \
                  __FILE__, __LINE__);                                       \
    ++g_launches;                                                            \
  } while (0)

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool init = false;
  int sm_count = 0;
  int pair_clusters = 0;   // co-resident clusters of the CTA-pair GEMM
  int bwd_pair_clusters = 0;   // same for the backward's CTA-pair GEMM
  int f8_pair_clusters = 0;    // same for the e4m3 CTA-pair GEMM
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

template <typename K>
cudaError_t allow_smem(K kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              bytes);
}

// Per-device one-time set-up: SM count and the dynamic shared-memory limits
// of the TMA/tcgen05 kernels.
moe_status device_setup(int* sm_count) {
  int dev = 0;
  MOE_CHECK_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices)
    return fail(MOE_ERR_UNSUPPORTED, "device index %d", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& di = g_dev[dev];
  if (!di.init) {
    MOE_CHECK_CUDA(cudaDeviceGetAttribute(&di.sm_count,
                                          cudaDevAttrMultiProcessorCount, dev));
    MOE_CHECK_CUDA(allow_smem(route_tc_kernel, RouteTcSmemLayout::alloc));
    MOE_CHECK_CUDA(allow_smem(grouped_gemm_kernel<256, 4>,
                              GemmSmem<256, 4>::alloc));
    MOE_CHECK_CUDA(allow_smem(grouped_gemm_kernel<32, 10>,
                              GemmSmem<32, 10>::alloc));
    MOE_CHECK_CUDA(allow_smem(grouped_gemm_pair_kernel, PairSmem::alloc));
#define MOE_FP8_SMEM(BN, CW, TWO, SW, ST)                                  \
  MOE_CHECK_CUDA(allow_smem(grouped_gemm_fp8_kernel<BN, CW, TWO, SW, ST>, \
                            Fp8Smem<BN, CW, TWO, ST>::alloc))
    MOE_FP8_SMEM(32, 1, true, true, 6);
    MOE_FP8_SMEM(32, 1, true, false, 6);
    MOE_FP8_SMEM(32, 1, false, false, 10);
    MOE_FP8_SMEM(128, 2, true, true, 4);
    MOE_FP8_SMEM(128, 2, true, false, 4);
    MOE_FP8_SMEM(128, 2, false, false, 6);
#undef MOE_FP8_SMEM
    MOE_CHECK_CUDA(allow_smem(bwd_gemm_kernel<kDgrad, 256, 4>,
                              BwdSmem<256, 4>::alloc));
    MOE_CHECK_CUDA(allow_smem(bwd_gemm_kernel<kRecomp, 256, 4>,
                              BwdSmem<256, 4>::alloc));
    MOE_CHECK_CUDA(allow_smem(bwd_gemm_kernel<kWgrad, 256, 4>,
                              BwdSmem<256, 4>::alloc));
    MOE_CHECK_CUDA(allow_smem(bwd_gemm_kernel<kWgrad, 128, 6>,
                              BwdSmem<128, 6>::alloc));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (di.sm_count / 2));
    cfg.blockDim = dim3(192);
    cfg.dynamicSmemBytes = PairSmem::alloc;
    int clusters = 0;
    MOE_CHECK_CUDA(cudaOccupancyMaxActiveClusters(
        &clusters, grouped_gemm_pair_kernel, &cfg));
    di.pair_clusters = clusters;
    MOE_CHECK_CUDA(allow_smem(bwd_gemm_pair_kernel<kDgrad>,
                              BwdPairSmem<kDgrad>::alloc));
    MOE_CHECK_CUDA(allow_smem(bwd_gemm_pair_kernel<kRecomp>,
                              BwdPairSmem<kRecomp>::alloc));
    MOE_CHECK_CUDA(allow_smem(bwd_gemm_pair_kernel<kWgrad>,
                              BwdPairSmem<kWgrad>::alloc));
    cfg.dynamicSmemBytes = BwdPairSmem<kWgrad>::alloc;
    cfg.blockDim = dim3(bwd_pair_threads<kWgrad>());
    clusters = 0;
    MOE_CHECK_CUDA(cudaOccupancyMaxActiveClusters(
        &clusters, bwd_gemm_pair_kernel<kWgrad>, &cfg));
    di.bwd_pair_clusters = clusters;
    MOE_CHECK_CUDA(allow_smem(grouped_gemm_fp8_pair_kernel, F8PairSmem::alloc));
    cfg.dynamicSmemBytes = F8PairSmem::alloc;
    cfg.blockDim = dim3(kF8PThreads);
    clusters = 0;
    MOE_CHECK_CUDA(cudaOccupancyMaxActiveClusters(
        &clusters, grouped_gemm_fp8_pair_kernel, &cfg));
    di.f8_pair_clusters = clusters;
    di.init = true;
  }
  *sm_count = di.sm_count;
  return MOE_OK;
}

int bwd_pair_clusters() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return 0;
  return g_dev[dev].bwd_pair_clusters;
}

int f8_pair_clusters() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return 0;
  return g_dev[dev].f8_pair_clusters;
}

int pair_clusters() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return 0;
  return g_dev[dev].pair_clusters;
}

moe_status get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (g_encode == nullptr)
    return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  return MOE_OK;
}

// 2-D bf16 K-major operand [rows, cols] (cols contiguous), 128-byte swizzle,
// box {64, box_rows}; out-of-range rows read as zero.
moe_status make_map(CUtensorMap* m, const void* ptr, long long rows,
                    long long cols, int box_rows) {
  moe_status st = get_encoder();
  if (st != MOE_OK) return st;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols),
                        static_cast<cuuint64_t>(rows > 0 ? rows : 1)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                        const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) rows=%lld "
                "cols=%lld box_rows=%d", static_cast<int>(r), rows, cols,
                box_rows);
  return MOE_OK;
}

// 3-D view of a K-major bf16 operand [rows, cols] as {64, rows, cols/64}
// with a box of {64, box_rows, atoms}: `atoms` consecutive 64-wide K-atoms
// of box_rows rows in one TMA load, stacked atom-major in shared memory,
// 128-byte swizzle.
moe_status make_map3(CUtensorMap* m, const void* ptr, long long rows,
                     long long cols, int box_rows, int atoms) {
  moe_status st = get_encoder();
  if (st != MOE_OK) return st;
  cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows > 0 ? rows : 1),
                        static_cast<cuuint64_t>(cols / 64)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2, 128};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows),
                       static_cast<cuuint32_t>(atoms)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                        const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled (3-D) failed (%d) "
                "rows=%lld cols=%lld box_rows=%d", static_cast<int>(r), rows,
                cols, box_rows);
  return MOE_OK;
}

// element size of activations (and of weights, except for MOE_FP8)
// e4m3 codes [rows, cols] (one byte each), box {128 bytes, box_rows},
// 128-byte swizzle.
moe_status make_map_u8(CUtensorMap* m, const void* ptr, long long rows,
                       long long cols, int box_rows) {
  moe_status st = get_encoder();
  if (st != MOE_OK) return st;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols),
                        static_cast<cuuint64_t>(rows > 0 ? rows : 1)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols)};
  cuuint32_t box[2] = {128, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                        const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled (u8) failed (%d) "
                "rows=%lld cols=%lld box_rows=%d", static_cast<int>(r), rows,
                cols, box_rows);
  return MOE_OK;
}

size_t elem_size(moe_dtype dt) { return dt == MOE_F32 ? 4 : 2; }

bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

inline long long cdiv(long long a, long long b) { return (a + b - 1) / b; }
inline size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// e4m3 operand buffers [rows, cols] (cols = the reduction): the codes, then
// at the next 256-byte boundary the fp32 scales, then at the next 256-byte
// boundary the same scales as a UE8M0 table [R][ue8_pitch(cols)].
// Activations: scales [cols/128][rows], R = rows.  Weights: scales
// [rows/128][cols/128], R = rows/128.
inline size_t fp8_codes_bytes(long long rows, long long cols) {
  return round256(static_cast<size_t>(rows) * cols);
}
inline size_t fp8_scales_bytes(long long rows, long long cols, bool weights) {
  return round256(static_cast<size_t>(weights ? rows / 128 : rows) *
                  (cols / 128) * 4);
}
inline size_t fp8_ue8_bytes(long long rows, long long cols, bool weights) {
  return round256(static_cast<size_t>(weights ? rows / 128 : rows) *
                  ue8_pitch(cols));
}
inline size_t fp8_buf_bytes(long long rows, long long cols, bool weights) {
  return fp8_codes_bytes(rows, cols) + fp8_scales_bytes(rows, cols, weights) +
         fp8_ue8_bytes(rows, cols, weights);
}
inline uint8_t* fp8_ue8(const void* base, long long rows, long long cols,
                        bool weights) {
  return static_cast<uint8_t*>(const_cast<void*>(base)) +
         fp8_codes_bytes(rows, cols) + fp8_scales_bytes(rows, cols, weights);
}

moe_status check_shape(const moe_shape* s) {
  if (s == nullptr) return fail(MOE_ERR_INVALID_ARG, "shape is NULL");
  if (s->dtype != MOE_F32 && s->dtype != MOE_BF16 && s->dtype != MOE_FP8)
    return fail(MOE_ERR_INVALID_ARG, "dtype %d", static_cast<int>(s->dtype));
  if (s->T < 0 || s->d <= 0 || s->n_routed <= 0 || s->top_k <= 0 ||
      s->n_shared < 0 || s->d_ff <= 0)
    return fail(MOE_ERR_INVALID_ARG, "non-positive size in shape");
  if (s->d % 128 != 0)
    return fail(MOE_ERR_UNSUPPORTED, "d=%d must be a multiple of 128", s->d);
  if (s->d_ff % 64 != 0)
    return fail(MOE_ERR_UNSUPPORTED, "d_ff=%d must be a multiple of 64",
                s->d_ff);
  if (s->top_k > kTopKMax || s->top_k > s->n_routed)
    return fail(MOE_ERR_UNSUPPORTED, "top_k=%d (max %d, <= n_routed)",
                s->top_k, kTopKMax);
  if (s->n_shared > 8)
    return fail(MOE_ERR_UNSUPPORTED, "n_shared=%d (max 8)", s->n_shared);
  if (s->dtype != MOE_F32) {
    if (s->n_routed > 256 || s->n_routed % 16 != 0)
      return fail(MOE_ERR_UNSUPPORTED,
                  "bf16 n_routed=%d must be a multiple of 16, <= 256",
                  s->n_routed);
    if (s->dtype == MOE_FP8 && s->d_ff % 128 != 0)
      return fail(MOE_ERR_UNSUPPORTED,
                  "fp8: d_ff=%d must be a multiple of 128", s->d_ff);
  } else {
    if (s->n_routed > 1024)
      return fail(MOE_ERR_UNSUPPORTED, "fp32 n_routed=%d (max 1024)",
                  s->n_routed);
    if (static_cast<long long>(s->T) * s->top_k > 65535LL * 4)
      return fail(MOE_ERR_UNSUPPORTED, "fp32 path: T*top_k too large");
  }
  const long long A = static_cast<long long>(s->T) * s->top_k;
  if (A > (1LL << 31) - 1 || static_cast<long long>(s->T) * s->d > (1LL << 40))
    return fail(MOE_ERR_UNSUPPORTED, "problem too large");
  return MOE_OK;
}

struct WsLayout {
  size_t sched, route_hist, perm_hist, h_routed, h_shared, u_q, h8_routed,
      h8_shared, total;
};

WsLayout ws_layout(const moe_shape* s) {
  WsLayout w;
  const size_t es = elem_size(s->dtype);
  const long long nblk = cdiv(s->T, kRouteTile);
  const long long A = static_cast<long long>(s->T) * s->top_k;
  size_t off = 0;
  w.sched = off;   // item counters: [0..1] whole / routed call, [2..3] shared
  off = round256(off + 4 * sizeof(int));
  w.route_hist = off;   // one histogram per router CTA (<= 8 per tile)
  off = round256(off + static_cast<size_t>(nblk) * kRtMaxSplit *
                           s->n_routed * 4);
  w.perm_hist = off;
  off = round256(off + static_cast<size_t>(cdiv(s->T, kPermChunk)) *
                           s->n_routed * 4);
  // H between the passes (MOE_FP8: the single-SM kernels' e4m3 codes and
  // scales of H)
  const long long SI = static_cast<long long>(s->n_shared) * s->d_ff;
  w.h_routed = off;
  off = round256(off + (s->dtype == MOE_FP8
                            ? fp8_buf_bytes(A, s->d_ff, false)
                            : static_cast<size_t>(A) * s->d_ff * es));
  w.h_shared = off;
  off = round256(off + (s->dtype == MOE_FP8
                            ? (SI > 0 ? fp8_buf_bytes(s->T, SI, false) : 0)
                            : static_cast<size_t>(s->T) * SI * es));
  w.u_q = off;          // MOE_FP8: e4m3 codes of u and their block scales
  if (s->dtype == MOE_FP8 && s->n_shared > 0)
    off += fp8_buf_bytes(s->T, s->d, false);
  // MOE_FP8 CTA-pair path: H as e4m3 codes, scales and UE8M0 tables, written
  // by the gate/up pass's epilogue
  w.h8_routed = off;
  if (s->dtype == MOE_FP8) off += fp8_buf_bytes(A, s->d_ff, false);
  w.h8_shared = off;
  if (s->dtype == MOE_FP8 && s->n_shared > 0)
    off += fp8_buf_bytes(s->T, static_cast<long long>(s->n_shared) * s->d_ff,
                         false);
  w.total = off;
  return w;
}

moe_status check_ws(const moe_shape* s, void* ws, size_t bytes) {
  const WsLayout w = ws_layout(s);
  if (ws == nullptr && w.total > 0)
    return fail(MOE_ERR_WORKSPACE, "workspace is NULL");
  if (bytes < w.total)
    return fail(MOE_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", bytes,
                w.total);
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return fail(MOE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  return MOE_OK;
}

#define NEED_PTR(p)                                                     \
  do {                                                                  \
    if ((p) == nullptr) return fail(MOE_ERR_INVALID_ARG, #p " is NULL"); \
    if (!aligned16(p))                                                  \
      return fail(MOE_ERR_INVALID_ARG, #p " not 16-byte aligned");      \
  } while (0)

inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

// grid of the fp32 FFN kernels: 64 columns x 4 rows per 256-thread block
inline dim3 grid2(long long cols, long long rows) {
  return dim3(static_cast<unsigned>(cdiv(cols, 64)),
              static_cast<unsigned>(cdiv(rows, 4)));
}

}  // namespace

namespace {

template <int BN, int STAGES>
moe_status launch_gemm(const CUtensorMap& a_r, const CUtensorMap& b_r,
                       const CUtensorMap& a_s, const CUtensorMap& b_s,
                       const GemmParams& p, int sms, cudaStream_t cs) {
  long long items = 0;
  if (p.shared_rows > 0)
    items += cdiv(p.shared_rows, BN) * (p.w_rows_shared / kGemmBM);
  if (p.n_groups > 0)
    items += (cdiv(p.max_routed_rows, BN) + p.n_groups) *
             (p.w_rows_routed / kGemmBM);
  if (items == 0) return MOE_OK;
  const int grid = static_cast<int>(items < sms ? items : sms);
  grouped_gemm_kernel<BN, STAGES><<<grid, 192, GemmSmem<BN, STAGES>::alloc,
                                    cs>>>(a_r, b_r, a_s, b_s, p);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

// Tensor maps of the CTA-pair GEMM: 3-D views (two K-atoms per box) of the
// weights (128-row boxes) and tokens (32/64/128-row boxes), routed/shared.
struct PairMaps {
  CUtensorMap a_r, a_s, b_r32, b_s32, b_r64, b_s64, b_r96, b_s96, b_r128,
      b_s128;
};

// k_r / k_s: reduction length (row length) of the routed / shared operands.
moe_status pair_maps(const void* w_r, long long w_r_rows, const void* x_r,
                     long long x_r_rows, long long k_r, const void* w_s,
                     long long w_s_rows, const void* x_s, long long x_s_rows,
                     long long k_s, PairMaps& m) {
  moe_status st;
  const int at = kPairAtoms;
  if ((st = make_map3(&m.a_r, w_r, w_r_rows, k_r, 128, at)) != MOE_OK)
    return st;
  if ((st = make_map3(&m.b_r32, x_r, x_r_rows, k_r, 32, at)) != MOE_OK)
    return st;
  if ((st = make_map3(&m.b_r64, x_r, x_r_rows, k_r, 64, at)) != MOE_OK)
    return st;
  if ((st = make_map3(&m.b_r96, x_r, x_r_rows, k_r, 96, at)) != MOE_OK)
    return st;
  if ((st = make_map3(&m.b_r128, x_r, x_r_rows, k_r, 128, at)) != MOE_OK)
    return st;
  if (w_s != nullptr) {
    if ((st = make_map3(&m.a_s, w_s, w_s_rows, k_s, 128, at)) != MOE_OK)
      return st;
    if ((st = make_map3(&m.b_s32, x_s, x_s_rows, k_s, 32, at)) != MOE_OK)
      return st;
    if ((st = make_map3(&m.b_s64, x_s, x_s_rows, k_s, 64, at)) != MOE_OK)
      return st;
    if ((st = make_map3(&m.b_s96, x_s, x_s_rows, k_s, 96, at)) != MOE_OK)
      return st;
    if ((st = make_map3(&m.b_s128, x_s, x_s_rows, k_s, 128, at)) != MOE_OK)
      return st;
  } else {
    m.a_s = m.a_r;
    m.b_s32 = m.b_r32;
    m.b_s64 = m.b_r64;
    m.b_s96 = m.b_r96;
    m.b_s128 = m.b_r128;
  }
  return MOE_OK;
}


template <int BN, int CW, bool TWO, bool SWIGLU, int STAGES>
moe_status launch_gemm_fp8(const CUtensorMap& a_r, const CUtensorMap& b_r,
                           const CUtensorMap& a_s, const CUtensorMap& b_s,
                           const Fp8Params& p, int sms, cudaStream_t cs) {
  using L = Fp8Smem<BN, CW, TWO, STAGES>;
  long long items = 0;
  if (p.shared_rows > 0)
    items += cdiv(p.shared_rows, BN) * (p.w_rows_shared / L::TR);
  if (p.n_groups > 0)
    items += (cdiv(p.max_routed_rows, BN) + p.n_groups) *
             (p.w_rows_routed / L::TR);
  if (items == 0) return MOE_OK;
  const int grid = static_cast<int>(items < sms ? items : sms);
  grouped_gemm_fp8_kernel<BN, CW, TWO, SWIGLU, STAGES>
      <<<grid, L::threads, L::alloc, cs>>>(a_r, b_r, a_s, b_s, p);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

moe_status launch_gemm_pair(const PairMaps& m, const GemmParams& p,
                            cudaStream_t cs) {
  long long items = 0;
  if (p.shared_rows > 0)
    items += cdiv(p.shared_rows, kPairBN) * (p.w_rows_shared / kPairBM);
  if (p.n_groups > 0)
    items += (cdiv(p.max_routed_rows, kPairBN) + p.n_groups) *
             (p.w_rows_routed / kPairBM);
  if (items == 0) return MOE_OK;
  const long long clusters = pair_clusters();
  if (clusters <= 0)
    return fail(MOE_ERR_CUDA, "CTA-pair GEMM cannot be resident on this GPU");
  const long long n = items < clusters ? items : clusters;
  grouped_gemm_pair_kernel<<<static_cast<int>(2 * n), 192, PairSmem::alloc,
                             cs>>>(m.a_r, m.b_r32, m.a_s, m.b_s32, m.b_r64,
                                   m.b_s64, m.b_r96, m.b_s96, m.b_r128,
                                   m.b_s128, p);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

// Tiled maps of e4m3 operands [rows, cols] (cols = the reduction) in
// 128-byte K-atoms with 128-byte swizzle, two atoms per box:
//   3-D {128, rows, cols/128}, box {128, box_rows, 2};
//   5-D gate/up view {128, 64 rows, 2 halves, rows/128 blocks, cols/128}
//   with a box of {128, 64, 1, 2, 2}: per atom, half h of row block w (gate)
//   and the same half of block w + 1 (up).
moe_status encode_u8(CUtensorMap* m, const void* ptr, int rank,
                     const cuuint64_t* dims, const cuuint64_t* strides,
                     const cuuint32_t* box) {
  moe_status st = get_encoder();
  if (st != MOE_OK) return st;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank,
                        const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled (%d-D u8) failed (%d)",
                rank, static_cast<int>(r));
  return MOE_OK;
}
moe_status make_map3_u8(CUtensorMap* m, const void* ptr, long long rows,
                        long long cols, int box_rows) {
  cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(rows > 0 ? rows : 1),
                        static_cast<cuuint64_t>(cols / 128)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols), 128};
  cuuint32_t box[3] = {128, static_cast<cuuint32_t>(box_rows), 2};
  return encode_u8(m, ptr, 3, dims, strides, box);
}
moe_status make_map_u8_gu5d(CUtensorMap* m, const void* ptr, long long rows,
                            long long cols) {
  const long long blocks = rows / 128 > 0 ? rows / 128 : 1;
  cuuint64_t dims[5] = {128, 64, 2, static_cast<cuuint64_t>(blocks),
                        static_cast<cuuint64_t>(cols / 128)};
  cuuint64_t strides[4] = {static_cast<cuuint64_t>(cols),
                           static_cast<cuuint64_t>(64 * cols),
                           static_cast<cuuint64_t>(128 * cols), 128};
  cuuint32_t box[5] = {128, 64, 1, 2, 2};
  return encode_u8(m, ptr, 5, dims, strides, box);
}

// Tensor maps of the e4m3 CTA-pair GEMM: weights (the 5-D gate/up view, or
// 128-row boxes for the down pass) and tokens (32 / 64 / 96-row boxes),
// routed and shared; two 128-byte K-atoms of e4m3 codes per box.
struct F8PairMaps {
  CUtensorMap a_r, a_s, b_r32, b_s32, b_r64, b_s64, b_r96, b_s96;
};

moe_status f8_pair_maps(const void* w_r, long long w_r_rows, const void* x_r,
                        long long x_r_rows, long long k_r, const void* w_s,
                        long long w_s_rows, const void* x_s, long long x_s_rows,
                        long long k_s, int a_box, F8PairMaps& m) {
  moe_status st;
  auto wmap = [&](CUtensorMap* mm, const void* w, long long rows,
                  long long k) {
    return a_box == 64 ? make_map_u8_gu5d(mm, w, rows, k)
                       : make_map3_u8(mm, w, rows, k, a_box);
  };
  if ((st = wmap(&m.a_r, w_r, w_r_rows, k_r)) != MOE_OK) return st;
  CUtensorMap* br[3] = {&m.b_r32, &m.b_r64, &m.b_r96};
  CUtensorMap* bs[3] = {&m.b_s32, &m.b_s64, &m.b_s96};
  const int boxes[3] = {32, 64, 96};
  for (int i = 0; i < 3; ++i)
    if ((st = make_map3_u8(br[i], x_r, x_r_rows, k_r, boxes[i])) != MOE_OK)
      return st;
  if (w_s != nullptr) {
    if ((st = wmap(&m.a_s, w_s, w_s_rows, k_s)) != MOE_OK) return st;
    for (int i = 0; i < 3; ++i)
      if ((st = make_map3_u8(bs[i], x_s, x_s_rows, k_s, boxes[i])) != MOE_OK)
        return st;
  } else {
    m.a_s = m.a_r;
    for (int i = 0; i < 3; ++i) *bs[i] = *br[i];
  }
  return MOE_OK;
}

moe_status launch_gemm_fp8_pair(const F8PairMaps& m, const F8PairParams& p,
                                cudaStream_t cs) {
  long long items = 0;
  if (p.shared_rows > 0)
    items += cdiv(p.shared_rows, kF8PBN) * (p.w_rows_shared / kF8PBM);
  if (p.n_groups > 0)
    items += (cdiv(p.max_routed_rows, kF8PBN) + p.n_groups) *
             (p.w_rows_routed / kF8PBM);
  if (items == 0) return MOE_OK;
  const long long clusters = f8_pair_clusters();
  if (clusters <= 0)
    return fail(MOE_ERR_CUDA, "e4m3 CTA-pair GEMM cannot be resident");
  const long long n = items < clusters ? items : clusters;
  grouped_gemm_fp8_pair_kernel<<<static_cast<int>(2 * n), kF8PThreads,
                                 F8PairSmem::alloc, cs>>>(
      m.a_r, m.a_s, m.b_r32, m.b_s32, m.b_r64, m.b_s64, m.b_r96, m.b_s96, p);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

// MOE_FP8 expert FFNs: quantize u for the shared experts, gate/up (+ SwiGLU
// + requantization of H), down.  d a multiple of 256: the block-scaled
// CTA-pair kernel for every group size.  Otherwise the single-SM kernels:
// 32-token chunks for a small average group size (weight streaming), else
// 128-token chunks.
moe_status expert_ffn_fp8(const moe_shape* s, const void* x_perm,
                          const int32_t* offsets, const void* w_gu8,
                          const void* w_down8, const void* u,
                          const void* ws_gu8, const void* ws_down8,
                          void* y_perm, void* y_shared, void* ws,
                          bool has_shared, int sms, cudaStream_t cs) {
  const WsLayout w = ws_layout(s);
  const long long A = static_cast<long long>(s->T) * s->top_k;
  const int N = s->n_routed, d = s->d, I = s->d_ff, SI = s->n_shared * s->d_ff;
  const long long T = s->T;
  char* wsb = static_cast<char*>(ws);
  // operands: codes, then scales at the next 256-byte boundary
  auto scales = [](const void* base, long long rows, long long cols) {
    return reinterpret_cast<float*>(static_cast<char*>(const_cast<void*>(base)) +
                                    fp8_codes_bytes(rows, cols));
  };
  uint8_t* h8 = reinterpret_cast<uint8_t*>(wsb + w.h_routed);
  uint8_t* h8s = reinterpret_cast<uint8_t*>(wsb + w.h_shared);
  uint8_t* u8 = reinterpret_cast<uint8_t*>(wsb + w.u_q);
  moe_status st;
  if (has_shared) {
    const long long warps = T * (d / kQBlock);
    quantize_rows_kernel<<<static_cast<unsigned>(cdiv(warps, 8)), 256, 0, cs>>>(
        static_cast<const __nv_bfloat16*>(u), s->T, d, u8, scales(u8, T, d), T,
        fp8_ue8(u8, T, d, false));
    MOE_CHECK_LAUNCH();
  }
  int* ctr = reinterpret_cast<int*>(wsb + w.sched);
  zero_i32_kernel<<<1, 32, 0, cs>>>(ctr, 2);
  MOE_CHECK_LAUNCH();
  const bool small = A <= 48LL * N;
  if (d % 256 == 0 && ue8_pitch(d) <= kF8PMaxPitch &&
      ue8_pitch(I) <= kF8PMaxPitch && ue8_pitch(SI) <= kF8PMaxPitch) {
    // e4m3 CTA pairs with the block scales applied in the tensor core, for
    // prefill- and decode-sized groups alike (a decode item's few tokens
    // cost the MMA about as much per instruction as a prefill item's, and
    // the weight stream bounds it).  The gate/up pass requantizes H to e4m3
    // 1 x 128 blocks (the same rule as every activation) in its epilogue,
    // for the down pass.
    uint8_t* q8 = reinterpret_cast<uint8_t*>(wsb + w.h8_routed);
    uint8_t* q8s = reinterpret_cast<uint8_t*>(wsb + w.h8_shared);
    // padding bytes of the H tables' rows (no block writes them); the gate/up
    // pass writes H's codes and scales only (its `out` is not used)
    if (ue8_pitch(I) * kQBlock > I && A > 0)
      MOE_CHECK_CUDA(cudaMemsetAsync(fp8_ue8(q8, A, I, false), 127,
                                     static_cast<size_t>(A) * ue8_pitch(I),
                                     cs));
    if (has_shared && ue8_pitch(SI) * kQBlock > SI)
      MOE_CHECK_CUDA(cudaMemsetAsync(fp8_ue8(q8s, T, SI, false), 127,
                                     static_cast<size_t>(T) * ue8_pitch(SI),
                                     cs));
    F8PairMaps m;
    F8PairParams q{};
    if ((st = f8_pair_maps(w_gu8, 2LL * N * I, x_perm, A, d,
                           has_shared ? ws_gu8 : nullptr, 2LL * SI, u8, T, d,
                           64, m)) != MOE_OK)
      return st;
    q.offsets = offsets;
    q.n_groups = N;
    q.max_routed_rows = A;
    q.shared_rows = has_shared ? s->T : 0;
    q.w_rows_routed = 2 * I;
    q.w_rows_shared = 2 * SI;
    q.k_routed = d;
    q.k_shared = d;
    q.gate_up = 1;
    q.sw_routed = fp8_ue8(w_gu8, 2LL * N * I, d, true);
    q.sw_shared = has_shared ? fp8_ue8(ws_gu8, 2LL * SI, d, true) : nullptr;
    q.sx_routed = fp8_ue8(x_perm, A, d, false);
    q.sx_shared = has_shared ? fp8_ue8(u8, T, d, false) : nullptr;
    q.pitch_routed = ue8_pitch(d);
    q.pitch_shared = ue8_pitch(d);
    q.out_routed = nullptr;
    q.ld_routed = I;
    q.out_shared = nullptr;
    q.ld_shared = SI;
    q.item_counter = ctr;
    q.q8_routed = q8;
    q.qs_routed = scales(q8, A, I);
    q.qe_routed = fp8_ue8(q8, A, I, false);
    q.qpitch_routed = ue8_pitch(I);
    if (has_shared) {
      q.q8_shared = q8s;
      q.qs_shared = scales(q8s, T, SI);
      q.qe_shared = fp8_ue8(q8s, T, SI, false);
      q.qpitch_shared = ue8_pitch(SI);
    }
    if ((st = launch_gemm_fp8_pair(m, q, cs)) != MOE_OK) return st;
    if ((st = f8_pair_maps(w_down8, static_cast<long long>(N) * d, q8, A, I,
                           has_shared ? ws_down8 : nullptr, d, q8s, T, SI, 128,
                           m)) != MOE_OK)
      return st;
    q.w_rows_routed = d;
    q.w_rows_shared = d;
    q.k_routed = I;
    q.k_shared = SI;
    q.gate_up = 0;
    q.sw_routed = fp8_ue8(w_down8, static_cast<long long>(N) * d, I, true);
    q.sw_shared = has_shared ? fp8_ue8(ws_down8, d, SI, true) : nullptr;
    q.sx_routed = fp8_ue8(q8, A, I, false);
    q.sx_shared = has_shared ? fp8_ue8(q8s, T, SI, false) : nullptr;
    q.pitch_routed = ue8_pitch(I);
    q.pitch_shared = ue8_pitch(SI);
    q.out_routed = y_perm;
    q.ld_routed = d;
    q.out_shared = y_shared;
    q.ld_shared = d;
    q.item_counter = ctr + 1;
    q.q8_routed = q.q8_shared = nullptr;
    return launch_gemm_fp8_pair(m, q, cs);
  }
  const int bn = small ? 32 : 128;
  CUtensorMap a_r, b_r, a_s, b_s;
  Fp8Params p{};
  // pass 1: gate/up (a_*: weights, b_*: tokens)
  if ((st = make_map_u8(&a_r, w_gu8, 2LL * N * I, d, 256)) != MOE_OK) return st;
  if ((st = make_map_u8(&b_r, x_perm, A, d, bn)) != MOE_OK) return st;
  if (has_shared) {
    if ((st = make_map_u8(&a_s, ws_gu8, 2LL * SI, d, 256)) != MOE_OK) return st;
    if ((st = make_map_u8(&b_s, u8, T, d, bn)) != MOE_OK) return st;
  } else {
    a_s = a_r;
    b_s = b_r;
  }
  p.offsets = offsets;
  p.n_groups = N;
  p.max_routed_rows = A;
  p.shared_rows = has_shared ? s->T : 0;
  p.w_rows_routed = 2 * I;
  p.w_rows_shared = 2 * SI;
  p.k_routed = d;
  p.k_shared = d;
  p.sw_routed = scales(w_gu8, 2LL * N * I, d);
  p.sw_shared = has_shared ? scales(ws_gu8, 2LL * SI, d) : nullptr;
  p.sx_routed = scales(x_perm, A, d);
  p.ldsx_routed = A;
  p.sx_shared = has_shared ? scales(u8, T, d) : nullptr;
  p.ldsx_shared = T;
  p.out_routed = h8;
  p.ld_routed = I;
  p.sh_routed = scales(h8, A, I);
  p.ldsh_routed = A;
  p.out_shared = h8s;
  p.ld_shared = SI;
  p.sh_shared = has_shared ? scales(h8s, T, SI) : nullptr;
  p.ldsh_shared = T;
  p.item_counter = ctr;
  st = small
             ? launch_gemm_fp8<32, 1, true, true, 6>(a_r, b_r, a_s, b_s, p, sms,
                                                     cs)
             : launch_gemm_fp8<128, 2, true, true, 4>(a_r, b_r, a_s, b_s, p,
                                                      sms, cs);
  if (st != MOE_OK) return st;
  // pass 2: down, two 128-row tiles of W_down per item when d allows
  const bool two = d % 256 == 0;
  const int tr = two ? 256 : 128;
  if ((st = make_map_u8(&a_r, w_down8, static_cast<long long>(N) * d, I, tr)) !=
      MOE_OK)
    return st;
  if ((st = make_map_u8(&b_r, h8, A, I, bn)) != MOE_OK) return st;
  if (has_shared) {
    if ((st = make_map_u8(&a_s, ws_down8, d, SI, tr)) != MOE_OK) return st;
    if ((st = make_map_u8(&b_s, h8s, T, SI, bn)) != MOE_OK) return st;
  } else {
    a_s = a_r;
    b_s = b_r;
  }
  p.w_rows_routed = d;
  p.w_rows_shared = d;
  p.k_routed = I;
  p.k_shared = SI;
  p.sw_routed = scales(w_down8, static_cast<long long>(N) * d, I);
  p.sw_shared = has_shared ? scales(ws_down8, d, SI) : nullptr;
  p.sx_routed = scales(h8, A, I);
  p.ldsx_routed = A;
  p.sx_shared = has_shared ? scales(h8s, T, SI) : nullptr;
  p.ldsx_shared = T;
  p.out_routed = y_perm;
  p.ld_routed = d;
  p.sh_routed = nullptr;
  p.out_shared = y_shared;
  p.ld_shared = d;
  p.sh_shared = nullptr;
  p.item_counter = ctr + 1;
  if (small)
    return two ? launch_gemm_fp8<32, 1, true, false, 6>(a_r, b_r, a_s, b_s, p,
                                                        sms, cs)
               : launch_gemm_fp8<32, 1, false, false, 10>(a_r, b_r, a_s, b_s,
                                                          p, sms, cs);
  return two ? launch_gemm_fp8<128, 2, true, false, 4>(a_r, b_r, a_s, b_s, p,
                                                       sms, cs)
             : launch_gemm_fp8<128, 2, false, false, 6>(a_r, b_r, a_s, b_s, p,
                                                        sms, cs);
}

// Shape, pointer and group checks shared by the routing entry points.
moe_status check_route_args(const moe_shape* s, int G, int M, const void* u,
                            const void* centroids, const float* bias,
                            const int32_t* topk_idx, const float* topk_gate,
                            const int32_t* counts) {
  moe_status st = check_shape(s);
  if (st != MOE_OK) return st;
  if (s->T > 0) {
    NEED_PTR(u);
    NEED_PTR(topk_idx);
    NEED_PTR(topk_gate);
  }
  NEED_PTR(centroids);
  NEED_PTR(bias);
  NEED_PTR(counts);
  if (G < 1 || G > kMaxExpertGroups || s->n_routed % G != 0 || M < 1 || M > G)
    return fail(MOE_ERR_INVALID_ARG,
                "n_groups=%d topk_groups=%d: need 1 <= topk_groups <= "
                "n_groups <= %d and n_routed %% n_groups == 0",
                G, M, kMaxExpertGroups);
  if (static_cast<long long>(M) * (s->n_routed / G) < s->top_k)
    return fail(MOE_ERR_INVALID_ARG,
                "top_k=%d exceeds the %d experts of %d kept groups",
                s->top_k, M * (s->n_routed / G), M);
  return MOE_OK;
}

// Router CTAs per 128-token tile on this device (bf16: split of d across a
// cluster; fp32: 1).
int route_ctas_per_tile(const moe_shape* s, int sms) {
  return s->dtype != MOE_F32 ? route_split(s->T, s->d, sms) : 1;
}

// Router launches; `hist` holds ceil(T/128) * route_ctas_per_tile int32
// histograms of n_routed entries.
moe_status launch_route(const moe_shape* s, int G, int M, const void* u,
                        const void* centroids, const float* bias,
                        int32_t* topk_idx, float* topk_gate, int32_t* counts,
                        int* hist, cudaStream_t cs) {
  int sms = 0;
  moe_status st = device_setup(&sms);
  if (st != MOE_OK) return st;
  const int nblk = static_cast<int>(cdiv(s->T, kRouteTile));
  const int S = route_ctas_per_tile(s, sms);
  if (nblk > 0) {
    if (s->dtype != MOE_F32) {     // bf16 router (also for MOE_FP8 layers)
      CUtensorMap tm_u, tm_e;
      st = make_map(&tm_u, u, s->T, s->d, kRouteTile);
      if (st != MOE_OK) return st;
      st = make_map(&tm_e, centroids, s->n_routed, s->d, s->n_routed);
      if (st != MOE_OK) return st;
      if (S == 1) {
        route_tc_kernel<<<nblk, kRouteThreads, RouteTcSmemLayout::alloc,
                          cs>>>(
            tm_u, tm_e, bias, s->T, s->d, s->n_routed, s->top_k, G, M, 1,
            topk_idx, topk_gate, hist);
      } else {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(nblk * S));
        cfg.blockDim = dim3(kRouteThreads);
        cfg.dynamicSmemBytes = RouteTcSmemLayout::alloc;
        cfg.stream = cs;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(S);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        MOE_CHECK_CUDA(cudaLaunchKernelEx(
            &cfg, route_tc_kernel, tm_u, tm_e, bias, s->T, s->d, s->n_routed,
            s->top_k, G, M, S, topk_idx, topk_gate, hist));
      }
      MOE_CHECK_LAUNCH();
    } else {
      route_f32_kernel<<<nblk, 128, 4 * s->n_routed * sizeof(float), cs>>>(
          static_cast<const float*>(u), static_cast<const float*>(centroids),
          bias, s->T, s->d, s->n_routed, s->top_k, G, M, topk_idx, topk_gate,
          hist);
      MOE_CHECK_LAUNCH();
    }
  }
  route_hist_reduce_kernel<<<static_cast<int>(cdiv(s->n_routed, 256)), 256, 0,
                             cs>>>(hist, nblk * S, s->n_routed, counts);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_workspace_size(const moe_shape* shape, size_t* bytes) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (bytes == nullptr) return fail(MOE_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = ws_layout(shape).total;
  return MOE_OK;
}

moe_status moe_fp8_weight_bytes(const moe_shape* s, int which,
                                size_t* bytes) {
  moe_status st = check_shape(s);
  if (st != MOE_OK) return st;
  if (bytes == nullptr) return fail(MOE_ERR_INVALID_ARG, "bytes is NULL");
  if (s->dtype != MOE_FP8)
    return fail(MOE_ERR_INVALID_ARG, "moe_fp8_weight_bytes needs MOE_FP8");
  const long long N = s->n_routed, d = s->d, I = s->d_ff,
                  SI = static_cast<long long>(s->n_shared) * s->d_ff;
  long long rows, cols;
  switch (which) {
    case 0: rows = 2 * N * I; cols = d; break;     // routed gate/up
    case 1: rows = N * d; cols = I; break;         // routed down
    case 2: rows = 2 * SI; cols = d; break;        // shared gate/up
    case 3: rows = d; cols = SI; break;            // shared down
    default:
      return fail(MOE_ERR_INVALID_ARG, "which=%d (0..3)", which);
  }
  *bytes = fp8_buf_bytes(rows, cols, true);
  return MOE_OK;
}

moe_status moe_x_perm_bytes(const moe_shape* s, size_t* bytes) {
  moe_status st = check_shape(s);
  if (st != MOE_OK) return st;
  if (bytes == nullptr) return fail(MOE_ERR_INVALID_ARG, "bytes is NULL");
  const long long A = static_cast<long long>(s->T) * s->top_k;
  if (s->dtype == MOE_FP8)
    *bytes = fp8_buf_bytes(A, s->d, false);
  else
    *bytes = static_cast<size_t>(A) * s->d * elem_size(s->dtype);
  return MOE_OK;
}

moe_status moe_pack_weights_fp8(const moe_shape* s, const void* w_gate,
                                const void* w_up, const void* w_down,
                                const void* ws_gate, const void* ws_up,
                                const void* ws_down, void* w_gu8,
                                void* w_down8, void* ws_gu8, void* ws_down8,
                                void* stream) {
  g_launches = 0;
  moe_status st = check_shape(s);
  if (st != MOE_OK) return st;
  if (s->dtype != MOE_FP8)
    return fail(MOE_ERR_INVALID_ARG, "moe_pack_weights_fp8 needs MOE_FP8");
  NEED_PTR(w_gate);
  NEED_PTR(w_up);
  NEED_PTR(w_down);
  NEED_PTR(w_gu8);
  NEED_PTR(w_down8);
  if (s->n_shared > 0) {
    NEED_PTR(ws_gate);
    NEED_PTR(ws_up);
    NEED_PTR(ws_down);
    NEED_PTR(ws_gu8);
    NEED_PTR(ws_down8);
  }
  cudaStream_t cs = as_stream(stream);
  const int N = s->n_routed, d = s->d, I = s->d_ff, SI = s->n_shared * s->d_ff;
  auto launch = [&](const void* a, const void* b, int mode, long long rows,
                    int K, void* dst) -> moe_status {
    uint8_t* q = static_cast<uint8_t*>(dst);
    float* sc = reinterpret_cast<float*>(q + fp8_codes_bytes(rows, K));
    const dim3 grid(static_cast<unsigned>(K / kQBlock),
                    static_cast<unsigned>(rows / kQBlock));
    quantize_weight_blocks_kernel<<<grid, 256, 0, cs>>>(
        static_cast<const __nv_bfloat16*>(a),
        static_cast<const __nv_bfloat16*>(b), mode, K, I, d, q, sc,
        fp8_ue8(q, rows, K, true));
    MOE_CHECK_LAUNCH();
    return MOE_OK;
  };
  if ((st = launch(w_gate, w_up, 1, 2LL * N * I, d, w_gu8)) != MOE_OK)
    return st;
  if ((st = launch(w_down, nullptr, 0, static_cast<long long>(N) * d, I,
                   w_down8)) != MOE_OK)
    return st;
  if (s->n_shared > 0) {
    if ((st = launch(ws_gate, ws_up, 1, 2LL * SI, d, ws_gu8)) != MOE_OK)
      return st;
    if ((st = launch(ws_down, nullptr, 2, d, SI, ws_down8)) != MOE_OK)
      return st;
  }
  return MOE_OK;
}

moe_status moe_pack_weights(const moe_shape* s, const void* w_gate,
                            const void* w_up, const void* ws_gate,
                            const void* ws_up, const void* ws_down,
                            void* w_gu_packed, void* ws_gu_packed,
                            void* ws_down_packed, void* stream) {
  g_launches = 0;
  moe_status st = check_shape(s);
  if (st != MOE_OK) return st;
  if (s->dtype == MOE_FP8)
    return fail(MOE_ERR_INVALID_ARG, "MOE_FP8 weights: moe_pack_weights_fp8");
  NEED_PTR(w_gate);
  NEED_PTR(w_up);
  NEED_PTR(w_gu_packed);
  if (s->n_shared > 0) {
    NEED_PTR(ws_gate);
    NEED_PTR(ws_up);
    NEED_PTR(ws_down);
    NEED_PTR(ws_gu_packed);
    NEED_PTR(ws_down_packed);
  }
  const int es = static_cast<int>(elem_size(s->dtype));
  const int rvec = s->d * es / 16;
  cudaStream_t cs = as_stream(stream);
  const long long rows_r = 2LL * s->n_routed * s->d_ff;
  pack_gate_up_kernel<<<static_cast<int>(rows_r < 65536 ? rows_r : 65536), 128,
                        0, cs>>>(
      static_cast<const uint4*>(w_gate), static_cast<const uint4*>(w_up),
      s->n_routed, 1, s->d_ff, rvec, static_cast<uint4*>(w_gu_packed));
  MOE_CHECK_LAUNCH();
  if (s->n_shared > 0) {
    const long long rows_s = 2LL * s->n_shared * s->d_ff;
    pack_gate_up_kernel<<<static_cast<int>(rows_s < 65536 ? rows_s : 65536),
                          128, 0, cs>>>(
        static_cast<const uint4*>(ws_gate), static_cast<const uint4*>(ws_up), 1,
        s->n_shared, s->d_ff, rvec, static_cast<uint4*>(ws_gu_packed));
    MOE_CHECK_LAUNCH();
    const long long rows_d = static_cast<long long>(s->n_shared) * s->d;
    pack_shared_down_kernel<<<static_cast<int>(rows_d < 65536 ? rows_d : 65536),
                              128, 0, cs>>>(
        static_cast<const uint4*>(ws_down), s->n_shared, s->d,
        s->d_ff * es / 16, static_cast<uint4*>(ws_down_packed));
    MOE_CHECK_LAUNCH();
  }
  return MOE_OK;
}

moe_status moe_route_grouped(const moe_shape* s, int n_groups,
                             int topk_groups, const void* u,
                             const void* centroids, const float* bias,
                             int32_t* topk_idx, float* topk_gate,
                             int32_t* counts, void* ws, size_t ws_bytes,
                             void* stream) {
  g_launches = 0;
  moe_status st = check_route_args(s, n_groups, topk_groups, u, centroids,
                                   bias, topk_idx, topk_gate, counts);
  if (st != MOE_OK) return st;
  st = check_ws(s, ws, ws_bytes);
  if (st != MOE_OK) return st;
  const WsLayout w = ws_layout(s);
  return launch_route(s, n_groups, topk_groups, u, centroids, bias, topk_idx,
                      topk_gate, counts,
                      reinterpret_cast<int*>(static_cast<char*>(ws) +
                                             w.route_hist),
                      as_stream(stream));
}

moe_status moe_route(const moe_shape* s, const void* u, const void* centroids,
                     const float* bias, int32_t* topk_idx, float* topk_gate,
                     int32_t* counts, void* ws, size_t ws_bytes, void* stream) {
  return moe_route_grouped(s, 1, 1, u, centroids, bias, topk_idx, topk_gate,
                           counts, ws, ws_bytes, stream);
}

moe_status moe_permute(const moe_shape* s, const void* u,
                       const int32_t* topk_idx, const int32_t* counts,
                       int32_t* offsets, int32_t* perm, int32_t* inv,
                       void* x_perm, void* ws, size_t ws_bytes, void* stream) {
  g_launches = 0;
  moe_status st = check_shape(s);
  if (st != MOE_OK) return st;
  if (s->T > 0) {
    NEED_PTR(u);
    NEED_PTR(topk_idx);
    NEED_PTR(perm);
    NEED_PTR(inv);
    NEED_PTR(x_perm);
  }
  NEED_PTR(counts);
  NEED_PTR(offsets);
  st = check_ws(s, ws, ws_bytes);
  if (st != MOE_OK) return st;
  const WsLayout w = ws_layout(s);
  int* chist = reinterpret_cast<int*>(static_cast<char*>(ws) + w.perm_hist);
  const int nch = static_cast<int>(cdiv(s->T, kPermChunk));
  cudaStream_t cs = as_stream(stream);
  if (nch > 0) {
    permute_chunk_hist_kernel<<<nch, 256, 0, cs>>>(topk_idx, s->T, s->top_k,
                                                   s->n_routed, chist);
    MOE_CHECK_LAUNCH();
  }
  permute_slots_kernel<<<nch > 0 ? nch : 1, 256, 0, cs>>>(
      topk_idx, counts, chist, s->T, s->top_k, s->n_routed, offsets, perm, inv);
  MOE_CHECK_LAUNCH();
  if (s->T > 0) {
    const int nvec = static_cast<int>(s->d * elem_size(s->dtype) / 16);
    int sms = 0;
    st = device_setup(&sms);
    if (st != MOE_OK) return st;
    const long long want = cdiv(s->T, 8);
    const int grid = static_cast<int>(want < sms * 8LL ? want : sms * 8LL);
    if (s->dtype == MOE_FP8) {
      const long long A = static_cast<long long>(s->T) * s->top_k;
      uint8_t* x8 = static_cast<uint8_t*>(x_perm);
      const long long wq = cdiv(static_cast<long long>(s->T) * (s->d / 128), 8);
      const int grid8 = static_cast<int>(wq < sms * 16LL ? wq : sms * 16LL);
      permute_gather_fp8_kernel<<<grid8, 256, 0, cs>>>(
          static_cast<const __nv_bfloat16*>(u), inv, s->T, s->top_k, s->d, A,
          x8, reinterpret_cast<float*>(x8 + fp8_codes_bytes(A, s->d)),
          fp8_ue8(x8, A, s->d, false));
      MOE_CHECK_LAUNCH();
      return MOE_OK;
    }
    permute_gather_kernel<<<grid, 256, 0, cs>>>(
        static_cast<const uint4*>(u), inv, s->T, s->top_k, nvec,
        static_cast<long long>(s->T) * s->top_k, static_cast<uint4*>(x_perm));
    MOE_CHECK_LAUNCH();
  }
  return MOE_OK;
}


static moe_status expert_ffn_impl(const moe_shape* s, int part,
                                  const void* x_perm, const int32_t* offsets,
                                  const void* w_gu_packed, const void* w_down,
                                  const void* u, const void* ws_gu_packed,
                                  const void* ws_down_packed, void* y_perm,
                                  void* y_shared, void* ws, size_t ws_bytes,
                                  void* stream, void* act = nullptr,
                                  void* act_shared = nullptr) {
  g_launches = 0;
  moe_status st = check_shape(s);
  if (st != MOE_OK) return st;
  const bool save = act != nullptr || act_shared != nullptr;
  if (save) {
    if (s->dtype != MOE_BF16)
      return fail(MOE_ERR_UNSUPPORTED,
                  "saved pre-activations: bf16 layers only (dtype %d)",
                  static_cast<int>(s->dtype));
    if (s->T > 0) NEED_PTR(act);
    if (s->T > 0 && s->n_shared > 0) NEED_PTR(act_shared);
  }
  if (part < 0 || part > 2)
    return fail(MOE_ERR_INVALID_ARG, "part=%d (0 both, 1 routed, 2 shared)",
                part);
  if (part != 0 && s->dtype == MOE_FP8)
    return fail(MOE_ERR_UNSUPPORTED, "MOE_FP8: expert FFN parts not split");
  const bool do_routed = part != 2;
  if (do_routed) {
    NEED_PTR(offsets);
    NEED_PTR(w_gu_packed);
    NEED_PTR(w_down);
    if (s->T > 0) {
      NEED_PTR(x_perm);
      NEED_PTR(y_perm);
    }
  }
  const bool has_shared = part != 1 && s->n_shared > 0 && s->T > 0;
  if (has_shared) {
    NEED_PTR(u);
    NEED_PTR(ws_gu_packed);
    NEED_PTR(ws_down_packed);
    NEED_PTR(y_shared);
  }
  st = check_ws(s, ws, ws_bytes);
  if (st != MOE_OK) return st;
  if (s->T == 0) return MOE_OK;
  int sms = 0;
  st = device_setup(&sms);
  if (st != MOE_OK) return st;
  const WsLayout w = ws_layout(s);
  void* h_r = static_cast<char*>(ws) + w.h_routed;
  void* h_s = static_cast<char*>(ws) + w.h_shared;
  const long long A = static_cast<long long>(s->T) * s->top_k;
  const int N = s->n_routed, d = s->d, I = s->d_ff, SI = s->n_shared * s->d_ff;
  cudaStream_t cs = as_stream(stream);

  if (s->dtype == MOE_F32) {
    const float* xp = static_cast<const float*>(x_perm);
    float* hr = static_cast<float*>(h_r);
    float* hs = static_cast<float*>(h_s);
    if (do_routed) {
      ffn_f32_gate_up_kernel<<<grid2(I, A), 256, 0, cs>>>(
          xp, static_cast<int>(A), offsets, N,
          static_cast<const float*>(w_gu_packed), I, d, hr);
      MOE_CHECK_LAUNCH();
      ffn_f32_down_kernel<<<grid2(d, A), 256, 0, cs>>>(
          hr, static_cast<int>(A), offsets, N,
          static_cast<const float*>(w_down), I, d,
          static_cast<float*>(y_perm));
      MOE_CHECK_LAUNCH();
    }
    if (has_shared) {
      ffn_f32_gate_up_kernel<<<grid2(SI, s->T), 256, 0, cs>>>(
          static_cast<const float*>(u), s->T, nullptr, 1,
          static_cast<const float*>(ws_gu_packed), SI, d, hs);
      MOE_CHECK_LAUNCH();
      ffn_f32_down_kernel<<<grid2(d, s->T), 256, 0, cs>>>(
          hs, s->T, nullptr, 1, static_cast<const float*>(ws_down_packed), SI,
          d, static_cast<float*>(y_shared));
      MOE_CHECK_LAUNCH();
    }
    return MOE_OK;
  }

  if (s->dtype == MOE_FP8)
    return expert_ffn_fp8(s, x_perm, offsets, w_gu_packed, w_down, u,
                          ws_gu_packed, ws_down_packed, y_perm, y_shared, ws,
                          has_shared, sms, cs);

  // bf16: tcgen05 grouped GEMMs.  Small average group size -> 32-token
  // chunks and a deeper ring (weight streaming); else 256-token chunks.
  const bool small = A <= 48LL * N;
  // CTA pairs (256 weight rows per item) when every weight group splits
  // into 256-row tiles; else the single-SM kernel.
  const bool pair = !small && d % 256 == 0 && I % 128 == 0;
  // a shared-only call counts its items apart, so it can run beside a
  // routed-only call on another stream
  int* ctr = reinterpret_cast<int*>(static_cast<char*>(ws) + w.sched) +
             (part == 2 ? 2 : 0);
  zero_i32_kernel<<<1, 32, 0, cs>>>(ctr, 2);
  MOE_CHECK_LAUNCH();
  if (!do_routed && !has_shared) return MOE_OK;
  // operands of the part that is not computed stand in for its maps
  const void* wgu_r = do_routed ? w_gu_packed : ws_gu_packed;
  const void* xr = do_routed ? x_perm : u;
  const long long rows_gu_r = do_routed ? 2LL * N * I : 2LL * SI;
  const long long rows_x_r = do_routed ? A : s->T;
  CUtensorMap a_r, b_r, a_s, b_s;
  const int box = kBoxRows;
  GemmParams p{};
  // pass 1: gate/up + SwiGLU -> H
  if ((st = make_map(&a_r, wgu_r, rows_gu_r, d, kGemmBM)) != MOE_OK)
    return st;
  PairMaps pm;
  if ((st = make_map(&b_r, xr, rows_x_r, d, box)) != MOE_OK) return st;
  if (has_shared) {
    if ((st = make_map(&a_s, ws_gu_packed, 2LL * SI, d, kGemmBM)) != MOE_OK)
      return st;
    if ((st = make_map(&b_s, u, s->T, d, box)) != MOE_OK) return st;
  } else {
    a_s = a_r;
    b_s = b_r;
  }
  p.offsets = offsets;
  p.n_groups = do_routed ? N : 0;
  p.w_rows_routed = 2 * I;
  p.k_routed = d;
  p.max_routed_rows = A;
  p.shared_rows = has_shared ? s->T : 0;
  p.w_rows_shared = 2 * SI;
  p.k_shared = d;
  p.out_routed = h_r;
  p.ld_routed = I;
  p.out_shared = h_s;
  p.ld_shared = SI;
  p.swiglu = 1;
  p.item_counter = ctr;
  if (save) {   // rows as H's: x_perm slots (routed), tokens (shared)
    p.act_routed = static_cast<__half*>(act);
    p.ld_act_routed = 2LL * I;
    p.act_shared = static_cast<__half*>(act_shared);
    p.ld_act_shared = 2LL * SI;
  }
  if (pair) {
    if ((st = pair_maps(wgu_r, rows_gu_r, xr, rows_x_r, d,
                        has_shared ? ws_gu_packed : nullptr, 2LL * SI,
                        u, s->T, d, pm)) != MOE_OK)
      return st;
    st = launch_gemm_pair(pm, p, cs);
  } else {
    st = small ? launch_gemm<32, 10>(a_r, b_r, a_s, b_s, p, sms, cs)
               : launch_gemm<256, 4>(a_r, b_r, a_s, b_s, p, sms, cs);
  }
  if (st != MOE_OK) return st;
  // pass 2: down -> y
  const void* wd_r = do_routed ? w_down : ws_down_packed;
  const long long rows_d_r = do_routed ? static_cast<long long>(N) * d : d;
  const long long k_r2 = do_routed ? I : SI;
  const void* hr_ = do_routed ? h_r : h_s;
  if ((st = make_map(&a_r, wd_r, rows_d_r, k_r2, kGemmBM)) != MOE_OK)
    return st;
  if ((st = make_map(&b_r, hr_, rows_x_r, k_r2, box)) != MOE_OK) return st;
  if (has_shared) {
    if ((st = make_map(&a_s, ws_down_packed, d, SI, kGemmBM)) != MOE_OK)
      return st;
    if ((st = make_map(&b_s, h_s, s->T, SI, box)) != MOE_OK) return st;
  } else {
    a_s = a_r;
    b_s = b_r;
  }
  p.w_rows_routed = d;
  p.k_routed = I;
  p.w_rows_shared = d;
  p.k_shared = SI;
  p.out_routed = y_perm;
  p.ld_routed = d;
  p.out_shared = y_shared;
  p.ld_shared = d;
  p.swiglu = 0;
  p.y_fp16 = 1;
  p.item_counter = ctr + 1;
  p.act_routed = p.act_shared = nullptr;
  if (pair) {
    if ((st = pair_maps(wd_r, rows_d_r, hr_, rows_x_r, k_r2,
                        has_shared ? ws_down_packed : nullptr, d, h_s, s->T,
                        SI, pm)) != MOE_OK)
      return st;
    return launch_gemm_pair(pm, p, cs);
  }
  return small ? launch_gemm<32, 10>(a_r, b_r, a_s, b_s, p, sms, cs)
               : launch_gemm<256, 4>(a_r, b_r, a_s, b_s, p, sms, cs);
}

moe_status moe_expert_ffn(const moe_shape* s, const void* x_perm,
                          const int32_t* offsets, const void* w_gu_packed,
                          const void* w_down, const void* u,
                          const void* ws_gu_packed, const void* ws_down_packed,
                          void* y_perm, void* y_shared, void* ws,
                          size_t ws_bytes, void* stream) {
  return expert_ffn_impl(s, 0, x_perm, offsets, w_gu_packed, w_down, u,
                         ws_gu_packed, ws_down_packed, y_perm, y_shared, ws,
                         ws_bytes, stream);
}

moe_status moe_expert_ffn_part(const moe_shape* s, int part,
                               const void* x_perm, const int32_t* offsets,
                               const void* w_gu_packed, const void* w_down,
                               const void* u, const void* ws_gu_packed,
                               const void* ws_down_packed, void* y_perm,
                               void* y_shared, void* ws, size_t ws_bytes,
                               void* stream) {
  return expert_ffn_impl(s, part, x_perm, offsets, w_gu_packed, w_down, u,
                         ws_gu_packed, ws_down_packed, y_perm, y_shared, ws,
                         ws_bytes, stream);
}

moe_status moe_expert_ffn_train(const moe_shape* s, const void* x_perm,
                                const int32_t* offsets,
                                const void* w_gu_packed, const void* w_down,
                                const void* u, const void* ws_gu_packed,
                                const void* ws_down_packed, void* y_perm,
                                void* y_shared, void* act, void* act_shared,
                                void* ws, size_t ws_bytes, void* stream) {
  if (act == nullptr) return fail(MOE_ERR_INVALID_ARG, "act is NULL");
  return expert_ffn_impl(s, 0, x_perm, offsets, w_gu_packed, w_down, u,
                         ws_gu_packed, ws_down_packed, y_perm, y_shared, ws,
                         ws_bytes, stream, act, act_shared);
}

moe_status moe_combine(const moe_shape* s, const void* u, const void* y_perm,
                       const void* y_shared, const int32_t* inv,
                       const float* topk_gate, void* h, moe_dtype h_dtype,
                       void* stream) {
  g_launches = 0;
  moe_status st = check_shape(s);
  if (st != MOE_OK) return st;
  if (h_dtype != MOE_F32 && h_dtype != MOE_BF16)
    return fail(MOE_ERR_INVALID_ARG, "h_dtype %d", static_cast<int>(h_dtype));
  if (s->T == 0) return MOE_OK;
  NEED_PTR(u);
  NEED_PTR(y_perm);
  NEED_PTR(inv);
  NEED_PTR(topk_gate);
  NEED_PTR(h);
  if (s->n_shared > 0) NEED_PTR(y_shared);
  const void* ys = s->n_shared > 0 ? y_shared : nullptr;
  const long long A = static_cast<long long>(s->T) * s->top_k;
  cudaStream_t cs = as_stream(stream);
  if (s->dtype != MOE_F32) {
    // bf16 and fp8 layers keep the expert outputs in fp16
    const __nv_bfloat16* a = static_cast<const __nv_bfloat16*>(u);
    const __half* y = static_cast<const __half*>(y_perm);
    const __half* z = static_cast<const __half*>(ys);
    if (h_dtype == MOE_F32)
      combine_kernel<__nv_bfloat16, __half, float><<<s->T, 128, 0, cs>>>(
          a, y, z, inv, topk_gate, s->T, s->d, s->top_k, A,
          static_cast<float*>(h));
    else
      combine_kernel<__nv_bfloat16, __half, __nv_bfloat16>
          <<<s->T, 128, 0, cs>>>(a, y, z, inv, topk_gate, s->T, s->d,
                                 s->top_k, A, static_cast<__nv_bfloat16*>(h));
  } else {
    const float* a = static_cast<const float*>(u);
    const float* y = static_cast<const float*>(y_perm);
    const float* z = static_cast<const float*>(ys);
    if (h_dtype == MOE_F32)
      combine_kernel<float, float, float><<<s->T, 128, 0, cs>>>(
          a, y, z, inv, topk_gate, s->T, s->d, s->top_k, A,
          static_cast<float*>(h));
    else
      combine_kernel<float, float, __nv_bfloat16><<<s->T, 128, 0, cs>>>(
          a, y, z, inv, topk_gate, s->T, s->d, s->top_k, A,
          static_cast<__nv_bfloat16*>(h));
  }
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

moe_status moe_update_bias(int n_routed, const int32_t* counts,
                           long long total_assign, float gamma, float* bias,
                           void* stream) {
  g_launches = 0;
  if (n_routed <= 0 || total_assign < 0)
    return fail(MOE_ERR_INVALID_ARG, "n_routed=%d total_assign=%lld", n_routed,
                total_assign);
  if (!(gamma >= 0.f) || gamma > 1e30f)
    return fail(MOE_ERR_INVALID_ARG, "gamma must be finite and >= 0");
  NEED_PTR(counts);
  NEED_PTR(bias);
  update_bias_kernel<<<static_cast<int>(cdiv(n_routed, 256)), 256, 0,
                       as_stream(stream)>>>(counts, n_routed, total_assign,
                                            gamma, bias);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

moe_status moe_get_device_error(void* stream) {
  MOE_CHECK_CUDA(cudaStreamSynchronize(as_stream(stream)));
  unsigned word = 0, info[2] = {0, 0};
  MOE_CHECK_CUDA(cudaMemcpyFromSymbol(&word, g_err_word, sizeof(word)));
  if (word == 0) return MOE_OK;
  MOE_CHECK_CUDA(cudaMemcpyFromSymbol(info, g_err_info, sizeof(info)));
  const unsigned zero[3] = {0, 0, 0};
  MOE_CHECK_CUDA(cudaMemcpyToSymbol(g_err_word, zero, sizeof(unsigned)));
  MOE_CHECK_CUDA(cudaMemcpyToSymbol(g_err_info, zero, 2 * sizeof(unsigned)));
  if (word & ERR_TIMEOUT)
    return fail(MOE_ERR_TIMEOUT, "device wait timed out (kernel %u, site %u)",
                info[0], info[1]);
  return fail(MOE_ERR_DEVICE_CHECK, "device bounds check (kernel %u, at %u)",
              info[0], info[1]);
}

moe_status moe_selftest_wait_timeout(unsigned limit_us, void* stream) {
  g_launches = 0;
  if (limit_us == 0 || limit_us > 1000000u)
    return fail(MOE_ERR_INVALID_ARG, "limit_us must be in [1, 1000000]");
  wait_timeout_selftest_kernel<<<1, 32, 0, as_stream(stream)>>>(
      1000ull * limit_us);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

const char* moe_status_string(moe_status st) {
  switch (st) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_TIMEOUT: return "device pipeline wait timed out";
    case MOE_ERR_DEVICE_CHECK: return "device bounds check failed";
  }
  return "unknown status";
}

const char* moe_last_error_detail(void) { return g_detail.c_str(); }

int moe_last_launch_count(void) { return g_launches; }

}  // extern "C"

// ---------------------------------------------------------------------------
// Workspace-free routing.  The per-block histograms of the router live in
// this file-scope device array instead of the caller's workspace.  Host code
// must not pass `g_route_noalloc_scratch` itself to a kernel: on the host
// that name is a stand-in, not a device address.  The device address is
// looked up once per device (cudaGetSymbolAddress, with that device current)
// and cached.
static __device__ __align__(256) int
    g_route_noalloc_scratch[MOE_ROUTE_NOALLOC_MAX_ENTRIES];

namespace {
int* g_noalloc_ptr[kMaxDevices] = {nullptr};
std::mutex g_noalloc_mu;

moe_status noalloc_scratch(int** out) {
  int dev = 0;
  MOE_CHECK_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices)
    return fail(MOE_ERR_UNSUPPORTED, "device index %d", dev);
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_route_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return fail(MOE_ERR_CUDA, "cudaGetSymbolAddress(route scratch): %s",
                  cudaGetErrorString(e));
    g_noalloc_ptr[dev] = static_cast<int*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return MOE_OK;
}
}  // namespace

extern "C" {

moe_status moe_route_noalloc(const moe_shape* s, const void* u,
                             const void* centroids, const float* bias,
                             int32_t* topk_idx, float* topk_gate,
                             int32_t* counts, void* stream) {
  g_launches = 0;
  moe_status st = check_route_args(s, 1, 1, u, centroids, bias, topk_idx,
                                   topk_gate, counts);
  if (st != MOE_OK) return st;
  int sms = 0;
  st = device_setup(&sms);
  if (st != MOE_OK) return st;
  const long long nblk = cdiv(s->T, kRouteTile);
  const long long need = nblk * route_ctas_per_tile(s, sms) * s->n_routed;
  if (need > MOE_ROUTE_NOALLOC_MAX_ENTRIES)
    return fail(MOE_ERR_UNSUPPORTED,
                "moe_route_noalloc: %lld router CTAs x n_routed = %lld "
                "histogram entries exceeds the static scratch of %d; use "
                "moe_route with a workspace",
                nblk * route_ctas_per_tile(s, sms), need,
                MOE_ROUTE_NOALLOC_MAX_ENTRIES);
  int* hist = nullptr;
  st = noalloc_scratch(&hist);
  if (st != MOE_OK) return st;
  return launch_route(s, 1, 1, u, centroids, bias, topk_idx, topk_gate,
                      counts, hist, as_stream(stream));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Backward pass.
namespace {

constexpr int kBwdCounters = 8;

// Workspace of moe_backward.  Per-assignment operands live in a padded
// layout: expert e's rows start at offpad[e] (a multiple of 16) and its
// segment is a whole number of 16-row blocks, so the layout needs at most
// A + 15 N rows (A = T K).
struct BwdLayout {
  long long A_pad;
  size_t ctr, offs, offpad, dz, X, dY, dH, H, dA, dX, dH_s, H_s, dA_s, dX_s,
      total;
};

BwdLayout bwd_layout(const moe_shape* s) {
  BwdLayout w;
  const long long A = static_cast<long long>(s->T) * s->top_k;
  const long long N = s->n_routed, d = s->d, I = s->d_ff;
  const long long SI = static_cast<long long>(s->n_shared) * I;
  w.A_pad = cdiv(A + (kPadRows - 1) * N, kPadRows) * kPadRows;
  const size_t R = static_cast<size_t>(w.A_pad);
  const size_t T = static_cast<size_t>(s->T);
  size_t off = 0;
  w.ctr = off;     off = round256(off + kBwdCounters * 4);
  w.offs = off;    off = round256(off + (N + 1) * 4);
  w.offpad = off;  off = round256(off + (N + 1) * 4);
  w.dz = off;      off = round256(off + R * 4);
  w.X = off;       off = round256(off + R * d * 2);
  w.dY = off;      off = round256(off + R * d * 2);
  w.dH = off;      off = round256(off + R * I * 2);
  w.H = off;       off = round256(off + R * I * 2);
  w.dA = off;      off = round256(off + R * 2 * I * 2);
  w.dX = off;      off = round256(off + R * d * 2);
  w.dH_s = off;    off = round256(off + T * SI * 2);
  w.H_s = off;     off = round256(off + T * SI * 2);
  w.dA_s = off;    off = round256(off + T * 2 * SI * 2);
  w.dX_s = off;    off = round256(off + (SI > 0 ? T * d * 2 : 0));
  w.total = off;
  return w;
}

moe_status check_bwd_shape(const moe_shape* s) {
  moe_status st = check_shape(s);
  if (st != MOE_OK) return st;
  if (s->dtype != MOE_BF16)
    return fail(MOE_ERR_UNSUPPORTED, "backward: bf16 layers only (dtype %d)",
                static_cast<int>(s->dtype));
  if (s->d_ff % 128 != 0)
    return fail(MOE_ERR_UNSUPPORTED,
                "backward: d_ff=%d must be a multiple of 128", s->d_ff);
  return MOE_OK;
}

template <int KIND, int BN, int STAGES>
moe_status launch_bwd_gemm(const CUtensorMap& a_r, const CUtensorMap& b_r,
                           const CUtensorMap& a_s, const CUtensorMap& b_s,
                           const BwdParams& p, long long max_items, int sms,
                           cudaStream_t cs) {
  if (max_items <= 0) return MOE_OK;
  const int grid = static_cast<int>(max_items < sms ? max_items : sms);
  bwd_gemm_kernel<KIND, BN, STAGES>
      <<<grid, 192, BwdSmem<BN, STAGES>::alloc, cs>>>(a_r, b_r, a_s, b_s, p);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

// 3-D maps of one backward pair launch: every operand as {64, rows,
// cols/64} with {64, box, 2}-element boxes (make_map3).  The A operands use
// 128-row boxes whether K-major (weight rows) or MN-major (K rows); the B
// operand gets 32/64/128-row boxes when it is the token operand, else only
// the 128-row one.
struct Op {
  const void* p;
  long long rows, cols;
};
moe_status bwd_pair_maps(Op a_r, Op b_r, Op a_s, Op b_s, bool shared,
                         bool tokens, BwdPairMaps& m, int kbox = 128) {
  // kbox: rows per box of the Wgrad operands (its K per stage); the token
  // kinds' weight boxes are always 128 rows
  moe_status st;
  if ((st = make_map3(&m.a_r, a_r.p, a_r.rows, a_r.cols, kbox, 2))) return st;
  if ((st = make_map3(&m.b_r128, b_r.p, b_r.rows, b_r.cols,
                      tokens ? 128 : kbox, 2)))
    return st;
  if (tokens) {
    if ((st = make_map3(&m.b_r32, b_r.p, b_r.rows, b_r.cols, 32, 2))) return st;
    if ((st = make_map3(&m.b_r64, b_r.p, b_r.rows, b_r.cols, 64, 2))) return st;
  } else {
    m.b_r32 = m.b_r64 = m.b_r128;
  }
  if (shared) {
    if ((st = make_map3(&m.a_s, a_s.p, a_s.rows, a_s.cols, kbox, 2)))
      return st;
    if ((st = make_map3(&m.b_s128, b_s.p, b_s.rows, b_s.cols,
                        tokens ? 128 : kbox, 2)))
      return st;
    if (tokens) {
      if ((st = make_map3(&m.b_s32, b_s.p, b_s.rows, b_s.cols, 32, 2)))
        return st;
      if ((st = make_map3(&m.b_s64, b_s.p, b_s.rows, b_s.cols, 64, 2)))
        return st;
    } else {
      m.b_s32 = m.b_s64 = m.b_s128;
    }
  } else {
    m.a_s = m.a_r;
    m.b_s32 = m.b_r32;
    m.b_s64 = m.b_r64;
    m.b_s128 = m.b_r128;
  }
  m.o_r = m.o2_r = m.o_s = m.o2_s = m.a_r;   // Wgrad sets its own
  return MOE_OK;
}

// Output map of a weight gradient [rows, cols] (bf16 or fp32) for the
// Wgrad TMA stores: boxes of 32 rows x 64 bytes (32 bf16 or 16 fp32
// columns) with 64-byte swizzle, the epilogue's shared-memory layout.
moe_status make_map_grad(CUtensorMap* m, const void* ptr, long long rows,
                         long long cols, bool bf16) {
  moe_status st = get_encoder();
  if (st != MOE_OK) return st;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols),
                        static_cast<cuuint64_t>(rows > 0 ? rows : 1)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * (bf16 ? 2 : 4)};
  cuuint32_t box[2] = {bf16 ? 32u : 16u, 32u};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(
      m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
      2, const_cast<void*>(ptr), dims, strides, box, estr,
      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
      CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled (gradient) failed (%d) "
                "rows=%lld cols=%lld", static_cast<int>(r), rows, cols);
  return MOE_OK;
}

// Outputs of the Dgrad (down) launch: dH (fp16) for the recompute pass, or,
// with the forward's saved pre-activations, H and dA straight from its
// epilogue (the SwiGLU backward fused, no recompute pass).
void set_dgrad_down_outputs(BwdParams& p, bool saved, const void* act,
                            const void* act_shared, int I, int SI, void* dH,
                            void* dH_s, void* H, void* H_s, void* dA,
                            void* dA_s) {
  p.ld_r = I;
  p.ld_s = SI;
  if (!saved) {
    p.out_r = dH;
    p.out_s = dH_s;
    p.act_r = p.act_s = nullptr;
    return;
  }
  p.out_r = H;
  p.out_s = H_s;
  p.out2_r = dA;    p.ld2_r = 2LL * I;
  p.out2_s = dA_s;  p.ld2_s = 2LL * SI;
  p.act_r = static_cast<const __half*>(act);
  p.ld_act_r = 2LL * I;
  p.act_s = static_cast<const __half*>(act_shared);
  p.ld_act_s = 2LL * SI;
}

template <int KIND>
moe_status launch_bwd_pair(const BwdPairMaps& m, const BwdParams& p,
                           long long max_items, cudaStream_t cs) {
  if (max_items <= 0) return MOE_OK;
  const long long clusters = bwd_pair_clusters();
  if (clusters <= 0)
    return fail(MOE_ERR_CUDA, "backward CTA-pair GEMM cannot be resident");
  const long long n = max_items < clusters ? max_items : clusters;
  bwd_gemm_pair_kernel<KIND>
      <<<static_cast<int>(2 * n), bwd_pair_threads<KIND>(),
         BwdPairSmem<KIND>::alloc, cs>>>(m, p);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_backward_workspace_size(const moe_shape* s, size_t* bytes) {
  g_launches = 0;
  moe_status st = check_bwd_shape(s);
  if (st != MOE_OK) return st;
  if (bytes == nullptr) return fail(MOE_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = bwd_layout(s).total;
  return MOE_OK;
}

moe_status moe_backward(const moe_shape* s, const void* dh, const void* u,
                        const void* centroids, const int32_t* topk_idx,
                        const float* topk_gate, const int32_t* offsets,
                        const int32_t* inv, const void* y_perm,
                        const void* act, const void* act_shared,
                        const void* w_gu_packed, const void* w_down,
                        const void* ws_gu_packed, const void* ws_down_packed,
                        float* du, float* dE, void* dw_gate, void* dw_up,
                        void* dw_down, void* dws_gate, void* dws_up,
                        void* dws_down, moe_dtype grad_dtype, void* ws,
                        size_t ws_bytes, void* stream) {
  g_launches = 0;
  moe_status st = check_bwd_shape(s);
  if (st != MOE_OK) return st;
  if (grad_dtype != MOE_F32 && grad_dtype != MOE_BF16)
    return fail(MOE_ERR_INVALID_ARG, "grad_dtype %d",
                static_cast<int>(grad_dtype));
  const int T = s->T, N = s->n_routed, d = s->d, I = s->d_ff,
            K = s->top_k, S = s->n_shared;
  const int SI = S * I;
  NEED_PTR(centroids);
  NEED_PTR(offsets);
  NEED_PTR(w_gu_packed);
  NEED_PTR(w_down);
  NEED_PTR(dE);
  NEED_PTR(dw_gate);
  NEED_PTR(dw_up);
  NEED_PTR(dw_down);
  if (T > 0) {
    NEED_PTR(dh);
    NEED_PTR(u);
    NEED_PTR(topk_idx);
    NEED_PTR(topk_gate);
    NEED_PTR(inv);
    NEED_PTR(y_perm);
    NEED_PTR(du);
  }
  if (S > 0) {
    NEED_PTR(ws_gu_packed);
    NEED_PTR(ws_down_packed);
    NEED_PTR(dws_gate);
    NEED_PTR(dws_up);
    NEED_PTR(dws_down);
  }
  // saved pre-activations (moe_expert_ffn_train): both or neither
  const bool saved = act != nullptr;
  if (!saved && act_shared != nullptr)
    return fail(MOE_ERR_INVALID_ARG, "act_shared given without act");
  if (saved && T > 0) {
    NEED_PTR(act);
    if (S > 0) NEED_PTR(act_shared);
  }
  const BwdLayout w = bwd_layout(s);
  if (ws == nullptr) return fail(MOE_ERR_WORKSPACE, "workspace is NULL");
  if (ws_bytes < w.total)
    return fail(MOE_ERR_WORKSPACE, "workspace %zu bytes < %zu needed",
                ws_bytes, w.total);
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return fail(MOE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  cudaStream_t cs = as_stream(stream);
  const size_t gsz = grad_dtype == MOE_BF16 ? 2 : 4;
  if (T == 0) {   // no tokens: every gradient is zero
    const size_t wn = static_cast<size_t>(N) * I * d * gsz;
    MOE_CHECK_CUDA(cudaMemsetAsync(dE, 0, static_cast<size_t>(N) * d * 4, cs));
    MOE_CHECK_CUDA(cudaMemsetAsync(dw_gate, 0, wn, cs));
    MOE_CHECK_CUDA(cudaMemsetAsync(dw_up, 0, wn, cs));
    MOE_CHECK_CUDA(cudaMemsetAsync(dw_down, 0, wn, cs));
    if (S > 0) {
      const size_t sn = static_cast<size_t>(SI) * d * gsz;
      MOE_CHECK_CUDA(cudaMemsetAsync(dws_gate, 0, sn, cs));
      MOE_CHECK_CUDA(cudaMemsetAsync(dws_up, 0, sn, cs));
      MOE_CHECK_CUDA(cudaMemsetAsync(dws_down, 0, sn, cs));
    }
    return MOE_OK;
  }
  int sms = 0;
  st = device_setup(&sms);
  if (st != MOE_OK) return st;
  char* base = static_cast<char*>(ws);
  int* ctr = reinterpret_cast<int*>(base + w.ctr);
  int* offs = reinterpret_cast<int*>(base + w.offs);    // checked offsets
  int* offpad = reinterpret_cast<int*>(base + w.offpad);
  float* dz = reinterpret_cast<float*>(base + w.dz);
  auto* X = reinterpret_cast<__nv_bfloat16*>(base + w.X);
  auto* dY = reinterpret_cast<__nv_bfloat16*>(base + w.dY);
  auto* dH = reinterpret_cast<__half*>(base + w.dH);
  auto* H = reinterpret_cast<__nv_bfloat16*>(base + w.H);
  auto* dA = reinterpret_cast<__nv_bfloat16*>(base + w.dA);
  auto* dX = reinterpret_cast<__half*>(base + w.dX);
  auto* dH_s = reinterpret_cast<__half*>(base + w.dH_s);
  auto* H_s = reinterpret_cast<__nv_bfloat16*>(base + w.H_s);
  auto* dA_s = reinterpret_cast<__nv_bfloat16*>(base + w.dA_s);
  auto* dX_s = reinterpret_cast<__half*>(base + w.dX_s);
  const long long A = static_cast<long long>(T) * K;
  const long long R = w.A_pad;

  // 1. checked and padded offsets; item counters
  bwd_offpad_kernel<<<1, 256, 0, cs>>>(offsets, N, A, offs, offpad, ctr,
                                       kBwdCounters);
  MOE_CHECK_LAUNCH();
  // 2. per-assignment operands and the gate gradient; zero padding rows
  bwd_gather_kernel<<<T, 128, 0, cs>>>(
      static_cast<const __nv_bfloat16*>(dh), static_cast<const __nv_bfloat16*>(u),
      topk_idx, topk_gate, inv, offs, offpad,
      static_cast<const __half*>(y_perm), d, K, N, A, R, dY, X, dz);
  MOE_CHECK_LAUNCH();
  bwd_zero_pad_kernel<<<N, 256, 0, cs>>>(offs, offpad, d, I, X, dY, H, dA,
                                         dz);
  MOE_CHECK_LAUNCH();

  const long long tok_items_r = cdiv(A, 256) + N;   // chunk bound
  const long long tok_items_s = S > 0 ? cdiv(T, 256) : 0;
  CUtensorMap a_r, b_r, a_s, b_s;
  BwdParams p{};
  p.offpad = offpad;
  p.offsets = offs;
  p.n_groups = N;
  p.shared_rows = S > 0 ? T : 0;
  p.I = I;

  // CTA pairs (256-row M tiles) when every M and N side splits into 256s
  const bool pair = d % 256 == 0 && I % 256 == 0;
  if (pair) {
    const bool sh = S > 0;
    const long long ti_r = cdiv(A, 256) + N;           // chunk bound
    const long long ti_s = sh ? cdiv(T, 256) : 0;
    const long long NI = static_cast<long long>(N) * I;
    BwdPairMaps m;
    // 3. Dgrad (down): dH = dY W_down, dH_s = dh Ws_down
    if ((st = bwd_pair_maps({w_down, static_cast<long long>(N) * d, I},
                            {dY, R, d}, {ws_down_packed, d, SI}, {dh, T, d},
                            sh, true, m)))
      return st;
    p.m_routed = I;  p.m_shared = SI;
    p.k_routed = d;  p.k_shared = d;
    set_dgrad_down_outputs(p, saved, act, act_shared, I, SI, dH, dH_s, H, H_s,
                           dA, dA_s);
    p.item_counter = ctr + 0;
    if ((st = launch_bwd_pair<kDgrad>(m, p, ti_r * (I / 256) +
                                                ti_s * (SI / 256), cs)))
      return st;
    p.act_r = p.act_s = nullptr;
    // 4. gate/up recomputed with the SwiGLU backward: H, dA (only without
    // the forward's saved pre-activations)
    if (!saved) {
      if ((st = bwd_pair_maps({w_gu_packed, 2 * NI, d}, {X, R, d},
                              {ws_gu_packed, 2LL * SI, d}, {u, T, d}, sh,
                              true, m)))
        return st;
      p.m_routed = 2 * I;  p.m_shared = 2 * SI;
      p.k_routed = d;      p.k_shared = d;
      p.dh_r = dH;         p.dh_s = dH_s;
      p.out_r = H;         p.ld_r = I;
      p.out_s = H_s;       p.ld_s = SI;
      p.out2_r = dA;       p.ld2_r = 2LL * I;
      p.out2_s = dA_s;     p.ld2_s = 2LL * SI;
      p.item_counter = ctr + 1;
      if ((st = launch_bwd_pair<kRecomp>(m, p, ti_r * (2 * I / 256) +
                                                   ti_s * (2 * SI / 256),
                                         cs)))
        return st;
    }
    // 5. Dgrad (gate/up): dX = dA W_gu, dX_s = dA_s Ws_gu
    if ((st = bwd_pair_maps({w_gu_packed, 2 * NI, d}, {dA, R, 2LL * I},
                            {ws_gu_packed, 2LL * SI, d}, {dA_s, T, 2LL * SI},
                            sh, true, m)))
      return st;
    p.m_routed = d;      p.m_shared = d;
    p.k_routed = 2 * I;  p.k_shared = 2 * SI;
    p.out_r = dX;        p.ld_r = d;
    p.out_s = dX_s;      p.ld_s = d;
    p.item_counter = ctr + 2;
    if ((st = launch_bwd_pair<kDgrad>(m, p, (ti_r + ti_s) * (d / 256), cs)))
      return st;
    // 6. Wgrad (gate/up): dW_gate / dW_up = dA^T X; shared dA_s^T u
    constexpr int kWbox = bwd_pair_bk<kWgrad>();
    if ((st = bwd_pair_maps({dA, R, 2LL * I}, {X, R, d},
                            {dA_s, T, 2LL * SI}, {u, T, d}, sh, false, m,
                            kWbox)))
      return st;
    p.m_routed = 2 * I;  p.m_shared = 2 * SI;
    p.n_routed = d;      p.n_shared = d;
    p.out_r = dw_gate;   p.out2_r = dw_up;   p.ld_r = d;
    p.out_s = dws_gate;  p.out2_s = dws_up;  p.ld_s = d;
    p.wgrad_gu = 1;
    p.out_bf16 = grad_dtype == MOE_BF16 ? 1 : 0;
    p.item_counter = ctr + 3;
    {
      const bool gb = p.out_bf16 != 0;
      if ((st = make_map_grad(&m.o_r, dw_gate, NI, d, gb))) return st;
      if ((st = make_map_grad(&m.o2_r, dw_up, NI, d, gb))) return st;
      if (sh) {
        if ((st = make_map_grad(&m.o_s, dws_gate, SI, d, gb))) return st;
        if ((st = make_map_grad(&m.o2_s, dws_up, SI, d, gb))) return st;
      } else {
        m.o_s = m.o_r;
        m.o2_s = m.o2_r;
      }
    }
    if ((st = launch_bwd_pair<kWgrad>(
             m, p,
             static_cast<long long>(N) * (2 * I / 256) * (d / 256) +
                 (sh ? static_cast<long long>(2 * SI / 256) * (d / 256) : 0),
             cs)))
      return st;
    // 7. Wgrad (down): dW_down = dY^T H; shared dh^T H_s
    if ((st = bwd_pair_maps({dY, R, d}, {H, R, I}, {dh, T, d}, {H_s, T, SI},
                            sh, false, m, kWbox)))
      return st;
    p.m_routed = d;   p.m_shared = d;
    p.n_routed = I;   p.n_shared = SI;
    p.out_r = dw_down;   p.out2_r = nullptr;  p.ld_r = I;
    p.out_s = dws_down;  p.out2_s = nullptr;  p.ld_s = I;
    p.wgrad_gu = 0;
    p.item_counter = ctr + 4;
    {
      const bool gb = p.out_bf16 != 0;
      if ((st = make_map_grad(&m.o_r, dw_down, static_cast<long long>(N) * d,
                              I, gb)))
        return st;
      if (sh) {
        if ((st = make_map_grad(&m.o_s, dws_down,
                                static_cast<long long>(S) * d, I, gb)))
          return st;
      } else {
        m.o_s = m.o_r;
      }
      m.o2_r = m.o_r;
      m.o2_s = m.o_s;
    }
    if ((st = launch_bwd_pair<kWgrad>(
             m, p,
             static_cast<long long>(N) * (d / 256) * (I / 256) +
                 (sh ? static_cast<long long>(d / 256) * (SI / 256) : 0),
             cs)))
      return st;
  } else {
    // 3. Dgrad (down): dH = dY W_down, dH_s = dh Ws_down
    if ((st = make_map(&a_r, w_down, static_cast<long long>(N) * d, I, 64)))
      return st;
    if ((st = make_map(&b_r, dY, R, d, kBoxRows))) return st;
    if (S > 0) {
      if ((st = make_map(&a_s, ws_down_packed, d, SI, 64))) return st;
      if ((st = make_map(&b_s, dh, T, d, kBoxRows))) return st;
    } else {
      a_s = a_r;
      b_s = b_r;
    }
    p.m_routed = I;  p.m_shared = SI;
    p.k_routed = d;  p.k_shared = d;
    set_dgrad_down_outputs(p, saved, act, act_shared, I, SI, dH, dH_s, H, H_s,
                           dA, dA_s);
    p.item_counter = ctr + 0;
    if ((st = launch_bwd_gemm<kDgrad, 256, 4>(
             a_r, b_r, a_s, b_s, p,
             tok_items_r * (I / 128) + tok_items_s * (SI / 128), sms, cs)))
      return st;
    p.act_r = p.act_s = nullptr;

    // 4. gate/up recomputed with the SwiGLU backward: H, dA (and shared),
    // only without the forward's saved pre-activations
    if (!saved) {
    if ((st = make_map(&a_r, w_gu_packed, 2LL * N * I, d, kGemmBM))) return st;
    if ((st = make_map(&b_r, X, R, d, kBoxRows))) return st;
    if (S > 0) {
      if ((st = make_map(&a_s, ws_gu_packed, 2LL * SI, d, kGemmBM))) return st;
      if ((st = make_map(&b_s, u, T, d, kBoxRows))) return st;
    } else {
      a_s = a_r;
      b_s = b_r;
    }
    p.m_routed = 2 * I;  p.m_shared = 2 * SI;
    p.k_routed = d;      p.k_shared = d;
    p.dh_r = dH;         p.dh_s = dH_s;
    p.out_r = H;         p.ld_r = I;
    p.out_s = H_s;       p.ld_s = SI;
    p.out2_r = dA;       p.ld2_r = 2LL * I;
    p.out2_s = dA_s;     p.ld2_s = 2LL * SI;
    p.item_counter = ctr + 1;
    if ((st = launch_bwd_gemm<kRecomp, 256, 4>(
             a_r, b_r, a_s, b_s, p,
             tok_items_r * (2 * I / 128) + tok_items_s * (2 * SI / 128), sms,
             cs)))
      return st;
    }

    // 5. Dgrad (gate/up): dX = dA W_gu, dX_s = dA_s Ws_gu
    if ((st = make_map(&a_r, w_gu_packed, 2LL * N * I, d, 64))) return st;
    if ((st = make_map(&b_r, dA, R, 2LL * I, kBoxRows))) return st;
    if (S > 0) {
      if ((st = make_map(&a_s, ws_gu_packed, 2LL * SI, d, 64))) return st;
      if ((st = make_map(&b_s, dA_s, T, 2LL * SI, kBoxRows))) return st;
    } else {
      a_s = a_r;
      b_s = b_r;
    }
    p.m_routed = d;      p.m_shared = d;
    p.k_routed = 2 * I;  p.k_shared = 2 * SI;
    p.out_r = dX;        p.ld_r = d;
    p.out_s = dX_s;      p.ld_s = d;
    p.item_counter = ctr + 2;
    if ((st = launch_bwd_gemm<kDgrad, 256, 4>(
             a_r, b_r, a_s, b_s, p,
             tok_items_r * (d / 128) + tok_items_s * (d / 128), sms, cs)))
      return st;

    // 6. Wgrad (gate/up): dW_gate / dW_up = dA^T X; shared dA_s^T u
    const bool gb = grad_dtype == MOE_BF16;
    if ((st = make_map(&a_r, dA, R, 2LL * I, 64))) return st;
    if ((st = make_map(&b_r, X, R, d, 64))) return st;
    if (S > 0) {
      if ((st = make_map(&a_s, dA_s, T, 2LL * SI, 64))) return st;
      if ((st = make_map(&b_s, u, T, d, 64))) return st;
    } else {
      a_s = a_r;
      b_s = b_r;
    }
    p.m_routed = 2 * I;  p.m_shared = 2 * SI;
    p.n_routed = d;      p.n_shared = d;
    p.out_r = dw_gate;   p.out2_r = dw_up;   p.ld_r = d;
    p.out_s = dws_gate;  p.out2_s = dws_up;  p.ld_s = d;
    p.wgrad_gu = 1;
    p.out_bf16 = gb ? 1 : 0;
    p.item_counter = ctr + 3;
    {
      const bool b256 = d % 256 == 0;
      const int bn = b256 ? 256 : 128;
      const long long items =
          static_cast<long long>(N) * (2 * I / 128) * cdiv(d, bn) +
          (S > 0 ? static_cast<long long>(2 * SI / 128) * cdiv(d, bn) : 0);
      st = b256 ? launch_bwd_gemm<kWgrad, 256, 4>(a_r, b_r, a_s, b_s, p, items,
                                                  sms, cs)
                : launch_bwd_gemm<kWgrad, 128, 6>(a_r, b_r, a_s, b_s, p, items,
                                                  sms, cs);
      if (st != MOE_OK) return st;
    }

    // 7. Wgrad (down): dW_down = dY^T H; shared dh^T H_s
    if ((st = make_map(&a_r, dY, R, d, 64))) return st;
    if ((st = make_map(&b_r, H, R, I, 64))) return st;
    if (S > 0) {
      if ((st = make_map(&a_s, dh, T, d, 64))) return st;
      if ((st = make_map(&b_s, H_s, T, SI, 64))) return st;
    } else {
      a_s = a_r;
      b_s = b_r;
    }
    p.m_routed = d;   p.m_shared = d;
    p.n_routed = I;   p.n_shared = SI;
    p.out_r = dw_down;   p.out2_r = nullptr;  p.ld_r = I;
    p.out_s = dws_down;  p.out2_s = nullptr;  p.ld_s = I;
    p.wgrad_gu = 0;
    p.item_counter = ctr + 4;
    {
      const bool b256 = I % 256 == 0 && SI % 256 == 0;
      const int bn = b256 ? 256 : 128;
      const long long items =
          static_cast<long long>(N) * (d / 128) * cdiv(I, bn) +
          (S > 0 ? static_cast<long long>(d / 128) * cdiv(SI, bn) : 0);
      st = b256 ? launch_bwd_gemm<kWgrad, 256, 4>(a_r, b_r, a_s, b_s, p, items,
                                                  sms, cs)
                : launch_bwd_gemm<kWgrad, 128, 6>(a_r, b_r, a_s, b_s, p, items,
                                                  sms, cs);
      if (st != MOE_OK) return st;
    }
  }

  // 8. centroid gradient; 9. input gradient
  bwd_centroid_grad_kernel<<<dim3(N, static_cast<unsigned>(cdiv(d, 1024))),
                             128, 0, cs>>>(offs, offpad, dz, X, d, dE);
  MOE_CHECK_LAUNCH();
  bwd_input_grad_kernel<<<T, 128, 0, cs>>>(
      static_cast<const __nv_bfloat16*>(dh), S > 0 ? dX_s : nullptr, dX,
      static_cast<const __nv_bfloat16*>(centroids), dz, topk_idx, inv, offs,
      offpad, d, K, N, A, du);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

}  // extern "C"
