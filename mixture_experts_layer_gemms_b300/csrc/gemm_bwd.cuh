// Grouped expert GEMMs of the layer BACKWARD pass on the tcgen05 tensor
// cores ("AI新顶流-DeepSeek 技术大揭秘", section "FP8混合精度训练框架": the
// Dgrad and Wgrad GEMMs of each linear operator; the layer is the FFN-output
// equation of "【推理llm論文精讀】DeepSeek V3技術論文", section 2.2).
//
// Three kinds of work, one persistent warp-specialised kernel (the forward's
// structure: TMA producer, single-thread MMA issuer, four epilogue warps,
// double-buffered TMEM accumulators, items claimed from a global counter):
//
//  kDgrad   D[m, n] = sum_k W[k, m] X[n, k]: the weight operand is read
//           MN-major (W stored [K rows, M contiguous]), tokens on N.
//           dH = dY W_down (W_down [d, I]: K = d, M = I) and
//           dX = dA W_gu   (packed W_gu [2I, d]: K = 2I, M = d).
//           Output fp16 [token][m]; or, for dH with the forward's saved
//           pre-activations a, c, the SwiGLU backward in the epilogue
//           (H and dA written instead of dH, as kRecomp writes them).
//  kRecomp  the forward's gate/up GEMM again (both operands K-major), with
//           the SwiGLU backward in the epilogue: from a, c (fp32, TMEM) and
//           dH it writes H = SiLU(a) c and dA = [dH c SiLU'(a) | dH SiLU(a)]
//           in the packed gate/up column order.  Only when the forward saved
//           no pre-activations.
//  kWgrad   D[m, n] = sum_k A[k, m] B[k, n] over the tokens of one group:
//           both operands MN-major (token rows, M or N contiguous); output
//           row-major per expert.  dW_gu = dA^T X  (gate/up rows unpacked to
//           W_gate / W_up), dW_down = dY^T H.
//
// Groups: the shared experts (all T tokens, one concatenated group) first,
// then the routed experts.  Routed token rows live in a padded layout: group
// e starts at offpad[e] (a multiple of 16) and holds cnt[e] rows, the rest
// of its 16-row blocks zero.  A Wgrad K block (64 rows) may run into the
// next group, but only its 16-row MMA steps up to the group's padded end
// are issued, so no product ever takes another group's rows.
#pragma once
#include "common.cuh"
#include "gemm.cuh"

namespace moe {

enum BwdKind : int { kDgrad = 0, kRecomp = 1, kWgrad = 2 };
constexpr int kPadRows = 16;   // routed groups are padded to this many rows
// epilogue staging: four warps x 32 x 33 floats (the Wgrad transpose; the
// Recomp exchange uses the first 4 x 32 x 17)
constexpr int kBwdStgBytes = 4 * 32 * 33 * 4;

// Shared-memory descriptor of an MN-major operand that TMA wrote as boxes of
// {64 MN elements (128 B), 64 K rows} with 128-byte swizzle.  Eight K rows
// form one 1024-byte swizzle atom (stride-dimension offset 1024 B between
// 8-row K groups); consecutive 64-wide MN blocks are one box apart
// (leading-dimension offset = box bytes).  Stepping K by 16 rows adds 2048 B
// to the start address.
__device__ __forceinline__ uint64_t sdesc_mn128(uint32_t saddr,
                                                uint32_t lbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}
// kind::f16 instruction descriptor with MN-major ("transposed") operands.
__host__ __device__ constexpr uint32_t idesc_bf16_mn(int M, int N, bool a_mn,
                                                     bool b_mn) {
  return idesc_bf16_f32(M, N) | (a_mn ? (1u << 15) : 0u) |
         (b_mn ? (1u << 16) : 0u);
}

struct BwdParams {
  const int* offpad;     // [n_groups+1] padded row offsets (device)
  const int* offsets;    // [n_groups+1] row offsets: cnt[e] = diff
  int n_groups;          // routed groups
  int shared_rows;       // T when there is a shared group, else 0
  int m_routed, m_shared;    // M-side rows of a group (multiples of 128)
  int k_routed, k_shared;    // Dgrad / Recomp: reduction length
  int n_routed, n_shared;    // Wgrad: N-side columns of a group
  int I;                     // one expert's intermediate size
  // outputs (meaning per kind, see the kernel comment)
  void* out_r;  long long ld_r;
  void* out_s;  long long ld_s;
  void* out2_r; long long ld2_r;     // Recomp: dA;   Wgrad gate/up: W_up grad
  void* out2_s; long long ld2_s;
  const __half* dh_r;  const __half* dh_s;   // Recomp: dH [token][i]
  // Dgrad of the down projection: when not null, the forward's saved
  // pre-activations [forward row][2I] (fp16, packed order); the epilogue
  // then writes H to out and dA to out2 instead of dH (no recompute pass)
  const __half* act_r;  long long ld_act_r;
  const __half* act_s;  long long ld_act_s;
  int wgrad_gu;          // Wgrad: 1 gate/up (unpack rows), 0 down
  int out_bf16;          // Wgrad: gradients stored as bf16 (else fp32)
  int* item_counter;
};

template <int BN, int STAGES>
struct BwdSmem {
  static constexpr int a_bytes = kGemmBM * kGemmBK * 2;   // 16 KB
  static constexpr int b_bytes = BN * kGemmBK * 2;
  static constexpr int a_off = 0;
  static constexpr int b_off = a_off + STAGES * a_bytes;
  static constexpr int stg_off = b_off + STAGES * b_bytes;
  static constexpr int stg_bytes = kBwdStgBytes;
  static constexpr int bar_off = stg_off + stg_bytes;
  static constexpr int n_bars = 2 * STAGES + 5 + 2 * kSchedDepth;
  static constexpr int misc_off = bar_off + n_bars * 8;
  static constexpr int epok_off = misc_off + 16;
  static constexpr int sched_off = epok_off + 16;
  static constexpr int tab_off = sched_off + 4 * kSchedDepth;
  static constexpr int total = tab_off + 3 * (kMaxGroups + 1) * 4;
  static constexpr int alloc = total + 1024;
  static constexpr int tmem_cols = 2 * BN;
  static_assert(alloc <= 227 * 1024, "shared memory");
};

struct BTile {
  int shared;    // 1: the shared group
  int e;         // routed group
  int wt;        // M tile inside the group
  int m0;        // first M row (wt * 128)
  int n0;        // tokens kinds: first token row; Wgrad: first column
  int n_valid;   // tokens kinds: tokens; Wgrad: columns
  int n_mma;     // MMA N
  int k_row0;    // first K row of the MN-major operands (Dgrad A, Wgrad A/B)
  int nk;        // K blocks (64 rows; 128 for the CTA-pair token kinds)
  int krows;     // K rows to multiply, a multiple of 16 (a Wgrad group's
                 // last block may hold fewer rows than the block)
};

// Item tables in shared memory: offpad, cnt and (tokens kinds) the prefix
// of BN-token chunks per group.
template <int KIND, int BN>
__device__ __forceinline__ BTile bwd_decode(int item, const BwdParams& p,
                                            int n_items_s, int nch_s,
                                            const int* offp, const int* cnt,
                                            const int* chunk_pre) {
  BTile t;
  if constexpr (KIND == kWgrad) {
    const int ntn_s = (p.n_shared + BN - 1) / BN;
    const int ntn_r = (p.n_routed + BN - 1) / BN;
    const int per_r = (p.m_routed / kGemmBM) * ntn_r;
    int local, ntn, ncols;
    if (item < n_items_s) {
      t.shared = 1;
      t.e = 0;
      local = item;
      ntn = ntn_s;
      ncols = p.n_shared;
      t.k_row0 = 0;
      t.nk = (p.shared_rows + kGemmBK - 1) / kGemmBK;
      t.krows = t.nk * kGemmBK;       // rows past T read as zero
    } else {
      const int j = item - n_items_s;
      t.shared = 0;
      t.e = j / per_r;
      local = j % per_r;
      ntn = ntn_r;
      ncols = p.n_routed;
      t.k_row0 = offp[t.e];
      t.krows = (cnt[t.e] + kPadRows - 1) / kPadRows * kPadRows;
      t.nk = (t.krows + kGemmBK - 1) / kGemmBK;
    }
    t.wt = local / ntn;
    t.m0 = t.wt * kGemmBM;
    t.n0 = (local % ntn) * BN;
    t.n_valid = min(BN, ncols - t.n0);
    t.n_mma = BN;
  } else {
    if (item < n_items_s) {
      const int wt = item / nch_s, ch = item % nch_s;
      t.shared = 1;
      t.e = 0;
      t.wt = wt;
      t.n0 = ch * BN;
      t.n_valid = min(BN, p.shared_rows - t.n0);
      t.k_row0 = 0;
      t.nk = p.k_shared / kGemmBK;
    } else {
      const int wt_r = p.m_routed / kGemmBM;
      const int j = item - n_items_s;
      int lo = 0, hi = p.n_groups;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (chunk_pre[mid] * wt_r <= j) lo = mid; else hi = mid;
      }
      const int e = lo;
      const int ce = chunk_pre[e + 1] - chunk_pre[e];
      const int local = j - chunk_pre[e] * wt_r;
      const int wt = local / ce, ch = local % ce;
      t.shared = 0;
      t.e = e;
      t.wt = wt;
      t.n0 = offp[e] + ch * BN;
      t.n_valid = min(BN, cnt[e] - ch * BN);
      t.k_row0 = e * p.k_routed;
      t.nk = p.k_routed / kGemmBK;
    }
    t.m0 = t.wt * kGemmBM;
    t.n_mma = (t.n_valid + 15) & ~15;
    t.krows = t.nk * kGemmBK;
  }
  return t;
}

// --- epilogues (four warps, 128 threads; thread (q, lane) owns M row
// q*32 + lane of the accumulator) ------------------------------------------

// kDgrad: out[token][m0 + row] (fp16), 32 tokens per tcgen05.ld.
__device__ __forceinline__ void bwd_ep_dgrad(uint32_t taddr, int n_valid,
                                             int b_row, __half* out,
                                             long long ld, int col, bool& ovf) {
  for (int n0 = 0; n0 < n_valid; n0 += 32) {
    uint32_t r[32];
    tmem_ld32(taddr + n0, r);
    tmem_ld_wait();
    const int nleft = n_valid - n0;
    __half* dst = out + static_cast<size_t>(b_row + n0) * ld + col;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < nleft) {
        const float v = __uint_as_float(r[j]);
        ovf |= !(fabsf(v) <= 65504.f);
        dst[static_cast<size_t>(j) * ld] = __float2half_rn(v);
      }
  }
}

// kDgrad of the down projection with the SwiGLU backward taken from the
// forward's saved pre-activations.  The thread's M row is intermediate
// column i = `col`; the accumulator holds dH (fp32) for 32 tokens per load.
// a and c of padded row `row` are at act[row + shift][ca] and [ca + 64]
// (fp16, packed order: ca = 128 (i / 64) + i % 64; shift maps the padded
// row to the forward's row), and
//   H[row][i]        = SiLU(a) c                                (bf16)
//   dA[row][ca]      = dH c SiLU'(a)   (gate half)              (bf16)
//   dA[row][ca + 64] = dH SiLU(a)      (up half)                (bf16)
// dH stays fp32 here (the recompute path rounds it to fp16 in between).
__device__ __forceinline__ void bwd_ep_dgrad_act(
    uint32_t taddr, int n_valid, int b_row, int col, long long shift,
    const __half* __restrict__ act, long long ld_act,
    __nv_bfloat16* H, long long ld_h, __nv_bfloat16* dA, long long ld_a) {
  const int ca = (col >> 6) * 128 + (col & 63);
  for (int n0 = 0; n0 < n_valid; n0 += 32) {
    const int nleft = n_valid - n0;
    // the chunk's a and c, loaded before the TMEM read so that their
    // latency overlaps it
    const __half* src =
        act + static_cast<size_t>(b_row + n0 + shift) * ld_act + ca;
    __half av[32], cv[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (j < nleft) {
        av[j] = src[static_cast<size_t>(j) * ld_act];
        cv[j] = src[static_cast<size_t>(j) * ld_act + 64];
      } else {
        av[j] = cv[j] = __float2half_rn(0.f);
      }
    }
    uint32_t r[32];
    tmem_ld32(taddr + n0, r);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (j >= nleft) continue;
      const float a = __half2float(av[j]);
      const float c = __half2float(cv[j]);
      const float g = __uint_as_float(r[j]);
      const float sg = 1.0f / (1.0f + expf(-a));
      const float si = a * sg;
      const size_t row = static_cast<size_t>(b_row + n0 + j);
      H[row * ld_h + col] = __float2bfloat16_rn(si * c);
      dA[row * ld_a + ca] =
          __float2bfloat16_rn(g * c * (sg * (1.0f + a * (1.0f - sg))));
      dA[row * ld_a + ca + 64] = __float2bfloat16_rn(g * si);
    }
  }
}

// kRecomp: rows 0..63 of the tile are gate pre-activations a, rows 64..127
// the up values c of intermediate columns i0 + 0..63 (packed order).  Warps
// q and q+2 swap half their tokens (as the forward's SwiGLU epilogue) so that
// each holds a and c of 16 tokens for its 32 columns, then write
//   H[token][i]           = SiLU(a) c                        (bf16)
//   dA[token][blk + i']   = dH c SiLU'(a)   (gate half)       (bf16)
//   dA[token][blk+64+i']  = dH SiLU(a)      (up half)         (bf16)
// with dH read from dH[token][i] (fp16).
// The warps of one exchange group (four warps, lane quarters 0..3) take
// the 32-token chunks n0 = c0, c0 + step, ... and synchronise on named
// barrier `bar` (several groups may split an item's chunks).
__device__ __forceinline__ void bwd_ep_recomp(
    uint32_t taddr, int n_valid, int b_row, int wt, const __half* dH,
    long long ld_h, __nv_bfloat16* H, __nv_bfloat16* dA, long long ld_a,
    float* xchg, int q, int lane, int c0 = 0, int step = 32, int bar = 1) {
  const bool gate_warp = q < 2;
  const int pair_q = q & 1;
  const int i = wt * 64 + pair_q * 32 + lane;        // column of H / dH
  const int ca = wt * 128 + pair_q * 32 + lane;      // packed column of da
  const int jbase = gate_warp ? 0 : 16;
  for (int n0 = c0; n0 < n_valid; n0 += step) {
    const int nleft = n_valid - n0;
    // this thread's 16 dH values, loaded before the TMEM read and the
    // exchange so that their latency overlaps them (the H / dA stores
    // below could alias dH as far as the compiler knows)
    float gv[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      gv[j] = jbase + j < nleft
                  ? __half2float(dH[static_cast<size_t>(b_row + n0 + jbase + j) *
                                        ld_h + i])
                  : 0.f;
    uint32_t r[32];
    tmem_ld32(taddr + n0, r);
    tmem_ld_wait();
    float* mine = xchg + ((q * 32) + lane) * 17;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      mine[j] = __uint_as_float(r[gate_warp ? 16 + j : j]);
    named_bar_sync(bar, 128);
    const float* theirs =
        xchg + (((gate_warp ? q + 2 : q - 2) * 32) + lane) * 17;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (jbase + j >= nleft) continue;
      const float a = gate_warp ? __uint_as_float(r[j]) : theirs[j];
      const float c = gate_warp ? theirs[j] : __uint_as_float(r[16 + j]);
      const size_t row = static_cast<size_t>(b_row + n0 + jbase + j);
      const float g = gv[j];
      const float sg = 1.0f / (1.0f + expf(-a));
      const float si = a * sg;
      H[row * ld_h + i] = __float2bfloat16_rn(si * c);
      dA[row * ld_a + ca] =
          __float2bfloat16_rn(g * c * (sg * (1.0f + a * (1.0f - sg))));
      dA[row * ld_a + ca + 64] = __float2bfloat16_rn(g * si);
    }
    named_bar_sync(bar, 128);
  }
}

// kWgrad output row m of a group's M side (gate/up: the packed row index,
// 128-row blocks of 64 gate then 64 up rows; down: the row of W_down): the
// address of its column 0, the byte stride to row m + 1 (rows of one warp
// are consecutive), and the column mapping of the shared down gradient
// (col_split = I: column c of the [d, S*I] tile is expert c / I's column
// c % I, s_stride elements apart).
struct WgradRow {
  char* p;
  long long row_bytes;
  int col_split;
  long long s_stride;
};
__device__ __forceinline__ WgradRow wgrad_row(const BwdParams& p, bool shared,
                                              int e, int m) {
  const int esz = p.out_bf16 ? 2 : 4;
  WgradRow w;
  w.col_split = 0;
  w.s_stride = 0;
  if (p.wgrad_gu) {
    const int within = m & 127;
    const long long irow = static_cast<long long>(m >> 7) * 64 + (within & 63);
    const long long ld = shared ? p.ld_s : p.ld_r;   // = d
    const long long base = shared ? 0 : static_cast<long long>(e) * p.I;
    char* g = static_cast<char*>(within < 64 ? (shared ? p.out_s : p.out_r)
                                             : (shared ? p.out2_s : p.out2_r));
    w.p = g + (base + irow) * ld * esz;
    w.row_bytes = ld * esz;
  } else {
    const long long ld = shared ? p.ld_s : p.ld_r;   // = I
    char* g = static_cast<char*>(shared ? p.out_s : p.out_r);
    if (shared) {       // [S][d][I]
      w.col_split = p.I;
      w.s_stride = static_cast<long long>(p.m_shared) * p.I;
      w.p = g + static_cast<long long>(m) * ld * esz;
    } else {            // [N][d][I]
      w.p = g + (static_cast<long long>(e) * p.m_routed + m) * ld * esz;
    }
    w.row_bytes = ld * esz;
  }
  return w;
}

// kWgrad epilogue of one warp: its 32 accumulator rows (TMEM lanes) x
// columns n0 .. n0 + n_valid of the tile, row-major.  Each 32-column chunk
// goes through a 32 x 33 float block in shared memory so that every store
// instruction writes whole column runs of one row (fp32: 128 B) or of two
// rows (bf16: 2 x 64 B).  `zero`: no accumulation happened (the group has
// no rows); zeros are stored.
__device__ __forceinline__ void bwd_ep_wgrad_warp(uint32_t taddr, int n0,
                                                  int n_valid, int bn,
                                                  bool zero, const WgradRow& w,
                                                  bool bf16, float* st,
                                                  int lane) {
  const int esz = bf16 ? 2 : 4;
#pragma unroll 1
  for (int c0 = 0; c0 < bn && c0 < n_valid; c0 += 32) {
    uint32_t r[32];
    if (!zero) {
      tmem_ld32(taddr + c0, r);
      tmem_ld_wait();
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) r[j] = 0u;
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) st[lane * 33 + j] = __uint_as_float(r[j]);
    __syncwarp();
    const long long c = n0 + c0;
    const long long off =
        w.col_split > 0 ? (c / w.col_split) * w.s_stride + c % w.col_split : c;
    char* base = w.p + off * esz;
    if (bf16) {
      const int half = lane >> 4, cc = (lane & 15) * 2;
#pragma unroll 4
      for (int rr = 0; rr < 32; rr += 2) {
        const int row = rr + half;
        *reinterpret_cast<uint32_t*>(base + row * w.row_bytes + cc * 2) =
            pack_bf16x2(st[row * 33 + cc], st[row * 33 + cc + 1]);
      }
    } else {
#pragma unroll 4
      for (int rr = 0; rr < 32; ++rr)
        *reinterpret_cast<float*>(base + rr * w.row_bytes + lane * 4) =
            st[rr * 33 + lane];
    }
    __syncwarp();
  }
}

// Operand maps: A (weights for the tokens kinds, token-row operand for
// Wgrad) and B, routed and shared.
template <int KIND, int BN, int STAGES>
__global__ void __launch_bounds__(192, 1)
bwd_gemm_kernel(const __grid_constant__ CUtensorMap tmA_r,
                const __grid_constant__ CUtensorMap tmB_r,
                const __grid_constant__ CUtensorMap tmA_s,
                const __grid_constant__ CUtensorMap tmB_s,
                const BwdParams p) {
  using L = BwdSmem<BN, STAGES>;
  constexpr bool kTokens = KIND != kWgrad;
  constexpr bool kAmn = KIND != kRecomp;
  constexpr bool kBmn = KIND == kWgrad;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + L::bar_off;
  const uint32_t bar_empty = bar_full + 8 * STAGES;
  const uint32_t bar_tfull = bar_empty + 8 * STAGES;    // [2]
  const uint32_t bar_tempty = bar_tfull + 16;           // [2]
  const uint32_t bar_final = bar_tempty + 16;
  volatile uint32_t* tmem_slot =
      reinterpret_cast<volatile uint32_t*>(smem + L::misc_off);
  volatile int* abort_flag =
      reinterpret_cast<volatile int*>(smem + L::misc_off + 4);
  volatile int* bad_flag =
      reinterpret_cast<volatile int*>(smem + L::misc_off + 8);
  volatile int* ep_ok = reinterpret_cast<volatile int*>(smem + L::epok_off);
  int* offp = reinterpret_cast<int*>(smem + L::tab_off);       // [G+1]
  int* cnt = offp + (kMaxGroups + 1);                          // [G]
  int* chunk_pre = cnt + (kMaxGroups + 1);                     // [G+1]
  float* stg = reinterpret_cast<float*>(smem + L::stg_off);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.n_groups;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_tfull + 8 * a, 1);
      mbar_init(bar_tempty + 8 * a, 128);
    }
    mbar_init(bar_final, 1);
    for (int i = 0; i < kSchedDepth; ++i) {
      mbar_init(bar_final + 8 + 8 * i, 1);
      mbar_init(bar_final + 8 + 8 * kSchedDepth + 8 * i, 5);
    }
    *abort_flag = 0;
    *bad_flag = 0;
    fence_mbar_init();
    if (G > 0) {
      tma_prefetch_desc(&tmA_r);
      tma_prefetch_desc(&tmB_r);
    }
    if (p.shared_rows > 0) {
      tma_prefetch_desc(&tmA_s);
      tma_prefetch_desc(&tmB_s);
    }
  }
  if (warp == 1) {
    tmem_alloc(sbase + L::misc_off, L::tmem_cols);
    tmem_relinquish();
  }
  for (int e = threadIdx.x; e < G; e += blockDim.x) {
    const int o = p.offpad[e], c = p.offsets[e + 1] - p.offsets[e];
    offp[e] = o;
    cnt[e] = c;
    if (c < 0 || o < 0 || (o & (kPadRows - 1)) != 0) *bad_flag = 1;
    chunk_pre[e + 1] = c > 0 ? (c + BN - 1) / BN : 0;
  }
  if (threadIdx.x == 0) chunk_pre[0] = 0;
  __syncthreads();
  for (int e = threadIdx.x; e < G; e += blockDim.x)   // segments fit
    if (e + 1 < G && offp[e] + cnt[e] > offp[e + 1]) *bad_flag = 1;
  if (kTokens && warp == 0) {
    int carry = 0;
    for (int base = 1; base <= G; base += 32) {
      const int i = base + lane;
      int v = (i <= G) ? chunk_pre[i] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
      }
      if (i <= G) chunk_pre[i] = v + carry;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool bad = *bad_flag != 0;
  if (bad && threadIdx.x == 0) report_error(ERR_CHECK, KID_GEMM_BWD, 0);

  int n_items_s = 0, nch_s = 0, n_items = 0;
  if constexpr (kTokens) {
    nch_s = p.shared_rows > 0 ? (p.shared_rows + BN - 1) / BN : 0;
    n_items_s = nch_s * (p.m_shared / kGemmBM);
    n_items = n_items_s +
              (G > 0 ? chunk_pre[G] * (p.m_routed / kGemmBM) : 0);
  } else {
    n_items_s = p.shared_rows > 0
                    ? (p.m_shared / kGemmBM) * ((p.n_shared + BN - 1) / BN)
                    : 0;
    n_items = n_items_s +
              G * (p.m_routed / kGemmBM) * ((p.n_routed + BN - 1) / BN);
  }
  if (bad) n_items = 0;
  const uint32_t bar_sfull = bar_final + 8;
  const uint32_t bar_sempty = bar_sfull + 8 * kSchedDepth;
  volatile int* sched = reinterpret_cast<volatile int*>(smem + L::sched_off);

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer + scheduler ----------------
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      int slot = 0;
      uint32_t sph = 0;
      int item = bad ? n_items : atomicAdd(p.item_counter, 1);
      while (!*abort_flag) {
        if (!mbar_wait(bar_sempty + 8 * slot, sph ^ 1, abort_flag,
                       KID_GEMM_BWD, 5))
          break;
        sched[slot] = item;
        mbar_arrive(bar_sfull + 8 * slot);
        if (++slot == kSchedDepth) {
          slot = 0;
          sph ^= 1;
        }
        if (item >= n_items) break;
        const BTile t = bwd_decode<KIND, BN>(item, p, n_items_s, nch_s, offp,
                                             cnt, chunk_pre);
        const int next = atomicAdd(p.item_counter, 1);
        const CUtensorMap* mA = t.shared ? &tmA_s : &tmA_r;
        const CUtensorMap* mB = t.shared ? &tmB_s : &tmB_r;
        int nbox = 0;
        uint32_t bytes = L::a_bytes;
        if constexpr (kTokens) {
          nbox = (t.n_mma + kBoxRows - 1) / kBoxRows;
          bytes += nbox * kBoxRows * kGemmBK * 2;
        } else {
          bytes += L::b_bytes;
        }
        bool ok = true;
        for (int i = 0; i < t.nk; ++i) {
          if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1, abort_flag,
                         KID_GEMM_BWD, 1)) {
            ok = false;
            break;
          }
          const int k0 = i * kGemmBK;
          const uint32_t fb = bar_full + 8 * stage;
          const uint32_t adst = sbase + L::a_off + stage * L::a_bytes;
          const uint32_t bdst = sbase + L::b_off + stage * L::b_bytes;
          mbar_arrive_expect_tx(fb, bytes);
          if constexpr (kAmn) {
            // two {64 M, 64 K} boxes
            tma_load_2d(adst, mA, t.m0, t.k_row0 + k0, fb);
            tma_load_2d(adst + 8192, mA, t.m0 + 64, t.k_row0 + k0, fb);
          } else {
            const int arow = (t.shared ? 0 : t.e * p.m_routed) + t.m0;
            tma_load_2d(adst, mA, k0, arow, fb);
          }
          if constexpr (kBmn) {
#pragma unroll
            for (int h = 0; h < BN / 64; ++h)
              tma_load_2d(bdst + h * 8192, mB, t.n0 + 64 * h, t.k_row0 + k0,
                          fb);
          } else {
            for (int bx = 0; bx < nbox; ++bx)
              tma_load_2d(bdst + bx * kBoxRows * kGemmBK * 2, mB, k0,
                          t.n0 + bx * kBoxRows, fb);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        item = next;
      }
      if (*abort_flag) {
        for (int j = 0; j < STAGES && j < issued; ++j) {
          int st = stage - 1 - j;
          uint32_t ph = phase;
          if (st < 0) {
            st += STAGES;
            ph ^= 1;
          }
          mbar_drain(bar_full + 8 * st, ph);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      int slot = 0;
      uint32_t sph = 0;
      while (!*abort_flag) {
        if (!mbar_wait(bar_sfull + 8 * slot, sph, abort_flag, KID_GEMM_BWD,
                       6))
          break;
        const int item = sched[slot];
        mbar_arrive(bar_sempty + 8 * slot);
        if (++slot == kSchedDepth) {
          slot = 0;
          sph ^= 1;
        }
        if (item >= n_items) break;
        const BTile t = bwd_decode<KIND, BN>(item, p, n_items_s, nch_s, offp,
                                             cnt, chunk_pre);
        if (!mbar_wait(bar_tempty + 8 * acc, acc_phase ^ 1, abort_flag,
                       KID_GEMM_BWD, 2))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * BN;
        const uint32_t idesc = idesc_bf16_mn(kGemmBM, t.n_mma, kAmn, kBmn);
        bool ok = true;
        for (int i = 0; i < t.nk; ++i) {
          if (!mbar_wait(bar_full + 8 * stage, phase, abort_flag,
                         KID_GEMM_BWD, 3)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = sbase + L::a_off + stage * L::a_bytes;
          const uint32_t b0 = sbase + L::b_off + stage * L::b_bytes;
          // 16-row K steps in this block (a Wgrad group's last block may
          // end early)
          const int nkk = min(kGemmBK, t.krows - i * kGemmBK) / 16;
#pragma unroll
          for (int kk = 0; kk < kGemmBK / 16; ++kk) {
            if (kk >= nkk) break;
            const uint64_t ad = kAmn ? sdesc_mn128(a0 + kk * 2048, 8192)
                                     : sdesc_k128(a0 + kk * 32);
            const uint64_t bd = kBmn ? sdesc_mn128(b0 + kk * 2048, 8192)
                                     : sdesc_k128(b0 + kk * 32);
            mma_bf16(d_tmem, ad, bd, idesc, (i | kk) != 0);
          }
          mma_commit(bar_empty + 8 * stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit(bar_tfull + 8 * acc);   // also fires for nk == 0
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      mma_commit(bar_final);
      mbar_drain(bar_final, 0);
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int ep = warp - 2;
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    int slot = 0;
    uint32_t sph = 0;
    bool ovf = false;
    while (true) {
      const bool got = mbar_wait(bar_sfull + 8 * slot, sph, abort_flag,
                                 KID_GEMM_BWD, 7);
      const int item = got ? sched[slot] : n_items;
      __syncwarp();
      if (got && lane == 0) mbar_arrive(bar_sempty + 8 * slot);
      if (++slot == kSchedDepth) {
        slot = 0;
        sph ^= 1;
      }
      bool ok = got;
      if (got && item < n_items)
        ok = mbar_wait(bar_tfull + 8 * acc, acc_phase, abort_flag,
                       KID_GEMM_BWD, 4);
      const bool wok = __all_sync(0xffffffffu, ok);
      if (lane == 0) ep_ok[ep] = wok ? 1 : 0;
      named_bar_sync(1, 128);
      if (!(ep_ok[0] && ep_ok[1] && ep_ok[2] && ep_ok[3])) break;
      if (item >= n_items) break;
      const BTile t = bwd_decode<KIND, BN>(item, p, n_items_s, nch_s, offp,
                                           cnt, chunk_pre);
      tc_fence_after();
      const uint32_t ta =
          tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      const int row = q * 32 + lane;   // M row of the tile
      if constexpr (KIND == kDgrad) {
        const __half* act = t.shared ? p.act_s : p.act_r;
        if (act != nullptr) {
          const long long shift =
              t.shared ? 0 : static_cast<long long>(p.offsets[t.e]) - offp[t.e];
          bwd_ep_dgrad_act(
              ta, t.n_valid, t.n0, t.m0 + row, shift, act,
              t.shared ? p.ld_act_s : p.ld_act_r,
              static_cast<__nv_bfloat16*>(t.shared ? p.out_s : p.out_r),
              t.shared ? p.ld_s : p.ld_r,
              static_cast<__nv_bfloat16*>(t.shared ? p.out2_s : p.out2_r),
              t.shared ? p.ld2_s : p.ld2_r);
        } else {
          __half* out = static_cast<__half*>(t.shared ? p.out_s : p.out_r);
          const long long ld = t.shared ? p.ld_s : p.ld_r;
          bwd_ep_dgrad(ta, t.n_valid, t.n0, out, ld, t.m0 + row, ovf);
        }
      } else if constexpr (KIND == kRecomp) {
        bwd_ep_recomp(ta, t.n_valid, t.n0, t.wt,
                      t.shared ? p.dh_s : p.dh_r,
                      t.shared ? p.ld_s : p.ld_r,
                      static_cast<__nv_bfloat16*>(t.shared ? p.out_s : p.out_r),
                      static_cast<__nv_bfloat16*>(t.shared ? p.out2_s
                                                           : p.out2_r),
                      t.shared ? p.ld2_s : p.ld2_r, stg, q, lane);
      } else {
        // this warp's rows t.m0 + q*32 .. +31
        const WgradRow w = wgrad_row(p, t.shared != 0, t.e, t.m0 + q * 32);
        bwd_ep_wgrad_warp(ta, t.n0, t.n_valid, BN, t.nk == 0, w,
                          p.out_bf16 != 0, stg + q * 32 * 33, lane);
      }
      tc_fence_before();
      mbar_arrive(bar_tempty + 8 * acc);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    if (ovf) report_error(ERR_CHECK, KID_GEMM_BWD, 200);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::tmem_cols);
  }
}

}  // namespace moe
