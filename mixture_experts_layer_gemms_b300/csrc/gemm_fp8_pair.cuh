// Grouped e4m3 expert GEMMs on CTA pairs with block scaling in the tensor
// core (tcgen05.mma kind::mxf8f6f4.block_scale).
// ("【推理llm論文精讀】DeepSeek V3技術論文", section 2.2: FFN^(r)_i of each
// selected expert and FFN^(s) of every shared expert; DeepSeek-V3 report
// commentary, cooktownmusic.com, FP8 part, Fig. 7a/7b: fine-grained block
// scales and partial sums kept in fp32.)
//
// Operands are the e4m3 codes and power-of-two block scales of the MOE_FP8
// layout (weights: 128 x 128 blocks, activations: 1 x 128 along the
// reduction).  The tensor core applies the scales itself: every 32 of the
// reduction carry one UE8M0 scale per row of each operand, so a 128-block's
// scale is given to its four 32-wide MMA steps.  Since the scales are powers
// of two, sum_k (2^ea x_k)(2^eb w_k) over a block equals 2^(ea+eb) times the
// block's partial sum -- the per-block promotion of the pages' Fig. 7b --
// and the fp32 accumulator carries the whole reduction, with no promotion
// pass on the CUDA cores.
//
// Items, orientation and schedule follow the bf16 CTA-pair kernel: weight
// rows on M (256 per item, 128 per CTA), tokens on N (at most 192 per item,
// in equal chunks), shared experts first, dynamic claim order, item table
// from the device offsets.  A stage is 256 of the reduction: two 128-byte
// K-atoms per row of e4m3, 32 KB of weights and <= 24 KB of tokens per CTA,
// three stages (each K-atom is a 128-byte-swizzled block of its rows).
// Gate/up items load each CTA's weight half as one 5-D box (per K-atom the
// CTA's 64 gate rows and the 64 up rows of the same intermediates), so SwiGLU pairs
// TMEM lanes l and l + 64 as in the bf16 kernel.  An item's 128 H columns
// (64 per CTA) are exactly one 1 x 128 quantization block of the down pass,
// so the epilogue requantizes H to e4m3 itself: per token, the block's
// largest |H| from both CTAs (exchanged through distributed shared memory),
// its exponent, the codes and the scales, from the same fp32 values the
// other e4m3 kernels quantize (a bf16 H would round twice).  Without the
// q8 outputs H leaves as fp32 instead.
//
// TMEM (512 columns per CTA): accumulators at columns 0 and 256 (192
// columns each), four scale groups at columns 192, 224, 448 and 480 (A
// scales 4 columns at +0, B scales 6 columns at +16).  One group holds the
// scales of four consecutive 128-blocks of the reduction (two stages): the
// MMAs of block kb use group kb / 4 and scale byte kb % 4; the scale warps
// run up to three groups ahead.
//
// Scales travel apart from the operands, as UE8M0 tables written by the
// quantizers (one byte per row and 128-block of the reduction, rows padded
// to 16-byte multiples).  At the start of an item each CTA's producer
// copies the item's token rows of the table and the two (gate/up) or one
// (down) weight row blocks into an item slot of shared memory with two bulk
// copies.  Four scale warps per CTA (one per lane quarter) then build each
// group from the slot -- one 32-bit word holds a row's four scale bytes of
// the group -- and store it with tcgen05.st; the even CTA's MMA thread
// waits for both CTAs' scale warps before a group's first MMA, and releases
// the group by an MMA commit after its last.
//
// Barriers (in each CTA; "L" = the even CTA): as the bf16 pair kernel, plus
//   isfull[j]  (both)   : the bulk copies of item scale slot j landed
//   isempty[j] (both)   : the 4 scale warps are done with item slot j
//   sffull[g]  (L only) : one arrival per scale warp of both CTAs
//   sfempty[g] (both)   : MMA commit multicast (group g's MMAs are done)
//   amx[c]     (both)   : the other CTA's 4 epilogue warps' token maxima of
//                         chunk parity c landed (st.async transaction bytes;
//                         fused requantization)
#pragma once
#include "common.cuh"
#include "gemm.cuh"
#include "quant.cuh"

namespace moe {

constexpr int kF8PBM = 256;       // packed weight rows per item (128 per CTA)
constexpr int kF8PBN = 192;       // max tokens per item
constexpr int kF8PStages = 3;
constexpr int kF8PAtoms = 2;      // 128-byte K-atoms per stage
constexpr int kF8PSfGroups = 4;   // scale groups in TMEM
constexpr int kF8PMaxPitch = 64;  // UE8M0 row bytes (reductions <= 8192)
// TMEM columns: accumulator a at a * 256; scale group g at 192 + 32 (g % 2)
// + 256 (g / 2)
__host__ __device__ constexpr uint32_t f8p_acc_col(int a) {
  return static_cast<uint32_t>(a) * 256u;
}
__host__ __device__ constexpr uint32_t f8p_sf_col(int g) {
  return 192u + 32u * static_cast<uint32_t>(g & 1) +
         256u * static_cast<uint32_t>(g >> 1);
}
constexpr int kF8PThreads = 320;  // producer, MMA, 4 epilogue, 4 scale warps

struct F8PairParams {
  const int* offsets;        // routed group row offsets [n_groups + 1]
  int n_groups;
  int w_rows_routed;         // packed weight rows per routed group
  int k_routed;              // reduction length (elements = bytes)
  long long max_routed_rows;
  int shared_rows;
  int w_rows_shared;
  int k_shared;
  int gate_up;               // 1: gate/up pass (SwiGLU epilogue, fp32 H)
  // UE8M0 scale tables, row pitch bytes (a multiple of 16): weights
  // [rows / 128][pitch] by packed row block, tokens [rows][pitch]
  const uint8_t* sw_routed;
  const uint8_t* sw_shared;
  const uint8_t* sx_routed;
  const uint8_t* sx_shared;
  int pitch_routed;
  int pitch_shared;
  void* out_routed;          // gate/up: H fp32; down: Y fp16
  long long ld_routed;
  void* out_shared;
  long long ld_shared;
  int* item_counter;         // zeroed before the launch
  // gate/up pass: when q8_routed is not null, H is requantized in the
  // epilogue instead of stored as fp32: e4m3 codes [rows][ld_*], fp32
  // scales [ld_* / 128][rows] (column = row) and the UE8M0 table
  // [rows][qpitch_*], the layout the activation quantizer writes
  uint8_t* q8_routed;
  float* qs_routed;
  uint8_t* qe_routed;
  int qpitch_routed;
  uint8_t* q8_shared;
  float* qs_shared;
  uint8_t* qe_shared;
  int qpitch_shared;
};

struct F8PairSmem {
  static constexpr int a_atom = 128 * 128;         // 16 KB per K-atom
  static constexpr int a_bytes = kF8PAtoms * a_atom;
  static constexpr int b_bytes = kF8PAtoms * 96 * 128;   // <= 96 token rows
  static constexpr int a_off = 0;
  static constexpr int b_off = a_off + kF8PStages * a_bytes;
  static constexpr int stg_off = b_off + kF8PStages * b_bytes;
  static constexpr int stg_bytes = 4 * 32 * 17 * 4;   // SwiGLU exchange
  // two item scale slots: the item's token rows of the UE8M0 table
  // [192][pitch], then its weight row blocks (2 x pitch)
  static constexpr int is_off = stg_off + stg_bytes;
  static constexpr int is_w = kF8PBN * kF8PMaxPitch;
  static constexpr int is_bytes = is_w + 2 * kF8PMaxPitch;
  static constexpr int bar_off = is_off + 2 * is_bytes;
  static constexpr int n_bars = 2 * kF8PStages + 4 + 5 + 2 * kSchedDepth +
                                2 * kF8PSfGroups;
  static constexpr int misc_off = bar_off + n_bars * 8;
  static constexpr int epok_off = misc_off + 16;
  static constexpr int sched_off = epok_off + 16;
  static constexpr int tab_off = sched_off + 4 * kSchedDepth;
  // fused requantization of H: per chunk parity, 4 warps x 16 token maxima,
  // this CTA's own and the peer CTA's; and two barriers the peer arrives on
  static constexpr int amx_off =
      (tab_off + 2 * (kMaxGroups + 1) * 4 + 15) / 16 * 16;   // float4 rows
  static constexpr int amx_bytes = 2 * 2 * 4 * 16 * 4;
  static constexpr int amxbar_off = amx_off + amx_bytes;
  static constexpr int total = amxbar_off + 16;
  static constexpr int alloc = total + 1024;
  static constexpr int tmem_cols = 512;
  static_assert(alloc <= 227 * 1024, "shared memory");
  static_assert(kF8PBN <= 192 && f8p_sf_col(3) + 24 <= 512, "TMEM map");
};

// The pair's two CTAs hold the 128 H columns of one 1 x 128 quantization
// block (64 each).  Hand-off of the per-token block maxima between them:
// each CTA's four epilogue warps write their 16 token maxima into their own
// `amx` slot of the chunk's parity and, by st.async, into the peer's; the
// st.async completes its bytes on the peer's barrier of that parity, where
// the peer's warp 0 expects 4 x 64 bytes per chunk.  No release fence is
// taken (one would wait for the epilogue's earlier global stores).  The
// slot of parity c is written again only after this CTA has received the
// peer's maxima of chunk c + 1, which the peer sends after its reads of
// chunk c.
struct F8Amx {
  float* own;            // [2][4][16]
  float* rem;            // [2][4][16], written by the peer
  uint32_t rem_peer;     // cluster address of the peer's `rem`
  uint32_t bar;          // this CTA's barriers [2]
  uint32_t bar_peer;     // cluster address of the peer's barriers
  int par;               // parity of the next chunk
  uint32_t ph;           // bit c: phase of barrier c
};

// 16 bytes into the peer CTA's shared memory, counted as transaction bytes
// on the peer's barrier `cluster_bar`.
__device__ __forceinline__ void st_async_v4f(uint32_t cluster_addr, float a,
                                             float b, float c, float d,
                                             uint32_t cluster_bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], "
      "{%1, %2, %3, %4}, [%5];" ::"r"(cluster_addr),
      "f"(a), "f"(b), "f"(c), "f"(d), "r"(cluster_bar)
      : "memory");
}

// Gate/up epilogue of the e4m3 CTA-pair GEMM with H requantized in place:
// SwiGLU as in epilogue_store (warps q and q+2 swap token halves so each
// thread holds H of one column, 16 tokens), then per token the largest |H|
// of the 128-column block (warp maximum, the partner warp's, the peer
// CTA's), the block exponent e and the e4m3 codes of H 2^-e; the rank-0
// CTA also writes the block's fp32 scale and UE8M0 byte.  H is the same
// fp32 value the separate quantizer would read, so the codes and scales are
// the same bit for bit.
__device__ __forceinline__ bool f8p_epilogue_swiglu_q8(
    uint32_t taddr, int n_valid, int b_row, int col0, long long ld,
    long long rows, uint8_t* q8, float* qs, uint8_t* qe, int qpitch,
    bool write_scales, float* xchg, F8Amx& am, int q, int lane,
    volatile int* abort_flag) {
  const bool gate_warp = q < 2;
  const int pair_q = q & 1;
  const int jbase = gate_warp ? 0 : 16;
  const int blk = col0 >> 7;                       // quantization block
  bool ok = true;
  for (int n0 = 0; n0 < n_valid; n0 += 32) {
    uint32_t r[32];
    tmem_ld32(taddr + n0, r);
    tmem_ld_wait();
    const int nleft = n_valid - n0;
    float* mine = xchg + ((q * 32) + lane) * 17;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      mine[j] = __uint_as_float(r[gate_warp ? 16 + j : j]);
    named_bar_sync(1, 128);
    const float* theirs =
        xchg + (((gate_warp ? q + 2 : q - 2) * 32) + lane) * 17;
    float h[16], mx[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float g = gate_warp ? __uint_as_float(r[j]) : theirs[j];
      const float u = gate_warp ? theirs[j] : __uint_as_float(r[16 + j]);
      // SiLU with the fast exponential and division intrinsics: H is
      // about to be rounded to 3 mantissa bits, so their few-ulp error
      // decides a code only at a rounding boundary (one e4m3 step)
      h[j] = jbase + j < nleft ? __fdividef(g, 1.0f + __expf(-g)) * u : 0.f;
      mx[j] = warp_amax(h[j]);
    }
    const int sl = am.par;
    if (lane == 0) {
      float* o = am.own + (sl * 4 + q) * 16;
      const uint32_t rp = am.rem_peer + ((sl * 4 + q) * 16) * 4;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        reinterpret_cast<float4*>(o)[v] =
            make_float4(mx[4 * v], mx[4 * v + 1], mx[4 * v + 2], mx[4 * v + 3]);
        st_async_v4f(rp + 16 * v, mx[4 * v], mx[4 * v + 1], mx[4 * v + 2],
                     mx[4 * v + 3], am.bar_peer + 8 * sl);
      }
      // this CTA's barrier: the peer's four warps' 64 bytes each
      if (q == 0) mbar_arrive_expect_tx(am.bar + 8 * sl, 4 * 64);
    }
    named_bar_sync(1, 128);          // the partner warp's maxima are in own
    if (!mbar_wait_cl(am.bar + 8 * sl, (am.ph >> sl) & 1u, abort_flag,
                      KID_GEMM_FP8, 120))
      ok = false;
    am.ph ^= 1u << sl;
    am.par ^= 1;
    const int qp = q ^ 1;
    const float* o1 = am.own + (sl * 4 + q) * 16;
    const float* o2 = am.own + (sl * 4 + qp) * 16;
    const float* r1 = am.rem + (sl * 4 + q) * 16;
    const float* r2 = am.rem + (sl * 4 + qp) * 16;
    // the warp's 16 tokens x 32 columns of codes, transposed through its own
    // (now free) 2 KB of the exchange buffer: lane pairs then store one
    // token's 32 codes as two 16-byte vectors
    uint8_t* tile = reinterpret_cast<uint8_t*>(xchg + q * 32 * 17);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float a = fmaxf(fmaxf(o1[j], o2[j]), fmaxf(r1[j], r2[j]));
      const int e = e4m3_scale_exp(a);
      const bool bad_e = e < -126 || e > 126;
      tile[j * 32 + lane] = bad_e ? 0 : static_cast<uint8_t>(
                                            e4m3_code(h[j], pow2f(-e)));
      if (jbase + j < nleft && write_scales && pair_q == 0 && lane == 0) {
        const long long row = b_row + n0 + jbase + j;
        const float sc = bad_e ? 0.f : pow2f(e);
        if (bad_e) report_error(ERR_CHECK, KID_QUANT, 1);
        qs[static_cast<long long>(blk) * rows + row] = sc;
        qe[row * qpitch + blk] = ue8_of(sc);
      }
    }
    __syncwarp();
    {
      const int j = lane >> 1, part = lane & 1;
      if (jbase + j < nleft) {
        const long long row = b_row + n0 + jbase + j;
        *reinterpret_cast<uint4*>(q8 + row * ld + col0 + pair_q * 32 +
                                  part * 16) =
            *reinterpret_cast<const uint4*>(tile + j * 32 + part * 16);
      }
    }
    named_bar_sync(1, 128);
  }
  return ok;
}

// Rows of the TMA box of a CTA's token half-tile: the smallest of 32, 64,
// 96 covering it (96 = 192 / 2).
__host__ __device__ __forceinline__ int f8p_token_box(int half) {
  return half <= 32 ? 32 : (half <= 64 ? 64 : 96);
}

// Item -> (pair weight tile, token chunk); chunk index fastest.
__device__ __forceinline__ Tile decode_f8p_item(int item,
                                                const F8PairParams& p,
                                                int n_items_s, int nch_s,
                                                const int* off_s,
                                                const int* chunk_pre) {
  Tile t;
  if (item < n_items_s) {
    const int wt = item / nch_s, ch = item % nch_s;
    t.shared = 1;
    t.wt = wt;
    t.a_row = wt * kF8PBM;
    t.b_row = ch * kF8PBN;
    t.n_valid = min(kF8PBN, p.shared_rows - t.b_row);
    t.k = p.k_shared;
  } else {
    const int wt_r = p.w_rows_routed / kF8PBM;
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
    const int m = off_s[e + 1] - off_s[e];
    const int sz = (((m + ce - 1) / ce) + 15) & ~15;   // equal chunks
    t.shared = 0;
    t.wt = wt;
    t.a_row = e * p.w_rows_routed + wt * kF8PBM;
    t.b_row = off_s[e] + ch * sz;
    t.n_valid = min(sz, off_s[e + 1] - t.b_row);
    t.k = p.k_routed;
  }
  t.n_mma = (t.n_valid + 15) & ~15;
  return t;
}

// UE8M0 byte of a power-of-two fp32 scale: its biased exponent.
__device__ __forceinline__ uint32_t ue8m0(float s) {
  return (__float_as_uint(s) >> 23) & 0xFFu;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kF8PThreads, 1)
grouped_gemm_fp8_pair_kernel(const __grid_constant__ CUtensorMap tmA_r,
                             const __grid_constant__ CUtensorMap tmA_s,
                             const __grid_constant__ CUtensorMap tmB_r32,
                             const __grid_constant__ CUtensorMap tmB_s32,
                             const __grid_constant__ CUtensorMap tmB_r64,
                             const __grid_constant__ CUtensorMap tmB_s64,
                             const __grid_constant__ CUtensorMap tmB_r96,
                             const __grid_constant__ CUtensorMap tmB_s96,
                             const F8PairParams p) {
  using L = F8PairSmem;
  constexpr int ST = kF8PStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + L::bar_off;
  const uint32_t bar_empty = bar_full + 8 * ST;
  const uint32_t bar_tfull = bar_empty + 8 * ST;     // [2]
  const uint32_t bar_tempty = bar_tfull + 16;        // [2]
  const uint32_t bar_final = bar_tempty + 16;
  const uint32_t bar_sfull = bar_final + 8;          // [kSchedDepth]
  const uint32_t bar_sempty = bar_sfull + 8 * kSchedDepth;
  const uint32_t bar_sffull = bar_sempty + 8 * kSchedDepth;  // [groups]
  const uint32_t bar_sfempty = bar_sffull + 8 * kF8PSfGroups; // [groups]
  const uint32_t bar_isfull = bar_sfempty + 8 * kF8PSfGroups;  // [2]
  const uint32_t bar_isempty = bar_isfull + 16;                 // [2]
  volatile uint32_t* tmem_slot =
      reinterpret_cast<volatile uint32_t*>(smem + L::misc_off);
  volatile int* abort_flag =
      reinterpret_cast<volatile int*>(smem + L::misc_off + 4);
  volatile int* bad_flag =
      reinterpret_cast<volatile int*>(smem + L::misc_off + 8);
  volatile int* ep_ok = reinterpret_cast<volatile int*>(smem + L::epok_off);
  volatile int* sched = reinterpret_cast<volatile int*>(smem + L::sched_off);
  int* off_s = reinterpret_cast<int*>(smem + L::tab_off);
  int* chunk_pre = off_s + (kMaxGroups + 1);
  float* stg = reinterpret_cast<float*>(smem + L::stg_off);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank() & 1u;
  const bool leader = rank == 0;
  const uint32_t lead = cluster_ctarank() & ~1u;
  const uint32_t peer = lead + 1;
  const int G = p.n_groups;

  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(bar_isfull + 8 * j, 1);       // producer's expect-tx
      mbar_init(bar_isempty + 8 * j, 4);      // the 4 scale warps
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_tfull + 8 * a, 1);
      mbar_init(bar_tempty + 8 * a, 8);       // 4 epilogue warps x 2 CTAs
    }
    for (int g = 0; g < kF8PSfGroups; ++g) {
      mbar_init(bar_sffull + 8 * g, 8);       // 4 scale warps x 2 CTAs
      mbar_init(bar_sfempty + 8 * g, 1);
    }
    mbar_init(bar_final, 1);
    for (int i = 0; i < kSchedDepth; ++i) {
      mbar_init(bar_sfull + 8 * i, 1);
      mbar_init(bar_sempty + 8 * i, 18);      // 9 consumers x 2 CTAs
    }
    for (int j = 0; j < 2; ++j)   // own expect-tx; the peer's st.async bytes
      mbar_init(sbase + L::amxbar_off + 8 * j, 1);
    *abort_flag = 0;
    *bad_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA_r);
    tma_prefetch_desc(&tmA_s);
  }
  if (warp == 1) {
    tmem_alloc_pair(sbase + L::misc_off, L::tmem_cols);
    tmem_relinquish_pair();
  }
  if (G > 0)
    for (int e = threadIdx.x; e <= G; e += blockDim.x) off_s[e] = p.offsets[e];
  __syncthreads();
  for (int e = threadIdx.x; e < G; e += blockDim.x) {
    const int m = off_s[e + 1] - off_s[e];
    if (m < 0 || off_s[e] < 0) *bad_flag = 1;
    chunk_pre[e + 1] = m > 0 ? (m + kF8PBN - 1) / kF8PBN : 0;
  }
  if (threadIdx.x == 0) {
    chunk_pre[0] = 0;
    if (G > 0 && static_cast<long long>(off_s[G]) > p.max_routed_rows)
      *bad_flag = 1;
  }
  __syncthreads();
  if (warp == 0) {
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
  cluster_sync();          // both CTAs' barriers exist before any remote use
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool bad = *bad_flag != 0;
  if (bad && threadIdx.x == 0) report_error(ERR_CHECK, KID_GEMM_FP8, 100);

  const int nch_s =
      p.shared_rows > 0 ? (p.shared_rows + kF8PBN - 1) / kF8PBN : 0;
  const int n_items_s = nch_s * (p.w_rows_shared / kF8PBM);
  const int n_items = bad ? 0
                          : n_items_s + (G > 0 ? chunk_pre[G] *
                                                     (p.w_rows_routed / kF8PBM)
                                               : 0);
  const uint32_t full_L = mapa_shared(bar_full, lead);
  const uint32_t tempty_L = mapa_shared(bar_tempty, lead);
  const uint32_t sempty_L = mapa_shared(bar_sempty, lead);
  const uint32_t sffull_L = mapa_shared(bar_sffull, lead);

  // Schedule ring consumer (every role but the even CTA's producer): the
  // next claimed item, or n_items when the ring gives out.
  int slot = 0;
  uint32_t sph = 0;
  auto next_item = [&](unsigned where) -> int {
    const bool got = mbar_wait_cl(bar_sfull + 8 * slot, sph, abort_flag,
                                  KID_GEMM_FP8, where);
    const int item = got ? sched[slot] : n_items;
    __syncwarp();
    if (got && lane == 0) mbar_arrive_cluster(sempty_L + 8 * slot);
    if (++slot == kSchedDepth) {
      slot = 0;
      sph ^= 1;
    }
    return got ? item : -1;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ----------- producer (both CTAs); scheduler in the even CTA ---------
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      int nitem = 0;       // items started (item scale slot = nitem % 2)
      int item = (leader && !bad) ? atomicAdd(p.item_counter, 1) : n_items;
      while (!*abort_flag) {
        if (leader) {
          if (!mbar_wait_cl(bar_sempty + 8 * slot, sph ^ 1, abort_flag,
                            KID_GEMM_FP8, 101))
            break;
          sched[slot] = item;
          st_cluster_u32(mapa_shared(sbase + L::sched_off + 4 * slot, peer),
                         static_cast<uint32_t>(item));
          mbar_arrive(bar_sfull + 8 * slot);
          mbar_arrive_cluster(mapa_shared(bar_sfull + 8 * slot, peer));
        } else {
          if (!mbar_wait_cl(bar_sfull + 8 * slot, sph, abort_flag,
                            KID_GEMM_FP8, 102))
            break;
          item = sched[slot];
          mbar_arrive_cluster(sempty_L + 8 * slot);
        }
        if (++slot == kSchedDepth) {
          slot = 0;
          sph ^= 1;
        }
        if (item >= n_items) break;
        int next = n_items;
        if (leader) next = atomicAdd(p.item_counter, 1);
        const Tile t = decode_f8p_item(item, p, n_items_s, nch_s, off_s,
                                       chunk_pre);
        // the item's scales: token rows and weight row blocks of the UE8M0
        // tables, into this CTA's item slot
        {
          const int j = nitem & 1;
          if (!mbar_wait(bar_isempty + 8 * j, ((nitem >> 1) & 1) ^ 1,
                         abort_flag, KID_GEMM_FP8, 113))
            break;
          const int pitch = t.shared ? p.pitch_shared : p.pitch_routed;
          const uint8_t* sx = t.shared ? p.sx_shared : p.sx_routed;
          const uint8_t* sw = t.shared ? p.sw_shared : p.sw_routed;
          const int rb = p.gate_up ? (t.a_row >> 7)
                                   : (t.a_row >> 7) + static_cast<int>(rank);
          const uint32_t tb = static_cast<uint32_t>(t.n_valid * pitch);
          const uint32_t wb = static_cast<uint32_t>((p.gate_up ? 2 : 1) * pitch);
          const uint32_t slot_s = sbase + L::is_off + j * L::is_bytes;
          mbar_arrive_expect_tx(bar_isfull + 8 * j, tb + wb);
          bulk_load(slot_s, sx + static_cast<size_t>(t.b_row) * pitch, tb,
                    bar_isfull + 8 * j);
          bulk_load(slot_s + L::is_w, sw + static_cast<size_t>(rb) * pitch, wb,
                    bar_isfull + 8 * j);
          ++nitem;
        }
        const CUtensorMap* mA = t.shared ? &tmA_s : &tmA_r;
        const int half = t.n_mma >> 1;
        const int box = f8p_token_box(half);
        const CUtensorMap* mB =
            box == 32   ? (t.shared ? &tmB_s32 : &tmB_r32)
            : box == 64 ? (t.shared ? &tmB_s64 : &tmB_r64)
                        : (t.shared ? &tmB_s96 : &tmB_r96);
        const int b_row = t.b_row + static_cast<int>(rank) * half;
        const uint32_t pair_bytes = 2u * static_cast<uint32_t>(
                                        L::a_bytes + kF8PAtoms * box * 128);
        const int nk = (t.k / 128 + kF8PAtoms - 1) / kF8PAtoms;   // stages
        bool ok = true;
        for (int i = 0; i < nk; ++i) {
          if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1, abort_flag,
                         KID_GEMM_FP8, 103)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(bar_full + 8 * stage, pair_bytes);
          const uint32_t fb = full_L + 8 * stage;
          const uint32_t adst = sbase + L::a_off + stage * L::a_bytes;
          if (p.gate_up) {
            // one 5-D box: per K-atom, the CTA's 64 gate rows (block
            // a_row / 128, half `rank`) then the 64 up rows of the same
            // intermediates (the next block, same half)
            tma_load_5d_pair(adst, mA, 0, 0, static_cast<int>(rank),
                             t.a_row >> 7, kF8PAtoms * i, fb);
          } else {
            tma_load_3d_pair(adst, mA, t.a_row + static_cast<int>(rank) * 128,
                             kF8PAtoms * i, fb);
          }
          tma_load_3d_pair(sbase + L::b_off + stage * L::b_bytes, mB, b_row,
                           kF8PAtoms * i, fb);
          ++issued;
          if (++stage == ST) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        item = next;
      }
      if (*abort_flag) {   // let the loads in flight land
        for (int j = 0; j < 2 && j < nitem; ++j) {
          const int n = nitem - 1 - j;
          mbar_drain(bar_isfull + 8 * (n & 1), (n >> 1) & 1);
        }
        if (leader)
          for (int j = 0; j < ST && j < issued; ++j) {
            int st = stage - 1 - j;
            uint32_t ph = phase;
            if (st < 0) {
              st += ST;
              ph ^= 1;
            }
            mbar_drain_cl(bar_full + 8 * st, ph);
          }
      }
    }
  } else if (warp == 1) {
    if (leader && lane == 0) {
      // ---------------- MMA issuer (even CTA) ----------------
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      int sfg = 0;
      uint32_t sf_phase = 0;
      while (!*abort_flag) {
        if (!mbar_wait_cl(bar_sfull + 8 * slot, sph, abort_flag, KID_GEMM_FP8,
                          104))
          break;
        const int item = sched[slot];
        mbar_arrive(bar_sempty + 8 * slot);
        if (++slot == kSchedDepth) {
          slot = 0;
          sph ^= 1;
        }
        if (item >= n_items) break;
        const Tile t = decode_f8p_item(item, p, n_items_s, nch_s, off_s,
                                       chunk_pre);
        if (!mbar_wait_cl(bar_tempty + 8 * acc, acc_phase ^ 1, abort_flag,
                          KID_GEMM_FP8, 105))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + f8p_acc_col(acc);
        const int nkb = t.k / 128;                              // blocks
        const int nk = (nkb + kF8PAtoms - 1) / kF8PAtoms;       // stages
        const uint32_t b_atom = static_cast<uint32_t>(
            f8p_token_box(t.n_mma >> 1) * 128);
        bool ok = true;
        for (int i = 0; i < nk; ++i) {
          if (((kF8PAtoms * i) & 3) == 0) {
            if (!mbar_wait_cl(bar_sffull + 8 * sfg, sf_phase, abort_flag,
                              KID_GEMM_FP8, 106)) {
              ok = false;
              break;
            }
          }
          if (!mbar_wait(bar_full + 8 * stage, phase, abort_flag, KID_GEMM_FP8,
                         107)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = sbase + L::a_off + stage * L::a_bytes;
          const uint32_t b0 = sbase + L::b_off + stage * L::b_bytes;
          const uint32_t sfa = tmem + f8p_sf_col(sfg);
#pragma unroll
          for (int at = 0; at < kF8PAtoms; ++at) {
            const int kb = kF8PAtoms * i + at;   // 128-block of the reduction
            if (kb < nkb) {
              const uint32_t idesc = idesc_mxf8_pair(t.n_mma, kb & 3);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_mxf8_pair(d_tmem,
                              sdesc_k128(a0 + at * L::a_atom + 32 * kk),
                              sdesc_k128(b0 + at * b_atom + 32 * kk), idesc,
                              sfa, sfa + 16, (kb | kk) != 0);
            }
          }
          mma_commit_pair_mc(bar_empty + 8 * stage, 0x3);
          if (++stage == ST) {
            stage = 0;
            phase ^= 1;
          }
          if (((kF8PAtoms * i + kF8PAtoms - 1) & 3) == 3 ||
              i == nk - 1) {                   // the group's last stage
            mma_commit_pair_mc(bar_sfempty + 8 * sfg, 0x3);
            if (++sfg == kF8PSfGroups) {
              sfg = 0;
              sf_phase ^= 1;
            }
          }
        }
        if (!ok) break;
        mma_commit_pair_mc(bar_tfull + 8 * acc, 0x3);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      mma_commit_pair_mc(bar_final, 0x1);   // every issued MMA complete
      mbar_drain_cl(bar_final, 0);
    }
  } else if (warp < 6) {
    // ---------------- epilogue (warps 2..5 of both CTAs) ----------------
    const int ep = warp - 2;
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    F8Amx amx;
    amx.own = reinterpret_cast<float*>(smem + L::amx_off);
    amx.rem = amx.own + 2 * 4 * 16;
    const uint32_t other = leader ? peer : lead;   // the pair's other CTA
    amx.rem_peer = mapa_shared(smem_u32(amx.rem), other);
    amx.bar = sbase + L::amxbar_off;
    amx.bar_peer = mapa_shared(amx.bar, other);
    amx.par = 0;
    amx.ph = 0;
    while (true) {
      int item = next_item(108);
      const bool got = item >= 0;
      if (!got) item = n_items;
      bool ok = got;
      if (got && item < n_items)
        ok = mbar_wait_cl(bar_tfull + 8 * acc, acc_phase, abort_flag,
                          KID_GEMM_FP8, 109);
      const bool wok = __all_sync(0xffffffffu, ok);
      if (lane == 0) ep_ok[ep] = wok ? 1 : 0;
      named_bar_sync(1, 128);
      if (!(ep_ok[0] && ep_ok[1] && ep_ok[2] && ep_ok[3])) break;
      if (item >= n_items) break;
      const Tile t = decode_f8p_item(item, p, n_items_s, nch_s, off_s,
                                     chunk_pre);
      tc_fence_after();
      void* out = t.shared ? p.out_shared : p.out_routed;
      const long long ld = t.shared ? p.ld_shared : p.ld_routed;
      const int tile128 = t.wt * 2 + static_cast<int>(rank);
      const uint32_t ta = tmem + (static_cast<uint32_t>(q * 32) << 16) +
                          f8p_acc_col(acc);
      bool eok = true;
      if (p.gate_up && p.q8_routed != nullptr) {
        eok = f8p_epilogue_swiglu_q8(
            ta, t.n_valid, t.b_row, tile128 * 64, ld,
            t.shared ? p.shared_rows : p.max_routed_rows,
            t.shared ? p.q8_shared : p.q8_routed,
            t.shared ? p.qs_shared : p.qs_routed,
            t.shared ? p.qe_shared : p.qe_routed,
            t.shared ? p.qpitch_shared : p.qpitch_routed, leader, stg, amx,
            q, lane, abort_flag);
      } else {
        epilogue_store(ta, t.n_valid, t.b_row, out, ld,
                       p.gate_up ? tile128 * 64 : tile128 * 128,
                       p.gate_up != 0, stg, q, ep, lane, true, true);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(tempty_L + 8 * acc);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
      if (!__all_sync(0xffffffffu, eok)) *abort_flag = 1;
    }
  } else {
    // ------------- scale warps (warps 6..9 of both CTAs) -------------------
    // Warp 6 + q writes TMEM lane quarter q: the A scale of its 32 weight
    // rows (column q of the group's A columns) and the B scales of all the
    // item's tokens (6 columns, the same in every quarter), from the item's
    // scale slot.
    const int q = warp & 3;
    const uint32_t lanebase = static_cast<uint32_t>(q * 32) << 16;
    const int R = q * 32 + lane;
    int nitem = 0;
    int sfg = 0;
    uint32_t sf_phase = 0;
    bool run = true;
    while (run) {
      const int item = next_item(110);
      if (item < 0 || item >= n_items) break;
      const Tile t = decode_f8p_item(item, p, n_items_s, nch_s, off_s,
                                     chunk_pre);
      const int nk = t.k / 128;
      const int pitch = t.shared ? p.pitch_shared : p.pitch_routed;
      const int j = nitem & 1;
      bool ok = mbar_wait(bar_isfull + 8 * j, (nitem >> 1) & 1, abort_flag,
                          KID_GEMM_FP8, 111);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const uint8_t* slot_p = smem + L::is_off + j * L::is_bytes;
      // the weight scale row of this lane's A row: 0 (gate, or the CTA's
      // down block) or 1 (up)
      const uint8_t* wrow =
          slot_p + L::is_w + ((p.gate_up && R >= 64) ? pitch : 0);
      for (int g = 0; g * 4 < nk; ++g) {
        // a row's four scale bytes of the group in one word (the table's
        // padding bytes hold 2^0 past the last block)
        const uint32_t wa = *reinterpret_cast<const uint32_t*>(wrow + 4 * g);
        uint32_t wb[8];   // columns 6, 7 unused (N <= 192)
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int n = 32 * c + lane;
          wb[c] = (c < 6 && n < t.n_valid)
                      ? *reinterpret_cast<const uint32_t*>(
                            slot_p + static_cast<size_t>(n) * pitch + 4 * g)
                      : 0x7F7F7F7Fu;
        }
        ok = mbar_wait_cl(bar_sfempty + 8 * sfg, sf_phase ^ 1, abort_flag,
                          KID_GEMM_FP8, 112);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          run = false;
          break;
        }
        const uint32_t col = tmem + f8p_sf_col(sfg);
        tc_fence_after();
        tmem_st1(col + lanebase + q, wa);
        tmem_st8(col + lanebase + 16, wb);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(sffull_L + 8 * sfg);
        if (++sfg == kF8PSfGroups) {
          sfg = 0;
          sf_phase ^= 1;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_isempty + 8 * j);
      ++nitem;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();          // no remote access to either CTA after this
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, L::tmem_cols);
  }
}

}  // namespace moe
