// Grouped expert GEMMs in e4m3 with block scales and promotion of the
// partial sums to fp32 every 128 elements of the reduction, on the CUDA
// cores: the kernels for shapes whose d is not a multiple of 256 (the
// others run on the block-scaled CTA-pair kernel, gemm_fp8_pair.cuh).
// (DeepSeek-V3 report commentary, cooktownmusic.com, FP8 training-framework
// part: FP8 GEMM inputs, fine-grained block scaling (Fig. 7a), partial
// results promoted to FP32 on the CUDA cores at N_C = 128 (Fig. 7b);
// "【推理llm論文精讀】DeepSeek V3技術論文", section 2.2: the expert FFNs of the
// FFN-output equation.)
//
// Same orientation and work items as the bf16 grouped GEMM (weights on the
// MMA's M side, tokens on N; items = (group, weight tile, token chunk), chunk
// fastest, claimed dynamically; the shared experts are one extra group
// scheduled first).  What differs:
//
//   * operands are e4m3 codes; one pipeline stage = one 128-wide block of
//     the reduction (128-byte swizzled rows, 4 MMAs of K = 32);
//   * each stage's MMAs write a fresh fp32 partial into one of NBUF TMEM
//     buffers; the epilogue warps read it and add it, times the two block
//     scales (weight block x token block, both powers of two), into fp32
//     registers -- the promotion of the pages' Fig. 7b, done by the warps
//     that also finish the item, while the tensor cores run the next block;
//   * an item covers two 128-row weight tiles (TWO) -- two M = 128 MMAs per
//     K-step on the same token operand -- or one;
//   * gate/up (SWIGLU, TWO): a weight tile is 128 gate rows followed by the 128 up
//     rows of the same intermediate indices, two M = 128 MMAs per K-step on
//     the same token operand, so a thread holds gate and up of one
//     intermediate index: H = SiLU(g) * u needs no exchange.  H is then
//     quantized in 1 x 128 blocks along the intermediate index (one block =
//     the tile's 128 rows, reduced over the four lane-quarter warps) and
//     stored as codes plus scales [I/128][rows] for the down pass;
//   * down (!SWIGLU): 128 or 256 output channels of Y, stored as fp16 (a
//     value beyond the fp16 range is reported, never written as inf).
//
// Warp roles (64 + 128 CW threads, one CTA per SM, persistent):
//   warp 0 lane 0: scheduler + TMA producer;  warp 1 lane 0: MMA issuer and
//   TMEM owner;  warps 2..: epilogue, warp w reads TMEM lane quarter w % 4
//   and token columns [(w-2)/4 * BN/CW, +BN/CW).
#pragma once
#include "common.cuh"
#include "gemm.cuh"
#include "quant.cuh"

namespace moe {

struct Fp8Params {
  const int* offsets;          // routed group row offsets [n_groups+1]
  int n_groups;
  long long max_routed_rows;   // rows of the routed token operand
  int shared_rows;             // tokens of the shared group (0: none)
  int w_rows_routed;           // packed weight rows per routed group
  int w_rows_shared;           // packed weight rows of the shared group
  int k_routed, k_shared;      // reduction lengths (multiples of 128)
  const float* sw_routed;      // weight block scales [row blocks][K/128]
  const float* sw_shared;
  const float* sx_routed;      // token block scales [K/128][ld]
  long long ldsx_routed;
  const float* sx_shared;
  long long ldsx_shared;
  void* out_routed;            // SwiGLU pass: H codes [rows][ld]; else Y fp16
  long long ld_routed;
  float* sh_routed;            // SwiGLU pass: H scales [I/128][ld]
  long long ldsh_routed;
  void* out_shared;
  long long ld_shared;
  float* sh_shared;
  long long ldsh_shared;
  int* item_counter;
};

template <int BN, int CW, bool TWO, int STAGES>
struct Fp8Smem {
  static constexpr int TR = TWO ? 256 : 128;            // weight rows / item
  static constexpr int a_bytes = TR * kQBlock;
  static constexpr int b_bytes = BN * kQBlock;
  static constexpr int a_off = 0;
  static constexpr int b_off = a_off + STAGES * a_bytes;
  static constexpr int amax_off = b_off + STAGES * b_bytes;   // [CW][4][BN/CW]
  static constexpr int PC = (TWO ? 2 : 1) * BN;          // TMEM cols / partial
  static constexpr int NBUF = (512 / PC) < 8 ? (512 / PC) : 8;
  static constexpr int bar_off = amax_off + 4 * BN * 4;
  static constexpr int n_bars = 2 * STAGES + 2 * NBUF + 1 + 2 * kSchedDepth;
  static constexpr int misc_off = bar_off + n_bars * 8;
  static constexpr int epok_off = misc_off + 16;
  static constexpr int sched_off = epok_off + 4 * 4 * CW;
  static constexpr int tab_off = sched_off + 4 * kSchedDepth;
  static constexpr int total = tab_off + 2 * (kMaxGroups + 1) * 4;
  static constexpr int alloc = total + 1024;
  static constexpr int cols_needed = NBUF * PC;
  static constexpr int tmem_cols = cols_needed <= 32 ? 32
                                   : cols_needed <= 64 ? 64
                                   : cols_needed <= 128 ? 128
                                   : cols_needed <= 256 ? 256 : 512;
  static constexpr int threads = 64 + 128 * CW;
  static_assert(alloc <= 227 * 1024, "shared memory");
  static_assert(BN % (32 * CW) == 0, "columns per epilogue warp");
  static_assert(NBUF >= 2, "at least two partial buffers");
};

template <int BN, int TR>
__device__ __forceinline__ Tile decode_item8(int item, const Fp8Params& p,
                                             int n_items_s, int nch_s,
                                             const int* off_s,
                                             const int* chunk_pre) {
  Tile t;
  if (item < n_items_s) {
    const int wt = item / nch_s, ch = item % nch_s;
    t.shared = 1;
    t.wt = wt;
    t.a_row = wt * TR;
    t.b_row = ch * BN;
    t.n_valid = min(BN, p.shared_rows - t.b_row);
    t.k = p.k_shared;
  } else {
    const int wt_r = p.w_rows_routed / TR;
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
    t.wt = wt;
    t.a_row = e * p.w_rows_routed + wt * TR;
    t.b_row = off_s[e] + ch * BN;
    t.n_valid = min(BN, off_s[e + 1] - t.b_row);
    t.k = p.k_routed;
  }
  t.n_mma = (t.n_valid + 15) & ~15;
  return t;
}

template <int BN, int CW, bool TWO, bool SWIGLU, int STAGES>
__global__ void __launch_bounds__(64 + 128 * CW, 1)
grouped_gemm_fp8_kernel(const __grid_constant__ CUtensorMap tmA_r,
                        const __grid_constant__ CUtensorMap tmB_r,
                        const __grid_constant__ CUtensorMap tmA_s,
                        const __grid_constant__ CUtensorMap tmB_s,
                        const Fp8Params p) {
  using L = Fp8Smem<BN, CW, TWO, STAGES>;
  static_assert(TWO || !SWIGLU, "SwiGLU needs gate and up tiles");
  constexpr bool DUAL = TWO;          // two 128-row tiles per item
  constexpr int TR = L::TR;
  constexpr int PC = L::PC;
  constexpr int NBUF = L::NBUF;
  constexpr int NW = 4 * CW;          // epilogue warps
  constexpr int NC = BN / CW;         // token columns per epilogue thread
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + L::bar_off;
  const uint32_t bar_empty = bar_full + 8 * STAGES;
  const uint32_t bar_pfull = bar_empty + 8 * STAGES;     // [NBUF]
  const uint32_t bar_pempty = bar_pfull + 8 * NBUF;      // [NBUF]
  const uint32_t bar_final = bar_pempty + 8 * NBUF;
  const uint32_t bar_sfull = bar_final + 8;              // [kSchedDepth]
  const uint32_t bar_sempty = bar_sfull + 8 * kSchedDepth;
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
  float* amax_s = reinterpret_cast<float*>(smem + L::amax_off);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.n_groups;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(bar_pfull + 8 * b, 1);
      mbar_init(bar_pempty + 8 * b, NW);
    }
    mbar_init(bar_final, 1);
    for (int i = 0; i < kSchedDepth; ++i) {
      mbar_init(bar_sfull + 8 * i, 1);
      mbar_init(bar_sempty + 8 * i, 1 + NW);   // MMA + epilogue warps
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
  if (G > 0)
    for (int e = threadIdx.x; e <= G; e += blockDim.x) off_s[e] = p.offsets[e];
  __syncthreads();
  for (int e = threadIdx.x; e < G; e += blockDim.x) {
    const int m = off_s[e + 1] - off_s[e];
    if (m < 0 || off_s[e] < 0) *bad_flag = 1;
    chunk_pre[e + 1] = m > 0 ? (m + BN - 1) / BN : 0;
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
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool bad = *bad_flag != 0;
  if (bad && threadIdx.x == 0) report_error(ERR_CHECK, KID_GEMM_FP8, 0);

  const int nch_s = p.shared_rows > 0 ? (p.shared_rows + BN - 1) / BN : 0;
  const int n_items_s = nch_s * (p.w_rows_shared / TR);
  const int n_items =
      bad ? 0
          : n_items_s + (G > 0 ? chunk_pre[G] * (p.w_rows_routed / TR) : 0);

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
                       KID_GEMM_FP8, 1))
          break;
        sched[slot] = item;
        mbar_arrive(bar_sfull + 8 * slot);
        if (++slot == kSchedDepth) {
          slot = 0;
          sph ^= 1;
        }
        if (item >= n_items) break;
        const int next = atomicAdd(p.item_counter, 1);
        const Tile t = decode_item8<BN, TR>(item, p, n_items_s, nch_s, off_s,
                                            chunk_pre);
        const CUtensorMap* mA = t.shared ? &tmA_s : &tmA_r;
        const CUtensorMap* mB = t.shared ? &tmB_s : &tmB_r;
        const int nk = t.k / kQBlock;
        bool ok = true;
        for (int i = 0; i < nk; ++i) {
          if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1, abort_flag,
                         KID_GEMM_FP8, 2)) {
            ok = false;
            break;
          }
          const uint32_t fb = bar_full + 8 * stage;
          mbar_arrive_expect_tx(fb, L::a_bytes + L::b_bytes);
          tma_load_2d(sbase + L::a_off + stage * L::a_bytes, mA, i * kQBlock,
                      t.a_row, fb);
          tma_load_2d(sbase + L::b_off + stage * L::b_bytes, mB, i * kQBlock,
                      t.b_row, fb);
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        item = next;
      }
      if (*abort_flag) {   // let loads in flight land before smem is freed
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
      int buf = 0;
      uint32_t bph = 0;
      int slot = 0;
      uint32_t sph = 0;
      while (!*abort_flag) {
        if (!mbar_wait(bar_sfull + 8 * slot, sph, abort_flag, KID_GEMM_FP8, 3))
          break;
        const int item = sched[slot];
        mbar_arrive(bar_sempty + 8 * slot);
        if (++slot == kSchedDepth) {
          slot = 0;
          sph ^= 1;
        }
        if (item >= n_items) break;
        const Tile t = decode_item8<BN, TR>(item, p, n_items_s, nch_s, off_s,
                                            chunk_pre);
        const uint32_t idesc = idesc_e4m3_f32(128, t.n_mma);
        const int nk = t.k / kQBlock;
        bool ok = true;
        for (int i = 0; i < nk; ++i) {
          if (!mbar_wait(bar_pempty + 8 * buf, bph ^ 1, abort_flag,
                         KID_GEMM_FP8, 4) ||
              !mbar_wait(bar_full + 8 * stage, phase, abort_flag, KID_GEMM_FP8,
                         5)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = sbase + L::a_off + stage * L::a_bytes;
          const uint32_t b0 = sbase + L::b_off + stage * L::b_bytes;
          const uint32_t d0 = tmem + buf * PC;
#pragma unroll
          for (int kk = 0; kk < kQBlock / 32; ++kk) {
            mma_e4m3(d0, sdesc_k128(a0 + kk * 32), sdesc_k128(b0 + kk * 32),
                     idesc, kk > 0);
            if constexpr (DUAL)
              mma_e4m3(d0 + BN, sdesc_k128(a0 + 128 * kQBlock + kk * 32),
                       sdesc_k128(b0 + kk * 32), idesc, kk > 0);
          }
          mma_commit(bar_empty + 8 * stage);
          mma_commit(bar_pfull + 8 * buf);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
          if (++buf == NBUF) {
            buf = 0;
            bph ^= 1;
          }
        }
        if (!ok) break;
      }
      mma_commit(bar_final);
      mbar_drain(bar_final, 0);
    }
  } else {
    // ---------------- epilogue: promotion + finish ----------------
    const int ep = warp - 2;
    const int q = warp & 3;            // TMEM lane quarter
    const int cg = ep >> 2;            // column group
    const int col0 = cg * NC;
    int buf = 0;
    uint32_t bph = 0;
    int slot = 0;
    uint32_t sph = 0;
    bool overflow = false;
    while (true) {
      const bool got = mbar_wait(bar_sfull + 8 * slot, sph, abort_flag,
                                 KID_GEMM_FP8, 6);
      const int item = got ? sched[slot] : n_items;
      __syncwarp();
      if (got && lane == 0) mbar_arrive(bar_sempty + 8 * slot);
      if (++slot == kSchedDepth) {
        slot = 0;
        sph ^= 1;
      }
      const bool wok = __all_sync(0xffffffffu, got);
      if (lane == 0) ep_ok[ep] = wok ? 1 : 0;
      named_bar_sync(1, 32 * NW);
      bool all_ok = true;
      for (int w = 0; w < NW; ++w) all_ok = all_ok && ep_ok[w];
      named_bar_sync(1, 32 * NW);      // ep_ok is rewritten next item
      if (!all_ok || item >= n_items) break;
      const Tile t = decode_item8<BN, TR>(item, p, n_items_s, nch_s, off_s,
                                          chunk_pre);
      const float* sw = t.shared ? p.sw_shared : p.sw_routed;
      const float* sx = t.shared ? p.sx_shared : p.sx_routed;
      const long long ldsx = t.shared ? p.ldsx_shared : p.ldsx_routed;
      const int nk = t.k / kQBlock;
      const int rb = t.a_row / 128;    // weight row block (gate; up = rb+1)
      float acc_g[NC], acc_u[DUAL ? NC : 1];
#pragma unroll
      for (int j = 0; j < NC; ++j) {
        acc_g[j] = 0.f;
        if constexpr (DUAL) acc_u[j] = 0.f;
      }
      bool ok = true;
      // Block scales of chunk i: weight (gate, up) and this lane's token
      // column in each 32-column slice.  They are loaded one chunk ahead so
      // that their latency hides behind the wait for the partial sums.
      auto load_scales = [&](int i, float& g, float& u, float* x) {
        g = __ldg(sw + static_cast<size_t>(rb) * nk + i);
        u = DUAL ? __ldg(sw + static_cast<size_t>(rb + 1) * nk + i) : 0.f;
#pragma unroll
        for (int c = 0; c < NC / 32; ++c) {
          const int col = col0 + c * 32 + lane;
          x[c] = col < t.n_valid
                     ? __ldg(sx + static_cast<size_t>(i) * ldsx + t.b_row + col)
                     : 0.f;
        }
      };
      float nswg, nswu, nsx[NC / 32];
      load_scales(0, nswg, nswu, nsx);
      for (int i = 0; i < nk; ++i) {
        const float swg = nswg, swu = nswu;
        float sxc[NC / 32];
#pragma unroll
        for (int c = 0; c < NC / 32; ++c) sxc[c] = nsx[c];
        if (i + 1 < nk) load_scales(i + 1, nswg, nswu, nsx);
        ok = mbar_wait(bar_pfull + 8 * buf, bph, abort_flag, KID_GEMM_FP8, 7) &&
             ok;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < NC / 32; ++c) {
          const int cbase = col0 + c * 32;
          if (cbase < t.n_mma) {
            // token scale of column cbase + lane, broadcast by shuffles
            const float sxl = sxc[c];
            uint32_t r[32];
            const uint32_t ta = tmem + (static_cast<uint32_t>(q * 32) << 16) +
                                buf * PC + cbase;
            if constexpr (DUAL && NC == 32) {
              // one 32-column slice per thread: both partials in flight
              // before the wait (registers allow it at this width)
              uint32_t r2[32];
              tmem_ld32(ta, r);
              tmem_ld32(ta + BN, r2);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const float sj = __shfl_sync(0xffffffffu, sxl, j);
                acc_g[c * 32 + j] =
                    fmaf(__uint_as_float(r[j]), swg * sj, acc_g[c * 32 + j]);
                acc_u[c * 32 + j] =
                    fmaf(__uint_as_float(r2[j]), swu * sj, acc_u[c * 32 + j]);
              }
            } else {
              tmem_ld32(ta, r);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const float sj = __shfl_sync(0xffffffffu, sxl, j);
                acc_g[c * 32 + j] =
                    fmaf(__uint_as_float(r[j]), swg * sj, acc_g[c * 32 + j]);
              }
              if constexpr (DUAL) {
                tmem_ld32(ta + BN, r);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                  const float sj = __shfl_sync(0xffffffffu, sxl, j);
                  acc_u[c * 32 + j] =
                      fmaf(__uint_as_float(r[j]), swu * sj, acc_u[c * 32 + j]);
                }
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_pempty + 8 * buf);
        if (++buf == NBUF) {
          buf = 0;
          bph ^= 1;
        }
      }
      const int row = q * 32 + lane;   // row of the 128-row output block
      if constexpr (SWIGLU) {
        // H = SiLU(g) * u for intermediate index wt*128 + row, then the
        // 1 x 128 block of each token: max over the four lane quarters
        float* am = amax_s + cg * 4 * NC;
#pragma unroll
        for (int j = 0; j < NC; ++j) {
          acc_g[j] = silu_f32(acc_g[j]) * acc_u[j];
          const float m = warp_amax(acc_g[j]);
          if (lane == 0) am[q * NC + j] = m;
        }
        named_bar_sync(2 + cg, 128);
        uint8_t* H = static_cast<uint8_t*>(t.shared ? p.out_shared
                                                     : p.out_routed);
        const long long ldh = t.shared ? p.ld_shared : p.ld_routed;
        float* sh = t.shared ? p.sh_shared : p.sh_routed;
        const long long ldsh = t.shared ? p.ldsh_shared : p.ldsh_routed;
        const int hcol = t.wt * 128 + row;
#pragma unroll
        for (int j = 0; j < NC; ++j) {
          const int col = col0 + j;
          const float a = fmaxf(fmaxf(am[j], am[NC + j]),
                                fmaxf(am[2 * NC + j], am[3 * NC + j]));
          const int e = e4m3_scale_exp(a);
          const bool eok = e >= -126 && e <= 126;
          overflow |= !eok;
          if (col < t.n_valid) {
            H[static_cast<size_t>(t.b_row + col) * ldh + hcol] =
                static_cast<uint8_t>(
                    eok ? e4m3_code(acc_g[j], pow2f(-e)) : 0u);
            if (q == 0 && lane == (j & 31))
              sh[static_cast<size_t>(t.wt) * ldsh + t.b_row + col] =
                  eok ? pow2f(e) : 0.f;
          }
        }
        named_bar_sync(2 + cg, 128);   // am is reused by the next item
      } else {
        __half* Y = static_cast<__half*>(t.shared ? p.out_shared
                                                  : p.out_routed);
        const long long ldy = t.shared ? p.ld_shared : p.ld_routed;
        const int ycol = t.wt * TR + row;     // second tile: + 128
#pragma unroll
        for (int j = 0; j < NC; ++j) {
          const int col = col0 + j;
          if (col < t.n_valid) {
            __half* yr = Y + static_cast<size_t>(t.b_row + col) * ldy + ycol;
            overflow |= !(fabsf(acc_g[j]) <= 65504.f);
            yr[0] = __float2half_rn(acc_g[j]);
            if constexpr (DUAL) {
              overflow |= !(fabsf(acc_u[j]) <= 65504.f);
              yr[128] = __float2half_rn(acc_u[j]);
            }
          }
        }
      }
      (void)ok;
    }
    if (overflow) report_error(ERR_CHECK, KID_GEMM_FP8, 100);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::tmem_cols);
  }
}

}  // namespace moe
