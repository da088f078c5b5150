// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM,
// operands staged by TMA).  ("【推理llm論文精讀】DeepSeek V3技術論文", section
// 2.2: FFN^(r)_i of each selected expert and FFN^(s) of every shared expert
// in the FFN-output equation; SwiGLU form is this library's reading.)
//
// Orientation: the weight rows sit on the MMA's M side (128 TMEM lanes) and
// the tokens on its N side, so a group of M_e tokens pads only to a multiple
// of 16 (tokens per tile = min(BN, remaining) rounded up to 16).
//
//   D[w, n] = sum_k W[a_row + w, k] * X[b_row + n, k]     (w < 128, n < N)
//
// Gate/up pass (swiglu = 1): a 128-row packed weight tile holds 64 gate rows
// then the 64 up rows of the same intermediate columns, so the epilogue
// emits 64 columns of H = SiLU(gate) * up (bf16, the next GEMM's operand).
// Down pass (swiglu = 0): 128 output columns of Y, kept in fp32.
//
// Work items: (group, weight tile, token chunk) with the chunk index
// fastest.  CTAs claim items in index order from a global counter, so the
// items that share a weight tile run side by side and the tile is fetched
// from HBM about once.  (An L2 prefetch of the weight stream ahead of the
// TMA ring measured slower: the extra TMA instructions cost more than the
// latency they hide.)  The shared experts form
// one extra group that spans all T tokens, scheduled first.  Offsets stay on
// the device: each CTA derives the item table from them in its prologue.
//
// Warp roles (192 threads, one CTA per SM, persistent):
//   warp 0 lane 0: scheduler + TMA producer over a STAGES-deep smem ring;
//   warp 1 lane 0: MMA issuer (also allocates / frees TMEM);
//   warps 2..5   : epilogue, double-buffered TMEM accumulators so that the
//                  epilogue of one item overlaps the mainloop of the next.
#pragma once
#include "common.cuh"

namespace moe {

constexpr int kGemmBM = 128;    // weight rows per tile (MMA M)
constexpr int kGemmBK = 64;     // K per pipeline stage (128 B of bf16)
constexpr int kBoxRows = 32;    // token rows per TMA box
constexpr int kMaxGroups = 256;
constexpr int kSchedDepth = 6;      // claimed items queued producer -> consumers

struct GemmParams {
  const int* offsets;   // routed group row offsets [n_groups+1] (device)
  int n_groups;         // routed groups (0: none)
  int w_rows_routed;    // weight rows per routed group
  int k_routed;         // reduction length of the routed pass
  long long max_routed_rows;  // rows of the routed B operand / output
  int shared_rows;      // tokens of the shared group (0: none)
  int w_rows_shared;    // weight rows of the shared group
  int k_shared;         // reduction length of the shared pass
  void* out_routed;     // swiglu: H bf16; else: Y (fp16 for bf16 layers, fp32 for fp32)
  long long ld_routed;
  void* out_shared;
  long long ld_shared;
  int swiglu;
  int y_fp16;           // down pass: store Y as fp16 (else fp32)
  int* item_counter;    // zeroed before the launch; CTAs claim items from it
  // bf16 gate/up pass: when not null, the gate and up pre-activations are
  // also stored (fp16, range checked; packed column order, the row of H)
  // for the backward
  __half* act_routed;
  long long ld_act_routed;
  __half* act_shared;
  long long ld_act_shared;
};

template <int BN, int STAGES>
struct GemmSmem {
  static constexpr int a_bytes = kGemmBM * kGemmBK * 2;
  static constexpr int b_bytes = BN * kGemmBK * 2;
  static constexpr int a_off = 0;
  static constexpr int b_off = a_off + STAGES * a_bytes;
  static constexpr int stg_off = b_off + STAGES * b_bytes;
  static constexpr int stg_bytes = 4 * 32 * 17 * 4;   // epilogue exchange
  static constexpr int bar_off = stg_off + stg_bytes;
  static constexpr int n_bars = 2 * STAGES + 5 + 2 * kSchedDepth;
  static constexpr int misc_off = bar_off + n_bars * 8;
  static constexpr int epok_off = misc_off + 16;
  static constexpr int sched_off = epok_off + 16;
  static constexpr int tab_off = sched_off + 4 * kSchedDepth;
  static constexpr int total = tab_off + 2 * (kMaxGroups + 1) * 4;
  static constexpr int alloc = total + 1024;
  static constexpr int tmem_cols = 2 * BN < 32 ? 32 : 2 * BN;
  static_assert(alloc <= 227 * 1024, "shared memory");
};

struct Tile {
  int a_row;      // first weight row (in its tensor map)
  int b_row;      // first token row (in its tensor map and output)
  int n_valid;    // tokens in this tile
  int n_mma;      // n_valid rounded up to 16
  int k;          // reduction length
  int wt;         // weight tile index inside the group
  int shared;     // 1: shared group
};

template <int BN>
__device__ __forceinline__ Tile decode_item(int item, const GemmParams& p,
                                            int n_items_s, int nch_s,
                                            const int* off_s,
                                            const int* chunk_pre) {
  Tile t;
  if (item < n_items_s) {
    const int wt = item / nch_s, ch = item % nch_s;
    t.shared = 1;
    t.wt = wt;
    t.a_row = wt * kGemmBM;
    t.b_row = ch * BN;
    t.n_valid = min(BN, p.shared_rows - t.b_row);
    t.k = p.k_shared;
  } else {
    const int wt_r = p.w_rows_routed / kGemmBM;
    const int j = item - n_items_s;
    // largest e with chunk_pre[e] * wt_r <= j
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
    t.a_row = e * p.w_rows_routed + wt * kGemmBM;
    t.b_row = off_s[e] + ch * BN;
    t.n_valid = min(BN, off_s[e + 1] - t.b_row);
    t.k = p.k_routed;
  }
  t.n_mma = (t.n_valid + 15) & ~15;
  return t;
}

// Epilogue of one work item, run by the four epilogue warps (128 threads,
// named barrier 1).  `taddr` is this warp's TMEM lane quarter at the item's
// accumulator; TMEM row = weight row of the tile, column = token.  Thread
// (q, lane) owns weight row q*32 + lane and, per 32-token chunk, reads that
// row's 32 values with one tcgen05.ld.
//   down (swiglu = 0): row r is output column col0 + r of Y (fp32).  For each
//     token the warp stores 32 consecutive floats (128 B), straight from
//     registers -- no shared memory.
//   gate/up (swiglu = 1): rows 0..63 are gate and rows 64..127 the up values
//     of H columns col0 + 0..63.  Warp q (gate) and warp q+2 (up) swap half
//     of their tokens through `xchg`: the gate warp finishes tokens 0..15,
//     the up warp tokens 16..31, each storing 32 consecutive bf16 per token.
//   xchg: 4 warps x 32 lanes x 17 floats (padded against bank conflicts).
__device__ __forceinline__ void epilogue_store(uint32_t taddr, int n_valid,
                                               int b_row, void* out,
                                               long long ld, int col0,
                                               bool swiglu, float* xchg, int q,
                                               int ep, int lane,
                                               bool y_fp16 = false,
                                               bool h_fp32 = false,
                                               __half* act = nullptr,
                                               long long ld_act = 0) {
  (void)ep;
  bool overflow = false;
  for (int n0 = 0; n0 < n_valid; n0 += 32) {
    uint32_t r[32];
    tmem_ld32(taddr + n0, r);
    tmem_ld_wait();
    const int nleft = n_valid - n0;   // tokens of this chunk that exist
    if (!swiglu) {
      const size_t off =
          static_cast<size_t>(b_row + n0) * ld + col0 + q * 32 + lane;
      if (y_fp16) {
        // fp16 keeps 11 significant bits (8x finer than bf16); values
        // beyond its range are reported, never written silently as inf.
        // The warp's 32 channels x 32 tokens are transposed through its
        // 2 KB of the exchange buffer (token rows of 64 bytes) and leave as
        // 16-byte stores, four lanes per token row.
        __half* tile = reinterpret_cast<__half*>(xchg + q * 32 * 17);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float v = __uint_as_float(r[j]);
          if (j < nleft) overflow |= !(fabsf(v) <= 65504.f);
          tile[j * 32 + lane] = __float2half_rn(v);
        }
        __syncwarp();
        __half* dst = static_cast<__half*>(out) +
                      static_cast<size_t>(b_row + n0) * ld + col0 + q * 32;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int piece = lane + 32 * c;        // 16-byte piece of the tile
          const int j = piece >> 2, part = piece & 3;
          if (j < nleft)
            *reinterpret_cast<uint4*>(dst + static_cast<size_t>(j) * ld +
                                      8 * part) =
                *reinterpret_cast<const uint4*>(tile + j * 32 + 8 * part);
        }
        __syncwarp();
      } else {
        float* dst = static_cast<float*>(out) + off;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j < nleft) dst[static_cast<size_t>(j) * ld] = __uint_as_float(r[j]);
      }
      continue;
    }
    if (act != nullptr) {
      // the pre-activation of packed row q*32 + lane (gate rows 0..63, up
      // rows 64..127 of H columns col0 ..) for the backward, in fp16 (11
      // significant bits; out of range is reported like y); a warp's 32
      // lanes write 64 contiguous bytes of each token row
      __half* ad = act + static_cast<size_t>(b_row + n0) * ld_act +
                   2 * col0 + q * 32 + lane;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < nleft) {
          const float v = __uint_as_float(r[j]);
          overflow |= !(fabsf(v) <= 65504.f);
          ad[static_cast<size_t>(j) * ld_act] = __float2half_rn(v);
        }
    }
    const bool gate_warp = q < 2;
    const int pair_q = q & 1;               // warps q and q+2 form a pair
    // publish the half the partner warp finishes
    float* mine = xchg + ((q * 32) + lane) * 17;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      mine[j] = __uint_as_float(r[gate_warp ? 16 + j : j]);
    named_bar_sync(1, 128);
    const float* theirs = xchg + (((gate_warp ? q + 2 : q - 2) * 32) + lane) * 17;
    const int jbase = gate_warp ? 0 : 16;
    const size_t o = static_cast<size_t>(b_row + n0 + jbase) * ld + col0 +
                     pair_q * 32 + lane;
    if (h_fp32) {   // fp32 H (requantized to e4m3 by the caller)
      float* dst = static_cast<float*>(out) + o;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float g = gate_warp ? __uint_as_float(r[j]) : theirs[j];
        const float u = gate_warp ? theirs[j] : __uint_as_float(r[16 + j]);
        if (jbase + j < nleft) dst[static_cast<size_t>(j) * ld] = silu_f32(g) * u;
      }
    } else {
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(out) + o;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float g = gate_warp ? __uint_as_float(r[j]) : theirs[j];
        const float u = gate_warp ? theirs[j] : __uint_as_float(r[16 + j]);
        if (jbase + j < nleft)
          dst[static_cast<size_t>(j) * ld] = __float2bfloat16_rn(silu_f32(g) * u);
      }
    }
    named_bar_sync(1, 128);
  }
  if (overflow) report_error(ERR_CHECK, KID_GEMM, 200);
}

// K-block visited at step i of an item (plain ascending order).
__device__ __forceinline__ int k_block(const Tile&, int i, int) { return i; }

template <int BN, int STAGES>
__global__ void __launch_bounds__(192, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA_r,
                    const __grid_constant__ CUtensorMap tmB_r,
                    const __grid_constant__ CUtensorMap tmA_s,
                    const __grid_constant__ CUtensorMap tmB_s,
                    const GemmParams p) {
  using L = GemmSmem<BN, STAGES>;
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
  int* off_s = reinterpret_cast<int*>(smem + L::tab_off);        // [G+1]
  int* chunk_pre = off_s + (kMaxGroups + 1);                     // [G+1]
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
      mbar_init(bar_final + 8 + 8 * i, 1);                    // sched full
      mbar_init(bar_final + 8 + 8 * kSchedDepth + 8 * i, 5);  // sched empty:
    }                                   // MMA thread + one per epilogue warp
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
  // Item table: offsets (checked) and the prefix of token chunks per group.
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
  if (warp == 0) {   // inclusive scan of chunk counts, 32 at a time
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
  if (bad && threadIdx.x == 0) report_error(ERR_CHECK, KID_GEMM, 0);

  const int nch_s = p.shared_rows > 0 ? (p.shared_rows + BN - 1) / BN : 0;
  const int n_items_s = nch_s * (p.w_rows_shared / kGemmBM);
  const int n_items = bad ? 0
                          : n_items_s + (G > 0 ? chunk_pre[G] *
                                                     (p.w_rows_routed / kGemmBM)
                                               : 0);
  // Dynamic schedule: the producer claims items from a global counter (so
  // the items that share a weight tile run side by side on neighbouring
  // SMs) and hands each claimed item to the MMA and epilogue warps through a
  // small ring in shared memory; an item >= n_items tells them to stop.
  const uint32_t bar_sfull = bar_final + 8;                 // [kSchedDepth]
  const uint32_t bar_sempty = bar_sfull + 8 * kSchedDepth;  // [kSchedDepth]
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
      Tile t{};
      if (item < n_items)
        t = decode_item<BN>(item, p, n_items_s, nch_s, off_s, chunk_pre);
      while (!*abort_flag) {
        if (!mbar_wait(bar_sempty + 8 * slot, sph ^ 1, abort_flag, KID_GEMM, 5))
          break;
        sched[slot] = item;
        mbar_arrive(bar_sfull + 8 * slot);
        if (++slot == kSchedDepth) {
          slot = 0;
          sph ^= 1;
        }
        if (item >= n_items) break;
        const int next = atomicAdd(p.item_counter, 1);
        Tile tn{};
        if (next < n_items)
          tn = decode_item<BN>(next, p, n_items_s, nch_s, off_s, chunk_pre);
        const CUtensorMap* mA = t.shared ? &tmA_s : &tmA_r;
        const CUtensorMap* mB = t.shared ? &tmB_s : &tmB_r;
        const int nbox = (t.n_mma + kBoxRows - 1) / kBoxRows;
        const uint32_t bytes = L::a_bytes + nbox * kBoxRows * kGemmBK * 2;
        const int nk = t.k / kGemmBK;
        bool ok = true;
        for (int i = 0; i < nk; ++i) {
          if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1, abort_flag,
                         KID_GEMM, 1)) {
            ok = false;
            break;
          }
          const int kx = k_block(t, i, nk) * kGemmBK;
          const uint32_t fb = bar_full + 8 * stage;
          mbar_arrive_expect_tx(fb, bytes);
          tma_load_2d(sbase + L::a_off + stage * L::a_bytes, mA, kx, t.a_row,
                      fb);
          const uint32_t bdst = sbase + L::b_off + stage * L::b_bytes;
          for (int bx = 0; bx < nbox; ++bx)
            tma_load_2d(bdst + bx * kBoxRows * kGemmBK * 2, mB, kx,
                        t.b_row + bx * kBoxRows, fb);
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        item = next;
        t = tn;
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
      int acc = 0;
      uint32_t acc_phase = 0;
      int slot = 0;
      uint32_t sph = 0;
      while (!*abort_flag) {
        if (!mbar_wait(bar_sfull + 8 * slot, sph, abort_flag, KID_GEMM, 6))
          break;
        const int item = sched[slot];
        mbar_arrive(bar_sempty + 8 * slot);
        if (++slot == kSchedDepth) {
          slot = 0;
          sph ^= 1;
        }
        if (item >= n_items) break;
        const Tile t = decode_item<BN>(item, p, n_items_s, nch_s, off_s,
                                       chunk_pre);
        if (!mbar_wait(bar_tempty + 8 * acc, acc_phase ^ 1, abort_flag,
                       KID_GEMM, 2))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * BN;
        const uint32_t idesc = idesc_bf16_f32(kGemmBM, t.n_mma);
        const int nk = t.k / kGemmBK;
        bool ok = true;
        for (int i = 0; i < nk; ++i) {
          if (!mbar_wait(bar_full + 8 * stage, phase, abort_flag, KID_GEMM,
                         3)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = sbase + L::a_off + stage * L::a_bytes;
          const uint32_t b0 = sbase + L::b_off + stage * L::b_bytes;
#pragma unroll
          for (int kk = 0; kk < kGemmBK / 16; ++kk)
            mma_bf16(d_tmem, sdesc_k128(a0 + kk * 32),
                     sdesc_k128(b0 + kk * 32), idesc, (i | kk) != 0);
          mma_commit(bar_empty + 8 * stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit(bar_tfull + 8 * acc);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      // every MMA issued above is complete once this fires
      mma_commit(bar_final);
      mbar_drain(bar_final, 0);
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int ep = warp - 2;          // column group of the store phase
    const int q = warp & 3;           // TMEM sub-partition this warp may read
    int acc = 0;
    uint32_t acc_phase = 0;
    int slot = 0;
    uint32_t sph = 0;
    while (true) {
      const bool got = mbar_wait(bar_sfull + 8 * slot, sph, abort_flag,
                                 KID_GEMM, 7);
      const int item = got ? sched[slot] : n_items;
      __syncwarp();
      if (got && lane == 0) mbar_arrive(bar_sempty + 8 * slot);
      if (++slot == kSchedDepth) {
        slot = 0;
        sph ^= 1;
      }
      bool ok = got;
      if (got && item < n_items)
        ok = mbar_wait(bar_tfull + 8 * acc, acc_phase, abort_flag, KID_GEMM,
                       4);
      // The four epilogue warps share named barrier 1, so they leave the
      // loop together: each posts its verdict, all read all four.
      const bool wok = __all_sync(0xffffffffu, ok);
      if (lane == 0) ep_ok[ep] = wok ? 1 : 0;
      named_bar_sync(1, 128);
      if (!(ep_ok[0] && ep_ok[1] && ep_ok[2] && ep_ok[3])) break;
      if (item >= n_items) break;
      const Tile t = decode_item<BN>(item, p, n_items_s, nch_s, off_s,
                                     chunk_pre);
      tc_fence_after();
      void* out = t.shared ? p.out_shared : p.out_routed;
      const long long ld = t.shared ? p.ld_shared : p.ld_routed;
      epilogue_store(tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * BN,
                     t.n_valid, t.b_row, out, ld,
                     p.swiglu ? t.wt * 64 : t.wt * 128, p.swiglu != 0, stg,
                     q, ep, lane, p.y_fp16 != 0, false,
                     t.shared ? p.act_shared : p.act_routed,
                     t.shared ? p.ld_act_shared : p.ld_act_routed);
      tc_fence_before();
      mbar_arrive(bar_tempty + 8 * acc);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::tmem_cols);
  }
}

}  // namespace moe
