// Grouped expert GEMMs on CTA pairs: tcgen05.mma.cta_group::2.
// ("【推理llm論文精讀】DeepSeek V3技術論文", section 2.2: FFN^(r)_i of each
// selected expert and FFN^(s) of every shared expert, as in gemm.cuh.)
//
// Same work as grouped_gemm_kernel (weights on M, tokens on N, fused SwiGLU
// or down epilogue with fp16 Y, shared group first, item table from the
// device offsets, dynamic claim order), but each item is a 256-row weight
// tile x up to 256 tokens computed by a cluster of two CTAs on two SMs:
//
//   CTA r (r = 0, 1) holds weight rows a_row + 128 r .. +128 (its half of
//   A) and token rows b_row + r N/2 .. + N/2 (its half of B) in its own
//   shared memory; the even CTA issues M=256 MMAs that read both halves and
//   write each CTA's TMEM (128 lanes = its weight rows, N columns).
//
// Per SM and K-block this moves 16 KB of A and 16 KB of B (instead of 16 KB
// + 32 KB for a 128 x 256 tile on one SM): the shared-memory traffic of the
// TMA fills plus the MMA operand reads stays within the SM's shared-memory
// bandwidth at full tensor rate.
//
// Synchronisation (barriers live in each CTA; "L" = the even CTA):
//   full[s]   (L only)  : L's expect-tx arrival + both CTAs' TMA bytes
//   empty[s]  (both)    : MMA commit multicast to both CTAs
//   tfull[a]  (both)    : MMA commit multicast (accumulator a ready)
//   tempty[a] (L only)  : one arrival per epilogue warp of both CTAs
//   sfull[i]  (both)    : L's producer publishes a claimed item to both
//   sempty[i] (L only)  : L's MMA and epilogue warps, the odd CTA's producer
//                         and epilogue warps release the slot
#pragma once
#include "common.cuh"
#include "gemm.cuh"

namespace moe {

constexpr int kPairBM = 256;       // weight rows per item (128 per CTA)
constexpr int kPairBN = 256;       // max tokens per item (128 per CTA)
// K per pipeline stage: two 64-wide swizzle atoms per operand, loaded by one
// 3-D TMA box each, one MMA commit per stage.
constexpr int kPairBK = 128;
constexpr int kPairAtoms = kPairBK / 64;
constexpr int kPairStages = 3;
constexpr int kPairHalfRows = kPairBN / 2;

struct PairSmem {
  static constexpr int a_bytes = 128 * kPairBK * 2;            // 32 KB
  static constexpr int b_bytes = kPairHalfRows * kPairBK * 2;  // 32 KB
  static constexpr int a_off = 0;
  static constexpr int b_off = a_off + kPairStages * a_bytes;
  static constexpr int stg_off = b_off + kPairStages * b_bytes;
  static constexpr int stg_bytes = 4 * 32 * 17 * 4;   // epilogue exchange
  static constexpr int bar_off = stg_off + stg_bytes;
  static constexpr int n_bars = 2 * kPairStages + 5 + 2 * kSchedDepth;
  static constexpr int misc_off = bar_off + n_bars * 8;
  static constexpr int epok_off = misc_off + 16;
  static constexpr int sched_off = epok_off + 16;
  static constexpr int tab_off = sched_off + 4 * kSchedDepth;
  static constexpr int total = tab_off + 2 * (kMaxGroups + 1) * 4;
  static constexpr int alloc = total + 1024;
  static constexpr int tmem_cols = 2 * kPairBN;   // two accumulators
  static_assert(alloc <= 227 * 1024, "shared memory");
};

// Rows of the TMA box that loads a CTA's token half-tile of `half` rows:
// the smallest of 32, 64, 96, 128 that covers it.  Each K-atom of the box
// is box * 128 bytes, a multiple of the 1024-byte swizzle-atom alignment.
__host__ __device__ __forceinline__ int pair_token_box(int half) {
  return half <= 32 ? 32 : (half <= 64 ? 64 : (half <= 96 ? 96 : 128));
}

// Item -> (pair weight tile, token chunk); chunk index fastest.
__device__ __forceinline__ Tile decode_pair_item(int item, const GemmParams& p,
                                                 int n_items_s, int nch_s,
                                                 const int* off_s,
                                                 const int* chunk_pre) {
  Tile t;
  if (item < n_items_s) {
    const int wt = item / nch_s, ch = item % nch_s;
    t.shared = 1;
    t.wt = wt;
    t.a_row = wt * kPairBM;
    t.b_row = ch * kPairBN;
    t.n_valid = min(kPairBN, p.shared_rows - t.b_row);
    t.k = p.k_shared;
  } else {
    const int wt_r = p.w_rows_routed / kPairBM;
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
    // ce = ceil(m / 256) chunks of equal size (rounded up to 16): two
    // balanced chunks each keep their MMAs busy while the weight tile
    // streams, where 256 + a few tokens would leave the second item with
    // almost no MMA work (measured ~1.5% faster at the V3 prefill shape).
    const int m = off_s[e + 1] - off_s[e];
    const int sz = (((m + ce - 1) / ce) + 15) & ~15;
    t.shared = 0;
    t.wt = wt;
    t.a_row = e * p.w_rows_routed + wt * kPairBM;
    t.b_row = off_s[e] + ch * sz;
    t.n_valid = min(sz, off_s[e + 1] - t.b_row);
    t.k = p.k_routed;
  }
  t.n_mma = (t.n_valid + 15) & ~15;
  return t;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(192, 1)
grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA_r,
                         const __grid_constant__ CUtensorMap tmB_r,
                         const __grid_constant__ CUtensorMap tmA_s,
                         const __grid_constant__ CUtensorMap tmB_s,
                         const __grid_constant__ CUtensorMap tmB_r64,
                         const __grid_constant__ CUtensorMap tmB_s64,
                         const __grid_constant__ CUtensorMap tmB_r96,
                         const __grid_constant__ CUtensorMap tmB_s96,
                         const __grid_constant__ CUtensorMap tmB_r128,
                         const __grid_constant__ CUtensorMap tmB_s128,
                         const GemmParams p) {
  using L = PairSmem;
  constexpr int ST = kPairStages;
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
  const uint32_t lead = cluster_ctarank() & ~1u;    // cluster rank of the even CTA
  const uint32_t peer = lead + 1;
  const int G = p.n_groups;

  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_tfull + 8 * a, 1);
      mbar_init(bar_tempty + 8 * a, 8);       // 4 epilogue warps x 2 CTAs
    }
    mbar_init(bar_final, 1);
    for (int i = 0; i < kSchedDepth; ++i) {
      mbar_init(bar_sfull + 8 * i, 1);
      mbar_init(bar_sempty + 8 * i, 10);      // 5 consumers x 2 CTAs
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
    tmem_alloc_pair(sbase + L::misc_off, L::tmem_cols);
    tmem_relinquish_pair();
  }
  if (G > 0)
    for (int e = threadIdx.x; e <= G; e += blockDim.x) off_s[e] = p.offsets[e];
  __syncthreads();
  for (int e = threadIdx.x; e < G; e += blockDim.x) {
    const int m = off_s[e + 1] - off_s[e];
    if (m < 0 || off_s[e] < 0) *bad_flag = 1;
    chunk_pre[e + 1] = m > 0 ? (m + kPairBN - 1) / kPairBN : 0;
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
  if (bad && threadIdx.x == 0) report_error(ERR_CHECK, KID_GEMM, 100);

  const int nch_s =
      p.shared_rows > 0 ? (p.shared_rows + kPairBN - 1) / kPairBN : 0;
  const int n_items_s = nch_s * (p.w_rows_shared / kPairBM);
  const int n_items = bad ? 0
                          : n_items_s + (G > 0 ? chunk_pre[G] *
                                                     (p.w_rows_routed / kPairBM)
                                               : 0);
  // cluster addresses of the even CTA's barriers that both CTAs signal
  const uint32_t full_L = mapa_shared(bar_full, lead);
  const uint32_t tempty_L = mapa_shared(bar_tempty, lead);
  const uint32_t sempty_L = mapa_shared(bar_sempty, lead);

  if (warp == 0) {
    if (lane == 0) {
      // ------------- producer (both CTAs); scheduler in the even CTA -------
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      int slot = 0;
      uint32_t sph = 0;
      int item = (leader && !bad) ? atomicAdd(p.item_counter, 1) : n_items;
      while (!*abort_flag) {
        if (leader) {
          if (!mbar_wait_cl(bar_sempty + 8 * slot, sph ^ 1, abort_flag,
                            KID_GEMM, 101))
            break;
          sched[slot] = item;
          st_cluster_u32(mapa_shared(sbase + L::sched_off + 4 * slot, peer),
                         static_cast<uint32_t>(item));
          mbar_arrive(bar_sfull + 8 * slot);
          mbar_arrive_cluster(mapa_shared(bar_sfull + 8 * slot, peer));
        } else {
          if (!mbar_wait_cl(bar_sfull + 8 * slot, sph, abort_flag, KID_GEMM,
                            102))
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
        const Tile t = decode_pair_item(item, p, n_items_s, nch_s, off_s,
                                        chunk_pre);
        const CUtensorMap* mA = t.shared ? &tmA_s : &tmA_r;
        // The CTA's token half-tile comes in ONE TMA box of 32, 64, 96 or
        // 128 rows (the smallest that covers it; rows past the half are
        // loaded and ignored): one TMA instruction per operand and stage,
        // and no more token bytes than the next multiple of 32 rows.
        const int half = t.n_mma >> 1;                 // token rows per CTA
        const int box = pair_token_box(half);
        const CUtensorMap* mB =
            box == 32    ? (t.shared ? &tmB_s : &tmB_r)
            : box == 64  ? (t.shared ? &tmB_s64 : &tmB_r64)
            : box == 96  ? (t.shared ? &tmB_s96 : &tmB_r96)
                         : (t.shared ? &tmB_s128 : &tmB_r128);
        const int a_row = t.a_row + static_cast<int>(rank) * 128;
        const int b_row = t.b_row + static_cast<int>(rank) * half;
        const uint32_t pair_bytes = 2u * (L::a_bytes + box * kPairBK * 2);
        const int nk = t.k / kPairBK;
        bool ok = true;
        for (int i = 0; i < nk; ++i) {
          if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1, abort_flag,
                         KID_GEMM, 103)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(bar_full + 8 * stage, pair_bytes);
          const uint32_t fb = full_L + 8 * stage;
          const int ka = i * kPairAtoms;
          tma_load_3d_pair(sbase + L::a_off + stage * L::a_bytes, mA, a_row, ka,
                           fb);
          tma_load_3d_pair(sbase + L::b_off + stage * L::b_bytes, mB, b_row, ka,
                           fb);
          ++issued;
          if (++stage == ST) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        item = next;
      }
      if (*abort_flag && leader) {   // let the pair's loads land
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
    if (lane == 0 && leader) {
      // ---------------- MMA issuer (even CTA) ----------------
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      int slot = 0;
      uint32_t sph = 0;
      while (!*abort_flag) {
        if (!mbar_wait_cl(bar_sfull + 8 * slot, sph, abort_flag, KID_GEMM,
                          104))
          break;
        const int item = sched[slot];
        mbar_arrive(bar_sempty + 8 * slot);
        if (++slot == kSchedDepth) {
          slot = 0;
          sph ^= 1;
        }
        if (item >= n_items) break;
        const Tile t = decode_pair_item(item, p, n_items_s, nch_s, off_s,
                                        chunk_pre);
        if (!mbar_wait_cl(bar_tempty + 8 * acc, acc_phase ^ 1, abort_flag,
                          KID_GEMM, 105))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * kPairBN;
        const uint32_t idesc = idesc_bf16_f32(kPairBM, t.n_mma);
        const int nk = t.k / kPairBK;
        // token box rows of this item (the K-atom stride of its B stage)
        const int half = t.n_mma >> 1;
        const uint32_t b_atom =
            static_cast<uint32_t>(pair_token_box(half)) * 128u;
        bool ok = true;
        for (int i = 0; i < nk; ++i) {
          if (!mbar_wait(bar_full + 8 * stage, phase, abort_flag, KID_GEMM,
                         106)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = sbase + L::a_off + stage * L::a_bytes;
          const uint32_t b0 = sbase + L::b_off + stage * L::b_bytes;
#pragma unroll
          for (int kk = 0; kk < kPairBK / 16; ++kk) {
            const uint32_t at = kk >> 2, w = (kk & 3) * 32;
            mma_bf16_pair(d_tmem, sdesc_k128(a0 + at * (128u * 128u) + w),
                          sdesc_k128(b0 + at * b_atom + w), idesc,
                          (i | kk) != 0);
          }
          mma_commit_pair_mc(bar_empty + 8 * stage, 0x3);
          if (++stage == ST) {
            stage = 0;
            phase ^= 1;
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
  } else {
    // ---------------- epilogue (warps 2..5 of both CTAs) ----------------
    const int ep = warp - 2;
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    int slot = 0;
    uint32_t sph = 0;
    while (true) {
      const bool got = mbar_wait_cl(bar_sfull + 8 * slot, sph, abort_flag,
                                    KID_GEMM, 107);
      const int item = got ? sched[slot] : n_items;
      __syncwarp();
      if (got && lane == 0) mbar_arrive_cluster(sempty_L + 8 * slot);
      if (++slot == kSchedDepth) {
        slot = 0;
        sph ^= 1;
      }
      bool ok = got;
      if (got && item < n_items)
        ok = mbar_wait(bar_tfull + 8 * acc, acc_phase, abort_flag, KID_GEMM,
                       108);
      const bool wok = __all_sync(0xffffffffu, ok);
      if (lane == 0) ep_ok[ep] = wok ? 1 : 0;
      named_bar_sync(1, 128);
      if (!(ep_ok[0] && ep_ok[1] && ep_ok[2] && ep_ok[3])) break;
      if (item >= n_items) break;
      const Tile t = decode_pair_item(item, p, n_items_s, nch_s, off_s,
                                      chunk_pre);
      tc_fence_after();
      void* out = t.shared ? p.out_shared : p.out_routed;
      const long long ld = t.shared ? p.ld_shared : p.ld_routed;
      const int tile128 = t.wt * 2 + static_cast<int>(rank);
      epilogue_store(tmem + (static_cast<uint32_t>(q * 32) << 16) +
                         acc * kPairBN,
                     t.n_valid, t.b_row, out, ld,
                     p.swiglu ? tile128 * 64 : tile128 * 128, p.swiglu != 0,
                     stg, q, ep, lane, p.y_fp16 != 0, false,
                     t.shared ? p.act_shared : p.act_routed,
                     t.shared ? p.ld_act_shared : p.ld_act_routed);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(tempty_L + 8 * acc);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
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
