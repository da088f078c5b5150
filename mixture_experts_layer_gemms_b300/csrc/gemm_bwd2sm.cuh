// The layer backward's grouped GEMMs on CTA pairs (tcgen05.mma.cta_group::2):
// the same three kinds of work as bwd_gemm_kernel (gemm_bwd.cuh) -- Dgrad
// with an MN-major weight operand (for dH optionally with the SwiGLU
// backward from saved pre-activations), the gate/up recompute with the
// SwiGLU backward epilogue, Wgrad with both operands MN-major -- on 256-row
// M tiles split over two SMs, as the forward's grouped_gemm_pair_kernel does
// ("AI新顶流-DeepSeek 技术大揭秘", section "FP8混合精度训练框架": the Dgrad and
// Wgrad GEMMs of each linear operator).
//
// CTA r of a pair holds M rows m0 + 128 r .. +128 of the A operand and its
// half of the B operand (tokens kinds: token rows n0 + r N/2 .. + N/2; Wgrad:
// columns n0 + 128 r .. +128) in its own shared memory; the even CTA issues
// M = 256 MMAs reading both halves, each CTA's TMEM receives its 128 rows x
// all N columns.  A stage of the token kinds is 128 of K: every operand
// half is one 3-D TMA box of two 64-element swizzle atoms (K-major: {64 K,
// rows, 2 K-atoms}; MN-major: {64 MN, 128 K rows, 2 MN-atoms}), 32 KB;
// Wgrad stages are 64 of K (16 KB per operand half), five of them.  Per SM and stage this
// moves 32 KB of A and at most 32 KB of B, where a 128 x 256 tile on one SM
// moves 16 + 32 KB per 64 of K: the shared-memory traffic of TMA fills plus
// MMA operand reads fits the SM's bandwidth at full tensor rate.
//
// Synchronisation is the forward pair kernel's (barriers in each CTA, the
// even CTA's full / tempty / sempty signalled by both).
#pragma once
#include "common.cuh"
#include "gemm.cuh"
#include "gemm_bwd.cuh"

namespace moe {

constexpr int kBwdPairBM = 256;      // M rows per item (128 per CTA)
constexpr int kBwdPairBN = 256;      // N per item
// Wgrad's store boxes: a ring of this many 2 KB boxes per epilogue warp
constexpr int kWgradBoxes = 3;

// K per stage and stages: 128 x 3 for the tokens kinds; 64 x 5 for Wgrad,
// whose epilogue (not its operand stream) is the bound and takes the shared
// memory freed for a ring of store boxes.
template <int KIND>
__host__ __device__ constexpr int bwd_pair_bk() {
  return KIND == kWgrad ? 64 : 128;
}
template <int KIND>
__host__ __device__ constexpr int bwd_pair_stages() {
  return KIND == kWgrad ? 5 : 3;
}

template <int KIND>
struct BwdPairSmem {
  static constexpr int BK = bwd_pair_bk<KIND>();
  static constexpr int ST = bwd_pair_stages<KIND>();
  static constexpr int a_bytes = 128 * BK * 2;   // 32 KB (16 KB for Wgrad)
  static constexpr int b_bytes = 128 * BK * 2;
  static constexpr int a_off = 0;
  static constexpr int b_off = a_off + ST * a_bytes;
  static constexpr int stg_off = b_off + ST * b_bytes;
  static constexpr int stg_bytes =
      KIND == kWgrad ? 8 * kWgradBoxes * 2048
                     : (KIND == kRecomp ? 2 * 128 * 17 * 4 : kBwdStgBytes);
  static constexpr int bar_off = stg_off + stg_bytes;
  static constexpr int n_bars = 2 * ST + 5 + 2 * kSchedDepth;
  static constexpr int misc_off = bar_off + n_bars * 8;
  static constexpr int epok_off = misc_off + 16;
  static constexpr int sched_off = epok_off + 32;     // 8 epilogue verdicts
  static constexpr int tab_off = sched_off + 4 * kSchedDepth;
  static constexpr int total = tab_off + 3 * (kMaxGroups + 1) * 4;
  static constexpr int alloc = total + 1024;
  static constexpr int tmem_cols = 2 * kBwdPairBN;
  static_assert(alloc <= 227 * 1024, "shared memory");
};

// Tensor maps of one pair launch.  Tokens kinds: A (weights; K-major 3-D
// {64, 128 rows, 2 K-atoms} for Recomp, MN-major {64, 128 K rows, 2
// M-atoms} for Dgrad) and the token operand with 32-, 64- and 128-row boxes
// (the smallest box that covers a CTA's token half is used).  Wgrad: A and
// B MN-major in the 128-row slots.
// Wgrad also takes the gradients' output maps: o (W_gate or W_down grads)
// and o2 (W_up grads), routed and shared, 2-D boxes of 32 x 32 elements
// with 64-byte (bf16) or 128-byte (fp32) swizzle.
struct BwdPairMaps {
  CUtensorMap a_r, a_s, b_r32, b_s32, b_r64, b_s64, b_r128, b_s128;
  CUtensorMap o_r, o2_r, o_s, o2_s;
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a,
                                             uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a),
               "r"(b), "r"(c), "r"(d)
               : "memory");
}

// kWgrad epilogue on CTA pairs: one warp's 32 accumulator rows x 128 of
// the tile's 256 columns (`cbeg` .. +128; two warps share each TMEM lane
// quarter): TMEM -> registers (all 128 columns, then the accumulator is
// released), then 32 columns at a time -> a box in the warp's
// 2 KB of shared memory, laid out as the output map's 64-byte swizzle
// expects (rows of 64 bytes: 32 bf16 or 16 fp32 columns) -> one TMA store
// per box, issued by lane 0.  The global writes leave as whole boxes, off
// the load/store path.  Box (x, y): x = column n0 + c, y = `y` (the warp's
// first output row); for the shared down gradient (col_split = I) column c
// is column c % I of rows y + (c / I) s_rows.  `zero`: the group had no
// rows, zeros are stored.
__device__ __forceinline__ void wgrad_store_box(const CUtensorMap* map, int c,
                                                int y, int col_split,
                                                int s_rows, uint32_t buf) {
  int x = c, yy = y;
  if (col_split > 0) {
    x = c % col_split;
    yy = y + (c / col_split) * s_rows;
  }
  tma_store_2d(map, x, yy, buf);
  bulk_commit();
}

// The warp's 128 accumulator columns, read from TMEM into registers in one
// go (four 32-column loads, one wait) so the accumulator can be handed back
// to the MMA before any of it is stored; zeros for a group with no rows.
__device__ __forceinline__ void bwd_ep_wgrad_take(uint32_t taddr, int cbeg,
                                                  bool zero,
                                                  uint32_t (&r)[4][32]) {
  if (!zero) {
#pragma unroll
    for (int j = 0; j < 4; ++j) tmem_ld32(taddr + cbeg + 32 * j, r[j]);
    tmem_ld_wait();
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int k = 0; k < 32; ++k) r[j][k] = 0u;
  }
}

// Stores what bwd_ep_wgrad_take read: each 32-column chunk becomes one bf16
// box (or two fp32 boxes) in the warp's ring, then a TMA store.
__device__ __forceinline__ void bwd_ep_wgrad_put(const uint32_t (&r)[4][32],
                                                 int cbeg,
                                                 const CUtensorMap* map,
                                                 int n0, int y, int col_split,
                                                 int s_rows, bool bf16,
                                                 uint32_t ring_base,
                                                 int& ring, int lane) {
  const int sw = (lane >> 1) & 3;            // 64-byte swizzle of this row
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int c0 = cbeg + 32 * j;
    if (bf16) {            // one box of 32 columns
      const uint32_t buf = ring_base + (ring % kWgradBoxes) * 2048u;
      const uint32_t row_addr = buf + lane * 64;
      ++ring;
      // the box written kWgradBoxes stores ago has been read
      if (lane == 0) bulk_wait_read<kWgradBoxes - 1>();
      __syncwarp();
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
#define MOE_F(k) __uint_as_float(r[j][cc * 8 + (k)])
        st_shared_v4(row_addr + ((cc ^ sw) * 16),
                     pack_bf16x2(MOE_F(0), MOE_F(1)),
                     pack_bf16x2(MOE_F(2), MOE_F(3)),
                     pack_bf16x2(MOE_F(4), MOE_F(5)),
                     pack_bf16x2(MOE_F(6), MOE_F(7)));
#undef MOE_F
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) wgrad_store_box(map, n0 + c0, y, col_split, s_rows, buf);
    } else {               // two boxes of 16 columns
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        const uint32_t buf = ring_base + (ring % kWgradBoxes) * 2048u;
        const uint32_t row_addr = buf + lane * 64;
        ++ring;
        if (lane == 0) bulk_wait_read<kWgradBoxes - 1>();
        __syncwarp();
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
          st_shared_v4(row_addr + ((cc ^ sw) * 16), r[j][hb * 16 + cc * 4],
                       r[j][hb * 16 + cc * 4 + 1], r[j][hb * 16 + cc * 4 + 2],
                       r[j][hb * 16 + cc * 4 + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0)
          wgrad_store_box(map, n0 + c0 + hb * 16, y, col_split, s_rows, buf);
      }
    }
  }
}

// Item -> tile.  Tokens kinds: (group, 256-row M tile, token chunk), chunk
// fastest; a group's chunks split its tokens evenly (each rounded up to
// 16), as in the forward.  Wgrad: (group, M tile, N tile), N fastest.
template <int KIND>
__device__ __forceinline__ BTile bwd_decode_pair(int item, const BwdParams& p,
                                                 int n_items_s, int nch_s,
                                                 const int* offp,
                                                 const int* cnt,
                                                 const int* chunk_pre) {
  constexpr int BK = bwd_pair_bk<KIND>();
  BTile t;
  if constexpr (KIND == kWgrad) {
    const int ntn_s = p.n_shared / kBwdPairBN;
    const int ntn_r = p.n_routed / kBwdPairBN;
    const int per_r = (p.m_routed / kBwdPairBM) * ntn_r;
    int local, ntn;
    if (item < n_items_s) {
      t.shared = 1;
      t.e = 0;
      local = item;
      ntn = ntn_s;
      t.k_row0 = 0;
      t.nk = (p.shared_rows + BK - 1) / BK;
      t.krows = t.nk * BK;            // rows past T read as zero
    } else {
      const int j = item - n_items_s;
      t.shared = 0;
      t.e = j / per_r;
      local = j % per_r;
      ntn = ntn_r;
      t.k_row0 = offp[t.e];
      t.krows = (cnt[t.e] + kPadRows - 1) / kPadRows * kPadRows;
      t.nk = (t.krows + BK - 1) / BK;
    }
    t.wt = local / ntn;
    t.m0 = t.wt * kBwdPairBM;
    t.n0 = (local % ntn) * kBwdPairBN;
    t.n_valid = kBwdPairBN;
    t.n_mma = kBwdPairBN;
  } else {
    if (item < n_items_s) {
      const int wt = item / nch_s, ch = item % nch_s;
      t.shared = 1;
      t.e = 0;
      t.wt = wt;
      t.n0 = ch * kBwdPairBN;
      t.n_valid = min(kBwdPairBN, p.shared_rows - t.n0);
      t.k_row0 = 0;
      t.nk = p.k_shared / BK;
    } else {
      const int wt_r = p.m_routed / kBwdPairBM;
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
      const int m = cnt[e];
      const int sz = (((m + ce - 1) / ce) + 15) & ~15;
      t.shared = 0;
      t.e = e;
      t.wt = wt;
      t.n0 = offp[e] + ch * sz;
      t.n_valid = min(sz, m - ch * sz);
      t.k_row0 = e * p.k_routed;
      t.nk = p.k_routed / BK;
    }
    t.m0 = t.wt * kBwdPairBM;
    t.n_mma = (t.n_valid + 15) & ~15;
    t.krows = t.nk * BK;
  }
  return t;
}

// Threads: producer warp, MMA warp, then 4 epilogue warps (8 for Wgrad,
// whose epilogue -- 128 x 256 stores per short K loop -- is its bound, and
// for the recompute, whose SwiGLU-backward epilogue reads dH and writes H
// and dA: two groups of four warps take alternate 32-token chunks).
template <int KIND>
__host__ __device__ constexpr int bwd_pair_epi_warps() {
  return KIND == kDgrad ? 4 : 8;
}
template <int KIND>
__host__ __device__ constexpr int bwd_pair_threads() {
  return 64 + 32 * bwd_pair_epi_warps<KIND>();
}

template <int KIND>
__global__ void __cluster_dims__(2, 1, 1)
__launch_bounds__(bwd_pair_threads<KIND>(), 1)
bwd_gemm_pair_kernel(const __grid_constant__ BwdPairMaps maps,
                     const BwdParams p) {
  using L = BwdPairSmem<KIND>;
  constexpr int ST = L::ST;
  constexpr int BK = L::BK;
  // MN-major operand atoms are BK rows x 128 B; K-major ones 128 rows
  constexpr uint32_t kMnAtom = BK * 128u;
  constexpr bool kTokens = KIND != kWgrad;
  constexpr bool kAmn = KIND != kRecomp;
  constexpr bool kBmn = KIND == kWgrad;
  constexpr int NEPI = bwd_pair_epi_warps<KIND>();
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
  int* offp = reinterpret_cast<int*>(smem + L::tab_off);
  int* cnt = offp + (kMaxGroups + 1);
  int* chunk_pre = cnt + (kMaxGroups + 1);
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
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_tfull + 8 * a, 1);
      mbar_init(bar_tempty + 8 * a, 2 * NEPI);   // epilogue warps x 2 CTAs
    }
    mbar_init(bar_final, 1);
    for (int i = 0; i < kSchedDepth; ++i) {
      mbar_init(bar_sfull + 8 * i, 1);
      mbar_init(bar_sempty + 8 * i, 2 * (1 + NEPI));   // consumers x 2 CTAs
    }
    *abort_flag = 0;
    *bad_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(sbase + L::misc_off, L::tmem_cols);
    tmem_relinquish_pair();
  }
  for (int e = threadIdx.x; e < G; e += blockDim.x) {
    const int o = p.offpad[e], c = p.offsets[e + 1] - p.offsets[e];
    offp[e] = o;
    cnt[e] = c;
    if (c < 0 || o < 0 || (o & (kPadRows - 1)) != 0) *bad_flag = 1;
    chunk_pre[e + 1] = c > 0 ? (c + kBwdPairBN - 1) / kBwdPairBN : 0;
  }
  if (threadIdx.x == 0) chunk_pre[0] = 0;
  __syncthreads();
  for (int e = threadIdx.x; e < G; e += blockDim.x)
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
  cluster_sync();          // both CTAs' barriers exist before any remote use
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool bad = *bad_flag != 0;
  if (bad && threadIdx.x == 0) report_error(ERR_CHECK, KID_GEMM_BWD, 100);

  int n_items_s = 0, nch_s = 0, n_items = 0;
  if constexpr (kTokens) {
    nch_s = p.shared_rows > 0 ? (p.shared_rows + kBwdPairBN - 1) / kBwdPairBN
                              : 0;
    n_items_s = nch_s * (p.m_shared / kBwdPairBM);
    n_items = n_items_s +
              (G > 0 ? chunk_pre[G] * (p.m_routed / kBwdPairBM) : 0);
  } else {
    n_items_s = p.shared_rows > 0 ? (p.m_shared / kBwdPairBM) *
                                        (p.n_shared / kBwdPairBN)
                                  : 0;
    n_items = n_items_s + G * (p.m_routed / kBwdPairBM) *
                              (p.n_routed / kBwdPairBN);
  }
  // the item tables are identical in both CTAs; a bad table in either
  // stops both (the odd CTA follows the even one's schedule)
  if (bad) n_items = 0;
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
                            KID_GEMM_BWD, 101))
            break;
          sched[slot] = item;
          st_cluster_u32(mapa_shared(sbase + L::sched_off + 4 * slot, peer),
                         static_cast<uint32_t>(item));
          mbar_arrive(bar_sfull + 8 * slot);
          mbar_arrive_cluster(mapa_shared(bar_sfull + 8 * slot, peer));
        } else {
          if (!mbar_wait_cl(bar_sfull + 8 * slot, sph, abort_flag,
                            KID_GEMM_BWD, 102))
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
        const BTile t = bwd_decode_pair<KIND>(item, p, n_items_s, nch_s, offp,
                                              cnt, chunk_pre);
        const CUtensorMap* mA = t.shared ? &maps.a_s : &maps.a_r;
        const CUtensorMap* mB;
        int half = 0;
        uint32_t b_bytes;
        if constexpr (kTokens) {
          half = t.n_mma >> 1;                       // token rows per CTA
          const int box = half <= 32 ? 32 : (half <= 64 ? 64 : 128);
          mB = box == 32 ? (t.shared ? &maps.b_s32 : &maps.b_r32)
                         : (box == 64 ? (t.shared ? &maps.b_s64 : &maps.b_r64)
                                      : (t.shared ? &maps.b_s128
                                                  : &maps.b_r128));
          b_bytes = static_cast<uint32_t>(box) * BK * 2;
        } else {
          mB = t.shared ? &maps.b_s128 : &maps.b_r128;
          b_bytes = L::b_bytes;
        }
        const uint32_t pair_bytes = 2u * (L::a_bytes + b_bytes);
        const int m_atom = (t.m0 + static_cast<int>(rank) * 128) / 64;
        const int a_row = (t.shared ? 0 : t.e * p.m_routed) + t.m0 +
                          static_cast<int>(rank) * 128;
        bool ok = true;
        for (int i = 0; i < t.nk; ++i) {
          if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1, abort_flag,
                         KID_GEMM_BWD, 103)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(bar_full + 8 * stage, pair_bytes);
          const uint32_t fb = full_L + 8 * stage;
          const uint32_t adst = sbase + L::a_off + stage * L::a_bytes;
          const uint32_t bdst = sbase + L::b_off + stage * L::b_bytes;
          const int krow = t.k_row0 + i * BK;
          if constexpr (kAmn)
            tma_load_3d_pair(adst, mA, krow, m_atom, fb);
          else
            tma_load_3d_pair(adst, mA, a_row, i * 2, fb);
          if constexpr (kBmn)
            tma_load_3d_pair(bdst, mB, krow,
                             (t.n0 + static_cast<int>(rank) * 128) / 64, fb);
          else
            tma_load_3d_pair(bdst, mB, t.n0 + static_cast<int>(rank) * half,
                             i * 2, fb);
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
        if (!mbar_wait_cl(bar_sfull + 8 * slot, sph, abort_flag, KID_GEMM_BWD,
                          104))
          break;
        const int item = sched[slot];
        mbar_arrive(bar_sempty + 8 * slot);
        if (++slot == kSchedDepth) {
          slot = 0;
          sph ^= 1;
        }
        if (item >= n_items) break;
        const BTile t = bwd_decode_pair<KIND>(item, p, n_items_s, nch_s, offp,
                                              cnt, chunk_pre);
        if (!mbar_wait_cl(bar_tempty + 8 * acc, acc_phase ^ 1, abort_flag,
                          KID_GEMM_BWD, 105))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * kBwdPairBN;
        const uint32_t idesc = idesc_bf16_mn(kBwdPairBM, t.n_mma, kAmn, kBmn);
        // K-major token operand: K-atom stride of this item's B stage
        const int half = t.n_mma >> 1;
        const uint32_t b_atom =
            (half <= 32 ? 32u : (half <= 64 ? 64u : 128u)) * 128u;
        bool ok = true;
        for (int i = 0; i < t.nk; ++i) {
          if (!mbar_wait(bar_full + 8 * stage, phase, abort_flag,
                         KID_GEMM_BWD, 106)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = sbase + L::a_off + stage * L::a_bytes;
          const uint32_t b0 = sbase + L::b_off + stage * L::b_bytes;
          // 16-row K steps in this stage (a Wgrad group's last block may
          // end early)
          const int nkk = min(BK, t.krows - i * BK) / 16;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            if (kk >= nkk) break;
            const uint32_t at = kk >> 2, w = (kk & 3) * 32;
            const uint64_t ad = kAmn ? sdesc_mn128(a0 + kk * 2048, kMnAtom)
                                     : sdesc_k128(a0 + at * 16384u + w);
            const uint64_t bd = kBmn ? sdesc_mn128(b0 + kk * 2048, kMnAtom)
                                     : sdesc_k128(b0 + at * b_atom + w);
            mma_bf16_pair(d_tmem, ad, bd, idesc, (i | kk) != 0);
          }
          mma_commit_pair_mc(bar_empty + 8 * stage, 0x3);
          if (++stage == ST) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit_pair_mc(bar_tfull + 8 * acc, 0x3);   // also for nk == 0
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      mma_commit_pair_mc(bar_final, 0x1);
      mbar_drain_cl(bar_final, 0);
    }
  } else {
    // ---------- epilogue (warps 2 .. 1 + NEPI of both CTAs) ----------
    const int ep = warp - 2;
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    int slot = 0;
    uint32_t sph = 0;
    bool ovf = false;
    int ring = 0;          // Wgrad: this warp's next store box
    while (true) {
      const bool got = mbar_wait_cl(bar_sfull + 8 * slot, sph, abort_flag,
                                    KID_GEMM_BWD, 107);
      const int item = got ? sched[slot] : n_items;
      __syncwarp();
      if (got && lane == 0) mbar_arrive_cluster(sempty_L + 8 * slot);
      if (++slot == kSchedDepth) {
        slot = 0;
        sph ^= 1;
      }
      bool ok = got;
      if (got && item < n_items)
        ok = mbar_wait(bar_tfull + 8 * acc, acc_phase, abort_flag,
                       KID_GEMM_BWD, 108);
      const bool wok = __all_sync(0xffffffffu, ok);
      if (lane == 0) ep_ok[ep] = wok ? 1 : 0;
      named_bar_sync(1, 32 * NEPI);
      bool all_ok = true;
#pragma unroll
      for (int w = 0; w < NEPI; ++w) all_ok = all_ok && ep_ok[w] != 0;
      if (!all_ok) break;
      if (item >= n_items) break;
      const BTile t = bwd_decode_pair<KIND>(item, p, n_items_s, nch_s, offp,
                                            cnt, chunk_pre);
      tc_fence_after();
      const uint32_t ta =
          tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * kBwdPairBN;
      const int m_cta = t.m0 + static_cast<int>(rank) * 128;  // CTA's rows
      if constexpr (KIND == kDgrad) {
        const __half* act = t.shared ? p.act_s : p.act_r;
        if (act != nullptr) {
          const long long shift =
              t.shared ? 0 : static_cast<long long>(p.offsets[t.e]) - offp[t.e];
          bwd_ep_dgrad_act(
              ta, t.n_valid, t.n0, m_cta + q * 32 + lane, shift, act,
              t.shared ? p.ld_act_s : p.ld_act_r,
              static_cast<__nv_bfloat16*>(t.shared ? p.out_s : p.out_r),
              t.shared ? p.ld_s : p.ld_r,
              static_cast<__nv_bfloat16*>(t.shared ? p.out2_s : p.out2_r),
              t.shared ? p.ld2_s : p.ld2_r);
        } else {
          __half* out = static_cast<__half*>(t.shared ? p.out_s : p.out_r);
          const long long ld = t.shared ? p.ld_s : p.ld_r;
          bwd_ep_dgrad(ta, t.n_valid, t.n0, out, ld, m_cta + q * 32 + lane,
                       ovf);
        }
      } else if constexpr (KIND == kRecomp) {
        const int grp = ep >> 2;            // exchange group of 4 warps
        bwd_ep_recomp(ta, t.n_valid, t.n0, m_cta / 128,
                      t.shared ? p.dh_s : p.dh_r, t.shared ? p.ld_s : p.ld_r,
                      static_cast<__nv_bfloat16*>(t.shared ? p.out_s : p.out_r),
                      static_cast<__nv_bfloat16*>(t.shared ? p.out2_s
                                                           : p.out2_r),
                      t.shared ? p.ld2_s : p.ld2_r, stg + grp * 128 * 17, q,
                      lane, 32 * grp, 64, 2 + grp);
      } else {
        const int m = m_cta + q * 32;       // the warp's first output row
        const CUtensorMap* om;
        int y, col_split = 0, s_rows = 0;
        if (p.wgrad_gu) {   // packed row -> gate / up row of [.., I, d]
          const int within = m & 127;
          const int irow = (m >> 7) * 64 + (within & 63);
          const bool gate = within < 64;
          om = t.shared ? (gate ? &maps.o_s : &maps.o2_s)
                        : (gate ? &maps.o_r : &maps.o2_r);
          y = (t.shared ? 0 : t.e * p.I) + irow;
        } else {            // [.., d, I]
          om = t.shared ? &maps.o_s : &maps.o_r;
          y = (t.shared ? 0 : t.e * p.m_routed) + m;
          if (t.shared) {
            col_split = p.I;
            s_rows = p.m_shared;
          }
        }
        uint32_t r[4][32];
        bwd_ep_wgrad_take(ta, (ep >> 2) * 128, t.nk == 0, r);
        // the accumulator is free once its columns are in registers: hand
        // it back before the stores, so the MMA runs on while they drain
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(tempty_L + 8 * acc);
        bwd_ep_wgrad_put(r, (ep >> 2) * 128, om, t.n0, y, col_split, s_rows,
                         p.out_bf16 != 0,
                         smem_u32(stg) + ep * (kWgradBoxes * 2048u), ring,
                         lane);
      }
      if constexpr (KIND != kWgrad) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(tempty_L + 8 * acc);
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    if (ovf) report_error(ERR_CHECK, KID_GEMM_BWD, 200);
    if constexpr (KIND == kWgrad)
      if (lane == 0) bulk_wait_all();   // stores done before smem goes away
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
