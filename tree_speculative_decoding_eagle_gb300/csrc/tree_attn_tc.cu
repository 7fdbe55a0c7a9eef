// Stage 3 (tensor-core path, bf16): tree-masked attention of the tree nodes
// over the KV prefix on the 5th-generation tensor cores.
//
// [EAGLE-1] sections "用語解説" (Tree Attention) and "Tree Attention の役割":
// the target scores every branch of the draft tree in one forward pass; with
// the [EAGLE-2] mask (section "注意マスクの調整") node i attends to the
// prefix and to its own ancestors only.
//
// One CTA per (sequence b, KV head g, group of MT 128-row M-tiles, KV split).
// Query rows are (node, head-in-group) pairs, so the m+1 nodes x G grouped
// heads of a KV head share every K/V tile.  Key tiles hold NK keys: first the
// prefix (positions 0..kv_len-1), then the tree nodes, masked with the
// ancestor bits.  Roles:
//   * producer warp: K/V tiles into a ring of shared-memory stages, by TMA
//     (128-byte swizzle) for full tiles, by plain loads with zero fill for
//     the ragged last prefix tile;
//   * MMA warp (one thread): S_t = Q_t K^T (A = Q from shared memory) and
//     O_t += P_t V (A = P from tensor memory), accumulators in tensor memory,
//     completion via tcgen05.commit on mbarriers.  Per tile j: S of tile j+1
//     for every M-tile as soon as its softmax has taken S(j) into registers,
//     then P(j).V for every M-tile once P(j) is in tensor memory;
//   * one softmax warpgroup per M-tile: reads its S rows from tensor memory
//     into registers once and releases S at once (so the next tile's
//     S = Q K^T runs while this tile's exponents are taken), takes the row
//     maximum and the exponents, writes P as packed bf16 pairs into tensor
//     memory, keeps the row sum, and rescales its O rows in tensor memory
//     only when the running maximum grows by more than 2^8.  A warp whose 32
//     rows all lie past the last (node, head) row only signals.
// Tensor memory per M-tile: S (NK columns), P (NK/2), O (dh).
// KV split (few heads: S <= 8 CTAs share one (b, g, M-group)): each CTA
// leaves its unnormalised fp32 O rows and (m, l) in its own workspace slot.
// When the launch is one wave the S CTAs are one thread-block cluster and
// each merges 1/S of the rows from all S slots after a cluster barrier;
// otherwise the CTAs leave at once (no co-scheduling, no waiting on peers)
// and tree_attn_merge_kernel merges.  The slots are read back from L2.
// Every wait is bounded; a timeout raises EAGLE_ERR_TIMEOUT in the status
// word and the CTA drains its copies and MMAs, frees tensor memory and exits.
#include <mutex>

#include "common.cuh"
#include "sm100.cuh"

namespace eagle {

using namespace sm100;

struct TcArgs {
  const __nv_bfloat16 *q, *k_cache, *v_cache;
  const int32_t *kv_len;
  const uint64_t *mask;
  int B, n, Hq, Hkv, G, Lmax, S, W;
  // paged prefix (block_table != nullptr): k_cache / v_cache are page pools
  // [num_pages, Hkv, page_size, dh]; logical position L of sequence b is row
  // L % page_size of page block_table[b * max_pages + L / page_size].  TMA
  // boxes are page_box = min(page_size, NK) rows.
  const int32_t *block_table;
  int max_pages, page_size, page_box, num_pages;
  float scale_log2;  // softmax scale times log2(e)
  __nv_bfloat16 *out;
  float *lse;
  int q_tma;          // 1: Q tiles arrive by TMA (G divides the region's rows), else plain loads
  int32_t *status;
  // KV split (S > 1) through the workspace: one slot per CTA, [slot_rows][DH]
  // fp32 O rows then [slot_rows] (m, l) pairs, the slots of a (b, g,
  // M-group) consecutive.
  float *part;
  int slot_rows;
};

// QR: query rows held per M-tile region.  128 normally; 64 when a group
// has at most 64 rows (node, grouped head): the 128-row MMAs then read
// rows 64-127 of each region from the neighbouring shared memory, and those
// rows' results are never written out (rows are independent in S = Q K^T
// and P.V), which frees shared memory for a third stage.
template <int DH, int MT, int NK, int STAGES, int QR = 128>
struct TcShape {
  static constexpr int kRegions = DH / 64;                   // 128-byte swizzle atoms per row
  static constexpr int kQRegionBytes = QR * 128;             // QR rows x 64 columns
  static constexpr int kQBytes = MT * kRegions * kQRegionBytes;
  static constexpr int kTileBytes = kRegions * NK * 128;     // one K (or V) tile
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kBarOff = kQBytes + STAGES * kStageBytes;
  static constexpr int kNumBars = 2 * STAGES + 4 * MT + 2;
  static constexpr int kBarBytes = kNumBars * 8 + 16;
  // QR = 128: buffers at the first 1 KB boundary, barriers after them.
  // QR = 64: the barriers sit in the gap before the 1 KB-aligned buffers
  // when it holds them, else after the buffers; with a 16-byte aligned base
  // either way ends within kBarOff + max(1008, 2 kBarBytes - 16) bytes.
  static constexpr int kSmem = QR == 128 ? kBarOff + kBarBytes + 1024
                                         : kBarOff + (1008 > 2 * kBarBytes - 16 ? 1008 : 2 * kBarBytes - 16);
  static_assert(QR == 128 || (QR == 64 && MT == 1), "64-row regions with one M-tile only");
  static constexpr int kThreads = MT * 128 + 64;
  static constexpr int kColS = 0;                            // S_t at t*NK
  static constexpr int kColP = MT * NK;                      // P_t at kColP + t*NK/2
  static constexpr int kColO = MT * NK + MT * NK / 2;        // O_t at kColO + t*DH
  static constexpr int kCols = kColO + MT * DH;
  static constexpr int kTmemCols = kCols <= 128 ? 128 : (kCols <= 256 ? 256 : 512);
  static_assert(kCols <= 512, "tensor memory budget");
  // split merge: fp32 O rows in the stage buffers, (m, l) in Q's
  static_assert(MT * 128 * DH * 4 <= STAGES * kStageBytes, "partial O fits the stage buffers");
  static_assert(MT * 128 * 8 <= kQBytes, "(m, l) fit the Q buffer");
};

// Most KV splits of one (sequence, KV head, M-group): one cluster of CTAs.
constexpr int kMaxClusterSplits = 8;

// MERGE: 0 the grid does not split the KV range (the merge code is compiled
// out); otherwise every CTA leaves its partial results in its workspace slot
// and 1 the S splits of an item (one cluster) merge after a cluster barrier,
// 2 tree_attn_merge_kernel merges them.
template <int DH, int MT, int NK, int STAGES, int MERGE, int QR>
__global__ void __launch_bounds__(MT * 128 + 64, MT == 1 ? 2 : 1)
    tree_attn_tc_kernel(const __grid_constant__ CUtensorMap kc_map, const __grid_constant__ CUtensorMap vc_map,
                        const __grid_constant__ CUtensorMap kt_map, const __grid_constant__ CUtensorMap vt_map,
                        const __grid_constant__ CUtensorMap q_map, TcArgs a) {
  using Sh = TcShape<DH, MT, NK, STAGES, QR>;
  constexpr bool SPLIT = MERGE != 0;
  constexpr bool kCluster = MERGE == 1;  // the splits merge in this kernel
  constexpr int NH = NK / 64;  // 64-key halves of a tile
  extern __shared__ unsigned char raw_smem[];
  const uintptr_t raw = reinterpret_cast<uintptr_t>(raw_smem);
  unsigned char *sm = reinterpret_cast<unsigned char *>((raw + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char *sQ = sm;
  unsigned char *sKV = sm + Sh::kQBytes;
  uint64_t *bars;
  if constexpr (QR == 128) {
    bars = reinterpret_cast<uint64_t *>(sm + Sh::kBarOff);
  } else {
    bars = reinterpret_cast<uint64_t *>(reinterpret_cast<uintptr_t>(sm) - raw >= static_cast<uintptr_t>(Sh::kBarBytes)
                                            ? raw_smem
                                            : sm + Sh::kBarOff);
  }
  uint64_t *kv_full = bars;
  uint64_t *kv_empty = bars + STAGES;
  uint64_t *s_full = bars + 2 * STAGES;
  uint64_t *s_free = s_full + MT;
  uint64_t *p_full = s_free + MT;
  uint64_t *o_done = p_full + MT;
  uint64_t *teardown = o_done + MT;
  uint64_t *q_full = teardown + 1;  // the Q tiles (TMA)
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + Sh::kNumBars);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, mg = blockIdx.y;
  const int bg = blockIdx.z, b = bg / a.Hkv, g = bg % a.Hkv;
  const int n = a.n;
  const int producer_warp = MT * 4, mma_warp = MT * 4 + 1;

  if (tid == 0) prefetch_l2(a.kv_len + b);  // its load below then waits on L2, not DRAM
  pdl_wait();  // inputs of this step (kv_len, queries, tree K/V, mask) come from earlier kernels
  const int L = min(max(a.kv_len[b], 0), a.Lmax);
  const int n_ptiles = (L + NK - 1) / NK;
  const int tps = (n_ptiles + a.S - 1) / a.S;
  const int p0 = min(n_ptiles, split * tps), p1 = min(n_ptiles, p0 + tps);
  const int np = p1 - p0;
  const int ntt = (split == a.S - 1) ? (n + NK - 1) / NK : 0;
  const int T = np + ntt;  // key tiles of this CTA
  // ---- Q tiles -> shared memory ---------------------------------------------
  // By TMA when the group size divides 128: a box of (64 columns, G heads,
  // 128/G nodes) lands as 128 rows in (node, grouped head) order, the M-tile
  // row order; rows past the batch are zero-filled, rows past this
  // sequence's last node hold the next sequence's queries (their outputs
  // are never written).  Otherwise plain loads with zero rows.
  const int rows_total = n * a.G;
  for (int idx = tid; !a.q_tma && idx < MT * QR * (DH / 8); idx += Sh::kThreads) {
    const int t = idx / (QR * (DH / 8));
    const int rem = idx % (QR * (DH / 8));
    const int r = rem / (DH / 8), c = rem % (DH / 8);
    const int rho = (mg * MT + t) * 128 + r;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (rho < rows_total) {
      const int i = rho / a.G, hh = rho % a.G;
      const __nv_bfloat16 *src = a.q + ((static_cast<int64_t>(b) * n + i) * a.Hq + g * a.G + hh) * DH;
      v = *reinterpret_cast<const uint4 *>(src + c * 8);
    }
    *reinterpret_cast<uint4 *>(sQ + (t * Sh::kRegions + c / 8) * Sh::kQRegionBytes + sw128_offset(r, c % 8)) = v;
  }
  fence_async_smem();
  if (tid == 0) {
    for (int q = 0; q < STAGES; ++q) {
      mbar_init(&kv_full[q], 1);
      mbar_init(&kv_empty[q], 1);
    }
    for (int t = 0; t < MT; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&s_free[t], 4);
      mbar_init(&p_full[t], 4);
      mbar_init(&o_done[t], 1);
    }
    mbar_init(teardown, 1);
    mbar_init(q_full, 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == mma_warp) {
    tmem_alloc(tmem_slot, Sh::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  int issued = 0;  // producer: tiles issued
  // softmax threads with S > 1: this row's final (m, l), kept for the merge
  bool part_have = false;
  float part_m = -INFINITY, part_l = 0.f;

  if (warp == producer_warp) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      if (a.q_tma) {
        mbar_arrive_expect_tx(q_full, MT * Sh::kRegions * Sh::kQRegionBytes);
        for (int t = 0; t < MT; ++t)
#pragma unroll
          for (int r = 0; r < Sh::kRegions; ++r)
            tma_load_3d(sQ + (t * Sh::kRegions + r) * Sh::kQRegionBytes, &q_map, r * 64, g * a.G,
                        b * n + (mg * MT + t) * (128 / a.G), q_full);
      }
      prefetch_tmap(&kc_map);
      prefetch_tmap(&vc_map);
      prefetch_tmap(&kt_map);
      prefetch_tmap(&vt_map);
    }
    for (int j = 0; j < T; ++j) {
      const int st = j % STAGES, use = j / STAGES;
      if (use >= 1 && !warp_wait(&kv_empty[st], (use - 1) & 1, abort_flag)) break;
      unsigned char *kst = sKV + st * Sh::kStageBytes;
      unsigned char *vst = kst + Sh::kTileBytes;
      const bool prefix = j < np;
      const int key0 = prefix ? (p0 + j) * NK : (j - np) * NK;
      const int valid = prefix ? min(NK, L - key0) : NK;
      if (!prefix || valid == NK) {
        if (lane == 0) {
          mbar_arrive_expect_tx(&kv_full[st], Sh::kStageBytes);
          if (prefix && a.block_table) {
            // one box per page-sized piece of the tile, each at its page's row
            for (int s0 = 0; s0 < NK; s0 += a.page_box) {
              const int key = key0 + s0;
              int page = a.block_table[static_cast<int64_t>(b) * a.max_pages + key / a.page_size];
              if (page < 0 || page >= a.num_pages) {  // outside the pool: report, read page 0
                report(a.status, EAGLE_ERR_INVALID);
                page = 0;
              }
              const int row = (page * a.Hkv + g) * a.page_size + key % a.page_size;
#pragma unroll
              for (int r = 0; r < Sh::kRegions; ++r) {
                tma_load_2d(kst + r * NK * 128 + s0 * 128, &kc_map, r * 64, row, &kv_full[st]);
                tma_load_2d(vst + r * NK * 128 + s0 * 128, &vc_map, r * 64, row, &kv_full[st]);
              }
            }
          } else {
            const CUtensorMap *km = prefix ? &kc_map : &kt_map;
            const CUtensorMap *vm = prefix ? &vc_map : &vt_map;
            const int row0 = prefix ? bg * a.Lmax + key0 : bg * n + key0;
#pragma unroll
            for (int r = 0; r < Sh::kRegions; ++r) {
              tma_load_2d(kst + r * NK * 128, km, r * 64, row0, &kv_full[st]);
              tma_load_2d(vst + r * NK * 128, vm, r * 64, row0, &kv_full[st]);
            }
          }
        }
      } else {
        // ragged last prefix tile: rows >= valid are zero (cache memory past
        // kv_len is never read)
        for (int idx = lane; idx < NK * (DH / 8); idx += 32) {
          const int r = idx / (DH / 8), c = idx % (DH / 8);
          uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
          if (r < valid) {
            int64_t row;
            if (a.block_table) {
              const int key = key0 + r;
              const int page = a.block_table[static_cast<int64_t>(b) * a.max_pages + key / a.page_size];
              row = (page >= 0 && page < a.num_pages)
                        ? (static_cast<int64_t>(page) * a.Hkv + g) * a.page_size + key % a.page_size
                        : -1;
              if (row < 0) report(a.status, EAGLE_ERR_INVALID);
            } else {
              row = static_cast<int64_t>(bg) * a.Lmax + key0 + r;
            }
            if (row >= 0) {
              kv = *reinterpret_cast<const uint4 *>(a.k_cache + row * DH + c * 8);
              vv = *reinterpret_cast<const uint4 *>(a.v_cache + row * DH + c * 8);
            }
          }
          const uint32_t off = (c / 8) * (NK * 128) + sw128_offset(r, c % 8);
          *reinterpret_cast<uint4 *>(kst + off) = kv;
          *reinterpret_cast<uint4 *>(vst + off) = vv;
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&kv_full[st]);
      }
      issued = j + 1;
    }
    // an empty split's Q copy (no MMA waits for it) lands before the
    // teardown barrier, so nothing written to the Q buffer after it races it
    if (a.q_tma && T == 0 && lane == 0) {
      volatile int never = 0;
      mbar_wait(q_full, 0, &never, 100000000ull);
    }
  } else if (warp == mma_warp) {
    // --------------------------------------------------------------------- MMA
    // Lane 0 issues every MMA and commit.  Shared-memory descriptors advance
    // by constants from per-stage bases: the start-address field holds the
    // byte address / 16 and never carries (shared memory is below 256 KB).
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(128, NK, false);
      constexpr uint32_t id_o = idesc_bf16(128, DH, true);
      const uint64_t q_desc0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t k_desc0 = sdesc_sw128(smem_u32(sKV), 16, 1024);
      const uint64_t v_desc0 = sdesc_sw128(smem_u32(sKV) + Sh::kTileBytes, NK * 128, 1024);
      auto issue_s = [&](int j, int t) {
        const uint64_t kd = k_desc0 + static_cast<uint64_t>((j % STAGES) * (Sh::kStageBytes >> 4));
        const uint64_t qd = q_desc0 + static_cast<uint64_t>(t * Sh::kRegions * (Sh::kQRegionBytes >> 4));
#pragma unroll
        for (int s = 0; s < DH / 16; ++s) {
          const uint64_t qoff = static_cast<uint64_t>(((s / 4) * Sh::kQRegionBytes + (s % 4) * 32) >> 4);
          const uint64_t koff = static_cast<uint64_t>(((s / 4) * (NK * 128) + (s % 4) * 32) >> 4);
          mma_bf16_ss(tmem + Sh::kColS + t * NK, qd + qoff, kd + koff, id_s, s > 0);
        }
        mma_commit(&s_full[t]);
      };
      bool ok = T == 0 || ((!a.q_tma || mbar_wait(q_full, 0, abort_flag)) && mbar_wait(&kv_full[0], 0, abort_flag));
      if (ok && T > 0) {
        tc_fence_after();
        for (int t = 0; t < MT; ++t) issue_s(0, t);
      }
      // per tile j: S(j+1) of every M-tile as soon as its softmax has taken
      // S(j) into registers, then P(j).V of every M-tile once P(j) is in
      // tensor memory
      for (int j = 0; j < T && ok; ++j) {
        const int st = j % STAGES;
        const bool next = j + 1 < T;
        if (next && !mbar_wait(&kv_full[(j + 1) % STAGES], ((j + 1) / STAGES) & 1, abort_flag)) break;
        const uint64_t vd = v_desc0 + static_cast<uint64_t>(st * (Sh::kStageBytes >> 4));
        for (int t = 0; t < MT && ok && next; ++t) {
          if (!mbar_wait(&s_free[t], j & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          issue_s(j + 1, t);
        }
        for (int t = 0; t < MT && ok; ++t) {
          if (!mbar_wait(&p_full[t], j & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t pcol = tmem + Sh::kColP + t * (NK / 2);
#pragma unroll
          for (int s = 0; s < NK / 16; ++s)
            mma_bf16_ts(tmem + Sh::kColO + t * DH, pcol + s * 8, vd + static_cast<uint64_t>(s * (2048 >> 4)), id_o,
                        (j > 0 || s > 0));
          mma_commit(&o_done[t]);
        }
        if (ok) mma_commit(&kv_empty[st]);
      }
    }
  } else {
    // ----------------------------------------------------------------- softmax
    const int t = warp >> 2, qtr = warp & 3;
    const int r = qtr * 32 + lane;
    const int rho = (mg * MT + t) * 128 + r;
    const bool row_ok = rho < rows_total;
    const bool warp_live = (mg * MT + t) * 128 + qtr * 32 < rows_total;  // warp-uniform
    const int i = row_ok ? rho / a.G : 0;
    const int hh = row_ok ? rho % a.G : 0;
    const uint32_t lane_base = static_cast<uint32_t>(qtr * 32) << 16;
    const uint32_t tS = tmem + lane_base + Sh::kColS + t * NK;
    const uint32_t tP = tmem + lane_base + Sh::kColP + t * (NK / 2);
    const uint32_t tO = tmem + lane_base + Sh::kColO + t * DH;
    const uint64_t *mrow = a.mask + (static_cast<int64_t>(b) * n + i) * a.W;
    // m is the exponent base of this row's P and O (scaled, base-2 units).  It
    // is raised only when the row maximum exceeds it by more than 8, so P
    // stays below 2^8 and O is rescaled rarely.
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < T; ++j) {
      if (!warp_wait(&s_full[t], j & 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
      // key validity per 64-key half: prefix positions below kv_len; tree
      // nodes that are ancestors-or-self of this row's node
      const bool prefix = j < np;
      uint64_t keep[NH];
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        if (prefix) {
          const int valid = min(NK, L - (p0 + j) * NK) - 64 * h;
          keep[h] = valid >= 64 ? ~0ull : (valid <= 0 ? 0ull : ((1ull << valid) - 1ull));
        } else {
          const int w = (j - np) * NH + h;
          keep[h] = (row_ok && w < a.W) ? mrow[w] : 0ull;
        }
      }
      bool dense = true;
#pragma unroll
      for (int h = 0; h < NH; ++h) dense = dense && keep[h] == ~0ull;
      dense = __all_sync(0xffffffffu, dense);
      auto half_max = [](const float (&sv)[64]) {
        float mx[4] = {sv[0], sv[1], sv[2], sv[3]};
#pragma unroll
        for (int c = 4; c < 64; c += 8) {
          mx[0] = fmax3(mx[0], sv[c], sv[c + 4]);
          mx[1] = fmax3(mx[1], sv[c + 1], sv[c + 5]);
          mx[2] = fmax3(mx[2], sv[c + 2], sv[c + 6]);
          mx[3] = fmax3(mx[3], sv[c + 3], sv[c + 7]);
        }
        return fmax3(fmax3(mx[0], mx[1], mx[2]), mx[3], -INFINITY);
      };
      // S into registers in one read; S's tensor memory is then released, so
      // the next tile's S = Q K^T runs while this tile's exponents are taken.
      // A warp whose 32 rows all lie past the last (node, head) row only
      // signals (its rows' results are never written out).
      float sv[NH][64];
      if (warp_live) {
#pragma unroll
        for (int h = 0; h < NH; ++h) tmem_ld64(tS + 64 * h, sv[h]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[t]);  // S has been read
      float tmax = -INFINITY;
      if (warp_live) {
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          if (!dense) {  // masked keys at -inf
#pragma unroll
            for (int c = 0; c < 64; ++c) sv[h][c] = ((keep[h] >> c) & 1ull) ? sv[h][c] : -INFINITY;
          }
          tmax = fmaxf(tmax, half_max(sv[h]));
        }
      }
      tmax *= a.scale_log2;  // scale > 0
      const bool raise = tmax > m + 8.f;
      const float base = raise ? tmax : m;
      const float alpha = raise ? ex2_approx(m - tmax) : 1.f;  // m = -inf gives 0
      m = base;
      if (j > 0) {  // P.V of the previous tile is done: P is free, O is final for it
        if (!warp_wait(&o_done[t], (j - 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
      }
      // P = exp2(s*scale - base), packed bf16 pairs into tensor memory (a row
      // with no valid key yet has base -inf and only -inf scores: any finite
      // exponent base then gives 0)
      const float nb = base > -INFINITY ? -base : 0.f;
      const uint64_t sc2 = f2_pack(a.scale_log2, a.scale_log2), nb2 = f2_pack(nb, nb);
      uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = acc0;
      // packed P in 16-column pieces, so only one piece's registers are live
      // next to the scores
      auto exp_half = [&](int h, const float (&sv)[64]) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          float pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int cc = 16 * q + c;
            float t0, t1;
            f2_unpack(f2_fma(f2_pack(sv[2 * cc], sv[2 * cc + 1]), sc2, nb2), t0, t1);
            const float p0v = ex2_approx(t0), p1v = ex2_approx(t1);
            if (c & 1) acc1 = f2_add(acc1, f2_pack(p0v, p1v));
            else acc0 = f2_add(acc0, f2_pack(p0v, p1v));
            __nv_bfloat162 h2 = __floats2bfloat162_rn(p0v, p1v);
            pk[c] = *reinterpret_cast<const float *>(&h2);
          }
          tmem_st16_async(tP + 32 * h + 16 * q, pk);
        }
      };
      if (warp_live) {
#pragma unroll
        for (int h = 0; h < NH; ++h) exp_half(h, sv[h]);
        tmem_wait_st();
      }
      float q0, q1, q2, q3;
      f2_unpack(acc0, q0, q1);
      f2_unpack(acc1, q2, q3);
      l = l * alpha + ((q0 + q1) + (q2 + q3));
      if (warp_live && j > 0 && __any_sync(0xffffffffu, raise)) {
#pragma unroll
        for (int c0 = 0; c0 < DH; c0 += 32) {
          float o[32];
          tmem_ld32(tO + c0, o);
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] *= alpha;
          tmem_st32(tO + c0, o);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[t]);
    }
    if (ok && T > 0 && !warp_wait(&o_done[t], (T - 1) & 1, abort_flag)) ok = false;
    tc_fence_after();
    // tcgen05.ld is warp-collective (.sync.aligned): every lane executes it,
    // rows past the last node only skip the global writes
    const int h = g * a.G + hh;
    const int64_t orow = (static_cast<int64_t>(b) * n + i) * a.Hq + h;
    const bool have = ok && T > 0;
    const float inv = (have && l > 0.f) ? 1.f / l : 0.f;
    if constexpr (SPLIT) {
      // split: (m, l) wait for the cluster merge; O stays in tensor memory
      // until every MMA of the CTA is done (the teardown barrier)
      part_have = have;
      part_m = m;
      part_l = l;
    } else {
#pragma unroll
      for (int c0 = 0; c0 < DH; c0 += 32) {
        float o[32];
        if (have) {
          tmem_ld32(tO + c0, o);
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = 0.f;
        }
        if (!row_ok) continue;
        __nv_bfloat162 hv[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) hv[e] = __floats2bfloat162_rn(o[2 * e] * inv, o[2 * e + 1] * inv);
        uint4 *dst = reinterpret_cast<uint4 *>(a.out + orow * DH + c0);
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[e] = reinterpret_cast<const uint4 *>(hv)[e];
      }
      if (row_ok && a.lse) a.lse[orow] = have ? (m + __log2f(l)) * kLn2 : -INFINITY;
    }
  }

  pdl_trigger();
  // ---- teardown --------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (*abort_flag) {
    if (tid == 0) report(a.status, EAGLE_ERR_TIMEOUT);
    volatile int never = 0;
    if (warp == mma_warp && lane == 0) {
      // every MMA issued so far completes before tensor memory is released
      mma_commit(teardown);
      mbar_wait(teardown, 0, &never, 100000000ull);
    }
    if (warp == producer_warp && lane == 0) {
      // copies still in flight complete before shared memory is released
      if (a.q_tma && T > 0) mbar_wait(q_full, 0, &never, 100000000ull);
      for (int j = max(0, issued - STAGES); j < issued; ++j)
        mbar_wait(&kv_full[j % STAGES], (j / STAGES) & 1, &never, 100000000ull);
    }
    __syncthreads();
  }
  if (SPLIT && warp < MT * 4) {
    // this CTA's unnormalised O rows (fp32) into the stage buffers and its
    // (m, l) pairs into the Q buffer: every MMA and copy has completed.  Row
    // r's 16-byte chunk c sits at chunk c ^ (r & 7) of the row, so the 32
    // rows of a warp store to distinct banks.
    const int t = warp >> 2, qtr = warp & 3, rl = t * 128 + qtr * 32 + lane;
    const uint32_t tO = tmem + (static_cast<uint32_t>(qtr * 32) << 16) + Sh::kColO + t * DH;
    const bool have = part_have && !*abort_flag;
    float4 *prow = reinterpret_cast<float4 *>(sKV) + rl * (DH / 4);
#pragma unroll
    for (int c0 = 0; c0 < DH; c0 += 32) {
      float o[32];
      if (__all_sync(0xffffffffu, have)) {
        tmem_ld32(tO + c0, o);
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) o[c] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e)
        prow[(c0 / 4 + e) ^ (rl & 7)] = make_float4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
    }
    reinterpret_cast<float2 *>(sQ)[rl] = have ? make_float2(part_m * kLn2, part_l) : make_float2(-INFINITY, 0.f);
  }
  const int r0 = mg * MT * 128, nr = max(0, min(rows_total, r0 + MT * 128) - r0);
  if constexpr (SPLIT) {
    tc_fence_before();
    __syncthreads();
    {
      // this CTA's rows [0, nr) into its workspace slot, one 16-byte chunk
      // per thread and store, a row's chunks contiguous (coalesced)
      constexpr int NV = DH / 4;
      const int64_t cl = static_cast<int64_t>(bg) * gridDim.y + mg;
      float *slot = a.part + (cl * a.S + split) * static_cast<int64_t>(a.slot_rows) * (DH + 2);
      for (int idx = tid; idx < nr * NV; idx += Sh::kThreads) {
        const int r = idx / NV, c = idx % NV;
        reinterpret_cast<float4 *>(slot)[idx] = reinterpret_cast<const float4 *>(sKV)[r * NV + (c ^ (r & 7))];
      }
      for (int r = tid; r < nr; r += Sh::kThreads)
        reinterpret_cast<float2 *>(slot + static_cast<int64_t>(a.slot_rows) * DH)[r] =
            reinterpret_cast<const float2 *>(sQ)[r];
    }
  }
  if (warp == mma_warp) tmem_dealloc(tmem, Sh::kTmemCols);

  // ---- split merge across the cluster ----------------------------------------
  // One-wave split launches (MERGE = 1): the S splits of this (b, g,
  // M-group) are one cluster.  Each CTA has put its unnormalised fp32 O rows
  // and (m, l) into its workspace slot; after one cluster barrier (release,
  // acquire) it merges rows [rank*per, (rank+1)*per) of the group from all S
  // slots, read from L2 skipping L1: out = sum_s w_s O_s with
  // w_s = exp(m_s - M) / L, M = max_s m_s, L = sum_s exp(m_s - M) l_s.
  // Global memory outlives every CTA, so no second round is needed.
  if constexpr (kCluster) {
    cluster_arrive_release();
    cluster_wait();
    const uint32_t rank = cluster_ctarank();
    const bool cok = *abort_flag == 0;
    const int per = (nr + a.S - 1) / a.S;
    const int q0 = min(nr, static_cast<int>(rank) * per), q1 = min(nr, q0 + per);
    const int64_t slot_floats = static_cast<int64_t>(a.slot_rows) * (DH + 2);
    const float *slots = a.part + (static_cast<int64_t>(bg) * gridDim.y + mg) * a.S * slot_floats;
    // four output columns per item, two items per thread at a time.  The NV
    // items of a row sit in NV consecutive lanes: lane c of the row loads
    // split c's (m, l) and the row's lanes share them by shuffles; every
    // item loads its S partial chunks, all in flight together.
    constexpr int NV = DH / 4;
    static_assert(NV == 16 || NV == 32, "a row's items fill half or all of a warp");
    constexpr int kItems = 2;
    const int n_items = (q1 - q0) * NV;  // a multiple of NV: a row's lanes agree on validity
    for (int base = tid; cok && base - lane < n_items; base += kItems * Sh::kThreads) {
      float2 mine[kItems];
      float4 po[kItems][kMaxClusterSplits];
#pragma unroll
      for (int u = 0; u < kItems; ++u) {
        const int item = base + u * Sh::kThreads;
        const int rr = q0 + item / NV, c = item % NV;
        const bool valid = item < n_items;
        mine[u] = (valid && c < a.S)
                      ? __ldcg(reinterpret_cast<const float2 *>(slots + c * slot_floats + static_cast<int64_t>(a.slot_rows) * DH) + rr)
                      : make_float2(-INFINITY, 0.f);
#pragma unroll
        for (int sp = 0; sp < kMaxClusterSplits; ++sp)
          po[u][sp] = (valid && sp < a.S) ? __ldcg(reinterpret_cast<const float4 *>(slots + sp * slot_floats) + rr * NV + c)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kItems; ++u) {
        const int item = base + u * Sh::kThreads;
        float2 ml[kMaxClusterSplits];
#pragma unroll
        for (int sp = 0; sp < kMaxClusterSplits; ++sp) {
          ml[sp].x = __shfl_sync(0xffffffffu, mine[u].x, sp, NV);
          ml[sp].y = __shfl_sync(0xffffffffu, mine[u].y, sp, NV);
          if (sp >= a.S) ml[sp] = make_float2(-INFINITY, 0.f);
        }
        if (item >= n_items) continue;
        const int rr = q0 + item / NV, c = item % NV;
        float M = -INFINITY;
#pragma unroll
        for (int sp = 0; sp < kMaxClusterSplits; ++sp) M = fmaxf(M, ml[sp].x);
        float Ls = 0.f;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int sp = 0; sp < kMaxClusterSplits; ++sp) {
          const float x = ml[sp].x;
          const float wgt = (M > -INFINITY && x > -INFINITY) ? ex2_approx((x - M) * kLog2e) : 0.f;
          Ls = fmaf(wgt, ml[sp].y, Ls);
          o.x = fmaf(wgt, po[u][sp].x, o.x); o.y = fmaf(wgt, po[u][sp].y, o.y);
          o.z = fmaf(wgt, po[u][sp].z, o.z); o.w = fmaf(wgt, po[u][sp].w, o.w);
        }
        const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
        const int rho = r0 + rr, i = rho / a.G, h = g * a.G + rho % a.G;
        const int64_t orow = (static_cast<int64_t>(b) * n + i) * a.Hq + h;
        __nv_bfloat162 lo = __floats2bfloat162_rn(o.x * inv, o.y * inv);
        __nv_bfloat162 hi = __floats2bfloat162_rn(o.z * inv, o.w * inv);
        uint2 packed;
        packed.x = *reinterpret_cast<const uint32_t *>(&lo);
        packed.y = *reinterpret_cast<const uint32_t *>(&hi);
        reinterpret_cast<uint2 *>(a.out + orow * DH)[c] = packed;
        if (c == 0 && a.lse) a.lse[orow] = Ls > 0.f ? M + __logf(Ls) : -INFINITY;
      }
    }
  }
}

// The merge of a split launch of several waves (MERGE = 2): one thread per (row, 4 output columns) of a
// (b, g, M-group), out = sum_s w_s O_s with w_s = exp(m_s - M) / L,
// M = max_s m_s, L = sum_s exp(m_s - M) l_s, reading the S slots from L2.
template <int DH>
__global__ void __launch_bounds__(256) tree_attn_merge_kernel(TcArgs a, int MT) {
  constexpr int NV = DH / 4;
  const int mg = blockIdx.y, bg = blockIdx.z, b = bg / a.Hkv, g = bg % a.Hkv;
  const int rows_total = a.n * a.G;
  const int r0 = mg * MT * 128, nr = max(0, min(rows_total, r0 + MT * 128) - r0);
  const int item = blockIdx.x * blockDim.x + threadIdx.x;
  pdl_wait();  // the partial results come from the attention kernel
  if (item >= nr * NV) return;
  const int rr = item / NV, c = item % NV;
  const int64_t slot_floats = static_cast<int64_t>(a.slot_rows) * (DH + 2);
  const float *slots = a.part + (static_cast<int64_t>(bg) * gridDim.y + mg) * a.S * slot_floats;
  float M = -INFINITY;
  for (int sp = 0; sp < a.S; ++sp)
    M = fmaxf(M, __ldcg(reinterpret_cast<const float2 *>(slots + sp * slot_floats + static_cast<int64_t>(a.slot_rows) * DH) + rr).x);
  float Ls = 0.f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int sp = 0; sp < a.S; ++sp) {
    const float2 ml = __ldcg(reinterpret_cast<const float2 *>(slots + sp * slot_floats + static_cast<int64_t>(a.slot_rows) * DH) + rr);
    const float4 po = __ldcg(reinterpret_cast<const float4 *>(slots + sp * slot_floats) + rr * NV + c);
    const float wgt = (M > -INFINITY && ml.x > -INFINITY) ? ex2_approx((ml.x - M) * kLog2e) : 0.f;
    Ls = fmaf(wgt, ml.y, Ls);
    o.x = fmaf(wgt, po.x, o.x); o.y = fmaf(wgt, po.y, o.y);
    o.z = fmaf(wgt, po.z, o.z); o.w = fmaf(wgt, po.w, o.w);
  }
  const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
  const int rho = r0 + rr, i = rho / a.G, h = g * a.G + rho % a.G;
  const int64_t orow = (static_cast<int64_t>(b) * a.n + i) * a.Hq + h;
  __nv_bfloat162 lo = __floats2bfloat162_rn(o.x * inv, o.y * inv);
  __nv_bfloat162 hi = __floats2bfloat162_rn(o.z * inv, o.w * inv);
  uint2 packed;
  packed.x = *reinterpret_cast<const uint32_t *>(&lo);
  packed.y = *reinterpret_cast<const uint32_t *>(&hi);
  reinterpret_cast<uint2 *>(a.out + orow * DH)[c] = packed;
  if (c == 0 && a.lse) a.lse[orow] = Ls > 0.f ? M + __logf(Ls) : -INFINITY;
}

// ---- host side ---------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2D bf16 tensor [rows, dh] viewed in boxes of 64 columns x `box_rows` rows
// with 128-byte swizzle.
static bool make_kv_map(CUtensorMap *map, const void *base, int64_t rows, int dh, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(dh), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(dh) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Q [B*n, Hq, dh] bf16 viewed as a 3D tensor with boxes of 64 columns x G
// heads x box_rows/G nodes (128-byte swizzle): one box is one M-tile region.
static bool make_q_map(CUtensorMap *map, const void *base, int64_t rows, int Hq, int dh, int G, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(dh), static_cast<cuuint64_t>(Hq), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(dh) * 2, static_cast<cuuint64_t>(Hq) * dh * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(box_rows / G)};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct TcPlan {
  int MT, NK, mgroups, S, ctas_per_sm, num_sms;
};

// Launch plan: M-tiles per CTA, key-tile width, and the KV split S chosen to
// minimise (waves of CTAs) x (key tiles per CTA + the cost of merging a
// split's partial results, in key-tile units).
static TcPlan tc_plan(int B, int n, int Hq, int Hkv, int dh, int Lmax, int num_sms) {
  TcPlan p;
  p.num_sms = num_sms;
  const int G = Hq / Hkv;
  const int tiles = (n * G + 127) / 128;
  p.MT = tiles <= 1 ? 1 : 2;
  p.NK = dh == 64 ? 128 : 64;
  p.mgroups = (tiles + p.MT - 1) / p.MT;
  p.ctas_per_sm = p.MT == 1 ? 2 : 1;
  const int64_t base = static_cast<int64_t>(B) * Hkv * p.mgroups;
  const int64_t slots = static_cast<int64_t>(num_sms) * p.ctas_per_sm;
  const int64_t ptiles = (Lmax + p.NK - 1) / p.NK;
  const double split_cost = static_cast<double>(G) * n * 64.0 / p.NK / 32.0 / p.mgroups;
  int best = 1;
  double best_cost = 1e30;
  for (int S = 1; S <= kMaxClusterSplits && S <= ptiles; ++S) {
    const int64_t waves = (base * S + slots - 1) / slots;
    const double per_cta = static_cast<double>((ptiles + S - 1) / S) + (S > 1 ? split_cost : 0.0);
    const double cost = waves * per_cta;
    if (cost < best_cost * 0.97) {  // prefer fewer splits unless clearly better
      best_cost = cost;
      best = S;
    }
  }
  p.S = best;
  return p;
}

// Rows of a split's workspace slot: the most (node, grouped head) rows of an
// M-group, rounded up to 8.
static int tc_slot_rows(const TcPlan &p, int n, int G) {
  const int rows = (n * G + 7) / 8 * 8;
  return rows < p.MT * 128 ? rows : p.MT * 128;
}

// A split launch passes its partial results through the workspace, one slot
// of fp32 O rows and (m, l) pairs per CTA, read back from L2.  When its CTAs
// are all resident at once (one wave) the splits of an item are one cluster
// and merge after a cluster barrier; otherwise every CTA leaves as soon as
// its slot is written (no cluster co-scheduling, no waiting on peers) and a
// second kernel merges.
static bool tc_one_wave(const TcPlan &p, int B, int Hkv, int num_sms) {
  return static_cast<int64_t>(B) * Hkv * p.mgroups * p.S <= static_cast<int64_t>(num_sms) * p.ctas_per_sm;
}

// Kernels one launch runs: the attention, plus the merge for a split
// launch of several waves.
int attn_tc_kernel_count(int B, int n, int Hq, int Hkv, int dh, int Lmax, int num_sms) {
  const TcPlan p = tc_plan(B, n, Hq, Hkv, dh, Lmax, num_sms);
  return p.S > 1 && !tc_one_wave(p, B, Hkv, num_sms) ? 2 : 1;
}

size_t attn_tc_workspace_bytes(int B, int n, int Hq, int Hkv, int dh, int Lmax, int num_sms) {
  const TcPlan p = tc_plan(B, n, Hq, Hkv, dh, Lmax, num_sms);
  if (p.S <= 1) return 0;
  return static_cast<size_t>(B) * Hkv * p.mgroups * p.S * tc_slot_rows(p, n, Hq / Hkv) * (dh + 2) * sizeof(float);
}

template <int DH, int MT, int NK, int STAGES, int MERGE, int QR>
static cudaError_t launch_tc_v(const CUtensorMap *maps, const TcArgs &a, const TcPlan &p, cudaStream_t st) {
  using Sh = TcShape<DH, MT, NK, STAGES, QR>;
  static_assert(Sh::kSmem <= 232448, "shared memory budget");
  // MT = 1 variants run two CTAs per SM (228 KB per SM, 1 KB reserved per CTA)
  static_assert(MT != 1 || 2 * (Sh::kSmem + 1024) <= 233472, "two CTAs per SM");
  static std::atomic<unsigned long long> configured{0};
  const cudaError_t e = set_smem_limit_once(tree_attn_tc_kernel<DH, MT, NK, STAGES, MERGE, QR>, Sh::kSmem, configured);
  if (e != cudaSuccess) return e;
  dim3 grid(p.S, p.mgroups, a.B * a.Hkv);
  if constexpr (MERGE == 2) {
    cudaError_t le = launch_chained(tree_attn_tc_kernel<DH, MT, NK, STAGES, MERGE, QR>, grid, dim3(Sh::kThreads),
                                    Sh::kSmem, st, maps[0], maps[1], maps[2], maps[3], maps[4], a);
    if (le != cudaSuccess) return le;
    const int rows = a.slot_rows;  // at least any M-group's rows
    const dim3 mgrid((rows * (DH / 4) + 255) / 256, p.mgroups, a.B * a.Hkv);
    return launch_chained(tree_attn_merge_kernel<DH>, mgrid, dim3(256), 0, st, a, MT);
  }
  // the S splits of one (b, g, M-group) form one cluster
  return launch_chained_cluster(tree_attn_tc_kernel<DH, MT, NK, STAGES, MERGE, QR>, grid, dim3(Sh::kThreads), Sh::kSmem,
                                st, p.S, maps[0], maps[1], maps[2], maps[3], maps[4], a);
}

template <int DH, int MT, int NK, int STAGES, int QR = 128>
static cudaError_t launch_tc_t(const CUtensorMap *maps, const TcArgs &a, const TcPlan &p, cudaStream_t st) {
  if (p.S <= 1) return launch_tc_v<DH, MT, NK, STAGES, 0, QR>(maps, a, p, st);
  return tc_one_wave(p, a.B, a.Hkv, p.num_sms) ? launch_tc_v<DH, MT, NK, STAGES, 1, QR>(maps, a, p, st)
                                              : launch_tc_v<DH, MT, NK, STAGES, 2, QR>(maps, a, p, st);
}

// Common launcher; block_table == nullptr is the contiguous cache, otherwise
// the page pools with Lmax = max_pages * page_size logical positions.
static cudaError_t launch_tc_common(const void *q, const void *k_cache, const void *v_cache, const int32_t *kv_len,
                                    const void *k_tree, const void *v_tree, const uint64_t *mask, int B, int n,
                                    int Hq, int Hkv, int dh, int Lmax, float scale, void *out, float *lse,
                                    void *ws, int32_t *status, int num_sms, cudaStream_t st,
                                    const int32_t *block_table, int max_pages, int page_size, int num_pages) {
  const TcPlan p = tc_plan(B, n, Hq, Hkv, dh, Lmax, num_sms);
  CUtensorMap maps[5];
  const int page_box = block_table ? min(page_size, p.NK) : p.NK;
  const int64_t cache_rows = block_table ? static_cast<int64_t>(num_pages) * Hkv * page_size
                                         : static_cast<int64_t>(B) * Hkv * Lmax;
  const int64_t tree_rows = static_cast<int64_t>(B) * Hkv * n;
  if (!make_kv_map(&maps[0], k_cache, cache_rows > 0 ? cache_rows : 1, dh, page_box) ||
      !make_kv_map(&maps[1], v_cache, cache_rows > 0 ? cache_rows : 1, dh, page_box) ||
      !make_kv_map(&maps[2], k_tree, tree_rows, dh, p.NK) || !make_kv_map(&maps[3], v_tree, tree_rows, dh, p.NK))
    return cudaErrorInvalidValue;
  const int G = Hq / Hkv;
  // at most 64 rows (node, grouped head) per group and dh = 128: 64-row Q
  // regions and a third stage
  const bool half_q = dh == 128 && n * G <= 64;
  const int q_rows = half_q ? 64 : 128;
  const bool q_tma = q_rows % G == 0 && make_q_map(&maps[4], q, static_cast<int64_t>(B) * n, Hq, dh, G, q_rows);
  if (!q_tma) maps[4] = maps[2];  // unused
  TcArgs a;
  a.q = reinterpret_cast<const __nv_bfloat16 *>(q);
  a.k_cache = reinterpret_cast<const __nv_bfloat16 *>(k_cache);
  a.v_cache = reinterpret_cast<const __nv_bfloat16 *>(v_cache);
  a.kv_len = kv_len;
  a.mask = mask;
  a.B = B; a.n = n; a.Hq = Hq; a.Hkv = Hkv; a.G = Hq / Hkv; a.Lmax = Lmax; a.S = p.S;
  a.W = (n + 63) / 64;
  a.block_table = block_table;
  a.max_pages = max_pages; a.page_size = page_size; a.page_box = page_box; a.num_pages = num_pages;
  a.scale_log2 = scale * kLog2e;
  a.out = reinterpret_cast<__nv_bfloat16 *>(out);
  a.lse = lse;
  a.q_tma = q_tma ? 1 : 0;
  a.status = status;
  a.part = p.S > 1 ? reinterpret_cast<float *>(ws) : nullptr;
  a.slot_rows = tc_slot_rows(p, n, G);
  if (p.S > 1 && !ws) return cudaErrorInvalidValue;
  cudaError_t e;
  // stages: as many as shared memory allows at the variant's CTAs per SM
  if (dh == 64) {
    e = p.MT == 1 ? launch_tc_t<64, 1, 128, 2>(maps, a, p, st) : launch_tc_t<64, 2, 128, 4>(maps, a, p, st);
  } else if (half_q) {
    e = launch_tc_t<128, 1, 64, 3, 64>(maps, a, p, st);
  } else {
    e = p.MT == 1 ? launch_tc_t<128, 1, 64, 2>(maps, a, p, st) : launch_tc_t<128, 2, 64, 4>(maps, a, p, st);
  }
  return e;
}

cudaError_t launch_tree_attn_tc(const void *q, const void *k_cache, const void *v_cache, const int32_t *kv_len,
                                const void *k_tree, const void *v_tree, const uint64_t *mask, int B, int n,
                                int Hq, int Hkv, int dh, int Lmax, float scale, void *out, float *lse, void *ws,
                                int32_t *status, int num_sms, cudaStream_t st) {
  return launch_tc_common(q, k_cache, v_cache, kv_len, k_tree, v_tree, mask, B, n, Hq, Hkv, dh, Lmax, scale, out,
                          lse, ws, status, num_sms, st, nullptr, 0, 0, 0);
}

cudaError_t launch_tree_attn_tc_paged(const void *q, const void *k_pages, const void *v_pages,
                                      const int32_t *block_table, int max_pages, int page_size, int num_pages,
                                      const int32_t *kv_len, const void *k_tree, const void *v_tree,
                                      const uint64_t *mask, int B, int n, int Hq, int Hkv, int dh, float scale,
                                      void *out, float *lse, void *ws, int32_t *status, int num_sms,
                                      cudaStream_t st) {
  return launch_tc_common(q, k_pages, v_pages, kv_len, k_tree, v_tree, mask, B, n, Hq, Hkv, dh,
                          max_pages * page_size, scale, out, lse, ws, status, num_sms, st, block_table, max_pages,
                          page_size, num_pages);
}

}  // namespace eagle
