// Stage 1: per-row softmax statistics and top-k of the draft logits.
//
// [EAGLE-2] section "ドラフトモデルのキャリブレーション": the confidence of a
// draft token is the probability the draft model assigns to it.  For every
// used row: M = max, Z = sum exp(x - M), the k largest logits (ties -> lower
// token id) and c = exp(x - M) / Z.
//
// One pass over HBM.  A row is split into S <= 8 parts, one CTA each; the
// parts of a row form one thread-block cluster.  Few rows (each part fits
// one segment per warp, and the parts of all rows fit three waves of two
// CTAs per SM) take 16-warp CTAs with 1024-token segments, held in
// registers (all 16-byte loads in flight at once); many rows take 8-warp
// CTAs, three per SM (or 4-warp CTAs, six per SM, when a warp would
// otherwise see fewer than eight segments), whose warps stream 1024-token
// segments through a three-stage ring in shared
// memory (asynchronous copies issued two segments ahead, so the loads stay
// in flight while a segment is being processed).  A warp visits each
// segment twice: lane maxima, then the sum of exp(x - segment max), folded
// into a running (max, sum).  Top-k selection works on unique 64-bit keys
// (logit order, then lower token id).  Each warp keeps its k best keys so
// far sorted in registers (lane i holds the i-th); a new key's place is the
// number of larger keys (one ballot) and the tail shifts down one lane.  The
// list's k-th key bounds the part from below, so values under the bound
// (shared block-wide as a maximum over the warps) are never looked at;
// before the list is full, the k-th largest lane maximum is the bound.  In
// the ring form the lanes also keep their running maxima in shared memory,
// and every eighth segment a warp raises the shared bound to the k-th
// largest of their group maxima (distinct elements, so a valid bound
// whenever read): the bound then reflects the whole block's progress
// rather than one warp's share of the row.  The warp lists
// merge block-wide: only keys at or above the block's bound are kept, and
// their ranks are counted.  With S > 1 every part pushes its k keys and
// (max, sum) into the shared memory of the row's first CTA and signals its
// mbarrier; that CTA merges them (a bounded wait; a timeout raises
// EAGLE_ERR_TIMEOUT and leaves the row unwritten).
#include "common.cuh"
#include "sm100.cuh"

namespace eagle {

using sm100::cluster_arrive_relaxed;
using sm100::cluster_ctarank;
using sm100::cluster_wait;
using sm100::mapa_shared;
using sm100::mbar_init;
using sm100::mbar_init_fence;
using sm100::mbar_wait_cluster;
using sm100::smem_u32;

struct DraftArgs {
  const void *logits;
  int B, D, k, V, R, S;  // R = used rows per sequence, S = parts per row (one cluster)
  int64_t ld;
  int32_t *tok;
  float *conf;
  float *stats;
  int32_t *status;
};

constexpr int kBatchCap = 128;    // candidates of one segment merged as a batch (the warp's buffer)
constexpr int kMaxDraftParts = 8;  // parts of one row: one cluster

// Number of keys of set[0..n) greater than `key` (set 16-byte aligned).
// Every lane of a warp reads the same addresses (broadcast), four 16-byte
// loads in flight.  Zero keys (empty slots) are never greater.
__device__ __forceinline__ int count_greater(uint64_t key, const uint64_t *set, int n) {
  const ulonglong2 *s2 = reinterpret_cast<const ulonglong2 *>(set);
  int r = 0;
#pragma unroll 4
  for (int q = 0; q < n / 2; ++q) {
    const ulonglong2 v = s2[q];
    r += (v.x > key) + (v.y > key);
  }
  if (n & 1) r += set[n - 1] > key;
  return r;
}

__device__ __forceinline__ uint64_t shfl_up_u64(uint64_t v, int d) {
  uint32_t lo = static_cast<uint32_t>(v), hi = static_cast<uint32_t>(v >> 32);
  lo = __shfl_up_sync(0xffffffffu, lo, d);
  hi = __shfl_up_sync(0xffffffffu, hi, d);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

// Bitonic sort of one float per lane across the warp, descending by lane.
__device__ __forceinline__ float warp_sort_desc(float x, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const float y = __shfl_xor_sync(0xffffffffu, x, stride);
      const bool desc = (lane & size) == 0;
      const bool lower = (lane & stride) == 0;
      x = (desc == lower) ? fmaxf(x, y) : fminf(x, y);
    }
  }
  return x;
}

// Element e of a 16-byte vector as float (no indexed register access).
template <typename T> __device__ __forceinline__ float elem_of(const uint4 &v, int e);
template <> __device__ __forceinline__ float elem_of<__nv_bfloat16>(const uint4 &v, int e) {
  const int q = e >> 1;
  const uint32_t w = q == 0 ? v.x : (q == 1 ? v.y : (q == 2 ? v.z : v.w));
  return (e & 1) ? bf16_hi(w) : bf16_lo(w);
}
template <> __device__ __forceinline__ float elem_of<float>(const uint4 &v, int e) {
  return __uint_as_float(e == 0 ? v.x : (e == 1 ? v.y : (e == 2 ? v.z : v.w)));
}

// Sum over a lane's vectors of 2^(x log2e + nmL): even and odd elements in
// the two halves of a packed pair, one FMA and one add for every two
// elements (each half rounds exactly as its scalar form).  kAll: every
// vector holds data (missing ones are -inf padding), so none is skipped.
template <typename T, int NVL, bool kAll = false>
__device__ __forceinline__ float segment_exp_sum(const uint4 (&vb)[NVL], int nvec, int lane, float nmL) {
  constexpr int VEC = VecTraits<T>::kElems;
  const uint64_t c2 = f2_pack(kLog2e, kLog2e), n2 = f2_pack(nmL, nmL);
  uint64_t acc = f2_pack(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < NVL; ++i) {
    if (kAll || lane + 32 * i < nvec) {
      float x[VEC];
      VecTraits<T>::unpack(vb[i], x);
#pragma unroll
      for (int e = 0; e < VEC; e += 2) {
        float y0, y1;
        f2_unpack(f2_fma(f2_pack(x[e], x[e + 1]), c2, n2), y0, y1);
        acc = f2_add(acc, f2_pack(ex2_approx(y0), ex2_approx(y1)));
      }
    }
  }
  float a0, a1;
  f2_unpack(acc, a0, a1);
  return a0 + a1;
}

// NW warps per CTA, NVL 16-byte vectors per lane and segment.
template <typename T, int NW, int NVL>
__global__ void __launch_bounds__(NW * 32, NW == 4 ? 6 : (NW == 8 ? 3 : 2)) draft_topk_kernel(DraftArgs a) {
  static_assert(NW == 4 || NW == 8 || NW == 16, "4- or 8-warp ring CTAs, 16-warp one-segment CTAs");
  using VT = VecTraits<T>;
  constexpr int VEC = VT::kElems;
  constexpr int SEG = 32 * NVL * VEC;  // tokens per warp and segment
  constexpr int NT = NW * 32;
  __shared__ __align__(16) uint64_t s_buf[NW][kBatchCap];  // a warp's candidates of one segment
  __shared__ __align__(16) uint64_t s_wl[NW][32];           // a warp's list for its batch merge
  __shared__ __align__(16) uint64_t s_tmp[NW][32];
  __shared__ __align__(16) uint64_t s_all[NW * 32];          // the warps' lists: k slots each
  // keys at or above a bound: at most NW*k (block merge) or S*k (part merge)
  __shared__ __align__(16) uint64_t s_cand[(NW > kMaxDraftParts ? NW : kMaxDraftParts) * 32];
  __shared__ __align__(16) uint64_t s_part_keys[kMaxDraftParts][32];  // first CTA: every part's top k
  __shared__ float2 s_part_ms[kMaxDraftParts];                       // first CTA: every part's (max, sum)
  __shared__ __align__(8) uint64_t s_part_bar;                      // first CTA: the parts have pushed
  __shared__ uint64_t s_top[32];
  __shared__ float s_m[NW], s_s[NW];
  __shared__ __align__(16) float s_lmax[NW * 32];  // ring form: each lane's running maximum
  __shared__ int s_nc;
  __shared__ unsigned s_thr;  // block prune bound (order-preserving bits)

  const int rg = blockIdx.y;  // b * R + r
  const int b = rg / a.R, r = rg % a.R;
  const int d = r == 0 ? 0 : 1 + (r - 1) / a.k;
  const int j = r == 0 ? 0 : (r - 1) % a.k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = a.k;
  const int part = a.S > 1 ? static_cast<int>(cluster_ctarank()) : 0;

  const T *row = reinterpret_cast<const T *>(a.logits) +
                 ((static_cast<int64_t>(b) * a.D + d) * a.k + j) * a.ld;
  // This CTA's part of the row is a range of segments; warp w takes
  // segments w, w+NW, ...  A segment is held in registers (all 16-byte
  // loads in flight together) and visited twice: lane maxima, then the sum
  // of exp(x - segment lane max).
  const int nseg = (a.V + SEG - 1) / SEG;
  const int spp = (nseg + a.S - 1) / a.S;
  const int g0 = part * spp, g1 = min(nseg, g0 + spp);
  uint4 vb[NVL];
  // ring form (4- or 8-warp CTAs): warp w's stages at s_ring[(w * kStages +
  // s) * NVL * 32], lane l's vectors l, l+32, ... of a segment in each;
  // every iteration commits one copy group (empty past the part's end)
  constexpr bool kRing = NW <= 8;
  constexpr int kStages = 3;
  extern __shared__ __align__(16) uint4 s_ring[];
  uint4 *my_ring = s_ring + warp * kStages * NVL * 32;
  // A full segment takes NVL unconditional copies at constant offsets; in
  // the row's last, partial segment a lane writes -inf padding into the
  // slots past the row's end (it alone reads them back), so every later
  // step handles all NVL vectors alike: -inf adds nothing to a maximum, an
  // exponential sum or a top-k list.
  auto issue_segment = [&](int gseg, int stage) {
    if (gseg < g1) {
      const int seg0 = gseg * SEG;
      const T *src = row + seg0 + lane * VEC;
      uint4 *dst = my_ring + stage * NVL * 32 + lane;
      if (seg0 + SEG <= a.V) {
#pragma unroll
        for (int i = 0; i < NVL; ++i) cp_async16(dst + 32 * i, src + 32 * i * VEC);
      } else {
        const int nvec = (a.V - seg0) / VEC;
#pragma unroll
        for (int i = 0; i < NVL; ++i) {
          if (lane + 32 * i < nvec) cp_async16(dst + 32 * i, src + 32 * i * VEC);
          else dst[32 * i] = VT::neg_inf_vec();
        }
      }
    }
    cp_async_commit();
  };
  auto load_segment = [&](int gseg) {
    const int seg0 = gseg * SEG;
    const int nvec = min(SEG, a.V - seg0) / VEC;
#pragma unroll
    for (int i = 0; i < NVL; ++i) {
      const int v = lane + 32 * i;
      if (v < nvec) vb[i] = ld_stream16(row + seg0 + v * VEC);
    }
  };
  pdl_wait();
  // in flight while the shared state is set up
  if constexpr (kRing) {
#pragma unroll
    for (int st = 0; st < kStages - 1; ++st) issue_segment(g0 + warp + st * NW, st);
  } else {
    if (g0 + warp < g1) load_segment(g0 + warp);
  }
  if (tid == 0) {
    s_thr = ordered_u32(-INFINITY);
    s_nc = 0;
    if (a.S > 1) {
      // the other parts' keys and (max, sum) arrive as transaction bytes
      mbar_init(&s_part_bar, 1);
      mbar_init_fence();
      if (part == 0) sm100::mbar_arrive_expect_tx(&s_part_bar, (a.S - 1) * (k * 8 + 8));
    }
  }
  if (tid < 32) s_top[tid] = 0ull;
  s_lmax[tid] = -INFINITY;
  __syncthreads();
  if (a.S > 1) cluster_arrive_relaxed();  // waited on before a part pushes to the first CTA

  float m = -INFINITY, sum = 0.f;  // this lane's running max and sum of exp(x - m)
  float lmax = -INFINITY;          // this lane's largest value so far
  float thr = -INFINITY;           // prune bound: at least k values of the part are >= thr
  float published = -INFINITY;     // this warp's bound as last raised in s_thr
  // The warp's top keys so far, sorted, in registers: lane i < k holds the
  // i-th (0 = empty); cnt of them are set (warp-uniform).  Once k are set,
  // lane k-1's key is the tightest prune bound.
  uint64_t mine = 0;
  int cnt = 0;
  auto insert = [&](uint64_t key) {  // called by the whole warp with one key
    const int pos = __popc(__ballot_sync(0xffffffffu, lane < k && mine > key));
    if (pos < k) {
      const uint64_t up = shfl_up_u64(mine, 1);
      if (lane > pos && lane < k) mine = up;
      if (lane == pos) mine = key;
      cnt = cnt < k ? cnt + 1 : k;
      if (cnt == k) thr = fmaxf(thr, key_value(shfl_u64(mine, k - 1)));
    }
  };
  float M = -INFINITY, Z = 0.f;  // the part's softmax statistics (warp 0)
  if constexpr (NW == 16) {
    // ---- one segment per warp: selection against one block-wide bound ----
    // The k-th largest of the warps' maxima, T: the warps whose maximum is
    // at or above T are at least k, each with a distinct element there, so
    // T bounds the part's k-th largest value from below.  (When fewer than
    // k warps hold a segment, T is the largest over the warps of each
    // warp's k-th largest lane maximum, a bound for the same reason.)  Every
    // element at or above T is gathered (one shared atomic per warp) and the
    // gathered keys are ranked by counting.  A flat row with more than
    // kGatherCap such elements takes the per-warp lists instead.
    constexpr int kGatherCap = 256;
    const int gseg = g0 + warp;
    const bool has = gseg < g1;  // warp-uniform
    const int seg0 = gseg * SEG;
    const int nvec = has ? min(SEG, a.V - seg0) / VEC : 0;
    float vmx[NVL];
    float smax = -INFINITY;
#pragma unroll
    for (int i = 0; i < NVL; ++i) {
      vmx[i] = (lane + 32 * i < nvec) ? vec_max<T>(vb[i]) : -INFINITY;
      smax = fmaxf(smax, vmx[i]);
    }
    const bool by_warps = k <= g1 - g0;  // at least k warps hold a segment (block-uniform)
    if (has && !by_warps) {
      const float y = warp_sort_desc(smax, lane);
      const float kth = __shfl_sync(0xffffffffu, y, k - 1);
      if (lane == 0 && kth > -INFINITY) atomicMax(&s_thr, ordered_u32(kth));
    }
    if (smax > -INFINITY) {
      m = smax;
      sum = segment_exp_sum<T, NVL>(vb, nvec, lane, -smax * kLog2e);
    }
    pdl_trigger();
    {
      const float mw = warp_max(m);
      const float sw = warp_sum((m == -INFINITY) ? 0.f : sum * ex2_approx((m - mw) * kLog2e));
      if (lane == 0) {
        s_m[warp] = mw;
        s_s[warp] = sw;
      }
    }
    __syncthreads();
    float bound = from_ordered_u32(s_thr);
    if (by_warps) {
      // the warp maximum of rank k-1 (greater, or equal at a lower warp, ranks first)
      const float wm = lane < NW ? s_m[lane] : -INFINITY;
      int rk = 0;
#pragma unroll
      for (int j = 0; j < NW; ++j) {
        const float o = s_m[j];
        rk += (o > wm) || (o == wm && j < lane);
      }
      const unsigned at = __ballot_sync(0xffffffffu, lane < NW && rk == k - 1 && wm > -INFINITY);
      if (at) bound = fmaxf(bound, __shfl_sync(0xffffffffu, wm, __ffs(at) - 1));
    }
    unsigned cms[NVL];
    int mycnt = 0;
#pragma unroll
    for (int i = 0; i < NVL; ++i) {
      cms[i] = 0;
      if (vmx[i] > -INFINITY && vmx[i] >= bound) {
        float x[VEC];
        VT::unpack(vb[i], x);
#pragma unroll
        for (int e = 0; e < VEC; ++e)
          if (x[e] >= bound && x[e] > -INFINITY) cms[i] |= 1u << e;
      }
      mycnt += __popc(cms[i]);
    }
    int pos = mycnt;  // inclusive prefix over the lanes, then exclusive
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, pos, o);
      if (lane >= o) pos += v;
    }
    const int total = __shfl_sync(0xffffffffu, pos, 31);
    pos -= mycnt;
    int base = 0;
    if (lane == 0 && total > 0) base = atomicAdd(&s_nc, total);
    base = __shfl_sync(0xffffffffu, base, 0);
    if (base + total <= kGatherCap) {
#pragma unroll
      for (int i = 0; i < NVL; ++i)
        for (unsigned cm = cms[i]; cm; cm &= cm - 1) {
          const int e = __ffs(cm) - 1;
          s_cand[base + pos++] = topk_key(elem_of<T>(vb[i], e), static_cast<uint32_t>(seg0 + (lane + 32 * i) * VEC + e));
        }
    }
    if (warp == 0) {
      const float mw = lane < NW ? s_m[lane] : -INFINITY;
      M = warp_max(mw);
      Z = warp_sum(mw == -INFINITY ? 0.f : s_s[lane] * ex2_approx((mw - M) * kLog2e));
    }
    __syncthreads();
    const int nc = s_nc;
    if (nc <= kGatherCap) {
      for (int i = tid; i < nc; i += NT) {
        const uint64_t key = s_cand[i];
        const int rk = count_greater(key, s_cand, nc);
        if (rk < k) s_top[rk] = key;
      }
    } else {
      // flat row: each warp keeps its k best of the gathered elements in
      // registers (one ballot-ranked insert per element), then the NW lists
      // are ranked together
#pragma unroll
      for (int i = 0; i < NVL; ++i) {
        unsigned cm = cms[i];
        for (unsigned lanes = __ballot_sync(0xffffffffu, cm != 0); lanes;
             lanes = __ballot_sync(0xffffffffu, cm != 0)) {
          const int src = __ffs(lanes) - 1;
          uint64_t key = 0;
          if (lane == src) {
            const int e = __ffs(cm) - 1;
            cm &= cm - 1;
            key = topk_key(elem_of<T>(vb[i], e), static_cast<uint32_t>(seg0 + (lane + 32 * i) * VEC + e));
          }
          insert(shfl_u64(key, src));
        }
      }
      if (lane < k) s_all[warp * k + lane] = mine;
      __syncthreads();
      for (int i = tid; i < NW * k; i += NT) {
        const uint64_t key = s_all[i];
        if (!key) continue;
        const int rk = count_greater(key, s_all, NW * k);
        if (rk < k) s_top[rk] = key;
      }
    }
    __syncthreads();
  } else {
    static_assert(kRing, "the streaming form is the shared-memory ring");
    int st_read = 0, st_issue = kStages - 1;  // ring stages, advanced without division
    for (int gseg = g0 + warp, it = 0; gseg < g1; gseg += NW, ++it) {
      const int seg0 = gseg * SEG;
      // the stage read one iteration ago takes the segment kStages-1 ahead;
      // this iteration's copies are then complete
      issue_segment(gseg + (kStages - 1) * NW, st_issue);
      st_issue = st_issue == kStages - 1 ? 0 : st_issue + 1;
      cp_async_wait<kStages - 1>();
      {
        const uint4 *src = my_ring + st_read * NVL * 32 + lane;
#pragma unroll
        for (int i = 0; i < NVL; ++i) vb[i] = src[32 * i];
      }
      st_read = st_read == kStages - 1 ? 0 : st_read + 1;
      float smax = -INFINITY;
      float vmx[NVL];
  #pragma unroll
      for (int i = 0; i < NVL; ++i) {
        vmx[i] = vec_max<T>(vb[i]);
        smax = fmaxf(smax, vmx[i]);
      }
      if (smax > -INFINITY) lse_combine(m, sum, smax, segment_exp_sum<T, NVL, true>(vb, 0, lane, -smax * kLog2e));
      lmax = fmaxf(lmax, smax);
      // block bound from the lanes' running maxima: a slot only ever holds an
      // element of this part (or -inf), whenever it is read, and distinct
      // slots hold distinct elements, so the k-th largest of any slots
      // bounds the part's k-th largest from below.  Every eighth segment a
      // warp takes the maxima of 32 groups of NW slots (lane l: slots
      // NW*l .. NW*l+NW-1 of the NW*32) and raises the shared bound to their
      // k-th largest.
      s_lmax[tid] = lmax;
      if (((it + warp) & 7) == 0) {
        float g[NW];
#pragma unroll
        for (int h = 0; h < NW; h += 4)
          asm volatile("ld.volatile.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                       : "=f"(g[h]), "=f"(g[h + 1]), "=f"(g[h + 2]), "=f"(g[h + 3])
                       : "r"(smem_u32(s_lmax + NW * lane + h)));
        float gm = g[0];
#pragma unroll
        for (int e = 1; e < NW; ++e) gm = fmaxf(gm, g[e]);
        const float y = warp_sort_desc(gm, lane);
        const float kth = __shfl_sync(0xffffffffu, y, k - 1);
        if (kth > thr) {
          thr = kth;
          if (lane == 0) atomicMax(&s_thr, ordered_u32(kth));
        }
      }
      // prune bound: before the list holds k keys, the k-th largest lane
      // maximum (lane maxima are distinct elements), sorted for only when at
      // least k lane maxima lie above the current bound (else it cannot
      // raise it); the block's shared maximum of its warps' bounds every
      // segment (one shared load)
      thr = fmaxf(thr, from_ordered_u32(*const_cast<volatile unsigned *>(&s_thr)));
      if (cnt < k && __popc(__ballot_sync(0xffffffffu, lmax > thr)) >= k) {
        const float y = warp_sort_desc(lmax, lane);
        thr = fmaxf(thr, __shfl_sync(0xffffffffu, y, k - 1));
      }
      if (!__any_sync(0xffffffffu, smax > -INFINITY && smax >= thr)) continue;
      unsigned cms[NVL];  // this lane's elements of each vector at or above the bound
      int mycnt = 0;
  #pragma unroll
      for (int i = 0; i < NVL; ++i) {
        cms[i] = 0;
        if (vmx[i] > -INFINITY && vmx[i] >= thr) {
          float x[VEC];
          VT::unpack(vb[i], x);
  #pragma unroll
          for (int e = 0; e < VEC; ++e)
            if (x[e] >= thr && x[e] > -INFINITY) cms[i] |= 1u << e;
        }
        mycnt += __popc(cms[i]);
      }
      const int total = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(mycnt)));
      if (total > 4 && total <= kBatchCap) {
        // many candidates (a warp's first segment): write them to the warp's
        // buffer, then keep the k best of list + buffer by counting larger keys
        int pos = mycnt;
  #pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, pos, o);
          if (lane >= o) pos += v;
        }
        pos -= mycnt;
        uint64_t *buf = s_buf[warp];
  #pragma unroll
        for (int i = 0; i < NVL; ++i)
          for (unsigned cm = cms[i]; cm; cm &= cm - 1) {
            const int e = __ffs(cm) - 1;
            buf[pos++] = topk_key(elem_of<T>(vb[i], e), static_cast<uint32_t>(seg0 + (lane + 32 * i) * VEC + e));
          }
        if (lane < cnt) s_wl[warp][lane] = mine;
        __syncwarp();
        for (int q = lane; q < cnt + total; q += 32) {
          const uint64_t key = q < cnt ? s_wl[warp][q] : buf[q - cnt];
          const int rk = count_greater(key, s_wl[warp], cnt) + count_greater(key, buf, total);
          if (rk < k) s_tmp[warp][rk] = key;
        }
        __syncwarp();
        cnt = cnt + total < k ? cnt + total : k;
        mine = lane < cnt ? s_tmp[warp][lane] : 0ull;
        if (cnt == k) thr = fmaxf(thr, key_value(shfl_u64(mine, k - 1)));
        __syncwarp();
      } else {
  #pragma unroll
      for (int i = 0; i < NVL; ++i) {
        unsigned cm = cms[i];
        // insert them one by one (lowest lane, lowest element first); each
        // insert may raise the bound and drop later ones
        for (unsigned lanes = __ballot_sync(0xffffffffu, cm != 0); lanes;
             lanes = __ballot_sync(0xffffffffu, cm != 0)) {
          const int src = __ffs(lanes) - 1;
          uint64_t key = 0;
          if (lane == src) {
            const int e = __ffs(cm) - 1;
            cm &= cm - 1;
            key = topk_key(elem_of<T>(vb[i], e), static_cast<uint32_t>(seg0 + (lane + 32 * i) * VEC + e));
          }
          key = shfl_u64(key, src);
          if (key_value(key) >= thr) insert(key);
          if (cm && !(vmx[i] >= thr)) cm = 0;  // the raised bound excludes the rest of this vector
        }
      }
      }
      if (cnt == k && thr > published) {  // raise the block's bound (rare once warm)
        if (lane == 0) atomicMax(&s_thr, ordered_u32(thr));
        published = thr;
      }
    }
    // this warp's list into its k slots (empty slots hold zero keys)
    if (lane < k) s_all[warp * k + lane] = mine;
    pdl_trigger();

    // ---- block: softmax statistics and the top k of the warp lists ------------
    {
      const float mw = warp_max(m);
      const float sw = warp_sum((m == -INFINITY) ? 0.f : sum * ex2_approx((m - mw) * kLog2e));
      if (lane == 0) {
        s_m[warp] = mw;
        s_s[warp] = sw;
      }
    }
    __syncthreads();
    // The top k of the block are among the keys at or above a lower bound
    // for its k-th largest key: the larger of the block's prune bound and the
    // k-th largest of a sample holding each warp's best ceil(k/NW) keys (at
    // least k keys of the block reach either).  The warps that gather the
    // keys at or above it each compute the sample bound themselves; the
    // gathered keys are then ranked by counting.
    static_assert(NW <= 32 && (NW & (NW - 1)) == 0, "NW * ceil(k/NW) <= 32 for every k <= 32");
    const int per_w = (k + NW - 1) / NW;
    if (warp * 32 < NW * k) {
      float sv = -INFINITY;
      if (lane < NW * per_w) {
        const uint64_t key = s_all[(lane / per_w) * k + lane % per_w];
        if (key) sv = key_value(key);
      }
      const float y = warp_sort_desc(sv, lane);
      const float bound = fmaxf(__shfl_sync(0xffffffffu, y, k - 1), from_ordered_u32(s_thr));
      const uint64_t key = tid < NW * k ? s_all[tid] : 0ull;
      const bool in = key && key_value(key) >= bound;
      const unsigned bal = __ballot_sync(0xffffffffu, in);
      int base = 0;
      if (lane == 0 && bal) base = atomicAdd(&s_nc, __popc(bal));
      base = __shfl_sync(0xffffffffu, base, 0);
      if (in) s_cand[base + __popc(bal & ((1u << lane) - 1u))] = key;
    }
    // the warps' (max, sum) pairs combined by one warp: the block maximum,
    // then each pair rescaled to it (one exponential per lane) and summed
    if (warp == 0) {
      const float mw = lane < NW ? s_m[lane] : -INFINITY;
      M = warp_max(mw);
      Z = warp_sum(mw == -INFINITY ? 0.f : s_s[lane] * ex2_approx((mw - M) * kLog2e));
    }
    __syncthreads();
    const int nc = s_nc;
    for (int i = tid; i < nc; i += NT) {
      const uint64_t key = s_cand[i];
      const int rk = count_greater(key, s_cand, nc);
      if (rk < k) s_top[rk] = key;
    }
    __syncthreads();
  }

  const int64_t slot = ((static_cast<int64_t>(b) * a.D + d) * a.k + j);
  auto finalize = [&](const uint64_t *top, float Mf, float Zf) {  // by warp 0
    if (lane < k) {
      const uint64_t key = top[lane];
      int32_t t = -1;
      float cf = 0.f;
      if (key) {
        t = static_cast<int32_t>(key_token(key));
        cf = expf(key_value(key) - Mf) / Zf;
      }
      a.tok[slot * a.k + lane] = t;
      a.conf[slot * a.k + lane] = cf;
    }
    if (lane == 0 && a.stats) {
      a.stats[slot * 2 + 0] = Mf;
      a.stats[slot * 2 + 1] = logf(Zf);
    }
  };
  if (a.S == 1) {
    if (warp == 0) finalize(s_top, M, Z);
    return;
  }

  // ---- parts of a row: push to the first CTA of the cluster, which merges --
  if (part != 0) {
    cluster_wait();  // the first CTA's barrier is initialised
    if (warp == 0) {
      // asynchronous stores into the first CTA, each completing its share
      // of the barrier's expected bytes
      const uint32_t bar = mapa_shared(smem_u32(&s_part_bar), 0);
      if (lane < k) {
        const uint32_t dst = mapa_shared(smem_u32(&s_part_keys[part][lane]), 0);
        const uint64_t key = s_top[lane];
        asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b64 [%0], %1, [%2];"
                     ::"r"(dst), "l"(key), "r"(bar) : "memory");
      }
      if (lane == 0) {
        const uint32_t dst = mapa_shared(smem_u32(&s_part_ms[part]), 0);
        asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];"
                     ::"r"(dst), "f"(M), "f"(Z), "r"(bar) : "memory");
      }
    }
    return;
  }
  cluster_wait();
  if (warp == 0) {
    bool ok = true;
    if (lane == 0) ok = mbar_wait_cluster(&s_part_bar, 0, 200000000ull);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (!ok) {
      if (lane == 0) report(a.status, EAGLE_ERR_TIMEOUT);
    } else {
      // own top k and (max, sum) as part 0, then the S*k keys ranked
      if (lane < k) s_part_keys[0][lane] = s_top[lane];
      float pm = lane == 0 ? M : -INFINITY, ps = lane == 0 ? Z : 0.f;
      if (lane > 0 && lane < a.S) {
        pm = s_part_ms[lane].x;
        ps = s_part_ms[lane].y;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, pm, o), z2 = __shfl_xor_sync(0xffffffffu, ps, o);
        lse_combine(pm, ps, m2, z2);
      }
      __syncwarp();
      // candidates: keys at or above the largest k-th key of any part
      float pb = -INFINITY;
      for (int q = lane; q < a.S; q += 32) {
        const uint64_t kth = s_part_keys[q][k - 1];
        if (kth) pb = fmaxf(pb, key_value(kth));
      }
      pb = warp_max(pb);
      int n = 0;
      for (int q = 0; q < a.S; ++q) {
        const uint64_t key = lane < k ? s_part_keys[q][lane] : 0ull;
        const bool in = key && key_value(key) >= pb;
        const unsigned bal = __ballot_sync(0xffffffffu, in);
        if (in) s_cand[n + __popc(bal & ((1u << lane) - 1u))] = key;
        n += __popc(bal);
      }
      if (lane < k) s_tmp[0][lane] = 0ull;
      __syncwarp();
      for (int q = lane; q < n; q += 32) {
        const uint64_t key = s_cand[q];
        const int rk = count_greater(key, s_cand, n);
        if (rk < k) s_tmp[0][rk] = key;
      }
      __syncwarp();
      finalize(s_tmp[0], pm, ps);
    }
  }
}

// ---- host side ---------------------------------------------------------------

struct DraftPlan {
  int NW, NVL, S;
};

// Few rows: 16-warp CTAs with 1024-token segments (bf16), when each row can
// be split into parts of one segment per warp and the parts take at most
// three waves of two CTAs per SM.  Otherwise 8-warp CTAs streaming 1024-token
// segments through a shared-memory ring: enough parts for about three CTAs
// per SM, but no part smaller than one segment per warp; or, when that
// leaves a warp fewer than eight segments, 4-warp CTAs (six per SM).  At
// most kMaxDraftParts parts per row (one cluster).
static DraftPlan draft_plan(int B, int R, int V, int vec, int num_sms) {
  const int64_t rows = static_cast<int64_t>(B) * R;
  DraftPlan p;
  {
    const int seg = 4 * 32 * vec;
    const int64_t nseg = (V + seg - 1) / seg;
    const int64_t parts = (nseg + 15) / 16;
    if (parts <= kMaxDraftParts && rows * parts <= 6 * static_cast<int64_t>(num_sms)) {
      p.NW = 16;
      p.NVL = 4;
      p.S = static_cast<int>(parts);
      return p;
    }
  }
  const int seg = 4 * 32 * vec;
  const int64_t nseg = (V + seg - 1) / seg;
  const int64_t max_parts = (nseg + 7) / 8;
  int64_t S = (static_cast<int64_t>(num_sms) * 3 + rows - 1) / rows;
  if (S > max_parts) S = max_parts;
  if (S > kMaxDraftParts) S = kMaxDraftParts;
  if (S < 1) S = 1;
  p.NW = 8;
  p.NVL = 4;
  p.S = static_cast<int>(S);
  // Fewer than eight segments per warp leave the ring's fill and the block
  // merge unamortised: 4-warp CTAs instead, six per SM, with parts of at
  // least eight segments per warp where the row has them.
  if ((nseg + S * 8 - 1) / (S * 8) < 8) {
    int64_t S4 = (static_cast<int64_t>(num_sms) * 6 + rows - 1) / rows;
    const int64_t max4 = nseg / 32 > 1 ? nseg / 32 : 1;
    if (S4 > max4) S4 = max4;
    if (S4 > kMaxDraftParts) S4 = kMaxDraftParts;
    if (S4 < 1) S4 = 1;
    p.NW = 4;
    p.S = static_cast<int>(S4);
  }
  return p;
}

// The parts of a row merge through the shared memory of their cluster: no
// workspace.
size_t draft_workspace_bytes(int, int, int, int, int, int) { return 0; }

// Ring CTAs of NW warps: three stages of 4 vectors per lane for each warp.
constexpr int ring_bytes(int nw) { return nw * 3 * 4 * 32 * 16; }

template <typename T, int NW>
static cudaError_t launch_ring(const DraftArgs &a, const dim3 &grid, cudaStream_t st) {
  static std::atomic<unsigned long long> configured{0};
  const cudaError_t e = set_smem_limit_once(draft_topk_kernel<T, NW, 4>, ring_bytes(NW), configured);
  if (e != cudaSuccess) return e;
  return launch_chained_cluster(draft_topk_kernel<T, NW, 4>, grid, dim3(NW * 32), ring_bytes(NW), st, a.S, a);
}

template <typename T>
static cudaError_t launch_t(const DraftArgs &a, const DraftPlan &p, cudaStream_t st) {
  const dim3 grid(a.S, a.B * a.R);
  if (p.NW == 16)
    return launch_chained_cluster(draft_topk_kernel<T, 16, 4>, grid, dim3(16 * 32), 0, st, a.S, a);
  if (p.NW == 4) return launch_ring<T, 4>(a, grid, st);
  return launch_ring<T, 8>(a, grid, st);
}

cudaError_t launch_draft_topk(const void *logits, int dtype, int B, int D, int k, int V,
                              int64_t ld, int32_t *tok, float *conf, float *stats,
                              void *, int32_t *status, int num_sms, cudaStream_t st) {
  DraftArgs a;
  a.logits = logits;
  a.B = B; a.D = D; a.k = k; a.V = V; a.ld = ld;
  a.R = 1 + (D - 1) * k;
  const int vec = dtype == EAGLE_BF16 ? 8 : 4;
  const DraftPlan p = draft_plan(B, a.R, V, vec, num_sms);
  a.S = p.S;
  a.tok = tok; a.conf = conf; a.stats = stats;
  a.status = status;
  return dtype == EAGLE_BF16 ? launch_t<__nv_bfloat16>(a, p, st) : launch_t<float>(a, p, st);
}

}  // namespace eagle
