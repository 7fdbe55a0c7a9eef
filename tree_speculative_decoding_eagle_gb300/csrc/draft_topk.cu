// Stage 1: per-row softmax statistics and top-k of the draft logits.
//
// [EAGLE-2] section "ドラフトモデルのキャリブレーション": the confidence of a
// draft token is the probability the draft model assigns to it.  For every
// used row: M = max, Z = sum exp(x - M), the k largest logits (ties -> lower
// token id) and c = exp(x - M) / Z.
//
// One pass over HBM.  A row is split into parts of 8 warps x 2048 tokens
// (bf16; 1024 for fp32), one CTA per part.  Each warp holds a segment in
// registers (all 16-byte loads in flight at once) and visits it twice: lane
// maxima, then the sum of exp(x - segment max), folded into a running
// (max, sum).  Top-k selection works on unique 64-bit keys (logit order,
// then lower token id).  Each warp keeps its k best keys so far sorted in
// registers (lane i holds the i-th); a new key's place is the number of
// larger keys (one ballot) and the tail shifts down one lane.  The list's
// k-th key bounds the part from below, so values under the bound (shared
// block-wide as a maximum over the warps) are never looked at; before the
// list is full, the k-th largest lane maximum is the bound.  The warp lists
// merge block-wide by rank counting in shared memory.  With S > 1 the last
// CTA of a row to finish (atomic ticket in the workspace) merges the S
// partial results; no CTA ever waits for another.
#include "common.cuh"

namespace eagle {

struct DraftArgs {
  const void *logits;
  int B, D, k, V, R, S;  // R = used rows per sequence, S = splits per row
  int64_t ld;
  int32_t *tok;
  float *conf;
  float *stats;
  unsigned char *ws;     // [counters (B*R u32, 256-aligned)][records]
  int32_t *status;
};

constexpr int kDraftThreads = 256;
constexpr int kBatchCap = 128;  // candidates of one segment merged as a batch (the warp's buffer)
constexpr int kDraftVecPerLane = 8;  // 16-byte vectors each lane holds in registers

// Workspace: [tickets: u32 per row][(max, sum) per row and split][k keys per
// row and split], each part 256-byte aligned.
__host__ __device__ inline size_t draft_counter_bytes(int B, int R) {
  return (static_cast<size_t>(B) * R * sizeof(uint32_t) + 255) / 256 * 256;
}
__host__ __device__ inline size_t draft_ms_bytes(int B, int R, int S) {
  return (static_cast<size_t>(B) * R * S * sizeof(float2) + 255) / 256 * 256;
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

// Rank of `key` among set[0..n): the number of larger keys (keys are unique).
__device__ __forceinline__ int rank_in(uint64_t key, const uint64_t *set, int n) {
  int r = 0;
  for (int q = 0; q < n; ++q) r += set[q] > key;
  return r;
}

__device__ __forceinline__ uint64_t shfl_up_u64(uint64_t v, int d) {
  uint32_t lo = static_cast<uint32_t>(v), hi = static_cast<uint32_t>(v >> 32);
  lo = __shfl_up_sync(0xffffffffu, lo, d);
  hi = __shfl_up_sync(0xffffffffu, hi, d);
  return (static_cast<uint64_t>(hi) << 32) | lo;
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

template <typename T>
__global__ void __launch_bounds__(kDraftThreads, 3) draft_topk_kernel(DraftArgs a) {
  using VT = VecTraits<T>;
  constexpr int VEC = VT::kElems;
  constexpr int NVL = kDraftVecPerLane;
  constexpr int SEG = 32 * NVL * VEC;  // tokens per warp
  constexpr int NW = kDraftThreads / 32;
  __shared__ uint64_t s_buf[NW][32 * 4];  // gathered keys of the block merge (NW*k, or S*k in the split merge)
  __shared__ uint64_t s_wl[NW][32], s_tmp[NW][32];
  __shared__ int s_wn[NW];
  __shared__ uint64_t s_top[32];
  __shared__ float s_m[NW], s_s[NW];
  __shared__ int s_last;
  __shared__ unsigned s_thr;  // block prune bound (order-preserving bits)

  const int s = blockIdx.x;
  const int rg = blockIdx.y;  // b * R + r
  const int b = rg / a.R, r = rg % a.R;
  const int d = r == 0 ? 0 : 1 + (r - 1) / a.k;
  const int j = r == 0 ? 0 : (r - 1) % a.k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = a.k;

  const T *row = reinterpret_cast<const T *>(a.logits) +
                 ((static_cast<int64_t>(b) * a.D + d) * a.k + j) * a.ld;
  if (tid == 0) s_thr = ordered_u32(-INFINITY);
  if (lane == 0) s_wn[warp] = 0;
  pdl_wait();
  __syncthreads();  // s_thr and list sizes initialised
  // This CTA's part of the row is a range of 2048-token segments (1024 for
  // fp32); warp w takes segments w, w+8, ...  A segment is held in
  // registers (all 16-byte loads in flight together) and visited twice:
  // lane maxima, then the sum of exp(x - segment lane max).
  const int nseg = (a.V + SEG - 1) / SEG;
  const int spp = (nseg + a.S - 1) / a.S;
  const int g0 = s * spp, g1 = min(nseg, g0 + spp);
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
  for (int gseg = g0 + warp; gseg < g1; gseg += NW) {
    const int seg0 = gseg * SEG;
    const int nvec = min(SEG, a.V - seg0) / VEC;
    uint4 vb[NVL];
#pragma unroll
    for (int i = 0; i < NVL; ++i) {
      const int v = lane + 32 * i;
      if (v < nvec) vb[i] = ld_stream16(row + seg0 + v * VEC);
    }
    float smax = -INFINITY;
    float vmx[NVL];
#pragma unroll
    for (int i = 0; i < NVL; ++i) {
      vmx[i] = (lane + 32 * i < nvec) ? vec_max<T>(vb[i]) : -INFINITY;
      smax = fmaxf(smax, vmx[i]);
    }
    if (smax > -INFINITY) {
      // sum of 2^(x*log2e - smax*log2e): per element one extract, FMA, ex2, add
      const float nmL = -smax * kLog2e;
      float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
      for (int i = 0; i < NVL; ++i) {
        if (lane + 32 * i < nvec) {
          float x[VEC];
          VT::unpack(vb[i], x);
#pragma unroll
          for (int e = 0; e < VEC; e += 2) {
            acc0 += ex2_approx(fmaf(x[e], kLog2e, nmL));
            acc1 += ex2_approx(fmaf(x[e + 1], kLog2e, nmL));
          }
        }
      }
      lse_combine(m, sum, smax, acc0 + acc1);
    }
    lmax = fmaxf(lmax, smax);
    // prune bound: before the list holds k keys, the k-th largest lane
    // maximum (lane maxima are distinct elements); the block's shared
    // maximum of its warps' bounds every segment (one shared load)
    if (cnt < k) {
      const float y = warp_sort_desc(lmax, lane);
      thr = fmaxf(thr, __shfl_sync(0xffffffffu, y, k - 1));
    }
    thr = fmaxf(thr, from_ordered_u32(*const_cast<volatile unsigned *>(&s_thr)));
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
      // buffer, then keep the k best of list + buffer by rank counting
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
        const int rk = rank_in(key, s_wl[warp], cnt) + rank_in(key, buf, total);
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
  if (lane < k) s_wl[warp][lane] = mine;
  if (lane == 0) s_wn[warp] = cnt;
  pdl_trigger();

  // ---- block: softmax statistics and the top k of the warp lists ------------
  {
    float mw = warp_max(m);
    float sw = (m == -INFINITY) ? 0.f : sum * ex2_approx((m - mw) * kLog2e);
    sw = warp_sum(sw);
    if (lane == 0) {
      s_m[warp] = mw;
      s_s[warp] = sw;
    }
  }
  __syncthreads();
  // gather the warp lists into one array (the first warp's buffer)
  uint64_t *U = s_buf[0];
  int C = 0;
  for (int w = 0; w < NW; ++w) {
    const int nw = s_wn[w];
    if (tid < nw) U[C + tid] = s_wl[w][tid];
    C += nw;
  }
  if (tid < 32) s_top[tid] = 0ull;
  __syncthreads();
  for (int i = tid; i < C; i += kDraftThreads) {
    const uint64_t key = U[i];
    const int rk = rank_in(key, U, C);
    if (rk < k) s_top[rk] = key;
  }
  float M = s_m[0], Z = s_s[0];
  for (int w = 1; w < NW; ++w) lse_combine(M, Z, s_m[w], s_s[w]);
  __syncthreads();

  const int64_t slot = ((static_cast<int64_t>(b) * a.D + d) * a.k + j);
  auto finalize = [&](const uint64_t *top, float Mf, float Zf) {
    if (tid < k) {
      const uint64_t key = top[tid];
      int32_t t = -1;
      float cf = 0.f;
      if (key) {
        t = static_cast<int32_t>(key_token(key));
        cf = expf(key_value(key) - Mf) / Zf;
      }
      a.tok[slot * a.k + tid] = t;
      a.conf[slot * a.k + tid] = cf;
    }
    if (tid == 0 && a.stats) {
      a.stats[slot * 2 + 0] = Mf;
      a.stats[slot * 2 + 1] = logf(Zf);
    }
  };
  if (a.S == 1) {
    finalize(s_top, M, Z);
    return;
  }

  // ---- split rows: publish the partial, the last CTA merges ---------------
  uint32_t *counters = reinterpret_cast<uint32_t *>(a.ws);
  float2 *parts_ms = reinterpret_cast<float2 *>(a.ws + draft_counter_bytes(a.B, a.R));
  uint64_t *parts_keys =
      reinterpret_cast<uint64_t *>(a.ws + draft_counter_bytes(a.B, a.R) + draft_ms_bytes(a.B, a.R, a.S));
  const int64_t prow = static_cast<int64_t>(rg) * a.S;
  if (tid < k) parts_keys[(prow + s) * k + tid] = s_top[tid];
  if (tid == 0) parts_ms[prow + s] = make_float2(M, Z);
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(counters + rg, 1u) == static_cast<uint32_t>(a.S - 1));
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  const int CS = a.S * k;
  for (int i = tid; i < CS; i += kDraftThreads)
    U[i] = __ldcg(reinterpret_cast<const unsigned long long *>(parts_keys + prow * k + i));
  if (tid < 32) s_top[tid] = 0ull;
  __syncthreads();
  for (int i = tid; i < CS; i += kDraftThreads) {
    const uint64_t key = U[i];
    if (!key) continue;  // a slice with fewer than k finite values
    const int rk = rank_in(key, U, CS);
    if (rk < k) s_top[rk] = key;
  }
  if (warp == 0) {
    float pm = -INFINITY, ps = 0.f;
    for (int q = lane; q < a.S; q += 32) {
      const float2 ms = __ldcg(parts_ms + prow + q);
      lse_combine(pm, ps, ms.x, ms.y);
    }
    const float Mw = warp_max(pm);
    const float Zw = warp_sum(pm == -INFINITY ? 0.f : ps * ex2_approx((pm - Mw) * kLog2e));
    if (lane == 0) {
      s_m[0] = Mw;
      s_s[0] = Zw;
    }
  }
  __syncthreads();
  finalize(s_top, s_m[0], s_s[0]);
  if (tid == 0) counters[rg] = 0;  // leave the ticket zeroed for the next call
}

// ---- host side ---------------------------------------------------------------

// Parts (CTAs) per row: enough CTAs for about three per SM, but no part
// smaller than one 2048-token segment per warp.
int draft_splits(int B, int R, int V, int vec, int num_sms) {
  const int64_t rows = static_cast<int64_t>(B) * R;
  const int seg = kDraftVecPerLane * 32 * vec;
  const int64_t nseg = (V + seg - 1) / seg;
  const int64_t max_parts = (nseg + (kDraftThreads / 32) - 1) / (kDraftThreads / 32);
  int64_t S = (static_cast<int64_t>(num_sms) * 3 + rows - 1) / rows;
  if (S > max_parts) S = max_parts;
  if (S > 32) S = 32;
  if (S < 1) S = 1;
  return static_cast<int>(S);
}

size_t draft_workspace_bytes(int B, int D, int k, int V, int vec, int num_sms) {
  const int R = 1 + (D - 1) * k;
  const int S = draft_splits(B, R, V, vec, num_sms);
  if (S == 1) return draft_counter_bytes(B, R);
  return draft_counter_bytes(B, R) + draft_ms_bytes(B, R, S) + static_cast<size_t>(B) * R * S * k * sizeof(uint64_t);
}

template <typename T>
static cudaError_t launch_t(const DraftArgs &a, cudaStream_t st) {
  return launch_chained(draft_topk_kernel<T>, dim3(a.S, a.B * a.R), dim3(kDraftThreads), 0, st, a);
}

cudaError_t launch_draft_topk(const void *logits, int dtype, int B, int D, int k, int V,
                              int64_t ld, int32_t *tok, float *conf, float *stats,
                              void *ws, int32_t *status, int num_sms, cudaStream_t st) {
  DraftArgs a;
  a.logits = logits;
  a.B = B; a.D = D; a.k = k; a.V = V; a.ld = ld;
  a.R = 1 + (D - 1) * k;
  const int vec = dtype == EAGLE_BF16 ? 8 : 4;
  a.S = draft_splits(B, a.R, V, vec, num_sms);
  a.tok = tok; a.conf = conf; a.stats = stats;
  a.ws = reinterpret_cast<unsigned char *>(ws);
  a.status = status;
  return dtype == EAGLE_BF16 ? launch_t<__nv_bfloat16>(a, st) : launch_t<float>(a, st);
}

}  // namespace eagle
