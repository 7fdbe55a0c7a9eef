// Stage 1: per-row softmax statistics and top-k of the draft logits.
//
// [EAGLE-2] section "ドラフトモデルのキャリブレーション": the confidence of a
// draft token is the probability the draft model assigns to it.  For every
// used row: M = max, Z = sum exp(x - M), the k largest logits (ties -> lower
// token id) and c = exp(x - M) / Z.
//
// One pass over HBM.  A row may be split across S CTAs (to fill the GPU when
// there are few rows); each CTA streams its slice through a ring of shared-
// memory stages filled by bulk copies and keeps an online (max, sum-exp) pair
// per thread.  Top-k selection works on unique 64-bit keys (logit order, then
// lower token id).  Every lane tracks its running maximum; the k-th largest
// lane maximum of a warp (a 32-lane bitonic sort per chunk) bounds the top k
// from below, and the block keeps the largest such bound.  Values at or
// above the bound are appended to a per-warp shared-memory buffer by a
// ballot scan, so only about k candidates per warp survive.  Merges keep the
// code small: the k best of a set of unique keys are found by counting, for
// each key, how many keys are larger (its rank), in shared memory.  Warp lists
// merge block-wide through shared memory.  With S > 1 the last CTA of a row
// to finish (atomic ticket in the workspace) merges the S partial results;
// no CTA ever waits for another.
#include "common.cuh"
#include "sm100.cuh"

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
constexpr int kDraftUnroll = 4;                                // vectors per thread per chunk
constexpr int kDraftChunkVec = kDraftThreads * kDraftUnroll;   // 16-byte vectors per chunk
constexpr int kDraftStages = 4;                                // chunks in flight per CTA
constexpr int kDraftSmem = kDraftStages * kDraftChunkVec * 16 + 128;

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

// The warp's k best of its list wl[0..*wn) and its buffer buf[0..fill),
// written back to wl in descending order (whole warp, rank by counting).
__device__ __forceinline__ void warp_compact(uint64_t *wl, int *wn, uint64_t *buf, int fill, uint64_t *tmp,
                                             int k, int lane) {
  __syncwarp();
  const int n0 = *wn;
  const int C = n0 + fill;
  for (int i = lane; i < C; i += 32) {
    const uint64_t key = i < n0 ? wl[i] : buf[i - n0];
    const int r = rank_in(key, wl, n0) + rank_in(key, buf, fill);
    if (r < k) tmp[r] = key;
  }
  __syncwarp();
  const int nk = C < k ? C : k;
  if (lane < nk) wl[lane] = tmp[lane];
  if (lane == 0) *wn = nk;
  __syncwarp();
}

template <typename T>
__global__ void __launch_bounds__(kDraftThreads) draft_topk_kernel(DraftArgs a) {
  using VT = VecTraits<T>;
  constexpr int VEC = VT::kElems;
  constexpr int CAP = 64 * VEC;  // candidate buffer per warp (two full vector steps)
  constexpr int NW = kDraftThreads / 32;
  __shared__ uint64_t s_buf[NW][CAP];
  __shared__ uint64_t s_wl[NW][32], s_tmp[NW][32];
  __shared__ int s_wn[NW];
  __shared__ uint64_t s_top[32];
  __shared__ float s_m[NW], s_s[NW];
  __shared__ int s_last;
  __shared__ volatile int s_abort;
  __shared__ unsigned s_thr;  // block prune bound (order-preserving bits)

  const int s = blockIdx.x;
  const int rg = blockIdx.y;  // b * R + r
  const int b = rg / a.R, r = rg % a.R;
  const int d = r == 0 ? 0 : 1 + (r - 1) / a.k;
  const int j = r == 0 ? 0 : (r - 1) % a.k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = a.k;
  uint64_t *buf = s_buf[warp];
  uint64_t *wl = s_wl[warp];

  const T *row = reinterpret_cast<const T *>(a.logits) +
                 ((static_cast<int64_t>(b) * a.D + d) * a.k + j) * a.ld;
  const int64_t NV = a.V / VEC;
  const int64_t v0 = NV * s / a.S, v1 = NV * (s + 1) / a.S;
  const int n_chunks = static_cast<int>((v1 - v0 + kDraftChunkVec - 1) / kDraftChunkVec);

  // the slice streams through a ring of shared-memory stages filled by bulk
  // copies (one elected thread), so many bytes are in flight per SM
  extern __shared__ __align__(128) unsigned char dsm[];
  uint4 *stage_buf = reinterpret_cast<uint4 *>(dsm);
  uint64_t *full = reinterpret_cast<uint64_t *>(dsm + kDraftStages * kDraftChunkVec * 16);
  if (tid == 0) {
    s_abort = 0;
    s_thr = ordered_u32(-INFINITY);
    for (int q = 0; q < kDraftStages; ++q) sm100::mbar_init(&full[q], 1);
    sm100::mbar_init_fence();
  }
  if (lane == 0) s_wn[warp] = 0;
  __syncthreads();
  auto issue = [&](int c) {
    const int64_t first = v0 + static_cast<int64_t>(c) * kDraftChunkVec;
    const uint32_t nvec = static_cast<uint32_t>(min(static_cast<int64_t>(kDraftChunkVec), v1 - first));
    uint64_t *bar = &full[c % kDraftStages];
    sm100::mbar_arrive_expect_tx(bar, nvec * 16u);
    sm100::bulk_load(stage_buf + (c % kDraftStages) * kDraftChunkVec, row + first * VEC, nvec * 16u, bar);
  };
  if (tid == 0)
    for (int c = 0; c < min(kDraftStages, n_chunks); ++c) issue(c);

  float m = -INFINITY, sum = 0.f;
  float lmax = -INFINITY;  // this lane's largest value so far
  float thr = -INFINITY;   // prune bound: at least k values of the slice are >= thr
  int fill = 0;            // candidates waiting in the warp buffer
  int consumed = 0;

  for (int c = 0; c < n_chunks; ++c) {
    const int st = c % kDraftStages;
    if (!sm100::mbar_wait(&full[st], (c / kDraftStages) & 1, &s_abort)) report(a.status, EAGLE_ERR_TIMEOUT);
    const int64_t first = v0 + static_cast<int64_t>(c) * kDraftChunkVec;
    const int nvec = static_cast<int>(min(static_cast<int64_t>(kDraftChunkVec), v1 - first));
    const uint4 *src = stage_buf + st * kDraftChunkVec;
    uint4 vb[kDraftUnroll];
    float vmx[kDraftUnroll];
#pragma unroll
    for (int u = 0; u < kDraftUnroll; ++u) {
      const int iv = u * kDraftThreads + tid;
      vmx[u] = -INFINITY;
      if (iv < nvec && !s_abort) {
        vb[u] = src[iv];
        float x[VEC];
        VT::unpack(vb[u], x);
        float vmax = x[0];
#pragma unroll
        for (int e = 1; e < VEC; ++e) vmax = fmaxf(vmax, x[e]);
        vmx[u] = vmax;
        if (vmax > -INFINITY) {
          if (vmax > m) {
            sum *= ex2_approx((m - vmax) * kLog2e);
            m = vmax;
          }
          const float mL = m * kLog2e;
          float p[VEC];
#pragma unroll
          for (int e = 0; e < VEC; ++e) p[e] = ex2_approx(fmaf(x[e], kLog2e, -mL));
#pragma unroll
          for (int w2 = VEC / 2; w2 > 0; w2 >>= 1)  // pairwise within the vector
#pragma unroll
            for (int e = 0; e < w2; ++e) p[e] += p[e + w2];
          sum += p[0];
        }
        lmax = fmaxf(lmax, vmax);
      }
    }
    // Lane maxima are distinct elements, so the k-th largest of the warp's
    // lane maxima has at least k elements at or above it; so has any other
    // warp's bound and the k-th key of a full warp list.  The block keeps the
    // largest bound.
    {
      const float y = warp_sort_desc(lmax, lane);
      float tw = __shfl_sync(0xffffffffu, y, k - 1);
      if (s_wn[warp] == k) tw = fmaxf(tw, key_value(wl[k - 1]));
      if (tw > -INFINITY) atomicMax(&s_thr, ordered_u32(tw));
      thr = fmaxf(thr, fmaxf(tw, from_ordered_u32(s_thr)));
    }
#pragma unroll
    for (int u = 0; u < kDraftUnroll; ++u) {
      const int iv = u * kDraftThreads + tid;
      const bool maybe = vmx[u] > -INFINITY && vmx[u] >= thr;
      if (__any_sync(0xffffffffu, maybe)) {
        unsigned cm = 0;
        float x[VEC];
        VT::unpack(vb[u], x);
        if (maybe) {
#pragma unroll
          for (int e = 0; e < VEC; ++e)
            if (x[e] >= thr && x[e] > -INFINITY) cm |= 1u << e;
        }
        const int cnt = __popc(cm);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        const int total = __shfl_sync(0xffffffffu, incl, 31);
        if (fill + total > CAP) {
          warp_compact(wl, &s_wn[warp], buf, fill, s_tmp[warp], k, lane);
          fill = 0;
        }
        if (cm) {
          int pos = fill + incl - cnt;
          const uint32_t t0 = static_cast<uint32_t>((first + iv) * VEC);
#pragma unroll
          for (int e = 0; e < VEC; ++e)
            if ((cm >> e) & 1u) buf[pos++] = topk_key(x[e], t0 + e);
        }
        fill += total;
      }
    }
    consumed = c + 1;
    __syncthreads();  // every thread is done with this stage
    if (s_abort) break;
    if (tid == 0 && c + kDraftStages < n_chunks) issue(c + kDraftStages);
  }
  if (s_abort) {
    // drain the copies still in flight before the CTA's shared memory goes away
    if (tid == 0) {
      volatile int never = 0;
      for (int c = max(0, consumed - 1); c < min(n_chunks, consumed - 1 + kDraftStages); ++c)
        sm100::mbar_wait(&full[c % kDraftStages], (c / kDraftStages) & 1, &never, 100000000ull);
    }
    return;
  }
  if (fill > 0) warp_compact(wl, &s_wn[warp], buf, fill, s_tmp[warp], k, lane);

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

int draft_splits(int B, int R, int V, int vec, int num_sms) {
  const int64_t rows = static_cast<int64_t>(B) * R;
  const int64_t NV = V / vec;
  const int64_t target = static_cast<int64_t>(num_sms) * 2;  // two CTAs fit per SM
  int64_t S = (target + rows - 1) / rows;
  // keep at least two full vector sweeps of the block per split
  int64_t max_by_len = NV / (2 * kDraftThreads);
  if (max_by_len < 1) max_by_len = 1;
  if (S > max_by_len) S = max_by_len;
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
  static bool configured = false;  // the attribute is per function, set once
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(draft_topk_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kDraftSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  draft_topk_kernel<T><<<dim3(a.S, a.B * a.R), kDraftThreads, kDraftSmem, st>>>(a);
  return cudaGetLastError();
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
