// Stage 1: per-row softmax statistics and top-k of the draft logits.
//
// [EAGLE-2] section "ドラフトモデルのキャリブレーション": the confidence of a
// draft token is the probability the draft model assigns to it.  For every
// used row: M = max, Z = sum exp(x - M), the k largest logits (ties -> lower
// token id) and c = exp(x - M) / Z.
//
// One pass over HBM.  A row may be split across S CTAs (to fill the GPU when
// there are few rows); each CTA streams its slice with 16-byte vector loads,
// keeps an online (max, sum-exp) pair and a per-thread top-K list of unique
// 64-bit keys (logit order, then lower token id), merges them warp-wide with
// bitonic shuffles and block-wide through shared memory.  With S > 1 the last
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
};

constexpr int kDraftThreads = 256;
constexpr int kDraftUnroll = 4;

template <int K>
struct alignas(16) DraftPartial {
  float m, s;
  uint32_t pad[2];
  uint64_t keys[K];
};

__host__ __device__ inline size_t draft_counter_bytes(int B, int R) {
  return (static_cast<size_t>(B) * R * sizeof(uint32_t) + 255) / 256 * 256;
}

template <int K>
__device__ __forceinline__ float list_floor(const uint64_t (&list)[K]) {
  return list[K - 1] ? key_value(list[K - 1]) : -INFINITY;
}

// Write the k best keys of a finished row (all lanes of the calling warp hold
// the same descending list).
template <int K>
__device__ __forceinline__ void draft_finalize(const DraftArgs &a, int b, int d, int j,
                                               const uint64_t (&list)[K], float M, float Z) {
  const int lane = threadIdx.x & 31;
  const int64_t slot = ((static_cast<int64_t>(b) * a.D + d) * a.k + j);
  if (lane < a.k) {
    uint64_t key = 0;
#pragma unroll
    for (int q = 0; q < K; ++q)
      if (q == lane) key = list[q];
    int32_t t = -1;
    float c = 0.f;
    if (key) {
      t = static_cast<int32_t>(key_token(key));
      c = expf(key_value(key) - M) / Z;
    }
    a.tok[slot * a.k + lane] = t;
    a.conf[slot * a.k + lane] = c;
  }
  if (lane == 0 && a.stats) {
    a.stats[slot * 2 + 0] = M;
    a.stats[slot * 2 + 1] = logf(Z);
  }
}

template <typename T, int K>
__global__ void __launch_bounds__(kDraftThreads) draft_topk_kernel(DraftArgs a) {
  using VT = VecTraits<T>;
  constexpr int VEC = VT::kElems;
  const int s = blockIdx.x;
  const int rg = blockIdx.y;  // b * R + r
  const int b = rg / a.R, r = rg % a.R;
  const int d = r == 0 ? 0 : 1 + (r - 1) / a.k;
  const int j = r == 0 ? 0 : (r - 1) % a.k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  const T *row = reinterpret_cast<const T *>(a.logits) +
                 ((static_cast<int64_t>(b) * a.D + d) * a.k + j) * a.ld;
  const int64_t NV = a.V / VEC;
  const int64_t v0 = NV * s / a.S, v1 = NV * (s + 1) / a.S;

  float m = -INFINITY, sum = 0.f;
  uint64_t list[K];
#pragma unroll
  for (int q = 0; q < K; ++q) list[q] = 0;
  float thr = -INFINITY, wthr = -INFINITY;

  for (int64_t base = v0; base < v1; base += kDraftThreads * kDraftUnroll) {
    uint4 buf[kDraftUnroll];
#pragma unroll
    for (int u = 0; u < kDraftUnroll; ++u) {
      int64_t idx = base + u * kDraftThreads + tid;
      if (idx < v1) buf[u] = ld_stream16(row + idx * VEC);
    }
#pragma unroll
    for (int u = 0; u < kDraftUnroll; ++u) {
      int64_t idx = base + u * kDraftThreads + tid;
      if (idx < v1) {
        float x[VEC];
        VT::unpack(buf[u], x);
        float vmax = x[0];
#pragma unroll
        for (int e = 1; e < VEC; ++e) vmax = fmaxf(vmax, x[e]);
        if (vmax > -INFINITY) {
          if (vmax > m) {
            sum *= ex2_approx((m - vmax) * kLog2e);
            m = vmax;
          }
          const float mL = m * kLog2e;
#pragma unroll
          for (int e = 0; e < VEC; ++e) sum += ex2_approx(fmaf(x[e], kLog2e, -mL));
          if (vmax > thr && vmax >= wthr) {
            const uint32_t t0 = static_cast<uint32_t>(idx * VEC);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
              if (x[e] > thr && x[e] >= wthr) {
                list_insert<K>(list, topk_key(x[e], t0 + e));
                thr = list_floor<K>(list);
              }
            }
          }
        }
      }
    }
    wthr = from_ordered_u32(__reduce_max_sync(0xffffffffu, ordered_u32(thr)));
  }

  // ---- warp merge -------------------------------------------------------
  warp_topk<K>(list);
  {
    float mw = warp_max(m);
    float sw = (m == -INFINITY) ? 0.f : sum * ex2_approx((m - mw) * kLog2e);
    sw = warp_sum(sw);
    m = mw;
    sum = sw;
  }
  __shared__ uint64_t s_keys[kDraftThreads / 32][K];
  __shared__ float s_m[kDraftThreads / 32], s_s[kDraftThreads / 32];
  __shared__ int s_last;
  if (lane == 0) {
    s_m[warp] = m;
    s_s[warp] = sum;
  }
  if (lane < K) {
#pragma unroll
    for (int q = 0; q < K; ++q)
      if (q == lane) s_keys[warp][q] = list[q];
  }
  __syncthreads();
  if (warp != 0) return;

  // ---- block merge (warp 0) -------------------------------------------------
  constexpr int NW = kDraftThreads / 32;
#pragma unroll
  for (int q = 0; q < K; ++q) list[q] = lane < NW ? s_keys[lane][q] : 0ull;
  warp_topk<K>(list);  // every lane ends with the block's top K
  float M = s_m[0], Z = s_s[0];
  for (int w = 1; w < NW; ++w) lse_combine(M, Z, s_m[w], s_s[w]);

  if (a.S == 1) {
    draft_finalize<K>(a, b, d, j, list, M, Z);
    return;
  }

  // ---- split rows: publish the partial, the last CTA merges ---------------
  uint32_t *counters = reinterpret_cast<uint32_t *>(a.ws);
  DraftPartial<K> *parts = reinterpret_cast<DraftPartial<K> *>(a.ws + draft_counter_bytes(a.B, a.R));
  DraftPartial<K> *mine = parts + static_cast<int64_t>(rg) * a.S + s;
  if (lane < K) {
#pragma unroll
    for (int q = 0; q < K; ++q)
      if (q == lane) mine->keys[q] = list[q];
  }
  if (lane == 0) {
    mine->m = M;
    mine->s = Z;
  }
  __threadfence();
  __syncwarp();
  if (lane == 0) s_last = (atomicAdd(counters + rg, 1u) == static_cast<uint32_t>(a.S - 1));
  __syncwarp();
  if (!s_last) return;
  __threadfence();

  const DraftPartial<K> *row_parts = parts + static_cast<int64_t>(rg) * a.S;
  float pm = -INFINITY, ps = 0.f;
  if (lane < a.S) {
#pragma unroll
    for (int q = 0; q < K; ++q) list[q] = __ldcg(reinterpret_cast<const unsigned long long *>(&row_parts[lane].keys[q]));
    pm = __ldcg(&row_parts[lane].m);
    ps = __ldcg(&row_parts[lane].s);
  } else {
#pragma unroll
    for (int q = 0; q < K; ++q) list[q] = 0;
  }
  warp_topk<K>(list);
  M = warp_max(pm);
  Z = warp_sum(pm == -INFINITY ? 0.f : ps * ex2_approx((pm - M) * kLog2e));
  draft_finalize<K>(a, b, d, j, list, M, Z);
  if (lane == 0) counters[rg] = 0;  // leave the ticket zeroed for the next call
}

// ---- host side ---------------------------------------------------------------

static int draft_kpow2(int k) {
  int K = 1;
  while (K < k) K <<= 1;
  return K;
}

int draft_splits(int B, int R, int V, int vec, int num_sms) {
  const int64_t rows = static_cast<int64_t>(B) * R;
  const int64_t NV = V / vec;
  const int64_t target = static_cast<int64_t>(num_sms) * 8;
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
  const int K = draft_kpow2(k);
  const size_t rec = 16 + 8 * static_cast<size_t>(K);
  return draft_counter_bytes(B, R) + (S > 1 ? static_cast<size_t>(B) * R * S * rec : 0);
}

template <typename T>
static cudaError_t launch_t(const DraftArgs &a, cudaStream_t st) {
  dim3 grid(a.S, a.B * a.R);
  const int K = draft_kpow2(a.k);
  switch (K) {
    case 1: draft_topk_kernel<T, 1><<<grid, kDraftThreads, 0, st>>>(a); break;
    case 2: draft_topk_kernel<T, 2><<<grid, kDraftThreads, 0, st>>>(a); break;
    case 4: draft_topk_kernel<T, 4><<<grid, kDraftThreads, 0, st>>>(a); break;
    case 8: draft_topk_kernel<T, 8><<<grid, kDraftThreads, 0, st>>>(a); break;
    case 16: draft_topk_kernel<T, 16><<<grid, kDraftThreads, 0, st>>>(a); break;
    case 32: draft_topk_kernel<T, 32><<<grid, kDraftThreads, 0, st>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_draft_topk(const void *logits, int dtype, int B, int D, int k, int V,
                              int64_t ld, int32_t *tok, float *conf, float *stats,
                              void *ws, int num_sms, cudaStream_t st) {
  DraftArgs a;
  a.logits = logits;
  a.B = B; a.D = D; a.k = k; a.V = V; a.ld = ld;
  a.R = 1 + (D - 1) * k;
  const int vec = dtype == EAGLE_BF16 ? 8 : 4;
  a.S = draft_splits(B, a.R, V, vec, num_sms);
  a.tok = tok; a.conf = conf; a.stats = stats;
  a.ws = reinterpret_cast<unsigned char *>(ws);
  return dtype == EAGLE_BF16 ? launch_t<__nv_bfloat16>(a, st) : launch_t<float>(a, st);
}

}  // namespace eagle
