// Stage 3 (CUDA-core path): tree-masked attention of the tree nodes over the
// KV prefix, plus the split-KV combine shared with the tensor-core path.
//
// [EAGLE-1] sections "用語解説" (Tree Attention) and "Tree Attention の役割":
// every branch of the draft tree is scored in one forward pass; with the
// [EAGLE-2] mask (section "注意マスクの調整") node i attends to the prefix and
// to its own ancestors only.
//
// This path serves fp32 inputs and is the plain reference for the tcgen05
// path: a warp owns one query row at a time, its lanes split the head
// dimension, and each key is folded into an online softmax.  The key range
// [0, kv_len[b] + n) (prefix, then tree nodes) may be split over S CTAs whose
// partial (acc, max, sum) triples are merged by attn_combine_kernel.
#include "common.cuh"

namespace eagle {

struct AttnArgs {
  const void *q, *k_cache, *v_cache, *k_tree, *v_tree;
  const int32_t *kv_len;
  const uint64_t *mask;
  int B, n, Hq, Hkv, dh, Lmax, S, W;
  float scale;
  void *out;
  float *lse;
  float *part_o;   // [B, Hq, S, n, dh]
  float *part_ml;  // [B, Hq, S, n, 2]
};

template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

template <typename T, int DH>
__global__ void __launch_bounds__(128) tree_attn_simt_kernel(AttnArgs a) {
  constexpr int PER = DH / 32;
  const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.Hq / a.Hkv, g = h / G;
  const int L = min(max(a.kv_len[b], 0), a.Lmax);  // lengths beyond the cache are clamped
  const int total = L + a.n;
  const int chunk = (total + a.S - 1) / a.S;
  const int k0 = s * chunk, k1 = min(total, k0 + chunk);
  const T *q = reinterpret_cast<const T *>(a.q);
  const T *kc = reinterpret_cast<const T *>(a.k_cache) + (static_cast<int64_t>(b) * a.Hkv + g) * a.Lmax * DH;
  const T *vc = reinterpret_cast<const T *>(a.v_cache) + (static_cast<int64_t>(b) * a.Hkv + g) * a.Lmax * DH;
  const T *kt = reinterpret_cast<const T *>(a.k_tree) + (static_cast<int64_t>(b) * a.Hkv + g) * a.n * DH;
  const T *vt = reinterpret_cast<const T *>(a.v_tree) + (static_cast<int64_t>(b) * a.Hkv + g) * a.n * DH;

  for (int i = warp; i < a.n; i += 4) {
    float qv[PER], acc[PER];
    const T *qrow = q + ((static_cast<int64_t>(b) * a.n + i) * a.Hq + h) * DH;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      qv[e] = to_f(qrow[lane * PER + e]) * a.scale;
      acc[e] = 0.f;
    }
    const uint64_t *mrow = a.mask + (static_cast<int64_t>(b) * a.n + i) * a.W;
    float m = -INFINITY, l = 0.f;
    for (int j = k0; j < k1; ++j) {
      const T *kr, *vr;
      if (j < L) {
        kr = kc + static_cast<int64_t>(j) * DH;
        vr = vc + static_cast<int64_t>(j) * DH;
      } else {
        const int t = j - L;
        if (!((mrow[t >> 6] >> (t & 63)) & 1ull)) continue;
        kr = kt + static_cast<int64_t>(t) * DH;
        vr = vt + static_cast<int64_t>(t) * DH;
      }
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < PER; ++e) dot = fmaf(qv[e], to_f(kr[lane * PER + e]), dot);
      dot = warp_sum(dot);
      if (dot > m) {
        const float corr = expf(m - dot);
        l = l * corr + 1.f;
#pragma unroll
        for (int e = 0; e < PER; ++e) acc[e] = fmaf(acc[e], corr, to_f(vr[lane * PER + e]));
        m = dot;
      } else {
        const float p = expf(dot - m);
        l += p;
#pragma unroll
        for (int e = 0; e < PER; ++e) acc[e] = fmaf(p, to_f(vr[lane * PER + e]), acc[e]);
      }
    }
    const int64_t orow = (static_cast<int64_t>(b) * a.n + i) * a.Hq + h;
    if (a.S == 1) {
      T *o = reinterpret_cast<T *>(a.out) + orow * DH;
      const float inv = 1.f / l;
#pragma unroll
      for (int e = 0; e < PER; ++e) o[lane * PER + e] = from_f<T>(acc[e] * inv);
      if (lane == 0 && a.lse) a.lse[orow] = m + logf(l);
    } else {
      const int64_t prow = ((static_cast<int64_t>(b) * a.Hq + h) * a.S + s) * a.n + i;
#pragma unroll
      for (int e = 0; e < PER; ++e) a.part_o[prow * DH + lane * PER + e] = acc[e];
      if (lane == 0) {
        a.part_ml[prow * 2 + 0] = m;
        a.part_ml[prow * 2 + 1] = l;
      }
    }
  }
}

// Merge S partial (acc, m, l) triples per (b, i, h): one warp per output row.
template <typename T, int DH>
__global__ void __launch_bounds__(256) attn_combine_kernel(AttnArgs a) {
  constexpr int PER = DH / 32;
  const int64_t rowid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t nrows = static_cast<int64_t>(a.B) * a.n * a.Hq;
  if (rowid >= nrows) return;
  const int h = static_cast<int>(rowid % a.Hq);
  const int i = static_cast<int>((rowid / a.Hq) % a.n);
  const int b = static_cast<int>(rowid / (static_cast<int64_t>(a.Hq) * a.n));
  const int64_t pbase = (static_cast<int64_t>(b) * a.Hq + h) * a.S * a.n + i;
  float M = -INFINITY;
  for (int s = 0; s < a.S; ++s) M = fmaxf(M, a.part_ml[(pbase + static_cast<int64_t>(s) * a.n) * 2]);
  float Lsum = 0.f, acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  for (int s = 0; s < a.S; ++s) {
    const int64_t pr = pbase + static_cast<int64_t>(s) * a.n;
    const float ms = a.part_ml[pr * 2], ls = a.part_ml[pr * 2 + 1];
    if (ms == -INFINITY) continue;
    const float w = expf(ms - M);
    Lsum += ls * w;
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = fmaf(a.part_o[pr * DH + lane * PER + e], w, acc[e]);
  }
  T *o = reinterpret_cast<T *>(a.out) + rowid * DH;
  const float inv = 1.f / Lsum;
#pragma unroll
  for (int e = 0; e < PER; ++e) o[lane * PER + e] = from_f<T>(acc[e] * inv);
  if (lane == 0 && a.lse) a.lse[rowid] = M + logf(Lsum);
}

// ---- host side ---------------------------------------------------------------

int attn_simt_splits(int B, int Hq, int n, int Lmax, int num_sms) {
  const int64_t ctas = static_cast<int64_t>(B) * Hq;
  int64_t S = (static_cast<int64_t>(num_sms) * 4 + ctas - 1) / ctas;
  const int64_t by_len = (Lmax + n) / 256;
  if (S > by_len) S = by_len;
  if (S > 64) S = 64;
  if (S < 1) S = 1;
  return static_cast<int>(S);
}

size_t attn_simt_workspace_bytes(int B, int n, int Hq, int dh, int Lmax, int num_sms) {
  const int S = attn_simt_splits(B, Hq, n, Lmax, num_sms);
  if (S == 1) return 0;
  return sizeof(float) * static_cast<size_t>(B) * Hq * S * n * (dh + 2);
}

template <typename T, int DH>
static cudaError_t launch_simt_t(AttnArgs a, cudaStream_t st) {
  dim3 grid(a.S, a.Hq, a.B);
  tree_attn_simt_kernel<T, DH><<<grid, 128, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || a.S == 1) return e;
  const int64_t rows = static_cast<int64_t>(a.B) * a.n * a.Hq;
  attn_combine_kernel<T, DH><<<static_cast<int>((rows * 32 + 255) / 256), 256, 0, st>>>(a);
  return cudaGetLastError();
}

// Split-KV merge for the tensor-core path (bf16 output, same partial layout).
cudaError_t launch_attn_combine_bf16(const float *part_o, const float *part_ml, int B, int n, int Hq, int dh,
                                     int S, void *out, float *lse, cudaStream_t st) {
  AttnArgs a = {};
  a.B = B; a.n = n; a.Hq = Hq; a.dh = dh; a.S = S;
  a.out = out; a.lse = lse;
  a.part_o = const_cast<float *>(part_o);
  a.part_ml = const_cast<float *>(part_ml);
  const int64_t rows = static_cast<int64_t>(B) * n * Hq;
  const int grid = static_cast<int>((rows * 32 + 255) / 256);
  if (dh == 64)
    attn_combine_kernel<__nv_bfloat16, 64><<<grid, 256, 0, st>>>(a);
  else
    attn_combine_kernel<__nv_bfloat16, 128><<<grid, 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_tree_attn_simt(const void *q, const void *k_cache, const void *v_cache,
                                  const int32_t *kv_len, const void *k_tree, const void *v_tree,
                                  const uint64_t *mask, int dtype, int B, int n, int Hq, int Hkv,
                                  int dh, int Lmax, float scale, void *out, float *lse, void *ws,
                                  int num_sms, cudaStream_t st) {
  AttnArgs a;
  a.q = q; a.k_cache = k_cache; a.v_cache = v_cache; a.k_tree = k_tree; a.v_tree = v_tree;
  a.kv_len = kv_len; a.mask = mask;
  a.B = B; a.n = n; a.Hq = Hq; a.Hkv = Hkv; a.dh = dh; a.Lmax = Lmax;
  a.S = attn_simt_splits(B, Hq, n, Lmax, num_sms);
  a.W = (n + 63) / 64;
  a.scale = scale;
  a.out = out; a.lse = lse;
  a.part_o = reinterpret_cast<float *>(ws);
  a.part_ml = a.part_o + static_cast<size_t>(B) * Hq * a.S * n * dh;
  if (dtype == EAGLE_BF16)
    return dh == 64 ? launch_simt_t<__nv_bfloat16, 64>(a, st) : launch_simt_t<__nv_bfloat16, 128>(a, st);
  return dh == 64 ? launch_simt_t<float, 64>(a, st) : launch_simt_t<float, 128>(a, st);
}

}  // namespace eagle
