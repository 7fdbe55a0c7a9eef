// Stage 2 for the EAGLE-1 static draft tree: the draft's top-k tokens placed
// on a fixed template.
//
// [EAGLE-2] sections "背景" and "EAGLE-1からの変更点": EAGLE-1 arranges its
// draft tokens on a tree shape fixed in advance and applies it to every
// input.  The template is an input: parent[i] (root -1, else < i) and
// rank[i] (node i is the rank[i]-th of its parent's top-k tokens).  The root
// uses draft row [0, 0]; the j-th node of depth d >= 1 that has children
// (node order) uses row [d, j].  Node score = float32 product of the
// confidences on the root path.  Outputs match eagle_tree_build's, so the
// attention and verification stages run on the result unchanged.
//
// One CTA per sequence.  The template is validated completely in shared
// memory before any index derived from it is used; an invalid template sets
// EAGLE_ERR_INVALID in the status word and the CTA writes nothing.
#include "common.cuh"

namespace eagle {

constexpr int kStaticThreads = 256;
constexpr int kStaticMaxDepth = 32;

struct StaticArgs {
  const int32_t *tok;
  const float *conf;
  int B, D, k, n;
  const int32_t *parent, *rank;
  const int32_t *root_tok;
  int32_t *node_tok, *node_parent, *node_depth, *node_src, *node_row;
  float *node_score;
  uint64_t *mask;
  int32_t *status;
};

__global__ void __launch_bounds__(kStaticThreads) static_tree_kernel(StaticArgs a) {
  extern __shared__ __align__(16) int sm[];
  const int n = a.n, k = a.k, D = a.D;
  int *s_par = sm;            // [n]
  int *s_rank = sm + n;       // [n]
  int *s_depth = sm + 2 * n;  // [n]
  int *s_kids = sm + 3 * n;   // [n] 1 if the node has children
  int *s_row = sm + 4 * n;    // [n] draft row slot d*k + j, root 0, else -1
  __shared__ int s_bad;
  const int b = blockIdx.x, tid = threadIdx.x;

  if (tid == 0) s_bad = 0;
  for (int i = tid; i < n; i += blockDim.x) {
    s_par[i] = a.parent[i];
    s_rank[i] = a.rank[i];
    s_kids[i] = 0;
  }
  __syncthreads();
  // structure: the root first, parents before children, ranks in [0, k)
  for (int i = tid; i < n; i += blockDim.x) {
    const int p = s_par[i];
    if (i == 0) {
      if (p != -1) s_bad = 1;
    } else if (p < 0 || p >= i || s_rank[i] < 0 || s_rank[i] >= k) {
      s_bad = 1;
    } else {
      s_kids[p] = 1;
    }
  }
  __syncthreads();
  if (s_bad) {
    if (tid == 0) report(a.status, EAGLE_ERR_INVALID);
    return;
  }
  // depths (parents precede children, so every walk ends at the root within
  // i steps) and distinct ranks among siblings
  for (int i = tid; i < n; i += blockDim.x) {
    int d = 0;
    for (int j = i; j > 0 && d <= D; j = s_par[j]) ++d;
    s_depth[i] = d;
    if (d > D || d > kStaticMaxDepth) s_bad = 1;
    for (int q = 1; q < i; ++q)
      if (s_par[q] == s_par[i] && s_rank[q] == s_rank[i] && i > 0) s_bad = 1;
  }
  __syncthreads();
  // draft rows of the nodes with children: at most k per depth, above depth D
  for (int i = tid; i < n; i += blockDim.x) {
    int row = -1;
    if (i == 0) {
      row = 0;
    } else if (s_kids[i]) {
      const int d = s_depth[i];
      int j = 0;
      for (int q = 1; q < i; ++q) j += (s_kids[q] && s_depth[q] == d) ? 1 : 0;
      if (d >= D || j >= k) s_bad = 1;
      row = d * k + j;
    }
    s_row[i] = row;
  }
  __syncthreads();
  if (s_bad) {
    if (tid == 0) report(a.status, EAGLE_ERR_INVALID);
    return;
  }

  // ---- tokens, scores and the mask ---------------------------------------
  const int32_t *tok = a.tok + static_cast<int64_t>(b) * D * k * k;
  const float *conf = a.conf + static_cast<int64_t>(b) * D * k * k;
  const int64_t ob = static_cast<int64_t>(b) * n;
  const int W = (n + 63) >> 6;
  for (int q = tid; q < n * W; q += blockDim.x) {
    const int i = q / W, w = q % W;
    if (w == 0) {
      int t = a.root_tok ? a.root_tok[b] : -1;
      float v = 1.0f;
      if (i > 0) {
        // confidences on the root path, deepest first, then multiplied from
        // the root down: V_child = fl32(V_parent * c)
        float c[kStaticMaxDepth];
        int depth = 0;
        for (int j = i; j > 0; j = s_par[j]) {
          const int slot = s_row[s_par[j]] * k + s_rank[j];
          c[depth++] = conf[slot];
          if (j == i) t = tok[slot];
        }
        for (int e = depth - 1; e >= 0; --e) v = __fadd_rn(__fmul_rn(v, c[e]), 0.0f);
      }
      a.node_tok[ob + i] = t;
      a.node_parent[ob + i] = s_par[i];
      if (a.node_depth) a.node_depth[ob + i] = s_depth[i];
      if (a.node_score) a.node_score[ob + i] = v;
      if (a.node_src) a.node_src[ob + i] = i;
      if (a.node_row) a.node_row[ob + i] = s_row[i];
    }
    if (a.mask) {
      uint64_t bits = 0;
      for (int j = i; j >= 0; j = s_par[j]) {
        if ((j >> 6) == w) bits |= 1ull << (j & 63);
        if (j == 0) break;
      }
      a.mask[(ob + i) * W + w] = bits;
    }
  }
}

cudaError_t launch_static_tree(const int32_t *tok, const float *conf, int B, int D, int k, const int32_t *parent,
                               const int32_t *rank, int n, const int32_t *root_tok, int32_t *node_tok,
                               int32_t *node_parent, int32_t *node_depth, float *node_score, int32_t *node_src,
                               int32_t *node_row, uint64_t *mask, int32_t *status, cudaStream_t st) {
  StaticArgs a;
  a.tok = tok; a.conf = conf;
  a.B = B; a.D = D; a.k = k; a.n = n;
  a.parent = parent; a.rank = rank; a.root_tok = root_tok;
  a.node_tok = node_tok; a.node_parent = node_parent; a.node_depth = node_depth;
  a.node_src = node_src; a.node_row = node_row; a.node_score = node_score;
  a.mask = mask; a.status = status;
  const size_t smem = sizeof(int) * 5 * static_cast<size_t>(n);
  if (smem > 48 * 1024) {
    static std::atomic<unsigned long long> configured{0};  // raised once per device, to the maximum
    const cudaError_t e = set_smem_limit_max_once(static_tree_kernel, configured);
    if (e != cudaSuccess) return e;
  }
  static_tree_kernel<<<B, kStaticThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace eagle
