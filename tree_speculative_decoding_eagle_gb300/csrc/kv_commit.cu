// After verification: the accepted path's keys and values join the KV cache.
//
// [EAGLE-1] section "検証方法" / [EAGLE-2]: the accepted draft tokens become
// part of the sequence and everything after a rejection is discarded.  The
// root's K/V is already the last prefix position; nodes path[1..a] are
// appended in path order at positions kv_len .. kv_len+a-1 and kv_len grows
// by a.  slot_mapping[b, i] is node i's position after the commit (root
// kv_len-1) or -1 for a node that is dropped.  The cache is either
// contiguous [B, Hkv, Lmax, dh] or paged: pages [num_pages, Hkv, P, dh] with
// block_table[b, p] the physical page of logical page p.
//
// One CTA per sequence: every thread reads kv_len[b] before the one write of
// the new length, so the length can be updated in place.  Indices and
// capacity are checked before anything is written; a violation sets
// EAGLE_ERR_INVALID and the sequence is left unchanged.
#include "common.cuh"

namespace eagle {

constexpr int kCommitThreads = 256;

struct CommitArgs {
  const unsigned char *k_tree, *v_tree;
  unsigned char *k_cache, *v_cache;
  int es, B, n, Hkv, dh, D, Lmax;
  const int32_t *accept_len, *path_nodes;
  const int32_t *block_table;
  int max_pages, page_size, num_pages;
  int32_t *kv_len, *slot_mapping, *status;
};

__global__ void __launch_bounds__(kCommitThreads) kv_commit_kernel(CommitArgs a) {
  __shared__ int s_ok;
  __shared__ int s_path[65];
  const int b = blockIdx.x, tid = threadIdx.x;
  const int L = a.kv_len[b];
  const int acc = a.accept_len[b];
  if (tid == 0) {
    int ok = acc >= 0 && acc <= a.D && acc <= 64 && L >= 1;
    for (int p = 1; ok && p <= acc; ++p) {
      const int node = a.path_nodes[static_cast<int64_t>(b) * (a.D + 1) + p];
      if (node < 1 || node >= a.n) ok = 0;
      s_path[p] = node;
      const int pos = L + p - 1;
      if (a.block_table) {
        const int lp = pos / a.page_size;
        if (lp >= a.max_pages) {
          ok = 0;
        } else {
          const int page = a.block_table[static_cast<int64_t>(b) * a.max_pages + lp];
          if (page < 0 || page >= a.num_pages) ok = 0;
        }
      } else if (pos >= a.Lmax) {
        ok = 0;
      }
    }
    s_ok = ok;
    if (!ok) report(a.status, EAGLE_ERR_INVALID);
  }
  __syncthreads();
  if (!s_ok) return;
  // rows of dh elements moved as 16-byte vectors
  const int vpr = a.dh * a.es / 16;
  const int64_t row_bytes = static_cast<int64_t>(a.dh) * a.es;
  for (int q = tid; q < acc * a.Hkv * vpr; q += blockDim.x) {
    const int p = 1 + q / (a.Hkv * vpr);
    const int g = (q / vpr) % a.Hkv;
    const int v = q % vpr;
    const int node = s_path[p];
    const int pos = L + p - 1;
    const int64_t src = ((static_cast<int64_t>(b) * a.Hkv + g) * a.n + node) * row_bytes + v * 16;
    int64_t dst;
    if (a.block_table) {
      const int page = a.block_table[static_cast<int64_t>(b) * a.max_pages + pos / a.page_size];
      dst = ((static_cast<int64_t>(page) * a.Hkv + g) * a.page_size + pos % a.page_size) * row_bytes + v * 16;
    } else {
      dst = ((static_cast<int64_t>(b) * a.Hkv + g) * a.Lmax + pos) * row_bytes + v * 16;
    }
    *reinterpret_cast<uint4 *>(a.k_cache + dst) = *reinterpret_cast<const uint4 *>(a.k_tree + src);
    *reinterpret_cast<uint4 *>(a.v_cache + dst) = *reinterpret_cast<const uint4 *>(a.v_tree + src);
  }
  if (a.slot_mapping) {
    for (int i = tid; i < a.n; i += blockDim.x) {
      int slot = i == 0 ? L - 1 : -1;
      for (int p = 1; p <= acc; ++p)
        if (s_path[p] == i) slot = L + p - 1;
      a.slot_mapping[static_cast<int64_t>(b) * a.n + i] = slot;
    }
  }
  __syncthreads();
  if (tid == 0) a.kv_len[b] = L + acc;
}

cudaError_t launch_kv_commit(const void *k_tree, const void *v_tree, int dtype, int B, int n, int Hkv, int dh,
                             const int32_t *accept_len, const int32_t *path_nodes, int D, void *k_cache,
                             void *v_cache, int Lmax, const int32_t *block_table, int max_pages, int page_size,
                             int num_pages, int32_t *kv_len, int32_t *slot_mapping, int32_t *status,
                             cudaStream_t st) {
  CommitArgs a;
  a.k_tree = reinterpret_cast<const unsigned char *>(k_tree);
  a.v_tree = reinterpret_cast<const unsigned char *>(v_tree);
  a.k_cache = reinterpret_cast<unsigned char *>(k_cache);
  a.v_cache = reinterpret_cast<unsigned char *>(v_cache);
  a.es = dtype == EAGLE_BF16 ? 2 : 4;
  a.B = B; a.n = n; a.Hkv = Hkv; a.dh = dh; a.D = D; a.Lmax = Lmax;
  a.accept_len = accept_len; a.path_nodes = path_nodes;
  a.block_table = block_table; a.max_pages = max_pages; a.page_size = page_size; a.num_pages = num_pages;
  a.kv_len = kv_len; a.slot_mapping = slot_mapping; a.status = status;
  kv_commit_kernel<<<B, kCommitThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace eagle
