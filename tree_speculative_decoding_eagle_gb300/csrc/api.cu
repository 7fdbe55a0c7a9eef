// C ABI of the library: argument validation, workspace sizing and dispatch
// to the stage kernels.  Every entry point returns an eagle_status and never
// throws, allocates or synchronises.
#include <cuda_runtime.h>

#include "common.cuh"

namespace eagle {
// draft_topk.cu
size_t draft_workspace_bytes(int B, int D, int k, int V, int vec, int num_sms);
cudaError_t launch_draft_topk(const void *logits, int dtype, int B, int D, int k, int V, int64_t ld,
                              int32_t *tok, float *conf, float *stats, void *ws, int32_t *status,
                              int num_sms, cudaStream_t st);
// tree_build.cu
cudaError_t launch_tree_build(const int32_t *tok, const float *conf, int B, int D, int k, int m, int flags,
                              const int32_t *root_tok, int32_t *node_tok, int32_t *node_parent,
                              int32_t *node_depth, float *node_score, int32_t *node_src,
                              int32_t *node_row, uint64_t *mask, int32_t *status, cudaStream_t st);
cudaError_t launch_tree_mask(const int32_t *parent, int B, int n, uint64_t *mask, cudaStream_t st);
// verify_draft.cu
cudaError_t launch_verify_draft(const void *target, const void *draft, int dtype, int64_t ld_t, int64_t ld_d,
                                const int32_t *node_tok, const int32_t *node_parent, const int32_t *node_row,
                                int B, int m, int D, int k, int V, float temperature, const float *uniforms,
                                int32_t *accept_len, int32_t *path_nodes, int32_t *out_tokens, int32_t *status,
                                cudaStream_t st);
// tree_attn_tc.cu (paged prefix)
cudaError_t launch_tree_attn_tc_paged(const void *q, const void *k_pages, const void *v_pages,
                                      const int32_t *block_table, int max_pages, int page_size, int num_pages,
                                      const int32_t *kv_len, const void *k_tree, const void *v_tree,
                                      const uint64_t *mask, int B, int n, int Hq, int Hkv, int dh, float scale,
                                      void *out, float *lse, void *ws, int32_t *status, int num_sms,
                                      cudaStream_t st);
// kv_commit.cu
cudaError_t launch_kv_commit(const void *k_tree, const void *v_tree, int dtype, int B, int n, int Hkv, int dh,
                             const int32_t *accept_len, const int32_t *path_nodes, int D, void *k_cache,
                             void *v_cache, int Lmax, const int32_t *block_table, int max_pages, int page_size,
                             int num_pages, int32_t *kv_len, int32_t *slot_mapping, int32_t *status,
                             cudaStream_t st);
// static_tree.cu
cudaError_t launch_static_tree(const int32_t *tok, const float *conf, int B, int D, int k, const int32_t *parent,
                               const int32_t *rank, int n, const int32_t *root_tok, int32_t *node_tok,
                               int32_t *node_parent, int32_t *node_depth, float *node_score, int32_t *node_src,
                               int32_t *node_row, uint64_t *mask, int32_t *status, cudaStream_t st);
size_t tree_smem_bytes(int D, int k, int m, int flags);
// tree_attn_simt.cu / tree_attn_tc.cu
size_t attn_simt_workspace_bytes(int B, int n, int Hq, int dh, int Lmax, int num_sms);
cudaError_t launch_tree_attn_simt(const void *q, const void *k_cache, const void *v_cache,
                                  const int32_t *kv_len, const void *k_tree, const void *v_tree,
                                  const uint64_t *mask, int dtype, int B, int n, int Hq, int Hkv,
                                  int dh, int Lmax, float scale, void *out, float *lse, void *ws,
                                  int num_sms, cudaStream_t st);
size_t attn_tc_workspace_bytes(int B, int n, int Hq, int Hkv, int dh, int Lmax, int num_sms);
int attn_tc_kernel_count(int B, int n, int Hq, int Hkv, int dh, int Lmax, int num_sms);
cudaError_t launch_tree_attn_tc(const void *q, const void *k_cache, const void *v_cache, const int32_t *kv_len,
                                const void *k_tree, const void *v_tree, const uint64_t *mask, int B, int n,
                                int Hq, int Hkv, int dh, int Lmax, float scale, void *out, float *lse, void *ws,
                                int32_t *status, int num_sms, cudaStream_t st);
// verify.cu
size_t verify_workspace_bytes(int B, int m, int V);
cudaError_t launch_verify(const void *target, int dtype, int64_t ld, const int32_t *node_tok,
                          const int32_t *node_parent, int B, int m, int D, int V, int mode,
                          float temperature, const float *u, int32_t *accept_len,
                          int32_t *path_nodes, int32_t *out_tokens, int32_t *status, void *ws,
                          int num_sms, cudaStream_t st);

// SM count of the current device (queried once per device).
int current_num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      sms = 148;
    cached[dev] = sms;
  }
  return cached[dev];
}

static inline int elem_size(int dtype) { return dtype == EAGLE_BF16 ? 2 : 4; }
static inline bool valid_dtype(int dtype) { return dtype == EAGLE_F32 || dtype == EAGLE_BF16; }
static inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static inline int from_cuda(cudaError_t e) { return e == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA; }

}  // namespace eagle

using namespace eagle;

extern "C" {

const char *eagle_status_string(int code) {
  switch (code) {
    case EAGLE_OK: return "ok";
    case EAGLE_ERR_INVALID: return "invalid argument";
    case EAGLE_ERR_UNSUPPORTED: return "unsupported configuration";
    case EAGLE_ERR_CUDA: return "CUDA error";
    case EAGLE_ERR_WORKSPACE: return "workspace too small";
    case EAGLE_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

int eagle_version(void) { return 100; }

size_t eagle_draft_topk_workspace_size(int B, int D, int k, int V) {
  if (B < 1 || D < 1 || k < 1 || V < 1) return 0;
  // the split count depends on the vector width; take the larger of the two
  size_t a = draft_workspace_bytes(B, D, k, V, 8, current_num_sms());
  size_t b = draft_workspace_bytes(B, D, k, V, 4, current_num_sms());
  return a > b ? a : b;
}

int eagle_draft_topk(const void *logits, int dtype, int B, int D, int k, int V, int64_t ld,
                     int32_t *tok, float *conf, float *stats, int32_t *status, void *workspace,
                     size_t workspace_bytes, eagle_stream_t stream) {
  if (!logits || !tok || !conf || !valid_dtype(dtype)) return EAGLE_ERR_INVALID;
  if (B < 1 || D < 1 || k < 1 || k > 32 || V < 1 || k > V || ld < V) return EAGLE_ERR_INVALID;
  const int es = elem_size(dtype);
  if ((static_cast<int64_t>(V) * es) % 16 || (ld * es) % 16 || !aligned16(logits)) return EAGLE_ERR_INVALID;
  if (static_cast<int64_t>(B) * (1 + (D - 1) * k) > 65535) return EAGLE_ERR_UNSUPPORTED;
  const int sms = current_num_sms();
  const size_t need = draft_workspace_bytes(B, D, k, V, 16 / es, sms);
  if (workspace_bytes < need || (need && !workspace)) return EAGLE_ERR_WORKSPACE;
  return from_cuda(launch_draft_topk(logits, dtype, B, D, k, V, ld, tok, conf, stats, workspace,
                                     status, sms, reinterpret_cast<cudaStream_t>(stream)));
}

int eagle_tree_build_variant(const int32_t *tok, const float *conf, int B, int D, int k, int m, int flags,
                             const int32_t *root_tok, int32_t *node_tok, int32_t *node_parent,
                             int32_t *node_depth, float *node_score, int32_t *node_src, int32_t *node_row,
                             uint64_t *mask, int32_t *status, eagle_stream_t stream) {
  if (!tok || !conf || !node_tok || !node_parent) return EAGLE_ERR_INVALID;
  if (B < 1 || D < 1 || k < 1 || k > 32 || m < 1) return EAGLE_ERR_INVALID;
  if (flags & ~(EAGLE_TREE_CONFIDENCE_ONLY | EAGLE_TREE_NO_RERANK)) return EAGLE_ERR_INVALID;
  const int64_t NC = k + static_cast<int64_t>(D - 1) * k * k;
  if (NC > 4095 || m > NC) return EAGLE_ERR_INVALID;
  if ((flags & EAGLE_TREE_NO_RERANK) && m > static_cast<int64_t>(D) * k) return EAGLE_ERR_INVALID;
  if (tree_smem_bytes(D, k, m, flags) > 227 * 1024) return EAGLE_ERR_UNSUPPORTED;  // one CTA's shared memory
  return from_cuda(launch_tree_build(tok, conf, B, D, k, m, flags, root_tok, node_tok, node_parent,
                                     node_depth, node_score, node_src, node_row, mask, status,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

int eagle_tree_build(const int32_t *tok, const float *conf, int B, int D, int k, int m,
                     const int32_t *root_tok, int32_t *node_tok, int32_t *node_parent,
                     int32_t *node_depth, float *node_score, int32_t *node_src, int32_t *node_row,
                     uint64_t *mask, int32_t *status, eagle_stream_t stream) {
  return eagle_tree_build_variant(tok, conf, B, D, k, m, 0, root_tok, node_tok, node_parent, node_depth,
                                  node_score, node_src, node_row, mask, status, stream);
}

int eagle_static_tree(const int32_t *tok, const float *conf, int B, int D, int k, const int32_t *tree_parent,
                      const int32_t *tree_rank, int n, const int32_t *root_tok, int32_t *node_tok,
                      int32_t *node_parent, int32_t *node_depth, float *node_score, int32_t *node_src,
                      int32_t *node_row, uint64_t *mask, int32_t *status, eagle_stream_t stream) {
  if (!tok || !conf || !tree_parent || !tree_rank || !node_tok || !node_parent) return EAGLE_ERR_INVALID;
  if (B < 1 || D < 1 || D > 32 || k < 1 || k > 32 || n < 1 || n > 1024) return EAGLE_ERR_INVALID;
  return from_cuda(launch_static_tree(tok, conf, B, D, k, tree_parent, tree_rank, n, root_tok, node_tok,
                                      node_parent, node_depth, node_score, node_src, node_row, mask, status,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

int eagle_tree_mask(const int32_t *node_parent, int B, int n, uint64_t *mask, eagle_stream_t stream) {
  if (!node_parent || !mask || B < 1 || n < 1 || n > 4096) return EAGLE_ERR_INVALID;
  return from_cuda(launch_tree_mask(node_parent, B, n, mask, reinterpret_cast<cudaStream_t>(stream)));
}

size_t eagle_tree_attn_workspace_size(int dtype, int B, int n, int Hq, int Hkv, int dh, int Lmax) {
  if (B < 1 || n < 1 || Hq < 1 || Hkv < 1 || dh < 1 || Lmax < 0) return 0;
  if (dtype == EAGLE_BF16) return attn_tc_workspace_bytes(B, n, Hq, Hkv, dh, Lmax, current_num_sms());
  return attn_simt_workspace_bytes(B, n, Hq, dh, Lmax, current_num_sms());
}

int eagle_tree_attn_kernel_count(int dtype, int B, int n, int Hq, int Hkv, int dh, int Lmax) {
  if (!valid_dtype(dtype) || B < 1 || n < 1 || Hq < 1 || Hkv < 1 || dh < 1 || Lmax < 0) return 0;
  if (dtype == EAGLE_BF16) return attn_tc_kernel_count(B, n, Hq, Hkv, dh, Lmax, current_num_sms());
  // fp32: a split prefix adds the combine kernel (it asks for a workspace)
  return attn_simt_workspace_bytes(B, n, Hq, dh, Lmax, current_num_sms()) > 0 ? 2 : 1;
}

int eagle_tree_attn(const void *q, const void *k_cache, const void *v_cache, const int32_t *kv_len,
                    const void *k_tree, const void *v_tree, const uint64_t *mask, int dtype, int B,
                    int n, int Hq, int Hkv, int dh, int Lmax, float scale, void *out, float *lse,
                    int32_t *status, void *workspace, size_t workspace_bytes, eagle_stream_t stream) {
  if (!q || !k_cache || !v_cache || !kv_len || !k_tree || !v_tree || !mask || !out) return EAGLE_ERR_INVALID;
  if (!valid_dtype(dtype) || B < 1 || n < 1 || n > 4096 || Hq < 1 || Hkv < 1 || Hq % Hkv || Lmax < 0)
    return EAGLE_ERR_INVALID;
  if (dh != 64 && dh != 128) return EAGLE_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(B) * Hkv > 65535) return EAGLE_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_tree) ||
      !aligned16(v_tree) || !aligned16(out))
    return EAGLE_ERR_INVALID;
  const int sms = current_num_sms();
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == EAGLE_BF16) {
    const size_t need = attn_tc_workspace_bytes(B, n, Hq, Hkv, dh, Lmax, sms);
    if (workspace_bytes < need || (need && !workspace)) return EAGLE_ERR_WORKSPACE;
    return from_cuda(launch_tree_attn_tc(q, k_cache, v_cache, kv_len, k_tree, v_tree, mask, B, n, Hq, Hkv, dh,
                                         Lmax, scale, out, lse, workspace, status, sms, st));
  }
  const size_t need = attn_simt_workspace_bytes(B, n, Hq, dh, Lmax, sms);
  if (workspace_bytes < need || (need && !workspace)) return EAGLE_ERR_WORKSPACE;
  return from_cuda(launch_tree_attn_simt(q, k_cache, v_cache, kv_len, k_tree, v_tree, mask, dtype, B, n, Hq,
                                         Hkv, dh, Lmax, scale, out, lse, workspace, sms, st));
}

static bool valid_pages(int max_pages, int page_size, int num_pages) {
  return max_pages >= 1 && num_pages >= 1 && page_size >= 16 && page_size <= 4096 &&
         (page_size & (page_size - 1)) == 0 && static_cast<int64_t>(max_pages) * page_size <= (1 << 24);
}

size_t eagle_tree_attn_paged_workspace_size(int dtype, int B, int n, int Hq, int Hkv, int dh, int max_pages,
                                            int page_size) {
  if (dtype != EAGLE_BF16 || B < 1 || n < 1 || Hq < 1 || Hkv < 1 || dh < 1 || max_pages < 1 || page_size < 1)
    return 0;
  return attn_tc_workspace_bytes(B, n, Hq, Hkv, dh, max_pages * page_size, current_num_sms());
}

int eagle_tree_attn_paged(const void *q, const void *k_pages, const void *v_pages, const int32_t *block_table,
                          int max_pages, int page_size, int num_pages, const int32_t *kv_len, const void *k_tree,
                          const void *v_tree, const uint64_t *mask, int dtype, int B, int n, int Hq, int Hkv,
                          int dh, float scale, void *out, float *lse, int32_t *status, void *workspace,
                          size_t workspace_bytes, eagle_stream_t stream) {
  if (!q || !k_pages || !v_pages || !block_table || !kv_len || !k_tree || !v_tree || !mask || !out)
    return EAGLE_ERR_INVALID;
  if (!valid_dtype(dtype) || B < 1 || n < 1 || n > 4096 || Hq < 1 || Hkv < 1 || Hq % Hkv ||
      !valid_pages(max_pages, page_size, num_pages))
    return EAGLE_ERR_INVALID;
  if (dtype != EAGLE_BF16 || (dh != 64 && dh != 128)) return EAGLE_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(B) * Hkv > 65535) return EAGLE_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(k_tree) || !aligned16(v_tree) ||
      !aligned16(out))
    return EAGLE_ERR_INVALID;
  const int sms = current_num_sms();
  const size_t need = attn_tc_workspace_bytes(B, n, Hq, Hkv, dh, max_pages * page_size, sms);
  if (workspace_bytes < need || (need && !workspace)) return EAGLE_ERR_WORKSPACE;
  return from_cuda(launch_tree_attn_tc_paged(q, k_pages, v_pages, block_table, max_pages, page_size, num_pages,
                                             kv_len, k_tree, v_tree, mask, B, n, Hq, Hkv, dh, scale, out, lse,
                                             workspace, status, sms, reinterpret_cast<cudaStream_t>(stream)));
}

int eagle_kv_commit(const void *k_tree, const void *v_tree, int dtype, int B, int n, int Hkv, int dh,
                    const int32_t *accept_len, const int32_t *path_nodes, int D, void *k_cache, void *v_cache,
                    int Lmax, const int32_t *block_table, int max_pages, int page_size, int num_pages,
                    int32_t *kv_len, int32_t *slot_mapping, int32_t *status, eagle_stream_t stream) {
  if (!k_tree || !v_tree || !accept_len || !path_nodes || !k_cache || !v_cache || !kv_len) return EAGLE_ERR_INVALID;
  if (!valid_dtype(dtype) || B < 1 || n < 1 || n > 4096 || Hkv < 1 || dh < 1 || D < 1 || D > 64)
    return EAGLE_ERR_INVALID;
  if ((dh * elem_size(dtype)) % 16) return EAGLE_ERR_INVALID;
  if (block_table ? !valid_pages(max_pages, page_size, num_pages) : Lmax < 1) return EAGLE_ERR_INVALID;
  if (!aligned16(k_tree) || !aligned16(v_tree) || !aligned16(k_cache) || !aligned16(v_cache))
    return EAGLE_ERR_INVALID;
  return from_cuda(launch_kv_commit(k_tree, v_tree, dtype, B, n, Hkv, dh, accept_len, path_nodes, D, k_cache,
                                    v_cache, Lmax, block_table, max_pages, page_size, num_pages, kv_len,
                                    slot_mapping, status, reinterpret_cast<cudaStream_t>(stream)));
}

size_t eagle_verify_workspace_size(int B, int m, int V) {
  if (B < 1 || m < 0 || V < 1) return 0;
  return verify_workspace_bytes(B, m, V);
}

int eagle_verify(const void *target, int dtype, int64_t ld, const int32_t *node_tok,
                 const int32_t *node_parent, int B, int m, int D, int V, int mode, float temperature,
                 const float *uniforms, int32_t *accept_len, int32_t *path_nodes,
                 int32_t *out_tokens, int32_t *status, void *workspace, size_t workspace_bytes,
                 eagle_stream_t stream) {
  if (!target || !node_tok || !node_parent || !accept_len || !path_nodes || !out_tokens)
    return EAGLE_ERR_INVALID;
  if (!valid_dtype(dtype) || B < 1 || m < 0 || m + 1 > 4096 || D < 1 || V < 1 || ld < V)
    return EAGLE_ERR_INVALID;
  if (mode != EAGLE_GREEDY && mode != EAGLE_SAMPLE) return EAGLE_ERR_INVALID;
  if (mode == EAGLE_SAMPLE && (!uniforms || !(temperature > 0.f))) return EAGLE_ERR_INVALID;
  const int es = elem_size(dtype);
  if ((static_cast<int64_t>(V) * es) % 16 || (ld * es) % 16 || !aligned16(target)) return EAGLE_ERR_INVALID;
  const size_t need = verify_workspace_bytes(B, m, V);
  if (workspace_bytes < need || !workspace) return EAGLE_ERR_WORKSPACE;
  return from_cuda(launch_verify(target, dtype, ld, node_tok, node_parent, B, m, D, V, mode,
                                 temperature, uniforms, accept_len, path_nodes, out_tokens, status,
                                 workspace, current_num_sms(), reinterpret_cast<cudaStream_t>(stream)));
}

int eagle_verify_draft(const void *target, const void *draft, int dtype, int64_t ld_t, int64_t ld_d,
                       const int32_t *node_tok, const int32_t *node_parent, const int32_t *node_row, int B,
                       int m, int D, int k, int V, float temperature, const float *uniforms,
                       int32_t *accept_len, int32_t *path_nodes, int32_t *out_tokens, int32_t *status,
                       eagle_stream_t stream) {
  if (!target || !draft || !node_tok || !node_parent || !node_row || !uniforms || !accept_len || !path_nodes ||
      !out_tokens)
    return EAGLE_ERR_INVALID;
  if (!valid_dtype(dtype) || B < 1 || m < 0 || m + 1 > 4096 || D < 1 || k < 1 || k > 32 || V < 1)
    return EAGLE_ERR_INVALID;
  if (ld_t < V || ld_d < V || !(temperature > 0.f)) return EAGLE_ERR_INVALID;
  const int es = elem_size(dtype);
  if ((static_cast<int64_t>(V) * es) % 16 || (ld_t * es) % 16 || (ld_d * es) % 16 || !aligned16(target) ||
      !aligned16(draft))
    return EAGLE_ERR_INVALID;
  if (B > 65535) return EAGLE_ERR_UNSUPPORTED;  // sequences index the grid's y dimension
  return from_cuda(launch_verify_draft(target, draft, dtype, ld_t, ld_d, node_tok, node_parent, node_row, B, m,
                                       D, k, V, temperature, uniforms, accept_len, path_nodes, out_tokens, status,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
