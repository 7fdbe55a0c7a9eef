// The whole step through the C ABI: the four stage calls in the method's
// order on one stream (eagle_step), and the same calls recorded once into a
// CUDA graph and replayed (eagle_step_graph_*).  Host code only: every
// kernel is the stages' own, launched by their entry points.
#include <cuda_runtime.h>

#include <new>

#include "eagle.h"

namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// The stages' workspace sizes, in the step workspace's order: draft, attention, verify.
bool stage_sizes(const eagle_step_args *a, size_t sz[3]) {
  if (!a || a->B < 1 || a->D < 1 || a->k < 1 || a->m < 1 || a->V < 1) return false;
  sz[0] = eagle_draft_topk_workspace_size(a->B, a->D, a->k, a->V);
  sz[1] = eagle_tree_attn_workspace_size(a->dtype, a->B, a->m + 1, a->Hq, a->Hkv, a->dh, a->Lmax);
  sz[2] = eagle_verify_workspace_size(a->B, a->m, a->V);
  return sz[2] != 0;  // verification always needs its records
}

unsigned char *piece(void *ws, size_t off, size_t bytes) {
  return bytes ? static_cast<unsigned char *>(ws) + off : nullptr;
}

}  // namespace

struct eagle_step_graph_s {
  cudaGraphExec_t exec;
};

extern "C" {

size_t eagle_step_workspace_size(const eagle_step_args *a) {
  size_t sz[3];
  if (!stage_sizes(a, sz)) return 0;
  return round_up(sz[0]) + round_up(sz[1]) + round_up(sz[2]);
}

int eagle_step(const eagle_step_args *a, void *ws, size_t ws_bytes, eagle_stream_t stream) {
  size_t sz[3];
  if (!stage_sizes(a, sz) || !a->mask) return EAGLE_ERR_INVALID;
  const size_t off_a = round_up(sz[0]), off_v = off_a + round_up(sz[1]);
  if (!ws || ws_bytes < off_v + round_up(sz[2])) return EAGLE_ERR_WORKSPACE;
  const int n = a->m + 1;
  int rc = eagle_draft_topk(a->draft_logits, a->dtype, a->B, a->D, a->k, a->V, a->draft_ld, a->tok, a->conf,
                            a->stats, a->status, piece(ws, 0, sz[0]), sz[0], stream);
  if (rc != EAGLE_OK) return rc;
  rc = eagle_tree_build(a->tok, a->conf, a->B, a->D, a->k, a->m, a->root_tok, a->node_tok, a->node_parent,
                        a->node_depth, a->node_score, a->node_src, a->node_row, a->mask, a->status, stream);
  if (rc != EAGLE_OK) return rc;
  rc = eagle_tree_attn(a->q, a->k_cache, a->v_cache, a->kv_len, a->k_tree, a->v_tree, a->mask, a->dtype, a->B, n,
                       a->Hq, a->Hkv, a->dh, a->Lmax, a->scale, a->attn_out, a->lse, a->status,
                       piece(ws, off_a, sz[1]), sz[1], stream);
  if (rc != EAGLE_OK) return rc;
  return eagle_verify(a->target, a->dtype, a->target_ld, a->node_tok, a->node_parent, a->B, a->m, a->D, a->V,
                      a->mode, a->temperature, a->uniforms, a->accept_len, a->path_nodes, a->out_tokens,
                      a->status, piece(ws, off_v, sz[2]), sz[2], stream);
}

int eagle_step_graph_create(const eagle_step_args *a, void *ws, size_t ws_bytes, eagle_step_graph_t *graph) {
  if (!graph) return EAGLE_ERR_INVALID;
  *graph = nullptr;
  cudaStream_t s = nullptr;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return EAGLE_ERR_CUDA;
  // one plain run: argument errors surface here, and each kernel's one-time
  // set-up (its shared-memory limit) happens outside the recording
  int rc = eagle_step(a, ws, ws_bytes, reinterpret_cast<eagle_stream_t>(s));
  if (rc == EAGLE_OK && cudaStreamSynchronize(s) != cudaSuccess) rc = EAGLE_ERR_CUDA;
  if (rc != EAGLE_OK) {
    cudaStreamDestroy(s);
    return rc;
  }
  if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaStreamDestroy(s);
    return EAGLE_ERR_CUDA;
  }
  rc = eagle_step(a, ws, ws_bytes, reinterpret_cast<eagle_stream_t>(s));
  cudaGraph_t g = nullptr;
  const cudaError_t ce = cudaStreamEndCapture(s, &g);
  cudaStreamDestroy(s);
  if (rc == EAGLE_OK && (ce != cudaSuccess || !g)) rc = EAGLE_ERR_CUDA;
  cudaGraphExec_t exec = nullptr;
  if (rc == EAGLE_OK && cudaGraphInstantiate(&exec, g, 0) != cudaSuccess) rc = EAGLE_ERR_CUDA;
  if (g) cudaGraphDestroy(g);
  if (rc != EAGLE_OK) return rc;
  eagle_step_graph_s *h = new (std::nothrow) eagle_step_graph_s{exec};
  if (!h) {
    cudaGraphExecDestroy(exec);
    return EAGLE_ERR_CUDA;
  }
  *graph = h;
  return EAGLE_OK;
}

int eagle_step_graph_launch(eagle_step_graph_t graph, eagle_stream_t stream) {
  if (!graph) return EAGLE_ERR_INVALID;
  return cudaGraphLaunch(graph->exec, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? EAGLE_OK
                                                                                             : EAGLE_ERR_CUDA;
}

int eagle_step_graph_destroy(eagle_step_graph_t graph) {
  if (!graph) return EAGLE_OK;
  const cudaError_t e = cudaGraphExecDestroy(graph->exec);
  delete graph;
  return e == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}

}  // extern "C"
