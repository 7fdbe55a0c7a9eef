// eagle_draft_topk_noalloc: the draft softmax / top-k stage for callers that
// cannot hand the library any scratch memory.
//
// Some callers only ever receive input and output buffers: plugins and
// custom-op hooks of a host runtime that owns all device memory and offers
// no scratch, or processes whose device-memory budget is fixed up front and
// may not grow.  The draft stage needs no scratch: the parts of a row merge
// through the shared memory of their thread-block cluster.  This entry point
// is eagle_draft_topk without the workspace arguments; it allocates nothing
// and calls on different streams may overlap.
#include "common.cuh"

namespace eagle {

cudaError_t launch_draft_topk(const void *logits, int dtype, int B, int D, int k, int V, int64_t ld,
                              int32_t *tok, float *conf, float *stats, void *ws, int32_t *status,
                              int num_sms, cudaStream_t st);
int current_num_sms();

}  // namespace eagle

using namespace eagle;

extern "C" int eagle_draft_topk_noalloc(const void *logits, int dtype, int B, int D, int k, int V, int64_t ld,
                                        int32_t *tok, float *conf, float *stats, int32_t *status,
                                        eagle_stream_t stream) {
  if (!logits || !tok || !conf || (dtype != EAGLE_F32 && dtype != EAGLE_BF16)) return EAGLE_ERR_INVALID;
  if (B < 1 || D < 1 || k < 1 || k > 32 || V < 1 || k > V || ld < V) return EAGLE_ERR_INVALID;
  const int es = dtype == EAGLE_BF16 ? 2 : 4;
  if ((static_cast<int64_t>(V) * es) % 16 || (ld * es) % 16 || (reinterpret_cast<uintptr_t>(logits) & 15u))
    return EAGLE_ERR_INVALID;
  if (static_cast<int64_t>(B) * (1 + (D - 1) * k) > 65535) return EAGLE_ERR_UNSUPPORTED;
  return launch_draft_topk(logits, dtype, B, D, k, V, ld, tok, conf, stats, nullptr, status, current_num_sms(),
                           reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? EAGLE_OK
             : EAGLE_ERR_CUDA;
}
