// eagle_draft_topk_noalloc: the draft softmax / top-k stage for callers that
// cannot hand the library any scratch memory.
//
// Some callers only ever receive input and output buffers: plugins and
// custom-op hooks of a host runtime that owns all device memory and offers
// no scratch, or processes whose device-memory budget is fixed up front and
// may not grow.  They cannot call cudaMalloc, and so cannot provide the
// workspace eagle_draft_topk needs for its split-row merges.  This entry
// point runs the same kernel with its scratch in a fixed array compiled into
// the library instead.
//
// The array is a file-scope __device__ variable of kNoallocScratchBytes, so
// every GPU that loads the library holds it until the process exits.  Host
// code cannot use the array's name as a device address: the address is
// looked up once per device with cudaGetSymbolAddress, on the first call
// made while that device is current.  All calls on a device share the array
// and it keeps the previous call's contents, so the part that must start at
// zero (the split-merge tickets) is cleared at the start of every call, and
// calls that may overlap on the GPU (other streams, other host threads) race
// on it and must be serialised by the caller.  Nothing here allocates.
#include <mutex>

#include "common.cuh"

namespace eagle {

size_t draft_workspace_bytes(int B, int D, int k, int V, int vec, int num_sms);
cudaError_t launch_draft_topk(const void *logits, int dtype, int B, int D, int k, int V, int64_t ld,
                              int32_t *tok, float *conf, float *stats, void *ws, int32_t *status,
                              int num_sms, cudaStream_t st);
int current_num_sms();

constexpr size_t kNoallocScratchBytes = EAGLE_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_draft_scratch[kNoallocScratchBytes];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (looked up once
// per device), or nullptr on failure.
void *scratch_for_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_draft_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}
}  // namespace

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
  const int sms = current_num_sms();
  const size_t need = draft_workspace_bytes(B, D, k, V, 16 / es, sms);
  if (need > kNoallocScratchBytes) return EAGLE_ERR_WORKSPACE;  // beyond the fixed array
  void *scratch = scratch_for_current_device();
  if (!scratch) return EAGLE_ERR_CUDA;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the merge tickets at the front of the scratch must start at zero
  const size_t tickets = (static_cast<size_t>(B) * (1 + (D - 1) * k) * sizeof(uint32_t) + 255) / 256 * 256;
  if (cudaMemsetAsync(scratch, 0, tickets < need ? tickets : need, st) != cudaSuccess) return EAGLE_ERR_CUDA;
  return launch_draft_topk(logits, dtype, B, D, k, V, ld, tok, conf, stats, scratch, status, sms, st) ==
                 cudaSuccess
             ? EAGLE_OK
             : EAGLE_ERR_CUDA;
}
