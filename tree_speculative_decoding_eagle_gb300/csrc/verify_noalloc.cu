// eagle_verify_noalloc: the verification stage with its scratch memory kept
// inside the library, for callers that cannot allocate device memory.
//
// eagle_verify needs scratch: for every target row and 2048-token chunk, a
// 16-byte record (max, sum of exponentials, argmax) that its statistics
// kernel writes and its walk kernel reads.  Its callers pass that scratch in
// as a workspace.  Some callers cannot: a plugin or custom-op hook in a host
// runtime that owns every device buffer and gives the op only its inputs and
// outputs; a serving loop that must not call cudaMalloc once it runs, since
// cudaMalloc can synchronise the device and stall the work in flight; a
// process that has handed all device memory to its own pool.
//
// Here the records live in one file-scope __device__ array of
// EAGLE_VERIFY_NOALLOC_SCRATCH_BYTES bytes.  Every GPU that loads the library
// holds it until the process exits; the call itself allocates nothing.  In
// host code the array's name is a host-side stand-in, not a device address,
// so the first call on each device looks the address up with
// cudaGetSymbolAddress (that device current) and keeps it; that first call
// should come before any stream capture.  No record needs clearing: every
// record a call reads, the same call writes first.  All calls share the one
// array and it keeps the last call's records, so calls that overlap on the
// GPU race on it.
#include <atomic>

#include "common.cuh"

static __device__ __align__(256) unsigned char verify_noalloc_scratch[EAGLE_VERIFY_NOALLOC_SCRATCH_BYTES];

namespace eagle {

size_t verify_workspace_bytes(int B, int m, int V);
cudaError_t launch_verify(const void *target, int dtype, int64_t ld, const int32_t *node_tok,
                          const int32_t *node_parent, int B, int m, int D, int V, int mode,
                          float temperature, const float *u, int32_t *accept_len,
                          int32_t *path_nodes, int32_t *out_tokens, int32_t *status, void *ws,
                          int num_sms, cudaStream_t st);
int current_num_sms();

namespace {

constexpr int kMaxDevices = 64;
std::atomic<void *> scratch_on_device[kMaxDevices];

// Device address of the scratch array on the current device (looked up once
// per device; devices beyond kMaxDevices look it up on every call).
cudaError_t scratch_address(void **addr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < kMaxDevices;
  if (cached) {
    void *p = scratch_on_device[dev].load(std::memory_order_acquire);
    if (p) {
      *addr = p;
      return cudaSuccess;
    }
  }
  void *p = nullptr;
  e = cudaGetSymbolAddress(&p, verify_noalloc_scratch);
  if (e != cudaSuccess) return e;
  if (cached) scratch_on_device[dev].store(p, std::memory_order_release);
  *addr = p;
  return cudaSuccess;
}

}  // namespace
}  // namespace eagle

using namespace eagle;

extern "C" int eagle_verify_noalloc(const void *target, int dtype, int64_t ld, const int32_t *node_tok,
                                    const int32_t *node_parent, int B, int m, int D, int V, int mode,
                                    float temperature, const float *uniforms, int32_t *accept_len,
                                    int32_t *path_nodes, int32_t *out_tokens, int32_t *status,
                                    eagle_stream_t stream) {
  // the argument rules of eagle_verify
  if (!target || !node_tok || !node_parent || !accept_len || !path_nodes || !out_tokens) return EAGLE_ERR_INVALID;
  if ((dtype != EAGLE_F32 && dtype != EAGLE_BF16) || B < 1 || m < 0 || m + 1 > 4096 || D < 1 || V < 1 || ld < V)
    return EAGLE_ERR_INVALID;
  if (mode != EAGLE_GREEDY && mode != EAGLE_SAMPLE) return EAGLE_ERR_INVALID;
  if (mode == EAGLE_SAMPLE && (!uniforms || !(temperature > 0.f))) return EAGLE_ERR_INVALID;
  const int es = dtype == EAGLE_BF16 ? 2 : 4;
  if ((static_cast<int64_t>(V) * es) % 16 || (ld * es) % 16 || (reinterpret_cast<uintptr_t>(target) & 15u))
    return EAGLE_ERR_INVALID;
  // the records must fit the library's array
  if (verify_workspace_bytes(B, m, V) > EAGLE_VERIFY_NOALLOC_SCRATCH_BYTES) return EAGLE_ERR_WORKSPACE;
  void *scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return EAGLE_ERR_CUDA;
  return launch_verify(target, dtype, ld, node_tok, node_parent, B, m, D, V, mode, temperature, uniforms,
                       accept_len, path_nodes, out_tokens, status, scratch, current_num_sms(),
                       reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? EAGLE_OK
             : EAGLE_ERR_CUDA;
}
