// Device helpers shared by the kernels of the tree-speculative step.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "../../include/eagle.h"

namespace eagle {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---- float <-> order-preserving unsigned ---------------------------------
// Maps floats to uint32 so that unsigned comparison equals float comparison
// (-0 is first folded into +0 so equal logits compare equal).
__device__ __forceinline__ uint32_t ordered_u32(float x) {
  x = x + 0.0f;  // -0 -> +0 under round-to-nearest
  uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float from_ordered_u32(uint32_t o) {
  uint32_t u = (o & 0x80000000u) ? (o & 0x7fffffffu) : ~o;
  return __uint_as_float(u);
}

// Top-k key of a logit: larger key = larger logit, then lower token id.
__device__ __forceinline__ uint64_t topk_key(float x, uint32_t tok) {
  return (static_cast<uint64_t>(ordered_u32(x)) << 32) | static_cast<uint64_t>(~tok);
}
__device__ __forceinline__ float key_value(uint64_t key) {
  return from_ordered_u32(static_cast<uint32_t>(key >> 32));
}
__device__ __forceinline__ uint32_t key_token(uint64_t key) {
  return ~static_cast<uint32_t>(key);
}

// ---- fast base-2 exponential (hardware approximation, PTX ex2.approx) ----
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- bf16 unpacking -------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <typename T> struct VecTraits;
template <> struct VecTraits<float> {
  static constexpr int kElems = 4;  // per 16-byte vector
  __device__ __forceinline__ static void unpack(const uint4 &v, float (&x)[4]) {
    x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y);
    x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
  }
  __device__ __forceinline__ static uint4 neg_inf_vec() { return make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u); }
  __device__ __forceinline__ static float load1(const void *p, int64_t i) {
    return __ldg(reinterpret_cast<const float *>(p) + i);
  }
};
template <> struct VecTraits<__nv_bfloat16> {
  static constexpr int kElems = 8;
  __device__ __forceinline__ static void unpack(const uint4 &v, float (&x)[8]) {
    x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
    x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z); x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
  }
  __device__ __forceinline__ static uint4 neg_inf_vec() { return make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u); }
  __device__ __forceinline__ static float load1(const void *p, int64_t i) {
    const unsigned short *s = reinterpret_cast<const unsigned short *>(p);
    return __uint_as_float(static_cast<uint32_t>(__ldg(s + i)) << 16);
  }
};

// ---- packed fp32 pairs (sm_100 family: one instruction for two lanes) ------
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float &a, float &b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Largest of the eight (bf16) or four (fp32) values of a 16-byte vector.
template <typename T> __device__ __forceinline__ float vec_max(const uint4 &v);
template <> __device__ __forceinline__ float vec_max<float>(const uint4 &v) {
  return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
               fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
}
template <> __device__ __forceinline__ float vec_max<__nv_bfloat16>(const uint4 &v) {
  const __nv_bfloat162 a = __hmax2(*reinterpret_cast<const __nv_bfloat162 *>(&v.x),
                                   *reinterpret_cast<const __nv_bfloat162 *>(&v.y));
  const __nv_bfloat162 b = __hmax2(*reinterpret_cast<const __nv_bfloat162 *>(&v.z),
                                   *reinterpret_cast<const __nv_bfloat162 *>(&v.w));
  const __nv_bfloat162 c = __hmax2(a, b);
  const uint32_t w = *reinterpret_cast<const uint32_t *>(&c);
  return fmaxf(bf16_lo(w), bf16_hi(w));
}

// Streaming 16-byte load that does not allocate in L1.
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// Asynchronous 16-byte copy global -> shared (L2 only), committed in groups;
// a thread waits for its own groups, so a lane that reads back only what it
// copied needs no barrier.
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
               ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))), "l"(gmem_src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---- warp reductions ------------------------------------------------------
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int o) {
  uint32_t lo = static_cast<uint32_t>(v), hi = static_cast<uint32_t>(v >> 32);
  lo = __shfl_xor_sync(0xffffffffu, lo, o);
  hi = __shfl_xor_sync(0xffffffffu, hi, o);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}
__device__ __forceinline__ uint64_t shfl_u64(uint64_t v, int src) {
  uint32_t lo = static_cast<uint32_t>(v), hi = static_cast<uint32_t>(v >> 32);
  lo = __shfl_sync(0xffffffffu, lo, src);
  hi = __shfl_sync(0xffffffffu, hi, src);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

// Merge of two (max, sum-of-exp relative to max) pairs.
__device__ __forceinline__ void lse_combine(float &m, float &s, float m2, float s2) {
  float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;  // both empty
  s = s * ex2_approx((m - mn) * kLog2e) + s2 * ex2_approx((m2 - mn) * kLog2e);
  m = mn;
}

// ---- launch configuration ----------------------------------------------------

// Raises a kernel's dynamic shared memory limit once per device (the limit
// belongs to the kernel as loaded on the current device).  `done` is the
// call site's record of the devices already configured: bit d for device
// d < 64; devices beyond are configured on every call.
template <typename Kernel>
inline cudaError_t set_smem_limit_once(Kernel kernel, int bytes, std::atomic<unsigned long long> &done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev >= 0 && dev < 64 ? 1ull << dev : 0ull;
  if (bit && (done.load(std::memory_order_relaxed) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_relaxed);
  return e;
}

// Raises a kernel's dynamic shared memory limit, once per device, to the
// most it can take: the device's opt-in maximum per block less the kernel's
// static shared memory.  The limit then only ever grows, so host threads
// launching the kernel with different sizes cannot lower it under each other.
template <typename Kernel>
inline cudaError_t set_smem_limit_max_once(Kernel kernel, std::atomic<unsigned long long> &done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev >= 0 && dev < 64 ? 1ull << dev : 0ull;
  if (bit && (done.load(std::memory_order_relaxed) & bit)) return cudaSuccess;
  int optin = 0;
  e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kernel);
  if (e != cudaSuccess) return e;
  const int bytes = optin - static_cast<int>(fa.sharedSizeBytes);
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_relaxed);
  return e;
}

// ---- chained launches (programmatic dependent launch) --------------------
// The step's kernels are launched so that each may be scheduled while the
// previous kernel in the stream finishes.  pdl_wait() blocks until that
// kernel has completed and its writes are visible; every chained kernel calls
// it before its first global read.  pdl_trigger() lets the next kernel be
// scheduled; kernels call it once their main work is done.  Both are no-ops
// for a kernel launched the ordinary way.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// Requests the line holding p into L2 without reading it into the SM: safe
// before pdl_wait() (L2 is coherent for the whole device, so a later load
// after the wait still sees the previous kernel's writes).
__device__ __forceinline__ void prefetch_l2(const void *p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)) : "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_chained(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                  Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// launch_chained with the grid's x dimension grouped into clusters of
// `cluster_x` CTAs (1: no clusters).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_chained_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                          cudaStream_t st, unsigned cluster_x, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cluster_x > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---- device-side status reporting -----------------------------------------
__device__ __forceinline__ void report(int32_t *status, int code) {
  if (status) atomicCAS(reinterpret_cast<int *>(status), 0, code);
}

}  // namespace eagle
