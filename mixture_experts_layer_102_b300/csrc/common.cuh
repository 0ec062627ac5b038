// Device helpers shared by the MoE forward kernels: element loads and stores in
// groups of 8 (one 16-byte vector for bf16), and the workspace status word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

namespace moe {

// Bits a kernel ORs into the workspace status word.
enum : uint32_t {
  STATUS_WAIT_TIMEOUT = 1u,  // a bounded mbarrier wait gave up
  STATUS_BAD_INDEX = 2u,     // an expert index or row outside its range
  STATUS_BAD_LAYOUT = 4u,    // a kernel's shared-memory carve did not fit its allocation
};

__device__ __forceinline__ void report(uint32_t* status, uint32_t bits) {
  if (status != nullptr) atomicOr(status, bits);
}

// Programmatic dependent launch. pdl_wait: block until the previous kernel of the
// stream has completed and its writes are visible (a no-op when this kernel was not
// launched as a dependent). pdl_trigger: let the next kernel of the stream start
// launching. Every kernel here calls both, in that order, after a prologue that reads
// at most the caller's own inputs (complete before the forward's first kernel, which
// is never a dependent launch, started) or the outputs of kernels two or more launches
// back (complete before the previous kernel, which triggers only after its own wait,
// let this one start), so at most two adjacent kernels overlap and all blocks of the
// earlier one are already resident when the later one starts.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch `kernel` on `stream`, as a programmatic dependent of the previous kernel of
// the stream when `pdl` is set.
template <typename... Exp, typename... Act>
inline cudaError_t launch_kernel(void (*kernel)(Exp...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t stream, bool pdl, Act&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = pdl ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<Act&&>(args)...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Let `kernel` use `bytes` of dynamic shared memory on the current device. The
// attribute is set once per kernel and device (and again only to raise it), so
// launches do not pay a driver call each time; safe to call from several threads.
inline cudaError_t ensure_dynamic_smem(const void* kernel, size_t bytes) {
  struct Entry {
    const void* fn;
    int dev;
    size_t bytes;
  };
  static std::mutex mu;
  static Entry table[256];
  static int used = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  int slot = -1;
  for (int i = 0; i < used; ++i)
    if (table[i].fn == kernel && table[i].dev == dev) {
      if (table[i].bytes >= bytes) return cudaSuccess;
      slot = i;
      break;
    }
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  if (slot < 0 && used < 256) slot = used++;
  if (slot >= 0) table[slot] = Entry{kernel, dev, bytes};
  return cudaSuccess;
}

// Opt-in shared memory per block of the current device (cached per device).
inline cudaError_t smem_optin_bytes(size_t* out) {
  static std::atomic<int> cached[64];  // 0 until the first query on that device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int c = dev >= 0 && dev < 64 ? cached[dev].load(std::memory_order_relaxed) : 0;
  if (c > 0) {
    *out = (size_t)c;
    return cudaSuccess;
  }
  int v = 0;
  e = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) cached[dev].store(v, std::memory_order_relaxed);
  *out = (size_t)v;
  return cudaSuccess;
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Two floats to a bf16 pair (round to nearest even), element 0 in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// 8 consecutive elements starting at p (p 16-byte aligned for bf16, 32 for f32).
__device__ __forceinline__ void load8(const float* p, float v[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float v[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x);
  v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
  v[4] = bf16_lo(u.z); v[5] = bf16_hi(u.z);
  v[6] = bf16_lo(u.w); v[7] = bf16_hi(u.w);
}

__device__ __forceinline__ void store8(float* p, const float v[8]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}

__device__ __forceinline__ void store8(__nv_bfloat16* p, const float v[8]) {
  uint4 u;
  u.x = pack_bf16x2(v[0], v[1]);
  u.y = pack_bf16x2(v[2], v[3]);
  u.z = pack_bf16x2(v[4], v[5]);
  u.w = pack_bf16x2(v[6], v[7]);
  *reinterpret_cast<uint4*>(p) = u;
}

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

// silu(z) = z * sigmoid(z) = z / (1 + e^-z)
__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

}  // namespace moe
