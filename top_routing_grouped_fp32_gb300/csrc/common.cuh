// common.cuh -- small device helpers shared by the kernels of this library.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr uint32_t kInvalid = 0xFFFFFFFFu;

// Every workspace starts with this header; word 0 is the device status.
constexpr size_t kWsHeader = 256;

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline size_t dtype_size(moe_dtype d) { return d == MOE_F32 ? 4 : 2; }

// ---- element conversions --------------------------------------------------
template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// ---- programmatic dependent launch ------------------------------------------
// Kernels of a call sequence are launched with programmatic stream
// serialisation: a kernel may be launched (and run its prologue) before its
// predecessor in the stream has finished.  pdl_wait() blocks until every
// predecessor grid has completed and its memory is visible, so each kernel
// calls it before its first read of anything a predecessor wrote;
// pdl_trigger() lets the successor be launched once every CTA of this grid has
// started.  Without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Reads element i of a weights array whose dtype is only known at run time.
__device__ __forceinline__ float load_dyn(const void* p, int dtype, size_t i) {
  if (dtype == MOE_F32) return static_cast<const float*>(p)[i];
  if (dtype == MOE_F16) return __half2float(static_cast<const __half*>(p)[i]);
  return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
}

// Packs 8 floats to 8 16-bit values (one 16-byte store).
template <typename T> __device__ __forceinline__ uint4 pack8(const float* f);
template <> __device__ __forceinline__ uint4 pack8<__nv_bfloat16>(const float* f) {
  uint4 r;
  __nv_bfloat162 v0 = __floats2bfloat162_rn(f[0], f[1]);
  __nv_bfloat162 v1 = __floats2bfloat162_rn(f[2], f[3]);
  __nv_bfloat162 v2 = __floats2bfloat162_rn(f[4], f[5]);
  __nv_bfloat162 v3 = __floats2bfloat162_rn(f[6], f[7]);
  r.x = *reinterpret_cast<uint32_t*>(&v0);
  r.y = *reinterpret_cast<uint32_t*>(&v1);
  r.z = *reinterpret_cast<uint32_t*>(&v2);
  r.w = *reinterpret_cast<uint32_t*>(&v3);
  return r;
}
template <> __device__ __forceinline__ uint4 pack8<__half>(const float* f) {
  uint4 r;
  __half2 v0 = __floats2half2_rn(f[0], f[1]);
  __half2 v1 = __floats2half2_rn(f[2], f[3]);
  __half2 v2 = __floats2half2_rn(f[4], f[5]);
  __half2 v3 = __floats2half2_rn(f[6], f[7]);
  r.x = *reinterpret_cast<uint32_t*>(&v0);
  r.y = *reinterpret_cast<uint32_t*>(&v1);
  r.z = *reinterpret_cast<uint32_t*>(&v2);
  r.w = *reinterpret_cast<uint32_t*>(&v3);
  return r;
}

// Unpacks 8 16-bit values from a 16-byte vector.
template <typename T> __device__ __forceinline__ void unpack8(uint4 v, float* f) {
  const T* e = reinterpret_cast<const T*>(&v);
#pragma unroll
  for (int i = 0; i < 8; ++i) f[i] = to_f32<T>(e[i]);
}

// Records the first device-side error in a workspace status word.
__device__ __forceinline__ void set_status(uint32_t* status, uint32_t code) {
  if (status) atomicCAS(status, 0u, code);
}

}  // namespace moe
