// combine.cu -- weighted combine back to token order.
//
// ruDNN user guide ("ruDNN Benutzerhandbuch"), section 6 "MoE aufrufen":
// combine uses the dispatch map to restore token order and merges the expert
// outputs with the routing weights.  Here y[t,:] = sum_j w[t,j] * out[r(t,j),:]
// with FP32 accumulation in ascending j (a fixed order, so the result is
// bit-reproducible), rounded once to the output dtype.
//
// The combines are HBM-bound streaming passes: each thread owns 8 consecutive
// columns of one token (one 16-byte vector for 16-bit types, two for FP32)
// and reads the k source rows of that token.  The combine backward (section
// 12) is one warp per dispatched row with 8-column vectors per lane.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

// slot_row[perm[r]] = r for every dispatched row (slot_row pre-filled with kInvalid)
__global__ void invert_perm_kernel(const uint32_t* __restrict__ perm, int64_t N,
                                   uint32_t* __restrict__ slot_row) {
  const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= N) return;
  const uint32_t s = perm[r];
  if (s < (uint64_t)N) slot_row[s] = (uint32_t)r;
}

// source rows are read once: evict-first loads
template <typename T>
__device__ __forceinline__ void load8(const T* p, float* f) {
  if constexpr (sizeof(T) == 2) {
    unpack8<T>(__ldcs(reinterpret_cast<const uint4*>(p)), f);
  } else {
    const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
    const float4 b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
}

// 8 elements as raw bits: one 16-byte vector (16-bit types) or two (FP32)
template <typename T>
struct Raw8 {
  uint4 q[sizeof(T) == 2 ? 1 : 2];
};
template <typename T, bool STREAM>
__device__ __forceinline__ Raw8<T> load_raw8(const T* p) {
  Raw8<T> r;
  const uint4* s = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int i = 0; i < (sizeof(T) == 2 ? 1 : 2); ++i) r.q[i] = STREAM ? __ldcs(s + i) : __ldg(s + i);
  return r;
}
template <typename T>
__device__ __forceinline__ void unpack_raw8(const Raw8<T>& r, float* f) {
  if constexpr (sizeof(T) == 2) {
    unpack8<T>(r.q[0], f);
  } else {
    f[0] = __uint_as_float(r.q[0].x); f[1] = __uint_as_float(r.q[0].y);
    f[2] = __uint_as_float(r.q[0].z); f[3] = __uint_as_float(r.q[0].w);
    f[4] = __uint_as_float(r.q[1].x); f[5] = __uint_as_float(r.q[1].y);
    f[6] = __uint_as_float(r.q[1].z); f[7] = __uint_as_float(r.q[1].w);
  }
}

template <typename T>
__device__ __forceinline__ void store8(T* p, const float* f) {
  if constexpr (sizeof(T) == 2) {
    *reinterpret_cast<uint4*>(p) = pack8<T>(f);
  } else {
    reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
  }
}

// y[t] = sum_j src[t*k+j], j in order (the fused forward's combine of the
// weighted slot rows).  VEC: H % 8 == 0 and 16-byte aligned rows, else one
// column per thread.
template <typename T, bool VEC>
__global__ void __launch_bounds__(256)
slot_sum_kernel(const T* __restrict__ src, int64_t T_rows, int k, int64_t H, T* __restrict__ y) {
  pdl_wait();
  pdl_trigger();
  constexpr int C = VEC ? 8 : 1;
  const int64_t groups = H / C;
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= T_rows * groups) return;
  const int64_t t = gid / groups;
  const int64_t c0 = (gid - t * groups) * C;
  float acc[C];
#pragma unroll
  for (int i = 0; i < C; ++i) acc[i] = 0.f;
  for (int j = 0; j < k; ++j) {
    const int64_t row = t * k + j;
    float v[C];
    if constexpr (VEC) {
      load8<T>(src + row * H + c0, v);
    } else {
      v[0] = to_f32<T>(src[row * H + c0]);
    }
#pragma unroll
    for (int i = 0; i < C; ++i) acc[i] += v[i];
  }
  if constexpr (VEC) {
    store8<T>(y + t * H + c0, acc);
  } else {
    y[t * H + c0] = from_f32<T>(acc[0]);
  }
}

constexpr int kBatch = 4;  // slots whose rows are loaded together in the weighted combine

// y[t] = sum_j w[t,j] * src[slot_row[t*k+j]], j in order (moe_combine; with
// no weights, the dispatch backward).  kBatch slots at a time: their row
// indices, then their raw rows, are loaded together and then added in slot
// order.  An undispatched slot makes the row NaN.
template <typename T, bool VEC>
__global__ void __launch_bounds__(256, 4)
combine_kernel(const T* __restrict__ src, const uint32_t* __restrict__ slot_row,
               const void* __restrict__ w, int wdt, int64_t T_rows, int k, int64_t H,
               T* __restrict__ y) {
  pdl_wait();
  pdl_trigger();
  constexpr int C = VEC ? 8 : 1;
  const int64_t groups = H / C;
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= T_rows * groups) return;
  const int64_t t = gid / groups;
  const int64_t c0 = (gid - t * groups) * C;
  float acc[C];
#pragma unroll
  for (int i = 0; i < C; ++i) acc[i] = 0.f;
  for (int j0 = 0; j0 < k; j0 += kBatch) {
    uint32_t rr[kBatch];
    float ww[kBatch];
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      rr[q] = kInvalid;
      ww[q] = 1.f;
      if (j0 + q < k) {
        rr[q] = __ldg(slot_row + t * k + j0 + q);
        if (w) ww[q] = load_dyn(w, wdt, (size_t)(t * k + j0 + q));
      }
    }
    // raw loads first, so that all of them are in flight before any is used
    Raw8<T> raw[VEC ? kBatch : 1];
    T one[kBatch];
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      if (j0 + q < k && rr[q] != kInvalid) {
        if constexpr (VEC) raw[q] = load_raw8<T, true>(src + (int64_t)rr[q] * H + c0);
        else one[q] = src[(int64_t)rr[q] * H + c0];
      }
    }
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      if (j0 + q >= k) break;
      if (rr[q] == kInvalid) {
#pragma unroll
        for (int i = 0; i < C; ++i) acc[i] = NAN;
      } else {
        float v[C];
        if constexpr (VEC) unpack_raw8<T>(raw[q], v);
        else v[0] = to_f32<T>(one[q]);
#pragma unroll
        for (int i = 0; i < C; ++i) acc[i] += ww[q] * v[i];
      }
    }
  }
  if constexpr (VEC) {
    store8<T>(y + t * H + c0, acc);
  } else {
    y[t * H + c0] = from_f32<T>(acc[0]);
  }
}

template <typename T, bool WEIGHTED>
cudaError_t launch_combine_t(const void* src, const uint32_t* slot_row, const void* w, moe_dtype wdt,
                             int64_t T_rows, int k, int64_t H, void* y, cudaStream_t s) {
  const bool vec = H % 8 == 0 && reinterpret_cast<uintptr_t>(src) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(y) % 16 == 0;
  const int64_t work = T_rows * (vec ? H / 8 : H);
  const unsigned grid = (unsigned)((work + 255) / 256);
  const T* sp = static_cast<const T*>(src);
  T* yp = static_cast<T*>(y);
  if constexpr (WEIGHTED) {
    if (vec)
      return launch_pdl(combine_kernel<T, true>, dim3(grid), dim3(256), 0, s, sp, slot_row, w, (int)wdt,
                        T_rows, k, H, yp);
    return launch_pdl(combine_kernel<T, false>, dim3(grid), dim3(256), 0, s, sp, slot_row, w, (int)wdt,
                      T_rows, k, H, yp);
  } else {
    if (vec) return launch_pdl(slot_sum_kernel<T, true>, dim3(grid), dim3(256), 0, s, sp, T_rows, k, H, yp);
    return launch_pdl(slot_sum_kernel<T, false>, dim3(grid), dim3(256), 0, s, sp, T_rows, k, H, yp);
  }
}

// Combine backward (user guide, section 12: combine_backward gives dexpert and
// FP32 dweights): one warp per dispatched row r holding slot s = t*k+j:
//   dexpert[r,:] = w[s] * dy[t,:]      dweights[s] = sum_h expert_out[r,h] dy[t,h]
// The dot product is summed per lane in column order, then by a butterfly
// (a fixed order).  Rows holding no slot (perm entry kInvalid or >= T*k) get
// dexpert = 0; slots no row holds keep the NaN the caller's buffer was filled
// with.
// VEC (H % 8 == 0, 16-byte aligned rows): each lane takes 8-column vectors
// lane, lane+32, ..., four in flight; its dot product runs over its vectors in
// order and over the 8 columns of each in order, then the butterfly.
template <typename T, bool VEC>
__global__ void __launch_bounds__(256)
combine_backward_kernel(const T* __restrict__ eo, const uint32_t* __restrict__ perm,
                        const void* __restrict__ w, int wdt, const T* __restrict__ dy, int64_t N,
                        int k, int64_t H, T* __restrict__ dexpert, float* __restrict__ dweights) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= N) return;
  const uint32_t s = __ldg(perm + r);
  T* dst = dexpert + r * H;
  if ((uint64_t)s >= (uint64_t)N) {  // no slot (kInvalid, or an entry past the T*k slots)
    for (int64_t c = lane; c < H; c += 32) dst[c] = from_f32<T>(0.f);
    return;
  }
  const int64_t t = s / (uint32_t)k;
  const float wv = load_dyn(w, wdt, s);
  const T* src = eo + r * H;
  const T* g = dy + t * H;
  float dot = 0.f;
  if constexpr (VEC) {
    const int64_t nv = H / 8;
    for (int64_t v0 = 0; v0 < nv; v0 += 4 * 32) {
      Raw8<T> ra[4], rb[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int64_t v = v0 + q * 32 + lane;
        if (v < nv) {
          ra[q] = load_raw8<T, true>(src + v * 8);
          rb[q] = load_raw8<T, false>(g + v * 8);
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int64_t v = v0 + q * 32 + lane;
        if (v < nv) {
          float a[8], b[8], o[8];
          unpack_raw8<T>(ra[q], a);
          unpack_raw8<T>(rb[q], b);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            o[i] = wv * b[i];
            dot = fmaf(a[i], b[i], dot);
          }
          store8<T>(dst + v * 8, o);
        }
      }
    }
  } else {
    for (int64_t c = lane; c < H; c += 32) {
      const float gv = to_f32<T>(g[c]);
      dst[c] = from_f32<T>(wv * gv);
      dot = fmaf(to_f32<T>(src[c]), gv, dot);
    }
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, d);
  if (lane == 0) dweights[s] = dot;
}

}  // namespace

cudaError_t launch_invert_perm(const uint32_t* perm, int64_t N, uint32_t* slot_row, cudaStream_t s) {
  cudaError_t err = cudaMemsetAsync(slot_row, 0xFF, (size_t)N * sizeof(uint32_t), s);
  if (err != cudaSuccess) return err;
  invert_perm_kernel<<<(unsigned)((N + 255) / 256), 256, 0, s>>>(perm, N, slot_row);
  return cudaGetLastError();
}

cudaError_t launch_combine(const void* expert_out, moe_dtype dt, const uint32_t* slot_row,
                           const void* weights, moe_dtype wdt, int64_t T, int k, int64_t H,
                           void* y, cudaStream_t s) {
  switch (dt) {
    case MOE_F32: return launch_combine_t<float, true>(expert_out, slot_row, weights, wdt, T, k, H, y, s);
    case MOE_F16: return launch_combine_t<__half, true>(expert_out, slot_row, weights, wdt, T, k, H, y, s);
    default: return launch_combine_t<__nv_bfloat16, true>(expert_out, slot_row, weights, wdt, T, k, H, y, s);
  }
}

cudaError_t launch_slot_sum(const void* slots, moe_dtype dt, int64_t T, int k, int64_t H, void* y,
                            cudaStream_t s) {
  switch (dt) {
    case MOE_F32: return launch_combine_t<float, false>(slots, nullptr, nullptr, dt, T, k, H, y, s);
    case MOE_F16: return launch_combine_t<__half, false>(slots, nullptr, nullptr, dt, T, k, H, y, s);
    default: return launch_combine_t<__nv_bfloat16, false>(slots, nullptr, nullptr, dt, T, k, H, y, s);
  }
}

cudaError_t launch_combine_backward(const void* expert_out, moe_dtype dt, const uint32_t* perm,
                                    const void* weights, moe_dtype wdt, const void* dy, int64_t T,
                                    int k, int64_t H, void* dexpert, float* dweights, cudaStream_t s) {
  const int64_t N = T * k;
  cudaError_t err = cudaMemsetAsync(dweights, 0xFF, (size_t)N * sizeof(float), s);  // NaN
  if (err != cudaSuccess) return err;
  const unsigned grid = (unsigned)((N + 7) / 8);
  const bool vec = H % 8 == 0 && reinterpret_cast<uintptr_t>(expert_out) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(dy) % 16 == 0 && reinterpret_cast<uintptr_t>(dexpert) % 16 == 0;
  auto go = [&](auto tag) {
    using T = decltype(tag);
    const T* eo = static_cast<const T*>(expert_out);
    const T* g = static_cast<const T*>(dy);
    T* dx = static_cast<T*>(dexpert);
    return vec ? launch_pdl(combine_backward_kernel<T, true>, dim3(grid), dim3(256), 0, s, eo, perm, weights,
                            (int)wdt, g, N, k, H, dx, dweights)
               : launch_pdl(combine_backward_kernel<T, false>, dim3(grid), dim3(256), 0, s, eo, perm, weights,
                            (int)wdt, g, N, k, H, dx, dweights);
  };
  switch (dt) {
    case MOE_F32: return go(float{});
    case MOE_F16: return go(__half{});
    default: return go(__nv_bfloat16{});
  }
}

}  // namespace moe
