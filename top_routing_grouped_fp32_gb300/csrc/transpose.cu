// transpose.cu -- layout changes that let the tensor-core engine run the
// expert backward (ExpertTrainingCache::backward in src/moe/experts.rs) with
// K-major operands only.
//
//  * pad_offsets: pad[e] = sum_{e' < e} roundup(count_e', 64): each expert's
//    dispatched rows start on a 64-column boundary once transposed, so every
//    TMA box of the weight-gradient products starts 128-byte aligned;
//  * transpose_rows: src [N, C] (dispatched rows) -> dst [C, ld], row r of
//    expert e landing in column pad[e] + (r - offsets[e]); padding columns
//    are zero, so they add nothing to the weight-gradient sums;
//  * transpose_weights: src [E, R, C] -> dst[e] [C, ld] at column col0 + r,
//    i.e. per-expert W^T (two of them side by side give [W_gate^T | W_up^T]).
// Each is a 32x32 shared-memory tile transpose (coalesced on both sides).
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kTile = 32;

__global__ void pad_offsets_kernel(const uint32_t* __restrict__ offsets, int E, uint32_t* __restrict__ pad) {
  // one warp: per-lane serial sums, then a warp scan (E <= 1024)
  const int lane = threadIdx.x;
  const int per = (E + 31) / 32;
  uint32_t loc = 0;
  for (int i = 0; i < per; ++i) {
    const int e = lane * per + i;
    if (e < E) loc += (offsets[e + 1] - offsets[e] + 63u) & ~63u;
  }
  uint32_t incl = loc;
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += o;
  }
  uint32_t run = incl - loc;
  for (int i = 0; i < per; ++i) {
    const int e = lane * per + i;
    if (e < E) {
      pad[e] = run;
      run += (offsets[e + 1] - offsets[e] + 63u) & ~63u;
    }
  }
  if (lane == 31) pad[E] = incl;
}

template <typename T>
__global__ void __launch_bounds__(256)
transpose_rows_kernel(const T* __restrict__ src, int64_t C, const uint32_t* __restrict__ offsets,
                      const uint32_t* __restrict__ pad, int E, T* __restrict__ dst, int64_t ld) {
  __shared__ float tile[kTile][kTile + 1];
  const int64_t j0 = (int64_t)blockIdx.x * kTile;  // padded column block of dst
  const int64_t c0 = (int64_t)blockIdx.y * kTile;  // column block of src
  if (j0 >= (int64_t)pad[E]) return;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  for (int i = ty; i < kTile; i += 8) {
    const int64_t j = j0 + i;  // padded index of the source row
    int lo = 0, hi = E;        // pad[lo] <= j < pad[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (pad[mid] <= (uint64_t)j) lo = mid; else hi = mid;
    }
    const int64_t r = (int64_t)offsets[lo] + (j - (int64_t)pad[lo]);
    const bool real = r < (int64_t)offsets[lo + 1];
    const int64_t c = c0 + tx;
    tile[i][tx] = (real && c < C) ? to_f32<T>(src[r * C + c]) : 0.f;
  }
  __syncthreads();
  for (int i = ty; i < kTile; i += 8) {
    const int64_t c = c0 + i;
    if (c < C) dst[c * ld + j0 + tx] = from_f32<T>(tile[tx][i]);
  }
}

template <typename T>
__global__ void __launch_bounds__(256)
transpose_weights_kernel(const T* __restrict__ src, int64_t R, int64_t C, T* __restrict__ dst,
                         int64_t ld, int64_t col0) {
  __shared__ T tile[kTile][kTile + 1];
  const int64_t e = blockIdx.z;
  const int64_t r0 = (int64_t)blockIdx.x * kTile, c0 = (int64_t)blockIdx.y * kTile;
  const T* s = src + e * R * C;
  T* d = dst + e * C * ld;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (int i = ty; i < kTile; i += 8) {
    const int64_t r = r0 + i, c = c0 + tx;
    if (r < R && c < C) tile[i][tx] = s[r * C + c];
  }
  __syncthreads();
  for (int i = ty; i < kTile; i += 8) {
    const int64_t c = c0 + i, r = r0 + tx;
    if (r < R && c < C) d[c * ld + col0 + r] = tile[tx][i];
  }
}

template <typename T>
cudaError_t rows_t(const void* src, int64_t C, const uint32_t* offsets, const uint32_t* pad, int E,
                   int64_t npad_max, void* dst, int64_t ld, cudaStream_t s) {
  dim3 grid((unsigned)((npad_max + kTile - 1) / kTile), (unsigned)((C + kTile - 1) / kTile));
  transpose_rows_kernel<T><<<grid, 256, 0, s>>>(static_cast<const T*>(src), C, offsets, pad, E,
                                                 static_cast<T*>(dst), ld);
  return cudaGetLastError();
}

template <typename T>
cudaError_t weights_t(const void* src, int64_t E, int64_t R, int64_t C, void* dst, int64_t ld,
                      int64_t col0, cudaStream_t s) {
  dim3 grid((unsigned)((R + kTile - 1) / kTile), (unsigned)((C + kTile - 1) / kTile), (unsigned)E);
  transpose_weights_kernel<T><<<grid, 256, 0, s>>>(static_cast<const T*>(src), R, C,
                                                    static_cast<T*>(dst), ld, col0);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pad_offsets(const uint32_t* offsets, int E, uint32_t* pad, cudaStream_t s) {
  pad_offsets_kernel<<<1, 32, 0, s>>>(offsets, E, pad);
  return cudaGetLastError();
}

cudaError_t launch_transpose_rows(const void* src, moe_dtype dt, int64_t C, const uint32_t* offsets,
                                  const uint32_t* pad, int E, int64_t npad_max, void* dst,
                                  int64_t ld, cudaStream_t s) {
  if (dt == MOE_BF16) return rows_t<__nv_bfloat16>(src, C, offsets, pad, E, npad_max, dst, ld, s);
  return rows_t<__half>(src, C, offsets, pad, E, npad_max, dst, ld, s);
}

cudaError_t launch_transpose_weights(const void* src, moe_dtype dt, int64_t E, int64_t R, int64_t C,
                                     void* dst, int64_t ld, int64_t col0, cudaStream_t s) {
  if (dt == MOE_BF16) return weights_t<__nv_bfloat16>(src, E, R, C, dst, ld, col0, s);
  return weights_t<__half>(src, E, R, C, dst, ld, col0, s);
}

}  // namespace moe
