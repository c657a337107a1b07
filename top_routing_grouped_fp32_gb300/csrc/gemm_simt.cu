// gemm_simt.cu -- segmented grouped GEMM on the FP32 FMA pipe.
//
// The products of SwiGluExperts::forward_dispatched_with_strategy in
// src/moe/experts.rs (ruDNN 0.1.25 source view): for a dispatched row r of
// expert e, out[r,:] = A[r,:] . W[e]^T ("NT" segmented grouped product).
// This path serves FP32 experts -- tensor-core TF32 would round the operands
// to 10-bit mantissas, too coarse for a 1e-4 relative tolerance -- and 16-bit
// shapes the tcgen05 path cannot take (rows not a multiple of 16 bytes).
//
// Tiles of 64 rows x 64 columns, 16-deep K slices staged in shared memory as
// FP32 (the next slice loaded into registers while the current one is
// multiplied); 256 threads each own a 4x4 block (two of them for gate/up).  Epilogues:
//   gate/up : h = silu(g) * u, with silu(z) = z / (1 + exp(-z))
//   down    : out[r,:] = o                           (moe_experts_forward)
//   weighted: slots[perm[r],:] = w[perm[r]] * o      (fused forward)
// Segments come from offsets[] on the device: the block computes the prefix of
// per-expert 64-row tile counts itself, so the host never reads offsets.
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int BM = 64, BN = 64, BK = 16;

// Locates m-tile `mt` among the experts' tiles: returns false when mt is past
// the last tile.  s_pref[e] = number of 64-row tiles of experts < e.
__device__ __forceinline__ bool find_tile(int mt, const uint32_t* s_pref, const uint32_t* offsets,
                                          int E, int& e_out, int64_t& m0, int& rows) {
  if ((uint32_t)mt >= s_pref[E]) return false;
  int lo = 0, hi = E;  // invariant: s_pref[lo] <= mt < s_pref[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_pref[mid] <= (uint32_t)mt) lo = mid; else hi = mid;
  }
  e_out = lo;
  m0 = (int64_t)offsets[lo] + (int64_t)(mt - (int)s_pref[lo]) * BM;
  const int64_t left = (int64_t)offsets[lo + 1] - m0;
  rows = (int)(left < BM ? left : BM);
  return true;
}

template <typename T, int MODE>
__global__ void __launch_bounds__(256)
grouped_gemm_simt(const T* __restrict__ A, const T* __restrict__ B0, const T* __restrict__ B1,
                  int E, int64_t K, int64_t n_out, const uint32_t* __restrict__ offsets,
                  T* __restrict__ out, const uint32_t* __restrict__ perm,
                  const void* __restrict__ weights, int wdt) {
  constexpr bool kDual = MODE == kGateUpSwiglu;
  __shared__ uint32_t s_pref[1025];
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[kDual ? 2 : 1][BK][BN + 4];
  pdl_wait();  // launched while the previous kernel finishes; its outputs are read below
  pdl_trigger();

  // prefix of per-expert tile counts (E <= 1024)
  if (threadIdx.x < 32) {
    const int per = (E + 31) / 32;
    uint32_t loc = 0;
    for (int i = 0; i < per; ++i) {
      const int e = threadIdx.x * per + i;
      if (e < E) loc += (offsets[e + 1] - offsets[e] + BM - 1) / BM;
    }
    uint32_t incl = loc;
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
      if ((int)threadIdx.x >= d) incl += o;
    }
    uint32_t run = incl - loc;
    for (int i = 0; i < per; ++i) {
      const int e = threadIdx.x * per + i;
      if (e < E) {
        s_pref[e] = run;
        run += (offsets[e + 1] - offsets[e] + BM - 1) / BM;
      }
    }
    if (threadIdx.x == 31) s_pref[E] = incl;
  }
  __syncthreads();

  int e, rows;
  int64_t m0;
  if (!find_tile(blockIdx.x, s_pref, offsets, E, e, m0, rows)) return;
  const int64_t n0 = (int64_t)blockIdx.y * BN;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const T* W0 = B0 + (size_t)e * n_out * K;
  const T* W1 = kDual ? B1 + (size_t)e * n_out * K : nullptr;

  float acc[2][4][4];
#pragma unroll
  for (int q = 0; q < 2; ++q)
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[q][i][j] = 0.f;

  // A[m0 .. m0+63][k0 .. k0+15] and W[n0 .. n0+63][k0 .. k0+15]: each thread
  // loads 4 elements of each; the next slice is loaded into registers while
  // the current one is multiplied from shared memory
  constexpr int PER = (BM * BK) / 256;
  float ra[PER], rb0[PER], rb1[PER];
  auto load_slice = [&](int64_t k0) {
#pragma unroll
    for (int it = 0; it < PER; ++it) {
      const int li = it * 256 + threadIdx.x;
      const int r = li / BK, kk = li % BK;
      ra[it] = (r < rows && k0 + kk < K) ? to_f32<T>(A[(m0 + r) * K + k0 + kk]) : 0.f;
      rb0[it] = rb1[it] = 0.f;
      if (n0 + r < n_out && k0 + kk < K) {
        rb0[it] = to_f32<T>(W0[(n0 + r) * K + k0 + kk]);
        if (kDual) rb1[it] = to_f32<T>(W1[(n0 + r) * K + k0 + kk]);
      }
    }
  };
  load_slice(0);
  for (int64_t k0 = 0; k0 < K; k0 += BK) {
    // stage the loaded slice, transposed
#pragma unroll
    for (int it = 0; it < PER; ++it) {
      const int li = it * 256 + threadIdx.x;
      const int r = li / BK, kk = li % BK;
      As[kk][r] = ra[it];
      Bs[0][kk][r] = rb0[it];
      if (kDual) Bs[kDual ? 1 : 0][kk][r] = rb1[it];
    }
    __syncthreads();
    if (k0 + BK < K) load_slice(k0 + BK);
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4], c[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[0][kk][tx + 16 * j];
      if (kDual) {
#pragma unroll
        for (int j = 0; j < 4; ++j) c[j] = Bs[kDual ? 1 : 0][kk][tx + 16 * j];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[0][i][j] = fmaf(a[i], b[j], acc[0][i][j]);
          if (kDual) acc[1][i][j] = fmaf(a[i], c[j], acc[1][i][j]);
        }
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = ty + 16 * i;
    if (r >= rows) continue;
    const int64_t grow = m0 + r;
    int64_t orow = grow;
    float scale = 1.f;
    if (MODE == kDownWeighted) {
      const uint32_t s = perm[grow];
      orow = s;
      scale = load_dyn(weights, wdt, s);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t c = n0 + tx + 16 * j;
      if (c >= n_out) continue;
      float v;
      if (MODE == kGateUpSwiglu) {
        const float g = acc[0][i][j];
        v = g / (1.f + expf(-g)) * acc[1][i][j];
      } else {
        v = acc[0][i][j] * scale;
      }
      out[orow * n_out + c] = from_f32<T>(v);
    }
  }
}

template <typename T>
cudaError_t launch_t(const GemmArgs& a, cudaStream_t s) {
  const int64_t mt_max = (a.N + BM - 1) / BM + std::min<int64_t>(a.E, a.N);
  dim3 grid((unsigned)mt_max, (unsigned)((a.n_out + BN - 1) / BN));
  const T* A = static_cast<const T*>(a.A);
  const T* B0 = static_cast<const T*>(a.B0);
  const T* B1 = static_cast<const T*>(a.B1);
  T* out = static_cast<T*>(a.out);
  const T* none = nullptr;
  switch (a.mode) {
    case kGateUpSwiglu:
      return launch_pdl(grouped_gemm_simt<T, kGateUpSwiglu>, grid, dim3(256), 0, s, A, B0, B1, a.E, a.K,
                        a.n_out, a.offsets, out, a.perm, a.weights, (int)a.wdt);
    case kDownPlain:
      return launch_pdl(grouped_gemm_simt<T, kDownPlain>, grid, dim3(256), 0, s, A, B0, none, a.E, a.K,
                        a.n_out, a.offsets, out, a.perm, a.weights, (int)a.wdt);
    default:
      return launch_pdl(grouped_gemm_simt<T, kDownWeighted>, grid, dim3(256), 0, s, A, B0, none, a.E, a.K,
                        a.n_out, a.offsets, out, a.perm, a.weights, (int)a.wdt);
  }
}

}  // namespace

cudaError_t launch_gemm_simt(const GemmArgs& a, cudaStream_t s) {
  switch (a.dt) {
    case MOE_F32: return launch_t<float>(a, s);
    case MOE_F16: return launch_t<__half>(a, s);
    default: return launch_t<__nv_bfloat16>(a, s);
  }
}

}  // namespace moe
