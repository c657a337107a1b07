// gemm_bwd.cu -- first-order backward of the SwiGLU experts (FP32 accumulate).
//
// ExpertTrainingCache::backward in src/moe/experts.rs (ruDNN 0.1.25 source
// view) and the ruDNN user guide, section 12: for each dispatched row r of
// expert e with forward g = x W_gate^T, u = x W_up^T, a = silu(g) u,
// o = a W_down^T and upstream gradient do = dL/do:
//   da     = do W_down                      dg = da u silu'(g),  du = da silu(g)
//   dinput = dg W_gate + du W_up            (per row, in the weight dtype)
//   ddown  = sum_r do_r^T a_r,  dgate = sum_r dg_r^T x_r,  dup = sum_r du_r^T x_r
// with the weight gradients in FP32 as on the pages.  g and u are recomputed
// from x (no forward cache), silu'(z) = s (1 + z (1 - s)), s = sigmoid(z).
//
// Two tiled FFMA kernels, both deterministic (every output element is summed
// by one thread in a fixed order):
//   row_gemm:    out[r, n] = sum_k A[r, k] * B_e[k, n] over an expert's rows,
//                with up to two (A, B) pairs and fused epilogues;
//   weight_grad: W_e[m, n] = sum_{r in e} P[r, m] * Q[r, n], one expert per
//                grid slice, K running over the expert's rows.
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int BM = 64, BN = 64, BK = 16;

// element (k, n) of expert e's operand in a strided view of the weights
template <typename T>
struct View {
  const T* p;
  int64_t se, sk, sn;  // strides of expert, k and n
  __device__ __forceinline__ float at(int e, int64_t k, int64_t n) const {
    return to_f32<T>(p[e * se + k * sk + n * sn]);
  }
};

enum RowEpi {
  kRawGU = 0,     // pair 0 -> g (FP32), pair 1 -> u (FP32): two outputs
  kSwigluBwd = 1, // da = acc; writes dg, du (FP32) from g, u; also a = silu(g) u
  kSum = 2,       // out = acc0 + acc1 in TO
};

__device__ __forceinline__ float sigmoidf_(float z) { return 1.f / (1.f + expf(-z)); }

// Prefix of per-expert 64-row tile counts (E <= 1024), computed by warp 0.
__device__ void tile_prefix(const uint32_t* offsets, int E, uint32_t* s_pref) {
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
}

template <typename TA, typename TW, typename TO, int NPAIR, int EPI>
__global__ void __launch_bounds__(256)
row_gemm(const TA* __restrict__ A0, const TA* __restrict__ A1, int64_t lda, View<TW> B0, View<TW> B1,
         int E, int64_t K, int64_t n_out, const uint32_t* __restrict__ offsets, TO* __restrict__ out0,
         float* __restrict__ out1, const float* __restrict__ g, const float* __restrict__ u,
         float* __restrict__ a_out) {
  __shared__ uint32_t s_pref[1025];
  __shared__ float As[NPAIR][BK][BM + 4];
  __shared__ float Bs[NPAIR][BK][BN + 4];
  tile_prefix(offsets, E, s_pref);
  const int mt = blockIdx.x;
  if ((uint32_t)mt >= s_pref[E]) return;
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_pref[mid] <= (uint32_t)mt) lo = mid; else hi = mid;
  }
  const int e = lo;
  const int64_t m0 = (int64_t)offsets[e] + (int64_t)(mt - (int)s_pref[e]) * BM;
  const int64_t left = (int64_t)offsets[e + 1] - m0;
  const int rows = (int)(left < BM ? left : BM);
  const int64_t n0 = (int64_t)blockIdx.y * BN;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;

  float acc[NPAIR][4][4];
#pragma unroll
  for (int q = 0; q < NPAIR; ++q)
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[q][i][j] = 0.f;

  for (int64_t k0 = 0; k0 < K; k0 += BK) {
#pragma unroll
    for (int it = 0; it < (BM * BK) / 256; ++it) {
      const int li = it * 256 + threadIdx.x;
      const int r = li / BK, kk = li % BK;
      const bool kin = k0 + kk < K;
      As[0][kk][r] = (r < rows && kin) ? to_f32<TA>(A0[(m0 + r) * lda + k0 + kk]) : 0.f;
      if (NPAIR == 2) As[NPAIR - 1][kk][r] = (r < rows && kin) ? to_f32<TA>(A1[(m0 + r) * lda + k0 + kk]) : 0.f;
      const bool nin = n0 + r < n_out;
      Bs[0][kk][r] = (nin && kin) ? B0.at(e, k0 + kk, n0 + r) : 0.f;
      if (NPAIR == 2) Bs[NPAIR - 1][kk][r] = (nin && kin) ? B1.at(e, k0 + kk, n0 + r) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
#pragma unroll
      for (int q = 0; q < NPAIR; ++q) {
        float av[4], bv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) av[i] = As[q][kk][ty + 16 * i];
#pragma unroll
        for (int j = 0; j < 4; ++j) bv[j] = Bs[q][kk][tx + 16 * j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[q][i][j] = fmaf(av[i], bv[j], acc[q][i][j]);
      }
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = ty + 16 * i;
    if (r >= rows) continue;
    const int64_t row = m0 + r;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t c = n0 + tx + 16 * j;
      if (c >= n_out) continue;
      const int64_t o = row * n_out + c;
      if constexpr (EPI == kRawGU) {
        reinterpret_cast<float*>(out0)[o] = acc[0][i][j];
        out1[o] = acc[NPAIR - 1][i][j];
      } else if constexpr (EPI == kSwigluBwd) {
        const float gg = g[o], uu = u[o], d = acc[0][i][j];
        const float s = sigmoidf_(gg);
        reinterpret_cast<float*>(out0)[o] = d * uu * s * (1.f + gg * (1.f - s));  // dg
        out1[o] = d * gg * s;                                                      // du
        a_out[o] = gg * s * uu;                                                    // a
      } else {
        float v = acc[0][i][j];
        if (NPAIR == 2) v += acc[NPAIR - 1][i][j];
        out0[o] = from_f32<TO>(v);
      }
    }
  }
}

// W_e[m, n] = sum over the expert's rows r of P[r, m] * Q[r, n]; FP32 output
// [E, M, N].  grid = (m-tiles, n-tiles, E).
template <typename TP, typename TQ>
__global__ void __launch_bounds__(256)
weight_grad(const TP* __restrict__ P, int64_t ldp, const TQ* __restrict__ Q, int64_t ldq,
            int64_t M, int64_t N, const uint32_t* __restrict__ offsets, float* __restrict__ W) {
  __shared__ float Ps[BK][BM + 4];
  __shared__ float Qs[BK][BN + 4];
  const int e = blockIdx.z;
  const int64_t m0 = (int64_t)blockIdx.x * BM, n0 = (int64_t)blockIdx.y * BN;
  const int64_t r0 = offsets[e], r1 = offsets[e + 1];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int64_t k0 = r0; k0 < r1; k0 += BK) {
#pragma unroll
    for (int it = 0; it < (BM * BK) / 256; ++it) {
      const int li = it * 256 + threadIdx.x;
      const int kk = li / BM, c = li % BM;  // coalesced along m / n
      const bool kin = k0 + kk < r1;
      Ps[kk][c] = (kin && m0 + c < M) ? to_f32<TP>(P[(k0 + kk) * ldp + m0 + c]) : 0.f;
      Qs[kk][c] = (kin && n0 + c < N) ? to_f32<TQ>(Q[(k0 + kk) * ldq + n0 + c]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float pv[4], qv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) pv[i] = Ps[kk][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) qv[j] = Qs[kk][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(pv[i], qv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t m = m0 + ty + 16 * i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t n = n0 + tx + 16 * j;
      if (n < N) W[((int64_t)e * M + m) * N + n] = acc[i][j];
    }
  }
}

template <typename T>
cudaError_t backward_t(const ExpertsBwdArgs& a, cudaStream_t s) {
  const int64_t N = a.N, H = a.H, I = a.I;
  const int E = a.E;
  const T* x = static_cast<const T*>(a.x_disp);
  const T* dout = static_cast<const T*>(a.dout);
  const T* Wg = static_cast<const T*>(a.gate);
  const T* Wu = static_cast<const T*>(a.up);
  const T* Wd = static_cast<const T*>(a.down);
  const int64_t mt = (N + BM - 1) / BM + std::min<int64_t>(E, N);
  // 1. g, u = x W_gate^T, x W_up^T       (B_e[k=h, n=i] = W[e, i, h])
  View<T> vg{Wg, I * H, 1, H}, vu{Wu, I * H, 1, H};
  row_gemm<T, T, float, 2, kRawGU><<<dim3((unsigned)mt, (unsigned)((I + BN - 1) / BN)), 256, 0, s>>>(
      x, x, H, vg, vu, E, H, I, a.offsets, a.g, a.u, nullptr, nullptr, nullptr);
  // 2. da = do W_down, then dg, du, a     (B_e[k=h, n=i] = W_down[e, h, i])
  View<T> vd{Wd, H * I, I, 1};
  row_gemm<T, T, float, 1, kSwigluBwd><<<dim3((unsigned)mt, (unsigned)((I + BN - 1) / BN)), 256, 0, s>>>(
      dout, nullptr, H, vd, vd, E, H, I, a.offsets, a.dg, a.du, a.g, a.u, a.act);
  // 3. dinput = dg W_gate + du W_up       (B_e[k=i, n=h] = W[e, i, h])
  View<T> vg2{Wg, I * H, H, 1}, vu2{Wu, I * H, H, 1};
  row_gemm<float, T, T, 2, kSum><<<dim3((unsigned)mt, (unsigned)((H + BN - 1) / BN)), 256, 0, s>>>(
      a.dg, a.du, I, vg2, vu2, E, I, H, a.offsets, static_cast<T*>(a.dinput), nullptr, nullptr,
      nullptr, nullptr);
  // 4. weight gradients (FP32)
  weight_grad<T, float><<<dim3((unsigned)((H + BM - 1) / BM), (unsigned)((I + BN - 1) / BN), E), 256, 0, s>>>(
      dout, H, a.act, I, H, I, a.offsets, a.ddown);                    // ddown[e,h,i]
  weight_grad<float, T><<<dim3((unsigned)((I + BM - 1) / BM), (unsigned)((H + BN - 1) / BN), E), 256, 0, s>>>(
      a.dg, I, x, H, I, H, a.offsets, a.dgate);                        // dgate[e,i,h]
  weight_grad<float, T><<<dim3((unsigned)((I + BM - 1) / BM), (unsigned)((H + BN - 1) / BN), E), 256, 0, s>>>(
      a.du, I, x, H, I, H, a.offsets, a.dup);                          // dup[e,i,h]
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_experts_backward(const ExpertsBwdArgs& a, cudaStream_t s) {
  switch (a.dt) {
    case MOE_F32: return backward_t<float>(a, s);
    case MOE_F16: return backward_t<__half>(a, s);
    default: return backward_t<__nv_bfloat16>(a, s);
  }
}

}  // namespace moe
