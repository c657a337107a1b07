// route.cu -- softmax / top-k routing, 8 to 32 lanes per token row.
//
// Implements the routing contract of the ruDNN user guide ("ruDNN
// Benutzerhandbuch"), section 4 "Routing-Vertrag": softmax over all experts in
// FP32 before the top-k selection, ties to the lower expert id, optional
// renormalisation of the selected weights followed by a cast to the logits
// dtype, NaN weights for rows holding NaN, +inf or only -inf.
//
// Readings of the contract used here:
//  * the selection key is the logit itself (softmax is strictly monotone, so
//    the k largest logits are the k largest probabilities, and the key is
//    exact in every logits dtype); equal logits go to the lower id, +0 == -0;
//  * slot j of a row holds the j-th selection (descending weight);
//  * a poisoned row is all-tied: idx = 0..k-1, weights NaN;
//  * renormalisation divides by the FP32 sum of the k selected values added
//    in slot order; weights are always stored in the logits dtype.
//
// Design: a row of E <= 1024 logits is held in registers by LPR lanes (8 for
// E <= 64, 16 for E <= 128, else 32), VPL values per lane in a blocked layout
// (lane l owns experts l*VPL .. l*VPL+VPL-1) so that each lane reads its share
// with one or a few vector loads; a warp routes 32/LPR rows at once.  Max,
// sum and each of the k arg-max rounds are butterflies over the row's lanes;
// a butterfly leaves the bit-identical value in every lane, so every lane
// agrees on each winner.
#include <math.h>

#include <atomic>
#include <map>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kRowsPerBlock = 8;  // 8 warps of 32 threads

// (va, ia) beats (vb, ib): larger logit, then lower id.
__device__ __forceinline__ bool beats(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

template <typename T, int VPL>
__device__ __forceinline__ void load_row(const T* row, int E, int lane, float (&v)[VPL]) {
  const int e0 = lane * VPL;
  constexpr int kBytes = VPL * (int)sizeof(T);
  const T* p = row + e0;
  bool full = e0 + VPL <= E;
  if (kBytes >= 4 && full && (reinterpret_cast<uintptr_t>(p) % (kBytes >= 16 ? 16 : kBytes)) == 0) {
    if constexpr (kBytes >= 16) {
      alignas(16) T buf[VPL];
#pragma unroll
      for (int c = 0; c < kBytes / 16; ++c)
        reinterpret_cast<uint4*>(buf)[c] = __ldg(reinterpret_cast<const uint4*>(p) + c);
#pragma unroll
      for (int i = 0; i < VPL; ++i) v[i] = to_f32<T>(buf[i]);
    } else if constexpr (kBytes == 8) {
      alignas(16) T buf[VPL];
      *reinterpret_cast<uint2*>(buf) = __ldg(reinterpret_cast<const uint2*>(p));
#pragma unroll
      for (int i = 0; i < VPL; ++i) v[i] = to_f32<T>(buf[i]);
    } else {
      alignas(16) T buf[VPL];
      *reinterpret_cast<uint32_t*>(buf) = __ldg(reinterpret_cast<const uint32_t*>(p));
#pragma unroll
      for (int i = 0; i < VPL; ++i) v[i] = to_f32<T>(buf[i]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < VPL; ++i) v[i] = (e0 + i < E) ? to_f32<T>(p[i]) : -INFINITY;
  }
}

// Selection key of a 16-bit logit: the logit's bits mapped to an unsigned
// order (negative values reversed; -0 taken as +0), above 0xFFFF - id, so that
// the larger unsigned key is the larger logit and, between equal logits, the
// lower id.  Key 0 is below every real key and marks a selected expert.  The
// logit is exact in its 16-bit type, so the key orders exactly what the FP32
// comparison (larger logit, then lower id) orders.
template <typename T>
__device__ __forceinline__ uint32_t bits16_of(float v) {
  if constexpr (std::is_same<T, __half>::value) return (uint32_t)__half_as_ushort(__float2half_rn(v));
  else return __float_as_uint(v) >> 16;  // bf16: the high half of the exact FP32 value
}
template <typename T>
__device__ __forceinline__ uint32_t sel_key(float v, int id) {
  uint32_t b = bits16_of<T>(v);
  if (b == 0x8000u) b = 0u;
  const uint32_t o = (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
  return (o << 16) | (0xFFFFu - (uint32_t)id);
}
template <typename T>
__device__ __forceinline__ float key_logit(uint32_t key) {
  const uint32_t o = key >> 16;
  const uint32_t b = (o & 0x8000u) ? (o & 0x7FFFu) : (~o & 0xFFFFu);
  if constexpr (std::is_same<T, __half>::value) return __half2float(__ushort_as_half((unsigned short)b));
  else return __uint_as_float(b << 16);
}

// LPR lanes per row (8, 16 or 32), so that a warp routes 32 / LPR rows at
// once: for E <= 64 one warp instruction serves four rows, and each butterfly
// has three steps instead of five.
template <typename T, int LPR, int VPL>
__global__ void __launch_bounds__(32 * kRowsPerBlock)
route_kernel(const T* __restrict__ logits, int64_t T_rows, int E, int k, int renorm,
             uint32_t* __restrict__ idx, T* __restrict__ w_out, float* __restrict__ w32,
             uint32_t* status_reset) {
  pdl_wait();
  pdl_trigger();
  if (status_reset && blockIdx.x == 0 && threadIdx.x == 0) *status_reset = 0u;
  constexpr int R = 32 / LPR;                 // rows per warp
  constexpr int SLOTS = (64 + LPR - 1) / LPR;  // slots one lane may own (top_k <= 64)
  const int lane = threadIdx.x & 31;
  const int sub = lane % LPR;                 // lane within its row's segment
  const int64_t t = ((int64_t)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5)) * R + lane / LPR;
  const bool live = t < T_rows;               // the whole warp stays for the shuffles

  float v[VPL];
  if (live) {
    load_row<T, VPL>(logits + t * E, E, sub, v);
  } else {
#pragma unroll
    for (int i = 0; i < VPL; ++i) v[i] = -INFINITY;
  }
  const int e0 = sub * VPL;

  // poisoned-row detection and the row maximum.  Padding entries (past E)
  // hold -inf: they move neither the maximum nor the sum, and in the arg-max
  // rounds a real expert beats them (a real -inf on the lower id), so with
  // k <= E they are never selected.
  float m = -INFINITY;
  int bad = 0;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    bad |= (isnan(v[i]) || v[i] == INFINITY) ? 1 : 0;
    m = fmaxf(m, v[i]);
  }
#pragma unroll
  for (int d = LPR / 2; d > 0; d >>= 1) {
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d, LPR));
    bad |= __shfl_xor_sync(0xffffffffu, bad, d, LPR);
  }
  const bool dead = bad != 0 || m == -INFINITY;  // poisoned (or past the end)

  // FP32 softmax denominator: per-lane sum, then a butterfly
  float s = 0.f;
  if (!dead) {
#pragma unroll
    for (int i = 0; i < VPL; ++i) s += expf(v[i] - m);
  }
#pragma unroll
  for (int d = LPR / 2; d > 0; d >>= 1) s += __shfl_xor_sync(0xffffffffu, s, d, LPR);

  // k rounds of arg-max over the not-yet-selected experts; slot j is kept by
  // lane j % LPR of the row, in its register slot j / LPR
  constexpr bool kKeys = sizeof(T) == 2;
  uint32_t key[kKeys ? VPL : 1];
  uint32_t taken = 0;  // FP32 logits: bit i set once expert e0+i is selected
  if constexpr (kKeys) {
#pragma unroll
    for (int i = 0; i < VPL; ++i) key[i] = sel_key<T>(v[i], e0 + i);
  }
  uint32_t my_idx[SLOTS];
  float my_p[SLOTS];
#pragma unroll
  for (int h = 0; h < SLOTS; ++h) my_idx[h] = 0u, my_p[h] = 0.f;
  float sel_sum = 0.f;
#pragma unroll
  for (int h = 0; h < SLOTS; ++h) {
    if (h * LPR >= k) break;
    const int jn = min(LPR, k - h * LPR);
    for (int jj = 0; jj < jn; ++jj) {
      float bv;
      int bi;
      if constexpr (kKeys) {
        uint32_t bk = key[0];
#pragma unroll
        for (int i = 1; i < VPL; ++i) bk = max(bk, key[i]);
#pragma unroll
        for (int d = LPR / 2; d > 0; d >>= 1) bk = max(bk, __shfl_xor_sync(0xffffffffu, bk, d, LPR));
#pragma unroll
        for (int i = 0; i < VPL; ++i) key[i] = key[i] == bk ? 0u : key[i];  // keys are unique per row
        bi = (int)(0xFFFFu - (bk & 0xFFFFu));
        bv = key_logit<T>(bk);
      } else {
        bv = -INFINITY;
        bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
          if (!(taken >> i & 1u) && beats(v[i], e0 + i, bv, bi)) {
            bv = v[i];
            bi = e0 + i;
          }
        }
#pragma unroll
        for (int d = LPR / 2; d > 0; d >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, d, LPR);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, d, LPR);
          if (beats(ov, oi, bv, bi)) {
            bv = ov;
            bi = oi;
          }
        }
        if (bi / VPL == sub) taken |= 1u << (bi % VPL);
      }
      const float p = dead ? 0.f : expf(bv - m) / s;
      sel_sum += p;  // every lane adds in slot order
      if (jj == sub) {
        my_idx[h] = (uint32_t)bi;
        my_p[h] = p;
      }
    }
  }
  if (!live) return;
  if (dead) {
    for (int j = sub; j < k; j += LPR) {
      idx[t * k + j] = (uint32_t)j;
      w_out[t * k + j] = from_f32<T>(NAN);
      if (w32) w32[t * k + j] = NAN;
    }
    return;
  }
#pragma unroll
  for (int h = 0; h < SLOTS; ++h) {
    const int j = h * LPR + sub;
    if (j < k) {
      const float w = renorm ? my_p[h] / sel_sum : my_p[h];
      idx[t * k + j] = my_idx[h];
      w_out[t * k + j] = from_f32<T>(w);
      if (w32) w32[t * k + j] = w;
    }
  }
}

template <typename T>
cudaError_t launch_typed(const void* logits, int64_t T_rows, int E, int k, int renorm,
                         uint32_t* idx, void* weights, float* w32, uint32_t* status_reset,
                         cudaStream_t s) {
  const T* l = static_cast<const T*>(logits);
  T* w = static_cast<T*>(weights);
  // lanes per row and values per lane: E <= 64 on 8 lanes, E <= 128 on 16, else 32
  auto go = [&](auto kernel, int lpr) {
    const int64_t rows_per_block = (int64_t)kRowsPerBlock * (32 / lpr);
    dim3 grid((unsigned)((T_rows + rows_per_block - 1) / rows_per_block));
    return launch_pdl(kernel, grid, dim3(32 * kRowsPerBlock), 0, s, l, T_rows, E, k, renorm, idx, w,
                      w32, status_reset);
  };
  if (E <= 8) return go(route_kernel<T, 8, 1>, 8);
  if (E <= 16) return go(route_kernel<T, 8, 2>, 8);
  if (E <= 32) return go(route_kernel<T, 8, 4>, 8);
  if (E <= 64) return go(route_kernel<T, 8, 8>, 8);
  if (E <= 128) return go(route_kernel<T, 16, 8>, 16);
  if (E <= 256) return go(route_kernel<T, 32, 8>, 32);
  if (E <= 512) return go(route_kernel<T, 32, 16>, 32);
  return go(route_kernel<T, 32, 32>, 32);
}

// ---------------------------------------------------------------------------
// Sigmoid group-limited routing: ruDNN user guide ("ruDNN Benutzerhandbuch"),
// section 10.  Scores are sigmoid(logit); an optional FP32 correction bias is
// added for the selection only; the E experts form `groups` contiguous
// groups of E/groups; a group scores the largest corrected value of its
// experts (or the FP32 sum of its two largest with group_top_two); the
// `sel_groups` best groups are kept and top_k experts are chosen among
// theirs by corrected score; ties go to the lower id; weights are the
// original sigmoid values, optionally renormalised (FP32 sum in slot order),
// times `scale`, rounded to the logits dtype.
//
// The selection is an FP32 decision, so the sigmoid is the correctly rounded
// FP32 value: computed with a double-precision exp and rounded once (for
// 16-bit logits looked up in a table of those values for all 65536 patterns).  A row
// with a NaN logit or NaN corrected score gets idx = 0..k-1 and NaN weights.
//
// One warp per row; the corrected scores of the row sit in the warp's slice
// of shared memory so that any group size can be scanned; the arg-max rounds
// run on registers as in the softmax router.
constexpr int kSigMaxGroups = 128;

// The selection score's sigmoid, correctly rounded to FP32 through FP64.
__device__ __forceinline__ float sigmoid_rn(float x) { return (float)(1.0 / (1.0 + exp(-(double)x))); }

// sigmoid_rn of every 16-bit logit pattern: [0] bf16, [1] f16.  Filled on the
// device by sigmoid_table_kernel with the same arithmetic, so a lookup gives
// the bits a per-element evaluation gives; 16-bit logits then need no FP64
// exp per expert (FP64 runs at a small fraction of the FP32 rate here).
__device__ float g_sigmoid16[2][65536];

__global__ void sigmoid_table_kernel() {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= 2 * 65536) return;
  const uint32_t b = (uint32_t)i & 0xFFFFu;
  const float x = i < 65536 ? __uint_as_float(b << 16) : __half2float(__ushort_as_half((unsigned short)b));
  g_sigmoid16[i >> 16][b] = sigmoid_rn(x);
}

template <typename T, int VPL>
__global__ void __launch_bounds__(32 * kRowsPerBlock)
route_sigmoid_grouped_kernel(const T* __restrict__ logits, int64_t T_rows, int E,
                             const float* __restrict__ bias, int k, int groups, int sel_groups,
                             int top_two, int renorm, float scale, uint32_t* __restrict__ idx,
                             T* __restrict__ w_out, float* __restrict__ w32) {
  extern __shared__ float sig_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * kRowsPerBlock + warp;
  float* c_row = sig_smem + warp * (E + 2 * kSigMaxGroups);  // corrected scores [E]
  float* gscore = c_row + E;                                  // group scores [groups]
  float* gsel = gscore + kSigMaxGroups;                       // 1.0 when kept
  if (t >= T_rows) return;

  float v[VPL];
  load_row<T, VPL>(logits + t * E, E, lane, v);
  const int e0 = lane * VPL;
  float sg[VPL], c[VPL];
  bool bad = false;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = e0 + i;
    if (e < E) {
      if constexpr (sizeof(T) == 2)
        sg[i] = g_sigmoid16[std::is_same<T, __half>::value ? 1 : 0][bits16_of<T>(v[i])];
      else
        sg[i] = sigmoid_rn(v[i]);
      c[i] = sg[i] + (bias ? __ldg(bias + e) : 0.f);
      bad |= isnan(v[i]) || isnan(c[i]);
      c_row[e] = c[i];
    } else {
      sg[i] = 0.f;
      c[i] = -INFINITY;
    }
  }
  if (__any_sync(0xffffffffu, bad)) {
    for (int j = lane; j < k; j += 32) {
      idx[t * k + j] = (uint32_t)j;
      w_out[t * k + j] = from_f32<T>(NAN);
      if (w32) w32[t * k + j] = NAN;
    }
    return;
  }
  __syncwarp();
  // group scores (lane g handles groups g, g+32, ...)
  const int gs = E / groups;
  for (int g = lane; g < groups; g += 32) {
    float best = -INFINITY, second = -INFINITY;
    int bi = -1;
    for (int e = g * gs; e < (g + 1) * gs; ++e) {
      const float x = c_row[e];
      if (bi < 0 || beats(x, e, best, bi)) {
        if (bi >= 0) second = fmaxf(second, best);
        best = x;
        bi = e;
      } else {
        second = fmaxf(second, x);
      }
    }
    gscore[g] = top_two ? best + second : best;
    gsel[g] = 0.f;
  }
  __syncwarp();
  // keep the sel_groups best groups
  for (int r = 0; r < sel_groups; ++r) {
    float bv = -INFINITY;
    int bg = 0x7fffffff;
    for (int g = lane; g < groups; g += 32)
      if (gsel[g] == 0.f && beats(gscore[g], g, bv, bg)) {
        bv = gscore[g];
        bg = g;
      }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, d);
      const int og = __shfl_xor_sync(0xffffffffu, bg, d);
      if (beats(ov, og, bv, bg)) {
        bv = ov;
        bg = og;
      }
    }
    if ((bg & 31) == lane) gsel[bg] = 1.f;
    __syncwarp();
  }
  // experts outside the kept groups take no part
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < VPL; ++i)
    if (e0 + i >= E || gsel[(e0 + i) / gs] == 0.f) taken |= 1u << i;

  uint32_t my_idx[2] = {0, 0};
  float my_p[2] = {0.f, 0.f};
  float sel_sum = 0.f;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY, bs = 0.f;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      if (!(taken >> i & 1u) && beats(c[i], e0 + i, bv, bi)) {
        bv = c[i];
        bi = e0 + i;
        bs = sg[i];
      }
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, d);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, d);
      const float os = __shfl_xor_sync(0xffffffffu, bs, d);
      if (beats(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
        bs = os;
      }
    }
    if (bi / VPL == lane) taken |= 1u << (bi % VPL);
    sel_sum += bs;
    if ((j & 31) == lane) {
      my_idx[j >> 5] = (uint32_t)bi;
      my_p[j >> 5] = bs;
    }
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int j = h * 32 + lane;
    if (j < k) {
      const float w = (renorm ? my_p[h] / sel_sum : my_p[h]) * scale;
      idx[t * k + j] = my_idx[h];
      w_out[t * k + j] = from_f32<T>(w);
      if (w32) w32[t * k + j] = w;
    }
  }
}

// ---------------------------------------------------------------------------
// Router weights of a fixed selection and their logit gradient (user guide,
// section 12: selected_router_weights / selected_router_backward).  Scoring 0:
// q_j = softmax(logits)[idx_j] over all E; scoring 1: q_j = sigmoid(logit
// idx_j).  w_j = scale * (renorm ? q_j / Q : q_j), Q = sum_m q_m (slot order).
// Given dw = dL/dw (FP32):  c_m = dL/dq_m = scale * (renorm ? dw_m/Q -
// (sum_j dw_j q_j)/Q^2 : dw_m), and
//   softmax: dL/dl_e = sum_{m: idx_m = e} c_m q_m - p_e * sum_m c_m q_m
//   sigmoid: dL/dl_e = sum_{m: idx_m = e} c_m q_m (1 - q_m)
// Repeated indices gather (each slot counts); an index >= E makes the row's
// weights and gradient NaN.  One warp per row, FP32 throughout; the row's
// logits sit in the warp's shared-memory slice.
template <typename T>
__global__ void __launch_bounds__(32 * kRowsPerBlock)
router_backward_kernel(const T* __restrict__ logits, int64_t T_rows, int E,
                       const uint32_t* __restrict__ idx, int k, const float* __restrict__ dw,
                       int scoring, int renorm, float scale, T* __restrict__ dlogits,
                       float* __restrict__ w_out) {
  extern __shared__ float rb_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * kRowsPerBlock + warp;
  float* lrow = rb_smem + warp * (E + 2 * 64);
  float* q = lrow + E;       // [k]
  float* cq = q + 64;        // [k]: c_m q_m (softmax) or c_m q_m (1 - q_m)
  if (t >= T_rows) return;
  const T* l = logits + t * E;
  float m = -INFINITY;
  for (int e = lane; e < E; e += 32) {
    const float v = to_f32<T>(l[e]);
    lrow[e] = v;
    m = fmaxf(m, v);
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
  bool bad = false;
  for (int j = lane; j < k; j += 32) bad |= __ldg(idx + t * k + j) >= (uint32_t)E;
  if (__any_sync(0xffffffffu, bad)) {
    for (int j = lane; j < k; j += 32)
      if (w_out) w_out[t * k + j] = NAN;
    if (dw)
      for (int e = lane; e < E; e += 32) dlogits[t * E + e] = from_f32<T>(NAN);
    return;
  }
  float ssum = 0.f;
  if (scoring == 0) {
    for (int e = lane; e < E; e += 32) ssum += expf(lrow[e] - m);
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, d);
  }
  __syncwarp();
  for (int j = lane; j < k; j += 32) {
    const float x = lrow[__ldg(idx + t * k + j)];
    q[j] = scoring == 0 ? expf(x - m) / ssum : 1.f / (1.f + expf(-x));
  }
  __syncwarp();
  // slot-order sums, computed identically by every lane
  float Q = 0.f, gq = 0.f;
  for (int j = 0; j < k; ++j) {
    Q += q[j];
    if (dw) gq += __ldg(dw + t * k + j) * q[j];
  }
  for (int j = lane; j < k; j += 32) {
    if (w_out) w_out[t * k + j] = scale * (renorm ? q[j] / Q : q[j]);
    if (dw) {
      const float dwj = __ldg(dw + t * k + j);
      const float c = renorm ? scale * (dwj / Q - gq / (Q * Q)) : scale * dwj;
      cq[j] = scoring == 0 ? c * q[j] : c * q[j] * (1.f - q[j]);
    }
  }
  if (!dw) return;
  __syncwarp();
  float tot = 0.f;
  for (int j = 0; j < k; ++j) tot += cq[j];
  for (int e = lane; e < E; e += 32) {
    float v = 0.f;
    for (int j = 0; j < k; ++j)
      if (__ldg(idx + t * k + j) == (uint32_t)e) v += cq[j];
    if (scoring == 0) v -= expf(lrow[e] - m) / ssum * tot;
    dlogits[t * E + e] = from_f32<T>(v);
  }
}

// The same routing with the softmax router's layout: LPR lanes per row (a warp
// routes 32/LPR rows), VPL values per lane in a blocked layout, for group
// sizes gs that are VPL times a power of two: a group is then LG = gs/VPL
// whole lanes.  A group's top-two score is each lane's top two, merged over
// the group's lanes; the kept groups and the top_k experts come from
// (score, id) arg-max butterflies over the row's lanes.  Every reduction is
// over a strict order of (value, id) pairs or an exact max, so the result is
// the oracle's sequential scan.  Other group sizes take the kernel above.
template <typename T, int LPR, int VPL>
__global__ void __launch_bounds__(32 * kRowsPerBlock)
route_sigmoid_lanes_kernel(const T* __restrict__ logits, int64_t T_rows, int E,
                           const float* __restrict__ bias, int k, int groups, int sel_groups,
                           int top_two, int renorm, float scale, uint32_t* __restrict__ idx,
                           T* __restrict__ w_out, float* __restrict__ w32) {
  pdl_wait();
  pdl_trigger();
  constexpr int R = 32 / LPR;
  constexpr int SLOTS = (64 + LPR - 1) / LPR;
  const int lane = threadIdx.x & 31;
  const int sub = lane % LPR;
  const int64_t t = ((int64_t)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5)) * R + lane / LPR;
  const bool live = t < T_rows;  // the whole warp stays for the shuffles
  float v[VPL];
  if (live) {
    load_row<T, VPL>(logits + t * E, E, sub, v);
  } else {
#pragma unroll
    for (int i = 0; i < VPL; ++i) v[i] = -INFINITY;
  }
  const int e0 = sub * VPL;
  float sg[VPL], c[VPL];
  int bad = 0;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = e0 + i;
    if (e < E) {
      if constexpr (sizeof(T) == 2)
        sg[i] = g_sigmoid16[std::is_same<T, __half>::value ? 1 : 0][bits16_of<T>(v[i])];
      else
        sg[i] = sigmoid_rn(v[i]);
      c[i] = sg[i] + (bias ? __ldg(bias + e) : 0.f);
      bad |= (isnan(v[i]) || isnan(c[i])) ? 1 : 0;
    } else {
      sg[i] = 0.f;
      c[i] = -INFINITY;
    }
  }
#pragma unroll
  for (int d = LPR / 2; d > 0; d >>= 1) bad |= __shfl_xor_sync(0xffffffffu, bad, d, LPR);

  // group score: this lane's two largest corrected scores, merged over the
  // LG lanes of its group (the two largest of a multiset of pairs)
  const int gs = E / groups;
  const int LG = gs / VPL;
  const int my_g = sub / LG;
  float b1 = -INFINITY, b2 = -INFINITY;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    if (c[i] > b1) {
      b2 = b1;
      b1 = c[i];
    } else if (c[i] > b2) {
      b2 = c[i];
    }
  }
  for (int d = 1; d < LG; d <<= 1) {
    const float o1 = __shfl_xor_sync(0xffffffffu, b1, d, LPR);
    const float o2 = __shfl_xor_sync(0xffffffffu, b2, d, LPR);
    const float n2 = fmaxf(fminf(b1, o1), fmaxf(b2, o2));
    b1 = fmaxf(b1, o1);
    b2 = n2;
  }
  const float gscore = top_two ? b1 + b2 : b1;
  // keep the sel_groups best groups; a group competes through its first lane
  bool kept = false;
  const bool leader = sub % LG == 0 && my_g < groups;
  for (int r = 0; r < sel_groups; ++r) {
    float bv = -INFINITY;
    int bg = 0x7fffffff;
    if (leader && !kept) {
      bv = gscore;
      bg = my_g;
    }
#pragma unroll
    for (int d = LPR / 2; d > 0; d >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, d, LPR);
      const int og = __shfl_xor_sync(0xffffffffu, bg, d, LPR);
      if (beats(ov, og, bv, bg)) {
        bv = ov;
        bg = og;
      }
    }
    kept |= bg == my_g;
  }
  // top_k experts of the kept groups by corrected score; slot j is kept by
  // lane j % LPR of the row, in its register slot j / LPR
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < VPL; ++i)
    if (!kept || e0 + i >= E) taken |= 1u << i;
  uint32_t my_idx[SLOTS];
  float my_p[SLOTS];
#pragma unroll
  for (int h = 0; h < SLOTS; ++h) my_idx[h] = 0u, my_p[h] = 0.f;
  float sel_sum = 0.f;
  const int row_lane0 = lane - sub;
#pragma unroll
  for (int h = 0; h < SLOTS; ++h) {
    if (h * LPR >= k) break;
    const int jn = min(LPR, k - h * LPR);
    for (int jj = 0; jj < jn; ++jj) {
      float bv = -INFINITY, bs = 0.f;
      int bi = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        if (!(taken >> i & 1u) && beats(c[i], e0 + i, bv, bi)) {
          bv = c[i];
          bi = e0 + i;
          bs = sg[i];
        }
      }
#pragma unroll
      for (int d = LPR / 2; d > 0; d >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, d, LPR);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, d, LPR);
        if (beats(ov, oi, bv, bi)) {
          bv = ov;
          bi = oi;
        }
      }
      // the winner's sigmoid, from the lane that holds it
      const int owner = row_lane0 + min(bi / VPL, LPR - 1);
      const float p = __shfl_sync(0xffffffffu, bs, owner);
      if (bi / VPL == sub) taken |= 1u << (bi % VPL);
      sel_sum += p;  // every lane adds in slot order
      if (jj == sub) {
        my_idx[h] = (uint32_t)bi;
        my_p[h] = p;
      }
    }
  }
  if (!live) return;
  if (bad) {
    for (int j = sub; j < k; j += LPR) {
      idx[t * k + j] = (uint32_t)j;
      w_out[t * k + j] = from_f32<T>(NAN);
      if (w32) w32[t * k + j] = NAN;
    }
    return;
  }
#pragma unroll
  for (int h = 0; h < SLOTS; ++h) {
    const int j = h * LPR + sub;
    if (j < k) {
      const float w = (renorm ? my_p[h] / sel_sum : my_p[h]) * scale;
      idx[t * k + j] = my_idx[h];
      w_out[t * k + j] = from_f32<T>(w);
      if (w32) w32[t * k + j] = w;
    }
  }
}

// Fills g_sigmoid16 before the first 16-bit sigmoid routing on a device, with
// no host synchronisation: the first call enqueues the fill on its stream;
// later calls on other streams wait for that fill's event until it is seen
// complete.  A stream being captured into a graph gets a fill of its own in
// the graph.  Refills write the same bits, so they cannot disturb a reader.
cudaError_t ensure_sigmoid_table(cudaStream_t s) {
  struct Fill {
    cudaEvent_t done_ev = nullptr;
    bool done = false;
  };
  static std::mutex mu;
  static std::map<int, Fill> fills;
  static std::atomic<uint64_t> done_mask{0};  // devices 0..63 whose fill is known complete
  auto fill = [s]() {
    sigmoid_table_kernel<<<2 * 65536 / 256, 256, 0, s>>>();
    return cudaGetLastError();
  };
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && (done_mask.load(std::memory_order_acquire) >> dev & 1u)) return cudaSuccess;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if ((e = cudaStreamIsCapturing(s, &cap)) != cudaSuccess) return e;
  if (cap != cudaStreamCaptureStatusNone) return fill();
  std::lock_guard<std::mutex> lock(mu);
  Fill& f = fills[dev];
  if (f.done) return cudaSuccess;
  if (!f.done_ev) {
    if ((e = fill()) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&f.done_ev, cudaEventDisableTiming)) != cudaSuccess) return e;
    return cudaEventRecord(f.done_ev, s);
  }
  e = cudaEventQuery(f.done_ev);
  if (e == cudaSuccess) {
    f.done = true;
    if (dev < 64) done_mask.fetch_or(1ull << dev, std::memory_order_release);
    return cudaSuccess;
  }
  if (e != cudaErrorNotReady) return e;
  return cudaStreamWaitEvent(s, f.done_ev, 0);
}

template <typename T>
cudaError_t launch_sigmoid_typed(const void* logits, int64_t T_rows, int E, const float* bias,
                                 int k, int groups, int sel_groups, int top_two, int renorm,
                                 float scale, uint32_t* idx, void* weights, float* w32,
                                 cudaStream_t s) {
  if constexpr (sizeof(T) == 2) {
    const cudaError_t e = ensure_sigmoid_table(s);
    if (e != cudaSuccess) return e;
  }
  {
    // the lanes layout of the softmax router, when a group is a power-of-two
    // number of whole lanes
    const T* l = static_cast<const T*>(logits);
    T* w = static_cast<T*>(weights);
    const int gs = E / groups;
    auto go = [&](auto kernel, int lpr, int vpl) -> int {
      if (gs % vpl != 0) return 0;
      const int lg = gs / vpl;
      if ((lg & (lg - 1)) != 0 || lg > lpr) return 0;
      const int64_t rows_per_block = (int64_t)kRowsPerBlock * (32 / lpr);
      dim3 grid((unsigned)((T_rows + rows_per_block - 1) / rows_per_block));
      const cudaError_t e = launch_pdl(kernel, grid, dim3(32 * kRowsPerBlock), 0, s, l, T_rows, E, bias, k,
                                       groups, sel_groups, top_two, renorm, scale, idx, w, w32);
      return e == cudaSuccess ? 1 : -(int)e;
    };
    int r;
    if (E <= 8) r = go(route_sigmoid_lanes_kernel<T, 8, 1>, 8, 1);
    else if (E <= 16) r = go(route_sigmoid_lanes_kernel<T, 8, 2>, 8, 2);
    else if (E <= 32) r = go(route_sigmoid_lanes_kernel<T, 8, 4>, 8, 4);
    else if (E <= 64) r = go(route_sigmoid_lanes_kernel<T, 8, 8>, 8, 8);
    else if (E <= 128) r = go(route_sigmoid_lanes_kernel<T, 16, 8>, 16, 8);
    else if (E <= 256) r = go(route_sigmoid_lanes_kernel<T, 32, 8>, 32, 8);
    else if (E <= 512) r = go(route_sigmoid_lanes_kernel<T, 32, 16>, 32, 16);
    else r = go(route_sigmoid_lanes_kernel<T, 32, 32>, 32, 32);
    if (r == 1) return cudaSuccess;
    if (r < 0) return (cudaError_t)(-r);
  }
  dim3 grid((unsigned)((T_rows + kRowsPerBlock - 1) / kRowsPerBlock));
  dim3 block(32 * kRowsPerBlock);
  const size_t smem = (size_t)kRowsPerBlock * (E + 2 * kSigMaxGroups) * sizeof(float);
  const T* l = static_cast<const T*>(logits);
  T* w = static_cast<T*>(weights);
#define MOE_SIG_CASE(V)                                                                          \
  route_sigmoid_grouped_kernel<T, V><<<grid, block, smem, s>>>(l, T_rows, E, bias, k, groups,    \
                                                               sel_groups, top_two, renorm,       \
                                                               scale, idx, w, w32);               \
  break;
  switch ((E + 31) / 32 <= 1 ? 1 : (E + 31) / 32 <= 2 ? 2 : (E + 31) / 32 <= 4 ? 4
          : (E + 31) / 32 <= 8 ? 8 : (E + 31) / 32 <= 16 ? 16 : 32) {
    case 1: MOE_SIG_CASE(1)
    case 2: MOE_SIG_CASE(2)
    case 4: MOE_SIG_CASE(4)
    case 8: MOE_SIG_CASE(8)
    case 16: MOE_SIG_CASE(16)
    default: MOE_SIG_CASE(32)
  }
#undef MOE_SIG_CASE
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_route(const void* logits, moe_dtype ldt, int64_t T, int E, int k, int renorm,
                         uint32_t* idx, void* weights, float* w32, uint32_t* status_reset,
                         cudaStream_t s) {
  switch (ldt) {
    case MOE_F32:
      return launch_typed<float>(logits, T, E, k, renorm, idx, weights, w32, status_reset, s);
    case MOE_F16:
      return launch_typed<__half>(logits, T, E, k, renorm, idx, weights, w32, status_reset, s);
    default:
      return launch_typed<__nv_bfloat16>(logits, T, E, k, renorm, idx, weights, w32, status_reset, s);
  }
}

cudaError_t launch_route_sigmoid_grouped(const void* logits, moe_dtype ldt, int64_t T, int E,
                                         const float* bias, int k, int groups, int sel_groups,
                                         int top_two, int renorm, float scale, uint32_t* idx,
                                         void* weights, float* w32, cudaStream_t s) {
  switch (ldt) {
    case MOE_F32:
      return launch_sigmoid_typed<float>(logits, T, E, bias, k, groups, sel_groups, top_two, renorm,
                                         scale, idx, weights, w32, s);
    case MOE_F16:
      return launch_sigmoid_typed<__half>(logits, T, E, bias, k, groups, sel_groups, top_two, renorm,
                                          scale, idx, weights, w32, s);
    default:
      return launch_sigmoid_typed<__nv_bfloat16>(logits, T, E, bias, k, groups, sel_groups, top_two,
                                                 renorm, scale, idx, weights, w32, s);
  }
}

cudaError_t launch_router_backward(const void* logits, moe_dtype ldt, int64_t T, int E,
                                   const uint32_t* idx, int k, const float* dw, int scoring,
                                   int renorm, float scale, void* dlogits, float* w_out,
                                   cudaStream_t s) {
  dim3 grid((unsigned)((T + kRowsPerBlock - 1) / kRowsPerBlock));
  dim3 block(32 * kRowsPerBlock);
  const size_t smem = (size_t)kRowsPerBlock * (E + 128) * sizeof(float);
  switch (ldt) {
    case MOE_F32:
      router_backward_kernel<float><<<grid, block, smem, s>>>(
          static_cast<const float*>(logits), T, E, idx, k, dw, scoring, renorm, scale,
          static_cast<float*>(dlogits), w_out);
      break;
    case MOE_F16:
      router_backward_kernel<__half><<<grid, block, smem, s>>>(
          static_cast<const __half*>(logits), T, E, idx, k, dw, scoring, renorm, scale,
          static_cast<__half*>(dlogits), w_out);
      break;
    default:
      router_backward_kernel<__nv_bfloat16><<<grid, block, smem, s>>>(
          static_cast<const __nv_bfloat16*>(logits), T, E, idx, k, dw, scoring, renorm, scale,
          static_cast<__nv_bfloat16*>(dlogits), w_out);
  }
  return cudaGetLastError();
}

}  // namespace moe
