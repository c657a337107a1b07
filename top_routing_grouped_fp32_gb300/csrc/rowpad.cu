// rowpad.cu -- the 64-padded row space of the tensor-core expert backward
// (ExpertTrainingCache::backward in src/moe/experts.rs), and the check of the
// offsets a caller passes to the staged expert calls.
//
// The weight gradients are per-expert sums over that expert's dispatched
// rows.  The tcgen05 engine reads them 64 rows per k-block; if each expert's
// rows start on a multiple of 64 and are followed by zero rows up to the next
// multiple, no k-block mixes two experts and the zero rows add nothing:
//
//  * pad_offsets: pad[e] = sum_{e' < e} roundup(count_e', 64), pad[E] the total;
//  * pad_rows: dst row pad[e] + j = src row offsets[e] + j for j < count_e,
//    zero for count_e <= j < pad[e+1] - pad[e]  (rows of C 16-bit elements,
//    C a multiple of 8, copied in 16-byte vectors: one warp per row).
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

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

// The offsets of a staged expert call as its kernels read them: each clamped
// to [previous, N], so that no segment runs backwards or past the N rows of
// the buffers; a clamped entry marks the status word MOE_ERR_INVALID_INDEX.
// One warp: per-lane serial running maxima, then a warp max-scan (E <= 1024).
__global__ void sanitize_offsets_kernel(const uint32_t* __restrict__ in, int E, int64_t N,
                                        uint32_t* __restrict__ out, uint32_t* __restrict__ status) {
  const int lane = threadIdx.x;
  const int n = E + 1;
  const int per = (n + 31) / 32;
  const uint32_t cap = N < (int64_t)0xFFFFFFFFu ? (uint32_t)N : 0xFFFFFFFEu;
  uint32_t run = 0;
  for (int i = 0; i < per; ++i) {
    const int e = lane * per + i;
    if (e < n) {
      const uint32_t v = in[e];
      run = max(run, v < cap ? v : cap);
    }
  }
  uint32_t incl = run;  // max over this lane's entries and every earlier lane's
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl = max(incl, o);
  }
  uint32_t prev = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 0) prev = 0;
  bool bad = false;
  for (int i = 0; i < per; ++i) {
    const int e = lane * per + i;
    if (e < n) {
      const uint32_t v = in[e];
      const uint32_t c = max(prev, v < cap ? v : cap);
      out[e] = c;
      bad |= c != v;
      prev = c;
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(status, (uint32_t)MOE_ERR_INVALID_INDEX);
}

constexpr int kRowsPerBlock = 8;  // one warp per row

__global__ void __launch_bounds__(32 * kRowsPerBlock)
pad_rows_kernel(const uint4* __restrict__ src, int64_t vecs, const uint32_t* __restrict__ offsets,
                const uint32_t* __restrict__ pad, int E, uint4* __restrict__ dst) {
  const int64_t j = (int64_t)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);  // padded row
  const int lane = threadIdx.x & 31;
  if (j >= (int64_t)pad[E]) return;
  int lo = 0, hi = E;  // pad[lo] <= j < pad[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if ((int64_t)pad[mid] <= j) lo = mid; else hi = mid;
  }
  const int64_t r = (int64_t)offsets[lo] + (j - (int64_t)pad[lo]);
  uint4* d = dst + j * vecs;
  if (r < (int64_t)offsets[lo + 1]) {
    const uint4* s = src + r * vecs;
    for (int64_t v = lane; v < vecs; v += 32) d[v] = __ldg(s + v);
  } else {
    for (int64_t v = lane; v < vecs; v += 32) d[v] = make_uint4(0u, 0u, 0u, 0u);
  }
}

}  // namespace

cudaError_t launch_sanitize_offsets(const uint32_t* offsets, int E, int64_t N, uint32_t* out,
                                   uint32_t* status, cudaStream_t s) {
  sanitize_offsets_kernel<<<1, 32, 0, s>>>(offsets, E, N, out, status);
  return cudaGetLastError();
}

cudaError_t launch_pad_offsets(const uint32_t* offsets, int E, uint32_t* pad, cudaStream_t s) {
  pad_offsets_kernel<<<1, 32, 0, s>>>(offsets, E, pad);
  return cudaGetLastError();
}

cudaError_t launch_pad_rows(const void* src, int64_t C, const uint32_t* offsets, const uint32_t* pad,
                            int E, int64_t npad_max, void* dst, cudaStream_t s) {
  const int64_t blocks = (npad_max + kRowsPerBlock - 1) / kRowsPerBlock;
  pad_rows_kernel<<<(unsigned)blocks, 32 * kRowsPerBlock, 0, s>>>(
      static_cast<const uint4*>(src), C / 8, offsets, pad, E, static_cast<uint4*>(dst));
  return cudaGetLastError();
}

}  // namespace moe
