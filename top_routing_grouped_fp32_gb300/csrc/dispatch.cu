// dispatch.cu -- deterministic capacity-free dispatch.
//
// The ruDNN user guide ("ruDNN Benutzerhandbuch"), section 5 "Expertengewichte
// und Verteilung", asks for a dispatch that drops no token and keeps a stored
// map that restores token order; its own slot order inside an expert is left
// unspecified (atomic).  The DispatchedTokens comment in src/moe/experts.rs
// states the invariant: complete, monotone expert segments.  Here the slot
// order is fixed: segment e lists its slots s = t*k + j in ascending s, i.e. a
// stable counting sort of the slots by expert id, so the result is
// bit-reproducible.
//
// Three kernels:
//  1. count:   per 256-token chunk, a shared-memory histogram of experts
//              (column E counts indices >= E).  Order-independent atomics.
//  2. scan:    one block turns the chunk histograms into offsets[E+1] and the
//              first row of every (chunk, expert) pair; it also writes the
//              device status and fills the unused tail of perm/row_experts.
//              For a small histogram table (chunks * (E+1) <= 16384 words) the
//              scatter blocks do this themselves and the kernel is skipped.
//  3. scatter: each warp walks the slots of its 32 tokens in order, 32
//              consecutive slots per step; __match_any_sync ranks equal
//              experts among the lanes, so ranks follow s exactly, duplicates
//              included.  A first pass counts per warp, a second writes
//              perm/row_experts (and slot_row, the inverse of perm, for the
//              fused forward).
// A fourth kernel gathers x rows into x_disp: in the fused forward one warp
// per token, which reads the token's row once and writes its top_k rows;
// in moe_dispatch (and for rows that are not whole 16-byte vectors) one
// warp per dispatched row.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kWarps = kDispatchChunk / 32;  // 8 warps, 32 tokens each
// histogram tables up to this many words are scanned by every scatter block
// (at most 64 KiB of L2 reads per block, instead of a one-block scan kernel)
constexpr int64_t kFusedScanWords = 16384;

__global__ void __launch_bounds__(256)
count_kernel(const uint32_t* __restrict__ idx, int64_t T, int E, int k,
             uint32_t* __restrict__ chunk_counts) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ uint32_t cnt[];  // E + 1
  for (int i = threadIdx.x; i <= E; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  const int64_t t0 = (int64_t)blockIdx.x * kDispatchChunk;
  const int64_t t1 = min(T, t0 + kDispatchChunk);
  const int64_t s0 = t0 * k, s1 = t1 * k;
  for (int64_t s = s0 + threadIdx.x; s < s1; s += blockDim.x) {
    const uint32_t e = __ldg(idx + s);
    atomicAdd(&cnt[e < (uint32_t)E ? e : (uint32_t)E], 1u);
  }
  __syncthreads();
  uint32_t* out = chunk_counts + (size_t)blockIdx.x * (E + 1);
  for (int i = threadIdx.x; i <= E; i += blockDim.x) out[i] = cnt[i];
}

// Inclusive block scan of one value per thread (blockDim.x <= 1024).
__device__ uint32_t block_inclusive_scan(uint32_t v, uint32_t* warp_sums) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    uint32_t o = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v += o;
  }
  if (lane == 31) warp_sums[w] = v;
  __syncthreads();
  if (w == 0) {
    const int nw = (blockDim.x + 31) >> 5;
    uint32_t x = lane < nw ? warp_sums[lane] : 0u;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      uint32_t o = __shfl_up_sync(0xffffffffu, x, d);
      if (lane >= d) x += o;
    }
    if (lane < nw) warp_sums[lane] = x;
  }
  __syncthreads();
  if (w > 0) v += warp_sums[w - 1];
  __syncthreads();
  return v;
}

__device__ __forceinline__ uint32_t warp_inclusive_scan(uint32_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t o = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v += o;
  }
  return v;
}

// One block of 1024 threads (32 warps).  Each warp owns experts w, w+32, ...
// and walks their chunk columns 32 chunks at a time, so the per-expert chunk
// loops are parallel over lanes (they were the latency of this kernel).
__global__ void __launch_bounds__(1024)
scan_kernel(const uint32_t* __restrict__ chunk_counts, int nchunks, int E, int64_t N,
            uint32_t* __restrict__ offsets, uint32_t* __restrict__ chunk_base,
            uint32_t* __restrict__ perm, uint32_t* __restrict__ row_experts,
            uint32_t* __restrict__ status) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint32_t warp_sums[32];
  __shared__ uint32_t s_tot[1025];  // per-expert totals, then segment starts; [E] = invalid
  __shared__ uint32_t s_total_valid;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  // 1. totals per expert (and of the invalid column E)
  for (int e = w; e <= E; e += 32) {
    uint32_t sum = 0;
    for (int b = lane; b < nchunks; b += 32) sum += chunk_counts[(size_t)b * (E + 1) + e];
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, d);
    if (lane == 0) s_tot[e] = sum;
  }
  __syncthreads();
  // 2. exclusive scan of the totals: segment starts (thread e owns expert e)
  const int e = threadIdx.x;
  const uint32_t total = e < E ? s_tot[e] : 0u;
  const uint32_t invalid = s_tot[E];
  const uint32_t incl = block_inclusive_scan(total, warp_sums);
  if (e < E) {
    s_tot[e] = incl - total;
    offsets[e] = incl - total;
    if (e == E - 1) {
      offsets[E] = incl;
      s_total_valid = incl;
    }
  }
  if (threadIdx.x == 0 && status) *status = invalid ? (uint32_t)MOE_ERR_INVALID_INDEX : 0u;
  __syncthreads();
  // 3. first row of every (chunk, expert): the segment start plus the
  //    expert's counts in earlier chunks
  for (int ex = w; ex < E; ex += 32) {
    uint32_t run = s_tot[ex];
    for (int b0 = 0; b0 < nchunks; b0 += 32) {
      const int b = b0 + lane;
      const uint32_t c = b < nchunks ? chunk_counts[(size_t)b * (E + 1) + ex] : 0u;
      const uint32_t x = warp_inclusive_scan(c);
      if (b < nchunks) chunk_base[(size_t)b * E + ex] = run + x - c;
      run += __shfl_sync(0xffffffffu, x, 31);
    }
  }
  // slots that were not dispatched leave the tail of perm / row_experts unused
  for (int64_t r = (int64_t)s_total_valid + threadIdx.x; r < N; r += blockDim.x) {
    perm[r] = kInvalid;
    if (row_experts) row_experts[r] = kInvalid;
  }
}

// SCAN: the scan is done here too (two kernels instead of three).  Every
// block reads the whole chunk histogram table (small: the launcher takes this
// form when chunks * (E+1) <= kFusedScanWords) and forms the per-expert totals
// and its own chunk's first rows; block 0 also writes offsets, the status and
// the tail of perm / row_experts, as the scan kernel does otherwise.
template <bool SCAN>
__global__ void __launch_bounds__(256)
scatter_kernel(const uint32_t* __restrict__ idx, int64_t T, int E, int k,
               const uint32_t* __restrict__ chunk_base, uint32_t* __restrict__ perm,
               uint32_t* __restrict__ row_experts, uint32_t* __restrict__ slot_row,
               const uint32_t* __restrict__ chunk_counts, int nchunks, uint32_t* __restrict__ offsets,
               uint32_t* __restrict__ status) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ uint32_t smem[];
  uint32_t* wcnt = smem;                 // [kWarps][E]: per-warp counters / running bases
  uint32_t* sidx = smem + kWarps * E;    // this chunk's idx slice, [tokens][k]
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kWarps * E; i += blockDim.x) wcnt[i] = 0;
  // one coalesced load of the chunk's indices; the walks below read them from
  // shared memory instead of issuing a dependent L2 load per token
  const int64_t tc0 = (int64_t)blockIdx.x * kDispatchChunk;
  const int64_t nslots = (min(T, tc0 + kDispatchChunk) - tc0) * k;
  for (int64_t i = threadIdx.x; i < nslots; i += blockDim.x) sidx[i] = __ldg(idx + tc0 * k + i);
  uint32_t* s_base = sidx + kDispatchChunk * k;  // SCAN: [E+1] this chunk's first rows
  if constexpr (SCAN) {
    uint32_t* s_tot = s_base + (E + 1);           // [E+1] totals, then segment starts
    __shared__ uint32_t warp_sums[32];
    __shared__ uint32_t s_valid;
    // per expert (and the invalid column E): the total over all chunks and
    // the part in the chunks before this one.  The table is read flat, 8
    // words per thread in flight, and summed with shared-memory integer
    // atomics (exact in any order).
    for (int i = threadIdx.x; i <= E; i += blockDim.x) s_tot[i] = s_base[i] = 0u;
    __syncthreads();
    const int64_t words = (int64_t)nchunks * (E + 1);
    const int64_t before = (int64_t)blockIdx.x * (E + 1);  // flat indices of earlier chunks
    for (int64_t f0 = threadIdx.x; f0 < words; f0 += 8 * (int64_t)blockDim.x) {
      uint32_t v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int64_t f = f0 + q * (int64_t)blockDim.x;
        v[q] = f < words ? __ldg(chunk_counts + f) : 0u;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int64_t f = f0 + q * (int64_t)blockDim.x;
        if (v[q] != 0u) {
          const int e = (int)(f % (E + 1));
          atomicAdd(&s_tot[e], v[q]);
          if (f < before) atomicAdd(&s_base[e], v[q]);
        }
      }
    }
    __syncthreads();
    // exclusive scan of the totals over experts, 4 experts per thread (E <= 1024)
    const int e0 = threadIdx.x * 4;
    uint32_t v[4], loc = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[i] = e0 + i < E ? s_tot[e0 + i] : 0u;
      loc += v[i];
    }
    const uint32_t incl = block_inclusive_scan(loc, warp_sums);
    const uint32_t invalid = s_tot[E];
    __syncthreads();  // every total read before the starts overwrite them
    uint32_t run = incl - loc;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (e0 + i < E) {
        s_tot[e0 + i] = run;
        s_base[e0 + i] += run;
        if (blockIdx.x == 0) offsets[e0 + i] = run;
      }
      run += v[i];
    }
    if (threadIdx.x == blockDim.x - 1) s_valid = incl;
    __syncthreads();
    if (blockIdx.x == 0) {
      if (threadIdx.x == 0) {
        offsets[E] = s_valid;
        if (status) *status = invalid ? (uint32_t)MOE_ERR_INVALID_INDEX : 0u;
      }
      for (int64_t r = (int64_t)s_valid + threadIdx.x; r < T * k; r += blockDim.x) {
        perm[r] = kInvalid;
        if (row_experts) row_experts[r] = kInvalid;
      }
    }
  }
  __syncthreads();
  // warp w walks the slots s = t*k + j of its 32 tokens in order, 32
  // consecutive slots per step (a step may span tokens): lane order is slot
  // order, so __match_any_sync ranks equal experts exactly as the stable sort
  const int64_t tw = tc0 + w * 32;
  const int64_t s_begin = tw * k, s_end = min(T, tw + 32) * k, s_chunk = tc0 * k;
  uint32_t* my = wcnt + w * E;
  const uint32_t lt_mask = (1u << lane) - 1u;

  // pass 1: per-warp counts
  for (int64_t q = s_begin; q < s_end; q += 32) {
    const int64_t sl = q + lane;
    const uint32_t e = sl < s_end ? sidx[sl - s_chunk] : kInvalid;
    const bool ok = e < (uint32_t)E;
    const uint32_t grp = __match_any_sync(0xffffffffu, ok ? e : kInvalid);
    if (ok && (grp & lt_mask) == 0) my[e] += __popc(grp);
    __syncwarp();
  }
  __syncthreads();
  // per-expert exclusive prefix over the warps, starting at the chunk's base
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    uint32_t run = SCAN ? s_base[e] : chunk_base[(size_t)blockIdx.x * E + e];
    for (int ww = 0; ww < kWarps; ++ww) {
      const uint32_t c = wcnt[ww * E + e];
      wcnt[ww * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  // pass 2: the same walk, now writing rows
  for (int64_t q = s_begin; q < s_end; q += 32) {
    const int64_t sl = q + lane;
    const bool in = sl < s_end;
    const uint32_t e = in ? sidx[sl - s_chunk] : kInvalid;
    const bool ok = e < (uint32_t)E;
    const uint32_t grp = __match_any_sync(0xffffffffu, ok ? e : kInvalid);
    const uint32_t base = ok ? my[e] : 0u;
    __syncwarp();
    if (ok) {
      const uint32_t r = base + __popc(grp & lt_mask);
      perm[r] = (uint32_t)sl;
      if (row_experts) row_experts[r] = e;
      if (slot_row) slot_row[sl] = r;
      if ((grp & lt_mask) == 0) my[e] = base + __popc(grp);
    } else if (slot_row && in) {
      slot_row[sl] = kInvalid;  // not dispatched
    }
    __syncwarp();
  }
}

// x_disp[r,:] = x[perm[r] / k, :] for r < offsets[E]; one warp per row.
template <int VEC_BYTES>
__global__ void __launch_bounds__(256)
gather_kernel(const char* __restrict__ x, int64_t row_bytes, int k, const uint32_t* __restrict__ perm,
              const uint32_t* __restrict__ offsets, int E, int64_t N, char* __restrict__ x_disp) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= N) return;
  const uint32_t valid_rows = __ldg(offsets + E);
  if (r >= (int64_t)valid_rows) return;
  const int64_t t = __ldg(perm + r) / (uint32_t)k;
  const char* src = x + t * row_bytes;
  char* dst = x_disp + r * row_bytes;
  if constexpr (VEC_BYTES == 16) {
    const int64_t nv = row_bytes / 16;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    // 8 loads in flight per lane (a 4 KiB row in one round); x_disp is
    // written with evict-first stores so that it does not push the token
    // rows, each read top_k times, out of L2
    int64_t v = lane;
    for (; v + 7 * 32 < nv; v += 8 * 32) {
      uint4 q[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) q[i] = __ldg(s4 + v + 32 * i);
#pragma unroll
      for (int i = 0; i < 8; ++i) __stcs(d4 + v + 32 * i, q[i]);
    }
    for (; v < nv; v += 32) __stcs(d4 + v, __ldg(s4 + v));
  } else {
    const int64_t nv = row_bytes / 2;
    const uint16_t* s2 = reinterpret_cast<const uint16_t*>(src);
    uint16_t* d2 = reinterpret_cast<uint16_t*>(dst);
    for (int64_t v = lane; v < nv; v += 32) d2[v] = s2[v];
  }
}

// The same rows in token order: one warp per token reads its row once (a
// 4 KiB chunk per round, 8 loads in flight per lane) and writes it to each of
// its top_k dispatched rows, slot_row[t*k+j] (kInvalid: not dispatched).  A
// token row is then fetched from DRAM once, instead of top_k times far apart.
__global__ void __launch_bounds__(256)
gather_tokens_kernel(const uint4* __restrict__ x, int64_t vecs, int k, const uint32_t* __restrict__ slot_row,
                     int64_t T, uint4* __restrict__ x_disp) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  // lane j holds the rows of slots j and 32 + j (top_k <= 64)
  const uint32_t* sr = slot_row + t * k;
  const uint32_t r_lo = lane < k ? __ldg(sr + lane) : kInvalid;
  const uint32_t r_hi = lane + 32 < k ? __ldg(sr + 32 + lane) : kInvalid;
  const uint4* src = x + t * vecs;
  for (int64_t v0 = 0; v0 < vecs; v0 += 8 * 32) {
    uint4 q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int64_t v = v0 + 32 * i + lane;
      if (v < vecs) q[i] = __ldg(src + v);
    }
    for (int j = 0; j < k; ++j) {
      const uint32_t r = __shfl_sync(0xffffffffu, j < 32 ? r_lo : r_hi, j & 31);
      if (r == kInvalid) continue;
      uint4* dst = x_disp + (int64_t)r * vecs;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int64_t v = v0 + 32 * i + lane;
        if (v < vecs) __stcs(dst + v, q[i]);
      }
    }
  }
}

}  // namespace

size_t dispatch_scratch_bytes(int64_t T, int E) {
  const int64_t nc = dispatch_chunks(T);
  return align_up((size_t)nc * (E + 1) * 4, 256) + align_up((size_t)nc * E * 4, 256);
}

cudaError_t launch_dispatch(const uint32_t* idx, int64_t T, int E, int k, uint32_t* offsets,
                            uint32_t* row_experts, uint32_t* perm, void* scratch,
                            uint32_t* status, cudaStream_t s, uint32_t* slot_row) {
  const int64_t nc = dispatch_chunks(T);
  uint32_t* counts = static_cast<uint32_t*>(scratch);
  uint32_t* bases = reinterpret_cast<uint32_t*>(static_cast<char*>(scratch) +
                                                align_up((size_t)nc * (E + 1) * 4, 256));
  cudaError_t err = launch_pdl(count_kernel, dim3((unsigned)nc), dim3(256), (E + 1) * sizeof(uint32_t), s,
                               idx, T, E, k, counts);
  if (err != cudaSuccess) return err;
  // a small histogram table: every scatter block scans it itself
  const bool fused = nc * (E + 1) <= kFusedScanWords;
  if (!fused) {
    err = launch_pdl(scan_kernel, dim3(1), dim3(1024), 0, s, counts, (int)nc, E, T * k, offsets, bases,
                     perm, row_experts, status);
    if (err != cudaSuccess) return err;
  }
  // at most 8*1024 + 256*64 + 2*1025 words = 104 KiB
  const size_t smem = ((size_t)kWarps * E + (size_t)kDispatchChunk * k + (fused ? 2 * (E + 1) : 0)) *
                      sizeof(uint32_t);
  auto kern = fused ? scatter_kernel<true> : scatter_kernel<false>;
  if (smem > 48 * 1024) {  // large E * k: opt in
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(kern, dim3((unsigned)nc), dim3(256), smem, s, idx, T, E, k, bases, perm, row_experts,
                    slot_row, counts, (int)nc, offsets, status);
}

cudaError_t launch_gather_tokens(const void* x, moe_dtype dt, int64_t H, int k, const uint32_t* slot_row,
                                 int64_t T, void* x_disp, cudaStream_t s) {
  const int64_t row_bytes = H * (int64_t)dtype_size(dt);
  if (row_bytes % 16 != 0 || reinterpret_cast<uintptr_t>(x) % 16 != 0 ||
      reinterpret_cast<uintptr_t>(x_disp) % 16 != 0 || k > 64)
    return cudaErrorInvalidValue;
  return launch_pdl(gather_tokens_kernel, dim3((unsigned)((T + 7) / 8)), dim3(256), 0, s,
                    static_cast<const uint4*>(x), row_bytes / 16, k, slot_row, T,
                    static_cast<uint4*>(x_disp));
}

cudaError_t launch_gather(const void* x, moe_dtype dt, int64_t H, int k, const uint32_t* perm,
                          const uint32_t* offsets, int E, int64_t N, void* x_disp, cudaStream_t s) {
  const int64_t row_bytes = H * (int64_t)dtype_size(dt);
  const unsigned grid = (unsigned)((N + 7) / 8);
  const bool vec = row_bytes % 16 == 0 && reinterpret_cast<uintptr_t>(x) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(x_disp) % 16 == 0;
  if (vec)
    return launch_pdl(gather_kernel<16>, dim3(grid), dim3(256), 0, s, static_cast<const char*>(x),
                      row_bytes, k, perm, offsets, E, N, static_cast<char*>(x_disp));
  return launch_pdl(gather_kernel<2>, dim3(grid), dim3(256), 0, s, static_cast<const char*>(x),
                    row_bytes, k, perm, offsets, E, N, static_cast<char*>(x_disp));
}


// ---------------------------------------------------------------------------
// Dispatch without a caller workspace (moe_dispatch_noalloc).
//
// Some callers cannot hand this library any scratch memory and cannot let it
// allocate: an inference engine whose plugin interface only passes the
// tensors of the layer, or a serving loop that fixed its memory plan at
// start-up and treats any later cudaMalloc (which may synchronise the device)
// as a fault.  For them the chunk counts and chunk bases of the dispatch live
// in this fixed device array.  It is part of the library image: every GPU that
// loads the library holds these bytes until the process exits.
//
// The kernels read only scratch entries that the same call wrote first (the
// count kernel writes every count of every chunk, the scan writes every
// base), so nothing has to be cleared between calls.  All calls share the one
// array: two such calls whose kernels overlap on the GPU (different streams
// without ordering) race on it and give wrong results.
constexpr size_t kNoAllocScratchBytes = size_t(2) << 20;  // 2 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

size_t dispatch_noalloc_scratch_limit() { return kNoAllocScratchBytes; }

// Device address of g_noalloc_scratch in the current CUDA context.  The
// host-side name of the array is only a stand-in, so the address is looked up
// with cudaGetSymbolAddress (with the device current) the first time a context
// calls, and cached under that context's unique id (cuCtxGetId): a context
// created later on the same device -- after cudaDeviceReset, or a driver-API
// context of its own -- loads the module anew and gets its own lookup, so a
// stale address is never reused.  For runtime-API callers this is once per
// device.
namespace {
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
template <typename F>
F driver_fn(const char* name, int version) {
  void* f = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &f, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<F>(f);
}
}  // namespace

cudaError_t dispatch_noalloc_scratch(void** out) {
  constexpr int kSlots = 64;
  static std::mutex mu;
  static unsigned long long ids[kSlots] = {};
  static void* addr[kSlots] = {};
  static int next = 0;
  static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent", 4000);
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId", 12000);
  if (!get_current || !get_id) return cudaErrorNotSupported;
  std::lock_guard<std::mutex> lock(mu);
  CUcontext ctx = nullptr;
  void* p = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) {
    // no context yet on this thread (or the driver not yet initialised): the
    // lookup itself makes the device's primary context current
    cudaError_t err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (err != cudaSuccess) return err;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorInvalidDevice;
  }
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS || id == 0) return cudaErrorInvalidDevice;
  for (int i = 0; i < kSlots; ++i) {
    if (ids[i] == id) {
      *out = addr[i];
      return cudaSuccess;
    }
  }
  if (!p) {
    cudaError_t err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (err != cudaSuccess) return err;
  }
  ids[next] = id;  // contexts beyond kSlots replace the oldest entry
  addr[next] = p;
  next = (next + 1) % kSlots;
  *out = p;
  return cudaSuccess;
}

}  // namespace moe
