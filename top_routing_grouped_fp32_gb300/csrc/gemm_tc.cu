// gemm_tc.cu -- persistent segmented grouped GEMM on Blackwell tensor cores.
//
// Computes the three expert products of SwiGluExperts::forward_dispatched_with_
// strategy in src/moe/experts.rs (ruDNN 0.1.25 source view): for every
// dispatched row r of expert e, A[r,:] . W[e]^T, with
//   gate/up : both products in one accumulator tile, epilogue h = silu(g) * u
//             (silu(z) = z * sigmoid(z), MindSpeed-Ops PR 163, rms_norm_gated
//             notes), stored as the 16-bit operand of the down product;
//   down    : o = h . W_down[e]^T, stored either in dispatch order
//             (moe_experts_forward) or multiplied by the routing weight of
//             its slot and stored at that token slot (fused forward: the
//             weight scale and the un-permute of the user guide's combine,
//             section 6, move into this epilogue).
// The pages' own grouped product is a scalar or "cooperative matrix" loop
// (prior art); this is an sm_103a design:
//
//   * persistent CTAs over a tile list built on the device from offsets[]
//     (segment lengths are never read by the host); a tile is 128*PAIR rows
//     x 256 FP32 accumulator columns of one expert, except that on CTA pairs
//     a segment's last tile holding at most 128 rows runs as a half tile
//     (M = 128 over the pair, 64 rows per CTA), halving its padding;
//   * PAIR = 2 (the default): a cluster of two CTAs on two SMs runs one
//     tcgen05.mma.cta_group::2 of M=256: each CTA stages its own 128 rows of A
//     and one 128-row half of B (for gate/up: 64 gate rows and the same 64 up
//     rows, so that every accumulator lane holds gate and up of the same
//     features; for down: one half of the 256 down rows), so an SM moves
//     32 KiB per 64-deep k-block instead of 48 KiB; the forward products
//     ring three 128-deep stages of 64 KiB (KS = 2), the backward products
//     and long-K down projections six 64-deep ones; PAIR = 1 is the
//     single-CTA form (M=128, both B halves staged locally, 4 stages; a tile
//     of at most 32 rows loads A through a 32-row box);
//   * warp 0: TMA producer (cp.async.bulk.tensor, 128-byte swizzle); its
//     copies complete on the leader CTA's "full" barrier;
//   * warp 1: allocates 512 TMEM columns; in the leader CTA one thread issues
//     the MMAs (kind::f16, FP32 accumulate) and tcgen05.commit frees ring
//     stages and hands finished accumulators to both CTAs' epilogues;
//   * warps 2-5: epilogue; each reads its 32 TMEM lanes (= 32 tile rows) with
//     tcgen05.ld while the MMA fills the other accumulator;
//   * rows past the end of a segment are computed (the A box may run into the
//     next expert's rows or past the buffer, where TMA fills zeros) and never
//     stored, so segments of any length are handled without padding;
//   * tiles are visited expert by expert; inside an expert, column panels of
//     `panel` n-blocks are swept over all its m-tiles so that CTAs running at
//     the same time share weight tiles in L2;
//   * the same kernel runs the five products of the expert backward
//     (ExpertTrainingCache::backward in src/moe/experts.rs): operands may be
//     MN-major in shared memory (weights and row blocks read as stored, no
//     transposes), the weight-gradient products take a per-expert K range
//     over 64-padded rows, and their epilogues store FP32 tiles.
//
// Every wait on an mbarrier is bounded: after ~2 s the CTA records
// MOE_ERR_DEVICE_TIMEOUT in the workspace status word, stops issuing work,
// waits (bounded) for its own copies and MMAs in flight, frees its TMEM and
// returns.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace moe {

// Prebuilt TMA descriptors of one expert-weight set (gate, up [E,I,H]; down [E,H,I]).
struct TcWeights {
  CUtensorMap gate;  // CUtensorMap carries its own 64-byte alignment
  CUtensorMap up;
  CUtensorMap down;
  CUtensorMap gate64;  // 64-row boxes: the interleaved gate/up operand of CTA pairs
  CUtensorMap up64;
  int64_t E, I, H;
};

namespace tc {

constexpr int BM = 128;        // rows per CTA
constexpr int BN = 256;        // FP32 accumulator columns per tile
constexpr int BK = 64;         // 64 16-bit elements = one 128-byte swizzle row
constexpr int UMMA_K = 16;
constexpr uint32_t A_BYTES = BM * BK * 2;        // 16 KiB
constexpr uint32_t B_HALF_BYTES = 128 * BK * 2;  // 16 KiB
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr int MAX_E = 1024;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// KS: 64-deep K sub-blocks per ring stage.  KS = 2 (forward CTA-pair GEMMs,
// K-major operands) halves the barrier round trips and commits per MMA: one
// stage holds A sub-blocks 0..KS-1, then B sub-blocks 0..KS-1, each in the
// 128-byte-swizzled layout of one TMA box.
template <int PAIR, int KS = 1>
struct Cfg {
  static constexpr int STAGES = KS == 2 ? 3 : (PAIR == 1 ? 4 : 6);
  static constexpr uint32_t B_BYTES = (PAIR == 1 ? 2u : 1u) * B_HALF_BYTES;  // B staged per CTA per sub-block
  static constexpr uint32_t STAGE_BYTES = KS * (A_BYTES + B_BYTES);
  static constexpr int TILE_M = BM * PAIR;
};

struct Params {
  const uint32_t* offsets;
  int E;
  int nb;             // n-blocks per m-tile
  int panel;          // n-blocks per raster panel
  int k_blocks;       // k-blocks per tile: 64-deep, 128-deep when KS = 2
  int mode;
  int cols_per_tile;  // output columns per tile: 128 (gate/up) or 256 (down)
  int b1_row_off;     // row offset of the second B box inside the n-block
  int64_t n_out;
  void* out;
  const uint32_t* perm;
  const void* weights;
  int wdt;
  uint32_t* status;
  // backward products
  void* out2;          // second output (kSwigluBwd: a; kWgrad: rows >= split)
  const void* da;      // kSwigluBwd: da = dout W_down, 16-bit [rows, n_out]
  const uint32_t* pad; // pad[e] = sum over e' < e of roundup(rows of e', 64)
  // operand forms: A K-major (rows x K) or MN-major (K rows x M columns);
  // B K-major 3-D, MN-major 3-D (experts x K rows x N columns) or MN-major 2-D
  int a_mn;
  int b_form;
  int a_row_pad;       // A rows live in the 64-padded row space (row - offsets[e] + pad[e])
  int kb_split;        // > 0: k-blocks from here on read map B1 and A columns from a_k2 on
  int a_k2;
  // kWgrad: per-expert product over the padded row range [pad[e], pad[e+1])
  int wgrad;
  int mb;              // m-tiles per expert
  int64_t m_total;     // M of the product
  int64_t split;       // output rows per buffer (M, or I for the [dgate; dup] pair)
  // forward products on CTA pairs: a segment's last m-tile holding at most
  // 128 rows runs as a half tile, an M = 128 tcgen05.mma.cta_group::2 (64 rows
  // per CTA, A loaded through mapA64): half the MMA work of a padded 256-row tile
  int half_tails;
  // gate/up on CTA pairs: B is staged interleaved, each CTA's 128-row half of
  // the N = 256 operand being [64 gate rows | the same 64 up rows] (mapB0 /
  // mapB1 then have 64-row boxes), so that every accumulator lane holds the
  // gate and up values of the same features in both tile forms
  int b_inter;
  int v8_out;  // out rows are 32-byte aligned segments (n_out % 16 == 0, 32-byte base)
  // single CTAs (decode-sized batches): a tile of at most 32 rows loads A
  // through a 32-row box (the mapA64 slot); the MMA still runs M = 128, and
  // its other 96 rows multiply whatever the ring stage held before -- rows
  // that are never stored
  int thin_a;
};

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t global_timer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// shared::cluster address of the same shared variable in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                   "memory");
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
template <bool CLUSTER>
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  if constexpr (CLUSTER) {
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 P, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, P;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, P;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
  }
  return ok != 0;
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// arrival on a barrier of another CTA of the cluster (shared::cluster address)
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cbar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cbar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
// Bounded wait for phase `parity` of `bar`.  Returns false if the CTA is
// aborting or the time limit passed (then the abort flag and status are set).
template <bool CLUSTER>
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                            uint32_t* status, uint64_t limit_ns) {
  const uint64_t t0 = global_timer();
  for (uint32_t n = 1;; ++n) {
    if (mbar_test<CLUSTER>(bar, parity)) return true;
    if ((n & 127u) == 0) {
      if (*abort_flag) return false;
      if (global_timer() - t0 > limit_ns) {
        *abort_flag = 1u;
        set_status(status, (uint32_t)MOE_ERR_DEVICE_TIMEOUT);
        return false;
      }
    }
  }
}
template <bool CLUSTER>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                          uint32_t* status, uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_test<CLUSTER>(bar, parity)) return true;  // fast path, inline
  return mbar_wait_slow<CLUSTER>(bar, parity, abort_flag, status, limit_ns);
}
// TMA tile loads into this CTA's shared memory.  PAIR == 2: the completion is
// counted on `bar`, a shared::cluster address that may be the leader CTA's.
template <int PAIR>
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar) {
  if constexpr (PAIR == 2) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
  } else {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
  }
}
template <int PAIR>
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t bar) {
  if constexpr (PAIR == 2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
  } else {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
  }
}
__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// TMEM allocation: PAIR == 2 allocates the same columns in both CTAs of the
// pair and is executed by one warp of each CTA.
template <int PAIR>
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t cols) {
  if constexpr (PAIR == 2) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
                 "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  } else {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
                 "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
}
template <int PAIR>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  if constexpr (PAIR == 2) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
                 : "memory");
  } else {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
                 : "memory");
  }
}
// D[tmem] (+)= A[smem] * B[smem]^T, both K-major, one (128*PAIR) x 256 x 16 step.
template <int PAIR>
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  if constexpr (PAIR == 2) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}
// Arrive on `bar` (same offset in every CTA of the pair) once all MMAs this
// thread issued have completed.  PAIR == 2: the arrival goes to both CTAs.
template <int PAIR>
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  if constexpr (PAIR == 2) {
    const uint16_t both = 3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"(both)
        : "memory");
  } else {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
  }
}
// Arrive on the issuing CTA's own `bar` once all its MMAs have completed.
template <int PAIR>
__device__ __forceinline__ void umma_commit_local(uint32_t bar) {
  if constexpr (PAIR == 2) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
  } else {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
  }
}
// 32 consecutive FP32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// An empty statement that the compiler must treat as rewriting r: placed after
// a wait, it keeps every use of r after that wait.
__device__ __forceinline__ void reg_fence(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),
                 "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]),
                 "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]),
                 "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]),
                 "+r"(r[31]));
}
// The same wait, naming the registers of a load still in flight as operands so
// that no use of them can be scheduled before it.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
        "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
        "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
        "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),
        "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
      :
      : "memory");
}

// 32 bytes (8 words) to a 32-byte-aligned global address: a whole sector per lane
__device__ __forceinline__ void st_v8(uint32_t* dst, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(w[0]), "r"(w[1]),
               "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// ---------------------------------------------------------------- epilogue stores
// Each lane of an epilogue warp holds one tile row; storing straight from
// registers would make every store instruction touch 32 rows.  Instead a
// warp's 32 rows x WORDS 32-bit words pass through its staging buffer (rows
// padded by 4 words against bank conflicts) and are written back CH = WORDS/4
// lanes per row, so each store instruction covers whole row segments
// (4 rows x 128 bytes for WORDS = 32, 8 rows x 64 bytes for WORDS = 16).
constexpr int STG_STRIDE = 36;                         // words per staged row
constexpr uint32_t STG_BYTES_PER_WARP = 32 * STG_STRIDE * 4;
constexpr uint32_t STG_BYTES = 4 * STG_BYTES_PER_WARP;  // 18 KiB

__device__ __forceinline__ void put4(uint32_t* w, uint4 q) {
  w[0] = q.x;
  w[1] = q.y;
  w[2] = q.z;
  w[3] = q.w;
}
// 32-bit words of a row segment that lie inside the output (cols_left >= 0)
template <typename V>
__device__ __forceinline__ int valid_words(int64_t cols_left) {
  const int64_t w = cols_left * (int64_t)sizeof(V) / 4;
  return w < 0 ? 0 : (int)(w < 32 ? w : 32);
}
// dst: this lane's row segment (nullptr: the row is not stored); the
// segment's first `valid` words are written (a multiple of 4).
template <int WORDS>
__device__ __forceinline__ void staged_store(uint32_t* stg, const uint32_t* w, uint32_t* dst, int valid,
                                             int lane) {
  constexpr int STRIDE = WORDS + 4;
  constexpr int CH = WORDS / 4;   // 16-byte chunks per row
  constexpr int RPI = 32 / CH;    // rows per store instruction
#pragma unroll
  for (int j = 0; j < CH; ++j)
    *reinterpret_cast<uint4*>(stg + lane * STRIDE + 4 * j) =
        make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  __syncwarp();
  const int j = lane % CH;
#pragma unroll
  for (int it = 0; it < CH; ++it) {
    const int r = lane / CH + RPI * it;
    const uint4 v = *reinterpret_cast<const uint4*>(stg + r * STRIDE + 4 * j);
    uint32_t* d = reinterpret_cast<uint32_t*>(
        __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(dst), r));
    if (d != nullptr && 4 * j < valid) *reinterpret_cast<uint4*>(d + 4 * j) = v;
  }
  __syncwarp();
}

// Shared-memory matrix descriptor of a K-major tile written by TMA with the
// 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4)      // start address
         | ((uint64_t)1 << 16)                     // leading offset (unused here)
         | ((uint64_t)(1024 >> 4) << 32)           // stride offset between 8-row groups
         | ((uint64_t)1 << 46)                     // descriptor version
         | ((uint64_t)2 << 61);                    // 128-byte swizzle
}
// The same for an MN-major tile: each TMA box holds 64 K rows of 64
// consecutive M (or N) elements, 128 bytes a row, swizzled in 8-row groups
// 1024 bytes apart (stride offset); boxes for the next 64 M/N elements follow
// 8 KiB apart (leading offset).
constexpr uint32_t MN_BOX_BYTES = 64 * BK * 2;  // 8 KiB
__device__ __forceinline__ uint64_t sw128_mn_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4)
         | ((uint64_t)(MN_BOX_BYTES >> 4) << 16)   // leading offset: next 64 M/N elements
         | ((uint64_t)(1024 >> 4) << 32)           // stride offset: next 8 K rows
         | ((uint64_t)1 << 46)
         | ((uint64_t)2 << 61);
}
enum BForm { kBKmajor3d = 0, kBMNmajor3d = 1, kBMNmajor2d = 2 };
// Instruction descriptor: FP32 accumulator, 16-bit A/B (bf16 or f16), both
// K-major (bits 15/16 set below make A/B MN-major), M = 128*PAIR, N = 256.
__host__ __device__ constexpr uint32_t make_idesc(bool bf16, int M) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---------------------------------------------------------------- tile list
struct Tile {
  int e;
  int nb;
  int64_t m0;  // first row of the (pair) tile
  int kx0;     // first K coordinate (0, or pad[e] for weight gradients)
  int nk;      // k-blocks of this tile
  bool half;   // M = 128 pair tile (64 rows per CTA): see Params::half_tails
  bool thin;   // single-CTA tile of at most 32 rows: see Params::thin_a
};

__device__ __forceinline__ Tile decode_tile(uint32_t tile, const Params& p, const uint32_t* s_pref,
                                            const uint32_t* s_off, int tile_m) {
  const uint32_t q = tile / (uint32_t)p.nb;
  int lo = 0, hi = p.E;  // s_pref[lo] <= q < s_pref[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_pref[mid] <= q) lo = mid; else hi = mid;
  }
  const uint32_t mte = s_pref[lo + 1] - s_pref[lo];
  const uint32_t L = tile - s_pref[lo] * (uint32_t)p.nb;
  const uint32_t w = (uint32_t)p.panel;
  const uint32_t pid = L / (mte * w);
  const uint32_t rem = L - pid * mte * w;
  const uint32_t width = min(w, (uint32_t)p.nb - pid * w);
  Tile t;
  t.e = lo;
  t.nb = (int)(pid * w + rem % width);
  t.m0 = (int64_t)s_off[lo] + (int64_t)(rem / width) * tile_m;
  t.kx0 = 0;
  t.nk = p.k_blocks;
  t.half = p.half_tails && (int64_t)s_off[lo + 1] - t.m0 <= BM;
  t.thin = p.thin_a && (int64_t)s_off[lo + 1] - t.m0 <= 32;
  return t;
}

// Weight-gradient tiles: expert-major, then m-tile, then n-block; the K range
// is the expert's padded column range of the transposed operands.
__device__ __forceinline__ Tile decode_wgrad(uint32_t tile, const Params& p, int tile_m) {
  const uint32_t per = (uint32_t)(p.mb * p.nb);
  Tile t;
  t.e = (int)(tile / per);
  const uint32_t rem = tile - (uint32_t)t.e * per;
  t.m0 = (int64_t)(rem / (uint32_t)p.nb) * tile_m;
  t.nb = (int)(rem % (uint32_t)p.nb);
  const uint32_t k0 = __ldg(p.pad + t.e), k1 = __ldg(p.pad + t.e + 1);
  t.kx0 = (int)k0;
  t.nk = (int)((k1 - k0) / BK);
  t.half = false;
  t.thin = false;
  return t;
}

// ---------------------------------------------------------------- the kernel
template <typename T, int PAIR, int KS>
__global__ void __launch_bounds__(THREADS, 1)
grouped_gemm_tc(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB0,
                const __grid_constant__ CUtensorMap mapB1, const __grid_constant__ CUtensorMap mapA64,
                const Params p) {
  using C = Cfg<PAIR, KS>;
  constexpr int STAGES = C::STAGES;
  constexpr bool kCluster = PAIR == 2;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t ring = (raw_s + 1023u) & ~1023u;  // 1024-byte aligned for the swizzle
  uint8_t* ring_ptr = smem_raw + (ring - raw_s);
  uint32_t* staging = reinterpret_cast<uint32_t*>(ring_ptr + STAGES * C::STAGE_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring_ptr + STAGES * C::STAGE_BYTES + STG_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  uint32_t* s_off = reinterpret_cast<uint32_t*>(ring_ptr + STAGES * C::STAGE_BYTES + STG_BYTES + 256);
  uint32_t* s_pref = s_off + (p.E + 1);

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;
  const uint32_t rank = kCluster ? cluster_rank() : 0u;  // this CTA's half of the pair tile
  const bool leader = rank == 0;
  const uint32_t cluster_id = blockIdx.x / PAIR, num_clusters = gridDim.x / PAIR;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 4 * PAIR);  // one arrival per epilogue warp of every CTA
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    prefetch_map(&mapA);
    if (p.half_tails || p.thin_a) prefetch_map(&mapA64);
    prefetch_map(&mapB0);
    prefetch_map(&mapB1);
  }
  if (warp == 1) tmem_alloc<PAIR>(smem_u32(tmem_slot), TMEM_COLS);
  // everything above overlaps the predecessor kernel (programmatic launch);
  // from here on the kernel reads what earlier kernels wrote
  pdl_wait();
  pdl_trigger();
  for (int i = threadIdx.x; i <= E; i += THREADS) s_off[i] = p.offsets[i];
  __syncthreads();
  if (warp == 2) {  // s_pref[e] = number of (128*PAIR)-row tiles of experts < e
    const int per = (E + 31) / 32;
    uint32_t loc = 0;
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      if (e < E) loc += (s_off[e + 1] - s_off[e] + C::TILE_M - 1) / C::TILE_M;
    }
    uint32_t incl = loc;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    uint32_t run = incl - loc;
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      if (e < E) {
        s_pref[e] = run;
        run += (s_off[e + 1] - s_off[e] + C::TILE_M - 1) / C::TILE_M;
      }
    }
    if (lane == 31) s_pref[E] = incl;
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (kCluster) cluster_sync();  // the peer's barriers exist before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t total_tiles =
      p.wgrad ? (uint32_t)E * (uint32_t)(p.mb * p.nb) : s_pref[E] * (uint32_t)p.nb;
  auto tile_at = [&](uint32_t tile) {
    return p.wgrad ? decode_wgrad(tile, p, C::TILE_M) : decode_tile(tile, p, s_pref, s_off, C::TILE_M);
  };
  // the leader CTA's barriers, as seen from this CTA
  const uint32_t full0_leader = kCluster ? mapa(full_bar(0), 0) : full_bar(0);
  const uint32_t tempty0_leader = kCluster ? mapa(tempty_bar(0), 0) : tempty_bar(0);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t last_fill[STAGES];
      bool filled[STAGES];
      for (int s = 0; s < STAGES; ++s) filled[s] = false, last_fill[s] = 0;
      bool ok = true;
      for (uint32_t tile = cluster_id; ok && tile < total_tiles; tile += num_clusters) {
        const Tile t = tile_at(tile);
        // A's row (K-major) or M column (MN-major) of this CTA's half: 128
        // rows, or 64 for a half tile
        int a_row = (int)(t.m0 + (int64_t)rank * (t.half ? BM / 2 : BM));
        if (p.a_row_pad) a_row += (int)(__ldg(p.pad + t.e) - s_off[t.e]);
        const int b0row = t.nb * p.cols_per_tile;
        const int b1row = b0row + p.b1_row_off;
        // interleaved gate/up B (pairs): this CTA's 64 gate rows and the same 64 up rows
        const int birow = b0row + (int)rank * 64;
        const CUtensorMap* ma = (t.half || t.thin) ? &mapA64 : &mapA;
        const uint32_t stage_tx = t.half   ? (C::STAGE_BYTES - KS * A_BYTES / 2) * PAIR
                                  : t.thin ? (C::STAGE_BYTES - KS * (A_BYTES - A_BYTES / 4)) * PAIR
                                           : C::STAGE_BYTES * PAIR;
        for (int kb = 0; kb < t.nk; ++kb) {
          if (!mbar_wait<kCluster>(empty_bar(stage), phase ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const uint32_t sa = ring + stage * C::STAGE_BYTES;
          const uint32_t fb = full0_leader + 8u * stage;
          // K coordinates of this k-block: A's, and B's (row or column)
          const bool second = p.kb_split > 0 && kb >= p.kb_split;  // [dg | du] . [W_gate ; W_up]: up half
          const int kx = second ? p.a_k2 + (kb - p.kb_split) * BK : t.kx0 + kb * BK * KS;
          const int kb_b = second ? (kb - p.kb_split) * BK : t.kx0 + kb * BK;
          const CUtensorMap* mb = second ? &mapB1 : &mapB0;
          if (leader) mbar_expect_tx(full_bar(stage), stage_tx);
          if constexpr (KS == 2) {  // K-major A and B only: KS sub-blocks of 64
#pragma unroll
            for (int sub = 0; sub < KS; ++sub) {
              const int kxs = kx + sub * BK;
              const uint32_t sbs = sa + KS * A_BYTES + sub * C::B_BYTES;
              tma_load_2d<PAIR>(sa + sub * A_BYTES, ma, kxs, a_row, fb);
              if constexpr (PAIR == 1) {
                tma_load_3d<PAIR>(sbs, &mapB0, kxs, b0row, t.e, fb);
                tma_load_3d<PAIR>(sbs + B_HALF_BYTES, &mapB1, kxs, b1row, t.e, fb);
              } else if (p.b_inter) {
                tma_load_3d<PAIR>(sbs, &mapB0, kxs, birow, t.e, fb);
                tma_load_3d<PAIR>(sbs + B_HALF_BYTES / 2, &mapB1, kxs, birow, t.e, fb);
              } else if (leader) {
                tma_load_3d<PAIR>(sbs, &mapB0, kxs, b0row, t.e, fb);
              } else {
                tma_load_3d<PAIR>(sbs, &mapB1, kxs, b1row, t.e, fb);
              }
            }
          } else if (p.a_mn) {  // two 64-column boxes of this CTA's 128 M values
            tma_load_2d<PAIR>(sa, &mapA, a_row, kx, fb);
            tma_load_2d<PAIR>(sa + MN_BOX_BYTES, &mapA, a_row + 64, kx, fb);
          } else {
            tma_load_2d<PAIR>(sa, ma, kx, a_row, fb);
          }
          if (KS == 2) {
            // loaded above
          } else if (p.b_form == kBKmajor3d) {
            if constexpr (PAIR == 1) {
              tma_load_3d<PAIR>(sa + A_BYTES, &mapB0, kx, b0row, t.e, fb);
              tma_load_3d<PAIR>(sa + A_BYTES + B_HALF_BYTES, &mapB1, kx, b1row, t.e, fb);
            } else if (p.b_inter) {
              tma_load_3d<PAIR>(sa + A_BYTES, &mapB0, kx, birow, t.e, fb);
              tma_load_3d<PAIR>(sa + A_BYTES + B_HALF_BYTES / 2, &mapB1, kx, birow, t.e, fb);
            } else if (leader) {
              tma_load_3d<PAIR>(sa + A_BYTES, &mapB0, kx, b0row, t.e, fb);
            } else {
              tma_load_3d<PAIR>(sa + A_BYTES, &mapB1, kx, b1row, t.e, fb);
            }
          } else {  // MN-major B: this CTA's N columns in boxes of 64
            const int n0 = t.nb * 256 + (PAIR == 2 ? (int)rank * 128 : 0);
#pragma unroll
            for (int j = 0; j < (PAIR == 2 ? 2 : 4); ++j) {
              const uint32_t dst = sa + A_BYTES + j * MN_BOX_BYTES;
              if (p.b_form == kBMNmajor3d) tma_load_3d<PAIR>(dst, mb, n0 + 64 * j, kb_b, t.e, fb);
              else tma_load_2d<PAIR>(dst, mb, n0 + 64 * j, kb_b, fb);
            }
          }
          filled[stage] = true;
          last_fill[stage] = phase;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && leader) {  // aborting: let the copies in flight land before exit
        for (int s = 0; s < STAGES; ++s) {
          if (!filled[s]) continue;
          const uint64_t t0 = global_timer();
          while (!mbar_test<kCluster>(full_bar(s), last_fill[s]) &&
                 global_timer() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader CTA)
    if (lane == 0 && leader) {
      const uint32_t idesc = make_idesc(sizeof(T) == 2 && !std::is_same<T, __half>::value, C::TILE_M) |
                             ((uint32_t)(p.a_mn != 0) << 15) | ((uint32_t)(p.b_form != kBKmajor3d) << 16);
      // half tile: M = 128 over the pair (the M field is bits 24-28, M >> 4)
      const uint32_t idesc_half = (idesc & ~(0x1Fu << 24)) | ((uint32_t)(C::TILE_M / 2 >> 4) << 24);
      // per 16-deep MMA step: 32 bytes along a K-major row, 16 rows of an MN-major box
      const uint32_t a_step = p.a_mn ? 16u * 128u : UMMA_K * 2u;
      const uint32_t b_step = p.b_form != kBKmajor3d ? 16u * 128u : UMMA_K * 2u;
      // descriptor bits other than the start address
      const uint64_t a_hi = p.a_mn ? sw128_mn_desc(0) : sw128_desc(0);
      const uint64_t b_hi = p.b_form != kBKmajor3d ? sw128_mn_desc(0) : sw128_desc(0);
      int stage = 0;
      uint32_t phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (uint32_t tile = cluster_id; ok && tile < total_tiles; tile += num_clusters) {
        const Tile tt = tile_at(tile);
        const int nk = tt.nk;  // 0 for an expert without rows (weight gradients)
        const uint32_t id = tt.half ? idesc_half : idesc;
        if (!mbar_wait<kCluster>(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait<kCluster>(full_bar(stage), phase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = ring + stage * C::STAGE_BYTES;
          const uint32_t sb = sa + KS * A_BYTES;
#pragma unroll
          for (int q = 0; q < KS * (BK / UMMA_K); ++q) {
            const int sub = q / (BK / UMMA_K), kk = q % (BK / UMMA_K);
            const uint32_t ak = sa + sub * A_BYTES + kk * a_step, bk = sb + sub * C::B_BYTES + kk * b_step;
            umma_f16<PAIR>(d_tmem, a_hi | ((ak & 0x3FFFFu) >> 4), b_hi | ((bk & 0x3FFFFu) >> 4), id,
                           (kb | q) != 0 ? 1u : 0u);
          }
          umma_commit<PAIR>(empty_bar(stage));  // ring stage free (in every CTA) once done
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit<PAIR>(tfull_bar(acc));  // accumulator ready for the epilogues
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      // every MMA this thread issued must be complete before TMEM is freed
      umma_commit_local<PAIR>(drain_bar);
      const uint64_t t0 = global_timer();
      while (!mbar_test<false>(drain_bar, 0) && global_timer() - t0 < kWaitLimitNs) {
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // this warp may access TMEM lanes 32*quarter .. +31
    uint32_t* stg = staging + quarter * (STG_BYTES_PER_WARP / 4);
    uint32_t acc = 0, acc_phase = 0;
    T* out = static_cast<T*>(p.out);
    for (uint32_t tile = cluster_id; tile < total_tiles; tile += num_clusters) {
      const Tile t = tile_at(tile);
      // full tile: lane l of quarter q is row 32q + l of this CTA's 128, all
      // N columns.  Half tile (M = 128 over the pair): the CTA's 64 rows sit
      // in lanes 0-63 with N columns 0-127 and again in lanes 64-127 with N
      // columns 128-255, each in TMEM columns 0-127; quarter q then holds rows
      // 32*(q & 1) + l and the N-column half q >> 1.
      const int row = t.half ? (quarter & 1) * 32 + lane : quarter * 32 + lane;
      const int nhalf = t.half ? quarter >> 1 : 0;
      const int64_t grow = t.m0 + (int64_t)rank * (t.half ? BM / 2 : BM) + row;
      const bool row_ok = p.wgrad ? grow < p.m_total : grow < (int64_t)s_off[t.e + 1];
      // the weighted epilogue's slot and routing weight: loaded before the
      // accumulator wait so that their latency overlaps the MMAs
      int64_t wslot = grow;
      float wscale = 1.f;
      if (p.mode == kDownWeighted && row_ok) {
        const uint32_t s = __ldg(p.perm + grow);
        wslot = s;
        wscale = load_dyn(p.weights, p.wdt, s);
      }
      int ok = 1;
      if (lane == 0) ok = mbar_wait<kCluster>(tfull_bar(acc), acc_phase, abort_flag, p.status) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * BN;
      if (p.mode == kGateUpSwiglu) {
        // h = silu(g) * u: stored straight from registers (one 16-byte vector
        // per 8 columns); this epilogue is not store-bound, and measured
        // faster without the staging round trip.  Interleaved B: accumulator
        // columns [128 b, 128 b + 64) hold gate features 64 b .. 64 b + 63 of
        // the tile (64 (b + nhalf) for a half tile) and the next 64 columns
        // the up values of the same features; otherwise gate columns 0-127,
        // up columns 128-255.
        const int fw = p.b_inter ? 64 : 128;       // features per block
        const int nblk = t.half ? 1 : 128 / fw;
        const int64_t col0 = (int64_t)t.nb * 128 + (int64_t)nhalf * 64;
        T* dst = out + grow * p.n_out + col0;
#pragma unroll 1
        for (int i32 = 0; i32 < nblk * fw; i32 += 32) {
          const int b = i32 / fw, c = i32 - b * fw;
          const uint32_t gcol = (uint32_t)(b * 2 * fw + c);
          uint32_t g[32], u[32];
          tmem_ld32(taddr + gcol, g);
          tmem_ld32(taddr + gcol + fw, u);
          tmem_wait_ld(g);
          reg_fence(u);
          if (row_ok) {
            uint32_t hw[16];
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              float f[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float gg = __uint_as_float(g[v * 8 + i]);
                const float uu = __uint_as_float(u[v * 8 + i]);
                // 16-bit output: the fast divide's ~2 ulp are far below its rounding
                f[i] = __fdividef(gg * uu, 1.f + __expf(-gg));
              }
              put4(hw + 4 * v, pack8<T>(f));
            }
            if (p.v8_out && col0 + i32 + 32 <= p.n_out) {
              uint32_t* d32 = reinterpret_cast<uint32_t*>(dst + i32);
              st_v8(d32, hw);
              st_v8(d32 + 8, hw + 8);
            } else {
#pragma unroll
              for (int v = 0; v < 4; ++v)
                if (col0 + i32 + v * 8 + 8 <= p.n_out)
                  *reinterpret_cast<uint4*>(dst + i32 + v * 8) =
                      make_uint4(hw[4 * v], hw[4 * v + 1], hw[4 * v + 2], hw[4 * v + 3]);
            }
          }
        }
      } else if (p.mode == kSwigluBwd) {
        // accumulators g = x . W_gate[e]^T, u = x . W_up[e]^T (recomputed); with
        // da = dout . W_down[e] (16-bit, from the previous product):
        // dg = da * u * silu'(g), du = da * silu(g) and the activation
        // a = silu(g) * u, stored in the 16-bit dtype in the 64-padded row
        // space (row - offsets[e] + pad[e]); the padding rows after an
        // expert's last row are written as zeros (a segment's padding ends
        // inside its last tile, half tiles included).  The gate and up
        // accumulator columns are laid out as in the forward gate/up product.
        const int fw = p.b_inter ? 64 : 128;
        const int64_t col0 = (int64_t)t.nb * 128 + (int64_t)nhalf * 64;  // this warp's first feature
        const int64_t I = p.n_out;
        const int64_t local = grow - (int64_t)s_off[t.e];
        const uint32_t pe = __ldg(p.pad + t.e);
        const bool zero_row = !row_ok && local < (int64_t)(__ldg(p.pad + t.e + 1) - pe);
        const int64_t prow = (int64_t)pe + local;
        const T* dasrc = static_cast<const T*>(p.da) + grow * I + col0;
        const bool store = row_ok || zero_row;
        uint32_t* dgp = store ? reinterpret_cast<uint32_t*>(out + prow * 2 * I + col0) : nullptr;
        uint32_t* dup_p = store ? reinterpret_cast<uint32_t*>(out + prow * 2 * I + I + col0) : nullptr;
        uint32_t* ap = store ? reinterpret_cast<uint32_t*>(static_cast<T*>(p.out2) + prow * I + col0) : nullptr;
        // da of this row (16-bit), 32 columns per chunk; the next chunk's loads
        // are issued before the current chunk is computed so that their latency
        // overlaps the TMEM reads and the arithmetic
        auto load_da = [&](int c, float (&d)[32]) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 q = make_uint4(0u, 0u, 0u, 0u);
            if (row_ok && col0 + c + v * 8 + 8 <= I) q = __ldg(reinterpret_cast<const uint4*>(dasrc + c + v * 8));
            unpack8<T>(q, d + v * 8);
          }
        };
        // NF features of this warp: 128 (full tile) or 64 (half tile)
        auto features = [&](auto nf) {
        constexpr int NF = decltype(nf)::value;
        float dcur[32];
        load_da(0, dcur);
#pragma unroll
        for (int c = 0; c < NF; c += 32) {
          float dnext[32];
          if (c + 32 < NF) load_da(c + 32, dnext);
          const int b = c / fw;
          const uint32_t gcol = (uint32_t)(b * 2 * fw + (c - b * fw));
          uint32_t g[32], u[32], wdg[16], wdu[16], wa[16];
          tmem_ld32(taddr + gcol, g);
          tmem_ld32(taddr + gcol + fw, u);
          tmem_wait_ld(g);
          reg_fence(u);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            float fdg[8], fdu[8], fa[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              // padding rows (and rows not stored) have da = 0 and store zeros
              const float gg = row_ok ? __uint_as_float(g[v * 8 + i]) : 0.f;
              const float uu = row_ok ? __uint_as_float(u[v * 8 + i]) : 0.f;
              const float dv = dcur[v * 8 + i];
              const float sg = __fdividef(1.f, 1.f + __expf(-gg));  // 16-bit outputs
              const float silu = gg * sg;
              fdg[i] = dv * uu * (sg + silu * (1.f - sg));
              fdu[i] = dv * silu;
              fa[i] = silu * uu;
            }
            put4(wdg + 4 * v, pack8<T>(fdg));
            put4(wdu + 4 * v, pack8<T>(fdu));
            put4(wa + 4 * v, pack8<T>(fa));
          }
          const int vw = valid_words<T>(I - col0 - c);
          staged_store<16>(stg, wdg, dgp ? dgp + c / 2 : nullptr, vw, lane);
          staged_store<16>(stg, wdu, dup_p ? dup_p + c / 2 : nullptr, vw, lane);
          staged_store<16>(stg, wa, ap ? ap + c / 2 : nullptr, vw, lane);
          if (c + 32 < NF) {
#pragma unroll
            for (int i = 0; i < 32; ++i) dcur[i] = dnext[i];
          }
        }
        };
        if (t.half) features(std::integral_constant<int, 64>{});
        else features(std::integral_constant<int, 128>{});
      } else if (p.mode == kWgrad) {
        // FP32 rows of a weight-gradient tile (rows at or past `split` go to
        // out2; an expert without rows gets zeros).  A half tile's warp holds
        // 128 of the 256 columns.
        const int64_t col0 = (int64_t)t.nb * 256 + (int64_t)nhalf * 128;
        float* rowf = nullptr;
        if (row_ok) {
          if (grow < p.split)
            rowf = static_cast<float*>(p.out) + ((int64_t)t.e * p.split + grow) * p.n_out + col0;
          else
            rowf = static_cast<float*>(p.out2) +
                   ((int64_t)t.e * (p.m_total - p.split) + grow - p.split) * p.n_out + col0;
        }
        uint32_t* rowp = reinterpret_cast<uint32_t*>(rowf);
        const bool empty = t.nk == 0;
        if (empty) {
          uint32_t z[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) z[i] = 0u;
#pragma unroll 1
          for (int c = 0; c < 256; c += 32)
            staged_store<32>(stg, z, rowp ? rowp + c : nullptr, valid_words<float>(p.n_out - col0 - c), lane);
        } else {
          // the next 32 columns are read from TMEM while this chunk is stored
          auto chunks = [&](auto nch) {
            constexpr int NCH = decltype(nch)::value;
            uint32_t ob[2][32];
            tmem_ld32(taddr, ob[0]);
            tmem_wait_ld(ob[0]);
#pragma unroll
            for (int ci = 0; ci < NCH; ++ci) {
              const int c = ci * 32;
              if (ci + 1 < NCH) tmem_ld32(taddr + c + 32, ob[(ci + 1) & 1]);
              staged_store<32>(stg, ob[ci & 1], rowp ? rowp + c : nullptr,
                               valid_words<float>(p.n_out - col0 - c), lane);
              if (ci + 1 < NCH) tmem_wait_ld(ob[(ci + 1) & 1]);
            }
          };
          if (t.half) chunks(std::integral_constant<int, 4>{});
          else chunks(std::integral_constant<int, 8>{});
        }
      } else {
        // the next 32 columns are read from TMEM while this chunk is scaled,
        // packed and stored.  A half tile's warp holds 128 of the 256 columns.
        const int64_t col0 = (int64_t)t.nb * 256 + (int64_t)nhalf * 128;
        uint32_t* rowp = row_ok ? reinterpret_cast<uint32_t*>(out + wslot * p.n_out + col0) : nullptr;
        // NCH 32-column chunks: 8 for a full tile, 4 for a half tile (a
        // compile-time count in each form, so the double buffer stays in registers)
        auto chunks = [&](auto nch) {
          constexpr int NCH = decltype(nch)::value;
          uint32_t ob[2][32];
          tmem_ld32(taddr, ob[0]);
          tmem_wait_ld(ob[0]);
#pragma unroll
          for (int ci = 0; ci < NCH; ++ci) {
            const int c = ci * 32;
            if (ci + 1 < NCH) tmem_ld32(taddr + c + 32, ob[(ci + 1) & 1]);
            const uint32_t* o = ob[ci & 1];
            uint32_t w[16];
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              float f[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(o[v * 8 + i]) * wscale;
              put4(w + 4 * v, pack8<T>(f));
            }
            if (p.v8_out && col0 + c + 32 <= p.n_out) {  // warp-uniform: whole 64-byte row segments
              if (rowp) {
                st_v8(rowp + c / 2, w);
                st_v8(rowp + c / 2 + 8, w + 8);
              }
            } else {
              staged_store<16>(stg, w, rowp ? rowp + c / 2 : nullptr, valid_words<T>(p.n_out - col0 - c), lane);
            }
            if (ci + 1 < NCH) tmem_wait_ld(ob[(ci + 1) & 1]);
          }
        };
        if (t.half) chunks(std::integral_constant<int, 4>{});
        else chunks(std::integral_constant<int, 8>{});
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (kCluster) mbar_arrive_cluster(tempty0_leader + 8u * acc);
        else mbar_arrive(tempty_bar(acc));
      }
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  __syncthreads();
  // PAIR == 2: the leader's MMAs write the peer's TMEM and the peer arrives on
  // the leader's barriers, so neither CTA frees TMEM or exits before both are done
  if constexpr (kCluster) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<PAIR>(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- self-test
// Exercises the path every bounded wait of this file takes when it gives up:
// one warp waits on an mbarrier that nothing will complete; after limit_ns
// the wait records MOE_ERR_DEVICE_TIMEOUT in the status word and the kernel
// returns normally, leaving the context usable.
__global__ void bounded_wait_selftest(uint32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait<false>(smem_u32(&bar), 0, &abort_flag, status, limit_ns);
  __syncthreads();
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

CUtensorMapDataType tmap_type(moe_dtype dt) {
  return dt == MOE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

// rows x cols (cols contiguous), box `box_rows` (128, or 64) rows x 64 columns
bool encode_2d(CUtensorMap* m, const void* base, moe_dtype dt, uint64_t rows, uint64_t cols,
               uint32_t box_rows = 128) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  return fn(m, tmap_type(dt), 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// experts x rows x cols (cols contiguous), box 1 x `box_rows` (128, or 64) x 64
bool encode_3d(CUtensorMap* m, const void* base, moe_dtype dt, uint64_t E, uint64_t rows,
               uint64_t cols, uint32_t box_rows = 128) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {cols, rows, E};
  cuuint64_t strides[2] = {cols * 2, rows * cols * 2};
  cuuint32_t box[3] = {(cuuint32_t)BK, box_rows, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  return fn(m, tmap_type(dt), 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int PAIR, int KS = 1>
size_t smem_bytes(int E) {
  return 1024 + (size_t)Cfg<PAIR, KS>::STAGES * Cfg<PAIR, KS>::STAGE_BYTES + STG_BYTES + 256 +
         8 * (size_t)(E + 1);
}

// Clusters of PAIR CTAs that can be resident at once (one CTA per SM).
template <typename T, int PAIR, int KS = 1>
cudaError_t resident_clusters(int num_sms, int* out) {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  static int clusters = 0;
  std::call_once(once, [num_sms] {
    err = cudaFuncSetAttribute(grouped_gemm_tc<T, PAIR, KS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem_bytes<PAIR, KS>(MAX_E));
    if (err != cudaSuccess) return;
    if (PAIR == 1) {
      clusters = num_sms;
      return;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = PAIR;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(PAIR * (num_sms / PAIR));
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = smem_bytes<PAIR, KS>(MAX_E);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaOccupancyMaxActiveClusters(&clusters, grouped_gemm_tc<T, PAIR, KS>, &cfg);
  });
  *out = clusters;
  return err;
}

// mA64: A with 64-row boxes, for the half tiles of p.half_tails (else unused)
template <typename T, int PAIR, int KS = 1>
cudaError_t launch_t(int64_t N, int E, const CUtensorMap& mA, const CUtensorMap& mB0,
                     const CUtensorMap& mB1, Params p, int num_sms, cudaStream_t s,
                     const CUtensorMap* mA64 = nullptr) {
  if (!mA64 || PAIR != 2) p.half_tails = 0;
  if (!mA64 || PAIR != 1) p.thin_a = 0;
  int clusters = 0;
  cudaError_t err = resident_clusters<T, PAIR, KS>(num_sms, &clusters);
  if (err != cudaSuccess) return err;
  if (clusters < 1) return cudaErrorLaunchOutOfResources;
  constexpr int TM = Cfg<PAIR>::TILE_M;
  int64_t tiles_max;
  if (p.wgrad) {
    tiles_max = (int64_t)E * p.mb * p.nb;
  } else {
    const int64_t mt_max = (N + TM - 1) / TM + std::min<int64_t>(E, N);
    tiles_max = mt_max * p.nb;
  }
  const int nclu = (int)std::max<int64_t>(1, std::min<int64_t>(clusters, tiles_max));
  // panel width: about one wave of clusters spread over an expert's expected m-tiles
  const int64_t mt_per_expert = std::max<int64_t>(1, (N + (int64_t)TM * E - 1) / ((int64_t)TM * E));
  p.panel = (int)std::max<int64_t>(1, std::min<int64_t>(p.nb, (nclu + mt_per_expert - 1) / mt_per_expert));
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = PAIR;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(nclu * PAIR);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem_bytes<PAIR, KS>(E);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, grouped_gemm_tc<T, PAIR, KS>, mA, mB0, mB1, mA64 ? *mA64 : mA, p);
}

template <typename T>
cudaError_t launch_any(bool pair, int64_t N, int E, const CUtensorMap& mA, const CUtensorMap& mB0,
                       const CUtensorMap& mB1, const Params& p, int num_sms, cudaStream_t s,
                       const CUtensorMap* mA64 = nullptr) {
  return pair ? launch_t<T, 2>(N, E, mA, mB0, mB1, p, num_sms, s, mA64)
              : launch_t<T, 1>(N, E, mA, mB0, mB1, p, num_sms, s);
}

// ---------------------------------------------------------------- backward
// Scratch of the tensor-core expert backward; every buffer 1024-byte aligned.
// Row buffers marked P live in the 64-padded row space (npad rows).
struct BwdLayout {
  int64_t npad;  // >= pad[E] for any offsets: N + 63 E
  size_t pad, da, dgduP, actP, xP, doutP, total;
};

BwdLayout bwd_layout(int64_t N, int E, int64_t H, int64_t I) {
  BwdLayout L{};
  L.npad = N + 63 * (int64_t)E;
  size_t off = 0;
  auto take = [&off](size_t bytes) {
    const size_t at = off;
    off += (bytes + 1023) & ~(size_t)1023;
    return at;
  };
  L.pad = take((size_t)(E + 1) * 4);
  L.da = take((size_t)N * I * 2);
  L.dgduP = take((size_t)L.npad * 2 * I * 2);
  L.actP = take((size_t)L.npad * I * 2);
  L.xP = take((size_t)L.npad * H * 2);
  L.doutP = take((size_t)L.npad * H * 2);
  L.total = off;
  return L;
}

// rows x cols (cols contiguous), box 64 rows x 64 columns: an MN-major operand
bool encode_2d_mn(CUtensorMap* m, const void* base, moe_dtype dt, uint64_t rows, uint64_t cols) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64u, (cuuint32_t)BK};
  cuuint32_t estr[2] = {1u, 1u};
  return fn(m, tmap_type(dt), 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// experts x rows x cols (cols contiguous), box 1 x 64 x 64: an MN-major weight operand
bool encode_3d_mn(CUtensorMap* m, const void* base, moe_dtype dt, uint64_t E, uint64_t rows,
                  uint64_t cols) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {cols, rows, E};
  cuuint64_t strides[2] = {cols * 2, rows * cols * 2};
  cuuint32_t box[3] = {64u, (cuuint32_t)BK, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  return fn(m, tmap_type(dt), 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Products of the backward, each one launch of grouped_gemm_tc, every weight
// read in its stored layout (MN-major where the product needs it transposed):
//   1. da     = dout W_down (W_down MN-major), in the 16-bit dtype
//   2. g, u   = x W_gate^T, x W_up^T recomputed; the epilogue forms dg, du
//               and a from them and da, in the padded row space
//   3. dinput = dg W_gate + du W_up (weights MN-major; one accumulator over
//               the gate k-blocks, then the up k-blocks)
//   4. [dgate ; dup] = [dg | du]^T x per expert   (both operands MN-major over
//   5. ddown         = dout^T a per expert         the expert's padded rows)
template <typename T>
cudaError_t backward_t(const ExpertsBwdArgs& a, const TcWeights* w, char* ws, int num_sms, cudaStream_t s) {
  const int64_t N = a.N, H = a.H, I = a.I;
  const int E = a.E;
  const moe_dtype dt = a.dt;
  const BwdLayout L = bwd_layout(N, E, H, I);
  uint32_t* pad = reinterpret_cast<uint32_t*>(ws + L.pad);
  void* da = ws + L.da;
  void* dgduP = ws + L.dgduP;
  void* actP = ws + L.actP;
  void* xP = ws + L.xP;
  void* doutP = ws + L.doutP;
  cudaError_t err;
#define MOE_TC_TRY(x) \
  if ((err = (x)) != cudaSuccess) return err
  CUtensorMap mX, mDo, mDgduP, mWdMN, mWgMN, mWuMN, mDgduMN, mXMN, mDoMN, mActMN;
  CUtensorMap mX64, mDo64, mDgduP64;  // 64-row A boxes: half tiles of products 1-3
  if (!encode_2d(&mX64, a.x_disp, dt, N, H, 64) || !encode_2d(&mDo64, a.dout, dt, N, H, 64) ||
      !encode_2d(&mDgduP64, dgduP, dt, L.npad, 2 * I, 64))
    return cudaErrorInvalidValue;
  if (!encode_2d(&mX, a.x_disp, dt, N, H) || !encode_2d(&mDo, a.dout, dt, N, H) ||
      !encode_2d(&mDgduP, dgduP, dt, L.npad, 2 * I) || !encode_3d_mn(&mWdMN, a.down, dt, E, H, I) ||
      !encode_3d_mn(&mWgMN, a.gate, dt, E, I, H) || !encode_3d_mn(&mWuMN, a.up, dt, E, I, H) ||
      !encode_2d_mn(&mDgduMN, dgduP, dt, L.npad, 2 * I) || !encode_2d_mn(&mXMN, xP, dt, L.npad, H) ||
      !encode_2d_mn(&mDoMN, doutP, dt, L.npad, H) || !encode_2d_mn(&mActMN, actP, dt, L.npad, I))
    return cudaErrorInvalidValue;
  MOE_TC_TRY(launch_pad_offsets(a.offsets, E, pad, s));
  // x and dout into the padded row space on a side stream: they are needed
  // only by products 4 and 5 and co-run with products 1-3 (whose CTAs leave
  // registers and threads free on every SM).  While `s` is being captured
  // into a CUDA graph they run on `s` itself (no per-call stream then).
  cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
  MOE_TC_TRY(cudaStreamIsCapturing(s, &capture));
  if (capture != cudaStreamCaptureStatusNone) {
    MOE_TC_TRY(launch_pad_rows(a.x_disp, H, a.offsets, pad, E, L.npad, xP, s));
    MOE_TC_TRY(launch_pad_rows(a.dout, H, a.offsets, pad, E, L.npad, doutP, s));
  }
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  if (capture == cudaStreamCaptureStatusNone)
    MOE_TC_TRY(cudaStreamCreateWithFlags(&side, cudaStreamNonBlocking));
  if (side) {
    err = cudaEventCreateWithFlags(&fork, cudaEventDisableTiming);
    if (err == cudaSuccess) err = cudaEventCreateWithFlags(&join, cudaEventDisableTiming);
    if (err == cudaSuccess) err = cudaEventRecord(fork, s);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(side, fork, 0);
    if (err == cudaSuccess) err = launch_pad_rows(a.x_disp, H, a.offsets, pad, E, L.npad, xP, side);
    if (err == cudaSuccess) err = launch_pad_rows(a.dout, H, a.offsets, pad, E, L.npad, doutP, side);
    if (err == cudaSuccess) err = cudaEventRecord(join, side);
    // destroying them now is legal: their resources go once the work is done
    cudaStreamDestroy(side);
    if (fork) cudaEventDestroy(fork);
  }
  struct EventGuard {
    cudaEvent_t e;
    ~EventGuard() {
      if (e) cudaEventDestroy(e);
    }
  } join_guard{join};
  if (err != cudaSuccess) return err;
  const bool pair = N >= (int64_t)BM * E;
  Params base{};
  base.offsets = a.offsets;
  base.E = E;
  base.status = a.status;
  base.wdt = (int)MOE_F32;
  base.pad = pad;
  // 1. da = dout W_down, stored in the 16-bit dtype
  Params p = base;
  p.mode = kDownPlain;
  p.b_form = kBMNmajor3d;
  p.k_blocks = (int)((H + BK - 1) / BK);
  p.cols_per_tile = 256;
  p.n_out = I;
  p.nb = (int)((I + 255) / 256);
  p.out = da;
  p.half_tails = 1;
  MOE_TC_TRY(launch_any<T>(pair, N, E, mDo, mWdMN, mWdMN, p, num_sms, s, &mDo64));
  // 2. g, u recomputed; epilogue: dg, du, a (padded rows)
  p = base;
  p.mode = kSwigluBwd;
  p.k_blocks = (int)((H + BK - 1) / BK);
  p.cols_per_tile = 128;
  p.b1_row_off = 0;
  p.n_out = I;
  p.nb = (int)((I + 127) / 128);
  p.out = dgduP;
  p.out2 = actP;
  p.da = da;
  p.half_tails = 1;
  p.b_inter = pair;  // gate/up staged as in the forward's CTA-pair product
  MOE_TC_TRY(launch_any<T>(pair, N, E, mX, pair ? w->gate64 : w->gate, pair ? w->up64 : w->up, p, num_sms, s,
                           &mX64));
  // 3. dinput
  const int kbI = (int)((I + BK - 1) / BK);
  p = base;
  p.mode = kDownPlain;
  p.b_form = kBMNmajor3d;
  p.a_row_pad = 1;
  p.kb_split = kbI;
  p.a_k2 = (int)I;
  p.k_blocks = 2 * kbI;
  p.cols_per_tile = 256;
  p.n_out = H;
  p.nb = (int)((H + 255) / 256);
  p.out = a.dinput;
  p.half_tails = 1;
  MOE_TC_TRY(launch_any<T>(pair, N, E, mDgduP, mWgMN, mWuMN, p, num_sms, s, &mDgduP64));
  // 4-5. weight gradients over the padded rows (after the side stream's copies)
  if (join) MOE_TC_TRY(cudaStreamWaitEvent(s, join, 0));
  constexpr int TM = Cfg<2>::TILE_M;
  p = base;
  p.mode = kWgrad;
  p.wgrad = 1;
  p.a_mn = 1;
  p.b_form = kBMNmajor2d;
  p.cols_per_tile = 256;
  p.m_total = 2 * I;
  p.split = I;
  p.mb = (int)((2 * I + TM - 1) / TM);
  p.n_out = H;
  p.nb = (int)((H + 255) / 256);
  p.out = a.dgate;
  p.out2 = a.dup;
  MOE_TC_TRY((launch_t<T, 2>(N, E, mDgduMN, mXMN, mXMN, p, num_sms, s)));
  p.m_total = H;
  p.split = H;
  p.mb = (int)((H + TM - 1) / TM);
  p.n_out = I;
  p.nb = (int)((I + 255) / 256);
  p.out = a.ddown;
  p.out2 = a.ddown;
  MOE_TC_TRY((launch_t<T, 2>(N, E, mDoMN, mActMN, mActMN, p, num_sms, s)));
#undef MOE_TC_TRY
  return cudaSuccess;
}

}  // namespace tc

bool tc_supported(moe_dtype dt, int64_t I, int64_t H) {
  return (dt == MOE_BF16 || dt == MOE_F16) && I % 8 == 0 && H % 8 == 0;
}

TcWeights* tc_weights_create(const void* gate, const void* up, const void* down, moe_dtype dt,
                             int64_t E, int64_t I, int64_t H, const char** err) {
  if (!tc::encode_fn()) {
    *err = "cuTensorMapEncodeTiled is not available from the driver";
    return nullptr;
  }
  TcWeights* w = new TcWeights();
  w->E = E;
  w->I = I;
  w->H = H;
  if (!tc::encode_3d(&w->gate, gate, dt, E, I, H) || !tc::encode_3d(&w->up, up, dt, E, I, H) ||
      !tc::encode_3d(&w->down, down, dt, E, H, I) || !tc::encode_3d(&w->gate64, gate, dt, E, I, H, 64) ||
      !tc::encode_3d(&w->up64, up, dt, E, I, H, 64)) {
    *err = "cuTensorMapEncodeTiled rejected an expert weight tensor";
    delete w;
    return nullptr;
  }
  return w;
}

void tc_weights_destroy(TcWeights* w) { delete w; }

cudaError_t launch_bounded_wait_selftest(uint32_t* status, uint64_t limit_ns, cudaStream_t s) {
  tc::bounded_wait_selftest<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_gemm_tc(const GemmArgs& a, const TcWeights* w, int num_sms, cudaStream_t s) {
  CUtensorMap mA, mA64;
  if (!tc::encode_2d(&mA, a.A, a.dt, (uint64_t)a.N, (uint64_t)a.K) ||
      !tc::encode_2d(&mA64, a.A, a.dt, (uint64_t)a.N, (uint64_t)a.K, 64))
    return cudaErrorInvalidValue;
  tc::Params p{};
  p.offsets = a.offsets;
  p.E = a.E;
  p.mode = a.mode;
  p.n_out = a.n_out;
  p.out = a.out;
  p.perm = a.perm;
  p.weights = a.weights;
  p.wdt = (int)a.wdt;
  p.status = a.status;
  p.k_blocks = (int)((a.K + tc::BK - 1) / tc::BK);
  p.half_tails = 1;
  p.v8_out = a.n_out % 16 == 0 && reinterpret_cast<uintptr_t>(a.out) % 32 == 0;
  // CTA pairs halve the B bytes each SM stages per k-block; they pay off when
  // experts hold at least a full 128-row tile on average.  With fewer rows per
  // expert (decode-sized batches) the GEMM streams weights from HBM and single
  // CTAs keep twice as many independent streams in flight.
  const bool pair = a.N >= (int64_t)tc::BM * a.E;
  const CUtensorMap* b0;
  const CUtensorMap* b1;
  if (a.mode == kGateUpSwiglu) {
    p.cols_per_tile = 128;
    p.b1_row_off = 0;
    p.b_inter = pair;
    b0 = pair ? &w->gate64 : &w->gate;
    b1 = pair ? &w->up64 : &w->up;
  } else {
    p.cols_per_tile = 256;
    p.b1_row_off = 128;
    b0 = &w->down;
    b1 = &w->down;
  }
  p.nb = (int)((a.n_out + p.cols_per_tile - 1) / p.cols_per_tile);
  if (pair && a.mode != kGateUpSwiglu && a.K > 4096) {
    // long-K down projection: six 64-deep stages rather than three 128-deep
    // ones (the same ring bytes); 0.5-5 % faster at K = 14336, 3 % slower at
    // K = 1408 (same-box A/B)
    if (a.dt == MOE_BF16) return tc::launch_t<__nv_bfloat16, 2>(a.N, a.E, mA, *b0, *b1, p, num_sms, s, &mA64);
    return tc::launch_t<__half, 2>(a.N, a.E, mA, *b0, *b1, p, num_sms, s, &mA64);
  }
  if (pair) {  // 128-deep k-blocks, two 64-deep sub-blocks per ring stage
    p.k_blocks = (int)((a.K + 2 * tc::BK - 1) / (2 * tc::BK));
    if (a.dt == MOE_BF16)
      return tc::launch_t<__nv_bfloat16, 2, 2>(a.N, a.E, mA, *b0, *b1, p, num_sms, s, &mA64);
    return tc::launch_t<__half, 2, 2>(a.N, a.E, mA, *b0, *b1, p, num_sms, s, &mA64);
  }
  CUtensorMap mA32;
  if (!tc::encode_2d(&mA32, a.A, a.dt, (uint64_t)a.N, (uint64_t)a.K, 32)) return cudaErrorInvalidValue;
  p.thin_a = 1;
  if (a.dt == MOE_BF16) return tc::launch_t<__nv_bfloat16, 1>(a.N, a.E, mA, *b0, *b1, p, num_sms, s, &mA32);
  return tc::launch_t<__half, 1>(a.N, a.E, mA, *b0, *b1, p, num_sms, s, &mA32);
}

size_t experts_backward_tc_workspace(int64_t N, int E, int64_t H, int64_t I) {
  return tc::bwd_layout(N, E, H, I).total;
}

cudaError_t launch_experts_backward_tc(const ExpertsBwdArgs& a, const TcWeights* w, void* ws,
                                       int num_sms, cudaStream_t s) {
  char* base = static_cast<char*>(ws);
  if (a.dt == MOE_BF16) return tc::backward_t<__nv_bfloat16>(a, w, base, num_sms, s);
  return tc::backward_t<__half>(a, w, base, num_sms, s);
}

}  // namespace moe
