// internal.h -- launchers shared between the translation units of the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// ---- routing (route.cu) ----------------------------------------------------
cudaError_t launch_route(const void* logits, moe_dtype ldt, int64_t T, int E, int k, int renorm,
                         uint32_t* idx, void* weights, float* w32, uint32_t* status_reset,
                         cudaStream_t s);

// selected router weights (FP32) and, when dw != nullptr, their logit gradient
cudaError_t launch_router_backward(const void* logits, moe_dtype ldt, int64_t T, int E,
                                   const uint32_t* idx, int k, const float* dw, int scoring,
                                   int renorm, float scale, void* dlogits, float* w_out,
                                   cudaStream_t s);
cudaError_t launch_route_sigmoid_grouped(const void* logits, moe_dtype ldt, int64_t T, int E,
                                         const float* bias, int k, int groups, int sel_groups,
                                         int top_two, int renorm, float scale, uint32_t* idx,
                                         void* weights, float* w32, cudaStream_t s);

// ---- dispatch (dispatch.cu) ------------------------------------------------
constexpr int kDispatchChunk = 256;  // tokens per block of the dispatch kernels
inline int64_t dispatch_chunks(int64_t T) { return (T + kDispatchChunk - 1) / kDispatchChunk; }
// bytes of scratch the dispatch kernels need (chunk counts and chunk bases)
size_t dispatch_scratch_bytes(int64_t T, int E);
cudaError_t launch_dispatch(const uint32_t* idx, int64_t T, int E, int k, uint32_t* offsets,
                            uint32_t* row_experts, uint32_t* perm, void* scratch,
                            uint32_t* status, cudaStream_t s, uint32_t* slot_row = nullptr);
// x_disp in token order from the slot -> row map the scatter wrote (16-byte
// rows and pointers, top_k <= 64; cudaErrorInvalidValue otherwise)
cudaError_t launch_gather_tokens(const void* x, moe_dtype dt, int64_t H, int k, const uint32_t* slot_row,
                                 int64_t T, void* x_disp, cudaStream_t s);
// fixed device scratch for moe_dispatch_noalloc (size limit and address)
size_t dispatch_noalloc_scratch_limit();
cudaError_t dispatch_noalloc_scratch(void** out);
cudaError_t launch_gather(const void* x, moe_dtype dt, int64_t H, int k, const uint32_t* perm,
                          const uint32_t* offsets, int E, int64_t N, void* x_disp, cudaStream_t s);

// ---- combine (combine.cu) --------------------------------------------------
cudaError_t launch_invert_perm(const uint32_t* perm, int64_t N, uint32_t* slot_row, cudaStream_t s);
cudaError_t launch_combine(const void* expert_out, moe_dtype dt, const uint32_t* slot_row,
                           const void* weights, moe_dtype wdt, int64_t T, int k, int64_t H,
                           void* y, cudaStream_t s);
// dexpert[r] = w[perm[r]] * dy[t], dweights[perm[r]] = <expert_out[r], dy[t]>
cudaError_t launch_combine_backward(const void* expert_out, moe_dtype dt, const uint32_t* perm,
                                    const void* weights, moe_dtype wdt, const void* dy, int64_t T,
                                    int k, int64_t H, void* dexpert, float* dweights, cudaStream_t s);
// y[t] = sum_j slots[t*k+j] (weights already applied), ascending j
cudaError_t launch_slot_sum(const void* slots, moe_dtype dt, int64_t T, int k, int64_t H, void* y,
                            cudaStream_t s);

// ---- grouped GEMMs ---------------------------------------------------------
enum GemmMode {
  kGateUpSwiglu = 0,
  kDownPlain = 1,
  kDownWeighted = 2,
  // backward products (tcgen05 path only; da = dout W_down and dinput use kDownPlain)
  kSwigluBwd = 4,   // g, u recomputed, then [dg | du] (out) and a (out2), 16-bit
  kWgrad = 5,       // per-expert FP32 weight-gradient tiles over the padded rows
};

struct GemmArgs {
  int mode;
  moe_dtype dt;
  int E;
  int64_t N;          // rows of the A operand (dispatched rows)
  int64_t K;          // reduction length
  int64_t n_out;      // output columns (I for gate/up, H for down)
  const void* A;      // [N, K]
  const void* B0;     // gate (gate/up) or down weights
  const void* B1;     // up (gate/up) or nullptr
  const uint32_t* offsets;
  void* out;          // [N, n_out] (or [T*k, n_out] slots for weighted mode)
  const uint32_t* perm;
  const void* weights;
  moe_dtype wdt;
  uint32_t* status;
};

// Backward of the SwiGLU experts (gemm_bwd.cu): FP32 accumulate, any dtype.
struct ExpertsBwdArgs {
  moe_dtype dt;
  int E;
  int64_t N, H, I;
  const void* x_disp;   // [N, H]
  const void* dout;     // [N, H] gradient of the expert outputs
  const void* gate;     // [E, I, H]
  const void* up;       // [E, I, H]
  const void* down;     // [E, H, I]
  const uint32_t* offsets;
  float* g;             // [N, I] scratch: recomputed gate product
  float* u;             // [N, I] scratch: recomputed up product
  float* act;           // [N, I] scratch: silu(g) * u
  float* dg;            // [N, I] scratch
  float* du;            // [N, I] scratch
  void* dinput;         // [N, H] in dt
  float* dgate;         // [E, I, H]
  float* dup;           // [E, I, H]
  float* ddown;         // [E, H, I]
  uint32_t* status;     // device status word (bounded waits of the tensor-core path)
};
cudaError_t launch_experts_backward(const ExpertsBwdArgs& a, cudaStream_t s);

// offsets of a staged expert call, clamped to [previous, N] (rowpad.cu); a
// clamped entry sets MOE_ERR_INVALID_INDEX in *status
cudaError_t launch_sanitize_offsets(const uint32_t* offsets, int E, int64_t N, uint32_t* out,
                                   uint32_t* status, cudaStream_t s);
// The 64-padded row space of the tensor-core backward (rowpad.cu)
cudaError_t launch_pad_offsets(const uint32_t* offsets, int E, uint32_t* pad, cudaStream_t s);
cudaError_t launch_pad_rows(const void* src, int64_t C, const uint32_t* offsets, const uint32_t* pad,
                            int E, int64_t npad_max, void* dst, cudaStream_t s);

// SIMT FP32-accumulate path (gemm_simt.cu): any dtype and shape
cudaError_t launch_gemm_simt(const GemmArgs& a, cudaStream_t s);

// tcgen05 path (gemm_tc.cu): F16/BF16, K and n_out multiples of 8, 16-byte aligned
struct TcWeights;  // prebuilt tensor maps of one expert-weight set
TcWeights* tc_weights_create(const void* gate, const void* up, const void* down, moe_dtype dt,
                             int64_t E, int64_t I, int64_t H, const char** err);
void tc_weights_destroy(TcWeights* w);
cudaError_t launch_gemm_tc(const GemmArgs& a, const TcWeights* w, int num_sms, cudaStream_t s);
bool tc_supported(moe_dtype dt, int64_t I, int64_t H);
// Expert backward on the tcgen05 engine (F16/BF16): scratch of
// experts_backward_tc_workspace(...) bytes at `ws` (1024-byte aligned);
// a.g/u/act/dg/du are not used.
size_t experts_backward_tc_workspace(int64_t N, int E, int64_t H, int64_t I);
cudaError_t launch_experts_backward_tc(const ExpertsBwdArgs& a, const TcWeights* w, void* ws,
                                       int num_sms, cudaStream_t s);
// a kernel whose bounded wait is made to expire (failure-path self-test)
cudaError_t launch_bounded_wait_selftest(uint32_t* status, uint64_t limit_ns, cudaStream_t s);

}  // namespace moe
