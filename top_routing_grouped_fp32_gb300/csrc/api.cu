// api.cu -- the C ABI declared in include/moe.h: argument validation, the
// workspace layouts and the order of kernel launches on the caller's stream.
//
// Validation follows the rules of SwiGluExperts::new and
// forward_dispatched_with_strategy in src/moe/experts.rs (rank-3 weights of
// one float dtype, non-zero dimensions, up shape == gate shape, down ==
// [E,H,I], dispatch/expert agreement) and the routing contract of the user
// guide, section 4 (F32/F16/BF16 logits, 1 <= top_k <= E).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <functional>
#include <string>

#include "common.cuh"
#include "internal.h"

struct moe_experts {
  const void* gate;
  const void* up;
  const void* down;
  moe_dtype dt;
  int64_t E, I, H;
  int device;
  int num_sms;
  moe::TcWeights* tc;  // null when the tcgen05 path does not apply (FP32, odd sizes)
};

namespace {

using moe::align_up;
using moe::dtype_size;
using moe::kWsHeader;

thread_local std::string g_error;

moe_status fail(moe_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_error = buf;
  return st;
}

moe_status ok() {
  g_error.clear();
  return MOE_OK;
}

moe_status cuda_fail(cudaError_t e, const char* what) {
  return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define MOE_TRY_CUDA(expr, what)                   \
  do {                                             \
    cudaError_t _e = (expr);                       \
    if (_e != cudaSuccess) return cuda_fail(_e, what); \
  } while (0)

constexpr int64_t kMaxE = 1024, kMaxK = 64, kMaxDim = int64_t(1) << 20;
constexpr int64_t kMaxRows = (int64_t(1) << 31) - 1;

bool valid_dtype(moe_dtype d) { return d == MOE_F32 || d == MOE_F16 || d == MOE_BF16; }
bool aligned16(const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }
bool aligned256(const void* p) { return reinterpret_cast<uintptr_t>(p) % 256 == 0; }

// Checks shared by the calls that take (T, E, top_k).
moe_status check_tek(int64_t T, int64_t E, int32_t k) {
  if (T < 0) return fail(MOE_ERR_SHAPE, "T must be >= 0 (got %lld)", (long long)T);
  if (E < 1) return fail(MOE_ERR_SHAPE, "E must be >= 1 (got %lld)", (long long)E);
  if (k < 1 || k > E)
    return fail(MOE_ERR_INVALID_ARG, "top_k must satisfy 1 <= top_k <= E (top_k=%d, E=%lld)", k,
                (long long)E);
  if (E > kMaxE) return fail(MOE_ERR_UNSUPPORTED, "E=%lld exceeds the supported 1024", (long long)E);
  if (k > kMaxK) return fail(MOE_ERR_UNSUPPORTED, "top_k=%d exceeds the supported 64", k);
  if (T > kMaxRows / k)
    return fail(MOE_ERR_UNSUPPORTED, "T*top_k=%lld exceeds 2^31-1", (long long)T * k);
  return MOE_OK;
}

// GroupRoutingOptions rules of the user guide, section 10.
moe_status check_group_options(int64_t T, int64_t E, const moe_group_routing_options* o) {
  if (!o) return fail(MOE_ERR_INVALID_ARG, "group routing options are NULL");
  if (T < 0) return fail(MOE_ERR_SHAPE, "T must be >= 0 (got %lld)", (long long)T);
  if (E < 1 || E > kMaxE)
    return fail(E < 1 ? MOE_ERR_SHAPE : MOE_ERR_UNSUPPORTED, "expert count must be in 1..=1024 (got %lld)",
                (long long)E);
  if (o->groups < 1 || o->groups > 128)
    return fail(MOE_ERR_INVALID_ARG, "group count must be in 1..=128 (got %d)", o->groups);
  if (E % o->groups != 0)
    return fail(MOE_ERR_INVALID_ARG, "expert count %lld is not divisible by %d groups", (long long)E, o->groups);
  if (o->selected_groups < 1 || o->selected_groups > o->groups)
    return fail(MOE_ERR_INVALID_ARG, "selected_groups must be in 1..=groups (got %d of %d)",
                o->selected_groups, o->groups);
  const int64_t per = E / o->groups;
  if (o->top_k < 1 || o->top_k > 64)
    return fail(MOE_ERR_INVALID_ARG, "top_k must be in 1..=64 (got %d)", o->top_k);
  if (o->top_k > o->selected_groups * per)
    return fail(MOE_ERR_INVALID_ARG, "top_k=%d exceeds the %lld experts of the selected groups", o->top_k,
                (long long)(o->selected_groups * per));
  if (o->group_top_two && per < 2)
    return fail(MOE_ERR_INVALID_ARG, "group_top_two needs at least two experts per group");
  if (!(o->scale > 0.f) || !std::isfinite(o->scale))
    return fail(MOE_ERR_INVALID_ARG, "scale must be finite and positive");
  if (T > kMaxRows / o->top_k) return fail(MOE_ERR_UNSUPPORTED, "T*top_k exceeds 2^31-1");
  return MOE_OK;
}

moe_status check_dim(int64_t v, const char* name) {
  if (v < 1) return fail(MOE_ERR_SHAPE, "%s must be >= 1 (got %lld)", name, (long long)v);
  if (v > kMaxDim) return fail(MOE_ERR_UNSUPPORTED, "%s=%lld exceeds 2^20", name, (long long)v);
  return MOE_OK;
}

moe_status check_ws(const void* ws, size_t have, size_t need) {
  if (!ws) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
  if (!aligned256(ws)) return fail(MOE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (have < need)
    return fail(MOE_ERR_INVALID_ARG, "workspace too small: %zu bytes given, %zu needed", have, need);
  return MOE_OK;
}

moe_status check_handle(const moe_experts* x) {
  if (!x) return fail(MOE_ERR_INVALID_ARG, "experts handle is NULL");
  int dev = -1;
  MOE_TRY_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  if (dev != x->device)
    return fail(MOE_ERR_INVALID_ARG, "experts live on device %d but device %d is current", x->device,
                dev);
  return MOE_OK;
}

// ---- workspace layouts -----------------------------------------------------
struct Cursor {
  size_t off = kWsHeader;
  size_t take(size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 1024);
    return at;
  }
};

struct ForwardLayout {
  size_t idx, weights, offsets, perm, scratch, x_disp, h, slots, slot_row, total;
};

ForwardLayout forward_layout(const moe_experts* x, int64_t T, int32_t k, moe_dtype ldt) {
  const size_t N = (size_t)T * k, s = dtype_size(x->dt);
  Cursor c;
  ForwardLayout L;
  L.idx = c.take(N * 4);
  L.weights = c.take(N * dtype_size(ldt));
  L.offsets = c.take((size_t)(x->E + 1) * 4);
  L.perm = c.take(N * 4);
  L.scratch = c.take(moe::dispatch_scratch_bytes(T, (int)x->E));
  L.x_disp = c.take(N * (size_t)x->H * s);
  L.h = c.take(N * (size_t)x->I * s);
  L.slots = c.take(N * (size_t)x->H * s);
  L.slot_row = c.take(N * 4);
  L.total = c.off;
  return L;
}

template <typename P>
P* at(void* base, size_t off) {
  return reinterpret_cast<P*>(static_cast<char*>(base) + off);
}

uint32_t* status_word(void* ws) { return static_cast<uint32_t*>(ws); }

// Runs the two expert GEMMs: gate/up + SwiGLU into h, then down.
moe_status run_experts(const moe_experts* x, const void* x_disp, int64_t N, const uint32_t* offsets,
                       void* h, void* out, int down_mode, const uint32_t* perm, const void* weights,
                       moe_dtype wdt, uint32_t* status, cudaStream_t s, void* ev_mid) {
  moe::GemmArgs g{};
  g.dt = x->dt;
  g.E = (int)x->E;
  g.N = N;
  g.offsets = offsets;
  g.status = status;
  g.mode = moe::kGateUpSwiglu;
  g.A = x_disp;
  g.K = x->H;
  g.n_out = x->I;
  g.B0 = x->gate;
  g.B1 = x->up;
  g.out = h;
  cudaError_t e = x->tc ? moe::launch_gemm_tc(g, x->tc, x->num_sms, s) : moe::launch_gemm_simt(g, s);
  if (e != cudaSuccess) return cuda_fail(e, "gate/up grouped GEMM launch");
  if (ev_mid) MOE_TRY_CUDA(cudaEventRecord((cudaEvent_t)ev_mid, s), "cudaEventRecord");
  g.mode = down_mode;
  g.A = h;
  g.K = x->I;
  g.n_out = x->H;
  g.B0 = x->down;
  g.B1 = nullptr;
  g.out = out;
  g.perm = perm;
  g.weights = weights;
  g.wdt = wdt;
  e = x->tc ? moe::launch_gemm_tc(g, x->tc, x->num_sms, s) : moe::launch_gemm_simt(g, s);
  if (e != cudaSuccess) return cuda_fail(e, "down grouped GEMM launch");
  return MOE_OK;
}

// The routing step of a fused forward: writes idx [T,k] and weights [T,k]
// (logits dtype) on the stream.
using RouteFn = std::function<cudaError_t(uint32_t* idx, void* w, cudaStream_t s)>;

moe_status forward_core(moe_experts_t x, const void* xin, const void* logits, moe_dtype ldt,
                        int64_t T, int32_t k, const RouteFn& route, void* y, void* ws,
                        size_t ws_bytes, cudaStream_t s, void* const* ev);

moe_status forward_impl(moe_experts_t x, const void* xin, const void* logits, moe_dtype ldt,
                        int64_t T, int32_t k, int renorm, void* y, void* ws, size_t ws_bytes,
                        cudaStream_t s, void* const* ev) {
  moe_status st = check_handle(x);
  if (st != MOE_OK) return st;
  if (!valid_dtype(ldt)) return fail(MOE_ERR_DTYPE, "logits dtype %d is not F32/F16/BF16", (int)ldt);
  if ((st = check_tek(T, x->E, k)) != MOE_OK) return st;
  const int E = (int)x->E;
  RouteFn route = [=](uint32_t* idx, void* w, cudaStream_t st_) {
    return moe::launch_route(logits, ldt, T, E, k, renorm, idx, w, nullptr, nullptr, st_);
  };
  return forward_core(x, xin, logits, ldt, T, k, route, y, ws, ws_bytes, s, ev);
}

moe_status forward_core(moe_experts_t x, const void* xin, const void* logits, moe_dtype ldt,
                        int64_t T, int32_t k, const RouteFn& route, void* y, void* ws,
                        size_t ws_bytes, cudaStream_t s, void* const* ev) {
  moe_status st;
  if (T == 0) return ok();
  if (!xin || !logits || !y) return fail(MOE_ERR_INVALID_ARG, "x, logits and y must be non-NULL");
  if (!aligned16(xin) || !aligned16(y))
    return fail(MOE_ERR_INVALID_ARG, "x and y must be 16-byte aligned");
  const ForwardLayout L = forward_layout(x, T, k, ldt);
  if ((st = check_ws(ws, ws_bytes, L.total)) != MOE_OK) return st;
  const int64_t N = T * k;
  const int E = (int)x->E;
  uint32_t* status = status_word(ws);
  uint32_t* idx = at<uint32_t>(ws, L.idx);
  void* w = at<void>(ws, L.weights);
  uint32_t* offsets = at<uint32_t>(ws, L.offsets);
  uint32_t* perm = at<uint32_t>(ws, L.perm);

  auto rec = [&](int i) -> cudaError_t {
    return ev && ev[i] ? cudaEventRecord((cudaEvent_t)ev[i], s) : cudaSuccess;
  };
  MOE_TRY_CUDA(rec(0), "cudaEventRecord");
  MOE_TRY_CUDA(route(idx, w, s), "routing kernel launch");
  MOE_TRY_CUDA(rec(1), "cudaEventRecord");
  // the gather walks tokens (each row read once, written to its top_k rows)
  // where rows are whole 16-byte vectors, else dispatched rows in order
  uint32_t* slot_row = at<uint32_t>(ws, L.slot_row);
  const bool by_token = (x->H * (int64_t)dtype_size(x->dt)) % 16 == 0;
  MOE_TRY_CUDA(moe::launch_dispatch(idx, T, E, k, offsets, nullptr, perm, at<void>(ws, L.scratch),
                                    status, s, by_token ? slot_row : nullptr),
               "dispatch kernel launch");
  if (by_token)
    MOE_TRY_CUDA(moe::launch_gather_tokens(xin, x->dt, x->H, k, slot_row, T, at<void>(ws, L.x_disp), s),
                 "gather kernel launch");
  else
    MOE_TRY_CUDA(moe::launch_gather(xin, x->dt, x->H, k, perm, offsets, E, N, at<void>(ws, L.x_disp), s),
                 "gather kernel launch");
  MOE_TRY_CUDA(rec(2), "cudaEventRecord");
  st = run_experts(x, at<void>(ws, L.x_disp), N, offsets, at<void>(ws, L.h), at<void>(ws, L.slots),
                   moe::kDownWeighted, perm, w, ldt, status, s, ev ? ev[3] : nullptr);
  if (st != MOE_OK) return st;
  MOE_TRY_CUDA(rec(4), "cudaEventRecord");
  MOE_TRY_CUDA(moe::launch_slot_sum(at<void>(ws, L.slots), x->dt, T, k, x->H, y, s),
               "combine kernel launch");
  MOE_TRY_CUDA(rec(5), "cudaEventRecord");
  return ok();
}

}  // namespace

extern "C" {

const char* moe_last_error(void) { return g_error.c_str(); }

const char* moe_status_string(moe_status st) {
  switch (st) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_SHAPE: return "MOE_ERR_SHAPE";
    case MOE_ERR_DTYPE: return "MOE_ERR_DTYPE";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_INVALID_INDEX: return "MOE_ERR_INVALID_INDEX";
    case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT";
  }
  return "unknown moe_status";
}

// ---- routing -------------------------------------------------------------
moe_status moe_route(const void* logits, moe_dtype ldt, int64_t T, int64_t E, int32_t top_k,
                     int renormalize, uint32_t* idx, void* weights, float* weights_f32,
                     cudaStream_t stream) {
  if (!valid_dtype(ldt)) return fail(MOE_ERR_DTYPE, "logits dtype %d is not F32/F16/BF16", (int)ldt);
  moe_status st = check_tek(T, E, top_k);
  if (st != MOE_OK) return st;
  if (T == 0) return ok();
  if (!logits || !idx || !weights) return fail(MOE_ERR_INVALID_ARG, "logits, idx and weights must be non-NULL");
  MOE_TRY_CUDA(moe::launch_route(logits, ldt, T, (int)E, top_k, renormalize, idx, weights,
                                 weights_f32, nullptr, stream),
               "routing kernel launch");
  return ok();
}

// ---- sigmoid group-limited routing ---------------------------------------
moe_status moe_route_sigmoid_grouped(const void* logits, moe_dtype ldt, int64_t T, int64_t E,
                                     const float* bias, const moe_group_routing_options* opt,
                                     uint32_t* idx, void* weights, float* weights_f32,
                                     cudaStream_t stream) {
  if (!valid_dtype(ldt)) return fail(MOE_ERR_DTYPE, "logits dtype %d is not F32/F16/BF16", (int)ldt);
  moe_status st = check_group_options(T, E, opt);
  if (st != MOE_OK) return st;
  if (T == 0) return ok();
  if (!logits || !idx || !weights) return fail(MOE_ERR_INVALID_ARG, "logits, idx and weights must be non-NULL");
  MOE_TRY_CUDA(moe::launch_route_sigmoid_grouped(logits, ldt, T, (int)E, bias, opt->top_k, opt->groups,
                                                 opt->selected_groups, opt->group_top_two,
                                                 opt->renormalize, opt->scale, idx, weights,
                                                 weights_f32, stream),
               "sigmoid routing kernel launch");
  return ok();
}

// ---- dispatch ------------------------------------------------------------
size_t moe_dispatch_workspace_size(int64_t T, int64_t E, int32_t top_k) {
  (void)top_k;
  if (T < 0 || E < 1 || E > kMaxE) return 0;
  return kWsHeader + align_up(moe::dispatch_scratch_bytes(T, (int)E), 1024);
}

moe_status moe_dispatch(const uint32_t* idx, int64_t T, int64_t E, int32_t top_k, const void* x,
                        moe_dtype x_dtype, int64_t H, uint32_t* offsets, uint32_t* row_experts,
                        uint32_t* perm, void* x_disp, void* ws, size_t ws_bytes, cudaStream_t stream) {
  moe_status st = check_tek(T, E, top_k);
  if (st != MOE_OK) return st;
  if ((x == nullptr) != (x_disp == nullptr))
    return fail(MOE_ERR_INVALID_ARG, "x and x_disp must both be given or both be NULL");
  if (x) {
    if (!valid_dtype(x_dtype)) return fail(MOE_ERR_DTYPE, "x dtype %d is not F32/F16/BF16", (int)x_dtype);
    if ((st = check_dim(H, "H")) != MOE_OK) return st;
  }
  if (!offsets) return fail(MOE_ERR_INVALID_ARG, "offsets must be non-NULL");
  if (T == 0) {
    // no rows: offsets are all zero, nothing else is written
    MOE_TRY_CUDA(cudaMemsetAsync(offsets, 0, (size_t)(E + 1) * 4, stream), "cudaMemsetAsync");
    return ok();
  }
  if (!idx || !perm) return fail(MOE_ERR_INVALID_ARG, "idx and perm must be non-NULL");
  if ((st = check_ws(ws, ws_bytes, moe_dispatch_workspace_size(T, E, top_k))) != MOE_OK) return st;
  MOE_TRY_CUDA(moe::launch_dispatch(idx, T, (int)E, top_k, offsets, row_experts, perm,
                                    static_cast<char*>(ws) + kWsHeader, status_word(ws), stream),
               "dispatch kernel launch");
  if (x)
    MOE_TRY_CUDA(moe::launch_gather(x, x_dtype, H, top_k, perm, offsets, (int)E, T * top_k, x_disp,
                                    stream),
                 "gather kernel launch");
  return ok();
}

moe_status moe_dispatch_noalloc(const uint32_t* idx, int64_t T, int64_t E, int32_t top_k,
                                const void* x, moe_dtype x_dtype, int64_t H, uint32_t* offsets,
                                uint32_t* row_experts, uint32_t* perm, void* x_disp,
                                cudaStream_t stream) {
  moe_status st = check_tek(T, E, top_k);
  if (st != MOE_OK) return st;
  if ((x == nullptr) != (x_disp == nullptr))
    return fail(MOE_ERR_INVALID_ARG, "x and x_disp must both be given or both be NULL");
  if (x) {
    if (!valid_dtype(x_dtype)) return fail(MOE_ERR_DTYPE, "x dtype %d is not F32/F16/BF16", (int)x_dtype);
    if ((st = check_dim(H, "H")) != MOE_OK) return st;
  }
  if (!offsets) return fail(MOE_ERR_INVALID_ARG, "offsets must be non-NULL");
  const size_t need = moe::dispatch_scratch_bytes(T, (int)E);
  const size_t limit = moe::dispatch_noalloc_scratch_limit();
  if (need > limit)
    return fail(MOE_ERR_UNSUPPORTED,
                "moe_dispatch_noalloc: T=%lld, E=%lld needs %zu bytes of scratch, above its fixed "
                "%zu bytes; use moe_dispatch with a workspace",
                (long long)T, (long long)E, need, limit);
  if (T == 0) {
    MOE_TRY_CUDA(cudaMemsetAsync(offsets, 0, (size_t)(E + 1) * 4, stream), "cudaMemsetAsync");
    return ok();
  }
  if (!idx || !perm) return fail(MOE_ERR_INVALID_ARG, "idx and perm must be non-NULL");
  void* scratch = nullptr;
  MOE_TRY_CUDA(moe::dispatch_noalloc_scratch(&scratch), "cudaGetSymbolAddress of the dispatch scratch");
  MOE_TRY_CUDA(moe::launch_dispatch(idx, T, (int)E, top_k, offsets, row_experts, perm, scratch,
                                    nullptr, stream),
               "dispatch kernel launch");
  if (x)
    MOE_TRY_CUDA(moe::launch_gather(x, x_dtype, H, top_k, perm, offsets, (int)E, T * top_k, x_disp,
                                    stream),
                 "gather kernel launch");
  return ok();
}

// ---- experts -------------------------------------------------------------
moe_status moe_experts_create(const void* gate, const void* up, const void* down, moe_dtype dt,
                              int64_t E, int64_t I, int64_t H, moe_experts_t* out) {
  if (!out) return fail(MOE_ERR_INVALID_ARG, "out handle pointer is NULL");
  *out = nullptr;
  if (!valid_dtype(dt)) return fail(MOE_ERR_DTYPE, "expert weight dtype %d is not F32/F16/BF16", (int)dt);
  if (E < 1 || I < 1 || H < 1)
    return fail(MOE_ERR_SHAPE, "MoE expert weight dimensions must be non-zero (E=%lld I=%lld H=%lld)",
                (long long)E, (long long)I, (long long)H);
  if (E > kMaxE) return fail(MOE_ERR_UNSUPPORTED, "E=%lld exceeds the supported 1024", (long long)E);
  moe_status st;
  if ((st = check_dim(I, "I")) != MOE_OK || (st = check_dim(H, "H")) != MOE_OK) return st;
  if ((unsigned __int128)E * I * H * dtype_size(dt) >= ((unsigned __int128)1 << 62))
    return fail(MOE_ERR_SHAPE, "expert weight element count overflows");
  if (!gate || !up || !down) return fail(MOE_ERR_INVALID_ARG, "gate, up and down must be non-NULL");
  if (!aligned16(gate) || !aligned16(up) || !aligned16(down))
    return fail(MOE_ERR_INVALID_ARG, "expert weights must be 16-byte aligned");
  int dev = -1;
  MOE_TRY_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  const void* ptrs[3] = {gate, up, down};
  for (const void* p : ptrs) {
    cudaPointerAttributes a{};
    MOE_TRY_CUDA(cudaPointerGetAttributes(&a, p), "cudaPointerGetAttributes");
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged)
      return fail(MOE_ERR_INVALID_ARG, "expert weights must be device memory");
    if (a.device != dev)
      return fail(MOE_ERR_INVALID_ARG, "expert weights must live on the current device %d", dev);
  }
  int sms = 0;
  MOE_TRY_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "cudaDeviceGetAttribute");
  moe_experts* x = new moe_experts{gate, up, down, dt, E, I, H, dev, sms, nullptr};
  if (moe::tc_supported(dt, I, H)) {
    const char* err = "";
    x->tc = moe::tc_weights_create(gate, up, down, dt, E, I, H, &err);
    if (!x->tc) {
      delete x;
      return fail(MOE_ERR_CUDA, "%s", err);
    }
  }
  *out = x;
  return ok();
}

void moe_experts_destroy(moe_experts_t x) {
  if (!x) return;
  moe::tc_weights_destroy(x->tc);
  delete x;
}

// the checked copy of a staged call's offsets, at the end of its workspace
static size_t offsets_copy_bytes(const moe_experts* x) { return align_up((size_t)(x->E + 1) * 4, 1024); }

size_t moe_experts_workspace_size(moe_experts_t x, int64_t N) {
  if (!x || N < 0) return 0;
  return kWsHeader + align_up((size_t)N * x->I * dtype_size(x->dt), 1024) + offsets_copy_bytes(x);
}

moe_status moe_experts_forward(moe_experts_t x, const void* x_disp, int64_t N, const uint32_t* offsets,
                               void* expert_out, void* ws, size_t ws_bytes, cudaStream_t stream) {
  moe_status st = check_handle(x);
  if (st != MOE_OK) return st;
  if (N < 0 || N > kMaxRows) return fail(MOE_ERR_SHAPE, "N=%lld out of range", (long long)N);
  if (N == 0) return ok();
  if (!x_disp || !offsets || !expert_out)
    return fail(MOE_ERR_INVALID_ARG, "x_disp, offsets and expert_out must be non-NULL");
  if (!aligned16(x_disp) || !aligned16(expert_out))
    return fail(MOE_ERR_INVALID_ARG, "x_disp and expert_out must be 16-byte aligned");
  if ((st = check_ws(ws, ws_bytes, moe_experts_workspace_size(x, N))) != MOE_OK) return st;
  MOE_TRY_CUDA(cudaMemsetAsync(ws, 0, 4, stream), "cudaMemsetAsync");
  uint32_t* off_ok = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + kWsHeader +
                                                 align_up((size_t)N * x->I * dtype_size(x->dt), 1024));
  MOE_TRY_CUDA(moe::launch_sanitize_offsets(offsets, (int)x->E, N, off_ok, status_word(ws), stream),
               "offsets check launch");
  st = run_experts(x, x_disp, N, off_ok, static_cast<char*>(ws) + kWsHeader, expert_out,
                   moe::kDownPlain, nullptr, nullptr, MOE_F32, status_word(ws), stream, nullptr);
  return st == MOE_OK ? ok() : st;
}

// ---- combine -------------------------------------------------------------
size_t moe_combine_workspace_size(int64_t T, int32_t top_k) {
  if (T < 0 || top_k < 1) return 0;
  return kWsHeader + align_up((size_t)T * top_k * 4, 1024);
}

moe_status moe_combine(const void* expert_out, moe_dtype dt, const uint32_t* perm, const void* weights,
                       moe_dtype wdt, int64_t T, int32_t top_k, int64_t H, void* y, void* ws,
                       size_t ws_bytes, cudaStream_t stream) {
  if (!valid_dtype(dt) || !valid_dtype(wdt)) return fail(MOE_ERR_DTYPE, "dtype is not F32/F16/BF16");
  if (T < 0) return fail(MOE_ERR_SHAPE, "T must be >= 0");
  if (top_k < 1) return fail(MOE_ERR_INVALID_ARG, "top_k must be >= 1");
  if (top_k > kMaxK) return fail(MOE_ERR_UNSUPPORTED, "top_k=%d exceeds the supported 64", top_k);
  if (T > kMaxRows / top_k) return fail(MOE_ERR_UNSUPPORTED, "T*top_k exceeds 2^31-1");
  moe_status st = check_dim(H, "H");
  if (st != MOE_OK) return st;
  if (T == 0) return ok();
  if (!expert_out || !perm || !weights || !y)
    return fail(MOE_ERR_INVALID_ARG, "expert_out, perm, weights and y must be non-NULL");
  if (!aligned16(expert_out) || !aligned16(y))
    return fail(MOE_ERR_INVALID_ARG, "expert_out and y must be 16-byte aligned");
  if ((st = check_ws(ws, ws_bytes, moe_combine_workspace_size(T, top_k))) != MOE_OK) return st;
  uint32_t* slot_row = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + kWsHeader);
  MOE_TRY_CUDA(moe::launch_invert_perm(perm, T * top_k, slot_row, stream), "perm inversion launch");
  MOE_TRY_CUDA(moe::launch_combine(expert_out, dt, slot_row, weights, wdt, T, top_k, H, y, stream),
               "combine kernel launch");
  return ok();
}

// ---- fused forward -------------------------------------------------------
size_t moe_forward_workspace_size(moe_experts_t x, int64_t T, int32_t top_k, moe_dtype ldt) {
  if (!x || T < 0 || top_k < 1 || !valid_dtype(ldt)) return 0;
  return forward_layout(x, T, top_k, ldt).total;
}

moe_status moe_forward_layout(moe_experts_t x, int64_t T, int32_t top_k, moe_dtype ldt,
                              moe_forward_layout_t* out) {
  if (!x || !out) return fail(MOE_ERR_INVALID_ARG, "NULL handle or output");
  if (T < 0 || top_k < 1 || !valid_dtype(ldt)) return fail(MOE_ERR_INVALID_ARG, "bad T, top_k or dtype");
  const ForwardLayout L = forward_layout(x, T, top_k, ldt);
  out->idx = L.idx;
  out->weights = L.weights;
  out->offsets = L.offsets;
  out->perm = L.perm;
  out->x_disp = L.x_disp;
  out->h = L.h;
  out->slots = L.slots;
  out->slot_row = L.slot_row;
  out->total = L.total;
  return ok();
}

moe_status moe_forward(moe_experts_t x, const void* xin, const void* logits, moe_dtype ldt, int64_t T,
                       int32_t top_k, int renormalize, void* y, void* ws, size_t ws_bytes,
                       cudaStream_t stream) {
  return forward_impl(x, xin, logits, ldt, T, top_k, renormalize, y, ws, ws_bytes, stream, nullptr);
}

moe_status moe_forward_sigmoid_grouped(moe_experts_t x, const void* xin, const void* logits,
                                       moe_dtype ldt, int64_t T, const float* bias,
                                       const moe_group_routing_options* opt, void* y, void* ws,
                                       size_t ws_bytes, cudaStream_t stream) {
  moe_status st = check_handle(x);
  if (st != MOE_OK) return st;
  if (!valid_dtype(ldt)) return fail(MOE_ERR_DTYPE, "logits dtype %d is not F32/F16/BF16", (int)ldt);
  if ((st = check_group_options(T, x->E, opt)) != MOE_OK) return st;
  const int E = (int)x->E;
  const moe_group_routing_options o = *opt;
  RouteFn route = [=](uint32_t* idx, void* w, cudaStream_t st_) {
    return moe::launch_route_sigmoid_grouped(logits, ldt, T, E, bias, o.top_k, o.groups,
                                             o.selected_groups, o.group_top_two, o.renormalize,
                                             o.scale, idx, w, nullptr, st_);
  };
  return forward_core(x, xin, logits, ldt, T, o.top_k, route, y, ws, ws_bytes, stream, nullptr);
}

moe_status moe_forward_timed(moe_experts_t x, const void* xin, const void* logits, moe_dtype ldt,
                             int64_t T, int32_t top_k, int renormalize, void* y, void* ws,
                             size_t ws_bytes, cudaStream_t stream, void* const* events, int n_events) {
  if (!events || n_events < 6) return fail(MOE_ERR_INVALID_ARG, "moe_forward_timed needs 6 events");
  return forward_impl(x, xin, logits, ldt, T, top_k, renormalize, y, ws, ws_bytes, stream, events);
}

size_t moe_forward_host_workspace_size(moe_experts_t x, int64_t T, int32_t top_k, moe_dtype ldt) {
  if (!x || T < 0 || top_k < 1 || !valid_dtype(ldt)) return 0;
  size_t total = forward_layout(x, T, top_k, ldt).total;
  total += align_up((size_t)T * x->H * dtype_size(x->dt), 1024) * 2;
  total += align_up((size_t)T * x->E * dtype_size(ldt), 1024);
  return total;
}

moe_status moe_forward_host(moe_experts_t x, const void* x_host, const void* logits_host, moe_dtype ldt,
                            int64_t T, int32_t top_k, int renormalize, void* y_host, void* ws,
                            size_t ws_bytes, cudaStream_t stream) {
  moe_status st = check_handle(x);
  if (st != MOE_OK) return st;
  if (!valid_dtype(ldt)) return fail(MOE_ERR_DTYPE, "logits dtype %d is not F32/F16/BF16", (int)ldt);
  if ((st = check_tek(T, x->E, top_k)) != MOE_OK) return st;
  if (T == 0) return ok();
  if (!x_host || !logits_host || !y_host)
    return fail(MOE_ERR_INVALID_ARG, "x_host, logits_host and y_host must be non-NULL");
  if ((st = check_ws(ws, ws_bytes, moe_forward_host_workspace_size(x, T, top_k, ldt))) != MOE_OK)
    return st;
  const size_t base = forward_layout(x, T, top_k, ldt).total;
  const size_t xb = (size_t)T * x->H * dtype_size(x->dt), lb = (size_t)T * x->E * dtype_size(ldt);
  char* xs = static_cast<char*>(ws) + base;
  char* ys = xs + align_up(xb, 1024);
  char* ls = ys + align_up(xb, 1024);
  MOE_TRY_CUDA(cudaMemcpyAsync(xs, x_host, xb, cudaMemcpyHostToDevice, stream), "cudaMemcpyAsync x");
  MOE_TRY_CUDA(cudaMemcpyAsync(ls, logits_host, lb, cudaMemcpyHostToDevice, stream),
               "cudaMemcpyAsync logits");
  st = forward_impl(x, xs, ls, ldt, T, top_k, renormalize, ys, ws, base, stream, nullptr);
  if (st != MOE_OK) return st;
  MOE_TRY_CUDA(cudaMemcpyAsync(y_host, ys, xb, cudaMemcpyDeviceToHost, stream), "cudaMemcpyAsync y");
  return ok();
}

// ---- pipelined host-buffer forward -----------------------------------------
struct moe_host_pipeline {
  static constexpr int kMaxDepth = 4;
  moe_experts* x;
  int64_t T_max;
  int32_t top_k;
  moe_dtype ldt;
  int renormalize;
  int depth;
  char* ws;
  size_t fwd_bytes;
  cudaStream_t stream, h2d, d2h;
  struct Slot {
    char *xs, *ls, *ys;
    cudaEvent_t loaded, computed, stored;
    bool used;
  } slot[kMaxDepth];
  uint64_t submitted;
};

namespace {
struct PipelineSizes {
  size_t fwd, xb, lb, per_slot;
};
PipelineSizes pipeline_sizes(const moe_experts* x, int64_t T, int32_t k, moe_dtype ldt) {
  PipelineSizes z;
  z.fwd = align_up(forward_layout(x, T, k, ldt).total, 1024);
  z.xb = align_up((size_t)T * x->H * dtype_size(x->dt), 1024);
  z.lb = align_up((size_t)T * x->E * dtype_size(ldt), 1024);
  z.per_slot = 2 * z.xb + z.lb;
  return z;
}
void pipeline_free(moe_host_pipeline* p) {
  for (int i = 0; i < moe_host_pipeline::kMaxDepth; ++i) {
    auto& sl = p->slot[i];
    if (sl.loaded) cudaEventDestroy(sl.loaded);
    if (sl.computed) cudaEventDestroy(sl.computed);
    if (sl.stored) cudaEventDestroy(sl.stored);
  }
  if (p->h2d) cudaStreamDestroy(p->h2d);
  if (p->d2h) cudaStreamDestroy(p->d2h);
  delete p;
}
}  // namespace

size_t moe_host_pipeline_workspace_size(moe_experts_t x, int64_t T_max, int32_t top_k, moe_dtype ldt,
                                        int depth) {
  if (!x || T_max < 1 || top_k < 1 || !valid_dtype(ldt) || depth < 2 ||
      depth > moe_host_pipeline::kMaxDepth)
    return 0;
  const PipelineSizes z = pipeline_sizes(x, T_max, top_k, ldt);
  return z.fwd + (size_t)depth * z.per_slot;
}

moe_status moe_host_pipeline_create(moe_experts_t x, int64_t T_max, int32_t top_k, moe_dtype ldt,
                                    int renormalize, int depth, void* ws, size_t ws_bytes,
                                    cudaStream_t stream, moe_host_pipeline_t* out) {
  moe_status st = check_handle(x);
  if (st != MOE_OK) return st;
  if (!out) return fail(MOE_ERR_INVALID_ARG, "out must be non-NULL");
  *out = nullptr;
  if (!valid_dtype(ldt)) return fail(MOE_ERR_DTYPE, "logits dtype %d is not F32/F16/BF16", (int)ldt);
  if (T_max < 1) return fail(MOE_ERR_SHAPE, "T_max must be >= 1");
  if ((st = check_tek(T_max, x->E, top_k)) != MOE_OK) return st;
  if (depth < 2 || depth > moe_host_pipeline::kMaxDepth)
    return fail(MOE_ERR_INVALID_ARG, "depth must be in 2..=4");
  if ((st = check_ws(ws, ws_bytes, moe_host_pipeline_workspace_size(x, T_max, top_k, ldt, depth))) != MOE_OK)
    return st;
  moe_host_pipeline* p = new moe_host_pipeline();
  p->x = x;
  p->T_max = T_max;
  p->top_k = top_k;
  p->ldt = ldt;
  p->renormalize = renormalize;
  p->depth = depth;
  p->ws = static_cast<char*>(ws);
  p->stream = stream;
  const PipelineSizes z = pipeline_sizes(x, T_max, top_k, ldt);
  p->fwd_bytes = z.fwd;
  cudaError_t e = cudaStreamCreateWithFlags(&p->h2d, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->d2h, cudaStreamNonBlocking);
  for (int i = 0; i < depth && e == cudaSuccess; ++i) {
    auto& sl = p->slot[i];
    sl.xs = p->ws + z.fwd + (size_t)i * z.per_slot;
    sl.ys = sl.xs + z.xb;
    sl.ls = sl.ys + z.xb;
    e = cudaEventCreateWithFlags(&sl.loaded, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&sl.computed, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&sl.stored, cudaEventDisableTiming);
  }
  if (e != cudaSuccess) {
    pipeline_free(p);
    return cuda_fail(e, "host pipeline streams and events");
  }
  *out = p;
  return ok();
}

moe_status moe_host_pipeline_submit(moe_host_pipeline_t p, const void* x_host, const void* logits_host,
                                    void* y_host, int64_t T) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "pipeline is NULL");
  if (T < 0 || T > p->T_max) return fail(MOE_ERR_SHAPE, "T=%lld outside 0..=T_max", (long long)T);
  if (T == 0) return ok();
  if (!x_host || !logits_host || !y_host)
    return fail(MOE_ERR_INVALID_ARG, "x_host, logits_host and y_host must be non-NULL");
  moe_experts* x = p->x;
  auto& sl = p->slot[p->submitted % (uint64_t)p->depth];
  const size_t xb = (size_t)T * x->H * dtype_size(x->dt), lb = (size_t)T * x->E * dtype_size(p->ldt);
  // inputs: into this slot once its previous forward has read it
  if (sl.used) MOE_TRY_CUDA(cudaStreamWaitEvent(p->h2d, sl.computed, 0), "cudaStreamWaitEvent");
  MOE_TRY_CUDA(cudaMemcpyAsync(sl.xs, x_host, xb, cudaMemcpyHostToDevice, p->h2d), "cudaMemcpyAsync x");
  MOE_TRY_CUDA(cudaMemcpyAsync(sl.ls, logits_host, lb, cudaMemcpyHostToDevice, p->h2d),
               "cudaMemcpyAsync logits");
  MOE_TRY_CUDA(cudaEventRecord(sl.loaded, p->h2d), "cudaEventRecord");
  // forward: after the inputs landed and the slot's previous y was copied out
  MOE_TRY_CUDA(cudaStreamWaitEvent(p->stream, sl.loaded, 0), "cudaStreamWaitEvent");
  if (sl.used) MOE_TRY_CUDA(cudaStreamWaitEvent(p->stream, sl.stored, 0), "cudaStreamWaitEvent");
  moe_status st = forward_impl(x, sl.xs, sl.ls, p->ldt, T, p->top_k, p->renormalize, sl.ys, p->ws,
                               p->fwd_bytes, p->stream, nullptr);
  if (st != MOE_OK) return st;
  MOE_TRY_CUDA(cudaEventRecord(sl.computed, p->stream), "cudaEventRecord");
  // output
  MOE_TRY_CUDA(cudaStreamWaitEvent(p->d2h, sl.computed, 0), "cudaStreamWaitEvent");
  MOE_TRY_CUDA(cudaMemcpyAsync(y_host, sl.ys, xb, cudaMemcpyDeviceToHost, p->d2h), "cudaMemcpyAsync y");
  MOE_TRY_CUDA(cudaEventRecord(sl.stored, p->d2h), "cudaEventRecord");
  sl.used = true;
  ++p->submitted;
  return ok();
}

moe_status moe_host_pipeline_sync(moe_host_pipeline_t p) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "pipeline is NULL");
  MOE_TRY_CUDA(cudaStreamSynchronize(p->h2d), "cudaStreamSynchronize");
  MOE_TRY_CUDA(cudaStreamSynchronize(p->stream), "cudaStreamSynchronize");
  MOE_TRY_CUDA(cudaStreamSynchronize(p->d2h), "cudaStreamSynchronize");
  return ok();
}

moe_status moe_host_pipeline_destroy(moe_host_pipeline_t p) {
  if (!p) return ok();
  const cudaError_t e1 = cudaStreamSynchronize(p->h2d);
  const cudaError_t e2 = cudaStreamSynchronize(p->d2h);
  pipeline_free(p);
  if (e1 != cudaSuccess) return cuda_fail(e1, "cudaStreamSynchronize");
  if (e2 != cudaSuccess) return cuda_fail(e2, "cudaStreamSynchronize");
  return ok();
}

// ---- first-order training backward (user guide, section 12) -------------
moe_status moe_combine_backward(const void* expert_out, moe_dtype dt, const uint32_t* perm,
                                const void* weights, moe_dtype wdt, const void* dy, int64_t T,
                                int32_t top_k, int64_t H, void* dexpert, float* dweights,
                                cudaStream_t stream) {
  if (!valid_dtype(dt) || !valid_dtype(wdt)) return fail(MOE_ERR_DTYPE, "dtype is not F32/F16/BF16");
  if (T < 0) return fail(MOE_ERR_SHAPE, "T must be >= 0");
  if (top_k < 1 || top_k > kMaxK) return fail(MOE_ERR_INVALID_ARG, "top_k must be in 1..=64");
  if (T > kMaxRows / top_k) return fail(MOE_ERR_UNSUPPORTED, "T*top_k exceeds 2^31-1");
  moe_status st = check_dim(H, "H");
  if (st != MOE_OK) return st;
  if (T == 0) return ok();
  if (!expert_out || !perm || !weights || !dy || !dexpert || !dweights)
    return fail(MOE_ERR_INVALID_ARG, "expert_out, perm, weights, dy, dexpert and dweights must be non-NULL");
  MOE_TRY_CUDA(moe::launch_combine_backward(expert_out, dt, perm, weights, wdt, dy, T, top_k, H, dexpert,
                                            dweights, stream),
               "combine backward launch");
  return ok();
}

moe_status moe_dispatch_backward(const void* dinput, moe_dtype dt, const uint32_t* perm, int64_t T,
                                 int32_t top_k, int64_t H, void* dx, void* ws, size_t ws_bytes,
                                 cudaStream_t stream) {
  if (!valid_dtype(dt)) return fail(MOE_ERR_DTYPE, "dtype is not F32/F16/BF16");
  if (T < 0) return fail(MOE_ERR_SHAPE, "T must be >= 0");
  if (top_k < 1 || top_k > kMaxK) return fail(MOE_ERR_INVALID_ARG, "top_k must be in 1..=64");
  if (T > kMaxRows / top_k) return fail(MOE_ERR_UNSUPPORTED, "T*top_k exceeds 2^31-1");
  moe_status st = check_dim(H, "H");
  if (st != MOE_OK) return st;
  if (T == 0) return ok();
  if (!dinput || !perm || !dx) return fail(MOE_ERR_INVALID_ARG, "dinput, perm and dx must be non-NULL");
  if (!aligned16(dinput) || !aligned16(dx))
    return fail(MOE_ERR_INVALID_ARG, "dinput and dx must be 16-byte aligned");
  if ((st = check_ws(ws, ws_bytes, moe_combine_workspace_size(T, top_k))) != MOE_OK) return st;
  uint32_t* slot_row = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + kWsHeader);
  MOE_TRY_CUDA(moe::launch_invert_perm(perm, T * top_k, slot_row, stream), "perm inversion launch");
  MOE_TRY_CUDA(moe::launch_combine(dinput, dt, slot_row, nullptr, MOE_F32, T, top_k, H, dx, stream),
               "dispatch backward launch");
  return ok();
}

// The tensor-core backward applies when the experts are F16/BF16 with the
// tcgen05 tensor maps and the 64-padded row space stays within the TMA
// coordinate range.
static bool bwd_tc_ok(const moe_experts* x, int64_t N) {
  return x->tc && N + 63 * x->E < (int64_t)INT32_MAX;
}

// scratch of either strategy: five FP32 [N, I] buffers, or the tensor-core layout
static size_t bwd_scratch_bytes(const moe_experts* x, int64_t N) {
  size_t need = 5 * align_up((size_t)N * x->I * 4, 1024);
  if (bwd_tc_ok(x, N))
    need = std::max(need, moe::experts_backward_tc_workspace(N, (int)x->E, x->H, x->I));
  return need;
}

size_t moe_experts_backward_workspace_size(moe_experts_t x, int64_t N) {
  if (!x || N < 0) return 0;
  return kWsHeader + bwd_scratch_bytes(x, N) + offsets_copy_bytes(x);
}

moe_status moe_experts_backward_with_strategy(moe_experts_t x, const void* x_disp, int64_t N,
                                              const uint32_t* offsets, const void* dout,
                                              void* dinput, float* dgate, float* dup, float* ddown,
                                              int strategy, void* ws, size_t ws_bytes,
                                              cudaStream_t stream) {
  moe_status st = check_handle(x);
  if (st != MOE_OK) return st;
  if (strategy != MOE_BWD_SCALAR && strategy != MOE_BWD_AUTO && strategy != MOE_BWD_TENSOR_CORE)
    return fail(MOE_ERR_INVALID_ARG, "strategy must be MOE_BWD_SCALAR, MOE_BWD_AUTO or MOE_BWD_TENSOR_CORE");
  if (N < 0 || N > kMaxRows) return fail(MOE_ERR_SHAPE, "N=%lld out of range", (long long)N);
  if (strategy == MOE_BWD_TENSOR_CORE && !bwd_tc_ok(x, N))
    return fail(MOE_ERR_UNSUPPORTED,
                "tensor-core backward needs F16/BF16 experts with H, I multiples of 8");
  if (!offsets || !dgate || !dup || !ddown)
    return fail(MOE_ERR_INVALID_ARG, "offsets, dgate, dup and ddown must be non-NULL");
  if (N > 0 && (!x_disp || !dout || !dinput))
    return fail(MOE_ERR_INVALID_ARG, "x_disp, dout and dinput must be non-NULL");
  const bool tc = strategy != MOE_BWD_SCALAR && bwd_tc_ok(x, N);
  if (tc && N > 0 && (!aligned16(x_disp) || !aligned16(dout) || !aligned16(dinput)))
    return fail(MOE_ERR_INVALID_ARG, "x_disp, dout and dinput must be 16-byte aligned");
  if ((st = check_ws(ws, ws_bytes, moe_experts_backward_workspace_size(x, N))) != MOE_OK) return st;
  const size_t part = align_up((size_t)N * x->I * 4, 1024);
  char* base = static_cast<char*>(ws) + kWsHeader;
  moe::ExpertsBwdArgs a{};
  a.dt = x->dt;
  a.E = (int)x->E;
  a.N = N;
  a.H = x->H;
  a.I = x->I;
  a.x_disp = x_disp;
  a.dout = dout;
  a.gate = x->gate;
  a.up = x->up;
  a.down = x->down;
  uint32_t* off_ok = reinterpret_cast<uint32_t*>(base + bwd_scratch_bytes(x, N));
  a.offsets = off_ok;
  a.g = reinterpret_cast<float*>(base);
  a.u = reinterpret_cast<float*>(base + part);
  a.act = reinterpret_cast<float*>(base + 2 * part);
  a.dg = reinterpret_cast<float*>(base + 3 * part);
  a.du = reinterpret_cast<float*>(base + 4 * part);
  a.dinput = dinput;
  a.dgate = dgate;
  a.dup = dup;
  a.ddown = ddown;
  a.status = status_word(ws);
  if (N == 0) {  // no rows: every weight gradient is zero
    const size_t wb = (size_t)x->E * x->I * x->H * 4;
    MOE_TRY_CUDA(cudaMemsetAsync(dgate, 0, wb, stream), "cudaMemsetAsync");
    MOE_TRY_CUDA(cudaMemsetAsync(dup, 0, wb, stream), "cudaMemsetAsync");
    MOE_TRY_CUDA(cudaMemsetAsync(ddown, 0, wb, stream), "cudaMemsetAsync");
    return ok();
  }
  MOE_TRY_CUDA(cudaMemsetAsync(ws, 0, 4, stream), "cudaMemsetAsync");
  MOE_TRY_CUDA(moe::launch_sanitize_offsets(offsets, (int)x->E, N, off_ok, a.status, stream),
               "offsets check launch");
  if (tc) {
    MOE_TRY_CUDA(moe::launch_experts_backward_tc(a, x->tc, base, x->num_sms, stream),
                 "tensor-core expert backward launch");
  } else {
    MOE_TRY_CUDA(moe::launch_experts_backward(a, stream), "expert backward launch");
  }
  return ok();
}

moe_status moe_experts_backward(moe_experts_t x, const void* x_disp, int64_t N, const uint32_t* offsets,
                                const void* dout, void* dinput, float* dgate, float* dup, float* ddown,
                                void* ws, size_t ws_bytes, cudaStream_t stream) {
  return moe_experts_backward_with_strategy(x, x_disp, N, offsets, dout, dinput, dgate, dup, ddown,
                                            MOE_BWD_SCALAR, ws, ws_bytes, stream);
}

static moe_status check_router_args(int64_t T, int64_t E, int32_t k, int scoring, float scale) {
  if (T < 0) return fail(MOE_ERR_SHAPE, "T must be >= 0");
  if (E < 1 || E > kMaxE) return fail(E < 1 ? MOE_ERR_SHAPE : MOE_ERR_UNSUPPORTED, "E must be in 1..=1024");
  if (k < 1 || k > kMaxK || k > E) return fail(MOE_ERR_INVALID_ARG, "top_k must satisfy 1 <= top_k <= min(E, 64)");
  if (scoring != 0 && scoring != 1) return fail(MOE_ERR_INVALID_ARG, "scoring must be 0 (softmax) or 1 (sigmoid)");
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(MOE_ERR_INVALID_ARG, "scale must be finite and positive");
  if (T > kMaxRows / k) return fail(MOE_ERR_UNSUPPORTED, "T*top_k exceeds 2^31-1");
  return MOE_OK;
}

moe_status moe_router_weights(const void* logits, moe_dtype ldt, const uint32_t* idx, int64_t T,
                              int64_t E, int32_t top_k, int scoring, int renormalize, float scale,
                              float* weights, cudaStream_t stream) {
  if (!valid_dtype(ldt)) return fail(MOE_ERR_DTYPE, "logits dtype is not F32/F16/BF16");
  moe_status st = check_router_args(T, E, top_k, scoring, scale);
  if (st != MOE_OK) return st;
  if (T == 0) return ok();
  if (!logits || !idx || !weights) return fail(MOE_ERR_INVALID_ARG, "logits, idx and weights must be non-NULL");
  MOE_TRY_CUDA(moe::launch_router_backward(logits, ldt, T, (int)E, idx, top_k, nullptr, scoring, renormalize,
                                           scale, nullptr, weights, stream),
               "router weights launch");
  return ok();
}

moe_status moe_router_backward(const void* logits, moe_dtype ldt, const uint32_t* idx,
                               const float* dweights, int64_t T, int64_t E, int32_t top_k, int scoring,
                               int renormalize, float scale, void* dlogits, cudaStream_t stream) {
  if (!valid_dtype(ldt)) return fail(MOE_ERR_DTYPE, "logits dtype is not F32/F16/BF16");
  moe_status st = check_router_args(T, E, top_k, scoring, scale);
  if (st != MOE_OK) return st;
  if (T == 0) return ok();
  if (!logits || !idx || !dweights || !dlogits)
    return fail(MOE_ERR_INVALID_ARG, "logits, idx, dweights and dlogits must be non-NULL");
  MOE_TRY_CUDA(moe::launch_router_backward(logits, ldt, T, (int)E, idx, top_k, dweights, scoring,
                                           renormalize, scale, dlogits, nullptr, stream),
               "router backward launch");
  return ok();
}

moe_status moe_selftest_bounded_wait(void* ws, uint32_t limit_ms, cudaStream_t stream) {
  if ((ws == nullptr) || !aligned256(ws))
    return fail(MOE_ERR_INVALID_ARG, "workspace must be non-NULL and 256-byte aligned");
  if (limit_ms < 1 || limit_ms > 2000) return fail(MOE_ERR_INVALID_ARG, "limit_ms must be in [1, 2000]");
  MOE_TRY_CUDA(cudaMemsetAsync(ws, 0, 4, stream), "cudaMemsetAsync");
  MOE_TRY_CUDA(moe::launch_bounded_wait_selftest(status_word(ws), (uint64_t)limit_ms * 1000000ull, stream),
               "self-test kernel launch");
  return ok();
}

moe_status moe_get_device_status(const void* ws, cudaStream_t stream) {
  if (!ws) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
  uint32_t v = 0;
  MOE_TRY_CUDA(cudaMemcpyAsync(&v, ws, 4, cudaMemcpyDeviceToHost, stream), "cudaMemcpyAsync status");
  MOE_TRY_CUDA(cudaStreamSynchronize(stream), "cudaStreamSynchronize");
  if (v == MOE_OK) return ok();
  if (v == MOE_ERR_INVALID_INDEX) return fail(MOE_ERR_INVALID_INDEX, "an expert index >= E reached dispatch");
  if (v == MOE_ERR_DEVICE_TIMEOUT)
    return fail(MOE_ERR_DEVICE_TIMEOUT, "a bounded wait inside a kernel expired");
  return fail(MOE_ERR_CUDA, "unknown device status %u", v);
}

}  // extern "C"
