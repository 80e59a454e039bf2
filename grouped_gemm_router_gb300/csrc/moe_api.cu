// C ABI of the MoE SwiGLU FFN forward pass: argument validation, workspace
// layout and the launch sequence.  All arithmetic runs in the kernels of
// route_permute.cu, grouped_gemm.cu and combine.cu.
#include <atomic>

#include "moe_kernels.cuh"

namespace moe {

static std::atomic<uint64_t> g_launches{0};
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

moe_status check_dims(const moe_dims& d) {
  if (d.T < 0 || d.D <= 0 || d.F <= 0 || d.E <= 0 || d.k <= 0) return MOE_ERR_INVALID_ARG;
  if (d.k > d.E) return MOE_ERR_INVALID_ARG;
  if (d.T > (1 << 24)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (d.D % 64 || d.F % 64 || d.D > MOE_MAX_DIM || d.F > MOE_MAX_DIM) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (d.E > MOE_MAX_EXPERTS || d.k > MOE_MAX_TOPK) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

struct Workspace {
  void* wpack;
  int32_t* ids;
  float* w;
  int32_t* hist;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv;
  uint16_t* x_sorted;
  uint16_t* h;
  uint16_t* y;
  float* ys;
  uint16_t* x_stage;
  uint16_t* out_stage;
  size_t bytes;
};

// Carves the workspace; with base == nullptr only computes the size.
Workspace carve(void* base, const moe_dims& d, bool shared, bool host_io) {
  Workspace w{};
  const size_t T = static_cast<size_t>(d.T), S = T * d.k;
  const size_t rows = S + (shared ? T : 0);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align_up(bytes);
    return base ? static_cast<char*>(base) + o : nullptr;
  };
  w.wpack = take(route_packed_bytes(d.D, d.E));
  w.ids = reinterpret_cast<int32_t*>(take(S * 4));
  w.w = reinterpret_cast<float*>(take(S * 4));
  w.hist = reinterpret_cast<int32_t*>(take(static_cast<size_t>(route_blocks_max(d.T)) * d.E * 4));
  w.counts = reinterpret_cast<int32_t*>(take(static_cast<size_t>(d.E) * 4));
  w.offsets = reinterpret_cast<int32_t*>(take(static_cast<size_t>(d.E + 1) * 4));
  w.perm = reinterpret_cast<int32_t*>(take(S * 4));
  w.inv = reinterpret_cast<int32_t*>(take(S * 4));
  w.x_sorted = reinterpret_cast<uint16_t*>(take(S * d.D * 2));
  w.h = reinterpret_cast<uint16_t*>(take(rows * d.F * 2));
  w.y = reinterpret_cast<uint16_t*>(take(S * d.D * 2));
  w.ys = shared ? reinterpret_cast<float*>(take(T * d.D * 4)) : nullptr;
  if (host_io) {
    w.x_stage = reinterpret_cast<uint16_t*>(take(T * d.D * 2));
    w.out_stage = reinterpret_cast<uint16_t*>(take(T * d.D * 2));
  }
  w.bytes = off;
  return w;
}

// Backward workspace: gradient buffers in the padded sorted layout.
struct BwdWorkspace {
  uint16_t* ybar;  // [S_pad, D]
  uint16_t* hbar;  // [S_pad + Tsh, F]
  uint16_t* gu;    // [S_pad + Tsh, 2F]
  uint16_t* h;     // [S_pad + Tsh, F]
  uint16_t* xbar;  // [S_pad + Tsh, D]
  float* wbar;     // [T, k]
  float* lbar;     // [T, k]
  float* rpart;    // router-gradient partials
  uint16_t* wgt;   // Wg^T [E, D]
  float* wpart;    // weight-gradient partial sums of split groups
  size_t bytes;
};

BwdWorkspace carve_bwd(void* base, const moe_dims& d, bool shared) {
  BwdWorkspace w{};
  const size_t T = static_cast<size_t>(d.T), S = T * d.k;
  const size_t Sp = static_cast<size_t>(bwd_padded_rows(d));
  const size_t rows = Sp + (shared ? T : 0);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align_up(bytes);
    return base ? static_cast<char*>(base) + o : nullptr;
  };
  w.ybar = reinterpret_cast<uint16_t*>(take(Sp * d.D * 2));
  w.hbar = reinterpret_cast<uint16_t*>(take(rows * d.F * 2));
  w.gu = reinterpret_cast<uint16_t*>(take(rows * d.F * 4));
  w.h = reinterpret_cast<uint16_t*>(take(rows * d.F * 2));
  w.xbar = reinterpret_cast<uint16_t*>(take(rows * d.D * 2));
  w.wbar = reinterpret_cast<float*>(take(S * 4));
  w.lbar = reinterpret_cast<float*>(take(S * 4));
  w.rpart = reinterpret_cast<float*>(take(bwd_router_part_floats(d) * 4));
  w.wgt = reinterpret_cast<uint16_t*>(take(static_cast<size_t>(d.E) * d.D * 2));
  w.wpart = reinterpret_cast<float*>(take(bwd_wgrad_part_floats(d, shared) * 4));
  w.bytes = off;
  return w;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shared-expert pointers: all three set or all three NULL.
int shared_state(const void* a, const void* b, const void* c) {
  const int n = (a != nullptr) + (b != nullptr) + (c != nullptr);
  return n == 0 ? 0 : (n == 3 ? 1 : -1);
}

void record(const moe_ffn_options* o, int i, cudaStream_t s) {
  if (o != nullptr && o->stage_events[i] != nullptr)
    cudaEventRecord(static_cast<cudaEvent_t>(o->stage_events[i]), s);
}

// The launch sequence of the layer on already validated arguments.
moe_status run_layer(const uint16_t* x, const uint16_t* Wg, const float* bias, const uint16_t* W1,
                     const uint16_t* W3, const uint16_t* W2, const uint16_t* Ws1,
                     const uint16_t* Ws3, const uint16_t* Ws2, const moe_dims& d, uint16_t* out,
                     const Workspace& ws, const moe_ffn_options* o, cudaStream_t s) {
  const bool shared = Ws1 != nullptr;
  const bool routed_in = o != nullptr && o->ids_in != nullptr && o->weights_in != nullptr;
  const int32_t* ids = routed_in ? o->ids_in : ws.ids;
  const float* w = routed_in ? o->weights_in : ws.w;
  cudaError_t e;
  // Every kernel after the first may start while its predecessor finishes
  // (programmatic dependent launch): it waits on the device before reading
  // the predecessor's results.  Stage events between kernels, when given,
  // serialise the launches again.
  record(o, 0, s);
  if (routed_in)
    e = launch_hist(ids, d, ws.hist, s, false);
  else
    e = launch_route(x, Wg, bias, d, ws.wpack, ws.ids, ws.w, ws.hist, s, false);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  record(o, 1, s);
  e = launch_scatter(ids, ws.hist, d, ws.counts, ws.offsets, ws.perm, ws.inv, x, ws.x_sorted, s, true);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  record(o, 2, s);
  if (o != nullptr && (o->flags & MOE_FFN_CHAINED)) {
    e = launch_chained_ffn(ws.x_sorted, x, W1, W3, W2, Ws1, Ws3, Ws2, ws.offsets, d, ws.y, ws.ys, s, true);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    record(o, 3, s);
  } else {
    e = launch_grouped_swiglu(ws.x_sorted, x, W1, W3, Ws1, Ws3, ws.offsets, d, ws.h, s, true);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    record(o, 3, s);
    e = launch_grouped_down(ws.h, W2, Ws2, ws.offsets, d, ws.y, ws.ys, s, true);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  record(o, 4, s);
  e = launch_combine(ws.y, shared ? ws.ys : nullptr, w, ws.inv, d, out, s, true);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  record(o, 5, s);
  return MOE_OK;
}

moe_status validate_layer(const void* x, const void* Wg, const float* bias, const void* W1,
                          const void* W3, const void* W2, const void* Ws1, const void* Ws3,
                          const void* Ws2, const moe_dims& d, const void* out, const void* ws,
                          const moe_ffn_options* o, bool x_out_on_host) {
  moe_status st = check_dims(d);
  if (st != MOE_OK) return st;
  if (!x || !Wg || !W1 || !W3 || !W2 || !out || !ws) return MOE_ERR_INVALID_ARG;
  if (shared_state(Ws1, Ws3, Ws2) < 0) return MOE_ERR_INVALID_ARG;
  const void* dev_ptrs[] = {Wg, W1, W3, W2, Ws1, Ws3, Ws2, ws, bias};
  for (const void* p : dev_ptrs)
    if (p != nullptr && !aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (!x_out_on_host && (!aligned16(x) || !aligned16(out))) return MOE_ERR_INVALID_ARG;
  if (o != nullptr && ((o->ids_in == nullptr) != (o->weights_in == nullptr))) return MOE_ERR_INVALID_ARG;
  if (o != nullptr && o->ids_in != nullptr && (!aligned16(o->ids_in) || !aligned16(o->weights_in)))
    return MOE_ERR_INVALID_ARG;
  if (o != nullptr && (o->flags & ~MOE_FFN_CHAINED) != 0) return MOE_ERR_INVALID_ARG;
  if (o != nullptr && (o->flags & MOE_FFN_CHAINED) && d.D > MOE_CHAINED_MAX_D)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

// The backward launch sequence on validated arguments.
moe_status run_backward(const uint16_t* x, const uint16_t* Wg, const uint16_t* W1, const uint16_t* W3,
                        const uint16_t* W2, const uint16_t* Ws1, const uint16_t* Ws3,
                        const uint16_t* Ws2, const uint16_t* d_out, const moe_dims& d,
                        const Workspace& fw, const BwdWorkspace& bw, uint16_t* dx, float* dWg,
                        float* dbias, float* dW1, float* dW3, float* dW2, float* dWs1, float* dWs3,
                        float* dWs2, const moe_ffn_options* o, cudaStream_t s) {
  const bool shared = Ws1 != nullptr;
  const bool routed_in = o != nullptr && o->ids_in != nullptr;
  const int32_t* ids = routed_in ? o->ids_in : fw.ids;
  const float* w = routed_in ? o->weights_in : fw.w;
  const BwdLayout L{d, shared, bwd_padded_rows(d)};
  const size_t Sp = static_cast<size_t>(L.S_pad);
  const size_t S = static_cast<size_t>(d.T) * d.k;
  // The unchained forward left h in its workspace (the recompute gives the
  // same bits); after a chained forward the recompute stores h itself.
  const bool fwd_h = o == nullptr || (o->flags & MOE_FFN_CHAINED) == 0;
  cudaError_t e;
  record(o, 0, s);
  e = launch_combine_bwd(L, d_out, fw.y, w, ids, fw.inv, fw.offsets, routed_in ? 1 : 0, bw.ybar, bw.wbar,
                         bw.lbar, Wg, bw.wgt, s, false);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  record(o, 1, s);
  e = launch_bwd_dgrad_w2(L, fw.offsets, bw.ybar, d_out, W2, Ws2, bw.hbar, s, true);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  record(o, 2, s);
  e = launch_bwd_act(L, fw.offsets, fw.x_sorted, x, W1, W3, Ws1, Ws3, bw.hbar, bw.gu, fwd_h ? nullptr : bw.h,
                     s, true);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  record(o, 3, s);
  e = launch_bwd_dgrad_x(L, fw.offsets, bw.gu, W1, W3, Ws1, Ws3, bw.xbar, s, true);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  record(o, 4, s);
  e = launch_bwd_wgrad(L, fw.offsets, fw.x_sorted, 0, d.D, x, bw.gu, 2 * d.F, bw.gu + Sp * 2 * d.F, d.F,
                       dW1, dW3, dWs1, dWs3, bw.wpart, s, true);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  record(o, 5, s);
  e = launch_bwd_wgrad(L, fw.offsets, fwd_h ? fw.h : bw.h, fwd_h ? 0 : 1, d.F,
                       fwd_h ? fw.h + S * d.F : bw.h + Sp * d.F, bw.ybar, d.D, d_out, d.D, dW2, nullptr, dWs2,
                       nullptr, bw.wpart, s, true);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  record(o, 6, s);
  e = launch_dx_gather(L, bw.xbar, ids, fw.inv, fw.offsets, routed_in ? nullptr : bw.lbar, bw.wgt, dx,
                       s, true);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  record(o, 7, s);
  if (!routed_in && (dWg != nullptr || dbias != nullptr)) {
    e = launch_router_bwd(L, fw.x_sorted, fw.perm, fw.offsets, bw.lbar, bw.rpart, dWg, dbias, s, true);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  record(o, 8, s);
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_ffn_backward_workspace_size(moe_dims d, int has_shared) {
  if (check_dims(d) != MOE_OK) return 0;
  return carve_bwd(nullptr, d, has_shared != 0).bytes;
}

moe_status moe_ffn_backward(const void* x, const void* Wg, const void* W1, const void* W3,
                            const void* W2, const void* Ws1, const void* Ws3, const void* Ws2,
                            const void* d_out, moe_dims d, const void* fwd_workspace,
                            size_t fwd_ws_bytes, void* dx, float* dWg, float* dbias, float* dW1,
                            float* dW3, float* dW2, float* dWs1, float* dWs3, float* dWs2,
                            void* workspace, size_t ws_bytes, const moe_ffn_options* opts,
                            void* stream) {
  moe_status st = check_dims(d);
  if (st != MOE_OK) return st;
  if (d.T == 0) return MOE_OK;  // nothing to differentiate (the gradient tensors are left as given)
  if (!x || !Wg || !W1 || !W3 || !W2 || !d_out || !fwd_workspace || !dx || !dW1 || !dW3 || !dW2 ||
      !workspace)
    return MOE_ERR_INVALID_ARG;
  const int sh = shared_state(Ws1, Ws3, Ws2);
  const int shg = shared_state(dWs1, dWs3, dWs2);
  if (sh < 0 || shg < 0 || sh != shg) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x, Wg, W1, W3, W2, Ws1, Ws3, Ws2, d_out, fwd_workspace, dx, dWg, dbias,
                        dW1, dW3, dW2, dWs1, dWs3, dWs2, workspace};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (opts != nullptr && ((opts->ids_in == nullptr) != (opts->weights_in == nullptr)))
    return MOE_ERR_INVALID_ARG;
  if (opts != nullptr && (opts->flags & ~MOE_FFN_CHAINED) != 0) return MOE_ERR_INVALID_ARG;
  const bool shared = sh == 1;
  const Workspace fw = carve(const_cast<void*>(fwd_workspace), d, shared, false);
  if (fwd_ws_bytes < fw.bytes) return MOE_ERR_WORKSPACE;
  const BwdWorkspace bw = carve_bwd(workspace, d, shared);
  if (ws_bytes < bw.bytes) return MOE_ERR_WORKSPACE;
  if (d.T == 0) return MOE_OK;
  return run_backward(static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(Wg),
                      static_cast<const uint16_t*>(W1), static_cast<const uint16_t*>(W3),
                      static_cast<const uint16_t*>(W2), static_cast<const uint16_t*>(Ws1),
                      static_cast<const uint16_t*>(Ws3), static_cast<const uint16_t*>(Ws2),
                      static_cast<const uint16_t*>(d_out), d, fw, bw, static_cast<uint16_t*>(dx),
                      dWg, dbias, dW1, dW3, dW2, dWs1, dWs3, dWs2, opts,
                      static_cast<cudaStream_t>(stream));
}

size_t moe_ffn_workspace_size(moe_dims d, int has_shared, int host_io) {
  if (check_dims(d) != MOE_OK) return 0;
  return carve(nullptr, d, has_shared != 0, host_io != 0).bytes;
}

moe_status moe_ffn_forward(const void* x, const void* Wg, const float* router_bias, const void* W1,
                           const void* W3, const void* W2, const void* Ws1, const void* Ws3,
                           const void* Ws2, moe_dims d, void* out, void* workspace, size_t ws_bytes,
                           const moe_ffn_options* opts, void* stream) {
  if (check_dims(d) == MOE_OK && d.T == 0) return MOE_OK;
  moe_status st = validate_layer(x, Wg, router_bias, W1, W3, W2, Ws1, Ws3, Ws2, d, out, workspace,
                                 opts, false);
  if (st != MOE_OK) return st;
  const bool shared = Ws1 != nullptr;
  const Workspace ws = carve(workspace, d, shared, false);
  if (ws_bytes < ws.bytes) return MOE_ERR_WORKSPACE;
  if (d.T == 0) return MOE_OK;
  return run_layer(static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(Wg), router_bias,
                   static_cast<const uint16_t*>(W1), static_cast<const uint16_t*>(W3),
                   static_cast<const uint16_t*>(W2), static_cast<const uint16_t*>(Ws1),
                   static_cast<const uint16_t*>(Ws3), static_cast<const uint16_t*>(Ws2), d,
                   static_cast<uint16_t*>(out), ws, opts, static_cast<cudaStream_t>(stream));
}

moe_status moe_ffn_forward_host(const void* x_host, const void* Wg, const float* router_bias,
                                const void* W1, const void* W3, const void* W2, const void* Ws1,
                                const void* Ws3, const void* Ws2, moe_dims d, void* out_host,
                                void* workspace, size_t ws_bytes, const moe_ffn_options* opts,
                                void* stream) {
  if (check_dims(d) == MOE_OK && d.T == 0) return MOE_OK;
  moe_status st = validate_layer(x_host, Wg, router_bias, W1, W3, W2, Ws1, Ws3, Ws2, d, out_host,
                                 workspace, opts, true);
  if (st != MOE_OK) return st;
  const bool shared = Ws1 != nullptr;
  const Workspace ws = carve(workspace, d, shared, true);
  if (ws_bytes < ws.bytes) return MOE_ERR_WORKSPACE;
  if (d.T == 0) return MOE_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t xbytes = static_cast<size_t>(d.T) * d.D * 2;
  record(opts, 6, s);
  if (cudaMemcpyAsync(ws.x_stage, x_host, xbytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  st = run_layer(ws.x_stage, static_cast<const uint16_t*>(Wg), router_bias,
                 static_cast<const uint16_t*>(W1), static_cast<const uint16_t*>(W3),
                 static_cast<const uint16_t*>(W2), static_cast<const uint16_t*>(Ws1),
                 static_cast<const uint16_t*>(Ws3), static_cast<const uint16_t*>(Ws2), d,
                 ws.out_stage, ws, opts, s);
  if (st != MOE_OK) return st;
  if (cudaMemcpyAsync(out_host, ws.out_stage, xbytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  record(opts, 7, s);
  return MOE_OK;
}

size_t moe_route_scratch_size(moe_dims d) {
  if (check_dims(d) != MOE_OK) return 0;
  return route_packed_bytes(d.D, d.E);
}

moe_status moe_route(const void* x, const void* Wg, const float* router_bias, moe_dims d,
                     int32_t* ids, float* weights, int32_t* block_hist, void* scratch,
                     size_t scratch_bytes, void* stream) {
  moe_status st = check_dims(d);
  if (st != MOE_OK) return st;
  if (!x || !Wg || !ids || !weights || !scratch) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Wg) || !aligned16(scratch)) return MOE_ERR_INVALID_ARG;
  if (scratch_bytes < route_packed_bytes(d.D, d.E)) return MOE_ERR_WORKSPACE;
  if (d.T == 0) return MOE_OK;
  return cuda_status(launch_route(static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(Wg),
                                  router_bias, d, scratch, ids, weights, block_hist,
                                  static_cast<cudaStream_t>(stream)));
}

int moe_route_block_tokens(int T) { return route_block_tokens(T); }

size_t moe_permute_scratch_size(moe_dims d) {
  if (check_dims(d) != MOE_OK) return 0;
  return static_cast<size_t>(route_blocks_max(d.T)) * d.E * 4;
}

moe_status moe_permute(const int32_t* ids, moe_dims d, int32_t* counts, int32_t* offsets,
                       int32_t* perm, int32_t* inv, const void* x, void* x_sorted, void* scratch,
                       size_t scratch_bytes, void* stream) {
  moe_status st = check_dims(d);
  if (st != MOE_OK) return st;
  if (!ids || !counts || !offsets || !perm || !inv || !scratch) return MOE_ERR_INVALID_ARG;
  if ((x == nullptr) != (x_sorted == nullptr)) return MOE_ERR_INVALID_ARG;
  if (x && (!aligned16(x) || !aligned16(x_sorted))) return MOE_ERR_INVALID_ARG;
  if (scratch_bytes < static_cast<size_t>(route_blocks(d.T)) * d.E * 4) return MOE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d.T == 0) {
    return cuda_status(cudaMemsetAsync(counts, 0, sizeof(int32_t) * d.E, s)) == MOE_OK
               ? cuda_status(cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (d.E + 1), s))
               : MOE_ERR_CUDA;
  }
  int32_t* hist = static_cast<int32_t*>(scratch);
  if (launch_hist(ids, d, hist, s) != cudaSuccess) return MOE_ERR_CUDA;
  return cuda_status(launch_scatter(ids, hist, d, counts, offsets, perm, inv,
                                    static_cast<const uint16_t*>(x), static_cast<uint16_t*>(x_sorted),
                                    s));
}

moe_status moe_grouped_swiglu(const void* x_sorted, const void* x, const void* W1, const void* W3,
                              const void* Ws1, const void* Ws3, const int32_t* offsets, moe_dims d,
                              void* h, void* stream) {
  moe_status st = check_dims(d);
  if (st != MOE_OK) return st;
  if (!x_sorted || !W1 || !W3 || !offsets || !h) return MOE_ERR_INVALID_ARG;
  if ((Ws1 == nullptr) != (Ws3 == nullptr)) return MOE_ERR_INVALID_ARG;
  if (Ws1 != nullptr && x == nullptr) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x_sorted, x, W1, W3, Ws1, Ws3, h};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (d.T == 0) return MOE_OK;
  return cuda_status(launch_grouped_swiglu(
      static_cast<const uint16_t*>(x_sorted), static_cast<const uint16_t*>(x),
      static_cast<const uint16_t*>(W1), static_cast<const uint16_t*>(W3),
      static_cast<const uint16_t*>(Ws1), static_cast<const uint16_t*>(Ws3), offsets, d,
      static_cast<uint16_t*>(h), static_cast<cudaStream_t>(stream)));
}

moe_status moe_grouped_ffn_chained(const void* x_sorted, const void* x, const void* W1,
                                   const void* W3, const void* W2, const void* Ws1,
                                   const void* Ws3, const void* Ws2, const int32_t* offsets,
                                   moe_dims d, void* y, float* ys, void* stream) {
  moe_status st = check_dims(d);
  if (st != MOE_OK) return st;
  if (d.D > MOE_CHAINED_MAX_D) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!x_sorted || !W1 || !W3 || !W2 || !offsets || !y) return MOE_ERR_INVALID_ARG;
  if (shared_state(Ws1, Ws3, Ws2) < 0) return MOE_ERR_INVALID_ARG;
  if (Ws1 != nullptr && (x == nullptr || ys == nullptr)) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x_sorted, x, W1, W3, W2, Ws1, Ws3, Ws2, y, ys};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (d.T == 0) return MOE_OK;
  return cuda_status(launch_chained_ffn(
      static_cast<const uint16_t*>(x_sorted), static_cast<const uint16_t*>(x),
      static_cast<const uint16_t*>(W1), static_cast<const uint16_t*>(W3),
      static_cast<const uint16_t*>(W2), static_cast<const uint16_t*>(Ws1),
      static_cast<const uint16_t*>(Ws3), static_cast<const uint16_t*>(Ws2), offsets, d,
      static_cast<uint16_t*>(y), Ws1 != nullptr ? ys : nullptr, static_cast<cudaStream_t>(stream)));
}

moe_status moe_grouped_down(const void* h, const void* W2, const void* Ws2, const int32_t* offsets,
                            moe_dims d, void* y, float* ys, void* stream) {
  moe_status st = check_dims(d);
  if (st != MOE_OK) return st;
  if (!h || !W2 || !offsets || !y) return MOE_ERR_INVALID_ARG;
  if (Ws2 != nullptr && ys == nullptr) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {h, W2, Ws2, y, ys};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (d.T == 0) return MOE_OK;
  return cuda_status(launch_grouped_down(static_cast<const uint16_t*>(h),
                                         static_cast<const uint16_t*>(W2),
                                         static_cast<const uint16_t*>(Ws2), offsets, d,
                                         static_cast<uint16_t*>(y), Ws2 != nullptr ? ys : nullptr,
                                         static_cast<cudaStream_t>(stream)));
}

moe_status moe_combine(const void* y, const float* ys, const float* weights, const int32_t* inv, moe_dims d,
                       void* out, void* stream) {
  moe_status st = check_dims(d);
  if (st != MOE_OK) return st;
  if (!y || !weights || !inv || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y) || !aligned16(out) || (ys != nullptr && !aligned16(ys))) return MOE_ERR_INVALID_ARG;
  if (d.T == 0) return MOE_OK;
  return cuda_status(launch_combine(static_cast<const uint16_t*>(y), ys, weights, inv, d,
                                    static_cast<uint16_t*>(out), static_cast<cudaStream_t>(stream)));
}

moe_status moe_device_error(void) {
  unsigned int v = 0;
  if (read_clear_device_error(&v) != cudaSuccess) return MOE_ERR_CUDA;
  return v ? MOE_ERR_DEVICE_TIMEOUT : MOE_OK;
}

moe_status moe_selftest_wait_timeout(int timeout_us, int32_t* gave_up, void* stream) {
  if (timeout_us < 1 || timeout_us > 1000000 || gave_up == nullptr) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_wait_timeout_selftest(static_cast<uint64_t>(timeout_us) * 1000ull, gave_up,
                                                  static_cast<cudaStream_t>(stream)));
}

uint64_t moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* moe_status_str(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_DEVICE_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

}  // extern "C"
