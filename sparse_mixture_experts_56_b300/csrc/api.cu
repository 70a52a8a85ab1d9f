// C ABI of libmoe.so: argument validation, workspace layout and the launch sequence of
// the MoE layer  y = sum_i G(x)_i · E_i(x),  G(x) = Softmax(TopK(x · W_g))
// ("Mixtral of Experts" (xyznot.com summary), Método; blog.csdn.net MOE数学公式).
// Everything is stream-ordered; nothing here synchronises except moe_check_device_error.
#include <atomic>
#include <mutex>

#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr unsigned long long kDefaultWaitNs = 2000000000ull;
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

struct Layout {
  size_t scratch, idx, w, offsets, perm, inv_perm, x_perm, h, y_perm;
  size_t permute_end, grouped_end, total;
};

Layout layout(long long T, long long d, long long f, int n, int k, int dtype) {
  const size_t esz = dtype == MOE_BF16 ? 2 : 4;
  const long long A = T * k;
  Layout L;
  size_t off = kAlign;  // status header
  L.scratch = off;
  off += align_up(permute_scratch_words(A, n) * sizeof(int32_t));
  L.permute_end = off;
  L.idx = off;
  off += align_up((size_t)A * sizeof(int32_t));
  L.w = off;
  off += align_up((size_t)A * sizeof(float));
  L.offsets = off;
  off += align_up((size_t)(n + 1) * sizeof(int32_t));
  L.perm = off;
  off += align_up((size_t)A * sizeof(int32_t));
  L.inv_perm = off;
  off += align_up((size_t)A * sizeof(int32_t));
  L.x_perm = off;
  off += align_up((size_t)A * d * esz);
  L.h = off;
  off += align_up((size_t)A * f * esz);
  L.grouped_end = off;
  L.y_perm = off;
  off += align_up((size_t)A * d * esz);
  L.total = off;
  return L;
}

// Backward workspace: the router / grouping part of the forward layout, then the padded
// expert-ordered buffers of the backward (rows_max rows each).
struct BwdLayout {
  size_t poff, wq, x_pad, g_pad, dx_pad, ab, da, db, hw, dwp, dl, part, total;
  int rows_max, ntiles;
};

inline bool use_tc(int dtype, int d, int f);

BwdLayout bwd_layout(long long T, long long d, long long f, int n, int k, int dtype) {
  const Layout L = layout(T, d, f, n, k, dtype);
  BwdLayout B;
  const long long A = T * k;
  const size_t esz = dtype == MOE_BF16 ? 2 : 4;
  B.rows_max = bwd_rows_max(A, n);
  B.ntiles = use_tc(dtype, (int)d, (int)f) ? bwd_dh_ntiles((int)f) : bwd_simt_ntiles((int)f);
  const size_t R = (size_t)B.rows_max;
  size_t off = L.x_perm;   // everything before x_perm is shared with the forward layout
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align_up(bytes);
    return at;
  };
  B.poff = take((size_t)(n + 1) * 4);
  B.wq = take(R * 4);
  B.x_pad = take(R * d * esz);
  B.g_pad = take(R * d * esz);
  B.dx_pad = take(R * d * esz);
  B.ab = take(R * 2 * f * esz);
  B.da = take(R * f * esz);
  B.db = take(R * f * esz);
  B.hw = take(R * f * esz);
  B.dwp = take(R * B.ntiles * 4);
  B.dl = take((size_t)T * n * 4);
  B.part = take((size_t)bwd_dwg_chunks((int)T) * (d + 1) * n * 4);
  B.total = off;
  return B;
}

// Decoder layer workspace: the MoE layer's workspace first (its status header is the
// decoder's), then the attention sub-block's buffers.
struct DecLayout {
  size_t offs, xn, q, k, v, o, oproj, h1, xn2, total;
};

DecLayout dec_layout(long long T, long long d, long long f, int n, int k, int hq, int hkv) {
  const Layout L = layout(T, d, f, n, k, MOE_BF16);
  DecLayout D;
  size_t off = L.total;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align_up(bytes);
    return at;
  };
  const size_t row = (size_t)T * 2;
  D.offs = take(2 * sizeof(int32_t));
  D.xn = take(row * d);
  D.q = take(row * hq * 128);
  D.k = take(row * hkv * 128);
  D.v = take(row * hkv * 128);
  D.o = take(row * hq * 128);
  D.oproj = take(row * d);
  D.h1 = take(row * d);
  D.xn2 = take(row * d);
  D.total = off;
  return D;
}

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
inline bool dtype_ok(int dt) { return dt == MOE_F32 || dt == MOE_BF16; }

bool sizes_ok(long long T, long long d, long long f, int n, int k) {
  if (T < 0 || d < 1 || f < 1) return false;
  if (n < 1 || n > kMaxExperts || k < 1 || k > n) return false;
  if (T * k >= (1ll << 31)) return false;
  if (d >= (1ll << 31) || f >= (1ll << 31)) return false;
  return true;
}

inline moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

inline uint32_t* status_word(void* ws) { return reinterpret_cast<uint32_t*>(ws); }

// The tensor-core path takes bf16 shapes whose rows are whole 64-element swizzle atoms.
inline bool use_tc(int dtype, int d, int f) { return dtype == MOE_BF16 && d % 64 == 0 && f % 64 == 0; }

moe_status up_impl(const void* x, const int32_t* perm, const int32_t* offsets, const void* w1,
                   const void* w3, int T, int d, int f, int n, int k, int dtype, void* h, void* ws,
                   const Layout& L, cudaStream_t s) {
  const int A = T * k;
  if (A == 0) return MOE_OK;
  void* x_perm = static_cast<char*>(ws) + L.x_perm;
  const size_t esz = dtype == MOE_BF16 ? 2 : 4;
  cudaError_t e = launch_gather_rows(x, perm, A, k, (size_t)d * esz, x_perm, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  const int nb = use_tc(dtype, d, f) ? swap_rows(T) : 0;
  if (nb > 0)
    e = launch_up_swap((const bf16*)x_perm, offsets, (const bf16*)w1, (const bf16*)w3, A, d, f, n,
                       nb, (bf16*)h, status_word(ws), g_wait_ns.load(), s);
  else if (use_tc(dtype, d, f))
    e = launch_up_tc((const bf16*)x_perm, offsets, (const bf16*)w1, (const bf16*)w3, A, d, f, n,
                     (bf16*)h, status_word(ws), g_wait_ns.load(), s);
  else
    e = launch_up_simt(x_perm, offsets, w1, w3, A, d, f, n, dtype, h, s);
  return cuda_status(e);
}

moe_status down_impl(const void* h, const int32_t* offsets, const void* w2, int T, int d, int f,
                     int n, int k, int dtype, void* y_perm, void* ws, cudaStream_t s) {
  const int A = T * k;
  if (A == 0) return MOE_OK;
  cudaError_t e;
  const int nb = use_tc(dtype, d, f) ? swap_rows(T) : 0;
  if (nb > 0)
    e = launch_down_swap((const bf16*)h, offsets, (const bf16*)w2, A, d, f, n, nb, (bf16*)y_perm,
                         status_word(ws), g_wait_ns.load(), s);
  else if (use_tc(dtype, d, f))
    e = launch_down_tc((const bf16*)h, offsets, (const bf16*)w2, A, d, f, n, (bf16*)y_perm,
                       status_word(ws), g_wait_ns.load(), s);
  else
    e = launch_down_simt(h, offsets, w2, A, d, f, n, dtype, y_perm, s);
  return cuda_status(e);
}

moe_status grouped_impl(const void* x, const int32_t* perm, const int32_t* offsets, const void* w1,
                        const void* w3, const void* w2, int T, int d, int f, int n, int k, int dtype,
                        void* y_perm, void* ws, const Layout& L, cudaStream_t s) {
  void* h = static_cast<char*>(ws) + L.h;
  moe_status st = up_impl(x, perm, offsets, w1, w3, T, d, f, n, k, dtype, h, ws, L, s);
  if (st != MOE_OK) return st;
  return down_impl(h, offsets, w2, T, d, f, n, k, dtype, y_perm, ws, s);
}

struct Routing {
  int32_t *idx, *offsets, *perm, *inv_perm, *poff;
  float* w;
};

// What moe_layer_forward_train keeps for moe_layer_backward_saved: the routing and the
// expert inputs a = x w1ᵀ, b = x w3ᵀ (bf16) in the expert-padded row order.
struct SavedLayout {
  size_t idx, w, offsets, perm, inv_perm, poff, ab, total;
};

SavedLayout saved_layout(long long T, long long d, long long f, int n, int k) {
  const long long A = T * k;
  SavedLayout S;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align_up(bytes);
    return at;
  };
  S.idx = take((size_t)A * 4);
  S.w = take((size_t)A * 4);
  S.offsets = take((size_t)(n + 1) * 4);
  S.perm = take((size_t)A * 4);
  S.inv_perm = take((size_t)A * 4);
  S.poff = take((size_t)(n + 1) * 4);
  S.ab = take((size_t)bwd_rows_max(A, n) * 2 * f * 2);
  S.total = off;
  (void)d;
  return S;
}

moe_status check_backward_args(const void* x, const void* w_gate, const void* w1, const void* w3,
                               const void* w2, const void* dy, int T, int d, int f, int n, int k,
                               int dtype, const void* dx, const float* dw_gate, const void* dw1,
                               const void* dw3, const void* dw2) {
  if (!dtype_ok(dtype) || !sizes_ok(T, d, f, n, k)) return MOE_ERR_INVALID_ARG;
  if (!w_gate || !w1 || !w3 || !w2 || !dw_gate || !dw1 || !dw3 || !dw2) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !dy || !dx)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w_gate) || !aligned16(w1) || !aligned16(w3) || !aligned16(w2) ||
      !aligned16(dw1) || !aligned16(dw3) || !aligned16(dw2) || ((uintptr_t)dw_gate & 3u) ||
      (T > 0 && (!aligned16(x) || !aligned16(dy) || !aligned16(dx))))
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// No tokens: every gradient is zero.
moe_status zero_grads(int d, int f, int n, int dtype, float* dw_gate, float* dlogit_bias, void* dw1,
                      void* dw3, void* dw2, cudaStream_t s) {
  const size_t wbytes = (size_t)n * f * d * (dtype == MOE_BF16 ? 2 : 4);
  cudaError_t e = cudaMemsetAsync(dw1, 0, wbytes, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(dw3, 0, wbytes, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(dw2, 0, wbytes, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(dw_gate, 0, (size_t)d * n * 4, s);
  if (e == cudaSuccess && dlogit_bias) e = cudaMemsetAsync(dlogit_bias, 0, (size_t)n * 4, s);
  return cuda_status(e);
}

// The backward after the routing (and its padded offsets) exists: gather, the expert GEMMs
// (recomputing a | b unless ab_saved holds them), the router's part and dW_g.
moe_status backward_core(const void* x, const void* w_gate, const void* w1, const void* w3,
                         const void* w2, const void* dy, int T, int d, int f, int n, int k,
                         int dtype, void* dx, float* dw_gate, float* dlogit_bias, void* dw1,
                         void* dw3, void* dw2, void* ws, const BwdLayout& B, const Routing& r,
                         const bf16* ab_saved, cudaStream_t s) {
  char* base = static_cast<char*>(ws);
  const size_t esz = dtype == MOE_BF16 ? 2 : 4;
  float* wq = reinterpret_cast<float*>(base + B.wq);
  // padded expert-ordered buffers in the storage dtype (bf16 on the tensor-core path)
  bf16* x_pad = reinterpret_cast<bf16*>(base + B.x_pad);
  bf16* g_pad = reinterpret_cast<bf16*>(base + B.g_pad);
  bf16* dx_pad = reinterpret_cast<bf16*>(base + B.dx_pad);
  bf16* ab = reinterpret_cast<bf16*>(base + B.ab);
  bf16* da = reinterpret_cast<bf16*>(base + B.da);
  bf16* db = reinterpret_cast<bf16*>(base + B.db);
  bf16* hw = reinterpret_cast<bf16*>(base + B.hw);
  float* dwp = reinterpret_cast<float*>(base + B.dwp);
  float* dl = reinterpret_cast<float*>(base + B.dl);
  float* part = reinterpret_cast<float*>(base + B.part);
  uint32_t* st = status_word(ws);
  const unsigned long long wn = g_wait_ns.load();
  const int R = B.rows_max;
  const int32_t* poff = r.poff;
  cudaError_t e = launch_gather_bwd(x, dy, r.offsets, poff, r.perm, r.w, n, k, R, (size_t)d * esz,
                                    x_pad, g_pad, wq, s);
  if (use_tc(dtype, d, f)) {
    // experts: a | b (saved by the forward, or recomputed), then dh' = dy w2 with the SwiGLU
    // backward in its epilogue
    if (!ab_saved && e == cudaSuccess)
      e = launch_bwd_store_ab(x_pad, poff, (const bf16*)w1, (const bf16*)w3, R, d, f, n, ab, st,
                              wn, s);
    if (e == cudaSuccess)
      e = launch_bwd_dh(g_pad, poff, (const bf16*)w2, ab_saved ? ab_saved : ab, wq, R, d, f, n,
                        dwp, da, db, hw, st, wn, s);
    if (e == cudaSuccess)
      e = launch_bwd_dgrad_x(da, db, poff, (const bf16*)w1, (const bf16*)w3, R, d, f, n, dx_pad,
                             st, wn, s);
    // weight gradients: dW1_e = da_eᵀ x_e, dW3_e = db_eᵀ x_e, dW2_e = dy_eᵀ (G h)_e
    if (e == cudaSuccess) e = launch_bwd_wgrad(da, x_pad, poff, R, f, d, n, (bf16*)dw1, st, wn, s);
    if (e == cudaSuccess) e = launch_bwd_wgrad(db, x_pad, poff, R, f, d, n, (bf16*)dw3, st, wn, s);
    if (e == cudaSuccess) e = launch_bwd_wgrad(g_pad, hw, poff, R, d, f, n, (bf16*)dw2, st, wn, s);
  } else if (e == cudaSuccess) {
    e = launch_bwd_experts_simt(x_pad, g_pad, poff, w1, w3, w2, wq, R, d, f, n, dtype, ab, dwp, da,
                                db, hw, dx_pad, dw1, dw3, dw2, s);
  }
  // router: gate and logit gradients, dx, then dW_g and the bias gradient
  if (e == cudaSuccess)
    e = launch_router_bwd(r.idx, r.w, r.offsets, poff, r.inv_perm, dwp, B.ntiles, dx_pad, w_gate,
                          T, d, n, k, dtype, dx, dl, s);
  if (e == cudaSuccess) e = launch_dwg(x, dl, T, d, n, dtype, part, dw_gate, dlogit_bias, s);
  return cuda_status(e);
}

}  // namespace

int device_sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    sms = 148;
  if (dev < 64) cache[dev] = sms;
  return sms;
}

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_DEVICE_INDEX: return "MOE_ERR_DEVICE_INDEX";
    default: return "MOE_ERR_UNKNOWN";
  }
}

int moe_version(void) { return 100; }

size_t moe_workspace_size(int T, int d, int f, int n, int k, int dtype) {
  if (!dtype_ok(dtype) || !sizes_ok(T, d, f, n, k)) return 0;
  return layout(T, d, f, n, k, dtype).total;
}

moe_status moe_router_topk(const void* x, const void* w_gate, const float* logit_bias, int T, int d,
                           int n, int k, int dtype, int32_t* topk_idx, float* topk_w, float* logits,
                           void* stream) {
  MOE_CALL_RANGE();
  if (!dtype_ok(dtype) || !sizes_ok(T, d, 1, n, k)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !w_gate || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_gate)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_router_topk(x, w_gate, logit_bias, T, d, n, k, dtype, topk_idx, topk_w,
                                        logits, (cudaStream_t)stream));
}

moe_status moe_permute(const int32_t* topk_idx, int T, int k, int n, int32_t* expert_offsets,
                       int32_t* perm, int32_t* inv_perm, void* ws, size_t ws_bytes, void* stream) {
  MOE_CALL_RANGE();
  if (!sizes_ok(T, 64, 64, n, k)) return MOE_ERR_INVALID_ARG;
  if (!expert_offsets || (T > 0 && (!topk_idx || !perm || !inv_perm))) return MOE_ERR_INVALID_ARG;
  const Layout L = layout(T, 64, 64, n, k, MOE_BF16);
  if (!ws || ws_bytes < L.permute_end || !aligned16(ws)) return MOE_ERR_WORKSPACE;
  char* base = static_cast<char*>(ws);
  return cuda_status(launch_permute(topk_idx, T * k, n, expert_offsets, perm, inv_perm,
                                    reinterpret_cast<int32_t*>(base + L.scratch), status_word(ws),
                                    (cudaStream_t)stream));
}

moe_status moe_grouped_swiglu(const void* x, const int32_t* perm, const int32_t* expert_offsets,
                              const void* w1, const void* w3, const void* w2, int T, int d, int f,
                              int n, int k, int dtype, void* y_perm, void* ws, size_t ws_bytes,
                              void* stream) {
  MOE_CALL_RANGE();
  if (!dtype_ok(dtype) || !sizes_ok(T, d, f, n, k)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !perm || !expert_offsets || !w1 || !w3 || !w2 || !y_perm) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w1) || !aligned16(w3) || !aligned16(w2) || !aligned16(y_perm))
    return MOE_ERR_INVALID_ARG;
  const Layout L = layout(T, d, f, n, k, dtype);
  if (!ws || ws_bytes < L.grouped_end || !aligned16(ws)) return MOE_ERR_WORKSPACE;
  return grouped_impl(x, perm, expert_offsets, w1, w3, w2, T, d, f, n, k, dtype, y_perm, ws, L,
                      (cudaStream_t)stream);
}

moe_status moe_expert_up(const void* x, const int32_t* perm, const int32_t* expert_offsets,
                         const void* w1, const void* w3, int T, int d, int f, int n, int k,
                         int dtype, void* h, void* ws, size_t ws_bytes, void* stream) {
  MOE_CALL_RANGE();
  if (!dtype_ok(dtype) || !sizes_ok(T, d, f, n, k)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !perm || !expert_offsets || !w1 || !w3 || !h) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w1) || !aligned16(w3) || !aligned16(h)) return MOE_ERR_INVALID_ARG;
  const Layout L = layout(T, d, f, n, k, dtype);
  if (!ws || ws_bytes < L.grouped_end || !aligned16(ws)) return MOE_ERR_WORKSPACE;
  return up_impl(x, perm, expert_offsets, w1, w3, T, d, f, n, k, dtype, h, ws, L,
                 (cudaStream_t)stream);
}

moe_status moe_expert_down(const void* h, const int32_t* expert_offsets, const void* w2, int T,
                           int d, int f, int n, int k, int dtype, void* y_perm, void* ws,
                           size_t ws_bytes, void* stream) {
  MOE_CALL_RANGE();
  if (!dtype_ok(dtype) || !sizes_ok(T, d, f, n, k)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!h || !expert_offsets || !w2 || !y_perm) return MOE_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(w2) || !aligned16(y_perm)) return MOE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < kAlign || !aligned16(ws)) return MOE_ERR_WORKSPACE;
  return down_impl(h, expert_offsets, w2, T, d, f, n, k, dtype, y_perm, ws, (cudaStream_t)stream);
}

moe_status moe_combine(const void* y_perm, const int32_t* inv_perm, const float* topk_w,
                       const void* residual, int T, int d, int k, int dtype, void* y, void* stream) {
  MOE_CALL_RANGE();
  if (!dtype_ok(dtype) || !sizes_ok(T, d, 1, k, k)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!y_perm || !inv_perm || !topk_w || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_perm) || !aligned16(y) || (residual && !aligned16(residual)))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine(y_perm, inv_perm, topk_w, residual, T, d, k, dtype, y,
                                    (cudaStream_t)stream));
}

moe_status moe_rmsnorm(const void* h, int T, int d, float eps, int dtype, void* x, void* stream) {
  MOE_CALL_RANGE();
  if (!dtype_ok(dtype) || !sizes_ok(T, d, 1, 1, 1) || !(eps >= 0.f)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!h || !x || h == x || !aligned16(h) || !aligned16(x)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_rmsnorm(h, T, d, eps, dtype, x, (cudaStream_t)stream));
}

moe_status moe_layer_forward(const void* x, const void* w_gate, const float* logit_bias,
                             const void* w1, const void* w3, const void* w2, const void* residual,
                             int T, int d, int f, int n, int k, int dtype, void* y,
                             int32_t* topk_idx_out, int32_t* expert_offsets_out, void* ws,
                             size_t ws_bytes, void* stream) {
  MOE_CALL_RANGE();
  if (!dtype_ok(dtype) || !sizes_ok(T, d, f, n, k)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (T == 0) {
    if (expert_offsets_out)
      return cuda_status(cudaMemsetAsync(expert_offsets_out, 0, (size_t)(n + 1) * 4, s));
    return MOE_OK;
  }
  if (!x || !w_gate || !w1 || !w3 || !w2 || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_gate) || !aligned16(w1) || !aligned16(w3) || !aligned16(w2) ||
      !aligned16(y) || (residual && !aligned16(residual)))
    return MOE_ERR_INVALID_ARG;
  const Layout L = layout(T, d, f, n, k, dtype);
  if (!ws || ws_bytes < L.total || !aligned16(ws)) return MOE_ERR_WORKSPACE;
  char* base = static_cast<char*>(ws);
  int32_t* idx = reinterpret_cast<int32_t*>(base + L.idx);
  float* w = reinterpret_cast<float*>(base + L.w);
  int32_t* offsets = reinterpret_cast<int32_t*>(base + L.offsets);
  int32_t* perm = reinterpret_cast<int32_t*>(base + L.perm);
  int32_t* inv_perm = reinterpret_cast<int32_t*>(base + L.inv_perm);
  void* y_perm = base + L.y_perm;
  const int A = T * k;

  cudaError_t e = launch_router_topk(x, w_gate, logit_bias, T, d, n, k, dtype, idx, w, nullptr, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  e = launch_permute(idx, A, n, offsets, perm, inv_perm, reinterpret_cast<int32_t*>(base + L.scratch),
                     status_word(ws), s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  moe_status st = grouped_impl(x, perm, offsets, w1, w3, w2, T, d, f, n, k, dtype, y_perm, ws, L, s);
  if (st != MOE_OK) return st;
  e = launch_combine(y_perm, inv_perm, w, residual, T, d, k, dtype, y, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  if (topk_idx_out &&
      cudaMemcpyAsync(topk_idx_out, idx, (size_t)A * 4, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (expert_offsets_out && cudaMemcpyAsync(expert_offsets_out, offsets, (size_t)(n + 1) * 4,
                                            cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

size_t moe_backward_workspace_size(int T, int d, int f, int n, int k, int dtype) {
  if (!dtype_ok(dtype) || !sizes_ok(T, d, f, n, k)) return 0;
  return bwd_layout(T, d, f, n, k, dtype).total;
}

moe_status moe_layer_backward(const void* x, const void* w_gate, const float* logit_bias,
                              const void* w1, const void* w3, const void* w2, const void* dy,
                              int T, int d, int f, int n, int k, int dtype, void* dx,
                              float* dw_gate, float* dlogit_bias, void* dw1, void* dw3, void* dw2,
                              void* ws, size_t ws_bytes, void* stream) {
  MOE_CALL_RANGE();
  moe_status st = check_backward_args(x, w_gate, w1, w3, w2, dy, T, d, f, n, k, dtype, dx,
                                      dw_gate, dw1, dw3, dw2);
  if (st != MOE_OK) return st;
  const BwdLayout B = bwd_layout(T, d, f, n, k, dtype);
  if (!ws || ws_bytes < B.total || !aligned16(ws)) return MOE_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  if (T == 0) return zero_grads(d, f, n, dtype, dw_gate, dlogit_bias, dw1, dw3, dw2, s);
  const Layout L = layout(T, d, f, n, k, dtype);
  char* base = static_cast<char*>(ws);
  Routing r;
  r.idx = reinterpret_cast<int32_t*>(base + L.idx);
  r.w = reinterpret_cast<float*>(base + L.w);
  r.offsets = reinterpret_cast<int32_t*>(base + L.offsets);
  r.perm = reinterpret_cast<int32_t*>(base + L.perm);
  r.inv_perm = reinterpret_cast<int32_t*>(base + L.inv_perm);
  r.poff = reinterpret_cast<int32_t*>(base + B.poff);
  // the forward's routing, recomputed (same kernels, same inputs, same result)
  cudaError_t e =
      launch_router_topk(x, w_gate, logit_bias, T, d, n, k, dtype, r.idx, r.w, nullptr, s);
  if (e == cudaSuccess)
    e = launch_permute(r.idx, T * k, n, r.offsets, r.perm, r.inv_perm,
                       reinterpret_cast<int32_t*>(base + L.scratch), status_word(ws), s);
  if (e == cudaSuccess) e = launch_pad_offsets(r.offsets, n, r.poff, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  return backward_core(x, w_gate, w1, w3, w2, dy, T, d, f, n, k, dtype, dx, dw_gate, dlogit_bias,
                       dw1, dw3, dw2, ws, B, r, nullptr, s);
}

size_t moe_train_saved_size(int T, int d, int f, int n, int k, int dtype) {
  if (!use_tc(dtype, d, f) || !sizes_ok(T, d, f, n, k)) return 0;
  return saved_layout(T, d, f, n, k).total;
}

moe_status moe_layer_forward_train(const void* x, const void* w_gate, const float* logit_bias,
                                   const void* w1, const void* w3, const void* w2,
                                   const void* residual, int T, int d, int f, int n, int k,
                                   int dtype, void* y, void* saved, size_t saved_bytes, void* ws,
                                   size_t ws_bytes, void* stream) {
  MOE_CALL_RANGE();
  if (!dtype_ok(dtype) || !sizes_ok(T, d, f, n, k)) return MOE_ERR_INVALID_ARG;
  if (!use_tc(dtype, d, f)) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!x || !w_gate || !w1 || !w3 || !w2 || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_gate) || !aligned16(w1) || !aligned16(w3) || !aligned16(w2) ||
      !aligned16(y) || (residual && !aligned16(residual)))
    return MOE_ERR_INVALID_ARG;
  const Layout L = layout(T, d, f, n, k, dtype);
  if (!ws || ws_bytes < L.total || !aligned16(ws)) return MOE_ERR_WORKSPACE;
  const SavedLayout S = saved_layout(T, d, f, n, k);
  if (!saved || saved_bytes < S.total || !aligned16(saved)) return MOE_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  char* base = static_cast<char*>(ws);
  char* sv = static_cast<char*>(saved);
  int32_t* idx = reinterpret_cast<int32_t*>(sv + S.idx);
  float* w = reinterpret_cast<float*>(sv + S.w);
  int32_t* offsets = reinterpret_cast<int32_t*>(sv + S.offsets);
  int32_t* perm = reinterpret_cast<int32_t*>(sv + S.perm);
  int32_t* inv_perm = reinterpret_cast<int32_t*>(sv + S.inv_perm);
  int32_t* poff = reinterpret_cast<int32_t*>(sv + S.poff);
  bf16* ab = reinterpret_cast<bf16*>(sv + S.ab);
  const int A = T * k;
  uint32_t* st = status_word(ws);
  cudaError_t e = launch_router_topk(x, w_gate, logit_bias, T, d, n, k, dtype, idx, w, nullptr, s);
  if (e == cudaSuccess)
    e = launch_permute(idx, A, n, offsets, perm, inv_perm,
                       reinterpret_cast<int32_t*>(base + L.scratch), st, s);
  if (e == cudaSuccess) e = launch_pad_offsets(offsets, n, poff, s);
  if (e == cudaSuccess) e = launch_zero_pad_rows(ab, offsets, poff, n, 2 * f, s);
  void* x_perm = base + L.x_perm;
  bf16* h = reinterpret_cast<bf16*>(base + L.h);
  void* y_perm = base + L.y_perm;
  if (e == cudaSuccess) e = launch_gather_rows(x, perm, A, k, (size_t)d * 2, x_perm, s);
  if (e == cudaSuccess)
    e = launch_up_tc((const bf16*)x_perm, offsets, (const bf16*)w1, (const bf16*)w3, A, d, f, n, h,
                     st, g_wait_ns.load(), s, ab, poff);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  moe_status ms = down_impl(h, offsets, w2, T, d, f, n, k, dtype, y_perm, ws, s);
  if (ms != MOE_OK) return ms;
  return cuda_status(launch_combine(y_perm, inv_perm, w, residual, T, d, k, dtype, y, s));
}

moe_status moe_layer_backward_saved(const void* x, const void* w_gate, const void* w1,
                                    const void* w3, const void* w2, const void* dy, int T, int d,
                                    int f, int n, int k, int dtype, const void* saved,
                                    size_t saved_bytes, void* dx, float* dw_gate,
                                    float* dlogit_bias, void* dw1, void* dw3, void* dw2, void* ws,
                                    size_t ws_bytes, void* stream) {
  MOE_CALL_RANGE();
  moe_status st = check_backward_args(x, w_gate, w1, w3, w2, dy, T, d, f, n, k, dtype, dx,
                                      dw_gate, dw1, dw3, dw2);
  if (st != MOE_OK) return st;
  if (!use_tc(dtype, d, f)) return MOE_ERR_UNSUPPORTED;
  const BwdLayout B = bwd_layout(T, d, f, n, k, dtype);
  if (!ws || ws_bytes < B.total || !aligned16(ws)) return MOE_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  if (T == 0) return zero_grads(d, f, n, dtype, dw_gate, dlogit_bias, dw1, dw3, dw2, s);
  const SavedLayout S = saved_layout(T, d, f, n, k);
  if (!saved || saved_bytes < S.total || !aligned16(saved)) return MOE_ERR_WORKSPACE;
  char* sv = const_cast<char*>(static_cast<const char*>(saved));
  Routing r;
  r.idx = reinterpret_cast<int32_t*>(sv + S.idx);
  r.w = reinterpret_cast<float*>(sv + S.w);
  r.offsets = reinterpret_cast<int32_t*>(sv + S.offsets);
  r.perm = reinterpret_cast<int32_t*>(sv + S.perm);
  r.inv_perm = reinterpret_cast<int32_t*>(sv + S.inv_perm);
  r.poff = reinterpret_cast<int32_t*>(sv + S.poff);
  return backward_core(x, w_gate, w1, w3, w2, dy, T, d, f, n, k, dtype, dx, dw_gate, dlogit_bias,
                       dw1, dw3, dw2, ws, B, r, reinterpret_cast<const bf16*>(sv + S.ab), s);
}

moe_status moe_attention_gqa(const void* q, const void* k, const void* v, int T, int seq_len,
                             int hq, int hkv, int dh, int dtype, void* out, void* ws,
                             size_t ws_bytes, void* stream) {
  MOE_CALL_RANGE();
  if (!dtype_ok(dtype) || T < 0 || seq_len < 0 || hq < 1 || hkv < 1 || dh < 1 || hq % hkv)
    return MOE_ERR_INVALID_ARG;
  if ((long long)T * hq * dh >= (1ll << 40)) return MOE_ERR_INVALID_ARG;
  if (dtype != MOE_BF16 || dh != 128) return MOE_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < kAlign || !aligned16(ws)) return MOE_ERR_WORKSPACE;
  if (T == 0) return MOE_OK;
  if (!q || !k || !v || !out || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_attention_gqa((const bf16*)q, (const bf16*)k, (const bf16*)v, T,
                                          seq_len, hq, hkv, (bf16*)out, status_word(ws),
                                          g_wait_ns.load(), (cudaStream_t)stream));
}

size_t moe_decoder_workspace_size(int T, int d, int f, int n, int k, int hq, int hkv) {
  if (!sizes_ok(T, d, f, n, k) || hq < 1 || hkv < 1 || hq % hkv) return 0;
  return dec_layout(T, d, f, n, k, hq, hkv).total;
}

moe_status moe_decoder_layer_forward(const void* h, const void* wq, const void* wk, const void* wv,
                                     const void* wo, const void* w_gate, const float* logit_bias,
                                     const void* w1, const void* w3, const void* w2, int T, int d,
                                     int f, int n, int k, int hq, int hkv, int seq_len, float eps,
                                     int dtype, void* y, int32_t* topk_idx_out, void* ws,
                                     size_t ws_bytes, void* stream) {
  MOE_CALL_RANGE();
  if (!dtype_ok(dtype) || !sizes_ok(T, d, f, n, k) || hq < 1 || hkv < 1 || hq % hkv ||
      seq_len < 0 || !(eps >= 0.f))
    return MOE_ERR_INVALID_ARG;
  if ((long long)T * hq * 128 >= (1ll << 40)) return MOE_ERR_INVALID_ARG;
  if (dtype != MOE_BF16 || !use_tc(dtype, d, f)) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!h || !wq || !wk || !wv || !wo || !w_gate || !w1 || !w3 || !w2 || !y)
    return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {h, wq, wk, wv, wo, w_gate, w1, w3, w2, y};
  for (const void* p : ptrs)
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  const Layout L = layout(T, d, f, n, k, dtype);
  const DecLayout D = dec_layout(T, d, f, n, k, hq, hkv);
  if (!ws || ws_bytes < D.total || !aligned16(ws)) return MOE_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  char* base = static_cast<char*>(ws);
  int32_t* offs = reinterpret_cast<int32_t*>(base + D.offs);
  bf16* xn = reinterpret_cast<bf16*>(base + D.xn);
  bf16* q = reinterpret_cast<bf16*>(base + D.q);
  bf16* kk = reinterpret_cast<bf16*>(base + D.k);
  bf16* v = reinterpret_cast<bf16*>(base + D.v);
  bf16* o = reinterpret_cast<bf16*>(base + D.o);
  bf16* oproj = reinterpret_cast<bf16*>(base + D.oproj);
  bf16* h1 = reinterpret_cast<bf16*>(base + D.h1);
  bf16* xn2 = reinterpret_cast<bf16*>(base + D.xn2);
  uint32_t* st = status_word(ws);
  const unsigned long long wn = g_wait_ns.load();
  const int dq = hq * 128, dkv = hkv * 128;
  // attention sub-block: RMSNorm, the three projections (plain GEMMs: the grouped tensor-core
  // kernel over one group holding every row), causal GQA attention, the output projection and
  // the residual
  cudaError_t e = launch_rmsnorm(h, T, d, eps, dtype, xn, s);
  if (e == cudaSuccess) e = launch_span_offsets(offs, T, s);
  if (e == cudaSuccess) e = launch_down_tc(xn, offs, (const bf16*)wq, T, dq, d, 1, q, st, wn, s);
  if (e == cudaSuccess) e = launch_down_tc(xn, offs, (const bf16*)wk, T, dkv, d, 1, kk, st, wn, s);
  if (e == cudaSuccess) e = launch_down_tc(xn, offs, (const bf16*)wv, T, dkv, d, 1, v, st, wn, s);
  if (e == cudaSuccess) e = launch_attention_gqa(q, kk, v, T, seq_len, hq, hkv, o, st, wn, s);
  if (e == cudaSuccess) e = launch_down_tc(o, offs, (const bf16*)wo, T, d, dq, 1, oproj, st, wn, s);
  if (e == cudaSuccess) e = launch_add_rows_bf16(h, oproj, (size_t)T * d, h1, s);
  // MoE sub-block: RMSNorm, the layer, the residual (in its combine)
  if (e == cudaSuccess) e = launch_rmsnorm(h1, T, d, eps, dtype, xn2, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  return moe_layer_forward(xn2, w_gate, logit_bias, w1, w3, w2, h1, T, d, f, n, k, dtype, y,
                           topk_idx_out, nullptr, ws, L.total, stream);
}

moe_status moe_routing_stats(const int32_t* topk_idx, int T, int k, int n, int seq_len,
                             int64_t* expert_counts, int64_t* pair_counts, void* stream) {
  MOE_CALL_RANGE();
  if (!sizes_ok(T, 1, 1, n, k) || seq_len < 0) return MOE_ERR_INVALID_ARG;
  if (!expert_counts || !pair_counts || (T > 0 && !topk_idx)) return MOE_ERR_INVALID_ARG;
  if (((uintptr_t)expert_counts & 7u) || ((uintptr_t)pair_counts & 7u) ||
      ((uintptr_t)topk_idx & 3u))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_routing_stats(topk_idx, T, k, n, seq_len, expert_counts, pair_counts,
                                          (cudaStream_t)stream));
}

moe_status moe_check_device_error(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || ws_bytes < kAlign) return MOE_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (word != 0) {
    if (cudaMemsetAsync(ws, 0, sizeof(word), s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (word & kDevErrTimeout) return MOE_ERR_TIMEOUT;
  if (word & kDevErrIndex) return MOE_ERR_DEVICE_INDEX;
  return MOE_OK;
}

void moe_set_wait_limit_ns(unsigned long long ns) { g_wait_ns.store(ns ? ns : kDefaultWaitNs); }

moe_status moe_set_tc_form(int form) {
  if (form != MOE_TC_FORM_AUTO && form != MOE_TC_FORM_SINGLE && form != MOE_TC_FORM_PAIR &&
      form != MOE_TC_FORM_SWAP)
    return MOE_ERR_INVALID_ARG;
  set_tc_form(form);
  set_swap_form(form);
  return MOE_OK;
}

}  // extern "C"
