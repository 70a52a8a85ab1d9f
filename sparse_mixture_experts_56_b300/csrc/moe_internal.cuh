// Internal declarations shared by the kernel files and the C-ABI layer of libmoe.so.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "moe.h"

namespace moe {

// Bits of the device status word (first 4 bytes of the workspace).
enum : uint32_t { kDevErrTimeout = 1u, kDevErrIndex = 2u };

constexpr int kMaxExperts = 32;

// Assignments handled by one block of the permutation kernels (32 warps x 1024).
constexpr int kPermuteChunk = 32768;

typedef __nv_bfloat16 bf16;

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<bf16>(bf16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ bf16 from_f32<bf16>(float v) { return __float2bfloat16_rn(v); }

// A named NVTX range around one call of the C ABI, so that a timeline tool (Nsight Systems,
// ncu's range filters) shows each call by name; without a tool attached the push and pop
// cost a few nanoseconds and do nothing.
struct CallRange {
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};
#define MOE_CALL_RANGE() ::moe::CallRange moe_call_range_(__func__)

// A setting that belongs to each device's context (a kernel's dynamic shared-memory limit):
// applied once per device, the first time a launch on that device needs it, and its result
// kept.  A process that drives several GPUs applies it on each.
constexpr int kMaxDevices = 64;
struct PerDeviceSetting {
  std::mutex mu;
  bool done[kMaxDevices] = {};
  cudaError_t err[kMaxDevices] = {};
  template <typename Apply>
  cudaError_t get(Apply apply) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
      return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev]) {
      err[dev] = apply();
      done[dev] = true;
    }
    return err[dev];
  }
};

// ---------------------------------------------------------------------------------------
// Launchers (host functions; every one returns the launch error of its kernels)
// ---------------------------------------------------------------------------------------
cudaError_t launch_router_topk(const void* x, const void* wg, const float* bias, int T, int d, int n,
                               int k, int dtype, int32_t* idx, float* w, float* logits,
                               cudaStream_t s);
cudaError_t launch_rmsnorm(const void* h, int T, int d, float eps, int dtype, void* x, cudaStream_t s);

// Permutation: per-block counts of the n experts and the trailing bucket of bad indices live
// in `scratch` (permute_scratch_words int32: 2 * nblocks * (n + 1)) when T*k > chunk.
int permute_blocks(long long A);
size_t permute_scratch_words(long long A, int n);
cudaError_t launch_permute(const int32_t* idx, int A, int n, int32_t* offsets, int32_t* perm,
                           int32_t* inv_perm, int32_t* scratch, uint32_t* status, cudaStream_t s);

// x_perm[p] = x[perm[p] / k]  (rows of `row_bytes` bytes)
cudaError_t launch_gather_rows(const void* x, const int32_t* perm, int A, int k, size_t row_bytes,
                               void* x_perm, cudaStream_t s);

// y = a + b for bf16 buffers of `elems` elements (a multiple of 8, 16-byte aligned)
cudaError_t launch_add_rows_bf16(const void* a, const void* b, size_t elems, void* y, cudaStream_t s);
// off[0] = 0, off[1] = rows: one group of every row (a plain GEMM through the grouped kernels)
cudaError_t launch_span_offsets(int32_t* off, int rows, cudaStream_t s);

cudaError_t launch_combine(const void* y_perm, const int32_t* inv_perm, const float* w,
                           const void* residual, int T, int d, int k, int dtype, void* y,
                           cudaStream_t s);

// fp32 / generic CUDA-core experts (x_perm already gathered).
cudaError_t launch_up_simt(const void* x_perm, const int32_t* offsets, const void* w1, const void* w3,
                           int A, int d, int f, int n, int dtype, void* h, cudaStream_t s);
cudaError_t launch_down_simt(const void* h, const int32_t* offsets, const void* w2, int A, int d,
                             int f, int n, int dtype, void* y_perm, cudaStream_t s);

// bf16 tcgen05 experts: up = w1|w3 GEMM with SiLU(a)*b fused; down = w2 GEMM.
// ab_save / poff_save (optional): also store a and b for the backward, in the expert-padded
// row order, as bf16 [rows, 2f].
cudaError_t launch_up_tc(const bf16* x_perm, const int32_t* offsets, const bf16* w1, const bf16* w3,
                         int A, int d, int f, int n, bf16* h, uint32_t* status,
                         unsigned long long wait_ns, cudaStream_t s, bf16* ab_save = nullptr,
                         const int32_t* poff_save = nullptr);
cudaError_t launch_down_tc(const bf16* h, const int32_t* offsets, const bf16* w2, int A, int d,
                           int f, int n, bf16* y_perm, uint32_t* status, unsigned long long wait_ns,
                           cudaStream_t s);

// The same two GEMMs for small token batches, operands swapped (weights as the 128-row MMA
// operand, the expert's token rows, in blocks of nb = 16..64, as the N operand); inference
// only (no a|b saved).  swap_rows(T): the block size the launchers use for a batch of T
// tokens, or 0 for the forms above.
int swap_rows(int T);
void set_swap_form(int form);
cudaError_t launch_up_swap(const bf16* x_perm, const int32_t* offsets, const bf16* w1,
                           const bf16* w3, int A, int d, int f, int n, int nb, bf16* h,
                           uint32_t* status, unsigned long long wait_ns, cudaStream_t s);
cudaError_t launch_down_swap(const bf16* h, const int32_t* offsets, const bf16* w2, int A, int d,
                             int f, int n, int nb, bf16* y_perm, uint32_t* status,
                             unsigned long long wait_ns, cudaStream_t s);

// Backward on the tensor cores, rows in the expert-padded layout (segments of `poff` are
// multiples of 128 rows; rows_max bounds the padded row count):
//   store_ab: ab[q] = [x_pad[q] w1_eᵀ | x_pad[q] w3_eᵀ]                         [rows, 2f]
//   dh:       dh' = g_pad[q] w2_e;  with a, b from ab and the row's gate G = wq[q]:
//             dwp[q, j] = <dh', SiLU(a) b> over column tile j,  da = G dh' b SiLU'(a),
//             db = G dh' SiLU(a),  hw = G SiLU(a) b                            [rows, f]
//   dgrad_x:  dx_pad[q] = da[q] w1_e + db[q] w3_e                              [rows, d]
//   wgrad:    dW_e = P_eᵀ Q_e over expert e's rows (P [rows, M], Q [rows, N]) [n, M, N]
int bwd_dh_ntiles(int f);
cudaError_t launch_bwd_store_ab(const bf16* x_pad, const int32_t* poff, const bf16* w1,
                                const bf16* w3, int rows_max, int d, int f, int n, bf16* ab,
                                uint32_t* status, unsigned long long wait_ns, cudaStream_t s);
cudaError_t launch_bwd_dh(const bf16* g_pad, const int32_t* poff, const bf16* w2, const bf16* ab,
                          const float* wq, int rows_max, int d, int f, int n, float* dwp, bf16* da,
                          bf16* db, bf16* hw, uint32_t* status, unsigned long long wait_ns,
                          cudaStream_t s);
cudaError_t launch_bwd_dgrad_x(const bf16* da, const bf16* db, const int32_t* poff, const bf16* w1,
                               const bf16* w3, int rows_max, int d, int f, int n, bf16* dx_pad,
                               uint32_t* status, unsigned long long wait_ns, cudaStream_t s);
cudaError_t launch_bwd_wgrad(const bf16* P, const bf16* Q, const int32_t* poff, int rows_max,
                             int M, int N, int n, bf16* dW, uint32_t* status,
                             unsigned long long wait_ns, cudaStream_t s);

// Steps of the backward around the GEMMs (backward.cu).
int bwd_rows_max(long long A, int n);
int bwd_dwg_chunks(int T);
cudaError_t launch_pad_offsets(const int32_t* off, int n, int32_t* poff, cudaStream_t s);
cudaError_t launch_gather_bwd(const void* x, const void* dy, const int32_t* off,
                              const int32_t* poff, const int32_t* perm, const float* topk_w,
                              int n, int k, int rows_max, size_t row_bytes, void* x_pad,
                              void* g_pad, float* wq, cudaStream_t s);
cudaError_t launch_router_bwd(const int32_t* idx, const float* topk_w, const int32_t* off,
                              const int32_t* poff, const int32_t* inv_perm, const float* dwp,
                              int ntiles, const void* dx_pad, const void* wg, int T, int d, int n,
                              int k, int dtype, void* dx, float* dl, cudaStream_t s);
cudaError_t launch_dwg(const void* x, const float* dl, int T, int d, int n, int dtype,
                       float* part, float* dwg, float* dbias, cudaStream_t s);
// Zero the padding rows of a padded [rows, row_elems] bf16 buffer: rows
// [poff[e] + (off[e+1] - off[e]), poff[e+1]) of every expert.
cudaError_t launch_zero_pad_rows(bf16* buf, const int32_t* off, const int32_t* poff, int n,
                                 int row_elems, cudaStream_t s);
// The backward's expert GEMMs on CUDA cores (fp32, or bf16 shapes outside the tensor-core
// path): recompute, dy w2 with the SwiGLU backward, dx_pad, and the three weight gradients.
int bwd_simt_ntiles(int f);
cudaError_t launch_bwd_experts_simt(const void* x_pad, const void* g_pad, const int32_t* poff,
                                    const void* w1, const void* w3, const void* w2,
                                    const float* wq, int rows_max, int d, int f, int n, int dtype,
                                    void* ab, float* dwp, void* da, void* db, void* hw,
                                    void* dx_pad, void* dw1, void* dw3, void* dw2,
                                    cudaStream_t s);

// Causal grouped-query attention, head dimension 128, bf16 (attention.cu).
cudaError_t launch_attention_gqa(const bf16* q, const bf16* k, const bf16* v, int T, int seq_len,
                                 int hq, int hkv, bf16* out, uint32_t* status,
                                 unsigned long long wait_ns, cudaStream_t s);

// Which tensor-core GEMM form the launchers pick (MOE_TC_FORM_*; process-wide).
void set_tc_form(int form);

// Routing statistics of one layer (counts [n], pair_counts [3]: pairs, same first, shared).
cudaError_t launch_routing_stats(const int32_t* idx, int T, int k, int n, int seq_len,
                                 int64_t* counts, int64_t* pair_counts, cudaStream_t s);

int device_sm_count();

}  // namespace moe
