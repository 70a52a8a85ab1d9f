// Gate-weighted sum back in token order:  y[t] = sum_slot G_slot(x_t) · E_slot(x_t) (+ residual)
//   "Mixtral of Experts" (xyznot.com summary), Método, eq. y = sum_i G(x)_i · SwiGLU_i(x);
//   the experts' outputs return to the original token positions (ja.news.hada.io,
//   実装と推論効率).
// One block per token row; 16-byte vectors; fp32 accumulation in ascending slot order, one
// rounding at the end (deterministic, no atomics).  A slot whose inv_perm entry lies outside
// [0, T*k) adds nothing (no row is read for it).
#include "moe_internal.cuh"

namespace moe {
namespace {

template <int K>
__global__ void __launch_bounds__(256) combine_bf16_vec_kernel(const uint4* __restrict__ y_perm,
                                                               const int32_t* __restrict__ inv_perm,
                                                               const float* __restrict__ w,
                                                               const uint4* residual, int Tn,
                                                               int row_vecs, int kk, uint4* y) {
  const int k = K > 0 ? K : kk;
  for (int t = blockIdx.x; t < Tn; t += gridDim.x) {
    int rows[kMaxExperts];
    float ws[kMaxExperts];
    const int A = Tn * k;
    for (int s = 0; s < k; ++s) {
      const int p = __ldg(inv_perm + (size_t)t * k + s);
      const bool ok = p >= 0 && p < A;
      rows[s] = ok ? p : -1;
      ws[s] = ok ? __ldg(w + (size_t)t * k + s) : 0.f;
    }
    for (int c = threadIdx.x; c < row_vecs; c += blockDim.x) {
      float acc[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = 0.f;
      for (int s = 0; s < k; ++s) {
        if (rows[s] < 0) continue;
        const uint4 v = __ldg(y_perm + (size_t)rows[s] * row_vecs + c);
        const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = __bfloat1622float2(p[j]);
          acc[2 * j] = fmaf(ws[s], f.x, acc[2 * j]);
          acc[2 * j + 1] = fmaf(ws[s], f.y, acc[2 * j + 1]);
        }
      }
      if (residual) {
        const uint4 v = residual[(size_t)t * row_vecs + c];
        const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = __bfloat1622float2(p[j]);
          acc[2 * j] += f.x;
          acc[2 * j + 1] += f.y;
        }
      }
      uint4 o;
      __nv_bfloat162* q = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
      for (int j = 0; j < 4; ++j) q[j] = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
      y[(size_t)t * row_vecs + c] = o;
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(256) combine_generic_kernel(const T* __restrict__ y_perm,
                                                              const int32_t* __restrict__ inv_perm,
                                                              const float* __restrict__ w,
                                                              const T* residual, int Tn, int d,
                                                              int k, T* y) {
  for (int t = blockIdx.x; t < Tn; t += gridDim.x) {
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
      float acc = 0.f;
      for (int s = 0; s < k; ++s) {
        const int p = __ldg(inv_perm + (size_t)t * k + s);
        if (p < 0 || p >= Tn * k) continue;
        acc = fmaf(__ldg(w + (size_t)t * k + s), to_f32(y_perm[(size_t)p * d + c]), acc);
      }
      if (residual) acc += to_f32(residual[(size_t)t * d + c]);
      y[(size_t)t * d + c] = from_f32<T>(acc);
    }
  }
}

// y = a + b row by row (bf16 storage, fp32 add, one rounding): the residual of a sub-block
// whose output is not already summed with it.
__global__ void __launch_bounds__(256) add_rows_bf16_kernel(const uint4* __restrict__ a,
                                                            const uint4* __restrict__ b,
                                                            size_t vecs, uint4* __restrict__ y) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < vecs;
       i += (size_t)gridDim.x * blockDim.x) {
    const uint4 u = __ldg(a + i), v = __ldg(b + i);
    const __nv_bfloat162* pu = reinterpret_cast<const __nv_bfloat162*>(&u);
    const __nv_bfloat162* pv = reinterpret_cast<const __nv_bfloat162*>(&v);
    uint4 o;
    __nv_bfloat162* po = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 x = __bfloat1622float2(pu[j]), z = __bfloat1622float2(pv[j]);
      po[j] = __floats2bfloat162_rn(x.x + z.x, x.y + z.y);
    }
    y[i] = o;
  }
}

// offsets of one group holding every row: {0, rows}
__global__ void span_offsets_kernel(int32_t* off, int rows) {
  if (threadIdx.x == 0) {
    off[0] = 0;
    off[1] = rows;
  }
}

}  // namespace

cudaError_t launch_add_rows_bf16(const void* a, const void* b, size_t elems, void* y,
                                 cudaStream_t s) {
  if (elems == 0) return cudaSuccess;
  const size_t vecs = elems / 8;
  const int cap = device_sm_count() * 8;
  const size_t want = (vecs + 255) / 256;
  const int grid = (int)(want < (size_t)cap ? (want > 0 ? want : 1) : cap);
  add_rows_bf16_kernel<<<grid, 256, 0, s>>>((const uint4*)a, (const uint4*)b, vecs, (uint4*)y);
  return cudaGetLastError();
}

cudaError_t launch_span_offsets(int32_t* off, int rows, cudaStream_t s) {
  span_offsets_kernel<<<1, 32, 0, s>>>(off, rows);
  return cudaGetLastError();
}

cudaError_t launch_combine(const void* y_perm, const int32_t* inv_perm, const float* w,
                           const void* residual, int T, int d, int k, int dtype, void* y,
                           cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int cap = device_sm_count() * 8;
  const int grid = T < cap ? T : cap;
  if (dtype == MOE_BF16 && d % 8 == 0) {
    const int rv = d / 8;
    const int threads = rv >= 256 ? 256 : ((rv + 31) / 32) * 32;
    if (k == 2)
      combine_bf16_vec_kernel<2><<<grid, threads, 0, s>>>((const uint4*)y_perm, inv_perm, w,
                                                          (const uint4*)residual, T, rv, k, (uint4*)y);
    else
      combine_bf16_vec_kernel<0><<<grid, threads, 0, s>>>((const uint4*)y_perm, inv_perm, w,
                                                          (const uint4*)residual, T, rv, k, (uint4*)y);
  } else if (dtype == MOE_BF16) {
    combine_generic_kernel<bf16><<<grid, 256, 0, s>>>((const bf16*)y_perm, inv_perm, w,
                                                      (const bf16*)residual, T, d, k, (bf16*)y);
  } else {
    combine_generic_kernel<float><<<grid, 256, 0, s>>>((const float*)y_perm, inv_perm, w,
                                                       (const float*)residual, T, d, k, (float*)y);
  }
  return cudaGetLastError();
}

}  // namespace moe
