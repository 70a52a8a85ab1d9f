// Experts on CUDA cores (fp32 storage, or bf16 shapes the tensor-core path does not take):
//   y_perm[p] = w2_e · (SiLU(w1_e · x_p) ⊙ (w3_e · x_p))   for the rows p of expert e
//   ("Mixtral of Experts" (xyznot.com summary), Método: every expert is a SwiGLU network).
// fp32 products and accumulation (fp32 storage keeps the intermediate in fp32; bf16 storage
// rounds it to bf16 like the tensor-core path).  Tiles of 32 rows x 64 columns, k-steps of
// 32, operands staged in shared memory.  A block's rows never cross an expert boundary: the
// block's m-tile index is mapped to (expert, tile) from the device-side offsets.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int BM = 32, BN = 64, BK = 32;

// Finds the expert and row range of global m-tile `mt`; returns false past the last tile.
__device__ __forceinline__ bool find_tile(const int32_t* offsets, int n, int mt, int& e, int& row0,
                                          int& rows) {
  for (int i = 0; i < n; ++i) {
    const int cnt = offsets[i + 1] - offsets[i];
    const int tiles = (cnt + BM - 1) / BM;
    if (mt < tiles) {
      e = i;
      row0 = offsets[i] + mt * BM;
      rows = min(BM, cnt - mt * BM);
      return true;
    }
    mt -= tiles;
  }
  return false;
}

__device__ __forceinline__ float silu_f32(float a) { return a / (1.0f + expf(-a)); }

template <typename T, bool SWIGLU>
__global__ void __launch_bounds__(256) simt_grouped_kernel(const T* __restrict__ act,
                                                           const int32_t* __restrict__ offsets,
                                                           const T* __restrict__ wa,
                                                           const T* __restrict__ wb, int n,
                                                           int kdim, int ndim, T* __restrict__ out) {
  __shared__ float xs[BM][BK + 1];
  __shared__ float as[BN][BK + 1];
  __shared__ float bs[SWIGLU ? BN : 1][BK + 1];
  __shared__ int s_e, s_row0, s_rows, s_ok;
  for (int mt = blockIdx.y;; mt += gridDim.y) {
    __syncthreads();
    if (threadIdx.x == 0) {
      int e = 0, r0 = 0, rows = 0;
      s_ok = find_tile(offsets, n, mt, e, r0, rows) ? 1 : 0;
      s_e = e;
      s_row0 = r0;
      s_rows = rows;
    }
    __syncthreads();
    if (!s_ok) return;
    const int e = s_e, row0 = s_row0, rows = s_rows;
    const int n0 = blockIdx.x * BN;
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    const T* wa_e = wa + (size_t)e * ndim * kdim;
    const T* wb_e = SWIGLU ? wb + (size_t)e * ndim * kdim : nullptr;
    float accA[2][4] = {}, accB[2][4] = {};
    for (int k0 = 0; k0 < kdim; k0 += BK) {
      for (int i = tid; i < BM * BK; i += 256) {
        const int r = i / BK, c = i % BK;
        xs[r][c] =
            (r < rows && k0 + c < kdim) ? to_f32(act[(size_t)(row0 + r) * kdim + k0 + c]) : 0.f;
      }
      for (int i = tid; i < BN * BK; i += 256) {
        const int j = i / BK, c = i % BK;
        const bool ok = (n0 + j < ndim) && (k0 + c < kdim);
        as[j][c] = ok ? to_f32(wa_e[(size_t)(n0 + j) * kdim + k0 + c]) : 0.f;
        if (SWIGLU) bs[j][c] = ok ? to_f32(wb_e[(size_t)(n0 + j) * kdim + k0 + c]) : 0.f;
      }
      __syncthreads();
#pragma unroll 8
      for (int c = 0; c < BK; ++c) {
        float xv[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) xv[r] = xs[ty * 2 + r][c];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const float av = as[tx + 16 * jj][c];
          const float bv = SWIGLU ? bs[tx + 16 * jj][c] : 0.f;
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            accA[r][jj] = fmaf(xv[r], av, accA[r][jj]);
            if (SWIGLU) accB[r][jj] = fmaf(xv[r], bv, accB[r][jj]);
          }
        }
      }
      __syncthreads();
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int row = ty * 2 + r;
      if (row >= rows) continue;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int col = n0 + tx + 16 * jj;
        if (col >= ndim) continue;
        const float v = SWIGLU ? silu_f32(accA[r][jj]) * accB[r][jj] : accA[r][jj];
        out[(size_t)(row0 + row) * ndim + col] = from_f32<T>(v);
      }
    }
  }
}

int simt_mtiles(int A, int n) {
  const int m = (A + BM - 1) / BM + n;  // upper bound over all experts; blocks stride over it
  return m > 32768 ? 32768 : m;
}

}  // namespace

cudaError_t launch_up_simt(const void* x_perm, const int32_t* offsets, const void* w1, const void* w3,
                           int A, int d, int f, int n, int dtype, void* h, cudaStream_t s) {
  if (A == 0) return cudaSuccess;
  dim3 g((f + BN - 1) / BN, simt_mtiles(A, n));
  if (dtype == MOE_BF16)
    simt_grouped_kernel<bf16, true><<<g, 256, 0, s>>>((const bf16*)x_perm, offsets, (const bf16*)w1,
                                                      (const bf16*)w3, n, d, f, (bf16*)h);
  else
    simt_grouped_kernel<float, true><<<g, 256, 0, s>>>((const float*)x_perm, offsets,
                                                       (const float*)w1, (const float*)w3, n, d, f,
                                                       (float*)h);
  return cudaGetLastError();
}

cudaError_t launch_down_simt(const void* h, const int32_t* offsets, const void* w2, int A, int d,
                             int f, int n, int dtype, void* y_perm, cudaStream_t s) {
  if (A == 0) return cudaSuccess;
  dim3 g((d + BN - 1) / BN, simt_mtiles(A, n));
  if (dtype == MOE_BF16)
    simt_grouped_kernel<bf16, false><<<g, 256, 0, s>>>((const bf16*)h, offsets, (const bf16*)w2,
                                                       nullptr, n, f, d, (bf16*)y_perm);
  else
    simt_grouped_kernel<float, false><<<g, 256, 0, s>>>((const float*)h, offsets, (const float*)w2,
                                                        nullptr, n, f, d, (float*)y_perm);
  return cudaGetLastError();
}

}  // namespace moe
