// The backward's expert GEMMs on CUDA cores, for the shapes the tensor-core path does not take
// (fp32 storage, or bf16 with d or f not a multiple of 64).  Same steps, same expert-padded
// row layout and the same results up to fp32 summation order as the tcgen05 modes:
//   kAB   [a | b] = x_pad [w1_e | w3_e]ᵀ                          (recompute, stored)
//   kDh   dh' = g_pad w2_e; epilogue: h = SiLU(a) b, per-tile partial <dh', h>,
//         da = G dh' b SiLU'(a), db = G dh' SiLU(a), hw = G h       (G = the row's gate)
//   kDx   dx_pad = da w1_e + db w3_e
//   kDW   dW_e = Pᵀ Q over expert e's padded rows
// ("Mixtral of Experts" (xyznot.com summary), Método: SwiGLU experts; the derivative of the
// forward by the chain rule.)  fp32 products and accumulation; stored values take the storage
// dtype.  Tiles of 32 rows x 64 columns, 32-deep k-steps through shared memory, operands
// read with arbitrary element strides (either operand may be stored transposed).
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int SBM = 32, SBN = 64, SBK = 32;
enum SimtMode { kAB = 0, kDh = 1, kDx = 2, kDW = 3 };

// operand element (r, c) = p[r * rs + c * cs]
template <typename T>
struct Operand {
  const T* p;
  long long rs, cs;
};

template <typename T>
__device__ __forceinline__ void stage(float (&dst)[SBM > SBN ? SBM : SBN][SBK + 1], int rows,
                                      const Operand<T>& op, int r0, int rmax, int k0, int kmax) {
  // rows x SBK elements (r, k) = op(r0 + r, k0 + k); the unit-stride index runs fastest
  const bool k_fast = op.cs == 1;
  for (int i = threadIdx.x; i < rows * SBK; i += blockDim.x) {
    const int r = k_fast ? i / SBK : i % rows;
    const int c = k_fast ? i % SBK : i / rows;
    const int gr = r0 + r, gk = k0 + c;
    dst[r][c] = (gr < rmax && gk < kmax) ? to_f32(op.p[(long long)gr * op.rs + (long long)gk * op.cs])
                                         : 0.f;
  }
}

template <typename T>
struct SimtArgs {
  const int32_t* poff;
  int n, rows_max;
  int M, N, K;           // per expert: output rows (kDW) / output columns / reduction length
  int ntiles;            // kDh: column tiles of f (partials per row)
  // per expert operand bases and strides; A is indexed (row, k), B (k, column)
  const T* a1; long long a1_rs, a1_cs;
  const T* a2;           // kDx: second A (db), same strides
  const T* b1; long long b1_rs, b1_cs; long long b_estride;   // expert e's B at b + e*b_estride
  const T* b2;           // kAB: w3; kDx: w3
  T* out;                // kAB: ab [rows, 2f]; kDx: dx_pad; kDW: dW [n, M, N]
  const T* ab;           // kDh
  const float* wq;       // kDh
  float* dwp;            // kDh
  T* da; T* db; T* hw;   // kDh
};

template <typename T, int MODE>
__global__ void __launch_bounds__(256) simt_bwd_kernel(const SimtArgs<T> args) {
  __shared__ float as[SBN][SBK + 1];   // rows of A (first SBM used)
  __shared__ float bs[SBN][SBK + 1];   // columns of B (stored transposed: [col][k])
  __shared__ float bs2[MODE == kAB ? SBN : 1][SBK + 1];
  __shared__ int s_e, s_r0, s_ok;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int n0 = blockIdx.x * SBN;
  const int mtiles_w = (args.M + SBM - 1) / SBM;
  for (int y = blockIdx.y;; y += gridDim.y) {
    __syncthreads();
    if (tid == 0) {
      int ok = 0, e = 0, r0 = 0;
      if (MODE == kDW) {
        if (y < args.n * mtiles_w) {
          ok = 1;
          e = y / mtiles_w;
          r0 = (y % mtiles_w) * SBM;
        }
      } else {
        r0 = y * SBM;
        if (r0 < args.poff[args.n] && r0 < args.rows_max) {
          ok = 1;
          while (e + 1 < args.n && args.poff[e + 1] <= r0) ++e;
        }
      }
      s_ok = ok;
      s_e = e;
      s_r0 = r0;
    }
    __syncthreads();
    if (!s_ok) return;
    const int e = s_e, r0 = s_r0;
    // operands of this tile
    Operand<T> A1, A2, B1, B2;
    int kmax, kb_split, rmax;
    if (MODE == kDW) {
      const int seg0 = args.poff[e], seg = args.poff[e + 1] - seg0;
      A1 = {args.a1 + (long long)seg0 * args.a1_cs, args.a1_rs, args.a1_cs};
      B1 = {args.b1 + (long long)seg0 * args.b1_rs, args.b1_rs, args.b1_cs};
      kmax = seg;
      kb_split = seg;
      rmax = args.M;
    } else {
      A1 = {args.a1, args.a1_rs, args.a1_cs};
      A2 = {args.a2, args.a1_rs, args.a1_cs};
      B1 = {args.b1 + (long long)e * args.b_estride, args.b1_rs, args.b1_cs};
      B2 = {args.b2 + (long long)e * args.b_estride, args.b1_rs, args.b1_cs};
      kmax = args.K;
      kb_split = MODE == kDx ? args.K / 2 : args.K;
      rmax = args.rows_max;
    }
    float acc[2][4] = {}, acc2[2][4] = {};
    // kDx runs the reduction in two halves (da with w1, then db with w3)
    const int klim = MODE == kDx ? kb_split : kmax;
    for (int half = 0; half < (MODE == kDx ? 2 : 1); ++half)
    for (int kk0 = 0; kk0 < klim; kk0 += SBK) {
      const bool second = half == 1;
      stage<T>(as, SBM, second ? A2 : A1, r0, rmax, kk0, klim);
      // B (k, col) staged as [col][k]: operand (col, k) has strides (cs, rs)
      const Operand<T>& Bk = second ? B2 : B1;
      stage<T>(bs, SBN, Operand<T>{Bk.p, Bk.cs, Bk.rs}, n0, args.N, kk0, klim);
      if constexpr (MODE == kAB)
        stage<T>(bs2, SBN, Operand<T>{B2.p, B2.cs, B2.rs}, n0, args.N, kk0, klim);
      __syncthreads();
#pragma unroll 8
      for (int c = 0; c < SBK; ++c) {
        const float xv0 = as[ty * 2][c], xv1 = as[ty * 2 + 1][c];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const float bv = bs[tx + 16 * jj][c];
          acc[0][jj] = fmaf(xv0, bv, acc[0][jj]);
          acc[1][jj] = fmaf(xv1, bv, acc[1][jj]);
          if (MODE == kAB) {
            const float bv2 = bs2[tx + 16 * jj][c];
            acc2[0][jj] = fmaf(xv0, bv2, acc2[0][jj]);
            acc2[1][jj] = fmaf(xv1, bv2, acc2[1][jj]);
          }
        }
      }
      __syncthreads();
    }
    // epilogue
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int row = r0 + ty * 2 + r;
      const bool row_ok = row < rmax;
      float dot = 0.f;
      const float gate = (MODE == kDh && row_ok) ? args.wq[row] : 0.f;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int col = n0 + tx + 16 * jj;
        if (!row_ok || col >= args.N) continue;
        const float v = acc[r][jj];
        if (MODE == kAB) {
          args.out[(size_t)row * 2 * args.N + col] = from_f32<T>(v);
          args.out[(size_t)row * 2 * args.N + args.N + col] = from_f32<T>(acc2[r][jj]);
        } else if (MODE == kDh) {
          const float a = to_f32(args.ab[(size_t)row * 2 * args.N + col]);
          const float b = to_f32(args.ab[(size_t)row * 2 * args.N + args.N + col]);
          const float sg = 1.0f / (1.0f + expf(-a));
          const float si = a * sg;
          dot = fmaf(v, si * b, dot);
          const size_t o = (size_t)row * args.N + col;
          args.da[o] = from_f32<T>(gate * v * b * sg * (1.0f + a * (1.0f - sg)));
          args.db[o] = from_f32<T>(gate * v * si);
          args.hw[o] = from_f32<T>(gate * si * b);
        } else if (MODE == kDx) {
          args.out[(size_t)row * args.N + col] = from_f32<T>(v);
        } else {
          args.out[((size_t)e * args.M + row) * args.N + col] = from_f32<T>(v);
        }
      }
      if (MODE == kDh) {
        // the 16 threads of this row pair sit in one half-warp: a fixed-order tree
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        if (tx == 0 && row_ok) args.dwp[(size_t)row * args.ntiles + blockIdx.x] = dot;
      }
    }
  }
}

template <typename T, int MODE>
cudaError_t launch(const SimtArgs<T>& a, int ytiles, cudaStream_t s) {
  dim3 g((a.N + SBN - 1) / SBN, ytiles < 65535 ? (ytiles > 0 ? ytiles : 1) : 65535);
  simt_bwd_kernel<T, MODE><<<g, 256, 0, s>>>(a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t run(const void* x_pad, const void* g_pad, const int32_t* poff, const void* w1,
                const void* w3, const void* w2, const float* wq, int rows_max, int d, int f, int n,
                void* ab, float* dwp, void* da, void* db, void* hw, void* dx_pad, void* dw1,
                void* dw3, void* dw2, cudaStream_t s) {
  const int rt = rows_max / SBM;
  SimtArgs<T> a = {};
  a.poff = poff;
  a.n = n;
  a.rows_max = rows_max;
  cudaError_t e;
  // recompute [a | b]: A = x_pad (rows, d); B(k in d, col in f) = w[e][col][k]
  a.M = rows_max; a.N = f; a.K = d;
  a.a1 = (const T*)x_pad; a.a1_rs = d; a.a1_cs = 1;
  a.b1 = (const T*)w1; a.b2 = (const T*)w3; a.b1_rs = 1; a.b1_cs = d; a.b_estride = (long long)f * d;
  a.out = (T*)ab;
  if ((e = launch<T, kAB>(a, rt, s)) != cudaSuccess) return e;
  // dh' = g_pad w2_e: B(k in d, col in f) = w2[e][k][col]
  a.a1 = (const T*)g_pad;
  a.b1 = (const T*)w2; a.b2 = nullptr; a.b1_rs = f; a.b1_cs = 1; a.b_estride = (long long)d * f;
  a.ab = (const T*)ab; a.wq = wq; a.dwp = dwp; a.ntiles = (f + SBN - 1) / SBN;
  a.da = (T*)da; a.db = (T*)db; a.hw = (T*)hw; a.out = nullptr;
  if ((e = launch<T, kDh>(a, rt, s)) != cudaSuccess) return e;
  // dx_pad = da w1_e + db w3_e: A = da | db (rows, f); B(k in f, col in d) = w[e][k][col]
  a.N = d; a.K = 2 * f;
  a.a1 = (const T*)da; a.a2 = (const T*)db; a.a1_rs = f; a.a1_cs = 1;
  a.b1 = (const T*)w1; a.b2 = (const T*)w3; a.b1_rs = d; a.b1_cs = 1; a.b_estride = (long long)f * d;
  a.out = (T*)dx_pad;
  if ((e = launch<T, kDx>(a, rt, s)) != cudaSuccess) return e;
  // weight gradients over each expert's rows: A(m, k) = P[k][m], B(k, j) = Q[k][j]
  struct W { const void* P; const void* Q; int M, N; void* out; } ws[3] = {
      {da, x_pad, f, d, dw1}, {db, x_pad, f, d, dw3}, {g_pad, hw, d, f, dw2}};
  for (const W& w : ws) {
    SimtArgs<T> b = {};
    b.poff = poff;
    b.n = n;
    b.rows_max = rows_max;
    b.M = w.M; b.N = w.N;
    b.a1 = (const T*)w.P; b.a1_rs = 1; b.a1_cs = w.M;
    b.b1 = (const T*)w.Q; b.b1_rs = w.N; b.b1_cs = 1;
    b.out = (T*)w.out;
    if ((e = launch<T, kDW>(b, n * ((w.M + SBM - 1) / SBM), s)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

int bwd_simt_ntiles(int f) { return (f + SBN - 1) / SBN; }

cudaError_t launch_bwd_experts_simt(const void* x_pad, const void* g_pad, const int32_t* poff,
                                    const void* w1, const void* w3, const void* w2,
                                    const float* wq, int rows_max, int d, int f, int n, int dtype,
                                    void* ab, float* dwp, void* da, void* db, void* hw,
                                    void* dx_pad, void* dw1, void* dw3, void* dw2,
                                    cudaStream_t s) {
  if (dtype == MOE_BF16)
    return run<bf16>(x_pad, g_pad, poff, w1, w3, w2, wq, rows_max, d, f, n, ab, dwp, da, db, hw,
                     dx_pad, dw1, dw3, dw2, s);
  return run<float>(x_pad, g_pad, poff, w1, w3, w2, wq, rows_max, d, f, n, ab, dwp, da, db, hw,
                    dx_pad, dw1, dw3, dw2, s);
}

}  // namespace moe
