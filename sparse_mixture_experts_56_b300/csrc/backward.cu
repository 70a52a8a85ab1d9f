// Backward of the layer y = sum_k G_k E_{e_k}(x), G = Softmax(TopK(x W_g + b)) ("Mixtral of
// Experts" (xyznot.com summary), Método, eqs. G and y; blog.csdn.net MOE数学公式 §2): the
// chain rule through the definitions, for L = <dy, y>.  TopK is piecewise constant, so only
// the kept logits receive gradient; the softmax over them gives
//     dl_k = G_k (dG_k - sum_j G_j dG_j),   dG_k = <dy, E_{e_k}(x)> = <w2ᵀ dy, h_k>.
// The experts' part runs on the tensor cores (grouped_tc.cu) in an expert-padded row layout:
// expert e's rows occupy [poff[e], poff[e+1]), a multiple of 128 rows, the padding rows being
// zero, so that no 128-row tile and no 64-row reduction block spans two experts.  This file
// holds the steps around those GEMMs:
//   pad_offsets   poff from the grouping's offsets
//   gather_bwd    x_pad, g_pad (rows of x and dy in padded expert order) and each row's gate G
//   router_bwd    per token: dG_k (sum of the GEMM epilogue's partial dot products, fixed
//                 order), dl over the kept experts, dx = sum_k dx_pad[q_k] + dl W_gᵀ
//   dwg_partial / dwg_reduce   dW_g = xᵀ dl and d(bias) = sum_t dl_t, in fixed order
#include <string.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kRowAlign = 128;
constexpr int kDwgChunk = 128;   // tokens per partial sum of dW_g
constexpr int kDwgBatch = 8;     // token rows of x in flight per thread (dW_g partial sums)

__global__ void pad_offsets_kernel(const int32_t* __restrict__ off, int n,
                                   int32_t* __restrict__ poff) {
  if (threadIdx.x == 0 && blockIdx.x == 0) {
    int acc = 0;
    for (int e = 0; e < n; ++e) {
      poff[e] = acc;
      const int m = off[e + 1] - off[e];
      acc += (m + kRowAlign - 1) / kRowAlign * kRowAlign;
    }
    poff[n] = acc;
  }
}

// One block per padded row q (grid-stride).  Rows past poff[n] are left alone.  V is the copy
// unit (16, 4 or 2 bytes, whichever divides the row).
template <typename V>
__global__ void __launch_bounds__(256) gather_bwd_kernel(
    const V* __restrict__ x, const V* __restrict__ dy, const int32_t* __restrict__ off,
    const int32_t* __restrict__ poff, const int32_t* __restrict__ perm,
    const float* __restrict__ topk_w, int n, int k, int rows_max, int row_vecs,
    V* __restrict__ x_pad, V* __restrict__ g_pad, float* __restrict__ wq) {
  __shared__ int s_poff[kMaxExperts + 1], s_off[kMaxExperts + 1];
  for (int i = threadIdx.x; i <= n; i += blockDim.x) {
    s_poff[i] = poff[i];
    s_off[i] = off[i];
  }
  __syncthreads();
  for (int q = blockIdx.x; q < rows_max && q < s_poff[n]; q += gridDim.x) {
    int e = 0;
    while (e + 1 < n && s_poff[e + 1] <= q) ++e;
    const int j = q - s_poff[e];
    V* xd = x_pad + (size_t)q * row_vecs;
    V* gd = g_pad + (size_t)q * row_vecs;
    if (j < s_off[e + 1] - s_off[e]) {
      const int a = __ldg(perm + s_off[e] + j);
      const int t = a / k;
      if (threadIdx.x == 0) wq[q] = __ldg(topk_w + a);
      const V* xs = x + (size_t)t * row_vecs;
      const V* gs = dy + (size_t)t * row_vecs;
      for (int c = threadIdx.x; c < row_vecs; c += blockDim.x) {
        xd[c] = __ldg(xs + c);
        gd[c] = __ldg(gs + c);
      }
    } else {
      if (threadIdx.x == 0) wq[q] = 0.f;
      V z;
      memset(&z, 0, sizeof(V));
      for (int c = threadIdx.x; c < row_vecs; c += blockDim.x) {
        xd[c] = z;
        gd[c] = z;
      }
    }
  }
}

// One warp per token (bf16, d % 8 == 0, n != 8).  dx[t] = sum_k dx_pad[q_k] + sum_k dl_k
// W_g[:, e_k]; dl [T, n] holds the logit gradient (zero outside the kept experts) for the dW_g
// reduction.
template <int KMAX>
__global__ void __launch_bounds__(256) router_bwd_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ topk_w,
    const int32_t* __restrict__ off, const int32_t* __restrict__ poff,
    const int32_t* __restrict__ inv_perm, const float* __restrict__ dwp, int ntiles,
    const bf16* __restrict__ dx_pad, const bf16* __restrict__ wg, int T, int d, int n, int k,
    bf16* __restrict__ dx, float* __restrict__ dl) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += warps) {
    int es[KMAX], qs[KMAX];
    float gate[KMAX], dG[KMAX];
    float sdot = 0.f;
#pragma unroll
    for (int s = 0; s < KMAX; ++s) {
      if (s < k) {
        const int a = t * k + s;
        const int e = __ldg(idx + a);
        es[s] = e;
        qs[s] = __ldg(poff + e) + (__ldg(inv_perm + a) - __ldg(off + e));
        gate[s] = __ldg(topk_w + a);
        // sum of the column-tile partials of <dw2ᵀ dy, h>: lane-strided, then a fixed tree
        float v = 0.f;
        for (int j = lane; j < ntiles; j += 32) v += __ldg(dwp + (size_t)qs[s] * ntiles + j);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        dG[s] = v;
        sdot = fmaf(gate[s], v, sdot);
      }
    }
    float dls[KMAX];
#pragma unroll
    for (int s = 0; s < KMAX; ++s)
      if (s < k) dls[s] = gate[s] * (dG[s] - sdot);
    // logit gradient row (zeros outside the kept experts)
    for (int e = lane; e < n; e += 32) {
      float v = 0.f;
#pragma unroll
      for (int s = 0; s < KMAX; ++s)
        if (s < k && es[s] == e) v = dls[s];
      dl[(size_t)t * n + e] = v;
    }
    // dx row, 8 columns per lane and step
    for (int c0 = lane * 8; c0 < d; c0 += 256) {
      float acc[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = 0.f;
#pragma unroll
      for (int s = 0; s < KMAX; ++s) {
        if (s < k) {
          const uint4 u = __ldg(reinterpret_cast<const uint4*>(dx_pad + (size_t)qs[s] * d + c0));
          const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 f2 = __bfloat1622float2(p[j]);
            acc[2 * j] += f2.x;
            acc[2 * j + 1] += f2.y;
          }
#pragma unroll
          for (int j = 0; j < 8; ++j)
            acc[j] = fmaf(dls[s], __bfloat162float(wg[(size_t)(c0 + j) * n + es[s]]), acc[j]);
        }
      }
      uint4 o;
      __nv_bfloat162* op = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
      for (int j = 0; j < 4; ++j) op[j] = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
      *reinterpret_cast<uint4*>(dx + (size_t)t * d + c0) = o;
    }
  }
}

// n == 8, bf16, d % 8 == 0: one warp per kRbTpw tokens.  The logit gradient of a token is
// kept as a dense row of 8 (zero outside its kept experts), so a row of W_g (8 bf16, one
// 16-byte load) serves every token of the warp and every slot without selecting an expert:
//     dx[t][c] = sum_k dx_pad[q_k][c] + sum_{e < 8} dl[t][e] W_g[c][e]
// (the second sum in ascending e; the zero terms add exactly nothing).
constexpr int kRbTpw = 4;
template <int KMAX>
__global__ void __launch_bounds__(256) router_bwd_n8_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ topk_w,
    const int32_t* __restrict__ off, const int32_t* __restrict__ poff,
    const int32_t* __restrict__ inv_perm, const float* __restrict__ dwp, int ntiles,
    const bf16* __restrict__ dx_pad, const bf16* __restrict__ wg, int T, int d, int k,
    bf16* __restrict__ dx, float* __restrict__ dl) {
  // per warp: the dense logit-gradient rows and the padded rows of its tokens
  __shared__ float s_dl[8][kRbTpw][8];
  __shared__ int s_q[8][kRbTpw][KMAX];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int t0 = ((blockIdx.x * blockDim.x + threadIdx.x) >> 5) * kRbTpw; t0 < T;
       t0 += warps * kRbTpw) {
    const int nt = min(kRbTpw, T - t0);
    const int slots = nt * k;   // (token i, slot s) pairs of the warp, p = i * k + s
    // lane p < slots: the padded row, expert and gate of pair p
    int my_e = 0, my_q = 0;
    float my_gate = 0.f;
    if (lane < slots) {
      const int i = lane / k, sl = lane - (lane / k) * k;
      const int a = (t0 + i) * k + sl;
      my_e = __ldg(idx + a);
      my_q = __ldg(poff + my_e) + (__ldg(inv_perm + a) - __ldg(off + my_e));
      my_gate = __ldg(topk_w + a);
      s_q[wib][i][sl] = my_q;
    }
    // dG of every pair: the sum of its column-tile partials of <dw2ᵀ dy, h>, lane-strided,
    // then a fixed tree; lane p keeps pair p's
    float my_dG = 0.f;
#pragma unroll
    for (int p = 0; p < kRbTpw * KMAX; ++p) {
      if (p >= slots) break;
      const int q = __shfl_sync(0xffffffffu, my_q, p);
      float v = 0.f;
      for (int j = lane; j < ntiles; j += 32) v += __ldg(dwp + (size_t)q * ntiles + j);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == p) my_dG = v;
    }
    // dl of pair p = G_p (dG_p - sum_s G_s dG_s over its token's slots, ascending s)
    const int first = (lane / k) * k;
    float sdot = 0.f;
    for (int sl = 0; sl < k; ++sl) {
      const float gv = __shfl_sync(0xffffffffu, my_gate, (first + sl) & 31);
      const float dv = __shfl_sync(0xffffffffu, my_dG, (first + sl) & 31);
      sdot = fmaf(gv, dv, sdot);
    }
    // the dense rows of 8 (zeros outside the kept experts), then the kept values
    s_dl[wib][lane >> 3][lane & 7] = 0.f;
    __syncwarp();
    if (lane < slots) s_dl[wib][lane / k][my_e] = my_gate * (my_dG - sdot);
    __syncwarp();
    if (lane < nt * 8) dl[(size_t)t0 * 8 + lane] = s_dl[wib][lane >> 3][lane & 7];
    // dx rows, 8 columns per lane and step: the 8 rows of W_g once for the warp's tokens
#pragma unroll 1
    for (int c0 = lane * 8; c0 < d; c0 += 256) {
      uint4 wr[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        wr[j] = __ldg(reinterpret_cast<const uint4*>(wg + (size_t)(c0 + j) * 8));
      // the dx_pad rows of every token of the warp are loaded before any is summed
      uint4 u[kRbTpw][KMAX];
#pragma unroll
      for (int i = 0; i < kRbTpw; ++i)
#pragma unroll
        for (int s = 0; s < KMAX; ++s)
          if (i < nt && s < k)
            u[i][s] = __ldg(reinterpret_cast<const uint4*>(dx_pad + (size_t)s_q[wib][i][s] * d + c0));
#pragma unroll
      for (int i = 0; i < kRbTpw; ++i) {
        if (i >= nt) break;
        const int t = t0 + i;
        float g[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) g[e] = s_dl[wib][i][e];
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.f;
#pragma unroll
        for (int s = 0; s < KMAX; ++s) {
          if (s < k) {
            const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u[i][s]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float2 f2 = __bfloat1622float2(p[j]);
              acc[2 * j] += f2.x;
              acc[2 * j + 1] += f2.y;
            }
          }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const __nv_bfloat162* wp = reinterpret_cast<const __nv_bfloat162*>(&wr[j]);
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const float2 f2 = __bfloat1622float2(wp[h]);
            acc[j] = fmaf(g[2 * h], f2.x, acc[j]);
            acc[j] = fmaf(g[2 * h + 1], f2.y, acc[j]);
          }
        }
        uint4 o;
        __nv_bfloat162* op = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
        for (int j = 0; j < 4; ++j) op[j] = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
        *reinterpret_cast<uint4*>(dx + (size_t)t * d + c0) = o;
      }
    }
    __syncwarp();
  }
}

// Generic form (any storage dtype, any d): one warp per token, one column per lane and step.
template <typename T, int KMAX>
__global__ void __launch_bounds__(256) router_bwd_generic_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ topk_w,
    const int32_t* __restrict__ off, const int32_t* __restrict__ poff,
    const int32_t* __restrict__ inv_perm, const float* __restrict__ dwp, int ntiles,
    const T* __restrict__ dx_pad, const T* __restrict__ wg, int Tn, int d, int n, int k,
    T* __restrict__ dx, float* __restrict__ dl) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < Tn; t += warps) {
    int es[KMAX], qs[KMAX];
    float gate[KMAX], dG[KMAX];
    float sdot = 0.f;
#pragma unroll
    for (int s = 0; s < KMAX; ++s) {
      if (s < k) {
        const int a = t * k + s;
        const int e = __ldg(idx + a);
        es[s] = e;
        qs[s] = __ldg(poff + e) + (__ldg(inv_perm + a) - __ldg(off + e));
        gate[s] = __ldg(topk_w + a);
        float v = 0.f;
        for (int j = lane; j < ntiles; j += 32) v += __ldg(dwp + (size_t)qs[s] * ntiles + j);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        dG[s] = v;
        sdot = fmaf(gate[s], v, sdot);
      }
    }
    float dls[KMAX];
#pragma unroll
    for (int s = 0; s < KMAX; ++s)
      if (s < k) dls[s] = gate[s] * (dG[s] - sdot);
    for (int e = lane; e < n; e += 32) {
      float v = 0.f;
#pragma unroll
      for (int s = 0; s < KMAX; ++s)
        if (s < k && es[s] == e) v = dls[s];
      dl[(size_t)t * n + e] = v;
    }
    for (int c = lane; c < d; c += 32) {
      float acc = 0.f;
#pragma unroll
      for (int s = 0; s < KMAX; ++s)
        if (s < k) {
          acc += to_f32(dx_pad[(size_t)qs[s] * d + c]);
          acc = fmaf(dls[s], to_f32(wg[(size_t)c * n + es[s]]), acc);
        }
      dx[(size_t)t * d + c] = from_f32<T>(acc);
    }
  }
}

// part[c][i][e] = sum over the tokens of chunk c of x[t, i] dl[t, e]; column i == d stands
// for the logit bias (x = 1).  Block: 256 columns x one chunk of tokens.
template <typename X>
__global__ void __launch_bounds__(256) dwg_partial_kernel(const X* __restrict__ x,
                                                          const float* __restrict__ dl, int Tn,
                                                          int d, int n,
                                                          float* __restrict__ part) {
  __shared__ float s_dl[kDwgChunk * kMaxExperts];
  const int c = blockIdx.y;
  const int t0 = c * kDwgChunk;
  const int tn = min(kDwgChunk, Tn - t0);
  for (int i = threadIdx.x; i < tn * n; i += blockDim.x) s_dl[i] = dl[(size_t)t0 * n + i];
  __syncthreads();
  const int col = blockIdx.x * blockDim.x + threadIdx.x;
  if (col > d) return;
  float acc[kMaxExperts];
  for (int e = 0; e < n; ++e) acc[e] = 0.f;
  for (int tt = 0; tt < tn; ++tt) {
    const float xv = col < d ? to_f32(x[(size_t)(t0 + tt) * d + col]) : 1.0f;
    for (int e = 0; e < n; ++e) acc[e] = fmaf(xv, s_dl[tt * n + e], acc[e]);
  }
  float* out = part + ((size_t)c * (d + 1) + col) * n;
  for (int e = 0; e < n; ++e) out[e] = acc[e];
}

// n == 8, d % 8 == 0: each thread owns 8 consecutive columns (one 16-byte load of x per
// token) and all 8 experts; the first block of a chunk also sums the chunk's logit gradients
// (the bias column, i == d).
__global__ void __launch_bounds__(128) dwg_partial_n8_kernel(const bf16* __restrict__ x,
                                                             const float* __restrict__ dl, int T,
                                                             int d, float* __restrict__ part) {
  __shared__ float s_dl[kDwgChunk * 8];
  const int c = blockIdx.y;
  const int t0 = c * kDwgChunk;
  const int tn = min(kDwgChunk, T - t0);
  for (int i = threadIdx.x; i < tn * 8; i += blockDim.x) s_dl[i] = dl[(size_t)t0 * 8 + i];
  __syncthreads();
  float* pc = part + (size_t)c * (d + 1) * 8;
  if (blockIdx.x == 0 && threadIdx.x < 8) {
    float v = 0.f;
    for (int tt = 0; tt < tn; ++tt) v += s_dl[tt * 8 + threadIdx.x];
    pc[(size_t)d * 8 + threadIdx.x] = v;
  }
  const int col0 = (blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (col0 >= d) return;
  float acc[8][8];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[j][e] = 0.f;
  // tokens in ascending order; the rows of kDwgBatch tokens are loaded together
  auto step = [&](const uint4& u, int tt) {
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
    float g[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) g[e] = s_dl[tt * 8 + e];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 xf = __bfloat1622float2(p[j]);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        acc[2 * j][e] = fmaf(xf.x, g[e], acc[2 * j][e]);
        acc[2 * j + 1][e] = fmaf(xf.y, g[e], acc[2 * j + 1][e]);
      }
    }
  };
  int tt = 0;
#pragma unroll 1
  for (; tt + kDwgBatch <= tn; tt += kDwgBatch) {
    uint4 u[kDwgBatch];
#pragma unroll
    for (int b = 0; b < kDwgBatch; ++b)
      u[b] = __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + tt + b) * d + col0));
#pragma unroll
    for (int b = 0; b < kDwgBatch; ++b) step(u[b], tt + b);
  }
#pragma unroll 1
  for (; tt < tn; ++tt)
    step(__ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + tt) * d + col0)), tt);
  float4* out = reinterpret_cast<float4*>(pc + (size_t)col0 * 8);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    out[2 * j] = make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
    out[2 * j + 1] = make_float4(acc[j][4], acc[j][5], acc[j][6], acc[j][7]);
  }
}

__global__ void __launch_bounds__(256) dwg_reduce_kernel(const float* __restrict__ part,
                                                         int chunks, int d, int n,
                                                         float* __restrict__ dwg,
                                                         float* __restrict__ dbias) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;   // flat (column, expert)
  if (i >= (d + 1) * n) return;
  float v = 0.f;
  for (int c = 0; c < chunks; ++c) v += part[(size_t)c * (d + 1) * n + i];
  if (i < d * n)
    dwg[i] = v;
  else if (dbias)
    dbias[i - d * n] = v;
}

// Block per (expert, padding row): padding rows follow each expert's rows in its segment.
__global__ void __launch_bounds__(256) zero_pad_rows_kernel(uint4* __restrict__ buf,
                                                            const int32_t* __restrict__ off,
                                                            const int32_t* __restrict__ poff,
                                                            int row_vecs) {
  const int e = blockIdx.y, j = blockIdx.x;
  const int row = poff[e] + (off[e + 1] - off[e]) + j;
  if (row >= poff[e + 1]) return;
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (int c = threadIdx.x; c < row_vecs; c += blockDim.x) buf[(size_t)row * row_vecs + c] = z;
}

}  // namespace

cudaError_t launch_zero_pad_rows(bf16* buf, const int32_t* off, const int32_t* poff, int n,
                                 int row_elems, cudaStream_t s) {
  dim3 grid(kRowAlign - 1, n);
  zero_pad_rows_kernel<<<grid, 256, 0, s>>>((uint4*)buf, off, poff, row_elems / 8);
  return cudaGetLastError();
}

int bwd_rows_max(long long A, int n) {
  const long long r = A + (long long)(kRowAlign - 1) * n;
  return (int)((r + kRowAlign - 1) / kRowAlign * kRowAlign);
}

int bwd_dwg_chunks(int T) { return (T + kDwgChunk - 1) / kDwgChunk; }

cudaError_t launch_pad_offsets(const int32_t* off, int n, int32_t* poff, cudaStream_t s) {
  pad_offsets_kernel<<<1, 32, 0, s>>>(off, n, poff);
  return cudaGetLastError();
}

cudaError_t launch_gather_bwd(const void* x, const void* dy, const int32_t* off,
                              const int32_t* poff, const int32_t* perm, const float* topk_w,
                              int n, int k, int rows_max, size_t row_bytes, void* x_pad,
                              void* g_pad, float* wq, cudaStream_t s) {
  if (rows_max == 0) return cudaSuccess;
  const int cap = device_sm_count() * 8;
  const int grid = rows_max < cap ? rows_max : cap;
  if (row_bytes % 16 == 0)
    gather_bwd_kernel<uint4><<<grid, 256, 0, s>>>(
        (const uint4*)x, (const uint4*)dy, off, poff, perm, topk_w, n, k, rows_max,
        (int)(row_bytes / 16), (uint4*)x_pad, (uint4*)g_pad, wq);
  else if (row_bytes % 4 == 0)
    gather_bwd_kernel<uint32_t><<<grid, 256, 0, s>>>(
        (const uint32_t*)x, (const uint32_t*)dy, off, poff, perm, topk_w, n, k, rows_max,
        (int)(row_bytes / 4), (uint32_t*)x_pad, (uint32_t*)g_pad, wq);
  else
    gather_bwd_kernel<uint16_t><<<grid, 256, 0, s>>>(
        (const uint16_t*)x, (const uint16_t*)dy, off, poff, perm, topk_w, n, k, rows_max,
        (int)(row_bytes / 2), (uint16_t*)x_pad, (uint16_t*)g_pad, wq);
  return cudaGetLastError();
}

cudaError_t launch_router_bwd(const int32_t* idx, const float* topk_w, const int32_t* off,
                              const int32_t* poff, const int32_t* inv_perm, const float* dwp,
                              int ntiles, const void* dx_pad_v, const void* wg_v, int T, int d,
                              int n, int k, int dtype, void* dx_v, float* dl, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const long long blocks = ((long long)T + 7) / 8;
  const long long cap = (long long)device_sm_count() * 16;
  const int grid = (int)(blocks < cap ? blocks : cap);
  if (dtype != MOE_BF16 || d % 8 != 0) {
    if (dtype == MOE_BF16) {
      if (k <= 2)
        router_bwd_generic_kernel<bf16, 2><<<grid, 256, 0, s>>>(
            idx, topk_w, off, poff, inv_perm, dwp, ntiles, (const bf16*)dx_pad_v,
            (const bf16*)wg_v, T, d, n, k, (bf16*)dx_v, dl);
      else
        router_bwd_generic_kernel<bf16, kMaxExperts><<<grid, 256, 0, s>>>(
            idx, topk_w, off, poff, inv_perm, dwp, ntiles, (const bf16*)dx_pad_v,
            (const bf16*)wg_v, T, d, n, k, (bf16*)dx_v, dl);
    } else {
      if (k <= 2)
        router_bwd_generic_kernel<float, 2><<<grid, 256, 0, s>>>(
            idx, topk_w, off, poff, inv_perm, dwp, ntiles, (const float*)dx_pad_v,
            (const float*)wg_v, T, d, n, k, (float*)dx_v, dl);
      else
        router_bwd_generic_kernel<float, kMaxExperts><<<grid, 256, 0, s>>>(
            idx, topk_w, off, poff, inv_perm, dwp, ntiles, (const float*)dx_pad_v,
            (const float*)wg_v, T, d, n, k, (float*)dx_v, dl);
    }
    return cudaGetLastError();
  }
  const bf16* dx_pad = (const bf16*)dx_pad_v;
  const bf16* wg = (const bf16*)wg_v;
  bf16* dx = (bf16*)dx_v;
  if (n == 8) {
    // four warps per block, so that small batches still spread over the SMs
    const long long nb = ((long long)T + 4 * kRbTpw - 1) / (4 * kRbTpw);
    const int g8 = (int)(nb < cap ? nb : cap);
    if (k <= 2)
      router_bwd_n8_kernel<2><<<g8, 128, 0, s>>>(idx, topk_w, off, poff, inv_perm, dwp, ntiles,
                                                dx_pad, wg, T, d, k, dx, dl);
    else
      router_bwd_n8_kernel<8><<<g8, 128, 0, s>>>(idx, topk_w, off, poff, inv_perm, dwp, ntiles,
                                                dx_pad, wg, T, d, k, dx, dl);
    return cudaGetLastError();
  }
  if (k <= 2)
    router_bwd_kernel<2><<<grid, 256, 0, s>>>(idx, topk_w, off, poff, inv_perm, dwp, ntiles,
                                              dx_pad, wg, T, d, n, k, dx, dl);
  else if (k <= 8)
    router_bwd_kernel<8><<<grid, 256, 0, s>>>(idx, topk_w, off, poff, inv_perm, dwp, ntiles,
                                              dx_pad, wg, T, d, n, k, dx, dl);
  else
    router_bwd_kernel<kMaxExperts><<<grid, 256, 0, s>>>(idx, topk_w, off, poff, inv_perm, dwp,
                                                        ntiles, dx_pad, wg, T, d, n, k, dx, dl);
  return cudaGetLastError();
}

cudaError_t launch_dwg(const void* x, const float* dl, int T, int d, int n, int dtype,
                       float* part, float* dwg, float* dbias, cudaStream_t s) {
  const int chunks = bwd_dwg_chunks(T);
  if (chunks > 0) {
    if (dtype == MOE_BF16 && n == 8 && d % 8 == 0) {
      dim3 grid((d / 8 + 127) / 128, chunks);
      dwg_partial_n8_kernel<<<grid, 128, 0, s>>>((const bf16*)x, dl, T, d, part);
    } else if (dtype == MOE_BF16) {
      dim3 grid((d + 1 + 255) / 256, chunks);
      dwg_partial_kernel<bf16><<<grid, 256, 0, s>>>((const bf16*)x, dl, T, d, n, part);
    } else {
      dim3 grid((d + 1 + 255) / 256, chunks);
      dwg_partial_kernel<float><<<grid, 256, 0, s>>>((const float*)x, dl, T, d, n, part);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int outs = (d + 1) * n;
  dwg_reduce_kernel<<<(outs + 255) / 256, 256, 0, s>>>(part, chunks, d, n, dwg, dbias);
  return cudaGetLastError();
}

}  // namespace moe
