// Router and gate:  l = x · W_g (+ b);  G(x) = Softmax(TopK(l))
//   "Mixtral of Experts" (xyznot.com summary), Método, eq. G;
//   blog.csdn.net "《Mixtral of Experts》…", MOE数学公式 §2.1 (logits), §2.2 (TopK keeps the K
//   largest logits, the rest become -inf), §2.3 (softmax over the TopK output: only the K
//   kept experts get weight, and those weights sum to 1).
// Also the row-wise RMSNorm used by stacked layers (not part of the pages' layer).
//
// One warp per token (for batches of at most 1024 tokens, one block per token, its 8 warps
// splitting the row).  The token's row of x is read once (16-byte loads); W_g (d x n, 64 KB
// for 4096 x 8 bf16) stays hot in L1/L2.  Products accumulate in fp32 per lane, then a
// butterfly reduction gives every lane all n logits.  Lane 0 selects the top K (ties ->
// lower index, descending order) and normalises exp(l - l_max) over them.
#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace {

template <int NP>
__device__ __forceinline__ void warp_allreduce(float (&acc)[NP]) {
#pragma unroll
  for (int e = 0; e < NP; ++e) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
  }
}

// Top-K selection and softmax over the kept logits; run by one lane.
template <int NP>
__device__ __forceinline__ void select_and_write(const float (&l)[NP], int n, int k,
                                                 int32_t* idx_row, float* w_row) {
  uint32_t taken = 0;
  int sel[kMaxExperts];
  float lmax = 0.f;
  for (int s = 0; s < k; ++s) {
    int best = -1;
    float bv = 0.f;
#pragma unroll
    for (int e = 0; e < NP; ++e) {
      if (e < n && !(taken >> e & 1u)) {
        // strict '>' keeps the lower index on equal logits
        if (best < 0 || l[e] > bv) {
          best = e;
          bv = l[e];
        }
      }
    }
    taken |= 1u << best;
    sel[s] = best;
    if (s == 0) lmax = bv;
  }
  float sum = 0.f;
  float ex[kMaxExperts];
  for (int s = 0; s < k; ++s) {
    float v = 0.f;
#pragma unroll
    for (int e = 0; e < NP; ++e)
      if (e == sel[s]) v = l[e];
    ex[s] = expf(v - lmax);
    sum += ex[s];
  }
  for (int s = 0; s < k; ++s) {
    idx_row[s] = sel[s];
    w_row[s] = ex[s] / sum;
  }
}

// Generic path: any d, any n <= NP, fp32 or bf16 storage.
template <typename T, int NP>
__global__ void __launch_bounds__(256) router_generic_kernel(const T* __restrict__ x,
                                                             const T* __restrict__ wg,
                                                             const float* __restrict__ bias, int Tn,
                                                             int d, int n, int k,
                                                             int32_t* __restrict__ idx,
                                                             float* __restrict__ w,
                                                             float* __restrict__ logits) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < Tn; t += warps) {
    float acc[NP];
#pragma unroll
    for (int e = 0; e < NP; ++e) acc[e] = 0.f;
    const T* xr = x + (size_t)t * d;
    for (int i = lane; i < d; i += 32) {
      const float xv = to_f32(xr[i]);
      const T* wr = wg + (size_t)i * n;
#pragma unroll
      for (int e = 0; e < NP; ++e)
        if (e < n) acc[e] = fmaf(xv, to_f32(wr[e]), acc[e]);
    }
    warp_allreduce<NP>(acc);
    if (bias) {
#pragma unroll
      for (int e = 0; e < NP; ++e)
        if (e < n) acc[e] += bias[e];
    }
    if (logits && lane < n) {
      float v = 0.f;
#pragma unroll
      for (int e = 0; e < NP; ++e)
        if (e == lane) v = acc[e];
      logits[(size_t)t * n + lane] = v;
    }
    if (lane == 0) select_and_write<NP>(acc, n, k, idx + (size_t)t * k, w + (size_t)t * k);
  }
}

// Fast path: bf16, n == 8, d % 256 == 0.  Each lane owns 8 consecutive elements of x per
// 256-element slab: eight 16-byte loads of the matching W_g rows, reused for the TPW tokens
// the warp handles at once, and one 16-byte load of x per token.  Every lane accumulates its
// elements in the same order whatever TPW is, so the logits do not depend on it.
template <int TPW>
__global__ void __launch_bounds__(256) router_bf16_n8_kernel(const bf16* __restrict__ x,
                                                             const bf16* __restrict__ wg,
                                                             const float* __restrict__ bias,
                                                             int Tn, int d, int k,
                                                             int32_t* __restrict__ idx,
                                                             float* __restrict__ w,
                                                             float* __restrict__ logits) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int t0 = ((blockIdx.x * blockDim.x + threadIdx.x) >> 5) * TPW; t0 < Tn;
       t0 += warps * TPW) {
    float acc[TPW][8];
#pragma unroll
    for (int j = 0; j < TPW; ++j)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[j][e] = 0.f;
    for (int i0 = lane * 8; i0 < d; i0 += 256) {
      const uint4* wr = reinterpret_cast<const uint4*>(wg + (size_t)i0 * 8);
      uint4 wv[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) wv[r] = __ldg(wr + r);
#pragma unroll
      for (int j = 0; j < TPW; ++j) {
        if (t0 + j < Tn) {
          const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + j) * d + i0));
          const __nv_bfloat162* xp = reinterpret_cast<const __nv_bfloat162*>(&xv);
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            const float2 xf = __bfloat1622float2(xp[r >> 1]);
            const float xs = (r & 1) ? xf.y : xf.x;
            const __nv_bfloat162* wp = reinterpret_cast<const __nv_bfloat162*>(&wv[r]);
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
              const float2 wf = __bfloat1622float2(wp[e2]);
              acc[j][2 * e2] = fmaf(xs, wf.x, acc[j][2 * e2]);
              acc[j][2 * e2 + 1] = fmaf(xs, wf.y, acc[j][2 * e2 + 1]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < TPW; ++j) {
      const int t = t0 + j;
      if (t >= Tn) break;
      warp_allreduce<8>(acc[j]);
      if (bias) {
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[j][e] += bias[e];
      }
      if (logits && lane < 8) {
        float v = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (e == lane) v = acc[j][e];
        logits[(size_t)t * 8 + lane] = v;
      }
      if (lane == 0) select_and_write<8>(acc[j], 8, k, idx + (size_t)t * k, w + (size_t)t * k);
    }
  }
}

// Large batches: W_g (d x 8 bf16, 64 KB at d = 4096) is staged in shared memory once per
// block, so the only global loads in the loop are the rows of x.  Four tokens per warp share
// each read of W_g from shared memory and its conversion to fp32, and the eight products of
// an element go through four packed two-wide fp32 FMAs (each half rounded as fmaf).  Each
// lane accumulates its elements in the same order as the kernel above, so the logits are
// identical.
constexpr int kRouterSmemTPW = 4;

// acc = (xs, xs) * (w_lo, w_hi) + acc, one packed fp32 FMA; w2 holds two bf16 (lo, hi)
__device__ __forceinline__ void fma2_bf16(uint64_t& acc, float xs, uint32_t w2) {
  const float wlo = __uint_as_float(w2 << 16), whi = __uint_as_float(w2 & 0xffff0000u);
  asm("{\n .reg .b64 a, b;\n mov.b64 a, {%1, %1};\n mov.b64 b, {%2, %3};\n"
      " fma.rn.f32x2 %0, a, b, %0;\n}\n"
      : "+l"(acc)
      : "f"(xs), "f"(wlo), "f"(whi));
}

__global__ void __launch_bounds__(256, 2) router_bf16_n8_smem_kernel(const bf16* __restrict__ x,
                                                                  const bf16* __restrict__ wg,
                                                                  const float* __restrict__ bias,
                                                                  int Tn, int d, int k,
                                                                  int32_t* __restrict__ idx,
                                                                  float* __restrict__ w,
                                                                  float* __restrict__ logits) {
  // d rows of 8 bf16; row i sits in slot 8*(i/8) + ((i%8) ^ ((i/8)%8)), so that the eight
  // lanes reading rows 8L + r (same r, consecutive L) hit eight different bank groups
  extern __shared__ uint4 s_wg[];
#pragma unroll 8
  for (int i = threadIdx.x; i < d; i += blockDim.x)
    s_wg[(i & ~7) | ((i ^ (i >> 3)) & 7)] = __ldg(reinterpret_cast<const uint4*>(wg) + i);
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  constexpr int TPW = kRouterSmemTPW;
  for (int t0 = ((blockIdx.x * blockDim.x + threadIdx.x) >> 5) * TPW; t0 < Tn;
       t0 += warps * TPW) {
    uint64_t acc2[TPW][4];   // experts (2e, 2e + 1) of token t0 + j in acc2[j][e]
#pragma unroll
    for (int j = 0; j < TPW; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc2[j][e] = 0ull;
    const int nt = Tn - t0 < TPW ? Tn - t0 : TPW;
#pragma unroll 2
    for (int i0 = lane * 8; i0 < d; i0 += 256) {
      uint4 xv[TPW];
#pragma unroll
      for (int j = 0; j < TPW; ++j)
        xv[j] = j < nt ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + j) * d + i0))
                       : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const uint4 wr = s_wg[i0 | ((r ^ (i0 >> 3)) & 7)];
        const uint32_t wq[4] = {wr.x, wr.y, wr.z, wr.w};
#pragma unroll
        for (int j = 0; j < TPW; ++j) {
          const uint32_t xw = (&xv[j].x)[r >> 1];
          const float xs = __uint_as_float((r & 1) ? (xw & 0xffff0000u) : (xw << 16));
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) fma2_bf16(acc2[j][e2], xs, wq[e2]);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < TPW; ++j) {
      const int t = t0 + j;
      if (t >= Tn) break;
      float acc[8];
#pragma unroll
      for (int e2 = 0; e2 < 4; ++e2) {
        acc[2 * e2] = __uint_as_float((uint32_t)acc2[j][e2]);
        acc[2 * e2 + 1] = __uint_as_float((uint32_t)(acc2[j][e2] >> 32));
      }
      warp_allreduce<8>(acc);
      if (bias) {
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] += bias[e];
      }
      if (logits && lane < 8) {
        float v = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (e == lane) v = acc[e];
        logits[(size_t)t * 8 + lane] = v;
      }
      if (lane == 0) select_and_write<8>(acc, 8, k, idx + (size_t)t * k, w + (size_t)t * k);
    }
  }
}

// Small batches (too few tokens to fill the GPU with one warp each): one block per token.
// The 8 warps split the row of x into 2048-element slabs, reduce within the warp, and meet
// in shared memory; warp 0 adds the 8 partial sums per expert in a fixed order.
__global__ void __launch_bounds__(256) router_bf16_n8_block_kernel(const bf16* __restrict__ x,
                                                                   const bf16* __restrict__ wg,
                                                                   const float* __restrict__ bias,
                                                                   int Tn, int d, int k,
                                                                   int32_t* __restrict__ idx,
                                                                   float* __restrict__ w,
                                                                   float* __restrict__ logits) {
  __shared__ float part[8][8];  // [warp][expert]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int t = blockIdx.x; t < Tn; t += gridDim.x) {
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * d);
#pragma unroll 2
    for (int i0 = threadIdx.x * 8; i0 < d; i0 += 2048) {
      const uint4 xv = __ldg(xr + (i0 >> 3));
      const __nv_bfloat162* xp = reinterpret_cast<const __nv_bfloat162*>(&xv);
      const uint4* wr = reinterpret_cast<const uint4*>(wg + (size_t)i0 * 8);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float2 xf = __bfloat1622float2(xp[j >> 1]);
        const float xs = (j & 1) ? xf.y : xf.x;
        const uint4 wv = __ldg(wr + j);
        const __nv_bfloat162* wp = reinterpret_cast<const __nv_bfloat162*>(&wv);
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) {
          const float2 wf = __bfloat1622float2(wp[e2]);
          acc[2 * e2] = fmaf(xs, wf.x, acc[2 * e2]);
          acc[2 * e2 + 1] = fmaf(xs, wf.y, acc[2 * e2 + 1]);
        }
      }
    }
    warp_allreduce<8>(acc);
    if (lane == 0) {
#pragma unroll
      for (int e = 0; e < 8; ++e) part[warp][e] = acc[e];
    }
    __syncthreads();
    if (warp == 0) {
      float l[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float v = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) v += part[q][e];
        l[e] = bias ? v + bias[e] : v;
      }
      if (logits && lane < 8) {
        float v = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (e == lane) v = l[e];
        logits[(size_t)t * 8 + lane] = v;
      }
      if (lane == 0) select_and_write<8>(l, 8, k, idx + (size_t)t * k, w + (size_t)t * k);
    }
    __syncthreads();
  }
}

template <typename T>
__global__ void __launch_bounds__(256) rmsnorm_kernel(const T* __restrict__ h, int Tn, int d,
                                                      float eps, T* __restrict__ x) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < Tn; t += warps) {
    const T* hr = h + (size_t)t * d;
    float ss = 0.f;
    for (int i = lane; i < d; i += 32) {
      const float v = to_f32(hr[i]);
      ss = fmaf(v, v, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = 1.0f / sqrtf(ss / (float)d + eps);
    T* xr = x + (size_t)t * d;
    for (int i = lane; i < d; i += 32) xr[i] = from_f32<T>(to_f32(hr[i]) * inv);
  }
}

// bf16 rows with d % 256 == 0: 16-byte loads, the row kept in registers between passes.
__global__ void __launch_bounds__(256) rmsnorm_bf16_vec_kernel(const bf16* __restrict__ h, int Tn,
                                                               int d, float eps,
                                                               bf16* __restrict__ x) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < Tn; t += warps) {
    const uint4* hr = reinterpret_cast<const uint4*>(h + (size_t)t * d);
    uint4* xr = reinterpret_cast<uint4*>(x + (size_t)t * d);
    float ss = 0.f;
    for (int c = lane; c < (d >> 3); c += 32) {
      const uint4 v = __ldg(hr + c);
      const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(p[j]);
        ss = fmaf(f.x, f.x, ss);
        ss = fmaf(f.y, f.y, ss);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = 1.0f / sqrtf(ss / (float)d + eps);
    for (int c = lane; c < (d >> 3); c += 32) {
      const uint4 v = __ldg(hr + c);
      const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
      uint4 o;
      __nv_bfloat162* q = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(p[j]);
        q[j] = __floats2bfloat162_rn(f.x * inv, f.y * inv);
      }
      xr[c] = o;
    }
  }
}

// Up to this many tokens the router gives each token a whole block (8 warps over d).
constexpr int kRouterBlockPerTokenMax = 1024;

// W_g rows staged in shared memory up to this d (16 bytes per row of 8 bf16).
constexpr int kRouterSmemMaxD = 12288;

cudaError_t router_smem_ready() {
  static PerDeviceSetting setting;
  return setting.get([] {
    return cudaFuncSetAttribute(router_bf16_n8_smem_kernel,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kRouterSmemMaxD * 16);
  });
}

int grid_for_warps(long long warps_needed) {
  const long long blocks = (warps_needed + 7) / 8;
  const long long cap = (long long)device_sm_count() * 16;
  return (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace

cudaError_t launch_router_topk(const void* x, const void* wg, const float* bias, int T, int d, int n,
                               int k, int dtype, int32_t* idx, float* w, float* logits,
                               cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int grid = grid_for_warps(T);
  if (dtype == MOE_BF16 && n == 8 && d % 256 == 0 && T <= kRouterBlockPerTokenMax) {
    router_bf16_n8_block_kernel<<<T, 256, 0, s>>>((const bf16*)x, (const bf16*)wg, bias, T, d, k,
                                                   idx, w, logits);
  } else if (dtype == MOE_BF16 && n == 8 && d % 256 == 0 && d <= kRouterSmemMaxD &&
             router_smem_ready() == cudaSuccess) {
    const long long warps_needed = (T + kRouterSmemTPW - 1) / kRouterSmemTPW;
    long long blocks = (warps_needed + 7) / 8;
    const long long cap = (long long)device_sm_count() * 2;   // two blocks fit per SM
    if (blocks > cap) blocks = cap;
    router_bf16_n8_smem_kernel<<<(int)blocks, 256, (size_t)d * 16, s>>>(
        (const bf16*)x, (const bf16*)wg, bias, T, d, k, idx, w, logits);
  } else if (dtype == MOE_BF16 && n == 8 && d % 256 == 0) {
    // four tokens per warp share each W_g load
    router_bf16_n8_kernel<4><<<grid_for_warps((T + 3) / 4), 256, 0, s>>>(
        (const bf16*)x, (const bf16*)wg, bias, T, d, k, idx, w, logits);
  } else if (dtype == MOE_BF16) {
    if (n <= 8)
      router_generic_kernel<bf16, 8><<<grid, 256, 0, s>>>((const bf16*)x, (const bf16*)wg, bias, T,
                                                          d, n, k, idx, w, logits);
    else
      router_generic_kernel<bf16, 32><<<grid, 256, 0, s>>>((const bf16*)x, (const bf16*)wg, bias, T,
                                                           d, n, k, idx, w, logits);
  } else {
    if (n <= 8)
      router_generic_kernel<float, 8><<<grid, 256, 0, s>>>((const float*)x, (const float*)wg, bias,
                                                           T, d, n, k, idx, w, logits);
    else
      router_generic_kernel<float, 32><<<grid, 256, 0, s>>>((const float*)x, (const float*)wg, bias,
                                                            T, d, n, k, idx, w, logits);
  }
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const void* h, int T, int d, float eps, int dtype, void* x, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int grid = grid_for_warps(T);
  if (dtype == MOE_BF16 && d % 256 == 0)
    rmsnorm_bf16_vec_kernel<<<grid, 256, 0, s>>>((const bf16*)h, T, d, eps, (bf16*)x);
  else if (dtype == MOE_BF16)
    rmsnorm_kernel<bf16><<<grid, 256, 0, s>>>((const bf16*)h, T, d, eps, (bf16*)x);
  else
    rmsnorm_kernel<float><<<grid, 256, 0, s>>>((const float*)h, T, d, eps, (float*)x);
  return cudaGetLastError();
}

}  // namespace moe
