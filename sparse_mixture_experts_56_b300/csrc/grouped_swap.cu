// Experts for small token batches (decode) on the 5th-generation tensor cores, with the
// operands swapped so that the weights fill the 128-row side of every MMA:
//   GEMM1ᵀ  aᵀ = w1_e · X_eᵀ,  bᵀ = w3_e · X_eᵀ,   h = SiLU(a) ⊙ b        (SwiGLU fused)
//   GEMM2ᵀ  y_permᵀ = w2_e · h_eᵀ
// for the rows p in [offsets[e], offsets[e+1]) of every expert e ("Mixtral of Experts"
// (xyznot.com summary), Método: each expert is a SwiGLU network of intermediate size 14336;
// ja.news.hada.io, 実装と推論効率: experts receive variable numbers of tokens).
//
// Why a second form: with a few tokens per expert the layer streams its weights from HBM, and
// the rate at which one SM streams is the bytes it keeps in flight divided by the memory
// latency.  In the token-rows-as-M form every stage also carries a 128-row token tile (16 KB,
// mostly rows of other experts) and an M=128 N=256 MMA; here a stage carries 32 KB of weights
// and only the expert's token rows (16-64 rows: 2-8 KB), the MMAs are M=128 N=16..64, and
// 5-6 stages fit in shared memory, so 160-192 KB of weights are in flight per SM instead of
// 128 KB.
//
// Design (persistent, one CTA per SM, 256 threads, warp-specialised):
//   warp 0      TMA producer: per stage two weight boxes [128 rows x 64 K] (GEMM1: the same
//               128 rows of w1_e and w3_e; GEMM2: rows r and r + 128 of w2_e) and the token
//               block, one box [NB rows x 64 K]; 128-byte swizzle.
//   warp 1      MMA issuer: tcgen05.mma.kind::f16 M=128 N=NB K=16, two per K slice (one per
//               weight box) into the tile's two accumulators; two tiles' accumulators in
//               TMEM (4 x 64 columns).
//   warp 2      allocates / frees the 256 TMEM columns.
//   warps 4-7   epilogue: tcgen05.ld 32x32b (TMEM lane = weight row), then GEMM1:
//               h[p, f0 + lane] = SiLU(a) b;  GEMM2: y_perm[p, d0 + lane] (and + 128).  For a
//               fixed token the 32 lanes of a warp write 32 consecutive columns.
// Work list: tiles (expert, token block of NB rows, weight tile) from expert_offsets on the
// device; an expert with more than NB rows takes several token blocks (each re-reads the
// expert's weights, so the launcher picks NB >= the tokens of the batch, which bounds the
// rows of any expert).  Balanced static schedule as in the token-rows-as-M form.
//
// Every wait is bounded (globaltimer).  A wait that runs past the limit raises the CTA's abort
// flag and sets the timeout bit of the device status word; every role then stops, the
// producer waits (bounded) for its copies in flight, the MMA warp for its MMAs, and the TMEM
// columns are freed before the CTA exits.
#include <cuda.h>

#include <atomic>

#include "moe_internal.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace ptx;

constexpr int kWRows = 128;                          // weight rows per MMA (TMEM lanes)
constexpr int kBK = 64;                              // K per stage (one swizzle atom of bf16)
constexpr int kUmmaK = 16;
constexpr uint32_t kWBytes = kWRows * kBK * 2;       // one weight box: 16 KB
constexpr int kMaxNB = 64;                           // token rows per block (MMA N), at most
constexpr int kMaxStages = 8;
constexpr uint32_t kTmemCols = 256;                  // 2 tiles x 2 accumulators x 64 columns
constexpr uint64_t kDrainNs = 200ull * 1000 * 1000;
constexpr size_t kSmemLimit = 232448;                // opt-in shared memory per block (227 KB)

enum SwapMode { kUp = 0, kDown = 1 };

struct SwapArgs {
  const int32_t* offsets;  // rows of each expert: [offsets[e], offsets[e+1])
  int mrows;               // rows of X; offsets are clamped into [0, mrows]
  int n;
  int kdim;                // reduction length: d (GEMM1) or f (GEMM2)
  int wrows;               // weight rows of one expert in the 2-D weight view: f or d
  int wstep;               // weight rows per tile: 128 (GEMM1) or 256 (GEMM2)
  int wt;                  // weight tiles per expert
  int nb;                  // token rows per block = MMA N (16, 32, 48 or 64)
  int stages;
  uint32_t stage_bytes;
  bf16* out;               // h [mrows, f] or y_perm [mrows, d]
  int ocols;               // columns of out
  uint32_t* status;
  unsigned long long wait_ns;
};

struct SwapShared {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int total;
  int tile_base[kMaxExperts + 1];
  int off[kMaxExperts + 1];
};

// stage layout: weight box 0 | weight box 1 | token block (all 1024-byte aligned)
__host__ __device__ constexpr uint32_t stage_bytes_for(int nb) {
  return 2 * kWBytes + (uint32_t)nb * kBK * 2;
}
__host__ __device__ constexpr size_t swap_smem_bytes(int stages, int nb) {
  return 1024 + (size_t)stages * stage_bytes_for(nb) + sizeof(SwapShared);
}

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B bf16 (7-9, 10-12 = 1),
// both K-major, N >> 3 at bits 17-22, M >> 4 at bits 24-28.
__device__ __forceinline__ uint32_t swap_idesc(int nb) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(nb >> 3) << 17) |
         ((uint32_t)(kWRows >> 4) << 24);
}

__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane, and the wait for them.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait16(uint32_t (&a)[16], uint32_t (&b)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]),
                 "+r"(a[6]), "+r"(a[7]), "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]),
                 "+r"(a[12]), "+r"(a[13]), "+r"(a[14]), "+r"(a[15]), "+r"(b[0]), "+r"(b[1]),
                 "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]), "+r"(b[7]),
                 "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]),
                 "+r"(b[14]), "+r"(b[15])::"memory");
}

// the four epilogue warps' barrier, returning whether `ok` holds in all of them
__device__ __forceinline__ int epilogue_all(int ok) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.and.pred p, 1, 128, q;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"(ok)
      : "memory");
  return (int)r;
}

struct SwapTile {
  int e, w;
  int row0;   // first token row of the block
  int rows;   // token rows of the block (<= nb)
};

__device__ __forceinline__ SwapTile decode_swap(const SwapShared& sh, int n, int wt, int nb,
                                                int tile) {
  int e = 0;
  while (e + 1 < n && sh.tile_base[e + 1] <= tile) ++e;
  const int u = tile - sh.tile_base[e];
  const int tb = u / wt;
  SwapTile t;
  t.e = e;
  t.w = u - tb * wt;
  t.row0 = sh.off[e] + tb * nb;
  t.rows = min(nb, sh.off[e + 1] - t.row0);
  return t;
}

__device__ __forceinline__ float silu_(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

template <int MODE>
__global__ void __launch_bounds__(256, 1)
    grouped_gemm_swap_kernel(const __grid_constant__ CUtensorMap tmW0,
                             const __grid_constant__ CUtensorMap tmW1,
                             const __grid_constant__ CUtensorMap tmX, const SwapArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int S = args.stages;
  const uint32_t SB = args.stage_bytes;
  SwapShared& sh = *reinterpret_cast<SwapShared*>(smem + (size_t)S * SB);
  volatile int* abort = &sh.abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = args.n, NB = args.nb, WT = args.wt;
  const int KB = args.kdim / kBK;

  if (threadIdx.x == 0) {
    // offsets made monotone inside [0, mrows], so that no block reaches past the buffers
    // whatever the device-side offsets hold
    auto clamp_off = [&](int v, int lo) { return v < lo ? lo : (v > args.mrows ? args.mrows : v); };
    int acc = 0;
    int o0 = clamp_off(args.offsets[0], 0);
    for (int e = 0; e < n; ++e) {
      const int o1 = clamp_off(args.offsets[e + 1], o0);
      sh.off[e] = o0;
      sh.tile_base[e] = acc;
      acc += ((o1 - o0 + NB - 1) / NB) * WT;
      o0 = o1;
    }
    sh.off[n] = o0;
    sh.tile_base[n] = acc;
    sh.total = acc;
    sh.abort = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&sh.full[s]), 1);
      mbar_init(smem_u32(&sh.empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&sh.tfull[a]), 1);
      mbar_init(smem_u32(&sh.tempty[a]), 4);   // the four epilogue warps
    }
    mbar_init(smem_u32(&sh.drain), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 2) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&sh.tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sh.tmem_base;
  const int total = sh.total;
  const uint64_t limit = args.wait_ns;
  // balanced static schedule: the fewest CTAs that still finish in the same number of rounds
  const int units = (int)gridDim.x;
  const int rounds = (total + units - 1) / units;
  const int gstride = rounds > 0 ? (total + rounds - 1) / rounds : units;
  const int first_tile = (int)blockIdx.x < gstride ? (int)blockIdx.x : total;
  const uint32_t tx_bytes = 2 * kWBytes + (uint32_t)NB * kBK * 2;

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer
    prefetch_map(&tmW0);
    if (MODE == kUp) prefetch_map(&tmW1);
    prefetch_map(&tmX);
    int stage = 0;
    uint32_t phase = 0, issued = 0, iphase = 0;
    bool ok = true;
    for (int tile = first_tile; ok && tile < total; tile += gstride) {
      const SwapTile t = decode_swap(sh, n, WT, NB, tile);
      const int wrow = t.e * args.wrows + t.w * args.wstep;
      for (int kb = 0; kb < KB; ++kb) {
        if (!wait_fast(smem_u32(&sh.empty[stage]), phase ^ 1u, abort, limit)) {
          raise_abort(abort, args.status);
          ok = false;
          break;
        }
        const uint32_t fb = smem_u32(&sh.full[stage]);
        const uint32_t base = smem_u32(smem + (size_t)stage * SB);
        mbar_expect_tx(fb, tx_bytes);
        tma_load_2d(base, &tmW0, fb, kb * kBK, wrow);
        if (MODE == kUp)   // the same rows of w3
          tma_load_2d(base + kWBytes, &tmW1, fb, kb * kBK, wrow);
        else               // the next 128 rows of w2
          tma_load_2d(base + kWBytes, &tmW0, fb, kb * kBK, wrow + kWRows);
        tma_load_2d(base + 2 * kWBytes, &tmX, fb, kb * kBK, t.row0);
        issued |= 1u << stage;
        iphase = (iphase & ~(1u << stage)) | (phase << stage);
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // every copy issued must have landed before the CTA may exit
    for (int s = 0; s < S; ++s)
      if ((issued >> s) & 1u)
        if (!drain_phase(smem_u32(&sh.full[s]), (iphase >> s) & 1u, kDrainNs))
          atomicOr(args.status, kDevErrTimeout);
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA issuer
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true, any_mma = false;
    const uint32_t idesc = swap_idesc(NB);
    const uint64_t dW0 = sw128_desc(smem_u32(smem));
    const uint64_t dW1 = sw128_desc(smem_u32(smem + kWBytes));
    const uint64_t dX = sw128_desc(smem_u32(smem + 2 * kWBytes));
    for (int tile = first_tile; ok && tile < total; tile += gstride) {
      if (!wait_fast(smem_u32(&sh.tempty[acc]), acc_phase ^ 1u, abort, limit)) {
        raise_abort(abort, args.status);
        break;
      }
      tc_fence_after();
      const uint32_t d0 = tmem_base + (uint32_t)(acc * 2 * kMaxNB);
      const uint32_t d1 = d0 + (uint32_t)kMaxNB;
      for (int kb = 0; kb < KB; ++kb) {
        if (!wait_fast(smem_u32(&sh.full[stage]), phase, abort, limit)) {
          raise_abort(abort, args.status);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t so = (uint32_t)stage * SB;
#pragma unroll
        for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
          const uint32_t ko = so + (uint32_t)kk * kUmmaK * 2;
          const uint32_t accum = (kb | kk) != 0 ? 1u : 0u;
          umma_f16(d0, desc_add(dW0, ko), desc_add(dX, ko), idesc, accum);
          umma_f16(d1, desc_add(dW1, ko), desc_add(dX, ko), idesc, accum);
        }
        any_mma = true;
        umma_commit(smem_u32(&sh.empty[stage]));
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      umma_commit(smem_u32(&sh.tfull[acc]));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // all MMAs issued by this thread must finish before the TMEM columns are freed
    if (any_mma) {
      umma_commit(smem_u32(&sh.drain));
      if (!drain_phase(smem_u32(&sh.drain), 0, kDrainNs)) atomicOr(args.status, kDevErrTimeout);
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- epilogue
    const int q = warp - 4;          // TMEM lane quarter
    const int r = q * 32 + lane;     // weight row of the tile held in this lane
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = first_tile; tile < total; tile += gstride) {
      const SwapTile t = decode_swap(sh, n, WT, NB, tile);
      int ok = 1;
      if (lane == 0) {
        ok = wait_fast(smem_u32(&sh.tfull[acc]), acc_phase, abort, limit) ? 1 : 0;
        if (!ok) raise_abort(abort, args.status);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!epilogue_all(ok)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * 2 * kMaxNB);
      // output columns of this lane: GEMM1 one column of h, GEMM2 two columns of y_perm
      const int col0 = t.w * args.wstep + r;
      const int col1 = col0 + kWRows;
      const bool ok0 = col0 < args.ocols;
      const bool ok1 = MODE == kDown && col1 < args.ocols;
#pragma unroll 1
      for (int c = 0; c < NB / 16; ++c) {
        uint32_t a[16], b[16];
        tmem_ld16(tb + c * 16, a);
        tmem_ld16(tb + kMaxNB + c * 16, b);
        tmem_wait16(a, b);
        if (c == NB / 16 - 1) {   // the accumulators are in registers: hand them back
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&sh.tempty[acc]));
        }
        const int jn = min(16, t.rows - c * 16);   // tokens of this chunk that exist
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          if (j < jn) {
            bf16* orow = args.out + (size_t)(t.row0 + c * 16 + j) * args.ocols;
            const float av = __uint_as_float(a[j]);
            const float bv = __uint_as_float(b[j]);
            if (MODE == kUp) {
              if (ok0) orow[col0] = __float2bfloat16_rn(silu_(av) * bv);
            } else {
              if (ok0) orow[col0] = __float2bfloat16_rn(av);
              if (ok1) orow[col1] = __float2bfloat16_rn(bv);
            }
          }
        }
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------

std::atomic<int> g_swap_form{MOE_TC_FORM_AUTO};

// Stages that fit in shared memory with token blocks of nb rows (6 for 16 or 32 rows, 5 for
// 48 or 64).
int swap_stages(int nb) {
  int s = kMaxStages;
  while (s > 2 && swap_smem_bytes(s, nb) > kSmemLimit) --s;
  return s;
}

template <int MODE>
cudaError_t set_swap_smem_attr() {
  static PerDeviceSetting setting;
  return setting.get([] {
    size_t most = 0;   // the largest layout any block size uses
    for (int nb = 16; nb <= kMaxNB; nb += 16) {
      const size_t b = swap_smem_bytes(swap_stages(nb), nb);
      most = b > most ? b : most;
    }
    return cudaFuncSetAttribute(grouped_gemm_swap_kernel<MODE>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)most);
  });
}

template <int MODE>
cudaError_t launch_swap(const CUtensorMap& mW0, const CUtensorMap& mW1, const CUtensorMap& mX,
                        SwapArgs a, int A, cudaStream_t s) {
  cudaError_t e = set_swap_smem_attr<MODE>();
  if (e != cudaSuccess) return e;
  a.stages = swap_stages(a.nb);
  a.stage_bytes = stage_bytes_for(a.nb);
  const long long tiles = ((long long)(A + a.nb - 1) / a.nb + a.n) * a.wt;
  const int sms = device_sm_count();
  const int grid = (int)(tiles < sms ? (tiles > 0 ? tiles : 1) : sms);
  grouped_gemm_swap_kernel<MODE><<<grid, 256, swap_smem_bytes(a.stages, a.nb), s>>>(mW0, mW1, mX,
                                                                                   a);
  return cudaGetLastError();
}

}  // namespace

void set_swap_form(int form) { g_swap_form.store(form, std::memory_order_relaxed); }

// Token rows per block of the swapped form for a batch of T tokens (no expert of a routed
// batch holds more than T rows: the K experts of a token are distinct), or 0 for the
// token-rows-as-M form.  On B300 at T = 32, d = 4096, f = 14336 the swapped up-projection
// streams its weights at 6.4 TB/s against 6.1 TB/s for the token-rows-as-M form (layer step
// 0.461 against 0.479 ms); above 64 tokens the token-rows-as-M form is used, whose larger
// token tiles suit the tensor-bound sizes.
int swap_rows(int T) {
  const int form = g_swap_form.load(std::memory_order_relaxed);
  if (form == MOE_TC_FORM_SINGLE || form == MOE_TC_FORM_PAIR) return 0;
  if (form == MOE_TC_FORM_AUTO && T > kMaxNB) return 0;
  const int r = (T + 15) / 16 * 16;
  return r < 16 ? 16 : (r > kMaxNB ? kMaxNB : r);
}

cudaError_t launch_up_swap(const bf16* x_perm, const int32_t* offsets, const bf16* w1,
                           const bf16* w3, int A, int d, int f, int n, int nb, bf16* h,
                           uint32_t* status, unsigned long long wait_ns, cudaStream_t s) {
  if (A == 0) return cudaSuccess;
  if (nb < 16 || nb > kMaxNB || nb % 16) return cudaErrorInvalidValue;
  CUtensorMap mW1, mW3, mX;
  if (!make_map(&mW1, w1, (uint64_t)n * f, (uint64_t)d, kWRows) ||
      !make_map(&mW3, w3, (uint64_t)n * f, (uint64_t)d, kWRows) ||
      !make_map(&mX, x_perm, (uint64_t)A, (uint64_t)d, (uint32_t)nb))
    return cudaErrorInvalidValue;
  SwapArgs a = {};
  a.offsets = offsets;
  a.mrows = A;
  a.n = n;
  a.kdim = d;
  a.wrows = f;
  a.wstep = kWRows;
  a.wt = (f + kWRows - 1) / kWRows;
  a.nb = nb;
  a.out = h;
  a.ocols = f;
  a.status = status;
  a.wait_ns = wait_ns;
  return launch_swap<kUp>(mW1, mW3, mX, a, A, s);
}

cudaError_t launch_down_swap(const bf16* h, const int32_t* offsets, const bf16* w2, int A, int d,
                             int f, int n, int nb, bf16* y_perm, uint32_t* status,
                             unsigned long long wait_ns, cudaStream_t s) {
  if (A == 0) return cudaSuccess;
  if (nb < 16 || nb > kMaxNB || nb % 16) return cudaErrorInvalidValue;
  CUtensorMap mW2, mX;
  if (!make_map(&mW2, w2, (uint64_t)n * d, (uint64_t)f, kWRows) ||
      !make_map(&mX, h, (uint64_t)A, (uint64_t)f, (uint32_t)nb))
    return cudaErrorInvalidValue;
  SwapArgs a = {};
  a.offsets = offsets;
  a.mrows = A;
  a.n = n;
  a.kdim = f;
  a.wrows = d;
  a.wstep = 2 * kWRows;
  a.wt = (d + 2 * kWRows - 1) / (2 * kWRows);
  a.nb = nb;
  a.out = y_perm;
  a.ocols = d;
  a.status = status;
  a.wait_ns = wait_ns;
  return launch_swap<kDown>(mW2, mW2, mX, a, A, s);
}

}  // namespace moe
