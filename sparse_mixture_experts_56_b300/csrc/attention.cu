// Causal grouped-query attention on the tensor cores (the attention sub-block of each decoder
// layer: "Mixtral of Experts" (xyznot.com summary), Método: 32 attention heads and 8 key-value
// heads at hidden size 4096, so head dimension 128; newsflash.city digest: the full dense 32k
// context, no sliding window).  For query head h, key-value head g = h / (Hq / Hkv) and
// query i of a sequence:
//     o_i = sum_{j <= i} softmax_j(q_i · k_j / sqrt(128)) v_j
//
// One CTA per (sequence, query head, block of 128 queries), 256 threads, warp-specialised:
//   warp 0      TMA producer: the Q tile once, then K and V tiles of 128 keys into a
//               two-stage ring (K-major K tile; V as MN-major B operand).
//   warp 1      MMA issuer: S = Q Kᵀ (M=N=K=128) into one of two TMEM score buffers, issued
//               one block ahead, and O += P V (V MN-major) into the TMEM output accumulator.
//   warp 2      allocates / frees the 512 TMEM columns (S0, S1, O).
//   warps 4-7   softmax, one query row per thread: scores from TMEM, causal / sequence mask,
//               online maximum and sum in fp32 (exp2 of log2e-scaled scores), O rescaled in
//               TMEM when the maximum grows, P written as bf16 into shared memory (128-byte
//               swizzle, the A operand of P V); finally O / l stored as bf16.
// Every wait is bounded (globaltimer) as in the expert GEMMs; a timeout sets the status bit,
// every role stops, the MMAs in flight are drained and TMEM is freed.
#include "moe_internal.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace ptx;

constexpr int kDh = 128;                         // head dimension
constexpr int kBlk = 128;                        // queries per CTA = keys per block
constexpr uint32_t kTile = 128 * 128 * 2;        // one 128 x 128 bf16 tile (32 KB)
constexpr uint32_t kHalf = kTile / 2;            // a 128 x 64 (or 64 x 128) half tile
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;                  // S0 at 0, S1 at 128, O at 256
constexpr uint64_t kAttnDrainNs = 200ull * 1000 * 1000;

// kind::f16, bf16 inputs, fp32 accumulation, M = N = 128; P V takes V MN-major (bit 16)
constexpr uint32_t kIdescQK =
    (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kIdescPV = kIdescQK | (1u << 16);

struct AttnArgs {
  int T, seq_len, nseq, nqb, hq, hkv;
  float scale_log2;      // log2(e) / sqrt(dh)
  bf16* out;             // [T, hq, dh]
  uint32_t* status;
  unsigned long long wait_ns;
};

struct AttnShared {
  uint64_t q_full;
  uint64_t kv_full[2], kv_empty[2];
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full, o_done, drain;
  uint32_t tmem_base;
  int abort;
};

// shared memory: Q | K0 | V0 | K1 | V1 | P0 | P1 | AttnShared, 1024-byte aligned tiles
constexpr size_t kAttnSmem = 1024 + 7 * (size_t)kTile + sizeof(AttnShared);
// The running maximum used as the exponent's offset is raised only when a block's maximum
// exceeds it by more than this (log2 units): P stays below 2^8, and most blocks skip the
// rescaling of O.
constexpr float kRescaleLog2 = 8.0f;

__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
// 32 consecutive fp32 columns of this thread's TMEM lane, written back
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
      "%29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// A lane of the softmax warps waits on `bar` for the warp (lane 0 polls); false on timeout.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          uint64_t limit, uint32_t* status, int lane) {
  int ok = 1;
  if (lane == 0) {
    ok = wait_phase(bar, parity, abort, limit) ? 1 : 0;
    if (!ok) raise_abort(abort, status);
  }
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__global__ void __launch_bounds__(256, 1)
    attention_gqa_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const AttnArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK[2] = {sQ + kTile, sQ + 3 * kTile};
  const uint32_t sV[2] = {sQ + 2 * kTile, sQ + 4 * kTile};
  const uint32_t sP[2] = {sQ + 5 * kTile, sQ + 6 * kTile};
  AttnShared& sh = *reinterpret_cast<AttnShared*>(smem + 7 * kTile);
  volatile int* abort = &sh.abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // work unit: heavy (late) query blocks first
  const int per_seq = args.nqb * args.hq;
  const int seq = blockIdx.x / per_seq;
  const int rem = blockIdx.x - seq * per_seq;
  const int h = rem / args.nqb;
  const int qb = args.nqb - 1 - (rem - h * args.nqb);
  const int g = h / (args.hq / args.hkv);
  const int s0 = seq * args.seq_len;                           // first token of the sequence
  const int n = min(args.seq_len, args.T - s0);                // tokens of the sequence
  const int nkv = qb + 1;                                      // key blocks 0 .. qb (causal)
  const uint64_t limit = args.wait_ns;

  if (threadIdx.x == 0) {
    sh.abort = 0;
    mbar_init(smem_u32(&sh.q_full), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&sh.kv_full[s]), 1);
      mbar_init(smem_u32(&sh.kv_empty[s]), 1);
      mbar_init(smem_u32(&sh.s_full[s]), 1);
      mbar_init(smem_u32(&sh.s_empty[s]), 4);
    }
    mbar_init(smem_u32(&sh.p_full), 4);
    mbar_init(smem_u32(&sh.o_done), 1);
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
  const uint32_t tmem = sh.tmem_base;

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer
    prefetch_map(&tmQ);
    prefetch_map(&tmK);
    prefetch_map(&tmV);
    const uint32_t qf = smem_u32(&sh.q_full);
    mbar_expect_tx(qf, kTile);
    tma_load_2d(sQ, &tmQ, qf, h * kDh, s0 + qb * kBlk);
    tma_load_2d(sQ + kHalf, &tmQ, qf, h * kDh + 64, s0 + qb * kBlk);
    uint32_t issued = 0, iphase = 0;
    for (int j = 0; j < nkv; ++j) {
      const int st = j & 1;
      const uint32_t ph = (uint32_t)(j >> 1) & 1u;
      if (!wait_phase(smem_u32(&sh.kv_empty[st]), ph ^ 1u, abort, limit)) {
        raise_abort(abort, args.status);
        break;
      }
      const uint32_t fb = smem_u32(&sh.kv_full[st]);
      mbar_expect_tx(fb, 2 * kTile);
      const int row = s0 + j * kBlk;
      // K: 128 keys x 128 dims as two K-major halves
      tma_load_2d(sK[st], &tmK, fb, g * kDh, row);
      tma_load_2d(sK[st] + kHalf, &tmK, fb, g * kDh + 64, row);
      // V: [key half kb][dim half nc] boxes of 64 keys x 64 dims (MN-major B operand)
      for (int kb = 0; kb < 2; ++kb)
        for (int nc = 0; nc < 2; ++nc)
          tma_load_2d(sV[st] + kb * kHalf + nc * (kHalf / 2), &tmV, fb, g * kDh + 64 * nc,
                      row + 64 * kb);
      issued |= 1u << st;
      iphase = (iphase & ~(1u << st)) | (ph << st);
    }
    drain_phase(qf, 0, kAttnDrainNs);
    for (int s = 0; s < 2; ++s)
      if ((issued >> s) & 1u)
        if (!drain_phase(smem_u32(&sh.kv_full[s]), (iphase >> s) & 1u, kAttnDrainNs))
          atomicOr(args.status, kDevErrTimeout);
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA issuer
    bool ok = wait_phase(smem_u32(&sh.q_full), 0, abort, limit);
    bool any = false;
    if (!ok) raise_abort(abort, args.status);
    // S_j = Q K_jᵀ into score buffer j % 2
    auto issue_s = [&](int j) -> bool {
      const int st = j & 1;
      const uint32_t ph = (uint32_t)(j >> 1) & 1u;
      if (!wait_phase(smem_u32(&sh.kv_full[st]), ph, abort, limit) ||
          !wait_phase(smem_u32(&sh.s_empty[st]), ph ^ 1u, abort, limit)) {
        raise_abort(abort, args.status);
        return false;
      }
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kDh / 16; ++kk) {
        const uint32_t off = (uint32_t)(kk >> 2) * kHalf + (uint32_t)(kk & 3) * 32;
        umma_f16(tmem + (uint32_t)st * 128, sw128_desc(sQ + off), sw128_desc(sK[st] + off),
                 kIdescQK, kk > 0 ? 1u : 0u);
      }
      umma_commit(smem_u32(&sh.s_full[st]));
      any = true;
      return true;
    };
    if (ok) ok = issue_s(0);
    for (int j = 0; ok && j < nkv; ++j) {
      if (j + 1 < nkv && !issue_s(j + 1)) break;
      // O += P_j V_j once the softmax has written P_j (and rescaled O)
      if (!wait_phase(smem_u32(&sh.p_full), (uint32_t)j & 1u, abort, limit)) {
        raise_abort(abort, args.status);
        break;
      }
      tc_fence_after();
      const int st = j & 1;
#pragma unroll
      for (int kk = 0; kk < kBlk / 16; ++kk) {
        const uint32_t aoff = (uint32_t)(kk >> 2) * kHalf + (uint32_t)(kk & 3) * 32;
        const uint32_t boff = (uint32_t)(kk >> 2) * kHalf + (uint32_t)(kk & 3) * 2048;
        umma_f16(tmem + kColO, sw128_desc(sP[st] + aoff), sw128_mn_desc(sV[st] + boff), kIdescPV,
                 (j > 0 || kk > 0) ? 1u : 0u);
      }
      umma_commit(smem_u32(&sh.o_done));
      umma_commit(smem_u32(&sh.kv_empty[st]));
    }
    if (any) {
      umma_commit(smem_u32(&sh.drain));
      if (!drain_phase(smem_u32(&sh.drain), 0, kAttnDrainNs)) atomicOr(args.status, kDevErrTimeout);
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- softmax
    const int q = warp - 4;
    const int r = q * 32 + lane;                    // query row of the tile (TMEM lane)
    const int qi = qb * kBlk + r;                   // query index within the sequence
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    float m = -1e30f, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const int st = j & 1;
      if (!warp_wait(smem_u32(&sh.s_full[st]), (uint32_t)(j >> 1) & 1u, abort, limit,
                     args.status, lane)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t u[32];
        tmem_ld32(tmem + lane_base + (uint32_t)st * 128 + c * 32, u);
        tmem_wait(u);
#pragma unroll
        for (int i = 0; i < 32; ++i) sv[c * 32 + i] = __uint_as_float(u[i]);
      }
      // the score buffer may be refilled
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.s_empty[st]));
      // mask (causal, sequence end) on the diagonal block, or where the block passes the end
      // of the sequence; every earlier block is entirely visible to every row
      const int k0 = j * kBlk;
      float mb = -1e30f;
      if (j == qb || k0 + kBlk > n) {
#pragma unroll
        for (int i = 0; i < 128; ++i) {
          const bool valid = (k0 + i <= qi) && (k0 + i < n);
          sv[i] = valid ? sv[i] * args.scale_log2 : -INFINITY;
          mb = fmaxf(mb, sv[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 128; ++i) {
          sv[i] *= args.scale_log2;
          mb = fmaxf(mb, sv[i]);
        }
      }
      // lazy rescaling: raise the offset only when the block's maximum passes it by more
      // than kRescaleLog2 (then every lane of the warp takes its own new offset)
      float corr = 1.0f;
      const bool rescale = __any_sync(0xffffffffu, mb > m + kRescaleLog2);
      if (rescale) {
        const float m_new = fmaxf(m, mb);
        corr = fast_exp2(m - m_new);
        m = m_new;
      }
      float sum = 0.f;
#pragma unroll
      for (int i = 0; i < 128; ++i) {
        sv[i] = fast_exp2(sv[i] - m);
        sum += sv[i];
      }
      l = l * corr + sum;
      // P row (bf16) into buffer j % 2, the swizzled A tile of P V: key half c/2, 16-byte
      // chunk ^ (r % 8).  P V of block j - 2, the buffer's previous reader, finished before
      // the wait of the previous step.
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t rowp = sP[st] + (uint32_t)(c >> 1) * kHalf + (uint32_t)r * 128u;
        const int j0 = (c & 1) * 4;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float* v = &sv[c * 32 + 8 * i];
          const uint32_t a = rowp + ((uint32_t)((j0 + i) ^ (r & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a),
                       "r"(pack_bf16x2(v[0], v[1])), "r"(pack_bf16x2(v[2], v[3])),
                       "r"(pack_bf16x2(v[4], v[5])), "r"(pack_bf16x2(v[6], v[7]))
                       : "memory");
        }
      }
      if (j > 0) {
        // P V of the previous block has finished with O: rescale it if the offset moved
        if (!warp_wait(smem_u32(&sh.o_done), (uint32_t)(j - 1) & 1u, abort, limit, args.status,
                       lane)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (rescale) {
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t u[32];
            tmem_ld32(tmem + lane_base + kColO + c * 32, u);
            tmem_wait(u);
#pragma unroll
            for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * corr);
            tmem_st32(tmem + lane_base + kColO + c * 32, u);
          }
          tmem_st_wait();
        }
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.p_full));
    }
    if (ok && warp_wait(smem_u32(&sh.o_done), (uint32_t)(nkv - 1) & 1u, abort, limit, args.status,
                        lane)) {
      tc_fence_after();
      const float inv = 1.0f / l;
      bf16* orow = args.out + ((size_t)(s0 + qi) * args.hq + h) * kDh;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t u[32];
        tmem_ld32(tmem + lane_base + kColO + c * 32, u);
        tmem_wait(u);
        if (qi < n) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 o;
            o.x = pack_bf16x2(__uint_as_float(u[8 * i + 0]) * inv, __uint_as_float(u[8 * i + 1]) * inv);
            o.y = pack_bf16x2(__uint_as_float(u[8 * i + 2]) * inv, __uint_as_float(u[8 * i + 3]) * inv);
            o.z = pack_bf16x2(__uint_as_float(u[8 * i + 4]) * inv, __uint_as_float(u[8 * i + 5]) * inv);
            o.w = pack_bf16x2(__uint_as_float(u[8 * i + 6]) * inv, __uint_as_float(u[8 * i + 7]) * inv);
            dst[i] = o;
          }
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

cudaError_t attn_smem_attr() {
  static cudaError_t err = cudaErrorNotReady;
  static std::once_flag once;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(attention_gqa_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kAttnSmem);
  });
  return err;
}

}  // namespace

cudaError_t launch_attention_gqa(const bf16* q, const bf16* k, const bf16* v, int T, int seq_len,
                                 int hq, int hkv, bf16* out, uint32_t* status,
                                 unsigned long long wait_ns, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  cudaError_t e = attn_smem_attr();
  if (e != cudaSuccess) return e;
  CUtensorMap mQ, mK, mV;
  if (!make_map(&mQ, q, (uint64_t)T, (uint64_t)hq * kDh, 128) ||
      !make_map(&mK, k, (uint64_t)T, (uint64_t)hkv * kDh, 128) ||
      !make_map(&mV, v, (uint64_t)T, (uint64_t)hkv * kDh, 64))
    return cudaErrorInvalidValue;
  AttnArgs a;
  a.T = T;
  a.seq_len = seq_len > 0 ? seq_len : T;
  a.nseq = (T + a.seq_len - 1) / a.seq_len;
  a.nqb = (a.seq_len + kBlk - 1) / kBlk;
  a.hq = hq;
  a.hkv = hkv;
  a.scale_log2 = 1.4426950408889634f / sqrtf((float)kDh);
  a.out = out;
  a.status = status;
  a.wait_ns = wait_ns;
  const long long ctas = (long long)a.nseq * hq * a.nqb;
  attention_gqa_kernel<<<(unsigned)ctas, 256, kAttnSmem, s>>>(mQ, mK, mV, a);
  return cudaGetLastError();
}

}  // namespace moe
