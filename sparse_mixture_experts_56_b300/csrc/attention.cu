// Causal grouped-query attention on the tensor cores (the attention sub-block of each decoder
// layer: "Mixtral of Experts" (xyznot.com summary), Método: 32 attention heads and 8 key-value
// heads at hidden size 4096, so head dimension 128; newsflash.city digest: the full dense 32k
// context, no sliding window).  For query head h, key-value head g = h / (Hq / Hkv) and
// query i of a sequence:
//     o_i = sum_{j <= i} softmax_j(q_i · k_j / sqrt(128)) v_j
//
// One CTA per (sequence, query head, 128-query tile), heaviest tiles first, 320 threads,
// warp-specialised:
//   warp 0      allocates / frees the TMEM columns (two score buffers S_a, S_b and O, 128
//               each); its lane 0 is the TMA producer: the Q tile once, then K and V tiles of
//               128 keys into two-stage rings (K-major K tile; V as MN-major B operand), K and
//               V stages freed separately.
//   warp 1      MMA issuer.  The scores of key block j go to buffer j mod 2, so the scores of
//               block j + 1 are computed while the softmax works on block j: the issue order is
//               S(0) S(1) | PV(0) S(2) | PV(1) S(3) | ..., with P(j) read from TMEM (it
//               overwrites S(j) in its buffer) and V MN-major.  The softmax therefore never
//               waits for a score product that depends on its own previous P.
//   warps 2-9   softmax, two threads per query row (warps 2-5 take the first 64 keys of a
//               block, warps 6-9 the last 64; a warp reaches the TMEM lanes 32 (w mod 4) ..
//               +31): the scores from TMEM into registers, causal / sequence mask on the
//               diagonal block only, the row maximum combined through shared memory, online
//               softmax with lazy rescaling of O in TMEM (the exponent offset moves only when
//               a block's maximum passes it by 2^8; O is rescaled after the P V product of the
//               previous block has finished), P written as bf16 into TMEM; finally O / l
//               stored as bf16.  The exchange of the row maximum also orders the second half's
//               P stores after the first half's score loads (P overwrites S columns 0-63).
// MMAs of one thread run in issue order: S(j + 2) is issued after P V(j), so the completion
// of S(j) tells the softmax that P V(j - 2) has finished reading buffer j mod 2.
// Every wait is bounded (globaltimer) as in the expert GEMMs; a timeout sets the status bit,
// every role stops, the MMAs in flight are drained and TMEM is freed.
#include "moe_internal.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace ptx;

constexpr int kDh = 128;                         // head dimension
constexpr int kBlk = 128;                        // queries per tile = keys per block
constexpr uint32_t kTile = 128 * 128 * 2;        // one 128 x 128 bf16 tile (32 KB)
constexpr uint32_t kHalf = kTile / 2;            // a 128 x 64 (or 64 x 128) half tile
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = 256;       // S/P of block j at 128 (j mod 2), O at 256
constexpr uint64_t kAttnDrainNs = 200ull * 1000 * 1000;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kThreads = 320;   // 2 control warps + 8 softmax warps

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
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
  uint64_t s_full[2], p_full[2], o_done;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  // the two threads of a query row (one per column half) exchange partial maxima and sums:
  // [slot][half][row] values and the number of the exchange they belong to (slot = parity of
  // the exchange)
  float xval[2][2][128];
  int xseq[2][2][128];
};

// shared memory: Q | K0 | V0 | K1 | V1 | AttnShared, 1024-byte aligned tiles
constexpr size_t kAttnSmem = 1024 + 5 * (size_t)kTile + sizeof(AttnShared);

__device__ __forceinline__ void umma_ss(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// A operand from TMEM (rows in lanes, K packed two bf16 per column)
__device__ __forceinline__ void umma_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
// 8 consecutive 32-bit columns of this thread's TMEM lane, loaded (the wait is separate)
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}
// 8 consecutive 32-bit columns (16 bf16 of P)
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
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

// max(a, b, c) in one instruction
__device__ __forceinline__ float max3(float a, float b, float c) {
  float m;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(m) : "f"(a), "f"(b), "f"(c));
  return m;
}
__device__ __forceinline__ uint64_t pair2(float lo, float hi) {
  return ((uint64_t)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}
// (x0, x1) * c + n for the pairs c = (c, c), n = (n, n): one packed fp32 FMA, each half
// rounded as fmaf
__device__ __forceinline__ void fma2(float x0, float x1, uint64_t c2, uint64_t n2, float& y0,
                                     float& y1) {
  asm("{\n .reg .b64 s, r;\n mov.b64 s, {%2, %3};\n fma.rn.f32x2 r, s, %4, %5;\n"
      " mov.b64 {%0, %1}, r;\n}\n"
      : "=f"(y0), "=f"(y1)
      : "f"(x0), "f"(x1), "l"(c2), "l"(n2));
}
// acc += (x0, x1), one packed fp32 add
__device__ __forceinline__ void add2(uint64_t& acc, float x0, float x1) {
  asm("{\n .reg .b64 t;\n mov.b64 t, {%1, %2};\n add.rn.f32x2 %0, %0, t;\n}\n"
      : "+l"(acc)
      : "f"(x0), "f"(x1));
}

// The two threads of a query row swap a value: publish (v, seq) in the slot of seq's parity,
// then wait (bounded) for the partner's entry of the same exchange in that slot.  A thread
// that runs ahead to exchange seq + 1 writes the other slot, and it cannot reach seq + 2
// before its partner has published seq + 1, which the partner does only after reading
// exchange seq -- so neither the value nor the sequence number the partner waits for is
// overwritten early.  A warp goes on only if every lane got its value.
__device__ __forceinline__ bool row_exchange(float* xval, volatile int* xseq, int mine,
                                             int other, float v, int seq, float& got,
                                             volatile int* abort, uint64_t limit,
                                             uint32_t* status) {
  const int so = (seq & 1) << 8;   // slot offset: [slot][half][row]
  xval[so + mine] = v;
  tc_fence_before();
  __threadfence_block();
  xseq[so + mine] = seq;
  bool ok = true;
  if (xseq[so + other] != seq) {
    const uint64_t t0 = gtimer();
    while (xseq[so + other] != seq) {
      if (*abort || gtimer() - t0 > limit) {
        ok = false;
        break;
      }
    }
  }
  __threadfence_block();
  tc_fence_after();
  got = reinterpret_cast<volatile float*>(xval)[so + other];
  if (!__all_sync(0xffffffffu, ok)) {
    if (!ok) raise_abort(abort, status);
    return false;
  }
  return true;
}

// Lane 0 of a softmax warp waits on `bar` for the warp; false on timeout.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          uint64_t limit, uint32_t* status, int lane) {
  int ok = 1;
  if (lane == 0) {
    ok = wait_fast(bar, parity, abort, limit) ? 1 : 0;
    if (!ok) raise_abort(abort, status);
  }
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__global__ void __launch_bounds__(kThreads, 1)
    attention_gqa_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const AttnArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK[2] = {sQ + kTile, sQ + 3 * kTile};
  const uint32_t sV[2] = {sQ + 2 * kTile, sQ + 4 * kTile};
  AttnShared& sh = *reinterpret_cast<AttnShared*>(smem + 5 * kTile);
  volatile int* abort = &sh.abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // work unit: one query tile; units of the same tile index (equal work) for every sequence
  // and head are adjacent, the heaviest tile index first
  const int per_qb = args.nseq * args.hq;
  const int qb = args.nqb - 1 - (int)(blockIdx.x / per_qb);
  const int rem = (int)(blockIdx.x % per_qb);
  const int seq = rem / args.hq;
  const int h = rem - seq * args.hq;
  const int g = h / (args.hq / args.hkv);
  const int s0 = seq * args.seq_len;                           // first token of the sequence
  const int n = min(args.seq_len, args.T - s0);                // tokens of the sequence
  const int nkv = qb + 1;                                      // causal key blocks
  const uint64_t limit = args.wait_ns;

  for (int i = threadIdx.x; i < 2 * 2 * 128; i += blockDim.x) (&sh.xseq[0][0][0])[i] = 0;
  if (threadIdx.x == 0) {
    sh.abort = 0;
    mbar_init(smem_u32(&sh.q_full), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&sh.k_full[s]), 1);
      mbar_init(smem_u32(&sh.k_empty[s]), 1);
      mbar_init(smem_u32(&sh.v_full[s]), 1);
      mbar_init(smem_u32(&sh.v_empty[s]), 1);
      mbar_init(smem_u32(&sh.s_full[s]), 1);
      mbar_init(smem_u32(&sh.p_full[s]), 8);
    }
    mbar_init(smem_u32(&sh.o_done), 1);
    mbar_init(smem_u32(&sh.drain), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0) {
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
    // bit b of issued / iphase: barrier b (K stage 0, K stage 1, V stage 0, V stage 1) has a
    // load in flight / the phase of its last load.  K runs one block ahead of V: the scores
    // of block j + 2 are issued right after P V(j), so K(j + 2) is loaded before the wait
    // for the V stage that P V(j - 2) frees.
    uint32_t issued = 0, iphase = 0;
    // K tile of block j: 128 keys x 128 dims as two K-major halves
    auto load_k = [&](int j) -> bool {
      const int st = j & 1;
      const uint32_t ph = (uint32_t)(j >> 1) & 1u;
      if (!wait_fast(smem_u32(&sh.k_empty[st]), ph ^ 1u, abort, limit)) {
        raise_abort(abort, args.status);
        return false;
      }
      const uint32_t kb_bar = smem_u32(&sh.k_full[st]);
      mbar_expect_tx(kb_bar, kTile);
      tma_load_2d(sK[st], &tmK, kb_bar, g * kDh, s0 + j * kBlk);
      tma_load_2d(sK[st] + kHalf, &tmK, kb_bar, g * kDh + 64, s0 + j * kBlk);
      issued |= 1u << st;
      iphase = (iphase & ~(1u << st)) | (ph << st);
      return true;
    };
    bool go = load_k(0);
    for (int j = 0; go && j < nkv; ++j) {
      const int st = j & 1;
      const uint32_t ph = (uint32_t)(j >> 1) & 1u;
      if (j + 1 < nkv && !load_k(j + 1)) break;
      // V: [key half kb][dim half nc] boxes of 64 keys x 64 dims (MN-major B operand)
      if (!wait_fast(smem_u32(&sh.v_empty[st]), ph ^ 1u, abort, limit)) {
        raise_abort(abort, args.status);
        break;
      }
      const uint32_t vb_bar = smem_u32(&sh.v_full[st]);
      mbar_expect_tx(vb_bar, kTile);
      for (int kb = 0; kb < 2; ++kb)
        for (int nc = 0; nc < 2; ++nc)
          tma_load_2d(sV[st] + kb * kHalf + nc * (kHalf / 2), &tmV, vb_bar, g * kDh + 64 * nc,
                      s0 + j * kBlk + 64 * kb);
      issued |= 4u << st;
      iphase = (iphase & ~(4u << st)) | (ph << (st + 2));
    }
    drain_phase(qf, 0, kAttnDrainNs);
    for (int b = 0; b < 4; ++b)
      if ((issued >> b) & 1u) {
        const uint32_t bar = b < 2 ? smem_u32(&sh.k_full[b]) : smem_u32(&sh.v_full[b - 2]);
        if (!drain_phase(bar, (iphase >> b) & 1u, kAttnDrainNs))
          atomicOr(args.status, kDevErrTimeout);
      }
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA issuer
    bool ok = wait_fast(smem_u32(&sh.q_full), 0, abort, limit);
    bool any = false;
    if (!ok) raise_abort(abort, args.status);
    // operand descriptors built once; every buffer, stage and K slice is a constant offset
    const uint64_t dQ = sw128_desc(sQ);             // Q | K0 | V0 | K1 | V1
    const uint64_t dV = sw128_mn_desc(sQ);
    // S(j) = Q K_jᵀ into score buffer j mod 2 (the K stage of block j must have landed); the
    // product frees the K stage
    auto issue_s = [&](int j) -> bool {
      const int st = j & 1;
      if (!wait_fast(smem_u32(&sh.k_full[st]), (uint32_t)(j >> 1) & 1u, abort, limit)) {
        raise_abort(abort, args.status);
        return false;
      }
      tc_fence_after();
      const uint64_t dk = desc_add(dQ, (uint32_t)(1 + 2 * st) * kTile);
      const uint32_t d_s = tmem + kColS + (uint32_t)st * 128;
#pragma unroll
      for (int kk = 0; kk < kDh / 16; ++kk) {
        const uint32_t off = (uint32_t)(kk >> 2) * kHalf + (uint32_t)(kk & 3) * 32;
        umma_ss(d_s, desc_add(dQ, off), desc_add(dk, off), kIdescQK, kk > 0 ? 1u : 0u);
      }
      umma_commit(smem_u32(&sh.s_full[st]));
      umma_commit(smem_u32(&sh.k_empty[st]));
      any = true;
      return true;
    };
    for (int j = 0; ok && j < 2 && j < nkv; ++j) ok = issue_s(j);
    for (int j = 0; ok && j < nkv; ++j) {
      const int st = j & 1;
      // O += P(j) V_j once the softmax has written P(j) into buffer j mod 2 (and rescaled O)
      // and the V tile of block j has landed
      if (!wait_fast(smem_u32(&sh.p_full[st]), (uint32_t)(j >> 1) & 1u, abort, limit) ||
          !wait_fast(smem_u32(&sh.v_full[st]), (uint32_t)(j >> 1) & 1u, abort, limit)) {
        raise_abort(abort, args.status);
        ok = false;
        break;
      }
      tc_fence_after();
      const uint64_t dv = desc_add(dV, (uint32_t)(2 + 2 * st) * kTile);
      const uint32_t d_o = tmem + kColO;
      const uint32_t a_p = tmem + kColS + (uint32_t)st * 128;
#pragma unroll
      for (int kk = 0; kk < kBlk / 16; ++kk) {
        const uint32_t boff = (uint32_t)(kk >> 2) * kHalf + (uint32_t)(kk & 3) * 2048;
        umma_ts(d_o, a_p + kk * 8, desc_add(dv, boff), kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
      }
      umma_commit(smem_u32(&sh.o_done));
      umma_commit(smem_u32(&sh.v_empty[st]));
      // the scores two blocks ahead go to the buffer P(j) came from (after P V(j) in issue
      // order)
      if (j + 2 < nkv && !issue_s(j + 2)) {
        ok = false;
        break;
      }
    }
    if (any) {
      umma_commit(smem_u32(&sh.drain));
      if (!drain_phase(smem_u32(&sh.drain), 0, kAttnDrainNs)) atomicOr(args.status, kDevErrTimeout);
    }
  } else if (warp >= 2) {
    // ---------------------------------------------------------------- softmax
    const int hh = (warp - 2) >> 2;                  // column half: keys 64 hh .. 64 hh + 63
    const int q = warp & 3;                          // TMEM lane quarter of this warp
    const int r = q * 32 + lane;                     // query row of the tile (TMEM lane)
    const int qi = qb * kBlk + r;                    // query index within the sequence
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const uint32_t tO = tmem + lane_base + kColO;
    float m = -1e30f, l = 0.f;
    bool ok = true;
    float* xval = &sh.xval[0][0][0];
    volatile int* xseq = &sh.xseq[0][0][0];
    const int xm = hh * 128 + r, xo = (hh ^ 1) * 128 + r;   // this thread's / the partner's slot
    int seq = 0;
    for (int j = 0; ok && j < nkv; ++j) {
      const int st = j & 1;
      const uint32_t tS = tmem + lane_base + kColS + (uint32_t)st * 128;
      if (!warp_wait(smem_u32(&sh.s_full[st]), (uint32_t)(j >> 1) & 1u, abort, limit, args.status,
                     lane)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int k0 = j * kBlk;
      // this half's 64 raw scores: two loads in flight, one wait
      uint32_t u0[32], u1[32];
      tmem_ld32(tS + hh * 64, u0);
      tmem_ld32(tS + hh * 64 + 32, u1);
      tmem_wait(u0);
      tmem_wait(u1);
#define SV(i) (*reinterpret_cast<float*>((i) < 32 ? &u0[(i)] : &u1[(i) - 32]))
      const int kh = k0 + hh * 64;                   // first key of this half
      // mask (diagonal block or past the sequence end only) and the block's maximum, taken on
      // the raw scores and scaled once (the scale is positive)
      // (eight independent partial maxima, three-input max instructions, and packed
      // two-wide fp32 FMAs and adds keep the chains short and the instruction count low)
      if (j == qb || k0 + kBlk > n) {
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          const bool valid = (kh + i <= qi) && (kh + i < n);
          SV(i) = valid ? SV(i) : -INFINITY;
        }
      }
      float mp[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) mp[a] = fmaxf(SV(2 * a), SV(2 * a + 1));
#pragma unroll
      for (int i = 8; i < 32; ++i) mp[i & 7] = max3(mp[i & 7], SV(2 * i), SV(2 * i + 1));
      float mb = max3(max3(mp[0], mp[1], mp[2]), max3(mp[3], mp[4], mp[5]), fmaxf(mp[6], mp[7]));
      {
        float mo;
        if (!row_exchange(xval, xseq, xm, xo, mb, ++seq, mo, abort, limit, args.status)) {
          ok = false;
          break;
        }
        mb = fmaxf(mb, mo);
      }
      mb *= args.scale_log2;
      // lazy rescaling of the exponent offset (warp-uniform decision, per-lane offsets)
      float corr = 1.0f;
      const bool rescale = __any_sync(0xffffffffu, mb > m + kRescaleLog2);
      if (rescale) {
        const float m_new = fmaxf(m, mb);
        corr = fast_exp2(m - m_new);
        m = m_new;
        if (j > 0) {
          // O may be rescaled once P V(j - 1) has finished accumulating into it (this half's
          // 64 columns, 8 at a time: the scores stay in registers meanwhile)
          if (!warp_wait(smem_u32(&sh.o_done), (uint32_t)(j - 1) & 1u, abort, limit, args.status,
                         lane)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int c = 8 * hh; c < 8 * hh + 8; ++c) {
            uint32_t u[8];
            tmem_ld8(tO + c * 8, u);
            asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(u[0]), "+r"(u[1]), "+r"(u[2]),
                         "+r"(u[3]), "+r"(u[4]), "+r"(u[5]), "+r"(u[6]), "+r"(u[7])::"memory");
#pragma unroll
            for (int i = 0; i < 8; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * corr);
            tmem_st8(tO + c * 8, u);
          }
        }
      }
      // P = exp2(score - offset) as bf16 over the first 64 columns of the buffer (columns
      // 16c .. 16c+15 hold keys 32c .. 32c+31; this half writes chunks 2 hh and 2 hh + 1)
      const uint64_t c2 = pair2(args.scale_log2, args.scale_log2), n2 = pair2(-m, -m);
      uint64_t sp[2] = {0, 0};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float x0, x1;
          fma2(SV(c * 16 + 2 * i), SV(c * 16 + 2 * i + 1), c2, n2, x0, x1);
          const float p0 = fast_exp2(x0);
          const float p1 = fast_exp2(x1);
          add2(sp[i & 1], p0, p1);
          pk[i] = pack_bf16x2(p0, p1);
        }
        tmem_st8(tS + hh * 32 + c * 8, pk);
      }
      float sum = 0.f;
#pragma unroll
      for (int a = 0; a < 2; ++a)
        sum += __uint_as_float((uint32_t)sp[a]) + __uint_as_float((uint32_t)(sp[a] >> 32));
#undef SV
      l = l * corr + sum;
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.p_full[st]));
    }
    // the row sum over both halves
    if (ok) {
      float lo;
      ok = row_exchange(xval, xseq, xm, xo, l, ++seq, lo, abort, limit, args.status);
      l += lo;
    }
    if (ok && warp_wait(smem_u32(&sh.o_done), (uint32_t)(nkv - 1) & 1u, abort, limit, args.status,
                        lane)) {
      tc_fence_after();
      const float inv = 1.0f / l;
      bf16* orow = args.out + ((size_t)(s0 + qi) * args.hq + h) * kDh;
#pragma unroll 1
      for (int c = 2 * hh; c < 2 * hh + 2; ++c) {
        uint32_t u[32];
        tmem_ld32(tO + c * 32, u);
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
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

cudaError_t attn_smem_attr() {
  static PerDeviceSetting setting;
  return setting.get([] {
    return cudaFuncSetAttribute(attention_gqa_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kAttnSmem);
  });
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
  attention_gqa_kernel<<<(unsigned)ctas, kThreads, kAttnSmem, s>>>(mQ, mK, mV, a);
  return cudaGetLastError();
}

}  // namespace moe
