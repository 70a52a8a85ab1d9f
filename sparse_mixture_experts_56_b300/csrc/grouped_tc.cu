// Experts on the 5th-generation tensor cores (bf16 in, fp32 accumulate in TMEM):
//   GEMM1  h[p, :]      = SiLU(x_p · w1_eᵀ) ⊙ (x_p · w3_eᵀ)      (SwiGLU fused in the epilogue)
//   GEMM2  y_perm[p, :] = h[p, :] · w2_eᵀ
// for the rows p in [offsets[e], offsets[e+1]) of every expert e ("Mixtral of Experts"
// (xyznot.com summary), Método: each expert is a SwiGLU network of intermediate size 14336;
// ja.news.hada.io, 実装と推論効率: experts receive variable numbers of tokens).
//
// Design (persistent, one CTA per SM, 256 threads, warp-specialised):
//   warp 0      TMA producer: A tile [128 x 64] + B tile [rows x 64] per stage, 128-byte
//               swizzle, into a shared-memory ring.
//   warp 1      MMA issuer: tcgen05.mma.kind::f16, N=256 K=16, four per stage, into one of two
//               TMEM accumulators (2 x 256 columns = all 512).
//   warp 2      allocates / frees the 512 TMEM columns.
//   warps 4-7   epilogue: tcgen05.ld 32x32b (warp w reads TMEM lanes 32*(w-4)...), then
//               GEMM1: SiLU(a)⊙b -> bf16 h;  GEMM2: -> bf16 y_perm.  Rows beyond the
//               expert's count are computed but never stored.
// Two forms share this code:
//   single CTA  (cta_group::1) M=128 tiles; each stage holds A [128 x 64] and all 256 B rows
//               (48 KB, 4 stages).  Used for small expert groups (decode), where the kernel
//               streams weights and the smaller tile wastes less of each MMA, and for GEMM1.
//   CTA pair    (cta_group::2, clusters of 2) M=256 tiles: each CTA loads its own 128 rows of
//               A and HALF of the 256 B rows (32 KB per stage, 6 stages); the even CTA issues
//               one MMA that reads both CTAs' shared memory and writes each CTA's 128 rows of
//               the accumulator into its own TMEM.  Per FLOP every SM moves a third less data
//               from L2 into shared memory.  Used for GEMM2 on large expert groups.
// For GEMM1 the 256 accumulator columns pair 128 rows of w1_e with the same 128 rows of w3_e
// (single CTA: both in one stage; pair: w1 in the even CTA, w3 in the odd one), so the SwiGLU
// epilogue finds a and b in columns c and 128 + c of the same TMEM lane.
// Work list: tiles (expert, m-tile, n-tile) enumerated on the device from expert_offsets
// (no host synchronisation); within an expert, groups of 16 m-tiles sweep all n-tiles so
// that the weight tiles of concurrently running CTAs are shared through L2.
//
// Every wait is bounded (globaltimer).  A wait that runs past the limit raises the CTA's
// abort flag and sets the timeout bit of the device status word; every role then stops,
// the producer waits (bounded) for its copies in flight, the MMA warp waits for its MMAs,
// and the TMEM columns are freed before the CTA exits.  In the pair form a CTA that gives up
// makes its peer's waits run out too; both meet at the final cluster barrier.
#include <cuda.h>

#include <atomic>
#include <mutex>

#include "moe_internal.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace ptx;

constexpr int BM = 128;                 // accumulator rows per CTA (TMEM lanes)
constexpr int BK = 64;                  // K per stage: one 128-byte swizzle atom of bf16
constexpr int BN = 256;                 // UMMA N = accumulator columns
constexpr int UMMA_K = 16;
constexpr int ACC = 2;                  // TMEM accumulators
constexpr uint32_t TMEM_COLS = 512;
constexpr int GROUP_M = 16;
constexpr uint64_t kDrainNs = 200ull * 1000 * 1000;
constexpr uint64_t kPeerGraceNs = 1000ull * 1000;

// Forward:  kSwiGLU  h = SiLU(x w1ᵀ) ⊙ (x w3ᵀ)          A = x rows,  B = w1|w3 (K-major)
//           kDown    y_perm = h w2ᵀ                     A = h rows,  B = w2 (K-major)
// Backward (rows in the expert-padded layout, every expert's segment a multiple of 128 rows):
//           kStoreAB [a | b] = x [w1 | w3]ᵀ, stored      A = x rows,  B = w1|w3 (K-major)
//           kDh      dh' = g w2 (g = dL/dy rows); the epilogue forms h, the gate gradient
//                    partial <dh', h>, and the gate-scaled da, db, G·h
//                                                        A = g rows,  B = w2 (MN-major)
//           kDgradX  dx = da w1 + db w3                  A = da|db,   B = w1|w3 (MN-major)
//           kWgrad   dW = Pᵀ Q over an expert's rows     A = P, B = Q (both MN-major)
enum Mode { kSwiGLU = 0, kDown = 1, kStoreAB = 2, kDh = 3, kDgradX = 4, kWgrad = 5 };

// Which operands sit in shared memory MN-major (the contiguous global dimension is M or N
// rather than the reduction dimension K).
constexpr bool a_mn(int mode) { return mode == kWgrad; }
constexpr bool b_mn(int mode) { return mode == kDh || mode == kDgradX || mode == kWgrad; }

// Geometry of the two forms.
template <bool PAIR>
struct Cfg {
  static constexpr int kCtas = PAIR ? 2 : 1;
  static constexpr int kTileM = BM * kCtas;            // rows of one tile
  static constexpr int kBRows = BN / kCtas;            // B rows each CTA loads per stage
  static constexpr int kStages = PAIR ? 6 : 4;
  static constexpr uint32_t kABytes = BM * BK * 2;
  static constexpr uint32_t kBBytes = kBRows * BK * 2;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
};

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A bf16 (7-9 = 1), B bf16 (10-12 =
// 1), A / B MN-major (bit 15 / 16), N >> 3 at bits 17-22, M >> 4 at bits 24-28 (M of the whole
// CTA pair in the pair form).
template <int MODE, bool PAIR>
constexpr uint32_t instr_desc() {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn(MODE) ? 1u : 0u) << 15) |
         ((b_mn(MODE) ? 1u : 0u) << 16) | ((uint32_t)(BN >> 3) << 17) |
         ((uint32_t)(Cfg<PAIR>::kTileM >> 4) << 24);
}

struct TcArgs {
  const int32_t* offsets;  // rows of each expert: [offsets[e], offsets[e+1])
  int mrows;               // rows of the row-indexed operands; offsets are clamped to [0, mrows]
  int n;
  int kdim;   // reduction length (not used by kWgrad, whose K is the expert's row count)
  int ndim;   // output columns
  int ntiles; // n-tiles per expert
  bf16* out;  // main output
  uint32_t* status;
  unsigned long long wait_ns;
  // backward only
  int brows;          // kDh / kDgradX: rows of one expert's B matrix in its 2-D view (d or f)
  int kb_split;       // kDgradX: k-blocks taken from (da, w1) before switching to (db, w3)
  int mdim;           // kWgrad: rows of the weight gradient (M)
  int mtiles_w;       // kWgrad: 128-row tiles of M
  const bf16* ab;     // kDh: [rows, 2 ndim] recomputed a | b
  const float* wq;    // kDh: gate weight of every row (0 on padding rows)
  float* dwp;         // kDh: [rows, ntiles] partial sums of <dh', h>
  bf16* da;           // kDh outputs [rows, ndim]
  bf16* db;
  bf16* hw;
  // kSwiGLU, optional: also store a and b (bf16) for the backward, row p of expert e at
  // padded row poff_save[e] + (p - offsets[e]) of ab_save [rows, 2 ndim]
  bf16* ab_save;
  const int32_t* poff_save;
};

template <int STAGES>
struct Shared {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[ACC];
  uint64_t tempty[ACC];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int total;
  int tile_base[kMaxExperts + 1];
  int mtiles[kMaxExperts];
  int off[kMaxExperts + 1];
};

// Output staging for the TMA store of full tiles: 128 rows x 128 bf16 columns as two
// 128-byte-swizzled boxes of [128 rows x 64 columns].
constexpr uint32_t kStageOutBytes = 128 * 128 * 2;

template <bool PAIR>
constexpr size_t smem_bytes() {
  return 1024 + (size_t)Cfg<PAIR>::kStages * Cfg<PAIR>::kStageBytes + kStageOutBytes +
         sizeof(Shared<Cfg<PAIR>::kStages>);
}

// ------------------------------------------------------------------------------------------
// PTX of the CTA-pair form and of the GEMM modes (the common pieces are in tc_ptx.cuh)
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address, in the cluster's shared window, of the same shared variable in CTA `rank`.
__device__ __forceinline__ uint32_t peer_addr(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
// Arrive on an mbarrier of another CTA of the cluster (address from peer_addr).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}
// Pair form: the copy lands in this CTA's shared memory and its bytes are counted on an
// mbarrier that may live in either CTA of the pair (`bar_cluster` from peer_addr).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"((uint64_t)map), "r"(bar_cluster), "r"(c0), "r"(c1)
      : "memory");
}
// Descriptor of an operand tile at `base`, and the byte step from one 16-deep K slice to
// the next: 16 K-rows of 128 bytes (MN-major) or 32 bytes along the swizzled row (K-major).
template <bool MN>
__device__ __forceinline__ uint64_t tile_desc(uint32_t base) {
  if constexpr (MN)
    return sw128_mn_desc(base);
  else
    return sw128_desc(base);
}
template <bool MN>
constexpr uint32_t kSliceBytes = MN ? 16 * 128 : UMMA_K * 2;
template <int MODE, bool PAIR>
__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                          uint32_t accumulate) {
  if constexpr (PAIR)
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(instr_desc<MODE, true>()), "r"(accumulate)
        : "memory");
  else
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(instr_desc<MODE, false>()), "r"(accumulate)
        : "memory");
}
// Arrives on `bar` once the MMAs issued so far by this thread are done: in the pair form on
// the barrier at that offset in both CTAs.
template <bool PAIR>
__device__ __forceinline__ void umma_commit_all(uint32_t bar) {
  if constexpr (PAIR)
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"((uint16_t)0x3)
        : "memory");
  else
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}
// Arrives on this CTA's `bar` only.
template <bool PAIR>
__device__ __forceinline__ void umma_commit_local(uint32_t bar) {
  if constexpr (PAIR)
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
  else
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}
template <bool PAIR>
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem) {
  if constexpr (PAIR) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     dst_smem),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  } else {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     dst_smem),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
}
template <bool PAIR>
__device__ __forceinline__ void tmem_dealloc(uint32_t base) {
  if constexpr (PAIR)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(base),
                 "r"(TMEM_COLS)
                 : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base),
                 "r"(TMEM_COLS)
                 : "memory");
}




// 32 consecutive columns (chunk c32 of the 128 staged ones) of row r into the staging buffer:
// box c32/2, 16-byte chunks (c32%2)*4 .. +3 of the row, at chunk ^ (r % 8) (128-byte swizzle),
// so the 32 lanes writing 32 consecutive rows spread over all banks.
__device__ __forceinline__ void stage_row32(uint32_t stage, int r, int c32, const float (&v)[32]) {
  const uint32_t row = stage + (uint32_t)(c32 >> 1) * (kStageOutBytes / 2) + (uint32_t)r * 128u;
  const int j0 = (c32 & 1) * 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t a = row + ((uint32_t)((j0 + i) ^ (r & 7)) << 4);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a),
                 "r"(pack_bf16x2(v[8 * i + 0], v[8 * i + 1])),
                 "r"(pack_bf16x2(v[8 * i + 2], v[8 * i + 3])),
                 "r"(pack_bf16x2(v[8 * i + 4], v[8 * i + 5])),
                 "r"(pack_bf16x2(v[8 * i + 6], v[8 * i + 7]))
                 : "memory");
  }
}
// barrier of the four epilogue warps only
__device__ __forceinline__ void epilogue_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// the same barrier, returning whether `ok` holds in every epilogue thread (the four warps then
// take the same decision, which their later barriers need)
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

__device__ __noinline__ void spin_ns(uint64_t ns) {
  const uint64_t t0 = gtimer();
  while (gtimer() - t0 < ns) {
  }
}

struct Tile {
  int e, mt, nt;
  int row0;   // first A row (token-row modes) / first K row of the expert (kWgrad)
  int rows;   // valid rows of the tile (token-row modes) / K rows of the expert (kWgrad)
};

template <int MODE, int TILE_M>
__device__ __forceinline__ Tile decode_tile(const int* tile_base, const int* mtiles,
                                            const int* off, int n, int ntiles, int tile) {
  int e = 0;
  while (e + 1 < n && tile_base[e + 1] <= tile) ++e;
  const int u = tile - tile_base[e];
  const int per_group = GROUP_M * ntiles;
  const int g = u / per_group, r = u - g * per_group;
  const int gsz = min(GROUP_M, mtiles[e] - g * GROUP_M);
  Tile t;
  t.e = e;
  t.mt = g * GROUP_M + r % gsz;
  t.nt = r / gsz;
  if (MODE == kWgrad) {
    t.row0 = off[e];
    t.rows = off[e + 1] - off[e];
  } else {
    t.row0 = off[e] + t.mt * TILE_M;
    t.rows = min(TILE_M, off[e + 1] - off[e] - t.mt * TILE_M);
  }
  return t;
}

__device__ __forceinline__ void store_row32(bf16* dst, const float (&v)[32]) {
  uint4* q = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint4 o;
    o.x = pack_bf16x2(v[8 * j + 0], v[8 * j + 1]);
    o.y = pack_bf16x2(v[8 * j + 2], v[8 * j + 3]);
    o.z = pack_bf16x2(v[8 * j + 4], v[8 * j + 5]);
    o.w = pack_bf16x2(v[8 * j + 6], v[8 * j + 7]);
    q[j] = o;
  }
}

__device__ __forceinline__ float sigmoidf_(float z) { return __fdividef(1.0f, 1.0f + __expf(-z)); }

// ------------------------------------------------------------------------------------------
// the kernel
// ------------------------------------------------------------------------------------------
template <int MODE, bool PAIR>
__global__ void __launch_bounds__(256, 1)
    grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmA2,
                           const __grid_constant__ CUtensorMap tmB0,
                           const __grid_constant__ CUtensorMap tmB1,
                           const __grid_constant__ CUtensorMap tmOut, const TcArgs args) {
  using C = Cfg<PAIR>;
  constexpr int STAGES = C::kStages;
  static_assert(!PAIR || MODE == kSwiGLU || MODE == kDown || MODE == kWgrad,
                "the pair form serves the forward GEMMs and the weight gradients");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;                                  // STAGES x 16 KB
  uint8_t* sB = smem + STAGES * C::kABytes;            // STAGES x B_BYTES
  const uint32_t s_out = smem_u32(smem + STAGES * C::kStageBytes);   // output staging
  Shared<STAGES>& sh =
      *reinterpret_cast<Shared<STAGES>*>(smem + STAGES * C::kStageBytes + kStageOutBytes);
  volatile int* abort = &sh.abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = args.n;
  const int KB = args.kdim / BK;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;   // 0 = the CTA that issues the MMAs
  const int unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int units = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  if (threadIdx.x == 0) {
    // offsets made monotone inside [0, mrows], so that no tile reaches past the buffers
    // whatever the device-side offsets hold
    auto clamp_off = [&](int v, int lo) { return v < lo ? lo : (v > args.mrows ? args.mrows : v); };
    int acc = 0;
    int o0 = clamp_off(args.offsets[0], 0);
    for (int e = 0; e < n; ++e) {
      const int o1 = clamp_off(args.offsets[e + 1], o0);
      const int mt = MODE == kWgrad ? args.mtiles_w : (o1 - o0 + C::kTileM - 1) / C::kTileM;
      sh.off[e] = o0;
      sh.mtiles[e] = mt;
      sh.tile_base[e] = acc;
      acc += mt * args.ntiles;
      o0 = o1;
    }
    sh.off[n] = o0;
    sh.tile_base[n] = acc;
    sh.total = acc;
    sh.abort = 0;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&sh.full[s]), 1);
      mbar_init(smem_u32(&sh.empty[s]), 1);
    }
    for (int a = 0; a < ACC; ++a) {
      mbar_init(smem_u32(&sh.tfull[a]), 1);
      mbar_init(smem_u32(&sh.tempty[a]), 4 * C::kCtas);   // the epilogue warps of every CTA
    }
    mbar_init(smem_u32(&sh.drain), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 2) tmem_alloc<PAIR>(smem_u32(&sh.tmem_base));
  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync_all();   // the peer's barriers are initialised before anyone signals them
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sh.tmem_base;
  const int total = sh.total;
  const uint64_t limit = args.wait_ns;
  // Balanced static schedule: the fewest CTAs (pairs) that still finish in the same number
  // of tile rounds, so every working unit gets the same number of tiles (+-1 only in the
  // last round); the spare units exit at once.  For weight-streaming (HBM-bound) launches
  // this removes the tail round in which a few CTAs stream alone.
  const int rounds = (total + units - 1) / units;
  const int gstride = rounds > 0 ? (total + rounds - 1) / rounds : units;
  const int first_tile = unit < gstride ? unit : total;

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer
    prefetch_map(&tmA);
    if (MODE == kDgradX) prefetch_map(&tmA2);
    prefetch_map(&tmB0);
    if (MODE == kSwiGLU || MODE == kStoreAB || MODE == kDgradX) prefetch_map(&tmB1);
    int stage = 0;
    uint32_t phase = 0, issued = 0, iphase = 0;
    bool ok = true;
    for (int tile = first_tile; ok && tile < total; tile += gstride) {
      const Tile t =
          decode_tile<MODE, C::kTileM>(sh.tile_base, sh.mtiles, sh.off, n, args.ntiles, tile);
      const int arow = t.row0 + (int)rank * BM;
      // first B row of this CTA's share: GEMM1 takes 128 rows of w1 (and of w3), GEMM2 256
      // rows of w2, split between the two CTAs of a pair
      const int brow = (MODE == kSwiGLU || MODE == kStoreAB)
                           ? t.e * args.ndim + t.nt * (BN / 2)
                           : t.e * args.ndim + t.nt * BN + (int)rank * C::kBRows;
      const CUtensorMap* bmap = (MODE == kSwiGLU && PAIR && rank == 1) ? &tmB1 : &tmB0;
      const int kbs = MODE == kWgrad ? t.rows / BK : KB;
      for (int kb = 0; kb < kbs; ++kb) {
        if (!wait_fast(smem_u32(&sh.empty[stage]), phase ^ 1u, abort, limit)) {
          raise_abort(abort, args.status);
          ok = false;
          break;
        }
        const uint32_t fb = smem_u32(&sh.full[stage]);
        const uint32_t a_dst = smem_u32(sA + stage * C::kABytes);
        const uint32_t b_dst = smem_u32(sB + stage * C::kBBytes);
        if constexpr (PAIR) {
          // both CTAs' bytes land on the even CTA's barrier, which the MMA issuer waits on
          if (rank == 0) mbar_expect_tx(fb, 2 * C::kStageBytes);
          const uint32_t fb0 = peer_addr(fb, 0);
          if constexpr (MODE == kWgrad) {
            // both operands MN-major: this CTA's 128 M columns of P and 128 N columns of Q,
            // as 64-column chunks of 64 K-rows
            const int m0 = t.mt * C::kTileM + (int)rank * BM;
            const int n0 = t.nt * BN + (int)rank * C::kBRows;
            const int krow = t.row0 + kb * BK;
            tma_load_2d_pair(a_dst, &tmA, fb0, m0, krow);
            tma_load_2d_pair(a_dst + kMnChunkBytes, &tmA, fb0, m0 + 64, krow);
            tma_load_2d_pair(b_dst, &tmB0, fb0, n0, krow);
            tma_load_2d_pair(b_dst + kMnChunkBytes, &tmB0, fb0, n0 + 64, krow);
          } else {
            tma_load_2d_pair(a_dst, &tmA, fb0, kb * BK, arow);
            tma_load_2d_pair(b_dst, bmap, fb0, kb * BK, brow);
          }
        } else {
          mbar_expect_tx(fb, C::kStageBytes);
          // A: 128 rows x 64 K (K-major), or for kWgrad 64 K-rows x 2 chunks of 64 M columns
          if constexpr (MODE == kWgrad) {
            tma_load_2d(a_dst, &tmA, fb, t.mt * BM, t.row0 + kb * BK);
            tma_load_2d(a_dst + kMnChunkBytes, &tmA, fb, t.mt * BM + 64, t.row0 + kb * BK);
          } else if constexpr (MODE == kDgradX) {
            if (kb < args.kb_split)
              tma_load_2d(a_dst, &tmA, fb, kb * BK, arow);
            else
              tma_load_2d(a_dst, &tmA2, fb, (kb - args.kb_split) * BK, arow);
          } else {
            tma_load_2d(a_dst, &tmA, fb, kb * BK, arow);
          }
          // B: K-major rows, or MN-major 64 K-rows x 4 chunks of 64 N columns
          if constexpr (b_mn(MODE)) {
            const CUtensorMap* bm = &tmB0;
            int krow;
            if constexpr (MODE == kWgrad) {
              krow = t.row0 + kb * BK;
            } else if constexpr (MODE == kDgradX) {
              const bool second = kb >= args.kb_split;
              bm = second ? &tmB1 : &tmB0;
              krow = t.e * args.brows + (second ? kb - args.kb_split : kb) * BK;
            } else {
              krow = t.e * args.brows + kb * BK;
            }
#pragma unroll
            for (int i = 0; i < BN / 64; ++i)
              tma_load_2d(b_dst + i * kMnChunkBytes, bm, fb, t.nt * BN + 64 * i, krow);
          } else {
            tma_load_2d(b_dst, &tmB0, fb, kb * BK, brow);
            if (MODE == kSwiGLU || MODE == kStoreAB)
              tma_load_2d(b_dst + C::kBBytes / 2, &tmB1, fb, kb * BK, brow);
          }
        }
        issued |= 1u << stage;
        iphase = (iphase & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // every copy issued must have landed before the CTA may exit
    if (!PAIR || rank == 0) {
      for (int s = 0; s < STAGES; ++s)
        if ((issued >> s) & 1u)
          if (!drain_phase(smem_u32(&sh.full[s]), (iphase >> s) & 1u, kDrainNs))
            atomicOr(args.status, kDevErrTimeout);
    } else if (issued && *abort) {
      // the odd CTA's copies are counted on the even CTA's barriers; after an abort the
      // even CTA may not wait for them, so give them time to land
      spin_ns(kPeerGraceNs);
    }
  } else if (warp == 1 && lane == 0 && (!PAIR || rank == 0)) {
    // ---------------------------------------------------------------- MMA issuer
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true, any_mma = false;
    // operand descriptors of stage 0, built once; stages and K slices are constant offsets
    const uint64_t dA0 = tile_desc<a_mn(MODE)>(smem_u32(sA));
    const uint64_t dB0 = tile_desc<b_mn(MODE)>(smem_u32(sB));
    for (int tile = first_tile; ok && tile < total; tile += gstride) {
      int kbs = KB;
      if (MODE == kWgrad) {
        const Tile t =
            decode_tile<MODE, C::kTileM>(sh.tile_base, sh.mtiles, sh.off, n, args.ntiles, tile);
        kbs = t.rows / BK;
      }
      if (!wait_fast(smem_u32(&sh.tempty[acc]), acc_phase ^ 1u, abort, limit)) {
        raise_abort(abort, args.status);
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
      for (int kb = 0; kb < kbs; ++kb) {
        if (!wait_fast(smem_u32(&sh.full[stage]), phase, abort, limit)) {
          raise_abort(abort, args.status);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t da = desc_add(dA0, (uint32_t)stage * C::kABytes);
        const uint64_t db = desc_add(dB0, (uint32_t)stage * C::kBBytes);
#pragma unroll
        for (int kk = 0; kk < BK / UMMA_K; ++kk)
          umma_bf16<MODE, PAIR>(d_tmem, desc_add(da, kk * kSliceBytes<a_mn(MODE)>),
                                desc_add(db, kk * kSliceBytes<b_mn(MODE)>),
                                (kb | kk) != 0 ? 1u : 0u);
        any_mma = true;
        umma_commit_all<PAIR>(smem_u32(&sh.empty[stage]));
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      // (a weight-gradient tile of an expert without rows has no MMA: the commit still
      // arrives, and the epilogue writes zeros)
      umma_commit_all<PAIR>(smem_u32(&sh.tfull[acc]));
      if (++acc == ACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // all MMAs issued by this thread must finish before the TMEM columns are freed
    if (any_mma) {
      umma_commit_local<PAIR>(smem_u32(&sh.drain));
      if (!drain_phase(smem_u32(&sh.drain), 0, kDrainNs)) atomicOr(args.status, kDevErrTimeout);
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- epilogue
    const int q = warp - 4;  // TMEM lane quarter
    const int r = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = first_tile; tile < total; tile += gstride) {
      const Tile t =
          decode_tile<MODE, C::kTileM>(sh.tile_base, sh.mtiles, sh.off, n, args.ntiles, tile);
      int ok = 1;
      if (lane == 0) {
        // The accumulator is ready once per tile.  A tile reducing over d or f runs for tens
        // of microseconds, so the epilogue sleeps between tests; a weight-gradient tile
        // reduces over an expert's rows only (a microsecond at small batches) and polls.
        const uint32_t tf = smem_u32(&sh.tfull[acc]);
        ok = (MODE == kWgrad ? wait_fast(tf, acc_phase, abort, limit)
                             : wait_phase_sleepy(tf, acc_phase, abort, limit))
                 ? 1
                 : 0;
        if (!ok) raise_abort(abort, args.status);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!epilogue_all(ok)) break;
      tc_fence_after();
      const int row = (int)rank * BM + r;   // row of the tile held in this TMEM lane
      // kWgrad: row of the weight gradient held in this TMEM lane
      const int wrow = t.mt * C::kTileM + (int)rank * BM + r;
      const bool row_ok = MODE == kWgrad ? wrow < args.mdim : row < t.rows;
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      const uint32_t tempty_local = smem_u32(&sh.tempty[acc]);
      // the even CTA's MMA issuer waits for the epilogue warps of both CTAs
      const uint32_t tempty = PAIR ? peer_addr(tempty_local, 0) : tempty_local;
      auto release_acc = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (PAIR)
            mbar_arrive_cluster(tempty);
          else
            mbar_arrive(tempty);
        }
      };
      // Full tiles of the forward GEMMs leave through shared memory and TMA stores (one
      // elected thread issues them); the ragged last tile of an expert, whose rows past the
      // expert's count must not be written, and the backward modes store row by row.
      constexpr bool kStaged = MODE == kSwiGLU || MODE == kDown;
      const bool staged = kStaged && (int)rank * BM + BM <= t.rows;
      const bool leader = warp == 4 && lane == 0;
      if (staged) {
        const int orow0 = t.row0 + (int)rank * BM;
        const int rounds = MODE == kSwiGLU ? 1 : 2;   // 128 output columns per round
        const int col0 = MODE == kSwiGLU ? t.nt * (BN / 2) : t.nt * BN;
        const size_t grow = (size_t)(t.row0 + row);
#pragma unroll 1
        for (int rd = 0; rd < rounds; ++rd) {
          if (leader) bulk_wait_read();
          epilogue_bar();
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            float v[32];
            if constexpr (MODE == kSwiGLU) {
              uint32_t a[32], b[32];
              tmem_ld32(tb + c * 32, a);
              tmem_ld32(tb + BN / 2 + c * 32, b);
              tmem_wait(a);
              tmem_wait(b);
              if (c == 3) release_acc();
              if (args.ab_save && col0 + c * 32 < args.ndim) {
                const size_t q = (size_t)(args.poff_save[t.e] + (int)grow - sh.off[t.e]);
                bf16* o = args.ab_save + q * 2 * args.ndim + col0 + c * 32;
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(a[j]);
                store_row32(o, v);
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(b[j]);
                store_row32(o + args.ndim, v);
              }
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const float av = __uint_as_float(a[j]);
                const float bv = __uint_as_float(b[j]);
                v[j] = __fdividef(av, 1.0f + __expf(-av)) * bv;
              }
            } else {
              uint32_t a[32];
              const int cc = rd * 4 + c;
              tmem_ld32(tb + cc * 32, a);
              tmem_wait(a);
              if (cc == BN / 32 - 1) release_acc();
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(a[j]);
            }
            stage_row32(s_out, r, c, v);
          }
          fence_async_smem();
          epilogue_bar();
          if (leader) {
            const int cb = col0 + rd * 128;
            if (cb < args.ndim) tma_store_2d(&tmOut, s_out, cb, orow0);
            if (cb + 64 < args.ndim) tma_store_2d(&tmOut, s_out + kStageOutBytes / 2, cb + 64, orow0);
            bulk_commit();
          }
        }
      } else if constexpr (MODE == kSwiGLU || MODE == kStoreAB) {
        const int col0 = t.nt * (BN / 2);
        const size_t grow = (size_t)(t.row0 + row);
#pragma unroll 1
        for (int c = 0; c < BN / 64; ++c) {
          uint32_t a[32], b[32];
          tmem_ld32(tb + c * 32, a);
          tmem_ld32(tb + BN / 2 + c * 32, b);
          tmem_wait(a);
          tmem_wait(b);
          if (c == BN / 64 - 1) release_acc();
          if (row_ok && col0 + c * 32 < args.ndim) {
            float v[32];
            if constexpr (MODE == kSwiGLU) {
              if (args.ab_save) {
                const size_t q = (size_t)(args.poff_save[t.e] + (int)grow - sh.off[t.e]);
                bf16* o = args.ab_save + q * 2 * args.ndim + col0 + c * 32;
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(a[j]);
                store_row32(o, v);
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(b[j]);
                store_row32(o + args.ndim, v);
              }
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const float av = __uint_as_float(a[j]);
                const float bv = __uint_as_float(b[j]);
                v[j] = __fdividef(av, 1.0f + __expf(-av)) * bv;
              }
              store_row32(args.out + grow * args.ndim + col0 + c * 32, v);
            } else {
              // [a | b] row of 2 * ndim columns
              bf16* o = args.out + grow * 2 * args.ndim + col0 + c * 32;
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(a[j]);
              store_row32(o, v);
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(b[j]);
              store_row32(o + args.ndim, v);
            }
          }
        }
      } else if constexpr (MODE == kDh) {
        // dh' = g w2 for 256 columns of f; with the recomputed a, b of the same columns:
        //   h = SiLU(a) b,  partial <dh', h>,  da = G dh' b SiLU'(a),  db = G dh' SiLU(a),
        //   hw = G h  (G = this row's gate weight, 0 on padding rows)
        // A thread holds one row of the tile, so a, b and the three outputs pass through this
        // warp's 8 KB of the staging buffer: each 32-column block of 32 rows (64 bytes a row)
        // is read and written by the warp with 16-byte accesses covering 8 whole rows per
        // instruction, and each thread reads or writes its own row in shared memory (16-byte
        // chunk c of row i at chunk c ^ ((i / 2) % 4): no bank conflicts either way).
        const int col0 = t.nt * BN;
        const size_t grow = (size_t)(t.row0 + row);
        const float gate = row_ok ? args.wq[grow] : 0.f;
        uint8_t* wsm = smem + STAGES * C::kStageBytes + q * (kStageOutBytes / 4);
        const int rows_here = t.rows - q * 32;   // rows of this warp's 32 that exist
        auto slot = [](int i, int ch) { return i * 64 + 16 * (ch ^ ((i >> 1) & 3)); };
        float dot = 0.f;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t dr[32];
          tmem_ld32(tb + c * 32, dr);
          tmem_wait(dr);
          if (c == BN / 32 - 1) release_acc();
          const int col = col0 + c * 32;
          if (col >= args.ndim) continue;   // the same for the whole warp
          // a | b of the warp's 32 rows into shared memory (a at 0, b at 2 KB)
#pragma unroll
          for (int s8 = 0; s8 < 4; ++s8) {
            const int i = s8 * 8 + (lane >> 2), ch = lane & 3;
            if (i < rows_here) {
              const bf16* src = args.ab + (size_t)(t.row0 + q * 32 + i) * 2 * args.ndim + col + ch * 8;
              *reinterpret_cast<uint4*>(wsm + slot(i, ch)) = __ldg(reinterpret_cast<const uint4*>(src));
              *reinterpret_cast<uint4*>(wsm + 2048 + slot(i, ch)) =
                  __ldg(reinterpret_cast<const uint4*>(src + args.ndim));
            }
          }
          __syncwarp();
          float av[32], bv[32], o1[32], o2[32];
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            const uint4 ua = *reinterpret_cast<const uint4*>(wsm + slot(lane, ch));
            const uint4 ub = *reinterpret_cast<const uint4*>(wsm + 2048 + slot(lane, ch));
            const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&ua);
            const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&ub);
#pragma unroll
            for (int i2 = 0; i2 < 4; ++i2) {
              const float2 fa = __bfloat1622float2(pa[i2]), fb = __bfloat1622float2(pb[i2]);
              av[8 * ch + 2 * i2] = fa.x;
              av[8 * ch + 2 * i2 + 1] = fa.y;
              bv[8 * ch + 2 * i2] = fb.x;
              bv[8 * ch + 2 * i2 + 1] = fb.y;
            }
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float dh = __uint_as_float(dr[j]);
            const float sg = sigmoidf_(av[j]);
            const float si = av[j] * sg;
            const float h = si * bv[j];
            dot = fmaf(dh, h, dot);
            o1[j] = gate * dh * bv[j] * sg * (1.0f + av[j] * (1.0f - sg));
            o2[j] = gate * dh * si;
            bv[j] = gate * h;
          }
          __syncwarp();   // every row of a | b has been read before the outputs overwrite it
          // da at 0, db at 2 KB, hw at 4 KB; then out to global memory by whole rows
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint4 u1, u2, u3;
            u1.x = pack_bf16x2(o1[8 * ch + 0], o1[8 * ch + 1]);
            u1.y = pack_bf16x2(o1[8 * ch + 2], o1[8 * ch + 3]);
            u1.z = pack_bf16x2(o1[8 * ch + 4], o1[8 * ch + 5]);
            u1.w = pack_bf16x2(o1[8 * ch + 6], o1[8 * ch + 7]);
            u2.x = pack_bf16x2(o2[8 * ch + 0], o2[8 * ch + 1]);
            u2.y = pack_bf16x2(o2[8 * ch + 2], o2[8 * ch + 3]);
            u2.z = pack_bf16x2(o2[8 * ch + 4], o2[8 * ch + 5]);
            u2.w = pack_bf16x2(o2[8 * ch + 6], o2[8 * ch + 7]);
            u3.x = pack_bf16x2(bv[8 * ch + 0], bv[8 * ch + 1]);
            u3.y = pack_bf16x2(bv[8 * ch + 2], bv[8 * ch + 3]);
            u3.z = pack_bf16x2(bv[8 * ch + 4], bv[8 * ch + 5]);
            u3.w = pack_bf16x2(bv[8 * ch + 6], bv[8 * ch + 7]);
            *reinterpret_cast<uint4*>(wsm + slot(lane, ch)) = u1;
            *reinterpret_cast<uint4*>(wsm + 2048 + slot(lane, ch)) = u2;
            *reinterpret_cast<uint4*>(wsm + 4096 + slot(lane, ch)) = u3;
          }
          __syncwarp();
#pragma unroll
          for (int s8 = 0; s8 < 4; ++s8) {
            const int i = s8 * 8 + (lane >> 2), ch = lane & 3;
            if (i < rows_here) {
              const size_t oo = (size_t)(t.row0 + q * 32 + i) * args.ndim + col + ch * 8;
              *reinterpret_cast<uint4*>(args.da + oo) = *reinterpret_cast<const uint4*>(wsm + slot(i, ch));
              *reinterpret_cast<uint4*>(args.db + oo) =
                  *reinterpret_cast<const uint4*>(wsm + 2048 + slot(i, ch));
              *reinterpret_cast<uint4*>(args.hw + oo) =
                  *reinterpret_cast<const uint4*>(wsm + 4096 + slot(i, ch));
            }
          }
          __syncwarp();   // the next block's a | b may overwrite the outputs only after this
        }
        if (row_ok) args.dwp[grow * args.ntiles + t.nt] = dot;
      } else {
        // kDown, kDgradX: rows of the tile; kWgrad: rows of expert e's gradient
        const int col0 = t.nt * BN;
        bf16* orow;
        if constexpr (MODE == kWgrad)
          orow = args.out + ((size_t)t.e * args.mdim + (size_t)wrow) * args.ndim + col0;
        else
          orow = args.out + (size_t)(t.row0 + row) * args.ndim + col0;
        const bool empty_k = MODE == kWgrad && t.rows == 0;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t a[32];
          tmem_ld32(tb + c * 32, a);
          tmem_wait(a);
          if (c == BN / 32 - 1) release_acc();
          if (row_ok && col0 + c * 32 < args.ndim) {
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = empty_k ? 0.f : __uint_as_float(a[j]);
            store_row32(orow + c * 32, v);
          }
        }
      }
      if (++acc == ACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // the TMA stores must finish reading the staging buffer (and land) before the CTA exits
    if (warp == 4 && lane == 0) bulk_wait_all();
  }

  __syncwarp();
  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync_all();   // neither CTA leaves while the other may still touch its memory
  else
    __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc<PAIR>(tmem_base);
  }
}

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------

template <int MODE, bool PAIR>
cudaError_t set_smem_attr() {
  static PerDeviceSetting setting;
  return setting.get([] {
    return cudaFuncSetAttribute(grouped_gemm_tc_kernel<MODE, PAIR>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem_bytes<PAIR>());
  });
}

// Clusters of two that can be resident at once (0 if the pair form cannot run here).
template <int MODE>
int max_pairs() {
  static int cache[64];
  static bool done[64] = {false};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!done[dev]) {
    int clusters = 0;
    if (set_smem_attr<MODE, true>() == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(2 * device_sm_count(), 1, 1);
      cfg.blockDim = dim3(256, 1, 1);
      cfg.dynamicSmemBytes = smem_bytes<true>();
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&clusters, grouped_gemm_tc_kernel<MODE, true>, &cfg) !=
          cudaSuccess)
        clusters = 0;
      (void)cudaGetLastError();
    }
    cache[dev] = clusters;
    done[dev] = true;
  }
  return cache[dev];
}

std::atomic<int> g_tc_form{MOE_TC_FORM_AUTO};

// Unless a form was forced with moe_set_tc_form: the pair form for GEMM2 (w2) when the
// experts hold on average at least one full 256-row tile, for GEMM1 (w1|w3 + SwiGLU) when
// they hold at least two; the single form otherwise.  Measured on B300 with interleaved runs
// at the prefill sizes (d = 4096, f = 14336, clocks held down by the power cap): at T = 4096
// the pair form runs GEMM1 6 % and GEMM2 12 % faster, at T = 16384 (skewed routing) GEMM1
// equally fast and GEMM2 9 % faster.  GEMM1's shorter reduction (K = 4096) gains less: its
// 256-row tiles waste more rows on the experts' ragged last tiles.
template <int MODE>
inline bool want_pair(int A, int n) {
  const int form = g_tc_form.load(std::memory_order_relaxed);
  if (form == MOE_TC_FORM_SINGLE) return false;
  if (form == MOE_TC_FORM_PAIR) return true;
  if (MODE == kDown) return (long long)A >= 256ll * n;
  if (MODE == kSwiGLU) return (long long)A >= 512ll * n;
  if (MODE == kWgrad) return true;   // M and N are weight dimensions: no row is wasted
  return false;
}

// Single-CTA launch over at most `tiles` tiles.
template <int MODE>
cudaError_t launch_single(const CUtensorMap& mA, const CUtensorMap& mA2, const CUtensorMap& mB0,
                          const CUtensorMap& mB1, const CUtensorMap& mOut, const TcArgs& a,
                          long long tiles, cudaStream_t s) {
  cudaError_t e = set_smem_attr<MODE, false>();
  if (e != cudaSuccess) return e;
  const int sms = device_sm_count();
  const int grid = (int)(tiles < sms ? (tiles > 0 ? tiles : 1) : sms);
  grouped_gemm_tc_kernel<MODE, false><<<grid, 256, smem_bytes<false>(), s>>>(mA, mA2, mB0, mB1,
                                                                           mOut, a);
  return cudaGetLastError();
}

// CTA-pair launch over at most `tiles` tiles on at most `pairs` resident clusters of two.
template <int MODE>
cudaError_t launch_pair(const CUtensorMap& mA, const CUtensorMap& mA2, const CUtensorMap& mB0,
                        const CUtensorMap& mB1, const CUtensorMap& mOut, const TcArgs& a,
                        long long tiles, int pairs, cudaStream_t s) {
  const int units = (int)(tiles < pairs ? (tiles > 0 ? tiles : 1) : pairs);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * units, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes<true>();
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, grouped_gemm_tc_kernel<MODE, true>, mA, mA2, mB0, mB1, mOut, a);
}

template <int MODE>
cudaError_t launch_gemm(const CUtensorMap& mA, const CUtensorMap& mB0, const CUtensorMap& mB1,
                        const CUtensorMap& mOut, const TcArgs& a, int A, cudaStream_t s) {
  const int pairs = want_pair<MODE>(A, a.n) ? max_pairs<MODE>() : 0;
  if (pairs > 0) {
    const long long tiles = ((long long)(A + 255) / 256 + a.n) * a.ntiles;
    return launch_pair<MODE>(mA, mA, mB0, mB1, mOut, a, tiles, pairs, s);
  }
  const long long tiles = ((long long)(A + BM - 1) / BM + a.n) * a.ntiles;
  return launch_single<MODE>(mA, mA, mB0, mB1, mOut, a, tiles, s);
}

}  // namespace

void set_tc_form(int form) { g_tc_form.store(form, std::memory_order_relaxed); }

cudaError_t launch_up_tc(const bf16* x_perm, const int32_t* offsets, const bf16* w1, const bf16* w3,
                         int A, int d, int f, int n, bf16* h, uint32_t* status,
                         unsigned long long wait_ns, cudaStream_t s, bf16* ab_save,
                         const int32_t* poff_save) {
  if (A == 0) return cudaSuccess;
  CUtensorMap mA, mW1, mW3, mH;
  if (!make_map(&mA, x_perm, (uint64_t)A, (uint64_t)d, BM) ||
      !make_map(&mW1, w1, (uint64_t)n * f, (uint64_t)d, BN / 2) ||
      !make_map(&mW3, w3, (uint64_t)n * f, (uint64_t)d, BN / 2) ||
      !make_map(&mH, h, (uint64_t)A, (uint64_t)f, BM))
    return cudaErrorInvalidValue;
  TcArgs a = {};
  a.offsets = offsets;
  a.mrows = A;
  a.n = n;
  a.kdim = d;
  a.ndim = f;
  a.ntiles = (f + BN / 2 - 1) / (BN / 2);
  a.out = h;
  a.status = status;
  a.wait_ns = wait_ns;
  a.ab_save = ab_save;
  a.poff_save = poff_save;
  return launch_gemm<kSwiGLU>(mA, mW1, mW3, mH, a, A, s);
}

cudaError_t launch_down_tc(const bf16* h, const int32_t* offsets, const bf16* w2, int A, int d,
                           int f, int n, bf16* y_perm, uint32_t* status, unsigned long long wait_ns,
                           cudaStream_t s) {
  if (A == 0) return cudaSuccess;
  // the pair form loads 128 of the 256 rows of a w2 tile per CTA, the single form all 256
  const uint32_t brows = want_pair<kDown>(A, n) && max_pairs<kDown>() > 0 ? BN / 2 : BN;
  CUtensorMap mA, mW2, mY;
  if (!make_map(&mA, h, (uint64_t)A, (uint64_t)f, BM) ||
      !make_map(&mW2, w2, (uint64_t)n * d, (uint64_t)f, brows) ||
      !make_map(&mY, y_perm, (uint64_t)A, (uint64_t)d, BM))
    return cudaErrorInvalidValue;
  TcArgs a = {};
  a.offsets = offsets;
  a.mrows = A;
  a.n = n;
  a.kdim = f;
  a.ndim = d;
  a.ntiles = (d + BN - 1) / BN;
  a.out = y_perm;
  a.status = status;
  a.wait_ns = wait_ns;
  return launch_gemm<kDown>(mA, mW2, mW2, mY, a, A, s);
}

// ------------------------------------------------------------------------------------------
// backward launchers (rows in the expert-padded layout: every expert's segment of
// `offsets` is a multiple of 128 rows; rows_max bounds the padded row count)
// ------------------------------------------------------------------------------------------
int bwd_dh_ntiles(int f) { return (f + BN - 1) / BN; }

cudaError_t launch_bwd_store_ab(const bf16* x_pad, const int32_t* poff, const bf16* w1,
                                const bf16* w3, int rows_max, int d, int f, int n, bf16* ab,
                                uint32_t* status, unsigned long long wait_ns, cudaStream_t s) {
  if (rows_max == 0) return cudaSuccess;
  CUtensorMap mA, mW1, mW3;
  if (!make_map(&mA, x_pad, (uint64_t)rows_max, (uint64_t)d, BM) ||
      !make_map(&mW1, w1, (uint64_t)n * f, (uint64_t)d, BN / 2) ||
      !make_map(&mW3, w3, (uint64_t)n * f, (uint64_t)d, BN / 2))
    return cudaErrorInvalidValue;
  TcArgs a = {};
  a.offsets = poff;
  a.mrows = rows_max;
  a.n = n;
  a.kdim = d;
  a.ndim = f;
  a.ntiles = (f + BN / 2 - 1) / (BN / 2);
  a.out = ab;
  a.status = status;
  a.wait_ns = wait_ns;
  return launch_single<kStoreAB>(mA, mA, mW1, mW3, mA, a, (long long)(rows_max / BM) * a.ntiles,
                                 s);
}

cudaError_t launch_bwd_dh(const bf16* g_pad, const int32_t* poff, const bf16* w2, const bf16* ab,
                          const float* wq, int rows_max, int d, int f, int n, float* dwp, bf16* da,
                          bf16* db, bf16* hw, uint32_t* status, unsigned long long wait_ns,
                          cudaStream_t s) {
  if (rows_max == 0) return cudaSuccess;
  CUtensorMap mA, mW2;
  if (!make_map(&mA, g_pad, (uint64_t)rows_max, (uint64_t)d, BM) ||
      !make_map(&mW2, w2, (uint64_t)n * d, (uint64_t)f, 64))
    return cudaErrorInvalidValue;
  TcArgs a = {};
  a.offsets = poff;
  a.mrows = rows_max;
  a.n = n;
  a.kdim = d;
  a.ndim = f;
  a.ntiles = bwd_dh_ntiles(f);
  a.brows = d;
  a.ab = ab;
  a.wq = wq;
  a.dwp = dwp;
  a.da = da;
  a.db = db;
  a.hw = hw;
  a.status = status;
  a.wait_ns = wait_ns;
  return launch_single<kDh>(mA, mA, mW2, mW2, mA, a, (long long)(rows_max / BM) * a.ntiles, s);
}

cudaError_t launch_bwd_dgrad_x(const bf16* da, const bf16* db, const int32_t* poff, const bf16* w1,
                               const bf16* w3, int rows_max, int d, int f, int n, bf16* dx_pad,
                               uint32_t* status, unsigned long long wait_ns, cudaStream_t s) {
  if (rows_max == 0) return cudaSuccess;
  CUtensorMap mDa, mDb, mW1, mW3;
  if (!make_map(&mDa, da, (uint64_t)rows_max, (uint64_t)f, BM) ||
      !make_map(&mDb, db, (uint64_t)rows_max, (uint64_t)f, BM) ||
      !make_map(&mW1, w1, (uint64_t)n * f, (uint64_t)d, 64) ||
      !make_map(&mW3, w3, (uint64_t)n * f, (uint64_t)d, 64))
    return cudaErrorInvalidValue;
  TcArgs a = {};
  a.offsets = poff;
  a.mrows = rows_max;
  a.n = n;
  a.kdim = 2 * f;
  a.kb_split = f / BK;
  a.ndim = d;
  a.ntiles = (d + BN - 1) / BN;
  a.brows = f;
  a.out = dx_pad;
  a.status = status;
  a.wait_ns = wait_ns;
  return launch_single<kDgradX>(mDa, mDb, mW1, mW3, mDa, a,
                                (long long)(rows_max / BM) * a.ntiles, s);
}

cudaError_t launch_bwd_wgrad(const bf16* P, const bf16* Q, const int32_t* poff, int rows_max,
                             int M, int N, int n, bf16* dW, uint32_t* status,
                             unsigned long long wait_ns, cudaStream_t s) {
  CUtensorMap mP, mQ;
  // rows_max >= 1 keeps the maps valid when no expert has rows (every tile then writes zeros)
  const uint64_t rows = rows_max > 0 ? (uint64_t)rows_max : 1;
  if (!make_map(&mP, P, rows, (uint64_t)M, 64) || !make_map(&mQ, Q, rows, (uint64_t)N, 64))
    return cudaErrorInvalidValue;
  TcArgs a = {};
  a.offsets = poff;
  a.mrows = rows_max;
  a.n = n;
  a.kdim = 0;
  a.mdim = M;
  a.ndim = N;
  a.ntiles = (N + BN - 1) / BN;
  a.out = dW;
  a.status = status;
  a.wait_ns = wait_ns;
  const int pairs = want_pair<kWgrad>(rows_max, n) ? max_pairs<kWgrad>() : 0;
  if (pairs > 0) {
    a.mtiles_w = (M + 2 * BM - 1) / (2 * BM);
    return launch_pair<kWgrad>(mP, mP, mQ, mQ, mP, a, (long long)n * a.mtiles_w * a.ntiles, pairs,
                               s);
  }
  a.mtiles_w = (M + BM - 1) / BM;
  return launch_single<kWgrad>(mP, mP, mQ, mQ, mP, a, (long long)n * a.mtiles_w * a.ntiles, s);
}

}  // namespace moe
