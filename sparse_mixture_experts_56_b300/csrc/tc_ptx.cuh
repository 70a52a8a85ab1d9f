// PTX building blocks shared by the tcgen05 kernels of libmoe.so (grouped expert GEMMs,
// attention): mbarriers with bounded waits, TMA tile loads and stores, shared-memory matrix
// descriptors (128-byte swizzle, K-major and MN-major), TMEM loads, and the host-side
// encoding of 2-D bf16 tensor maps.
#pragma once

#include <cuda.h>

#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace ptx {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.b32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"((uint64_t)map), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)map) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row atoms 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) |
         (1ull << 46) | (2ull << 61);
}

// The descriptor of the same layout `bytes` further on: the start address is the low field
// (16-byte units, shared-memory addresses below 256 KB), so a byte offset is one 64-bit add.
// Issue loops build their descriptors once and step them this way; recomputing the full
// descriptor before every MMA measurably slowed the MMA issue (N = 256: about 10 %).
__device__ __forceinline__ uint64_t desc_add(uint64_t desc, uint32_t bytes) {
  return desc + (uint64_t)(bytes >> 4);
}

// MN-major, 128-byte swizzle: each TMA box is 64 K-rows of 64 contiguous M/N elements (8 KB);
// boxes for successive 64-element M/N chunks sit 8 KB apart (leading byte offset), 8-row K
// groups 1024 bytes apart (stride byte offset).
constexpr uint32_t kMnChunkBytes = 64 * 64 * 2;
__device__ __forceinline__ uint64_t sw128_mn_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(kMnChunkBytes >> 4) << 16) |
         ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

#define MOE_R32(r)                                                                               \
  "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),           \
      "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),   \
      "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),             \
      "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),             \
      "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
#define MOE_P32(r)                                                                               \
  "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),           \
      "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),   \
      "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),             \
      "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),             \
      "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : MOE_R32(r)
      : "r"(taddr));
}
// Waits for the thread's outstanding tcgen05.ld; the registers are threaded through the asm
// so that no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : MOE_P32(r)::"memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   (uint64_t)map),
               "r"(src), "r"(c0), "r"(c1)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// a TMA store source may be overwritten once the stores issued so far have read it
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void raise_abort(volatile int* abort, uint32_t* status) {
  if (!*abort) {
    *abort = 1;
    atomicOr(status, kDevErrTimeout);
  }
}

// Waits for the phase of parity `parity` of `bar`; false on abort or after limit_ns.
static __device__ __noinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort,
                                        uint64_t limit_ns) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = gtimer();
  for (;;) {
    if (mbar_test(bar, parity)) return true;
    if (*abort) return false;
    if (gtimer() - t0 > limit_ns) return false;
  }
}

// wait_phase with the common case inline: a phase that has already completed costs one
// try_wait instead of a call (the call saves and restores registers, a few hundred cycles in
// a kernel with a large register budget).
__device__ __forceinline__ bool wait_fast(uint32_t bar, uint32_t parity, volatile int* abort,
                                          uint64_t limit_ns) {
  return mbar_test(bar, parity) || wait_phase(bar, parity, abort, limit_ns);
}

// wait_phase for a role that waits long and whose wake-up can be a little late (an epilogue
// waiting for the next accumulator while the MMAs of a whole tile run): between tests the
// thread sleeps, 64 ns at first and doubling up to 2 us, instead of polling.  In a GEMM held
// back by the power limit the polling threads' power is taken from the tensor cores (1 % of
// the layer step at 16384 tokens in interleaved runs).
static __device__ __noinline__ bool wait_phase_sleepy(uint32_t bar, uint32_t parity,
                                                      volatile int* abort, uint64_t limit_ns) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = gtimer();
  uint32_t ns = 64;
  for (;;) {
    __nanosleep(ns);
    if (mbar_test(bar, parity)) return true;
    if (*abort) return false;
    if (gtimer() - t0 > limit_ns) return false;
    if (ns < 2048) ns <<= 1;
  }
}

// Same, ignoring the abort flag (used to drain work already in flight).
static __device__ __noinline__ bool drain_phase(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = gtimer();
  for (;;) {
    if (mbar_test(bar, parity)) return true;
    if (gtimer() - t0 > limit_ns) return false;
  }
}

// ------------------------------------------------------------------------------------------
// host side: 2-D bf16 tensor maps
// ------------------------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D bf16 tensor [rows, cols] (cols contiguous), boxes of [box_rows, 64], 128-byte swizzle.
inline bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64u, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace ptx
}  // namespace moe
