// Grouping of the T*k token->expert assignments by expert, and the row gather that builds the
// expert-ordered copy of x.
//   Experts whose gate is 0 are not computed ("Mixtral 8x7B: 疎な専門家混合言語モデル",
//   ja.news.hada.io, MoEレイヤーの計算方式); each expert receives a variable number of tokens
//   and the outputs go back to the original token positions (same page, 実装と推論効率).
//
// Outputs: expert_offsets[n+1] (exclusive prefix sum of per-expert counts), perm[p] = the
// assignment a = t*k + slot at position p, positions ordered by (expert, a), and
// inv_perm[a] = p.  Stable and deterministic: no atomics decide any position.
// An expert index outside [0, n) (a caller's mistake, reported through the status word) puts
// its assignment in a trailing bucket after every expert: expert_offsets[n] counts the valid
// assignments only, and perm / inv_perm stay a permutation of [0, T*k), so that every row
// index a later step reads from them is in bounds.
//
// A block of 32 warps handles a chunk of kPermuteChunk assignments; warp w owns a contiguous
// sub-chunk.  Ranks within a 32-wide round come from __match_any_sync + popc of the lanes
// below; per-(warp, expert) counters in shared memory carry the rank across rounds.  One
// block covers the whole problem when T*k <= kPermuteChunk (a single launch); otherwise a
// count kernel, a scan kernel and a scatter kernel run over the chunks.
#include <cuda.h>

#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kWarps = 32;

struct ChunkBounds {
  int begin, end;
};

__device__ __forceinline__ ChunkBounds warp_range(int chunk_begin, int chunk_end, int warp) {
  const int len = chunk_end - chunk_begin;
  int per = (len + kWarps - 1) / kWarps;
  per = (per + 31) & ~31;
  const int b = chunk_begin + warp * per;
  const int e = min(chunk_end, b + per);
  return {b, e};
}

// Zeroes the kMaxExperts + 1 counters of one warp's row.
__device__ __forceinline__ void clear_row(int* row, int lane) {
  row[lane] = 0;
  if (lane == 0) row[kMaxExperts] = 0;
}

// A warp's range holds at most kPermuteChunk / kWarps = 1024 assignments: 32 rounds of 32.
// Each lane loads the raw indices of a batch of 16 rounds first, with nothing between the
// loads so that they are all in flight together; the rounds then classify them (reporting
// bad ones) and run from registers.
constexpr int kBatch = 16;
static_assert(kPermuteChunk / kWarps % (32 * kBatch) == 0, "a warp's range is whole batches");

__device__ __forceinline__ void load_batch(const int32_t* __restrict__ idx, int base, int end,
                                           int lane, int (&v)[kBatch]) {
#pragma unroll
  for (int j = 0; j < kBatch; ++j) {
    const int i = base + 32 * j + lane;
    v[j] = i < end ? __ldg(idx + i) : 0;
  }
}

// Bucket of assignment i with raw expert index v: the expert, n (the trailing bucket) for an
// index outside [0, n), which is reported when `status` is not null, or -1 past the range.
__device__ __forceinline__ int bucket_of(int v, int i, int end, int n, uint32_t* status) {
  if (i >= end) return -1;
  if (v < 0 || v >= n) {
    if (status) atomicOr(status, kDevErrIndex);
    return n;
  }
  return v;
}

// cnt[w][e] <- number of assignments of warp w's range that go to bucket e.
__device__ void count_warp(const int32_t* __restrict__ idx, ChunkBounds r, int n, int lane,
                           int* cnt_row, uint32_t* status) {
  for (int b0 = r.begin; b0 < r.end; b0 += 32 * kBatch) {
    int ev[kBatch];
    load_batch(idx, b0, r.end, lane, ev);
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int base = b0 + 32 * j;
      if (base >= r.end) break;
      const int e = bucket_of(ev[j], base + lane, r.end, n, status);
      const unsigned m = __match_any_sync(0xffffffffu, e);
      if (e >= 0 && lane == __ffs(m) - 1) cnt_row[e] += __popc(m);
      __syncwarp();
    }
  }
}

// Writes perm / inv_perm for warp w's range; run_row[e] holds the first position of the
// warp's assignments to expert e and is advanced as rounds go by.
__device__ void scatter_warp(const int32_t* __restrict__ idx, ChunkBounds r, int n, int lane,
                             int* run_row, int32_t* __restrict__ perm,
                             int32_t* __restrict__ inv_perm, uint32_t* status) {
  const unsigned lt = (1u << lane) - 1u;
  for (int b0 = r.begin; b0 < r.end; b0 += 32 * kBatch) {
    int ev[kBatch];
    load_batch(idx, b0, r.end, lane, ev);
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int base = b0 + 32 * j;
      if (base >= r.end) break;
      const int i = base + lane;
      const int e = bucket_of(ev[j], i, r.end, n, status);
      const unsigned m = __match_any_sync(0xffffffffu, e);
      int pos = 0;
      if (e >= 0) {
        pos = run_row[e] + __popc(m & lt);
        perm[pos] = i;
        inv_perm[i] = pos;
      }
      __syncwarp();
      if (e >= 0 && lane == __ffs(m) - 1) run_row[e] += __popc(m);
      __syncwarp();
    }
  }
}

// Single block: count, scan, scatter.
__global__ void __launch_bounds__(1024) permute_single_kernel(const int32_t* __restrict__ idx,
                                                              int A, int n,
                                                              int32_t* __restrict__ offsets,
                                                              int32_t* __restrict__ perm,
                                                              int32_t* __restrict__ inv_perm,
                                                              uint32_t* status) {
  __shared__ int cnt[kWarps][kMaxExperts + 1];
  __shared__ int ebase[kMaxExperts + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  clear_row(cnt[warp], lane);
  __syncwarp();
  const ChunkBounds r = warp_range(0, A, warp);
  count_warp(idx, r, n, lane, cnt[warp], status);
  __syncthreads();
  if (warp == 0) {
    // lane = bucket (bucket 32, the trailing one when n = 32, in lane 0's second counter):
    // exclusive prefix over warps, then over buckets
    const bool second = lane == 0 && n == kMaxExperts;
    int run = 0, run2 = 0;
    for (int w = 0; w < kWarps; ++w) {
      const int c = cnt[w][lane];
      cnt[w][lane] = run;
      run += c;
      if (second) {
        const int c2 = cnt[w][kMaxExperts];
        cnt[w][kMaxExperts] = run2;
        run2 += c2;
      }
    }
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const int excl = incl - run;
    const int total32 = __shfl_sync(0xffffffffu, incl, 31);
    ebase[lane] = excl;
    if (lane == 0) ebase[kMaxExperts] = total32;
    // offsets[e] for e < n, and offsets[n] = the trailing bucket's start = valid assignments
    if (lane <= n) offsets[lane] = excl;
    if (second) offsets[kMaxExperts] = total32;
  }
  __syncthreads();
  cnt[warp][lane] += ebase[lane];
  if (lane == 0) cnt[warp][kMaxExperts] += ebase[kMaxExperts];
  __syncwarp();
  scatter_warp(idx, r, n, lane, cnt[warp], perm, inv_perm, status);
}

// Multi-block, step 1: per-block counts -> block_cnt[b * n + e].
__global__ void __launch_bounds__(1024) permute_count_kernel(const int32_t* __restrict__ idx, int A,
                                                             int n, int32_t* __restrict__ block_cnt,
                                                             uint32_t* status) {
  __shared__ int cnt[kWarps][kMaxExperts + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  clear_row(cnt[warp], lane);
  __syncwarp();
  const int cb = blockIdx.x * kPermuteChunk, ce = min(A, cb + kPermuteChunk);
  count_warp(idx, warp_range(cb, ce, warp), n, lane, cnt[warp], status);
  __syncthreads();
  if (warp == 0) {
    for (int b = lane; b <= n; b += 32) {
      int s = 0;
      for (int w = 0; w < kWarps; ++w) s += cnt[w][b];
      block_cnt[blockIdx.x * (n + 1) + b] = s;
    }
  }
}

// Multi-block, step 2 (one warp): block_base[b * (n+1) + e] = offsets[e] + counts of bucket e
// in blocks < b, for the buckets e = 0..n (n: the trailing bucket of bad indices).
__global__ void permute_scan_kernel(const int32_t* __restrict__ block_cnt, int nblocks, int n,
                                    int32_t* __restrict__ block_base,
                                    int32_t* __restrict__ offsets) {
  const int lane = threadIdx.x & 31;
  const int nb1 = n + 1;
  const bool first = lane < nb1, second = lane + 32 < nb1;   // second: bucket 32 in lane 0
  int run = 0, run2 = 0;
  for (int b = 0; b < nblocks; ++b) {
    if (first) {
      const int c = block_cnt[b * nb1 + lane];
      block_base[b * nb1 + lane] = run;
      run += c;
    }
    if (second) {
      const int c = block_cnt[b * nb1 + lane + 32];
      block_base[b * nb1 + lane + 32] = run2;
      run2 += c;
    }
  }
  int incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  const int excl = incl - run;
  const int total32 = __shfl_sync(0xffffffffu, incl, 31);
  if (first) {
    offsets[lane] = excl;
    for (int b = 0; b < nblocks; ++b) block_base[b * nb1 + lane] += excl;
  }
  if (second) {
    offsets[lane + 32] = total32;
    for (int b = 0; b < nblocks; ++b) block_base[b * nb1 + lane + 32] += total32;
  }
}

// Multi-block, step 3: recount per warp, add the block base, scatter.
__global__ void __launch_bounds__(1024) permute_scatter_kernel(const int32_t* __restrict__ idx,
                                                               int A, int n,
                                                               const int32_t* __restrict__ block_base,
                                                               int32_t* __restrict__ perm,
                                                               int32_t* __restrict__ inv_perm,
                                                               uint32_t* status) {
  __shared__ int cnt[kWarps][kMaxExperts + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  clear_row(cnt[warp], lane);
  __syncwarp();
  const int cb = blockIdx.x * kPermuteChunk, ce = min(A, cb + kPermuteChunk);
  const ChunkBounds r = warp_range(cb, ce, warp);
  // bad indices were already reported by the count kernel
  count_warp(idx, r, n, lane, cnt[warp], nullptr);
  __syncthreads();
  if (warp == 0) {
    for (int b = lane; b <= n; b += 32) {
      int run = block_base[blockIdx.x * (n + 1) + b];
      for (int w = 0; w < kWarps; ++w) {
        const int c = cnt[w][b];
        cnt[w][b] = run;
        run += c;
      }
    }
  }
  __syncthreads();
  scatter_warp(idx, r, n, lane, cnt[warp], perm, inv_perm, nullptr);
  (void)status;
}

// x_perm[p] = x[perm[p] / k], 16-byte vectors when the row allows it.  A perm entry outside
// [0, T*k) (a caller's buffer that no permutation wrote) gives a zero row instead of a read
// out of bounds.
__global__ void __launch_bounds__(256) gather_rows_vec_kernel(const uint4* __restrict__ x,
                                                              const int32_t* __restrict__ perm,
                                                              int A, int k, int row_vecs,
                                                              uint4* __restrict__ x_perm) {
  for (int p = blockIdx.x; p < A; p += gridDim.x) {
    const int a = __ldg(perm + p);
    const bool ok = a >= 0 && a < A;
    const uint4* src = x + (size_t)(ok ? a / k : 0) * row_vecs;
    uint4* dst = x_perm + (size_t)p * row_vecs;
    for (int c = threadIdx.x; c < row_vecs; c += blockDim.x)
      dst[c] = ok ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
  }
}

__global__ void __launch_bounds__(256) gather_rows_byte_kernel(const uint8_t* __restrict__ x,
                                                               const int32_t* __restrict__ perm,
                                                               int A, int k, size_t row_bytes,
                                                               uint8_t* __restrict__ x_perm) {
  for (int p = blockIdx.x; p < A; p += gridDim.x) {
    const int a = __ldg(perm + p);
    const bool ok = a >= 0 && a < A;
    const size_t t = ok ? (size_t)(a / k) : 0;
    for (size_t c = threadIdx.x; c < row_bytes; c += blockDim.x)
      x_perm[(size_t)p * row_bytes + c] = ok ? x[t * row_bytes + c] : (uint8_t)0;
  }
}

}  // namespace

int permute_blocks(long long A) { return (int)((A + kPermuteChunk - 1) / kPermuteChunk); }

size_t permute_scratch_words(long long A, int n) {
  const int nb = permute_blocks(A);
  return nb <= 1 ? 0 : (size_t)2 * nb * (n + 1);
}

cudaError_t launch_permute(const int32_t* idx, int A, int n, int32_t* offsets, int32_t* perm,
                           int32_t* inv_perm, int32_t* scratch, uint32_t* status, cudaStream_t s) {
  const int nb = permute_blocks(A);
  if (nb <= 1) {
    permute_single_kernel<<<1, 1024, 0, s>>>(idx, A, n, offsets, perm, inv_perm, status);
    return cudaGetLastError();
  }
  int32_t* block_cnt = scratch;
  int32_t* block_base = scratch + permute_scratch_words(A, n) / 2;
  permute_count_kernel<<<nb, 1024, 0, s>>>(idx, A, n, block_cnt, status);
  permute_scan_kernel<<<1, 32, 0, s>>>(block_cnt, nb, n, block_base, offsets);
  permute_scatter_kernel<<<nb, 1024, 0, s>>>(idx, A, n, block_base, perm, inv_perm, status);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const void* x, const int32_t* perm, int A, int k, size_t row_bytes,
                               void* x_perm, cudaStream_t s) {
  if (A == 0) return cudaSuccess;
  const int cap = device_sm_count() * 8;
  const int grid = A < cap ? A : cap;
  if (row_bytes % 16 == 0 && ((uintptr_t)x % 16) == 0 && ((uintptr_t)x_perm % 16) == 0) {
    gather_rows_vec_kernel<<<grid, 256, 0, s>>>((const uint4*)x, perm, A, k, (int)(row_bytes / 16),
                                                (uint4*)x_perm);
  } else {
    gather_rows_byte_kernel<<<grid, 256, 0, s>>>((const uint8_t*)x, perm, A, k, row_bytes,
                                                 (uint8_t*)x_perm);
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------------
// Allocation-free permutation: the same launches as launch_permute, with the per-block
// counts and the status word in a fixed array of this library instead of a workspace.
// ---------------------------------------------------------------------------------------
namespace {

constexpr int kNoAllocMaxBlocks = 128;  // T*k up to 128 * 32768 = 4,194,304 assignments
constexpr int kNoAllocStatusWords = 64;  // the status word, padded to 256 bytes
constexpr int kNoAllocWords = kNoAllocStatusWords + 2 * kNoAllocMaxBlocks * (kMaxExperts + 1);

// Shared by every call on a device; holds the last call's contents.
static __device__ __align__(256) int32_t g_noalloc_scratch[kNoAllocWords];

struct NoAllocSlot {
  int32_t* ptr = nullptr;
  unsigned long long ctx_id = 0;   // the context the address belongs to
  bool valid = false;
};
std::mutex g_noalloc_mu;
NoAllocSlot g_noalloc_slot[64];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Process-unique id of the calling thread's current CUDA context (false if there is none or
// the driver lacks the query).  Ids are never reused within a process, so an id that differs
// from the cached one means a new context: another one made current, or the device's primary
// context re-created after cudaDeviceReset (which unloads this library's device array too).
bool current_ctx_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext c = nullptr;
  if (!get_current || !get_id || get_current(&c) != CUDA_SUCCESS || !c) return false;
  return get_id(c, id) == CUDA_SUCCESS;
}

// Device address of the array in the current context.  Looked up with cudaGetSymbolAddress
// once per context (the name is only a host-side stand-in and must never be handed to a
// kernel itself) and looked up again whenever the current context is not the one the cached
// address belongs to.
cudaError_t noalloc_scratch(int32_t** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocSlot& slot = g_noalloc_slot[dev];
  unsigned long long id = 0;
  if (!slot.valid || !current_ctx_id(&id) || id != slot.ctx_id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);   // also makes the context current
    if (e != cudaSuccess) {
      slot.valid = false;
      return e;
    }
    slot.ptr = static_cast<int32_t*>(p);
    slot.valid = current_ctx_id(&slot.ctx_id);   // without an id, look up again next call
  }
  *out = slot.ptr;
  return cudaSuccess;
}

}  // namespace

}  // namespace moe

extern "C" moe_status moe_permute_noalloc(const int32_t* topk_idx, int T, int k, int n,
                                          int32_t* expert_offsets, int32_t* perm,
                                          int32_t* inv_perm, void* stream) {
  using namespace moe;
  if (T < 0 || n < 1 || n > kMaxExperts || k < 1 || k > n) return MOE_ERR_INVALID_ARG;
  const long long A = (long long)T * k;
  if (A >= (1ll << 31)) return MOE_ERR_INVALID_ARG;
  if (!expert_offsets || (A > 0 && (!topk_idx || !perm || !inv_perm))) return MOE_ERR_INVALID_ARG;
  if (permute_blocks(A) > kNoAllocMaxBlocks) return MOE_ERR_UNSUPPORTED;
  int32_t* scratch = nullptr;
  if (noalloc_scratch(&scratch) != cudaSuccess || !scratch) return MOE_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t* status = reinterpret_cast<uint32_t*>(scratch);
  // the status word must start at zero; the per-block counts are written before being read
  if (cudaMemsetAsync(status, 0, sizeof(uint32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
  const cudaError_t e = launch_permute(topk_idx, (int)A, n, expert_offsets, perm, inv_perm,
                                       scratch + kNoAllocStatusWords, status, s);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
