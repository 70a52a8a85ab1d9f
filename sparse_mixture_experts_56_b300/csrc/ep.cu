// Expert parallelism (EP): the bookkeeping a rank needs around the two all-to-all exchanges.
//   Tokens that an expert must process are sent to the GPU holding that expert, and the
//   expert outputs return to the original token positions (newsflash.city digest, section
//   "专家层的混合"; "Mixtral 8x7B: 疎な専門家混合言語モデル" (ja.news.hada.io), section
//   "実装と推論効率").
// Rank g holds the experts [g*E, (g+1)*E).  Its receive buffer holds, source rank after source
// rank, each source's rows for those experts in the source's grouping order (expert, then
// assignment).  moe_ep_regroup orders those rows by local expert, then by source, which is the
// row order the grouped expert GEMMs take; moe_gather_rows moves rows by an index vector
// (into that order before the experts, and back to receive order after them).
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kMaxSources = 1024;

// One block per (source s, local expert j): the block's rows sit at receive positions
// src_base(s) + sum_{j' < j} c[s][j'] + i and at grouped positions
// local_offsets[j] + sum_{s' < s} c[s'][j] + i, i < c[s][j].  Counts are clamped to >= 0, the
// sums taken in 64 bits, and positions outside [0, R) are never written.
__global__ void __launch_bounds__(256) ep_regroup_kernel(const int32_t* __restrict__ counts,
                                                         int G, int E, int R,
                                                         int32_t* __restrict__ local_offsets,
                                                         int32_t* __restrict__ row_map,
                                                         int32_t* __restrict__ inv_row_map) {
  const int s = blockIdx.x / E, j = blockIdx.x % E;
  __shared__ long long s_recv0, s_group0;
  __shared__ int s_cnt;
  if (threadIdx.x == 0) {
    auto c = [&](int ss, int jj) -> long long {
      const int v = counts[ss * E + jj];
      return v > 0 ? v : 0;
    };
    long long recv0 = 0, group0 = 0;
    for (int ss = 0; ss < s; ++ss)
      for (int jj = 0; jj < E; ++jj) recv0 += c(ss, jj);
    for (int jj = 0; jj < j; ++jj) recv0 += c(s, jj);
    for (int jj = 0; jj < j; ++jj)
      for (int ss = 0; ss < G; ++ss) group0 += c(ss, jj);
    for (int ss = 0; ss < s; ++ss) group0 += c(ss, j);
    s_recv0 = recv0;
    s_group0 = group0;
    s_cnt = (int)c(s, j);
    if (blockIdx.x == 0) {
      long long run = 0;
      for (int jj = 0; jj < E; ++jj) {
        local_offsets[jj] = (int32_t)(run < R ? run : R);
        for (int ss = 0; ss < G; ++ss) run += c(ss, jj);
      }
      local_offsets[E] = (int32_t)(run < R ? run : R);
    }
  }
  __syncthreads();
  const long long recv0 = s_recv0, group0 = s_group0;
  const int cnt = s_cnt;
  for (int i = threadIdx.x; i < cnt; i += blockDim.x) {
    const long long q = recv0 + i, p = group0 + i;
    if (q < R && p < R) {
      row_map[p] = (int32_t)q;
      inv_row_map[q] = (int32_t)p;
    }
  }
}

// dst[p] = src[index[p] / k]; an index outside [0, rows_src * k) gives a zero row.
__global__ void __launch_bounds__(256) gather_index_vec_kernel(const uint4* __restrict__ src,
                                                               const int32_t* __restrict__ index,
                                                               int rows, long long limit, int k,
                                                               int row_vecs,
                                                               uint4* __restrict__ dst) {
  for (int p = blockIdx.x; p < rows; p += gridDim.x) {
    const int a = __ldg(index + p);
    const bool ok = a >= 0 && a < limit;
    const uint4* s = src + (size_t)(ok ? a / k : 0) * row_vecs;
    uint4* d = dst + (size_t)p * row_vecs;
    for (int c = threadIdx.x; c < row_vecs; c += blockDim.x)
      d[c] = ok ? __ldg(s + c) : make_uint4(0u, 0u, 0u, 0u);
  }
}

__global__ void __launch_bounds__(256) gather_index_byte_kernel(const uint8_t* __restrict__ src,
                                                                const int32_t* __restrict__ index,
                                                                int rows, long long limit, int k,
                                                                size_t row_bytes,
                                                                uint8_t* __restrict__ dst) {
  for (int p = blockIdx.x; p < rows; p += gridDim.x) {
    const int a = __ldg(index + p);
    const bool ok = a >= 0 && a < limit;
    const size_t t = ok ? (size_t)(a / k) : 0;
    for (size_t c = threadIdx.x; c < row_bytes; c += blockDim.x)
      dst[(size_t)p * row_bytes + c] = ok ? src[t * row_bytes + c] : (uint8_t)0;
  }
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_ep_regroup(const int32_t* recv_counts, int G, int E, int R,
                                     int32_t* local_offsets, int32_t* row_map,
                                     int32_t* inv_row_map, void* stream) {
  MOE_CALL_RANGE();
  using namespace moe;
  if (G < 1 || G > kMaxSources || E < 1 || E > kMaxExperts || R < 0) return MOE_ERR_INVALID_ARG;
  if (!recv_counts || !local_offsets || (R > 0 && (!row_map || !inv_row_map)))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  ep_regroup_kernel<<<G * E, 256, 0, s>>>(recv_counts, G, E, R, local_offsets, row_map,
                                          inv_row_map);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" moe_status moe_gather_rows(const void* src, int rows_src, const int32_t* index,
                                      int rows, int k, size_t row_bytes, void* dst,
                                      void* stream) {
  MOE_CALL_RANGE();
  using namespace moe;
  if (rows < 0 || rows_src < 0 || k < 1 || row_bytes == 0) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!src || !index || !dst) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const int cap = device_sm_count() * 8;
  const int grid = rows < cap ? rows : cap;
  const long long limit = (long long)rows_src * k;
  if (row_bytes % 16 == 0 && ((uintptr_t)src % 16) == 0 && ((uintptr_t)dst % 16) == 0)
    gather_index_vec_kernel<<<grid, 256, 0, s>>>((const uint4*)src, index, rows, limit, k,
                                                 (int)(row_bytes / 16), (uint4*)dst);
  else
    gather_index_byte_kernel<<<grid, 256, 0, s>>>((const uint8_t*)src, index, rows, limit, k,
                                                  row_bytes, (uint8_t*)dst);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
