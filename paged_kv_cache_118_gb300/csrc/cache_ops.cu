// Cache writes of a decode step, sm_103a.
//
// * reshape_and_cache — every new token's key and value rows go to their slot
//   (block = slot / B, row = slot % B) of the paged cache; the pages only say
//   the new token is written into the sequence's tail block ("079｜vLLM 与
//   PagedAttention", wq-win.github.io, §2 "共享与写时复制" and the §3
//   algorithm box). With the [num_blocks][B][H_kv][D] layout, slot s of head h
//   starts at element (s * H_kv + h) * D, so the scatter is a gather of 16-byte
//   pieces along a flat row index.
// * swap_blocks — the copies of a swap between two pools, one of which is
//   usually pinned host memory reached directly over the CPU-GPU link (same
//   review, §3 algorithm box).
// * copy_blocks — copy-on-write copies of whole blocks (same review, §2
//   "一次分叉什么时候真的要复制缓存块": only a shared, partly filled tail is ever
//   copied). The pair list travels in the kernel parameters (no device buffer,
//   no host-to-device copy); lists longer than one parameter block are split
//   over several launches.
// Both are bandwidth-bound bitwise copies with 16-byte vector accesses and
// grids sized to the SM count.

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <unordered_set>
#include <vector>

#include "pagedkv.h"
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {

__global__ void __launch_bounds__(256)
    reshape_and_cache_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                             uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                             const int64_t* __restrict__ slots, int64_t num_rows, int kv_heads,
                             int chunks, int64_t capacity, int32_t* err) {
  const int64_t total = num_rows * chunks;  // num_rows = tokens * kv_heads
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = i / chunks;              // token * kv_heads + head
    const int c = static_cast<int>(i - row * chunks);
    const int64_t t = row / kv_heads;
    const int h = static_cast<int>(row - t * kv_heads);
    const int64_t slot = __ldg(slots + t);
    if (slot < 0) continue;
    if (slot >= capacity) {
      if (c == 0 && h == 0) flag_error(err, PKV_DEVERR_SLOT);
      continue;
    }
    const int64_t dst = (slot * kv_heads + h) * chunks + c;
    k_cache[dst] = __ldg(k + i);
    v_cache[dst] = __ldg(v + i);
  }
}

constexpr int kPairsPerLaunch = 1024;  // 8 KB of kernel parameters

struct PairList {
  int32_t src[kPairsPerLaunch];
  int32_t dst[kPairsPerLaunch];
};

// grid.y = pair, grid.x strides over the block's 16-byte pieces.
__global__ void __launch_bounds__(256)
    copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                       int64_t block_chunks, const __grid_constant__ PairList pairs) {
  const int pair = blockIdx.y;
  const int64_t s = static_cast<int64_t>(pairs.src[pair]) * block_chunks;
  const int64_t d = static_cast<int64_t>(pairs.dst[pair]) * block_chunks;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < block_chunks;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 a = __ldcs(k_cache + s + i);
    const uint4 b = __ldcs(v_cache + s + i);
    k_cache[d + i] = a;
    v_cache[d + i] = b;
  }
}

// grid.y = pair; source and destination pools differ (one may be host memory).
__global__ void __launch_bounds__(256)
    swap_blocks_kernel(uint4* __restrict__ dk, uint4* __restrict__ dv, const uint4* __restrict__ sk,
                       const uint4* __restrict__ sv, int64_t block_chunks,
                       const __grid_constant__ PairList pairs) {
  const int pair = blockIdx.y;
  const int64_t s = static_cast<int64_t>(pairs.src[pair]) * block_chunks;
  const int64_t d = static_cast<int64_t>(pairs.dst[pair]) * block_chunks;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < block_chunks;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 a = __ldcs(sk + s + i);
    const uint4 b = __ldcs(sv + s + i);
    __stcs(dk + d + i, a);
    __stcs(dv + d + i, b);
  }
}

// SM count of the current device (152 on GB300 if the lookup fails: it only
// sizes the grid of a grid-stride loop).
static int sm_count() {
  int n = 0;
  return device_sm_count(&n) == cudaSuccess ? n : 152;
}

}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_reshape_and_cache(const void* k, const void* v, void* k_cache,
                                            void* v_cache, const int64_t* slot_mapping,
                                            int num_tokens, int num_kv_heads, int head_size,
                                            int num_blocks, int block_size, int dtype,
                                            int32_t* err_flag, void* stream) {
  if (num_tokens < 0) return PKV_EINVAL;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PKV_EINVAL;
  if (dtype != PKV_F16 && dtype != PKV_BF16) return PKV_EINVAL;
  if (num_kv_heads < 1 || head_size < 1 || (head_size * 2) % 16 != 0) return PKV_EINVAL;
  if (num_blocks < 1 || block_size < 1) return PKV_EINVAL;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_EINVAL;
  const int chunks = head_size * 2 / 16;
  const int64_t rows = static_cast<int64_t>(num_tokens) * num_kv_heads;
  const int64_t total = rows * chunks;
  const int threads = 256;
  const int64_t want = (total + threads - 1) / threads;
  const int grid = static_cast<int>(std::min<int64_t>(want, static_cast<int64_t>(sm_count()) * 8));
  reshape_and_cache_kernel<<<grid, threads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), static_cast<uint4*>(k_cache),
      static_cast<uint4*>(v_cache), slot_mapping, rows, num_kv_heads, chunks,
      static_cast<int64_t>(num_blocks) * block_size, err_flag);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

extern "C" pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, const int32_t* src_dst_pairs,
                                      int num_pairs, int num_blocks, size_t block_bytes,
                                      void* stream) {
  if (num_pairs < 0) return PKV_EINVAL;
  if (num_pairs == 0) return PKV_OK;
  if (!k_cache || !v_cache || !src_dst_pairs || num_blocks < 1) return PKV_EINVAL;
  if (block_bytes == 0 || block_bytes % 16 != 0) return PKV_EINVAL;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PKV_EINVAL;
  std::unordered_set<int32_t> dsts;
  dsts.reserve(num_pairs * 2);
  for (int i = 0; i < num_pairs; ++i) {
    const int32_t s = src_dst_pairs[2 * i], d = src_dst_pairs[2 * i + 1];
    if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) return PKV_ERANGE;
    if (!dsts.insert(d).second) return PKV_EINVAL;
  }
  for (int i = 0; i < num_pairs; ++i)
    if (dsts.count(src_dst_pairs[2 * i])) return PKV_EINVAL;

  const int64_t chunks = static_cast<int64_t>(block_bytes / 16);
  const int threads = 256;
  const int per_pair = static_cast<int>(std::min<int64_t>((chunks + threads - 1) / threads, 64));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int base = 0; base < num_pairs; base += kPairsPerLaunch) {
    const int n = std::min(kPairsPerLaunch, num_pairs - base);
    PairList pl;
    for (int i = 0; i < n; ++i) {
      pl.src[i] = src_dst_pairs[2 * (base + i)];
      pl.dst[i] = src_dst_pairs[2 * (base + i) + 1];
    }
    copy_blocks_kernel<<<dim3(per_pair, n), threads, 0, s>>>(
        static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), chunks, pl);
    if (cudaGetLastError() != cudaSuccess) return PKV_ECUDA;
  }
  return PKV_OK;
}

// Device address of p (device memory or pinned host memory the GPU maps), or
// nullptr if the GPU cannot address it.
static void* device_address(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return const_cast<void*>(p);
  if (a.type == cudaMemoryTypeHost) return a.devicePointer;
  return nullptr;
}

extern "C" pkv_status pkv_swap_blocks(void* dst_k, void* dst_v, const void* src_k,
                                      const void* src_v, const int32_t* src_dst_pairs,
                                      int num_pairs, int src_blocks, int dst_blocks,
                                      size_t block_bytes, void* stream) {
  if (num_pairs < 0) return PKV_EINVAL;
  if (num_pairs == 0) return PKV_OK;
  if (!dst_k || !dst_v || !src_k || !src_v || !src_dst_pairs || src_blocks < 1 || dst_blocks < 1)
    return PKV_EINVAL;
  if (block_bytes == 0 || block_bytes % 16 != 0) return PKV_EINVAL;
  void* dk = device_address(dst_k);
  void* dv = device_address(dst_v);
  void* sk = device_address(src_k);
  void* sv = device_address(src_v);
  if (!dk || !dv || !sk || !sv) return PKV_EINVAL;
  if (!aligned16(dk) || !aligned16(dv) || !aligned16(sk) || !aligned16(sv)) return PKV_EINVAL;
  std::unordered_set<int32_t> dsts;
  dsts.reserve(num_pairs * 2);
  for (int i = 0; i < num_pairs; ++i) {
    const int32_t s = src_dst_pairs[2 * i], d = src_dst_pairs[2 * i + 1];
    if (s < 0 || s >= src_blocks || d < 0 || d >= dst_blocks) return PKV_ERANGE;
    if (!dsts.insert(d).second) return PKV_EINVAL;
  }
  const int64_t chunks = static_cast<int64_t>(block_bytes / 16);
  const int threads = 256;
  const int per_pair = static_cast<int>(std::min<int64_t>((chunks + threads - 1) / threads, 64));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  for (int base = 0; base < num_pairs; base += kPairsPerLaunch) {
    const int n = std::min(kPairsPerLaunch, num_pairs - base);
    PairList pl;
    for (int i = 0; i < n; ++i) {
      pl.src[i] = src_dst_pairs[2 * (base + i)];
      pl.dst[i] = src_dst_pairs[2 * (base + i) + 1];
    }
    swap_blocks_kernel<<<dim3(per_pair, n), threads, 0, st>>>(
        static_cast<uint4*>(dk), static_cast<uint4*>(dv), static_cast<const uint4*>(sk),
        static_cast<const uint4*>(sv), chunks, pl);
    if (cudaGetLastError() != cudaSuccess) return PKV_ECUDA;
  }
  return PKV_OK;
}
