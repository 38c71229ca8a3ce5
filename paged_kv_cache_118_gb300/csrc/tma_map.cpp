// TMA tensor maps of a KV cache [num_blocks][block_size][num_kv_heads][D]
// (16-bit elements), shared by the attention kernels' launchers. The driver's
// encoder is reached through the runtime's entry-point query, so the library
// does not link the driver library.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "pkv_host.h"

namespace pkv {

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// Recently encoded maps, keyed by every argument of the encoding (a map is a
// pure function of them): a decode loop passes the same caches call after
// call, and the encoder costs a few microseconds of host time per map.
namespace {
struct MapKey {
  const void* base;
  int64_t extent;                      // slots (caches) or rows (queries)
  int d, heads, box, view;             // view -1: a query map
  bool operator==(const MapKey& o) const {
    return base == o.base && extent == o.extent && d == o.d && heads == o.heads &&
           box == o.box && view == o.view;
  }
};
constexpr int kMapCache = 32;
std::mutex g_map_mu;
MapKey g_map_key[kMapCache];
CUtensorMap g_map_val[kMapCache];
int g_map_used = 0, g_map_next = 0;

bool cached_map(const MapKey& k, CUtensorMap* out) {
  std::lock_guard<std::mutex> lock(g_map_mu);
  for (int i = 0; i < g_map_used; ++i)
    if (g_map_key[i] == k) {
      *out = g_map_val[i];
      return true;
    }
  return false;
}

void remember_map(const MapKey& k, const CUtensorMap& m) {
  std::lock_guard<std::mutex> lock(g_map_mu);
  const int i = g_map_used < kMapCache ? g_map_used++ : (g_map_next++ % kMapCache);
  g_map_key[i] = k;
  g_map_val[i] = m;
}
}  // namespace

bool encode_cache_map(CUtensorMap* tm, const void* base, int D, int num_kv_heads,
                             int64_t slots, int box_rows, CacheView view) {
  const MapKey key{base, slots, D, num_kv_heads, box_rows, static_cast<int>(view)};
  if (cached_map(key, tm)) return true;
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  CUresult r;
  if (view == kRowsPlain) {
    // 3-D view: x = element within the head (D), y = KV head, z = slot; box D x 1 x rows.
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(num_kv_heads),
                          static_cast<cuuint64_t>(slots)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                             static_cast<cuuint64_t>(D) * 2 * num_kv_heads};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(D), 1, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[3] = {1, 1, 1};
    r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    // 4-D view: x = 64 elements (128 bytes), y = slot, z = KV head, w = which
    // 64-element line of the head; box 64 x rows x 1 x D/64 with the 128-byte
    // swizzle. One copy moves whole rows of a block, stored line-major: all
    // rows' first 128 bytes, then all rows' second 128 bytes, so that eight
    // consecutive rows of one line fall in eight different swizzle phases.
    cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(slots),
                          static_cast<cuuint64_t>(num_kv_heads), static_cast<cuuint64_t>(D / 64)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2 * num_kv_heads,
                             static_cast<cuuint64_t>(D) * 2, 128};
    cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_rows), 1,
                         static_cast<cuuint32_t>(view == kLineSwizzled ? 1 : D / 64)};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS) return false;
  remember_map(key, *tm);
  return true;
}

bool encode_query_map(CUtensorMap* tm, const void* base, int D, int64_t rows, int box_rows) {
  const MapKey key{base, rows, D, 0, box_rows, -1};
  if (cached_map(key, tm)) return true;
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(D / 64), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(D) * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  remember_map(key, *tm);
  return true;
}

bool encode_token_query_map(CUtensorMap* tm, const void* base, int D, int num_heads,
                            int64_t tokens, int group) {
  const MapKey key{base, tokens, D, num_heads, group, -2};
  if (cached_map(key, tm)) return true;
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(D / 64), static_cast<cuuint64_t>(num_heads),
                        static_cast<cuuint64_t>(tokens)};
  cuuint64_t strides[3] = {128, static_cast<cuuint64_t>(D) * 2,
                           static_cast<cuuint64_t>(num_heads) * D * 2};
  cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(128 / group)};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  remember_map(key, *tm);
  return true;
}

}  // namespace pkv
