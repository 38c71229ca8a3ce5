// Host-side helpers shared by the pagedkv launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace pkv {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Unique id of the CUDA context current on this thread (0 if none is); false
// if the driver cannot tell.
bool current_context_id(unsigned long long* id);
// SM count of the current device, looked up once per device.
cudaError_t device_sm_count(int* sms);
// Sets a kernel's dynamic shared-memory limit to smem_bytes on the current
// device and returns how many CTAs of `threads` threads fit on one SM (both
// once per device, kernel and size; ctas_per_sm may be NULL).
cudaError_t prepare_kernel(const void* kernel, int threads, int smem_bytes, int* ctas_per_sm);

// TMA map of one cache.
//  kRowsPlain: 3-D view (D, KV head, slot), box D x 1 x box_rows.
//  kRowsSwizzled: 4-D view (64 elements, slot, KV head, D/64 lines), box
//    64 x box_rows x 1 x D/64 with the 128-byte swizzle: whole rows of box_rows
//    slots per copy, stored line-major.
//  kLineSwizzled: the same view with the box 64 x box_rows x 1 x 1: one
//    128-byte line of box_rows slots per copy, so that a tile's rows of one
//    line can sit contiguously (the layout tcgen05 operands are read in).
// Returns false if the encoder is missing or refuses the view.
enum CacheView { kRowsPlain = 0, kRowsSwizzled = 1, kLineSwizzled = 2 };
bool encode_cache_map(CUtensorMap* tm, const void* base, int D, int num_kv_heads, int64_t slots,
                      int box_rows, CacheView view);

// TMA map of the queries [rows][D] (16-bit elements) as (64 elements, D/64
// lines, row) with the box 64 x 1 x box_rows and the 128-byte swizzle: one
// line of box_rows consecutive rows per copy.
bool encode_query_map(CUtensorMap* tm, const void* base, int D, int64_t rows, int box_rows);

// TMA map of packed queries [tokens][num_heads][D] (16-bit elements) as (64
// elements, D/64 lines, head, token) with the box 64 x 1 x group x 128/group
// and the 128-byte swizzle: one line of 128 rows (token-major, head-minor) of
// one KV head's query group per copy; tokens past the end read as zeros.
bool encode_token_query_map(CUtensorMap* tm, const void* base, int D, int num_heads,
                            int64_t tokens, int group);

struct DecodeTcArgs {
  float* part_acc;
  float2* part_ml;
  int* counter;                        // zero at launch
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  int32_t* err;
  int num_seqs, num_heads, num_kv_heads, head_size, num_blocks, block_size, max_blocks_per_seq;
  int partition_tokens, max_parts;
  bool bf16;
  float q_scale;                       // scale * log2(e)
  uint64_t wait_ns;                    // limit of every pipeline wait (1 s normally)
  int stall_unit;                      // test hook (see pkv_test_decode_wait_timeout); -1: none
};
// The tensor-memory decode path for large query groups (decode_tc.cu): writes
// the same partition partials as the other decode paths.
bool decode_tc_supported(int group, int head_size, int block_size, int partition_tokens);
cudaError_t launch_decode_tc(const DecodeTcArgs& a, cudaStream_t stream);

}  // namespace pkv
