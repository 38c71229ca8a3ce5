// Paged decode attention for sm_103a.
//
// What is computed: for each sequence and query head, softmax attention of the
// single decode query over the sequence's whole cached history, which sits in
// fixed-size physical blocks reached through the sequence's block table, with
// one softmax denominator shared by every block and the unfilled rows of the
// last block masked ("079｜vLLM 与 PagedAttention", wq-win.github.io, §2
// "分块以后，注意力仍需对整个历史归一化", the equation for Z and o).
//
// How (GB300 design, not the pages' A100 kernel):
//  * decode_partition_kernel — one CTA per (sequence, KV head [or a slice of
//    its query-head group], context partition of `partition_tokens` tokens).
//    One producer thread streams 32-token tiles of K and V into a 4-stage
//    shared-memory ring with 3-D TMA tensor copies (a copy per physical block,
//    or a 32-row slice of one when blocks are larger), completing on mbarriers.
//    Four consumer warps split each tile into 8-lane token groups; each group
//    keeps its own running maximum, denominator and fp32 accumulator for the
//    GS query heads that share the KV head (online softmax in base 2, with the
//    rescale taken only when the maximum grows by more than 2^8). The groups
//    are merged at the end into one unnormalised partial (m, l, acc[d]).
//  * decode_reduce_kernel — one warp per (sequence, query head) merges the
//    partition partials: M = max m_p, Z = sum l_p 2^(m_p - M),
//    o = sum acc_p 2^(m_p - M) / Z, rounded to the output type.
// Every wait on an mbarrier has a time limit (see pkv_device.cuh); a block id
// or context length out of range is skipped and reported through err_flag.

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "pagedkv.h"
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {

constexpr int kTile = 32;           // tokens per pipeline stage
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kGroupLanes = 8;      // lanes that share one token row
constexpr int kGroups = kConsumerWarps * 32 / kGroupLanes;  // token groups per CTA (16)
constexpr int kStages = 4;
constexpr float kRescaleThreshold = 8.0f;  // base-2 growth of the max that forces a rescale
constexpr float kLog2e = 1.4426950408889634f;

struct DecodeParams {
  float* part_acc;            // [rows][D], rows = num_seqs * num_heads * max_parts
  float2* part_ml;            // [rows] = (m in base-2 units, l)
  const uint16_t* q;          // [num_seqs][num_heads][D]
  const int32_t* block_tables;
  const int32_t* context_lens;
  int32_t* err;
  int num_heads;
  int group;                  // query heads per KV head (num_heads / num_kv_heads)
  int num_blocks;
  int block_size;
  int max_blocks_per_seq;
  int partition_tokens;
  int max_parts;
  int box_rows;               // rows per TMA copy: min(block_size, kTile)
  float q_scale;              // scale * log2(e)
};

template <int D, int GS>
struct DecodeLayout {
  static constexpr int kRowBytes = D * 2;
  static constexpr int kTileBytes = kTile * kRowBytes;        // K (or V) of one stage
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kCombineFloats = kConsumerWarps * GS * (D + 2);
  static constexpr int kChunks = D / 64;                      // 16-byte pieces per lane per row
  static constexpr int kE = 8 * kChunks;                      // elements per lane per row
  static int smem_bytes(int table_slice) {
    return 1024 /*alignment slack*/ + kRingBytes + kCombineFloats * 4 + 2 * kStages * 8 +
           ((table_slice * 4 + 15) / 16) * 16;
  }
};

template <int D, int GS, typename T>
__global__ void __launch_bounds__(kThreads, 2)
    decode_partition_kernel(const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
  using Lay = DecodeLayout<D, GS>;
  constexpr int E = Lay::kE;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* ring = smem;
  float* combine = reinterpret_cast<float*>(smem + Lay::kRingBytes);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(combine + Lay::kCombineFloats);
  uint64_t* empty_bar = full_bar + kStages;
  int32_t* slice = reinterpret_cast<int32_t*>(empty_bar + kStages);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int subs = p.group / GS;                 // CTAs per KV head
  const int kvh = blockIdx.x / subs;
  const int head0 = kvh * p.group + (blockIdx.x % subs) * GS;
  const int seq = blockIdx.y;
  const int part = blockIdx.z;
  const int B = p.block_size;

  const int L = __ldg(p.context_lens + seq);
  if (L < 1 || L > p.max_blocks_per_seq * B) {
    if (threadIdx.x == 0 && part == 0 && blockIdx.x == 0) flag_error(p.err, PKV_DEVERR_CONTEXT);
    return;
  }
  const int t_begin = part * p.partition_tokens;
  if (t_begin >= L) return;
  const int t_end = min(L, t_begin + p.partition_tokens);
  const int n_tiles = (t_end - t_begin + kTile - 1) / kTile;
  const int jb0 = t_begin / B;
  const int nb = (t_end - 1) / B - jb0 + 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], kConsumerWarps);
    }
    fence_barrier_init();
  }
  if (warp == kConsumerWarps) {
    if (lane == 0) {
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
    }
    const int32_t* row = p.block_tables + static_cast<int64_t>(seq) * p.max_blocks_per_seq + jb0;
    for (int i = lane; i < nb; i += 32) {
      int32_t id = __ldg(row + i);
      if (id < 0 || id >= p.num_blocks) {
        flag_error(p.err, PKV_DEVERR_BLOCK_ID);
        id = 0;
      }
      slice[i] = id;
    }
  }
  __syncthreads();

  // ------------------------------------------------------------ producer
  if (warp == kConsumerWarps) {
    if (lane != 0) return;
    const uint64_t policy = l2_evict_first_policy();
    const uint32_t copy_bytes = static_cast<uint32_t>(p.box_rows) * Lay::kRowBytes;
    int last_issued[kStages];
#pragma unroll
    for (int i = 0; i < kStages; ++i) last_issued[i] = -1;
    bool ok = true;
    for (int i = 0; i < n_tiles; ++i) {
      const int st = i % kStages;
      if (i >= kStages && !mbar_wait(&empty_bar[st], ((i / kStages) & 1) ^ 1)) {
        ok = false;
        break;
      }
      const int t0 = t_begin + i * kTile;
      const int valid = min(kTile, t_end - t0);
      const int copies = B >= kTile ? 1 : (valid + B - 1) / B;
      uint8_t* kdst = ring + st * Lay::kStageBytes;
      uint8_t* vdst = kdst + Lay::kTileBytes;
      mbar_arrive_expect_tx(&full_bar[st], 2u * copies * copy_bytes);
      for (int c = 0; c < copies; ++c) {
        int z;
        if (B >= kTile) {
          z = slice[t0 / B - jb0] * B + (t0 % B);
        } else {
          z = slice[t0 / B + c - jb0] * B;
        }
        tma_load_3d(kdst + c * copy_bytes, &tm_k, &full_bar[st], 0, kvh, z, policy);
        tma_load_3d(vdst + c * copy_bytes, &tm_v, &full_bar[st], 0, kvh, z, policy);
      }
      last_issued[st] = i;
    }
    if (!ok) {
      flag_error(p.err, PKV_DEVERR_TIMEOUT);
      // Let the copies already in flight land before the CTA can retire.
      for (int st = 0; st < kStages; ++st)
        if (last_issued[st] >= 0) mbar_wait(&full_bar[st], (last_issued[st] / kStages) & 1);
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int grp = lane >> 3;                      // group within the warp
  const int gi = warp * 4 + grp;                  // group within the CTA (0..15)
  const int j = lane & 7;                         // lane within the group
  const unsigned gmask = 0xffu << (grp * 8);

  float qf[GS][E];
#pragma unroll
  for (int g = 0; g < GS; ++g) {
    const uint16_t* qrow = p.q + (static_cast<int64_t>(seq) * p.num_heads + head0 + g) * D;
#pragma unroll
    for (int c = 0; c < Lay::kChunks; ++c) {
      uint4 raw = __ldg(reinterpret_cast<const uint4*>(qrow + c * 64 + 8 * j));
      widen8<T>(raw, &qf[g][c * 8]);
#pragma unroll
      for (int e = 0; e < 8; ++e) qf[g][c * 8 + e] *= p.q_scale;
    }
  }
  float m[GS], l[GS], acc[GS][E];
#pragma unroll
  for (int g = 0; g < GS; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[g][e] = 0.f;
  }

  bool ok = true;
  for (int i = 0; i < n_tiles; ++i) {
    const int st = i % kStages;
    if (!mbar_wait(&full_bar[st], (i / kStages) & 1)) {
      ok = false;
      break;
    }
    const int valid = min(kTile, t_end - (t_begin + i * kTile));
    const uint16_t* ks = reinterpret_cast<const uint16_t*>(ring + st * Lay::kStageBytes);
    const uint16_t* vs = ks + kTile * D;
#pragma unroll
    for (int r = 0; r < kTile / kGroups; ++r) {
      const int tk = gi + r * kGroups;
      if (tk < valid) {
        float s[GS];
#pragma unroll
        for (int g = 0; g < GS; ++g) s[g] = 0.f;
#pragma unroll
        for (int c = 0; c < Lay::kChunks; ++c) {
          uint4 raw = *reinterpret_cast<const uint4*>(ks + tk * D + c * 64 + 8 * j);
          float kf[8];
          widen8<T>(raw, kf);
#pragma unroll
          for (int g = 0; g < GS; ++g)
#pragma unroll
            for (int e = 0; e < 8; ++e) s[g] = fmaf(qf[g][c * 8 + e], kf[e], s[g]);
        }
        float pr[GS];
#pragma unroll
        for (int g = 0; g < GS; ++g) {
          s[g] += __shfl_xor_sync(gmask, s[g], 1);
          s[g] += __shfl_xor_sync(gmask, s[g], 2);
          s[g] += __shfl_xor_sync(gmask, s[g], 4);
          if (s[g] > m[g] + kRescaleThreshold) {
            const float corr = ex2(m[g] - s[g]);
            l[g] *= corr;
#pragma unroll
            for (int e = 0; e < E; ++e) acc[g][e] *= corr;
            m[g] = s[g];
          }
          pr[g] = ex2(s[g] - m[g]);
          l[g] += pr[g];
        }
#pragma unroll
        for (int c = 0; c < Lay::kChunks; ++c) {
          uint4 raw = *reinterpret_cast<const uint4*>(vs + tk * D + c * 64 + 8 * j);
          float vf[8];
          widen8<T>(raw, vf);
#pragma unroll
          for (int g = 0; g < GS; ++g)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[g][c * 8 + e] = fmaf(pr[g], vf[e], acc[g][c * 8 + e]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[st]);
  }
  if (!ok) flag_error(p.err, PKV_DEVERR_TIMEOUT);

  // Merge the four groups of this warp (lanes j, j+8, j+16, j+24 hold the same
  // elements), then the four warps through shared memory.
#pragma unroll
  for (int g = 0; g < GS; ++g) {
    float mx = fmaxf(m[g], __shfl_xor_sync(0xffffffffu, m[g], 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    const float f = (mx == -INFINITY) ? 0.f : ex2(m[g] - mx);
    float ls = l[g] * f;
    ls += __shfl_xor_sync(0xffffffffu, ls, 8);
    ls += __shfl_xor_sync(0xffffffffu, ls, 16);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      float a = acc[g][e] * f;
      a += __shfl_xor_sync(0xffffffffu, a, 8);
      a += __shfl_xor_sync(0xffffffffu, a, 16);
      acc[g][e] = a;
    }
    float* cw = combine + (warp * GS + g) * (D + 2);
    if (grp == 0) {
#pragma unroll
      for (int c = 0; c < Lay::kChunks; ++c)
#pragma unroll
        for (int e = 0; e < 8; ++e) cw[2 + c * 64 + 8 * j + e] = acc[g][c * 8 + e];
      if (j == 0) {
        cw[0] = mx;
        cw[1] = ls;
      }
    }
  }
  named_sync(1, kConsumerWarps * 32);

  const int64_t row0 =
      (static_cast<int64_t>(seq) * p.num_heads + head0) * p.max_parts + part;
  for (int idx = threadIdx.x; idx < GS * D; idx += kConsumerWarps * 32) {
    const int g = idx / D;
    const int e = idx % D;
    float mw[kConsumerWarps];
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      mw[w] = combine[(w * GS + g) * (D + 2)];
      M = fmaxf(M, mw[w]);
    }
    float a = 0.f, lsum = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float f = (mw[w] == -INFINITY) ? 0.f : ex2(mw[w] - M);
      a = fmaf(combine[(w * GS + g) * (D + 2) + 2 + e], f, a);
      lsum = fmaf(combine[(w * GS + g) * (D + 2) + 1], f, lsum);
    }
    const int64_t row = row0 + static_cast<int64_t>(g) * p.max_parts;
    p.part_acc[row * D + e] = a;
    if (e == 0) p.part_ml[row] = make_float2(M, lsum);
  }
}

template <typename O>
__device__ __forceinline__ void store_out(O* dst, float v);
template <>
__device__ __forceinline__ void store_out<float>(float* dst, float v) { *dst = v; }
template <>
__device__ __forceinline__ void store_out<__half>(__half* dst, float v) {
  *dst = __float2half_rn(v);
}
template <>
__device__ __forceinline__ void store_out<__nv_bfloat16>(__nv_bfloat16* dst, float v) {
  *dst = __float2bfloat16_rn(v);
}

struct ReduceParams {
  const float* part_acc;
  const float2* part_ml;
  const int32_t* context_lens;
  int num_seqs;
  int num_heads;
  int max_parts;
  int partition_tokens;
  int max_context;
};

template <int D, typename O>
__global__ void __launch_bounds__(128) decode_reduce_kernel(O* out, const ReduceParams p) {
  constexpr int PER = D / 32;
  const int w = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (w >= p.num_seqs * p.num_heads) return;
  const int seq = w / p.num_heads;
  O* dst = out + static_cast<int64_t>(w) * D + lane * PER;
  const int L = __ldg(p.context_lens + seq);
  if (L < 1 || L > p.max_context) {
#pragma unroll
    for (int k = 0; k < PER; ++k) store_out<O>(dst + k, 0.f);
    return;
  }
  const int np = (L + p.partition_tokens - 1) / p.partition_tokens;
  const int64_t row0 = static_cast<int64_t>(w) * p.max_parts;
  float M = -INFINITY;
  for (int i = lane; i < np; i += 32) M = fmaxf(M, p.part_ml[row0 + i].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float Z = 0.f;
  for (int i = lane; i < np; i += 32) {
    const float2 ml = p.part_ml[row0 + i];
    Z = fmaf(ml.y, ex2(ml.x - M), Z);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) Z += __shfl_xor_sync(0xffffffffu, Z, o);
  float acc[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) acc[k] = 0.f;
  for (int i = 0; i < np; ++i) {
    const float wgt = ex2(p.part_ml[row0 + i].x - M);
    const float* src = p.part_acc + (row0 + i) * D + lane * PER;
    if constexpr (PER == 4) {
      const float4 v = *reinterpret_cast<const float4*>(src);
      acc[0] = fmaf(v.x, wgt, acc[0]);
      acc[1] = fmaf(v.y, wgt, acc[1]);
      acc[2] = fmaf(v.z, wgt, acc[2]);
      acc[3] = fmaf(v.w, wgt, acc[3]);
    } else {
#pragma unroll
      for (int k = 0; k < PER; ++k) acc[k] = fmaf(src[k], wgt, acc[k]);
    }
  }
#pragma unroll
  for (int k = 0; k < PER; ++k) store_out<O>(dst + k, acc[k] / Z);
}

// ---------------------------------------------------------------- host side

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

// 3-D view of a cache: x = element within the head (D), y = KV head,
// z = slot (block * B + row); box = D x 1 x box_rows.
static bool encode_cache_map(CUtensorMap* tm, const void* base, int D, int num_kv_heads,
                             int64_t slots, int box_rows) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(num_kv_heads),
                        static_cast<cuuint64_t>(slots)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                           static_cast<cuuint64_t>(D) * 2 * num_kv_heads};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(D), 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static int pick_group_slice(int group) {
  for (int gs = 4; gs > 1; --gs)
    if (group % gs == 0) return gs;
  return 1;
}

template <int D, int GS, typename T>
static cudaError_t launch_partition(const CUtensorMap& tk, const CUtensorMap& tv,
                                    const DecodeParams& p, int num_kv_heads, int num_seqs,
                                    cudaStream_t stream) {
  auto kern = decode_partition_kernel<D, GS, T>;
  const int slice = p.partition_tokens / p.block_size + 2;
  const int smem = DecodeLayout<D, GS>::smem_bytes(slice);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(num_kv_heads * (p.group / GS), num_seqs, p.max_parts);
  kern<<<grid, kThreads, smem, stream>>>(tk, tv, p);
  return cudaGetLastError();
}

template <int D, typename T>
static cudaError_t dispatch_gs(int gs, const CUtensorMap& tk, const CUtensorMap& tv,
                               const DecodeParams& p, int num_kv_heads, int num_seqs,
                               cudaStream_t s) {
  switch (gs) {
    case 1: return launch_partition<D, 1, T>(tk, tv, p, num_kv_heads, num_seqs, s);
    case 2: return launch_partition<D, 2, T>(tk, tv, p, num_kv_heads, num_seqs, s);
    case 3: return launch_partition<D, 3, T>(tk, tv, p, num_kv_heads, num_seqs, s);
    default: return launch_partition<D, 4, T>(tk, tv, p, num_kv_heads, num_seqs, s);
  }
}

template <int D>
static cudaError_t launch_reduce(void* out, int out_dtype, const ReduceParams& rp,
                                 cudaStream_t s) {
  const int warps = rp.num_seqs * rp.num_heads;
  dim3 grid((warps + 3) / 4);
  switch (out_dtype) {
    case PKV_F32:
      decode_reduce_kernel<D, float><<<grid, 128, 0, s>>>(static_cast<float*>(out), rp);
      break;
    case PKV_F16:
      decode_reduce_kernel<D, __half><<<grid, 128, 0, s>>>(static_cast<__half*>(out), rp);
      break;
    default:
      decode_reduce_kernel<D, __nv_bfloat16>
          <<<grid, 128, 0, s>>>(static_cast<__nv_bfloat16*>(out), rp);
  }
  return cudaGetLastError();
}

}  // namespace pkv

using namespace pkv;

static int effective_partition(int partition_tokens) {
  return partition_tokens == 0 ? 512 : partition_tokens;
}

// A 32-token tile is a whole number of blocks, or a whole number of tiles is a block.
static bool block_size_ok(int b) { return b >= 1 && b <= 256 && (b & (b - 1)) == 0; }

extern "C" size_t pkv_decode_workspace_size(int num_seqs, int num_heads, int head_size,
                                            int max_blocks_per_seq, int block_size,
                                            int partition_tokens) {
  const int pt = effective_partition(partition_tokens);
  if (num_seqs < 0 || num_heads < 1 || head_size < 1 || max_blocks_per_seq < 1 ||
      block_size < 1 || pt < 1)
    return 0;
  const int64_t parts = (static_cast<int64_t>(max_blocks_per_seq) * block_size + pt - 1) / pt;
  const int64_t rows = static_cast<int64_t>(num_seqs) * num_heads * parts;
  return static_cast<size_t>(rows * head_size * 4 + rows * 8 + 16);
}

extern "C" pkv_status pkv_paged_attention_decode(
    void* out, int out_dtype, const void* q, const void* k_cache, const void* v_cache,
    int kv_dtype, const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
    int num_heads, int num_kv_heads, int head_size, int num_blocks, int block_size,
    int max_blocks_per_seq, float scale, int partition_tokens, void* workspace,
    size_t workspace_bytes, int32_t* err_flag, void* stream) {
  const int pt = effective_partition(partition_tokens);
  if (num_seqs < 0 || num_seqs > 65535) return PKV_EINVAL;
  if (num_seqs == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !workspace)
    return PKV_EINVAL;
  if (kv_dtype != PKV_F16 && kv_dtype != PKV_BF16) return PKV_EINVAL;
  if (out_dtype != PKV_F16 && out_dtype != PKV_BF16 && out_dtype != PKV_F32) return PKV_EINVAL;
  if (head_size != 64 && head_size != 128) return PKV_EINVAL;
  if (num_kv_heads < 1 || num_heads < num_kv_heads || num_heads % num_kv_heads != 0)
    return PKV_EINVAL;
  if (!block_size_ok(block_size) || num_blocks < 1 || max_blocks_per_seq < 1) return PKV_EINVAL;
  if (static_cast<int64_t>(num_blocks) * block_size > INT32_MAX) return PKV_EINVAL;
  if (static_cast<int64_t>(max_blocks_per_seq) * block_size > INT32_MAX / 2) return PKV_EINVAL;
  if (pt < kTile || pt > 4096 || pt % kTile != 0) return PKV_EINVAL;
  if (!std::isfinite(scale)) return PKV_EINVAL;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(workspace))
    return PKV_EINVAL;
  const int64_t max_ctx = static_cast<int64_t>(max_blocks_per_seq) * block_size;
  const int64_t parts = (max_ctx + pt - 1) / pt;
  if (parts > 65535) return PKV_EINVAL;
  const size_t need = pkv_decode_workspace_size(num_seqs, num_heads, head_size,
                                                max_blocks_per_seq, block_size, pt);
  if (workspace_bytes < need) return PKV_EWORKSPACE;

  const int box_rows = std::min(block_size, kTile);
  CUtensorMap tk, tv;
  const int64_t slots = static_cast<int64_t>(num_blocks) * block_size;
  if (!encode_cache_map(&tk, k_cache, head_size, num_kv_heads, slots, box_rows) ||
      !encode_cache_map(&tv, v_cache, head_size, num_kv_heads, slots, box_rows))
    return PKV_ECUDA;

  const int64_t rows = static_cast<int64_t>(num_seqs) * num_heads * parts;
  DecodeParams p{};
  p.part_acc = static_cast<float*>(workspace);
  p.part_ml = reinterpret_cast<float2*>(static_cast<float*>(workspace) + rows * head_size);
  p.q = static_cast<const uint16_t*>(q);
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.err = err_flag;
  p.num_heads = num_heads;
  p.group = num_heads / num_kv_heads;
  p.num_blocks = num_blocks;
  p.block_size = block_size;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.partition_tokens = pt;
  p.max_parts = static_cast<int>(parts);
  p.box_rows = box_rows;
  p.q_scale = scale * kLog2e;
  const int gs = pick_group_slice(p.group);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  cudaError_t e;
  if (head_size == 128) {
    e = kv_dtype == PKV_F16 ? dispatch_gs<128, F16>(gs, tk, tv, p, num_kv_heads, num_seqs, s)
                            : dispatch_gs<128, BF16>(gs, tk, tv, p, num_kv_heads, num_seqs, s);
  } else {
    e = kv_dtype == PKV_F16 ? dispatch_gs<64, F16>(gs, tk, tv, p, num_kv_heads, num_seqs, s)
                            : dispatch_gs<64, BF16>(gs, tk, tv, p, num_kv_heads, num_seqs, s);
  }
  if (e != cudaSuccess) return PKV_ECUDA;

  ReduceParams rp{};
  rp.part_acc = p.part_acc;
  rp.part_ml = p.part_ml;
  rp.context_lens = context_lens;
  rp.num_seqs = num_seqs;
  rp.num_heads = num_heads;
  rp.max_parts = p.max_parts;
  rp.partition_tokens = pt;
  rp.max_context = static_cast<int>(max_ctx);
  e = head_size == 128 ? launch_reduce<128>(out, out_dtype, rp, s)
                       : launch_reduce<64>(out, out_dtype, rp, s);
  return e == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

// ---------------------------------------------------------------------------
// Allocation-free variant of the decode call.
//
// Some callers cannot hand the decode call a workspace: for example a plugin
// that a host application gives only its input and output buffers while the
// application owns every byte of device memory, or a serving loop that has
// reserved the whole pool up front and must not call cudaMalloc (which can
// stall the device) once decoding runs. For them, the partition partials live
// in this fixed array, part of the library's image: every GPU that loads the
// library holds its PKV_NOALLOC_SCRATCH_BYTES until the process exits. The
// kernels are the same as those of pkv_paged_attention_decode; only the place
// of the partials differs.
// ---------------------------------------------------------------------------

static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};
}  // namespace

// Device address of g_noalloc_scratch on the current device. Host code only
// sees a host-side stand-in under the array's name, so the address is looked
// up once per device (with that device current) and remembered.
static pkv_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ECUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return PKV_ECUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return PKV_OK;
}

extern "C" pkv_status pkv_paged_attention_decode_noalloc(
    void* out, int out_dtype, const void* q, const void* k_cache, const void* v_cache,
    int kv_dtype, const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
    int num_heads, int num_kv_heads, int head_size, int num_blocks, int block_size,
    int max_blocks_per_seq, float scale, int partition_tokens, int32_t* err_flag, void* stream) {
  if (num_seqs == 0) return PKV_OK;
  const size_t need = pkv_decode_workspace_size(num_seqs, num_heads, head_size,
                                                max_blocks_per_seq, block_size, partition_tokens);
  if (need == 0) return PKV_EINVAL;
  if (need > PKV_NOALLOC_SCRATCH_BYTES) return PKV_EWORKSPACE;
  void* scratch = nullptr;
  const pkv_status st = noalloc_scratch(&scratch);
  if (st != PKV_OK) return st;
  // Nothing in the array has to start at zero: the merge reads only partials
  // that the same call wrote first, in stream order.
  return pkv_paged_attention_decode(out, out_dtype, q, k_cache, v_cache, kv_dtype, block_tables,
                                    context_lens, num_seqs, num_heads, num_kv_heads, head_size,
                                    num_blocks, block_size, max_blocks_per_seq, scale,
                                    partition_tokens, scratch, PKV_NOALLOC_SCRATCH_BYTES, err_flag,
                                    stream);
}
