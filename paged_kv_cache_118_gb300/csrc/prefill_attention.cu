// Paged chunked-prefill attention for sm_103a.
//
// What is computed: a sequence with L tokens in its cache receives a chunk of
// C query tokens, its last C positions (their keys and values already
// written); query i (position L - C + i) attends over positions 0..L-C+i of the
// sequence's paged history with one softmax denominator (chunked prefill,
// zhy-blog.vercel.app §4: a long prompt is processed in chunks whose masks
// follow their position; "079｜vLLM 与 PagedAttention" §2 for the single global
// denominator). Decode is the case C = 1.
//
// How (FlashAttention-2 structure over a paged cache, warp-level tensor cores):
//  * one CTA per (tile of 64 rows, KV head, sequence); a row is one (query
//    token, query head of the KV head's group), so 64/G tokens per tile;
//  * a producer warp streams 32-key tiles of K and V over the causal range
//    only, one 4-D TMA box per physical block with the 128-byte swizzle, into
//    a 4-stage ring completing on mbarriers (bounded waits);
//  * each of four consumer warps owns 16 rows and every key: S = Q K^T with
//    mma.m16n8k16 (Q fragments in registers), causal mask and online softmax
//    (base 2, lazy rescale) in the accumulator layout, P fed straight from
//    the score fragments into P V with mma.m16n8k16 (bfloat16 P as hi + lo
//    halves), fp32 accumulation; a warp skips tiles past its last query.
// A chunk or context length out of range is skipped and reported.

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <type_traits>

#include "pagedkv.h"
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {
namespace prefill {

constexpr int kTile = 32;              // keys per pipeline stage
constexpr int kRows = 64;              // query rows per CTA (16 per consumer warp)
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 4;
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLog2e = 1.4426950408889634f;

struct Params {
  void* out;
  int out_dtype;
  const uint16_t* q;                   // [total_queries][num_heads][D]
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* query_start;          // [num_seqs + 1]
  int32_t* err;
  int num_heads;
  int group;                           // query heads per KV head
  int num_blocks;
  int block_size;
  int max_blocks_per_seq;
  int max_query_len;
  int box_rows;                        // min(block_size, kTile)
  float q_scale;                       // scale * log2(e)
};

template <int D>
struct Layout {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kSmem = 1024 + kRingBytes + 2 * kStages * 8;
};

__device__ __forceinline__ void store_elem(void* out, int64_t i, float v, int dtype) {
  if (dtype == PKV_F32) static_cast<float*>(out)[i] = v;
  else if (dtype == PKV_F16) static_cast<__half*>(out)[i] = __float2half_rn(v);
  else static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(v);
}

template <int D, typename T>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const Params p) {
  using Lay = Layout<D>;
  constexpr int KS = D / 16;           // k-steps of q.k
  constexpr int NT = D / 8;            // 8-column tiles of the output
  const int rows_shift = 31 - __clz(p.box_rows);  // rows per TMA copy = 2^rows_shift
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* ring = smem;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + Lay::kRingBytes);
  uint64_t* empty_bar = full_bar + kStages;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int seq = blockIdx.z;
  const int kvh = blockIdx.y;
  const int G = p.group;
  const int tokens_per_tile = kRows / G;
  const int tok0 = blockIdx.x * tokens_per_tile;          // first chunk token of the tile
  const int B = p.block_size;

  const int qs = __ldg(p.query_start + seq);
  const int C = __ldg(p.query_start + seq + 1) - qs;
  const int L = __ldg(p.context_lens + seq);
  if (C < 0 || C > p.max_query_len || C > L || L > p.max_blocks_per_seq * B) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && kvh == 0 && C != 0)
      flag_error(p.err, PKV_DEVERR_CONTEXT);
    return;
  }
  if (tok0 >= C) return;
  const int tok_end = min(C, tok0 + tokens_per_tile);
  const int kv_end = L - C + tok_end;                      // keys this tile can see
  const int n_tiles = (kv_end + kTile - 1) / kTile;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], kConsumerWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();

  // ------------------------------------------------------------ producer
  if (warp == kConsumerWarps) {
    if (lane != 0) return;
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    const uint64_t policy = l2_evict_first_policy();
    const uint32_t copy_bytes = static_cast<uint32_t>(p.box_rows) * D * 2;
    const int32_t* row = p.block_tables + static_cast<int64_t>(seq) * p.max_blocks_per_seq;
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
      const int t0 = i * kTile;
      const int valid = min(kTile, kv_end - t0);
      const int copies = B >= kTile ? 1 : (valid + B - 1) / B;
      uint8_t* kdst = ring + st * Lay::kStageBytes;
      uint8_t* vdst = kdst + Lay::kTileBytes;
      mbar_arrive_expect_tx(&full_bar[st], 2u * copies * copy_bytes);
      for (int c = 0; c < copies; ++c) {
        const int j = B >= kTile ? t0 / B : t0 / B + c;
        int32_t id = __ldg(row + j);
        if (id < 0 || id >= p.num_blocks) {
          flag_error(p.err, PKV_DEVERR_BLOCK_ID);
          id = 0;
        }
        const int z = id * B + (B >= kTile ? t0 % B : 0);
        tma_load_4d(kdst + c * copy_bytes, &tm_k, &full_bar[st], 0, z, kvh, 0, policy);
        tma_load_4d(vdst + c * copy_bytes, &tm_v, &full_bar[st], 0, z, kvh, 0, policy);
      }
      last_issued[st] = i;
    }
    if (!ok) {
      flag_error(p.err, PKV_DEVERR_TIMEOUT);
      for (int st = 0; st < kStages; ++st)
        if (last_issued[st] >= 0) mbar_wait(&full_bar[st], (last_issued[st] / kStages) & 1);
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int g = lane >> 2, t = lane & 3;
  const int r0 = warp * 16;            // this warp's first row of the tile
  // rows r0 + g and r0 + g + 8: (token, head) and their query positions
  int tokA = tok0 + (r0 + g) / G, tokB = tok0 + (r0 + g + 8) / G;
  const int headA = kvh * G + (r0 + g) % G, headB = kvh * G + (r0 + g + 8) % G;
  const bool liveA = tokA < C, liveB = tokB < C;
  const int posA = L - C + tokA, posB = L - C + tokB;
  // the warp's last query position: tiles past it are skipped
  const int warp_last_tok = min(C - 1, tok0 + (r0 + 15) / G);
  const int warp_kv_end = L - C + warp_last_tok + 1;

  uint32_t qa[KS][4];
  {
    const uint16_t* qrA = p.q + (static_cast<int64_t>(qs + (liveA ? tokA : 0)) * p.num_heads + headA) * D;
    const uint16_t* qrB = p.q + (static_cast<int64_t>(qs + (liveB ? tokB : 0)) * p.num_heads + headB) * D;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qa[ks][0] = liveA ? __ldg(reinterpret_cast<const uint32_t*>(qrA + 16 * ks + 2 * t)) : 0u;
      qa[ks][1] = liveB ? __ldg(reinterpret_cast<const uint32_t*>(qrB + 16 * ks + 2 * t)) : 0u;
      qa[ks][2] = liveA ? __ldg(reinterpret_cast<const uint32_t*>(qrA + 16 * ks + 8 + 2 * t)) : 0u;
      qa[ks][3] = liveB ? __ldg(reinterpret_cast<const uint32_t*>(qrB + 16 * ks + 8 + 2 * t)) : 0u;
    }
  }
  float o[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
  const int r = lane & 7, mat = lane >> 3;

  bool ok = true;
  for (int i = 0; i < n_tiles; ++i) {
    const int st = i % kStages;
    if (!mbar_wait(&full_bar[st], (i / kStages) & 1)) {
      ok = false;
      break;
    }
    const int t0 = i * kTile;
    if (t0 < warp_kv_end) {
      const uint8_t* kt = ring + st * Lay::kStageBytes;
      const uint8_t* vt = kt + Lay::kTileBytes;
      // S = Q K^T for 4 groups of 8 keys
      float s[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
        for (int kp = 0; kp < KS / 2; ++kp) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(swizzled_chunk<D / 64>(kt, 8 * nt + r, 4 * kp + mat, rows_shift), b0, b1, b2, b3);
          T::mma16816(s[nt], qa[2 * kp][0], qa[2 * kp][1], qa[2 * kp][2], qa[2 * kp][3], b0, b1);
          T::mma16816(s[nt], qa[2 * kp + 1][0], qa[2 * kp + 1][1], qa[2 * kp + 1][2],
                      qa[2 * kp + 1][3], b2, b3);
        }
      }
      // causal mask (also hides keys past the context and rows past the chunk)
      float tmA = -INFINITY, tmB = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = t0 + 8 * nt + 2 * t + e;
          s[nt][e] = (liveA && key <= posA) ? s[nt][e] * p.q_scale : -INFINITY;
          s[nt][2 + e] = (liveB && key <= posB) ? s[nt][2 + e] * p.q_scale : -INFINITY;
          tmA = fmaxf(tmA, s[nt][e]);
          tmB = fmaxf(tmB, s[nt][2 + e]);
        }
      tmA = fmaxf(tmA, __shfl_xor_sync(0xffffffffu, tmA, 1));
      tmA = fmaxf(tmA, __shfl_xor_sync(0xffffffffu, tmA, 2));
      tmB = fmaxf(tmB, __shfl_xor_sync(0xffffffffu, tmB, 1));
      tmB = fmaxf(tmB, __shfl_xor_sync(0xffffffffu, tmB, 2));
      const bool needA = tmA > mA + kRescaleThreshold, needB = tmB > mB + kRescaleThreshold;
      if (__any_sync(0xffffffffu, needA || needB)) {
        const float cA = needA ? ex2(mA - tmA) : 1.f, cB = needB ? ex2(mB - tmB) : 1.f;
        if (needA) mA = tmA;
        if (needB) mB = tmB;
        lA *= cA;
        lB *= cB;
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          o[j][0] *= cA;
          o[j][1] *= cA;
          o[j][2] *= cB;
          o[j][3] *= cB;
        }
      }
      // probabilities, and the P fragments of the two 16-key k-steps
      uint32_t ph[2][4], pl[2][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const float p0 = s[nt][0] == -INFINITY ? 0.f : ex2(s[nt][0] - mA);
        const float p1 = s[nt][1] == -INFINITY ? 0.f : ex2(s[nt][1] - mA);
        const float p2 = s[nt][2] == -INFINITY ? 0.f : ex2(s[nt][2] - mB);
        const float p3 = s[nt][3] == -INFINITY ? 0.f : ex2(s[nt][3] - mB);
        lA += p0 + p1;
        lB += p2 + p3;
        const int ks = nt >> 1, hi = (nt & 1) * 2;   // A regs: [row g | row g+8] x [k lo | k hi]
        const uint32_t hA = T::pack(p0, p1), hB = T::pack(p2, p3);
        ph[ks][hi] = hA;
        ph[ks][hi + 1] = hB;
        if constexpr (std::is_same<T, BF16>::value) {
          const float2 fa = T::to_float2(hA), fb = T::to_float2(hB);
          pl[ks][hi] = T::pack(p0 - fa.x, p1 - fa.y);
          pl[ks][hi + 1] = T::pack(p2 - fb.x, p3 - fb.y);
        }
      }
      // keys past the context: their V rows may hold anything
      const int kmax = kv_end - t0;                     // keys of this tile that exist
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
        for (int jq = 0; jq < NT / 2; ++jq) {          // two output tiles per ldmatrix
          // matrices: (keys 0-7, d-tile 2jq), (keys 8-15, 2jq), (keys 0-7, 2jq+1), (keys 8-15, 2jq+1)
          const int krow = 16 * ks + 8 * (mat & 1) + r;
          uint32_t b[4];
          ldsm_x4_t(swizzled_chunk<D / 64>(vt, krow, 2 * jq + (mat >> 1), rows_shift), b[0], b[1],
                    b[2], b[3]);
          if (kmax < kTile) {
            const int k0 = 16 * ks + 2 * t;
            const uint32_t keep0 = (k0 < kmax ? 0x0000ffffu : 0u) | (k0 + 1 < kmax ? 0xffff0000u : 0u);
            const uint32_t keep1 = (k0 + 8 < kmax ? 0x0000ffffu : 0u) | (k0 + 9 < kmax ? 0xffff0000u : 0u);
            b[0] &= keep0; b[2] &= keep0;
            b[1] &= keep1; b[3] &= keep1;
          }
          T::mma16816(o[2 * jq], ph[ks][0], ph[ks][1], ph[ks][2], ph[ks][3], b[0], b[1]);
          T::mma16816(o[2 * jq + 1], ph[ks][0], ph[ks][1], ph[ks][2], ph[ks][3], b[2], b[3]);
          if constexpr (std::is_same<T, BF16>::value) {
            T::mma16816(o[2 * jq], pl[ks][0], pl[ks][1], pl[ks][2], pl[ks][3], b[0], b[1]);
            T::mma16816(o[2 * jq + 1], pl[ks][0], pl[ks][1], pl[ks][2], pl[ks][3], b[2], b[3]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[st]);
  }
  if (!ok) flag_error(p.err, PKV_DEVERR_TIMEOUT);

  lA += __shfl_xor_sync(0xffffffffu, lA, 1);
  lA += __shfl_xor_sync(0xffffffffu, lA, 2);
  lB += __shfl_xor_sync(0xffffffffu, lB, 1);
  lB += __shfl_xor_sync(0xffffffffu, lB, 2);
  if (liveA) {
    const int64_t base = (static_cast<int64_t>(qs + tokA) * p.num_heads + headA) * D;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      store_elem(p.out, base + 8 * j + 2 * t, o[j][0] / lA, p.out_dtype);
      store_elem(p.out, base + 8 * j + 2 * t + 1, o[j][1] / lA, p.out_dtype);
    }
  }
  if (liveB) {
    const int64_t base = (static_cast<int64_t>(qs + tokB) * p.num_heads + headB) * D;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      store_elem(p.out, base + 8 * j + 2 * t, o[j][2] / lB, p.out_dtype);
      store_elem(p.out, base + 8 * j + 2 * t + 1, o[j][3] / lB, p.out_dtype);
    }
  }
}

template <int D, typename T>
static cudaError_t launch(const CUtensorMap& tk, const CUtensorMap& tv, const Params& p,
                          int num_kv_heads, int num_seqs, cudaStream_t s) {
  auto kern = prefill_kernel<D, T>;
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [&] {
    attr = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Layout<D>::kSmem);
  });
  if (attr != cudaSuccess) return attr;
  const int tiles = (p.max_query_len * p.group + kRows - 1) / kRows;
  dim3 grid(tiles, num_kv_heads, num_seqs);
  kern<<<grid, kThreads, Layout<D>::kSmem, s>>>(tk, tv, p);
  return cudaGetLastError();
}

}  // namespace prefill
}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_paged_attention_prefill(
    void* out, int out_dtype, const void* q, const void* k_cache, const void* v_cache,
    int kv_dtype, const int32_t* block_tables, const int32_t* context_lens,
    const int32_t* query_start, int num_seqs, int num_heads, int num_kv_heads, int head_size,
    int num_blocks, int block_size, int max_blocks_per_seq, int max_query_len, float scale,
    int32_t* err_flag, void* stream) {
  if (num_seqs < 0 || num_seqs > 65535) return PKV_EINVAL;
  if (num_seqs == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start)
    return PKV_EINVAL;
  if (kv_dtype != PKV_F16 && kv_dtype != PKV_BF16) return PKV_EINVAL;
  if (out_dtype != PKV_F16 && out_dtype != PKV_BF16 && out_dtype != PKV_F32) return PKV_EINVAL;
  if (head_size != 64 && head_size != 128) return PKV_EINVAL;
  if (num_kv_heads < 1 || num_heads < num_kv_heads || num_heads % num_kv_heads != 0)
    return PKV_EINVAL;
  const int group = num_heads / num_kv_heads;
  if (prefill::kRows % group != 0) return PKV_EINVAL;
  if (block_size < 8 || block_size > 256 || (block_size & (block_size - 1)) != 0)
    return PKV_EINVAL;
  if (num_blocks < 1 || max_blocks_per_seq < 1 || max_query_len < 1) return PKV_EINVAL;
  if (static_cast<int64_t>(num_blocks) * block_size > INT32_MAX) return PKV_EINVAL;
  if (static_cast<int64_t>(max_blocks_per_seq) * block_size > INT32_MAX / 2) return PKV_EINVAL;
  if (static_cast<int64_t>(max_query_len) * group / prefill::kRows > 65535) return PKV_EINVAL;
  if (!std::isfinite(scale)) return PKV_EINVAL;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_EINVAL;

  const int box_rows = std::min(block_size, prefill::kTile);
  CUtensorMap tk, tv;
  const int64_t slots = static_cast<int64_t>(num_blocks) * block_size;
  if (!encode_cache_map(&tk, k_cache, head_size, num_kv_heads, slots, box_rows, true) ||
      !encode_cache_map(&tv, v_cache, head_size, num_kv_heads, slots, box_rows, true))
    return PKV_ECUDA;
  prefill::Params p{};
  p.out = out;
  p.out_dtype = out_dtype;
  p.q = static_cast<const uint16_t*>(q);
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.query_start = query_start;
  p.err = err_flag;
  p.num_heads = num_heads;
  p.group = group;
  p.num_blocks = num_blocks;
  p.block_size = block_size;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.max_query_len = max_query_len;
  p.box_rows = box_rows;
  p.q_scale = scale * prefill::kLog2e;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (head_size == 128)
    e = kv_dtype == PKV_F16 ? prefill::launch<128, F16>(tk, tv, p, num_kv_heads, num_seqs, s)
                            : prefill::launch<128, BF16>(tk, tv, p, num_kv_heads, num_seqs, s);
  else
    e = kv_dtype == PKV_F16 ? prefill::launch<64, F16>(tk, tv, p, num_kv_heads, num_seqs, s)
                            : prefill::launch<64, BF16>(tk, tv, p, num_kv_heads, num_seqs, s);
  return e == cudaSuccess ? PKV_OK : PKV_ECUDA;
}
