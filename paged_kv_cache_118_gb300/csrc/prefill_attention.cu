// Paged chunked-prefill attention for sm_103a on the 5th-generation tensor
// cores.
//
// What is computed: a sequence with L tokens in its cache receives a chunk of
// C query tokens, its last C positions (their keys and values already
// written); query i (position L - C + i) attends over positions 0..L-C+i of the
// sequence's paged history with one softmax denominator (chunked prefill,
// zhy-blog.vercel.app §4: a long prompt is processed in chunks whose masks
// follow their position; "079｜vLLM 与 PagedAttention" §2 for the single global
// denominator). Decode is the case C = 1.
//
// How (one CTA per 256 query rows, KV head and sequence: two query tiles of
// 128 rows; a row is one (query token, query head of the KV head's group), so
// 128/G tokens per query tile):
//  * warp 0 streams 64-key tiles of K and V over the causal range only, one
//    TMA copy per physical block and 128-byte line (128-byte swizzle), each
//    lane issuing one, into a 5-stage ring completing on mbarriers; both
//    query tiles use each K/V tile;
//  * warp 1 owns the tensor memory (per query tile: two 64-column score
//    buffers and the D-column output) and issues, from one thread, S = Q K^T
//    (M = 128, N = 64, K = D) into a score buffer and O += P V (M = 128,
//    N = D, K = 64, P read from tensor memory) into the output, each
//    followed by a commit to an mbarrier; the next tile's S is issued before
//    this tile's P V;
//  * a softmax warpgroup per query tile, one thread per query row (its TMEM
//    lane): the row's 64 scores come out of tensor memory, the causal mask
//    and a base-2 online softmax with lazy rescale (the output row is
//    rescaled in place only when the running maximum grows by more than 2^8)
//    give P, written back over the scores as 16-bit pairs, where the P V
//    product reads it; the output row is divided by the row sum at the end.
// Every wait is bounded; a chunk or context length out of range is skipped
// and reported.

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

constexpr int kRows = 128;             // query rows of one query tile: the TMEM lanes
constexpr int kQTiles = 2;             // query tiles per CTA, sharing every K/V tile
constexpr int kKeys = 64;              // keys per tile
constexpr int kStages = 5;
constexpr int kThreads = 128 + kQTiles * 128;   // warp 0: copies; warp 1: MMA; 4 warps per query tile
constexpr int kSoftmaxWarp0 = 4;
// per query tile t, from column 256 t: S0 [0, 64), S1 [64, 128), O [128, 128 + D)
constexpr uint32_t kTmemCols = 256 * kQTiles;
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
  int box_rows;                        // rows per TMA copy: min(block_size, kKeys)
  float q_scale;                       // scale * log2(e)
};

// Shared memory, from a 1024-byte aligned base. Every operand is stored as
// 128-byte rows with the 128-byte swizzle (16-byte chunk c of the row at
// position n sits at c ^ (n % 8)), 8-row groups 1024 bytes apart:
//  Q, per query tile: D/64 column blocks of 128 rows (A of S, K-major);
//  each stage: K then V, each D/64 line blocks of 64 key rows (B of S,
//  K-major; B of P V, MN-major with the next 64 columns one line block on);
//  (P stays in tensor memory.)
template <int D>
struct Layout {
  static constexpr int NH = D / 64;
  static constexpr int kQBytes = kRows * D * 2;
  static constexpr int kLineBytes = kKeys * 128;          // one line block of a K or V tile
  static constexpr int kTileBytes = NH * kLineBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kOffStages = kQTiles * kQBytes;
  static constexpr int kOffBars = kOffStages + kStages * kStageBytes;
  // stage_full[S], stage_empty[S], q_full, per query tile s_full[2], p_full[2],
  // pv_done[2]; drain, tail (V rows past the last key zeroed)
  static constexpr int kNumBars = 2 * kStages + 1 + 6 * kQTiles + 2;
  static constexpr int kOffTmem = kOffBars + kNumBars * 8;
  static constexpr int kSmem = 1024 + kOffTmem + 16;
};

template <typename T>
__device__ __forceinline__ void store_row(void* out, int out_dtype, int64_t base, const float* v,
                                          int n) {
  // n values of one output row, 16 bytes at a time
  if (out_dtype == PKV_F32) {
    float4* d = reinterpret_cast<float4*>(static_cast<float*>(out) + base);
    for (int i = 0; i < n / 4; ++i) d[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  } else {
    uint4* d = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + base);
    for (int i = 0; i < n / 8; ++i) {
      uint4 w;
      if (out_dtype == PKV_F16) {
        w.x = F16::pack(v[8 * i], v[8 * i + 1]);
        w.y = F16::pack(v[8 * i + 2], v[8 * i + 3]);
        w.z = F16::pack(v[8 * i + 4], v[8 * i + 5]);
        w.w = F16::pack(v[8 * i + 6], v[8 * i + 7]);
      } else {
        w.x = BF16::pack(v[8 * i], v[8 * i + 1]);
        w.y = BF16::pack(v[8 * i + 2], v[8 * i + 3]);
        w.z = BF16::pack(v[8 * i + 4], v[8 * i + 5]);
        w.w = BF16::pack(v[8 * i + 6], v[8 * i + 7]);
      }
      d[i] = w;
    }
  }
}

template <int D, typename T>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const Params p) {
  using Lay = Layout<D>;
  constexpr int NH = Lay::NH;
  constexpr bool kBF16 = std::is_same<T, BF16>::value;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* qtiles = smem;
  uint8_t* stages = smem + Lay::kOffStages;
  uint64_t* stage_full = reinterpret_cast<uint64_t*>(smem + Lay::kOffBars);
  uint64_t* stage_empty = stage_full + kStages;
  uint64_t* q_full = stage_empty + kStages;
  uint64_t* tbars = q_full + 1;                 // per query tile: s_full[2], p_full[2], pv_done[2]
  uint64_t* drain = tbars + 6 * kQTiles;
  uint64_t* tail = drain + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kOffTmem);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int seq = blockIdx.z;
  const int kvh = blockIdx.y;
  const int G = p.group;
  const int tok_per_qt = kRows / G;                        // chunk tokens per query tile
  const int tok0 = blockIdx.x * kQTiles * tok_per_qt;      // first chunk token of the CTA
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
  // key tiles each query tile reads (0 for a tile wholly past the chunk)
  int nt[kQTiles];
#pragma unroll
  for (int t = 0; t < kQTiles; ++t) {
    const int first = tok0 + t * tok_per_qt;
    const int kv_end_t = L - C + min(C, first + tok_per_qt);
    nt[t] = first < C ? (kv_end_t + kKeys - 1) / kKeys : 0;
  }
  const int kv_end = L - C + min(C, tok0 + kQTiles * tok_per_qt);   // keys the CTA reads
  const int n_tiles = (kv_end + kKeys - 1) / kKeys;
  // the lowest query tile that reads the last key tile zeroes its V rows past kv_end
  int zt = 0;
  while (nt[zt] != n_tiles) ++zt;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&stage_full[i], 1);
      mbar_init(&stage_empty[i], 1);
    }
    mbar_init(q_full, kQTiles * kRows);
    for (int t = 0; t < kQTiles; ++t)
      for (int i = 0; i < 2; ++i) {
        mbar_init(&tbars[6 * t + i], 1);              // s_full
        mbar_init(&tbars[6 * t + 2 + i], kRows);      // p_full
        mbar_init(&tbars[6 * t + 4 + i], 1);          // pv_done
      }
    mbar_init(drain, 1);
    mbar_init(tail, kRows);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------- copies
    // Lane l copies line (l / 2) % NH of K (l even) or V (l odd) for the
    // tile's copy l / (2 NH); it reads that copy's block id before the wait
    // for the stage, so the read overlaps the wait.
    if (lane == 0) {
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
    }
    const uint64_t policy = l2_evict_first_policy();
    const int R = p.box_rows;
    const uint32_t copy_bytes = static_cast<uint32_t>(R) * 128;
    const int32_t* row = p.block_tables + static_cast<int64_t>(seq) * p.max_blocks_per_seq;
    const int my_c = lane / (2 * NH);
    const int my_h = (lane >> 1) % NH;
    const CUtensorMap* my_map = (lane & 1) ? &tm_v : &tm_k;
    const uint32_t my_off =
        (lane & 1) * Lay::kTileBytes + my_h * Lay::kLineBytes + my_c * copy_bytes;
    int last_issued[kStages];
#pragma unroll
    for (int i = 0; i < kStages; ++i) last_issued[i] = -1;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int st = j % kStages;
      const int t0 = j * kKeys;
      const int copies = (min(kKeys, kv_end - t0) + R - 1) / R;   // copies of R rows cover the keys
      const bool mine = my_c < copies;
      const int tk = t0 + my_c * R;                        // first key of the lane's copy
      int32_t id = mine ? __ldg(row + tk / B) : 0;
      bool e_ok = true;
      if (lane == 0 && j >= kStages) e_ok = mbar_wait(&stage_empty[st], ((j / kStages) & 1) ^ 1);
      if (!__shfl_sync(0xffffffffu, e_ok, 0)) {
        ok = false;
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&stage_full[st], 2u * NH * copies * copy_bytes);
        last_issued[st] = j;
      }
      __syncwarp();
      if (mine) {
        if (id < 0 || id >= p.num_blocks) {
          flag_error(p.err, PKV_DEVERR_BLOCK_ID);
          id = 0;
        }
        tma_load_4d(stages + st * Lay::kStageBytes + my_off, my_map, &stage_full[st], 0,
                    id * B + tk % B, kvh, my_h, policy);
      }
    }
    if (!ok && lane == 0) {
      flag_error(p.err, PKV_DEVERR_TIMEOUT);
      for (int st = 0; st < kStages; ++st)
        if (last_issued[st] >= 0) mbar_wait(&stage_full[st], (last_issued[st] / kStages) & 1);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t kIdescS = mma_idesc_f16(kBF16, kRows, kKeys, false);
      constexpr uint32_t kIdescO = mma_idesc_f16(kBF16, kRows, D, true);
      bool ok = mbar_wait(q_full, 0);
      tc_fence_after();
      // Descriptors are built once; a k-step or another buffer only moves the
      // start address (bits 0-13, in 16-byte units), so it is an addition.
      const uint64_t dq0 = smem_desc_sw128(qtiles, 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(stages, 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(stages + Lay::kTileBytes, Lay::kLineBytes, 1024);
      // S of query tile t for key tile j, into its score buffer j % 2, once
      // the P V product two tiles back has read the P held there
      auto issue_s = [&](int t, int j) -> bool {
        const int b = j & 1;
        if (j >= 2 && !mbar_wait(&tbars[6 * t + 4 + b], ((j - 2) >> 1) & 1)) return false;
        tc_fence_after();
        const uint64_t dq = dq0 + (t * Lay::kQBytes >> 4);
        const uint64_t dk = dk0 + ((j % kStages) * Lay::kStageBytes >> 4);
        const uint32_t d = tbase + 256 * t + b * kKeys;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          // 64-element column block ks / 4, 32 bytes per k-step inside it
          const uint32_t qo = ((ks >> 2) * kRows * 128 + (ks & 3) * 32) >> 4;
          const uint32_t ko = ((ks >> 2) * Lay::kLineBytes + (ks & 3) * 32) >> 4;
          tc_mma_f16(d, dq + qo, dk + ko, kIdescS, ks > 0 ? 1u : 0u);
        }
        tc_commit(&tbars[6 * t + b]);                       // s_full
        return true;
      };
      // O of query tile t += P V for key tile j; P (16-bit, two per column)
      // is in the first 32 columns of score buffer j % 2, 8 columns per k-step
      auto issue_pv = [&](int t, int j) -> bool {
        const int b = j & 1;
        if (!mbar_wait(&tbars[6 * t + 2 + b], (j >> 1) & 1)) return false;   // p_full
        tc_fence_after();
        // V as B, MN-major: 16 keys are two 8-row groups; the next 64 columns
        // of D are one line block (kLineBytes) on
        const uint64_t dv = dv0 + ((j % kStages) * Lay::kStageBytes >> 4);
        const uint32_t a = tbase + 256 * t + b * kKeys;
        const uint32_t d = tbase + 256 * t + 128;
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          tc_mma_f16_ts(d, a + kk * 8, dv + ((kk * 16 * 128) >> 4), kIdescO,
                        (j > 0 || kk > 0) ? 1u : 0u);
        if constexpr (kBF16) {                              // + (p - hi) V
#pragma unroll
          for (int kk = 0; kk < kKeys / 16; ++kk)
            tc_mma_f16_ts(d, a + kKeys / 2 + kk * 8, dv + ((kk * 16 * 128) >> 4), kIdescO, 1u);
        }
        tc_commit(&tbars[6 * t + 4 + b]);                   // pv_done
        return true;
      };
      auto issue_s_all = [&](int j) -> bool {
        if (!mbar_wait(&stage_full[j % kStages], (j / kStages) & 1)) return false;
        for (int t = 0; t < kQTiles; ++t)
          if (j < nt[t] && !issue_s(t, j)) return false;
        return true;
      };
      if (ok) ok = issue_s_all(0);
      for (int j = 0; ok && j < n_tiles; ++j) {
        if (j + 1 < n_tiles) ok = issue_s_all(j + 1);
        for (int t = 0; ok && t < kQTiles; ++t)
          if (j < nt[t]) ok = issue_pv(t, j);
        if (ok) tc_commit(&stage_empty[j % kStages]);       // K and V of tile j are read
      }
      if (!ok) flag_error(p.err, PKV_DEVERR_TIMEOUT);
      // everything issued has completed before the columns are freed
      tc_commit(drain);
      if (!mbar_wait(drain, 0)) flag_error(p.err, PKV_DEVERR_TIMEOUT);
    }
  } else if (warp >= kSoftmaxWarp0) {
    // ---------------------------------------------------------- softmax
    const int t = (warp - kSoftmaxWarp0) >> 2;             // query tile
    const int r = ((warp - kSoftmaxWarp0) & 3) * 32 + lane;   // row of the tile = TMEM lane
    const uint32_t tl = tbase + 256 * t + ((static_cast<uint32_t>(warp & 3) * 32) << 16);
    uint64_t* s_full = &tbars[6 * t];
    uint64_t* p_full = s_full + 2;
    uint64_t* pv_done = s_full + 4;
    uint8_t* qtile = qtiles + t * Lay::kQBytes;
    const int n_my = nt[t];
    const int tok = tok0 + t * tok_per_qt + r / G;
    const int head = kvh * G + r % G;
    const bool live = tok < C;
    const int pos = L - C + tok;
    // this row of Q into the A layout of S (zeros past the chunk)
    {
      const uint4* src = reinterpret_cast<const uint4*>(
          p.q + (static_cast<int64_t>(qs + (live ? tok : 0)) * p.num_heads + head) * D);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const int h = c >> 3, cc = c & 7;
        uint4 v = live ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(qtile + h * kRows * 128 + r * 128 + ((cc ^ (r & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();
      mbar_arrive(q_full);
    }
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_my; ++j) {
      const int b = j & 1;
      // tcgen05.ld/st are warp-collective: every wait result is made warp-uniform
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[b], (j >> 1) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[kKeys];
#pragma unroll
      for (int h = 0; h < kKeys / 32; ++h) {
        uint32_t raw[32];
        tmem_ld32(tl + b * kKeys + h * 32, raw);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[h * 32 + i] = __uint_as_float(raw[i]);
      }
      // causal mask (also hides keys past the context and rows past the chunk);
      // the row maximum is taken on unscaled scores (the scale is positive)
      const int key0 = j * kKeys;
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (live && key0 + kKeys - 1 <= pos) {              // every key of the tile is visible
#pragma unroll
        for (int i = 0; i < kKeys; ++i) mx[i & 3] = fmaxf(mx[i & 3], s[i]);
      } else {
#pragma unroll
        for (int i = 0; i < kKeys; ++i) {
          s[i] = (live && key0 + i <= pos) ? s[i] : -INFINITY;
          mx[i & 3] = fmaxf(mx[i & 3], s[i]);
        }
      }
      const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * p.q_scale;
      const bool need = mt > m + kRescaleThreshold;
      if (__any_sync(0xffffffffu, need)) {                 // the whole warp takes this branch
        const float mn = need ? mt : m;
        if (j > 0) {
          // the output rows hold earlier tiles: rescale them once their P V is
          // done (factor 1 on rows that keep their max or hold nothing yet)
          if (!__all_sync(0xffffffffu, mbar_wait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float c = (need && m != -INFINITY) ? ex2(m - mn) : 1.f;
#pragma unroll
          for (int h = 0; h < D / 32; ++h) {
            uint32_t raw[32];
            tmem_ld32(tl + 128 + h * 32, raw);
#pragma unroll
            for (int i = 0; i < 32; ++i) raw[i] = __float_as_uint(__uint_as_float(raw[i]) * c);
            tmem_st32(tl + 128 + h * 32, raw);
          }
          l *= c;
        }
        m = mn;
      }
      // p = 2^(scale s - m): a masked score is -inf and gives 0 (m is finite
      // on a live row from its first tile on; a row past the chunk writes 0)
      const float nm = live ? -m : 0.f;
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
      // P as 16-bit pairs over the first 32 columns of the scores; bf16 P also
      // keeps its rounding error (p - hi) in the next 32, read by a second P V
      uint32_t pk[kKeys / 2], pl[kKeys / 2];
#pragma unroll
      for (int i = 0; i < kKeys; i += 2) {
        const float e0 = live ? ex2(fmaf(s[i], p.q_scale, nm)) : 0.f;
        const float e1 = live ? ex2(fmaf(s[i + 1], p.q_scale, nm)) : 0.f;
        ls[(i >> 1) & 3] += e0 + e1;
        pk[i >> 1] = T::pack(e0, e1);
        if constexpr (kBF16) {
          const float2 h = T::to_float2(pk[i >> 1]);
          pl[i >> 1] = T::pack(e0 - h.x, e1 - h.y);
        }
      }
      l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      tmem_st32(tl + b * kKeys, pk);                        // over the scores of this tile
      if constexpr (kBF16) tmem_st32(tl + b * kKeys + kKeys / 2, pl);
      if (j == n_tiles - 1 && kv_end - key0 < kKeys) {
        if (t == zt) {
          // V rows past the last key may hold anything (0 x NaN is NaN): zero them
          uint8_t* vt = stages + (j % kStages) * Lay::kStageBytes + Lay::kTileBytes;
          const int valid = kv_end - key0;
          for (int idx = r; idx < NH * kKeys; idx += kRows) {
            const int kr = idx % kKeys, h = idx / kKeys;
            if (kr >= valid) {
              uint4* d = reinterpret_cast<uint4*>(vt + h * Lay::kLineBytes + kr * 128);
#pragma unroll
              for (int i = 0; i < 8; ++i) d[i] = make_uint4(0u, 0u, 0u, 0u);
            }
          }
          fence_proxy_async_smem();
          mbar_arrive(tail);
        } else if (!mbar_wait(tail, 0)) {                   // a lower query tile zeroes them
          ok = false;
          break;
        }
      }
      tc_fence_before();
      mbar_arrive(&p_full[b]);
    }
    if (n_my > 0) {
      if (__all_sync(0xffffffffu,
                     ok && mbar_wait(&pv_done[(n_my - 1) & 1], ((n_my - 1) >> 1) & 1))) {
        tc_fence_after();
        float o[D];
#pragma unroll
        for (int h = 0; h < D / 32; ++h) {
          uint32_t raw[32];
          tmem_ld32(tl + 128 + h * 32, raw);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[h * 32 + i] = __uint_as_float(raw[i]);
        }
        if (live) {
          const float inv = 1.f / l;
#pragma unroll
          for (int i = 0; i < D; ++i) o[i] *= inv;
          store_row<T>(p.out, p.out_dtype,
                       (static_cast<int64_t>(qs + tok) * p.num_heads + head) * D, o, D);
        }
      } else {
        flag_error(p.err, PKV_DEVERR_TIMEOUT);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

template <int D, typename T>
static cudaError_t launch(const CUtensorMap& tk, const CUtensorMap& tv, const Params& p,
                          int num_kv_heads, int num_seqs, cudaStream_t s) {
  auto kern = prefill_kernel<D, T>;
  // one CTA per SM: it holds all 512 tensor-memory columns, so shared memory is
  // requested past half an SM even where the layout needs less (d = 64)
  constexpr int kSmemLaunch = Layout<D>::kSmem > 120 * 1024 ? Layout<D>::kSmem : 120 * 1024;
  const cudaError_t attr =
      prepare_kernel(reinterpret_cast<const void*>(kern), kThreads, kSmemLaunch, nullptr);
  if (attr != cudaSuccess) return attr;
  const int tiles = (p.max_query_len * p.group + kQTiles * kRows - 1) / (kQTiles * kRows);
  dim3 grid(tiles, num_kv_heads, num_seqs);
  kern<<<grid, kThreads, kSmemLaunch, s>>>(tk, tv, p);
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
  if (!std::isfinite(scale) || !(scale > 0.f)) return PKV_EINVAL;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_EINVAL;

  const int box_rows = std::min(block_size, prefill::kKeys);
  CUtensorMap tk, tv;
  const int64_t slots = static_cast<int64_t>(num_blocks) * block_size;
  if (!encode_cache_map(&tk, k_cache, head_size, num_kv_heads, slots, box_rows, kLineSwizzled) ||
      !encode_cache_map(&tv, v_cache, head_size, num_kv_heads, slots, box_rows, kLineSwizzled))
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
