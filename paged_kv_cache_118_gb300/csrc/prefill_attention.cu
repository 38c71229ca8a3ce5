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
// How (persistent: one CTA per SM takes work items, each 256 query rows, a
// KV head and a sequence: two query tiles of 128 rows; a row is one (query
// token, query head of the KV head's group), so 128/G tokens per query tile;
// items with more keys first, the CTA's own index first, then claims from a
// counter in the caller's workspace):
//  * warp 0 claims items and publishes them to the other warps, then streams
//    each item's causal key range in 128-key tiles, K and V of a tile into
//    two slots of one ring (so a K tile is released as soon as its score
//    products are done), one TMA copy per physical block and 128-byte line
//    (128-byte swizzle), each lane issuing one; both query tiles use each
//    K/V tile, and the ring runs on from one item into the next;
//  * warp 1 owns the tensor memory (per query tile: a 128-column score
//    buffer and the D-column output) and issues, from one thread,
//    S = Q K^T (M = 128, N = 128, K = D) and O += P V (M = 128, N = D,
//    K = 128, P read from tensor memory), each followed by a commit to an
//    mbarrier; a query tile's next S follows its P V. A product issue
//    costs one thread tens of cycles whatever its size, so the products
//    are made as wide as tensor memory allows;
//  * one thread of warp 2 loads each item's query rows by TMA once the
//    previous item's S products are done;
//  * a softmax warpgroup per query tile, one thread per query row (its TMEM
//    lane): it reads the row's 128 scores from tensor memory in one load (a
//    tensor-memory round trip costs hundreds of cycles under load, so a tile
//    takes one load and one store), runs a
//    base-2 online softmax with lazy rescale (the output row is rescaled in
//    place only when the running maximum grows by more than 2^8) and writes
//    P back over the scores as 16-bit pairs, where the P V product reads it;
//    the output row is divided by the row sum at the item's end and the
//    output columns are handed back to the MMA.
// Every wait is bounded; a chunk or context length out of range, or a chunk
// whose rows would pass the end of q, is skipped and reported.

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <type_traits>

#include "pagedkv.h"
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {
namespace prefill {

constexpr int kRows = 128;             // query rows of one query tile: the TMEM lanes
constexpr int kQTiles = 2;             // query tiles per item, sharing every K/V tile
constexpr int kKeys = 128;             // keys per tile
constexpr int kThreads = 128 + kQTiles * 128;   // warp 0: items, K/V; warp 1: MMA; warp 2: Q; 4 warps per query tile
constexpr int kSoftmaxWarp0 = 4;
// per query tile t, from column 256 t: S (P over it) [0, 128), O [128, 128 + D)
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
  int* counter;                        // item counter, zero at launch
  int num_seqs;
  int num_heads;
  int num_kv_heads;
  int group;                           // query heads per KV head
  int num_blocks;
  int block_size;
  int max_blocks_per_seq;
  int max_query_len;
  int total_queries;                   // rows of q and out
  int qblocks;                         // 256-row query blocks of the longest chunk
  int total_items;                     // qblocks * num_seqs * num_kv_heads
  int box_rows;                        // rows per TMA copy: min(block_size, 64)
  float q_scale;                       // scale * log2(e)
};

// One work item: query block qb (rows 256 qb ..) of sequence seq and KV head
// kvh; qs, C, L: the sequence's first query row, chunk length and context.
struct Item {
  int seq;                             // -1: no more items
  int kvh, qb, qs, C, L;
};

// What an item reads: key tiles of each query tile (the causal range of its
// last row), keys and key tiles of the whole item, and the lowest query tile
// that reads the last key tile (it zeroes that tile's V rows past the last key).
struct Shape {
  int nt[kQTiles];
  int kv_end, n_tiles, zt;
};

__device__ __forceinline__ Shape item_shape(const Item& it, int G) {
  Shape sh;
  const int tok_per_qt = kRows / G;
  const int tok0 = it.qb * kQTiles * tok_per_qt;
#pragma unroll
  for (int t = 0; t < kQTiles; ++t) {
    const int first = tok0 + t * tok_per_qt;
    const int kv_end_t = it.L - it.C + min(it.C, first + tok_per_qt);
    sh.nt[t] = first < it.C ? (kv_end_t + kKeys - 1) / kKeys : 0;
  }
  sh.kv_end = it.L - it.C + min(it.C, tok0 + kQTiles * tok_per_qt);
  sh.n_tiles = (sh.kv_end + kKeys - 1) / kKeys;
  sh.zt = 0;
  while (sh.nt[sh.zt] != sh.n_tiles) ++sh.zt;
  return sh;
}

// Shared memory, from a 1024-byte aligned base. Every operand is stored as
// 128-byte rows with the 128-byte swizzle (16-byte chunk c of the row at
// position n sits at c ^ (n % 8)), 8-row groups 1024 bytes apart:
//  Q, per query tile: D/64 column blocks of 128 rows (A of S, K-major);
//  a ring of slots, each holding a K tile or a V tile: D/64 line blocks of
//  128 key rows (K: B of S, K-major; V: B of P V, MN-major with the next 64
//  columns one line block on); (P stays in tensor memory.) Then the
//  barriers and two item slots.
template <int D>
struct Layout {
  static constexpr int NH = D / 64;
  static constexpr int kQBytes = kRows * D * 2;
  static constexpr int kLineBytes = kKeys * 128;          // one line block of a K or V tile
  static constexpr int kSlotBytes = NH * kLineBytes;      // one K or V tile
  static constexpr int kSlots = D == 128 ? 5 : 8;
  static constexpr int kOffSlots = kQTiles * kQBytes;
  static constexpr int kOffBars = kOffSlots + kSlots * kSlotBytes;
  // slot_full[S], slot_empty[S], item_full[2], item_empty[2], q_full, q_free,
  // per query tile s_full, p_full, pv_done, o_free; drain, tail
  static constexpr int kNumBars = 2 * kSlots + 4 + 2 + 4 * kQTiles + 2;
  static constexpr int kOffItems = kOffBars + kNumBars * 8;
  static constexpr int kOffTmem = kOffItems + 2 * static_cast<int>(sizeof(Item));
  static constexpr int kSmem = 1024 + kOffTmem + 16;
  static_assert(kSmem <= 232448, "shared memory of one CTA");
};

template <typename T>
__device__ __forceinline__ void store_row(void* out, int out_dtype, int64_t base, const float* v,
                                          int n) {
  // n values of one output row, 32 bytes per store where the output is
  // 32-byte aligned (the ABI asks for 16), else 16 bytes per store
  if ((reinterpret_cast<uintptr_t>(out) & 31) == 0) {
    if (out_dtype == PKV_F32) {
      float* d = static_cast<float*>(out) + base;
      for (int i = 0; i < n / 8; ++i)
        asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(d + 8 * i),
                     "f"(v[8 * i]), "f"(v[8 * i + 1]), "f"(v[8 * i + 2]), "f"(v[8 * i + 3]),
                     "f"(v[8 * i + 4]), "f"(v[8 * i + 5]), "f"(v[8 * i + 6]), "f"(v[8 * i + 7])
                     : "memory");
    } else {
      uint16_t* d = static_cast<uint16_t*>(out) + base;
      for (int i = 0; i < n / 16; ++i) {
        uint32_t w[8];
        for (int j = 0; j < 8; ++j)
          w[j] = out_dtype == PKV_F16 ? F16::pack(v[16 * i + 2 * j], v[16 * i + 2 * j + 1])
                                      : BF16::pack(v[16 * i + 2 * j], v[16 * i + 2 * j + 1]);
        asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(d + 16 * i),
                     "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]),
                     "r"(w[7])
                     : "memory");
      }
    }
    return;
  }
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

// Barrier phases. Each barrier completes one phase per event, and every wait
// names the parity of the phase it needs; no barrier can run two phases ahead
// of a waiter, because each producer's next phase needs the waiter's
// progress:
//  * slot_full / slot_empty: per K or V tile of the CTA (g, counted over all
//    items: K of key tile j in slot g, its V in slot g + 1); item_full /
//    item_empty: per item, two slots;
//  * q_full (256 arrivals: every softmax thread wrote its query row) and
//    q_free (the item's S products are done): once per item;
//  * s_full / p_full / pv_done of query tile t: per key tile that t reads,
//    counted over all items (gt); o_free of t: per item in which t reads keys
//    (its output columns were read back);
//  * tail: per item whose last key tile is partial.
template <int D, typename T>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const __grid_constant__ CUtensorMap tm_q, const Params p) {
  using Lay = Layout<D>;
  constexpr int NH = Lay::NH;
  constexpr int S = Lay::kSlots;
  constexpr bool kBF16 = std::is_same<T, BF16>::value;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* qtiles = smem;
  uint8_t* slots = smem + Lay::kOffSlots;
  uint64_t* slot_full = reinterpret_cast<uint64_t*>(smem + Lay::kOffBars);
  uint64_t* slot_empty = slot_full + S;
  uint64_t* item_full = slot_empty + S;
  uint64_t* item_empty = item_full + 2;
  uint64_t* q_full = item_empty + 2;
  uint64_t* q_free = q_full + 1;
  uint64_t* tbars = q_free + 1;                 // per query tile: s_full, p_full, pv_done, o_free
  uint64_t* drain = tbars + 4 * kQTiles;
  uint64_t* tail = drain + 1;
  Item* items = reinterpret_cast<Item*>(smem + Lay::kOffItems);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kOffTmem);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;
  const int B = p.block_size;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&slot_full[i], 1);
      mbar_init(&slot_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&item_full[i], 1);
      mbar_init(&item_empty[i], kQTiles * kRows + 2);   // the softmax, MMA and query threads
    }
    mbar_init(q_full, 1);
    mbar_init(q_free, 1);
    for (int t = 0; t < kQTiles; ++t) {
      mbar_init(&tbars[4 * t], 1);              // s_full
      mbar_init(&tbars[4 * t + 1], kRows);      // p_full
      mbar_init(&tbars[4 * t + 2], 1);          // pv_done
      mbar_init(&tbars[4 * t + 3], kRows);      // o_free
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
    // ---------------------------------------------------------- items, copies
    // Lane l copies line l % NH of the tile's copy l / NH (R rows of one
    // block); it reads that copy's block id before the waits for the slots,
    // and issues the copy into the K slot and then into the V slot.
    if (lane == 0) {
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
    }
    const uint64_t policy = l2_evict_first_policy();
    const int R = p.box_rows;
    const uint32_t copy_bytes = static_cast<uint32_t>(R) * 128;
    const int my_c = lane / NH;
    const int my_h = lane % NH;
    const uint32_t my_off = my_h * Lay::kLineBytes + my_c * copy_bytes;
    const int per_qb = p.num_seqs * p.num_kv_heads;
    const int tok_per_item = kQTiles * (kRows / G);
    const int max_ctx = p.max_blocks_per_seq * B;
    int g = 0;                                  // slots filled
    int k = 0;                                  // items published
    bool ok = true;
    for (int claim = 0; ok; ++claim) {
      // the CTA's own index first (no round trip), then the shared counter;
      // items with more keys (later query blocks) come first
      int u = static_cast<int>(blockIdx.x);
      if (claim > 0) {
        if (lane == 0) u = static_cast<int>(gridDim.x) + atomicAdd(p.counter, 1);
        u = __shfl_sync(0xffffffffu, u, 0);
      }
      Item it{-1, 0, 0, 0, 0, 0};
      if (u < p.total_items) {
        const int qb = p.qblocks - 1 - u / per_qb;
        const int rem = u - (p.qblocks - 1 - qb) * per_qb;
        const int seq = rem / p.num_kv_heads;
        const int kvh = rem - seq * p.num_kv_heads;
        int v = 0;
        if (lane < 3) v = __ldg(lane == 2 ? p.context_lens + seq : p.query_start + seq + lane);
        const int qs = __shfl_sync(0xffffffffu, v, 0);
        const int C = __shfl_sync(0xffffffffu, v, 1) - qs;
        const int L = __shfl_sync(0xffffffffu, v, 2);
        if (C < 0 || C > p.max_query_len || C > L || L > max_ctx || qs < 0 ||
            qs > p.total_queries - C) {
          if (lane == 0 && qb == 0 && kvh == 0 && C != 0) flag_error(p.err, PKV_DEVERR_CONTEXT);
          continue;
        }
        if (qb * tok_per_item >= C) continue;   // no query rows in this block
        it = Item{seq, kvh, qb, qs, C, L};
      }
      const int slot = k & 1;
      if (k >= 2 && !__all_sync(0xffffffffu, mbar_wait(&item_empty[slot], ((k >> 1) & 1) ^ 1))) {
        ok = false;
        break;
      }
      if (lane == 0) {
        items[slot] = it;
        mbar_arrive(&item_full[slot]);
      }
      ++k;
      if (it.seq < 0) break;
      const Shape sh = item_shape(it, G);
      const int32_t* row = p.block_tables + static_cast<int64_t>(it.seq) * p.max_blocks_per_seq;
      for (int j = 0; ok && j < sh.n_tiles; ++j) {
        const int t0 = j * kKeys;
        const int copies = (min(kKeys, sh.kv_end - t0) + R - 1) / R;   // copies of R rows cover the keys
        const bool mine = my_c < copies;
        const int tk = t0 + my_c * R;                      // first key of the lane's copy
        int32_t id = mine ? __ldg(row + tk / B) : 0;
        if (mine && (id < 0 || id >= p.num_blocks)) {
          flag_error(p.err, PKV_DEVERR_BLOCK_ID);
          id = 0;
        }
        for (int kv = 0; kv < 2; ++kv, ++g) {
          const int st = g % S;
          if (g >= S &&
              !__all_sync(0xffffffffu, mbar_wait(&slot_empty[st], ((g / S) & 1) ^ 1))) {
            ok = false;
            break;
          }
          if (lane == 0) mbar_arrive_expect_tx(&slot_full[st], NH * copies * copy_bytes);
          __syncwarp();
          if (mine)
            tma_load_4d(slots + st * Lay::kSlotBytes + my_off, kv ? &tm_v : &tm_k, &slot_full[st], 0,
                        id * B + tk % B, it.kvh, my_h, policy);
        }
      }
    }
    if (!ok && lane == 0) {
      flag_error(p.err, PKV_DEVERR_TIMEOUT);
      // let the copies in flight (the last S slots filled) land
      for (int i = max(0, g - S); i < g; ++i) mbar_wait(&slot_full[i % S], (i / S) & 1);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t kIdescS = mma_idesc_f16(kBF16, kRows, kKeys, false);
      constexpr uint32_t kIdescO = mma_idesc_f16(kBF16, kRows, D, true);
      // Descriptors are built once; a k-step or another slot only moves the
      // start address (bits 0-13, in 16-byte units), so it is an addition.
      const uint64_t dq0 = smem_desc_sw128(qtiles, 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(slots, 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(slots, Lay::kLineBytes, 1024);
      int g = 0;                                // slots consumed
      int gt[kQTiles] = {0, 0};                 // key tiles each query tile has read
      int no[kQTiles] = {0, 0};                 // items in which each query tile read keys
      bool ok = true;
      auto slot_landed = [&](int gg) -> bool {
        if (!mbar_wait(&slot_full[gg % S], (gg / S) & 1)) return false;
        tc_fence_after();
        return true;
      };
      // S of query tile t from the K tile in slot gg, into its score columns
      auto issue_s = [&](int t, int gg) {
        const uint64_t dq = dq0 + (t * Lay::kQBytes >> 4);
        const uint64_t dk = dk0 + ((gg % S) * Lay::kSlotBytes >> 4);
        const uint32_t d = tbase + 256 * t;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          // 64-element column block ks / 4, 32 bytes per k-step inside it
          const uint32_t qo = ((ks >> 2) * kRows * 128 + (ks & 3) * 32) >> 4;
          const uint32_t ko = ((ks >> 2) * Lay::kLineBytes + (ks & 3) * 32) >> 4;
          tc_mma_f16(d, dq + qo, dk + ko, kIdescS, ks > 0 ? 1u : 0u);
        }
        tc_commit(&tbars[4 * t]);                           // s_full
      };
      // O of query tile t (+)= P V with the V tile in slot gg; P (16-bit, two
      // per column) is in the first 64 score columns, 8 columns per k-step;
      // an item's first P V overwrites O
      auto issue_pv = [&](int t, int gg, bool first) {
        // V as B, MN-major: 16 keys are two 8-row groups; the next 64 columns
        // of D are one line block (kLineBytes) on
        const uint64_t dv = dv0 + ((gg % S) * Lay::kSlotBytes >> 4);
        const uint32_t a = tbase + 256 * t;
        const uint32_t d = a + 128;
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          tc_mma_f16_ts(d, a + kk * 8, dv + ((kk * 16 * 128) >> 4), kIdescO,
                        (!first || kk > 0) ? 1u : 0u);
        if constexpr (kBF16) {                              // + (p - hi) V
#pragma unroll
          for (int kk = 0; kk < kKeys / 16; ++kk)
            tc_mma_f16_ts(d, a + kKeys / 2 + kk * 8, dv + ((kk * 16 * 128) >> 4), kIdescO, 1u);
        }
        tc_commit(&tbars[4 * t + 2]);                       // pv_done
      };
      for (int k = 0; ok; ++k) {
        const int slot = k & 1;
        if (!mbar_wait(&item_full[slot], (k >> 1) & 1)) {
          ok = false;
          break;
        }
        const Item it = items[slot];
        mbar_arrive(&item_empty[slot]);
        if (it.seq < 0) break;
        const Shape sh = item_shape(it, G);
        if (!mbar_wait(q_full, k & 1)) {                  // this item's query rows
          ok = false;
          break;
        }
        tc_fence_after();
        // S of the first key tile: it follows the previous item's last P V
        // of each query tile (which read P there), and that P V's softmax
        // threads are done with the scores
        if (!slot_landed(g)) {
          ok = false;
          break;
        }
        for (int t = 0; t < kQTiles; ++t)
          if (sh.nt[t] > 0) issue_s(t, g);
        tc_commit(&slot_empty[g % S]);                     // K tile 0 read
        if (sh.n_tiles == 1) tc_commit(q_free);            // the item's S products are issued
        for (int j = 0; ok && j < sh.n_tiles; ++j) {
          const int gk = g + 2 * j;                        // K of tile j; its V in gk + 1
          if (!slot_landed(gk + 1)) {
            ok = false;
            break;
          }
          bool k_next = false;
          for (int t = 0; ok && t < kQTiles; ++t) {
            if (j >= sh.nt[t]) continue;
            const int gi = gt[t] + j;
            if (!mbar_wait(&tbars[4 * t + 1], gi & 1)) {   // p_full: P of tile j written
              ok = false;
              break;
            }
            // the item's first P V overwrites O: the softmax threads have read
            // back the last item in which this query tile read keys
            if (j == 0 && no[t] >= 1 && !mbar_wait(&tbars[4 * t + 3], (no[t] - 1) & 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_pv(t, gk + 1, j == 0);
            if (j + 1 < sh.nt[t]) {
              // the next S overwrites the P this P V reads; products issued
              // by one thread run in issue order, so it follows at once
              if (!k_next && !slot_landed(gk + 2)) {
                ok = false;
                break;
              }
              k_next = true;
              tc_fence_after();
              issue_s(t, gk + 2);
            }
          }
          if (!ok) break;
          tc_commit(&slot_empty[(gk + 1) % S]);            // V tile j read
          if (k_next) {
            tc_commit(&slot_empty[(gk + 2) % S]);          // K tile j + 1 read
            if (j + 2 == sh.n_tiles) tc_commit(q_free);    // the item's S products are issued
          }
        }
        g += 2 * sh.n_tiles;
        for (int t = 0; t < kQTiles; ++t) {
          gt[t] += sh.nt[t];
          no[t] += sh.nt[t] > 0 ? 1 : 0;
        }
      }
      if (!ok) flag_error(p.err, PKV_DEVERR_TIMEOUT);
      // everything issued has completed before the columns are freed
      tc_commit(drain);
      if (!mbar_wait(drain, 0)) flag_error(p.err, PKV_DEVERR_TIMEOUT);
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------- query rows
    // One thread copies each item's 256 query rows into the A layout of S by
    // TMA (four boxes at d = 128: two query tiles x two 64-element lines) as
    // soon as the previous item's S products are done, while the softmax
    // threads still finish that item. Rows past the chunk read the next
    // tokens' queries (or zeros past the last token): they are masked out.
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      const uint64_t policy = l2_evict_first_policy();
      const int tok_per_qt = kRows / G;
      bool ok = true;
      int issued = 0;                                       // items whose query rows were loaded
      for (int k = 0; ok; ++k) {
        const int slot = k & 1;
        if (!mbar_wait(&item_full[slot], (k >> 1) & 1)) {
          ok = false;
          break;
        }
        const Item it = items[slot];
        mbar_arrive(&item_empty[slot]);
        if (it.seq < 0) break;
        if (k >= 1 && !mbar_wait(q_free, (k - 1) & 1)) {
          ok = false;
          break;
        }
        ++issued;
        mbar_arrive_expect_tx(q_full, kQTiles * Lay::kQBytes);
#pragma unroll
        for (int t = 0; t < kQTiles; ++t)
#pragma unroll
          for (int h = 0; h < NH; ++h)
            tma_load_4d(qtiles + t * Lay::kQBytes + h * kRows * 128, &tm_q, q_full, 0, h, it.kvh * G,
                        it.qs + it.qb * kQTiles * tok_per_qt + t * tok_per_qt, policy);
      }
      if (!ok) {
        flag_error(p.err, PKV_DEVERR_TIMEOUT);
        // let the last copy in flight land before the CTA leaves
        if (issued > 0) mbar_wait(q_full, (issued - 1) & 1);
      }
    }
  } else if (warp >= kSoftmaxWarp0) {
    // ---------------------------------------------------------- softmax
    const int t = (warp - kSoftmaxWarp0) >> 2;             // query tile
    const int r = ((warp - kSoftmaxWarp0) & 3) * 32 + lane;   // row of the tile = TMEM lane
    const uint32_t tl = tbase + 256 * t + ((static_cast<uint32_t>(warp & 3) * 32) << 16);
    uint64_t* s_full = &tbars[4 * t];
    uint64_t* p_full = s_full + 1;
    uint64_t* pv_done = s_full + 2;
    uint64_t* o_free = s_full + 3;
    const int tok_per_qt = kRows / G;
    int gt = 0;                                            // key tiles this query tile read, over all items
    int gall = 0;                                          // slots of the CTA, over all items
    int ntail = 0;                                         // items whose last key tile was partial
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int slot = k & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&item_full[slot], (k >> 1) & 1))) {
        ok = false;
        break;
      }
      const Item it = items[slot];
      mbar_arrive(&item_empty[slot]);
      if (it.seq < 0) break;
      const Shape sh = item_shape(it, G);
      const int n_my = sh.nt[t];
      const int tok = it.qb * kQTiles * tok_per_qt + t * tok_per_qt + r / G;
      const int head = it.kvh * G + r % G;
      const bool live = tok < it.C;
      const int pos = it.L - it.C + tok;
      const bool partial_end = sh.kv_end % kKeys != 0;     // the item's last key tile is partial
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < n_my; ++j) {
        const int gi = gt + j;
        // tcgen05.ld/st are warp-collective: every wait result is made warp-uniform
        if (!__all_sync(0xffffffffu, mbar_wait(s_full, gi & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        // the row's 128 scores in one load; the causal mask (also hides keys
        // past the context and rows past the chunk) only on tiles that cross
        // the row's causal edge; the row maximum is taken on unscaled scores
        // (the scale is positive)
        const int key0 = j * kKeys;
        uint32_t sc[kKeys];
        tmem_ld128(tl, sc);
        if (!(live && key0 + kKeys - 1 <= pos)) {
#pragma unroll
          for (int i = 0; i < kKeys; ++i)
            if (!(live && key0 + i <= pos)) sc[i] = __float_as_uint(-INFINITY);
        }
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int i = 0; i < kKeys; ++i) mx[i & 3] = fmaxf(mx[i & 3], __uint_as_float(sc[i]));
        const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * p.q_scale;
        const bool need = mt > m + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {                 // the whole warp takes this branch
          const float mn = need ? mt : m;
          if (j > 0) {
            // the output rows hold earlier tiles: rescale them once their P V is
            // done (factor 1 on rows that keep their max or hold nothing yet)
            if (!__all_sync(0xffffffffu, mbar_wait(pv_done, (gi - 1) & 1))) {
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
        // on a live row from its first tile on; a row past the chunk has only
        // -inf scores and nm = 0, so it writes 0 without a select); P goes
        // over the scores as 16-bit pairs in one store; bf16 P also keeps its
        // rounding error (p - hi) in the next 64 columns, read by a second
        // P V. This loop is bound by instruction issue, so the scale, the
        // shift and the row sum run as packed f32x2 pairs.
        const float nm = live ? -m : 0.f;
        const f32x2 sc2 = pack2(p.q_scale, p.q_scale), nm2 = pack2(nm, nm);
        f32x2 ls2[2] = {pack2(0.f, 0.f), pack2(0.f, 0.f)};
        uint32_t pk[kKeys / 2];
#pragma unroll
        for (int i = 0; i < kKeys; i += 2) {
          float x0, x1;
          unpack2(fma2(pack2_bits(sc[i], sc[i + 1]), sc2, nm2), x0, x1);
          const float e0 = ex2(x0);
          const float e1 = ex2(x1);
          ls2[(i >> 1) & 1] = add2(ls2[(i >> 1) & 1], pack2(e0, e1));
          pk[i >> 1] = T::pack(e0, e1);
          if constexpr (kBF16) {
            const float2 h = T::to_float2(pk[i >> 1]);
            sc[i >> 1] = T::pack(e0 - h.x, e1 - h.y);        // sc[0 .. i] are no longer needed
          }
        }
        tmem_st64(tl, pk);
        if constexpr (kBF16) {
          uint32_t pl[kKeys / 2];
#pragma unroll
          for (int i = 0; i < kKeys / 2; ++i) pl[i] = sc[i];
          tmem_st64(tl + kKeys / 2, pl);
        }
        float l0, l1;
        unpack2(add2(ls2[0], ls2[1]), l0, l1);
        l += l0 + l1;
        if (j == sh.n_tiles - 1 && partial_end) {
          if (t == sh.zt) {
            // V rows past the last key may hold anything (0 x NaN is NaN): zero
            // them, once the tile's V copies have landed
            const int gv = gall + 2 * j + 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&slot_full[gv % S], (gv / S) & 1))) {
              ok = false;
              break;
            }
            uint8_t* vt = slots + (gv % S) * Lay::kSlotBytes;
            const int valid = sh.kv_end - key0;
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
          } else if (!__all_sync(0xffffffffu, mbar_wait(tail, ntail & 1))) {   // a lower query tile zeroes them
            ok = false;
            break;
          }
        }
        tc_fence_before();
        mbar_arrive(p_full);
      }
      if (!ok) break;
      gt += n_my;
      if (n_my > 0) {
        if (!__all_sync(0xffffffffu, mbar_wait(pv_done, (gt - 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        float o[D];
        {
          uint32_t raw[D];
          if constexpr (D == 128) tmem_ld128(tl + 128, raw);
          else tmem_ld64(tl + 128, raw);
#pragma unroll
          for (int i = 0; i < D; ++i) o[i] = __uint_as_float(raw[i]);
        }
        tc_fence_before();
        mbar_arrive(o_free);                                 // the output columns may be reused
        if (live) {
          const float inv = 1.f / l;
#pragma unroll
          for (int i = 0; i < D; ++i) o[i] *= inv;
          store_row<T>(p.out, p.out_dtype,
                       (static_cast<int64_t>(it.qs + tok) * p.num_heads + head) * D, o, D);
        }
      }
      gall += 2 * sh.n_tiles;
      if (partial_end) ++ntail;
    }
    if (!ok) flag_error(p.err, PKV_DEVERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

template <int D, typename T>
static cudaError_t launch(const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq,
                          const Params& p, cudaStream_t s) {
  auto kern = prefill_kernel<D, T>;
  // one CTA per SM: it holds all 512 tensor-memory columns, so shared memory is
  // requested past half an SM even where the layout needs less (d = 64)
  constexpr int kSmemLaunch = Layout<D>::kSmem > 120 * 1024 ? Layout<D>::kSmem : 120 * 1024;
  const cudaError_t attr =
      prepare_kernel(reinterpret_cast<const void*>(kern), kThreads, kSmemLaunch, nullptr);
  if (attr != cudaSuccess) return attr;
  int sms = 0;
  cudaError_t e = device_sm_count(&sms);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(p.counter, 0, sizeof(int), s);
  if (e != cudaSuccess) return e;
  const int grid = std::min(p.total_items, sms);           // persistent: one CTA per SM at most
  kern<<<grid, kThreads, kSmemLaunch, s>>>(tk, tv, tq, p);
  return cudaGetLastError();
}

}  // namespace prefill
}  // namespace pkv

using namespace pkv;

extern "C" size_t pkv_prefill_workspace_size(void) { return 16; }

extern "C" pkv_status pkv_paged_attention_prefill(
    void* out, int out_dtype, const void* q, const void* k_cache, const void* v_cache,
    int kv_dtype, const int32_t* block_tables, const int32_t* context_lens,
    const int32_t* query_start, int num_seqs, int num_heads, int num_kv_heads, int head_size,
    int num_blocks, int block_size, int max_blocks_per_seq, int max_query_len, int total_queries,
    float scale, void* workspace, size_t workspace_bytes, int32_t* err_flag, void* stream) {
  if (num_seqs < 0 || num_seqs > 65535) return PKV_EINVAL;
  if (num_seqs == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start)
    return PKV_EINVAL;
  if (!workspace || workspace_bytes < pkv_prefill_workspace_size() || !aligned16(workspace))
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
  if (num_blocks < 1 || max_blocks_per_seq < 1 || max_query_len < 1 || total_queries < 0)
    return PKV_EINVAL;
  if (static_cast<int64_t>(num_blocks) * block_size > INT32_MAX) return PKV_EINVAL;
  if (static_cast<int64_t>(max_blocks_per_seq) * block_size > INT32_MAX / 2) return PKV_EINVAL;
  // work items: 256-row query blocks x sequences x KV heads, counted in an int
  const int64_t qblocks = (static_cast<int64_t>(max_query_len) * group + prefill::kQTiles * prefill::kRows - 1) /
                          (prefill::kQTiles * prefill::kRows);
  const int64_t items = qblocks * num_seqs * num_kv_heads;
  if (items > INT32_MAX / 2) return PKV_EINVAL;
  if (!std::isfinite(scale) || !(scale > 0.f)) return PKV_EINVAL;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_EINVAL;

  const int box_rows = std::min(block_size, 64);
  if (total_queries == 0) return PKV_OK;                  // no chunk has a row
  CUtensorMap tk, tv, tq;
  const int64_t slots = static_cast<int64_t>(num_blocks) * block_size;
  if (!encode_cache_map(&tk, k_cache, head_size, num_kv_heads, slots, box_rows, kLineSwizzled) ||
      !encode_cache_map(&tv, v_cache, head_size, num_kv_heads, slots, box_rows, kLineSwizzled) ||
      !encode_token_query_map(&tq, q, head_size, num_heads, total_queries, group))
    return PKV_ECUDA;
  prefill::Params p{};
  p.out = out;
  p.out_dtype = out_dtype;
  p.q = static_cast<const uint16_t*>(q);
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.query_start = query_start;
  p.err = err_flag;
  p.counter = static_cast<int*>(workspace);
  p.num_seqs = num_seqs;
  p.num_heads = num_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = group;
  p.num_blocks = num_blocks;
  p.block_size = block_size;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.max_query_len = max_query_len;
  p.total_queries = total_queries;
  p.qblocks = static_cast<int>(qblocks);
  p.total_items = static_cast<int>(items);
  p.box_rows = box_rows;
  p.q_scale = scale * prefill::kLog2e;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (head_size == 128)
    e = kv_dtype == PKV_F16 ? prefill::launch<128, F16>(tk, tv, tq, p, s)
                            : prefill::launch<128, BF16>(tk, tv, tq, p, s);
  else
    e = kv_dtype == PKV_F16 ? prefill::launch<64, F16>(tk, tv, tq, p, s)
                            : prefill::launch<64, BF16>(tk, tv, tq, p, s);
  return e == cudaSuccess ? PKV_OK : PKV_ECUDA;
}
