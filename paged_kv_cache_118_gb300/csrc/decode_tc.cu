// Paged decode attention for large query groups on the 5th-generation tensor
// cores (tcgen05), accumulators in tensor memory.
//
// What is computed is the decode call's partition partial ("079｜vLLM 与
// PagedAttention" §2 and the split-context form of [R] §3): for sequence s,
// KV head h and a context partition [t0, t1) of its L tokens, every query head
// g of h's group gets m = max_u scale q_g.k_u (base-2 units), l = sum_u
// 2^(scale q_g.k_u - m) and acc = sum_u 2^(scale q_g.k_u - m) v_u, which the
// decode reduce kernel merges with one global denominator.
//
// Why a second path: the warp-level tensor path serves at most 8 query heads
// per KV head in a CTA, so a group of G > 8 heads reads each K/V byte G/8
// times. Here the G heads (32, 64 or 128 of them) are the rows of one 128-row
// product, and each K/V byte is read once.
//
// How (persistent CTAs, one per SM, 256 threads):
//  * all warps first build the call's work list: up to 1024 sequences, only
//    units (sequence, partition, KV head) that exist are numbered, every whole
//    partition first, then the partial last ones largest first, so that the
//    run ends with its shortest units; larger batches number them all and skip
//    the empty ones. Warp 0 then takes units: its CTA's index first, then
//    claims from a global counter. Per unit it reads the partition's block ids (one per lane),
//    loads the G query rows by TMA into a staging buffer and streams
//    the partition's 64-key K tiles into a ring of 4 to 6 stages (as many
//    as shared memory holds beside the rest), while warp 2 follows the same
//    units and streams their V tiles into the same stages: one TMA copy per
//    physical block and 128-byte line, each warp's lanes issuing a tile's
//    copies at once (one warp issuing all of them was the stream's limit
//    below 16-row blocks);
//  * one thread of warp 1 owns the 512 tensor-memory columns (two 64-column
//    score buffers, two D-column output buffers and two query buffers, one of
//    each per unit in flight), copies each unit's query rows from the staging
//    buffer into tensor memory (tcgen05.cp) and issues S = Q K^T (M = 128,
//    N = 64, K = D; Q from tensor memory) and O += P V (P from tensor memory),
//    committing each to an mbarrier; a tile's S is issued before the
//    previous tile's P V, and the next unit's first S as soon as its queries
//    are in;
//  * warps 4-7 run the softmax, one thread per query row (its TMEM lane). The
//    query rows hold 128 / G copies of the group's G heads, and copy c of a
//    head takes keys [c 64 G / 128, (c + 1) 64 G / 128) of every tile (its P
//    is 0 elsewhere), so every thread works on 64 G / 128 keys per tile. At
//    the end of a unit the copies of a head are merged through shared memory
//    (two copies exchange halves of D and each writes one; with four, copy 0
//    takes the others' rows half of D at a time) and the partials written,
//    while the next unit runs in the other output buffer.
// Every wait is bounded; bad block ids and lengths are reported and skipped.

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>
#include <type_traits>

#include "pagedkv.h"
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {
namespace tcdec {

constexpr int kRows = 128;             // product rows: 128 / G copies of the group's query heads
constexpr int kKeys = 64;              // keys per tile
constexpr int kMaxStages = 6;
constexpr int kSmemLimit = 232448;     // shared memory one CTA may ask for
constexpr int kThreads = 256;          // warp 0: claims, K copies; 1: MMA; 2: V copies; 4-7: softmax
constexpr int kSoftmaxWarp0 = 4;
constexpr int kMaxIds = 256;           // block ids of one unit, read ahead of its copies
constexpr int kCompactMaxSeqs = 1024;  // batches up to this size get a compact work list
// S0 [0, 64), S1 [64, 128), O0 [128, 128 + D), O1 [256, 256 + D),
// Q0 [384, 384 + D/2), Q1 [448, 448 + D/2) (16-bit pairs)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kQCol = 384;
constexpr float kRescaleThreshold = 8.0f;

struct Params {
  float* part_acc;                     // [rows][D], rows = num_seqs * num_heads * max_parts
  float2* part_ml;                     // [rows] = (m in base-2 units, l)
  int* counter;
  const int32_t* block_tables;
  const int32_t* context_lens;
  int32_t* err;
  int num_seqs, num_heads, num_kv_heads, group;
  int num_blocks, block_size, max_blocks_per_seq;
  int partition_tokens, max_parts, total_units, box_rows;
  float q_scale;
  uint64_t wait_ns;                    // limit of every pipeline wait
  int stall_unit;                      // test hook: the softmax warps wait out this unit; -1: none
};

struct UnitInfo {
  int seq;                             // -1: no more units
  int kvh;
  int part;
  int len;
};

// Shared memory from a 1024-byte aligned base; operands are 128-byte rows with
// the 128-byte swizzle, 8-row groups 1024 bytes apart:
//  Q staging: D/64 column blocks of 128 rows, 128 / G copies of the G query
//  rows (K-major; copied to tensor memory at the start of the unit);
//  each stage: K then V, D/64 line blocks of 64 key rows (B of S, K-major; B
//  of P V, MN-major with the next 64 columns one line block on);
//  merge area (two or four copies): rows of D/2 + 1 floats (an odd stride, so
//  a warp writing its rows meets no bank conflict), then the rows' (m, l):
//  with two copies every row passes the half of D its partner writes; with
//  four the rows of copies 1-3 pass half of D per round to copy 0;
//  then the barriers, the unit slots and the work list (the Q staging buffer
//  serves as scratch while the list is built, before the first query copy).
// The ring takes as many stages (up to kMaxStages) as the rest leaves room for.
template <int D, int C>
struct Layout {
  static constexpr int NH = D / 64;
  static constexpr int kQBytes = kRows * D * 2;
  static constexpr int kLineBytes = kKeys * 128;
  static constexpr int kTileBytes = NH * kLineBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kOffStages = kQBytes;
  static constexpr int kHalf = D / 2;
  // two copies exchange halves (all 128 rows write one); four pass the
  // later copies' rows to the first
  static constexpr int kMergeRows = C == 2 ? kRows : kRows - kRows / C;
  static constexpr int kMergeStride = kHalf + 1;
  static constexpr int kMergeBytes = kMergeRows * (kMergeStride + 2) * 4;
  // barriers: stage_full[S], stage_empty[S], unit_full[2], unit_empty[2],
  // q_full, q_free, s_full[2], p_full[2], pv_done[2], o_free[2], drain,
  // mrg_full, mrg_free, never (one that nothing completes: the test hook's)
  static constexpr int kTailBytes = (2 * kMaxStages + 2 * 8 + 4) * 8 +
                                    2 * static_cast<int>(sizeof(UnitInfo)) + 2 * kMaxIds * 4 +
                                    (kCompactMaxSeqs + 4) * 4 + kCompactMaxSeqs * 2 +
                                    kCompactMaxSeqs * 4 + 16;
  static constexpr int kFit =
      (kSmemLimit - 1024 - kOffStages - kMergeBytes - kTailBytes - 16) / kStageBytes;
  static constexpr int kStages = kFit < kMaxStages ? kFit : kMaxStages;
  static constexpr int kOffMerge = kOffStages + kStages * kStageBytes;
  static constexpr int kOffBars = (kOffMerge + kMergeBytes + 15) / 16 * 16;
  static constexpr int kNumBars = 2 * kStages + 2 * 8 + 4;
  static constexpr int kOffUnits = kOffBars + kNumBars * 8;
  static constexpr int kOffIds = kOffUnits + 2 * static_cast<int>(sizeof(UnitInfo));
  static constexpr int kOffPref = kOffIds + 2 * kMaxIds * 4;  // whole partitions per sequence
  static constexpr int kOffOrder = kOffPref + (kCompactMaxSeqs + 4) * 4;  // partial ones, largest first
  static constexpr int kOffLens = kOffOrder + kCompactMaxSeqs * 2;
  static constexpr int kOffTmem = kOffLens + kCompactMaxSeqs * 4;
  static constexpr int kSmem = 1024 + kOffTmem + 16;
  static_assert(kStages >= 3 && kSmem <= kSmemLimit, "shared memory of one CTA");
};

// Builds the compact work list with all the CTA's threads (every CTA builds
// the same list: claims index into it, so no step may depend on the order of
// concurrent events): per sequence its length, the prefix of whole
// partitions, and the sequences with a partial last partition in a stable
// counting sort by tile count, largest first. `scratch` is the Q staging
// buffer, before any query copy reaches it; a proxy fence hands it back.
// Ends with a block-wide barrier.
__device__ __forceinline__ void build_list(const Params& p, int max_ctx, int* scratch, int* pref,
                                           uint16_t* porder, int* lens, int& whole_units,
                                           int& partial_units) {
  constexpr int kWarps = kThreads / 32;
  constexpr int kChunks = kCompactMaxSeqs / 32;
  constexpr int kChunksPerWarp = (kChunks + kWarps - 1) / kWarps;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = p.num_seqs;
  const int nchunks = (n + 31) / 32;
  const int PT = p.partition_tokens;
  const int nbk = PT / kKeys;                          // tile counts 1 .. nbk <= 64
  int* chunk_sum = scratch;                            // [32]
  int* totals = scratch + 32;                          // [2]
  int* base = scratch + 40;                            // [nbk + 1]
  int* cnt = base + (nbk + 1);                         // [(nbk + 1) * 32]
  uint8_t* tiles_of = reinterpret_cast<uint8_t*>(cnt + (nbk + 1) * kChunks);
  uint8_t* rank_of = tiles_of + kCompactMaxSeqs;
  for (int i = tid; i < (nbk + 1) * kChunks; i += kThreads) cnt[i] = 0;
  int Ls[kChunksPerWarp];
#pragma unroll
  for (int j = 0; j < kChunksPerWarp; ++j) {          // every load of this warp in flight at once
    const int s = (warp + j * kWarps) * 32 + lane;
    Ls[j] = s < n ? __ldg(p.context_lens + s) : 0;
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kChunksPerWarp; ++j) {
    const int ch = warp + j * kWarps;
    if (ch >= nchunks) break;
    const int s = ch * 32 + lane;
    const int L = Ls[j];
    const bool valid = s < n && L >= 1 && L <= max_ctx;
    if (s < n && !valid && blockIdx.x == 0) flag_error(p.err, PKV_DEVERR_CONTEXT);
    int x = valid ? L / PT : 0;                        // whole partitions
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (s < n) {
      pref[s + 1] = x;
      lens[s] = L;
    }
    if (lane == 31) chunk_sum[ch] = x;
    const int r = valid ? L % PT : 0;
    const int t = (r + kKeys - 1) / kKeys;
    const unsigned same = __match_any_sync(0xffffffffu, t);
    if (s < n) {
      tiles_of[s] = static_cast<uint8_t>(t);
      rank_of[s] = static_cast<uint8_t>(__popc(same & ((1u << lane) - 1u)));
    }
    if (t > 0 && lane == __ffs(same) - 1) cnt[t * kChunks + ch] = __popc(same);
  }
  __syncthreads();
  if (warp == 0) {                                     // chunk offsets of the whole partitions
    const int v = lane < nchunks ? chunk_sum[lane] : 0;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane < nchunks) chunk_sum[lane] = x - v;
    if (lane == 31) totals[0] = x;
  }
  for (int b = 1 + tid; b <= nbk; b += kThreads) {    // places within each tile count
    int acc = 0;
    for (int ch = 0; ch < nchunks; ++ch) {
      const int v = cnt[b * kChunks + ch];
      cnt[b * kChunks + ch] = acc;
      acc += v;
    }
    base[b] = acc;
  }
  __syncthreads();
  if (warp == 0) {                                     // first place of each count, largest first
    int carry = 0;
    for (int top = nbk; top >= 1; top -= 32) {
      const int b = top - lane;
      const int v = b >= 1 ? base[b] : 0;
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      __syncwarp();
      if (b >= 1) base[b] = carry + x - v;
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) totals[1] = carry;
  }
  __syncthreads();
  for (int s = tid; s < n; s += kThreads) {
    pref[s + 1] += chunk_sum[s >> 5];
    const int t = tiles_of[s];
    if (t > 0) porder[base[t] + cnt[t * kChunks + (s >> 5)] + rank_of[s]] = static_cast<uint16_t>(s);
  }
  if (tid == 0) pref[0] = 0;
  whole_units = totals[0];
  partial_units = totals[1];
  fence_proxy_async_smem();
  __syncthreads();
}

// C: copies of the G = 128 / C query rows in the product's rows.
template <int D, typename T, int C>
__global__ void __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_q, const Params p) {
  using Lay = Layout<D, C>;
  constexpr int kStages = Lay::kStages;
  constexpr int NH = Lay::NH;
  constexpr bool kBF16 = std::is_same<T, BF16>::value;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* qstage = smem;
  uint8_t* stages = smem + Lay::kOffStages;
  uint64_t* stage_full = reinterpret_cast<uint64_t*>(smem + Lay::kOffBars);
  uint64_t* stage_empty = stage_full + kStages;
  uint64_t* unit_full = stage_empty + kStages;
  uint64_t* unit_empty = unit_full + 2;
  uint64_t* q_full = unit_empty + 2;                     // the staging buffer
  uint64_t* q_free = q_full + 1;
  uint64_t* s_full = q_free + 1;
  uint64_t* p_full = s_full + 2;
  uint64_t* pv_done = p_full + 2;
  uint64_t* o_free = pv_done + 2;
  uint64_t* drain = o_free + 2;
  uint64_t* mrg_full = drain + 1;
  uint64_t* mrg_free = mrg_full + 1;
  uint64_t* never = mrg_free + 1;
  float* merge = reinterpret_cast<float*>(smem + Lay::kOffMerge);
  float2* mrg_ml = reinterpret_cast<float2*>(merge + Lay::kMergeRows * Lay::kMergeStride);
  UnitInfo* units = reinterpret_cast<UnitInfo*>(smem + Lay::kOffUnits);
  int32_t* ids = reinterpret_cast<int32_t*>(smem + Lay::kOffIds);
  int32_t* pref = reinterpret_cast<int32_t*>(smem + Lay::kOffPref);
  uint16_t* porder = reinterpret_cast<uint16_t*>(smem + Lay::kOffOrder);
  int32_t* lens = reinterpret_cast<int32_t*>(smem + Lay::kOffLens);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kOffTmem);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int B = p.block_size;
  const int PT = p.partition_tokens;
  const int G = p.group;
  const int max_ctx = p.max_blocks_per_seq * B;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&stage_full[i], 2);                 // the K and the V copy warps
      mbar_init(&stage_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&unit_full[i], 1);
      mbar_init(&unit_empty[i], kRows + 2);          // softmax threads, MMA thread, V copy warp
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], kRows);
      mbar_init(&pv_done[i], 1);
      mbar_init(&o_free[i], kRows);
    }
    mbar_init(q_full, 1);
    mbar_init(q_free, 1);
    mbar_init(drain, 1);
    // two copies: every row; four: the copies past the first, then the first
    mbar_init(mrg_full, C == 2 ? kRows : (C > 1 ? kRows - kRows / C : 1));
    mbar_init(mrg_free, C == 2 ? kRows : kRows / C);
    mbar_init(never, 1);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const bool compact = p.num_seqs <= kCompactMaxSeqs;
  int whole_units = 0, partial_units = 0;
  if (compact)
    build_list(p, max_ctx, reinterpret_cast<int*>(qstage), pref, porder, lens, whole_units,
               partial_units);

  if (warp == 0 || warp == 2) {
    // ---------------------------------------------------------- claims, copies
    // Warp 0 takes the units (claims, block ids, query rows) and copies each
    // tile's K; warp 2 follows the published units and copies the tiles' V.
    // Each lane issues one copy (one physical block, one 128-byte line), and
    // each warp's lane 0 arrives on the stage with the bytes of its own copies.
    const bool leader = warp == 0;
    if (lane == 0) {
      prefetch_tmap(leader ? &tm_k : &tm_v);
      if (leader) prefetch_tmap(&tm_q);
    }
    const uint64_t policy = l2_evict_first_policy();
    const int R = p.box_rows;
    const uint32_t copy_bytes = static_cast<uint32_t>(R) * 128;
    const int Hkv = p.num_kv_heads;
    const int total = compact ? (whole_units + partial_units) * Hkv : p.total_units;
    // lane l copies line l % NH of the tile's copy l / NH
    const int my_c = lane / NH;
    const int my_h = lane % NH;
    const CUtensorMap* my_map = leader ? &tm_k : &tm_v;
    const uint32_t my_off =
        (leader ? 0u : static_cast<uint32_t>(Lay::kTileBytes)) + my_h * Lay::kLineBytes +
        my_c * copy_bytes;
    int g = 0;                                             // tiles issued
    int k = 0;                                             // units published / followed
    int last_issued[kStages];
#pragma unroll
    for (int i = 0; i < kStages; ++i) last_issued[i] = -1;
    bool ok = true;
    for (int claim = 0; ok; ++claim) {
      const int slot = k & 1;
      int32_t* uids = ids + slot * kMaxIds;                // this unit's block ids
      UnitInfo info{-1, 0, 0, 0};
      int t_begin = 0, t_end = 0;
      if (leader) {
        // the CTA's own index first (no round trip), then the shared counter
        int u = blockIdx.x;
        if (claim > 0) {
          if (lane == 0) u = static_cast<int>(gridDim.x) + atomicAdd(p.counter, 1);
          u = __shfl_sync(0xffffffffu, u, 0);
        }
        if (u < total) {
          int seq, kvh, part, L;
          if (compact) {
            const int w = u / Hkv;
            kvh = u - w * Hkv;
            if (w >= whole_units) {                        // a partial last partition
              seq = porder[w - whole_units];
              L = lens[seq];
              part = L / PT;
            } else {
              int lo = 0, hi = p.num_seqs;                 // largest lo with pref[lo] <= w
              while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (pref[mid] <= w) lo = mid; else hi = mid;
              }
              seq = lo;
              L = lens[lo];
              part = w - pref[lo];
            }
          } else {
            const int per_part = p.num_seqs * Hkv;
            part = u / per_part;
            const int rem = u - part * per_part;
            seq = rem / Hkv;
            kvh = rem - seq * Hkv;
            L = __ldg(p.context_lens + seq);
            if (L < 1 || L > max_ctx) {
              if (lane == 0 && part == 0 && kvh == 0) flag_error(p.err, PKV_DEVERR_CONTEXT);
              continue;
            }
            if (part * PT >= L) continue;                  // this sequence has no such partition
          }
          t_begin = part * PT;
          t_end = min(L, t_begin + PT);
          info = UnitInfo{seq, kvh, part, L};
        }
        // the slot's unit two back has been read by all its consumers, and its
        // block ids by warp 2 (its last arrival)
        bool w_ok = true;
        if (lane == 0 && k >= 2) w_ok = mbar_wait(&unit_empty[slot], ((k >> 1) & 1) ^ 1, p.wait_ns);
        if (!__shfl_sync(0xffffffffu, w_ok, 0)) {
          ok = false;
          break;
        }
        if (info.seq >= 0) {
          const int b0 = t_begin / B;
          const int32_t* row =
              p.block_tables + static_cast<int64_t>(info.seq) * p.max_blocks_per_seq;
          const int nb = (t_end - 1) / B - b0 + 1;
          for (int i = lane; i < nb; i += 32) {
            int32_t id = __ldg(row + b0 + i);
            if (id < 0 || id >= p.num_blocks) {
              flag_error(p.err, PKV_DEVERR_BLOCK_ID);
              id = 0;
            }
            uids[i] = id;
          }
        }
        __threadfence_block();
        __syncwarp();
        // the staging buffer, once the previous unit's rows are in tensor memory
        if (lane == 0 && k >= 1 && info.seq >= 0) w_ok = mbar_wait(q_free, (k - 1) & 1, p.wait_ns);
        if (!__shfl_sync(0xffffffffu, w_ok, 0)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          units[slot] = info;
          if (info.seq >= 0) {
            // the group's query rows, once per copy
            mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(NH) * kRows * 128);
            const int row0 = info.seq * p.num_heads + info.kvh * G;
#pragma unroll
            for (int c = 0; c < C; ++c)
#pragma unroll
              for (int h = 0; h < NH; ++h)
                tma_load_3d(qstage + h * kRows * 128 + c * G * 128, &tm_q, q_full, 0, h, row0,
                            policy);
          }
          // the release orders the ids' stores before warp 2's reads
          mbar_arrive(&unit_full[slot]);
        }
      } else {
        if (!__all_sync(0xffffffffu, mbar_wait(&unit_full[slot], (k >> 1) & 1, p.wait_ns))) {
          ok = false;
          break;
        }
        info = units[slot];
        if (info.seq >= 0) {
          t_begin = info.part * PT;
          t_end = min(info.len, t_begin + PT);
        }
      }
      ++k;
      if (info.seq < 0) break;
      const int b0 = t_begin / B;
      const int n_tiles = (t_end - t_begin + kKeys - 1) / kKeys;
      for (int i = 0; i < n_tiles; ++i, ++g) {
        const int st = g % kStages;
        bool e_ok = true;
        if (lane == 0 && g >= kStages) e_ok = mbar_wait(&stage_empty[st], ((g / kStages) & 1) ^ 1, p.wait_ns);
        if (!__shfl_sync(0xffffffffu, e_ok, 0)) {
          ok = false;
          break;
        }
        const int t0 = t_begin + i * kKeys;
        const int copies = (min(kKeys, t_end - t0) + R - 1) / R;
        if (lane == 0) {
          mbar_arrive_expect_tx(&stage_full[st], static_cast<uint32_t>(NH) * copies * copy_bytes);
          last_issued[st] = g;
        }
        __syncwarp();
        if (my_c < copies) {
          const int tk = t0 + my_c * R;
          const int z = uids[tk / B - b0] * B + tk % B;
          tma_load_4d(stages + st * Lay::kStageBytes + my_off, my_map, &stage_full[st], 0, z,
                      info.kvh, my_h, policy);
        }
      }
      __syncwarp();
      // warp 2 is done with the unit's block ids
      if (ok && !leader && lane == 0) mbar_arrive(&unit_empty[slot]);
    }
    if (!ok && lane == 0) {
      flag_error(p.err, PKV_DEVERR_TIMEOUT);
      for (int st = 0; st < kStages; ++st)
        if (last_issued[st] >= 0) mbar_wait(&stage_full[st], (last_issued[st] / kStages) & 1, p.wait_ns);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t kIdescS = mma_idesc_f16(kBF16, kRows, kKeys, false);
      constexpr uint32_t kIdescO = mma_idesc_f16(kBF16, kRows, D, true);
      const uint64_t dq0 = smem_desc_sw128(qstage, 16, 1024);   // the staging buffer
      const uint64_t dk0 = smem_desc_sw128(stages, 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(stages + Lay::kTileBytes, Lay::kLineBytes, 1024);
      int g = 0;                                           // tiles consumed
      bool ok = true;
      // S of global tile gi (its stage, score buffer gi % 2) from query buffer qb
      auto issue_s = [&](int gi, int qb) -> bool {
        const int st = gi % kStages, b = gi & 1;
        if (!mbar_wait(&stage_full[st], (gi / kStages) & 1, p.wait_ns)) return false;
        // the score buffer's P was read by the P V product two tiles back
        if (gi >= 2 && !mbar_wait(&pv_done[b], ((gi - 2) >> 1) & 1, p.wait_ns)) return false;
        tc_fence_after();
        const uint32_t qt = tbase + kQCol + qb * (D / 2);
        const uint64_t dk = dk0 + ((st * Lay::kStageBytes) >> 4);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t ko = ((ks >> 2) * Lay::kLineBytes + (ks & 3) * 32) >> 4;
          tc_mma_f16_ts(tbase + b * kKeys, qt + ks * 8, dk + ko, kIdescS, ks > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[b]);
        return true;
      };
      // O of output buffer ob (+)= P V of global tile gi
      auto issue_pv = [&](int gi, int ob, bool first) -> bool {
        const int st = gi % kStages, b = gi & 1;
        if (!mbar_wait(&p_full[b], (gi >> 1) & 1, p.wait_ns)) return false;
        tc_fence_after();
        const uint64_t dv = dv0 + ((st * Lay::kStageBytes) >> 4);
        const uint32_t a = tbase + b * kKeys;
        const uint32_t d = tbase + 128 + ob * 128;
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          tc_mma_f16_ts(d, a + kk * 8, dv + ((kk * 16 * 128) >> 4), kIdescO,
                        (!first || kk > 0) ? 1u : 0u);
        if constexpr (kBF16) {                              // + (p - hi) V
#pragma unroll
          for (int kk = 0; kk < kKeys / 16; ++kk)
            tc_mma_f16_ts(d, a + kKeys / 2 + kk * 8, dv + ((kk * 16 * 128) >> 4), kIdescO, 1u);
        }
        tc_commit(&pv_done[b]);
        tc_commit(&stage_empty[st]);
        return true;
      };
      for (int k = 0; ok; ++k) {
        const int slot = k & 1;
        if (!mbar_wait(&unit_full[slot], (k >> 1) & 1, p.wait_ns)) {
          ok = false;
          break;
        }
        const UnitInfo info = units[slot];
        mbar_arrive(&unit_empty[slot]);
        if (info.seq < 0) break;
        const int t_begin = info.part * PT;
        const int n_tiles = (min(info.len, t_begin + PT) - t_begin + kKeys - 1) / kKeys;
        if (!mbar_wait(q_full, k & 1, p.wait_ns)) {
          ok = false;
          break;
        }
        // the output buffer was read out at the end of the unit two back
        if (k >= 2 && !mbar_wait(&o_free[slot], ((k >> 1) & 1) ^ 1, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // the query rows into this unit's query columns, one 16-element k-step
        // (128 rows x 32 bytes) per copy, in order with the products around
        // them (the unit two back read these columns before); the staging
        // buffer is free once the copies are done
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          tc_cp_128x256b(tbase + kQCol + slot * (D / 2) + ks * 8,
                         dq0 + (((ks >> 2) * kRows * 128 + (ks & 3) * 32) >> 4));
        tc_commit(q_free);
        ok = issue_s(g, slot);
        for (int i = 0; ok && i < n_tiles; ++i) {
          if (i + 1 < n_tiles) ok = issue_s(g + i + 1, slot);
          if (ok) ok = issue_pv(g + i, slot, i == 0);
        }
        g += n_tiles;
      }
      if (!ok) flag_error(p.err, PKV_DEVERR_TIMEOUT);
      tc_commit(drain);
      if (!mbar_wait(drain, 0, p.wait_ns)) flag_error(p.err, PKV_DEVERR_TIMEOUT);
    }
  } else if (warp >= kSoftmaxWarp0) {
    // ---------------------------------------------------------- softmax
    constexpr int KC = kKeys / C;                          // keys of a tile per copy
    const int r = (warp - kSoftmaxWarp0) * 32 + lane;     // row = TMEM lane
    const uint32_t tl = tbase + ((static_cast<uint32_t>(warp & 3) * 32) << 16);
    const int cp = r / G;                                  // copy (the same across a warp)
    const int hr = r - cp * G;                             // head of the group
    int g = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int slot = k & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&unit_full[slot], (k >> 1) & 1, p.wait_ns))) {
        ok = false;
        break;
      }
      const UnitInfo info = units[slot];
      mbar_arrive(&unit_empty[slot]);
      if (info.seq < 0) break;
      // test hook: wait on a barrier nothing completes, so that this wait (and
      // then the MMA thread's and the copy warp's) runs out
      if (k == p.stall_unit && !__all_sync(0xffffffffu, mbar_wait(never, 0, p.wait_ns))) {
        ok = false;
        break;
      }
      const int t_begin = info.part * PT;
      const int t_end = min(info.len, t_begin + PT);
      const int n_tiles = (t_end - t_begin + kKeys - 1) / kKeys;
      const uint32_t to = tl + 128 + slot * 128;          // this unit's output columns
      float m = -INFINITY, l = 0.f;
      for (int i = 0; i < n_tiles; ++i, ++g) {
        const int b = g & 1;
        // tcgen05.ld/st are warp-collective: every wait result is made warp-uniform
        if (!__all_sync(0xffffffffu, mbar_wait(&s_full[b], (g >> 1) & 1, p.wait_ns))) {
          ok = false;
          break;
        }
        tc_fence_after();
        // this copy's KC scores of the tile (its columns only)
        float s[KC];
        if constexpr (KC == 16) {
          uint32_t raw[16];
          tmem_ld16(tl + b * kKeys + cp * KC, raw);
#pragma unroll
          for (int e = 0; e < 16; ++e) s[e] = __uint_as_float(raw[e]);
        } else {
#pragma unroll
          for (int h = 0; h < KC / 32; ++h) {
            uint32_t raw[32];
            tmem_ld32(tl + b * kKeys + cp * KC + h * 32, raw);
#pragma unroll
            for (int e = 0; e < 32; ++e) s[h * 32 + e] = __uint_as_float(raw[e]);
          }
        }
        const int tile_valid = t_end - (t_begin + i * kKeys);   // keys of the tile that exist
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (tile_valid >= kKeys) {
#pragma unroll
          for (int e = 0; e < KC; ++e) mx[e & 3] = fmaxf(mx[e & 3], s[e]);
        } else {
#pragma unroll
          for (int e = 0; e < KC; ++e) {
            s[e] = cp * KC + e < tile_valid ? s[e] : -INFINITY;
            mx[e & 3] = fmaxf(mx[e & 3], s[e]);
          }
        }
        const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * p.q_scale;
        const bool need = mt > m + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {               // the whole warp takes this branch
          const float mn = need ? mt : m;
          if (i > 0) {
            // the output rows hold earlier tiles of the unit: rescale them
            // once their P V is done (factor 1 on rows that keep their max)
            if (!__all_sync(0xffffffffu, mbar_wait(&pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, p.wait_ns))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const float c = (need && m != -INFINITY) ? ex2(m - mn) : 1.f;
#pragma unroll
            for (int h = 0; h < D / 32; ++h) {
              uint32_t raw[32];
              tmem_ld32(to + h * 32, raw);
#pragma unroll
              for (int e = 0; e < 32; ++e) raw[e] = __float_as_uint(__uint_as_float(raw[e]) * c);
              tmem_st32(to + h * 32, raw);
            }
            l *= c;
          }
          m = mn;
        }
        // p = 2^(scale s - m) on this copy's keys, 0 on the others' (a slice
        // with no key yet keeps m = -inf and gives 0)
        const float nm = m == -INFINITY ? 0.f : -m;
        const f32x2 sc2 = pack2(p.q_scale, p.q_scale), nm2 = pack2(nm, nm), neg1 = pack2(-1.f, -1.f);
        f32x2 ls2[2] = {pack2(0.f, 0.f), pack2(0.f, 0.f)};
        uint32_t vh[KC / 2], vl[KC / 2];
#pragma unroll
        for (int e = 0; e < KC; e += 2) {
          float x0, x1;
          unpack2(fma2(pack2(s[e], s[e + 1]), sc2, nm2), x0, x1);
          const float e0 = ex2(x0);
          const float e1 = ex2(x1);
          const f32x2 ee = pack2(e0, e1);
          ls2[(e >> 1) & 1] = add2(ls2[(e >> 1) & 1], ee);
          vh[e >> 1] = T::pack(e0, e1);
          if constexpr (kBF16) {
            float d0, d1;
            unpack2(fma2(T::to_pair(vh[e >> 1]), neg1, ee), d0, d1);
            vl[e >> 1] = T::pack(d0, d1);
          }
        }
        {
          float l0, l1;
          unpack2(add2(ls2[0], ls2[1]), l0, l1);
          l += l0 + l1;
        }
        // P as 16-bit pairs over the first 32 columns of the scores; bf16 P also
        // keeps its rounding error (p - hi) in the next 32, read by a second P V
        if constexpr (C == 2) {
          // this copy's 16 columns, and zeros over the other copy's
          uint32_t zero[KC / 2];
#pragma unroll
          for (int e = 0; e < KC / 2; ++e) zero[e] = 0u;
          tmem_st16_issue(tl + b * kKeys + cp * (KC / 2), vh);
          tmem_st16_issue(tl + b * kKeys + (1 - cp) * (KC / 2), zero);
          if constexpr (kBF16) {
            tmem_st16_issue(tl + b * kKeys + kKeys / 2 + cp * (KC / 2), vl);
            tmem_st16_issue(tl + b * kKeys + kKeys / 2 + (1 - cp) * (KC / 2), zero);
          }
          tmem_wait_st();
        } else {
          uint32_t pk[kKeys / 2], pl[kKeys / 2];
#pragma unroll
          for (int cc = 0; cc < C; ++cc)
#pragma unroll
            for (int e = 0; e < KC / 2; ++e) {
              pk[cc * KC / 2 + e] = cp == cc ? vh[e] : 0u;
              if constexpr (kBF16) pl[cc * KC / 2 + e] = cp == cc ? vl[e] : 0u;
            }
          tmem_st32(tl + b * kKeys, pk);                    // over the scores of this tile
          if constexpr (kBF16) tmem_st32(tl + b * kKeys + kKeys / 2, pl);
        }
        if (tile_valid < kKeys) {
          // V rows past the last key may hold anything (0 x NaN is NaN): zero them
          uint8_t* vt = stages + (g % kStages) * Lay::kStageBytes + Lay::kTileBytes;
          for (int idx = r; idx < NH * kKeys; idx += kRows) {
            const int kr = idx % kKeys, h = idx / kKeys;
            if (kr >= tile_valid) {
              uint4* d = reinterpret_cast<uint4*>(vt + h * Lay::kLineBytes + kr * 128);
#pragma unroll
              for (int e = 0; e < 8; ++e) d[e] = make_uint4(0u, 0u, 0u, 0u);
            }
          }
          fence_proxy_async_smem();
        }
        tc_fence_before();
        mbar_arrive(&p_full[b]);
      }
      if (!ok) break;
      // the unit's partials, once its last P V is done
      if (!__all_sync(0xffffffffu, mbar_wait(&pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, p.wait_ns))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int64_t prow = (static_cast<int64_t>(info.seq) * p.num_heads + info.kvh * G + hr) *
                               p.max_parts + info.part;
      if constexpr (C == 1) {
        uint32_t raw[D];                                    // one tensor-memory round trip
        if constexpr (D == 128) tmem_ld128(to, raw);
        else tmem_ld64(to, raw);
        float4* dst = reinterpret_cast<float4*>(p.part_acc + prow * D);
#pragma unroll
        for (int e = 0; e < D / 4; ++e)
          dst[e] = make_float4(__uint_as_float(raw[4 * e]), __uint_as_float(raw[4 * e + 1]),
                               __uint_as_float(raw[4 * e + 2]), __uint_as_float(raw[4 * e + 3]));
        p.part_ml[prow] = make_float2(m, l);
      } else if constexpr (C == 2) {
        // Copy c merges and writes the half [c D/2, (c + 1) D/2) of the head's
        // row; it hands its other half, with its (m, l), to the other copy.
        if (k >= 1 && !__all_sync(0xffffffffu, mbar_wait(mrg_free, (k - 1) & 1, p.wait_ns))) {
          ok = false;
          break;
        }
        float* out_row = merge + (cp * G + hr) * Lay::kMergeStride;
        {
          uint32_t raw[Lay::kHalf];                        // one tensor-memory round trip
          if constexpr (Lay::kHalf == 64) tmem_ld64(to + (1 - cp) * Lay::kHalf, raw);
          else tmem_ld32(to + (1 - cp) * Lay::kHalf, raw);
#pragma unroll
          for (int e = 0; e < Lay::kHalf; ++e) out_row[e] = __uint_as_float(raw[e]);
        }
        mrg_ml[cp * G + hr] = make_float2(m, l);
        mbar_arrive(mrg_full);
        if (!__all_sync(0xffffffffu, mbar_wait(mrg_full, k & 1, p.wait_ns))) {
          ok = false;
          break;
        }
        const float* in_row = merge + ((1 - cp) * G + hr) * Lay::kMergeStride;
        const float2 mo = mrg_ml[(1 - cp) * G + hr];
        const float M = fmaxf(m, mo.x);
        const float fm = m == -INFINITY ? 0.f : ex2(m - M);
        const float fo = mo.x == -INFINITY ? 0.f : ex2(mo.x - M);
        if (cp == 0) p.part_ml[prow] = make_float2(M, fmaf(mo.y, fo, l * fm));
        {
          uint32_t raw[Lay::kHalf];
          if constexpr (Lay::kHalf == 64) tmem_ld64(to + cp * Lay::kHalf, raw);
          else tmem_ld32(to + cp * Lay::kHalf, raw);
          float4* dst = reinterpret_cast<float4*>(p.part_acc + prow * D + cp * Lay::kHalf);
#pragma unroll
          for (int j = 0; j < Lay::kHalf / 4; ++j) {
            float o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
              o[i] = fmaf(in_row[4 * j + i], fo, __uint_as_float(raw[4 * j + i]) * fm);
            dst[j] = make_float4(o[0], o[1], o[2], o[3]);
          }
        }
        mbar_arrive(mrg_free);
      } else {
        // the copies' output rows meet in shared memory, half of D per round
        // (rounds 2k and 2k + 1 of this CTA's k-th unit)
        float f[C], M = m, lt = 0.f;
        for (int hf = 0; hf < 2 && ok; ++hf) {
          const int round = 2 * k + hf;
          if (cp > 0) {
            if (round >= 1 && !__all_sync(0xffffffffu, mbar_wait(mrg_free, (round - 1) & 1, p.wait_ns))) {
              ok = false;
              break;
            }
            float* row = merge + ((cp - 1) * G + hr) * Lay::kMergeStride;
#pragma unroll
            for (int h = 0; h < Lay::kHalf / 32; ++h) {
              uint32_t raw[32];
              tmem_ld32(to + hf * Lay::kHalf + h * 32, raw);
#pragma unroll
              for (int e = 0; e < 32; ++e) row[h * 32 + e] = __uint_as_float(raw[e]);
            }
            if (hf == 0) mrg_ml[(cp - 1) * G + hr] = make_float2(m, l);
            mbar_arrive(mrg_full);
          } else {
            if (!__all_sync(0xffffffffu, mbar_wait(mrg_full, round & 1, p.wait_ns))) {
              ok = false;
              break;
            }
            if (hf == 0) {
#pragma unroll
              for (int cc = 1; cc < C; ++cc) M = fmaxf(M, mrg_ml[(cc - 1) * G + hr].x);
              f[0] = m == -INFINITY ? 0.f : ex2(m - M);
              lt = l * f[0];
#pragma unroll
              for (int cc = 1; cc < C; ++cc) {
                const float2 ml = mrg_ml[(cc - 1) * G + hr];
                f[cc] = ml.x == -INFINITY ? 0.f : ex2(ml.x - M);
                lt = fmaf(ml.y, f[cc], lt);
              }
              p.part_ml[prow] = make_float2(M, lt);
            }
#pragma unroll
            for (int h = 0; h < Lay::kHalf / 32; ++h) {
              uint32_t raw[32];
              tmem_ld32(to + hf * Lay::kHalf + h * 32, raw);
              float4* dst = reinterpret_cast<float4*>(p.part_acc + prow * D + hf * Lay::kHalf + h * 32);
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                float o[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  o[i] = __uint_as_float(raw[4 * j + i]) * f[0];
#pragma unroll
                  for (int cc = 1; cc < C; ++cc)
                    o[i] = fmaf(merge[((cc - 1) * G + hr) * Lay::kMergeStride + h * 32 + 4 * j + i],
                                f[cc], o[i]);
                }
                dst[j] = make_float4(o[0], o[1], o[2], o[3]);
              }
            }
            mbar_arrive(mrg_free);
          }
        }
        if (!ok) break;
      }
      tc_fence_before();
      mbar_arrive(&o_free[slot]);
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

template <int D, typename T, int C>
static cudaError_t launch(const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq,
                          const Params& p, cudaStream_t s) {
  auto kern = decode_tc_kernel<D, T, C>;
  using Lay = Layout<D, C>;
  // one CTA per SM: it holds all 512 tensor-memory columns, so shared memory is
  // requested past half an SM even where the layout needs less (d = 64)
  constexpr int kSmemLaunch = Lay::kSmem > 120 * 1024 ? Lay::kSmem : 120 * 1024;
  int sms = 0;
  cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), kThreads, kSmemLaunch,
                                 nullptr);
  if (e == cudaSuccess) e = device_sm_count(&sms);
  if (e != cudaSuccess) return e;
  const int grid = std::max(1, std::min(p.total_units, sms));
  e = cudaMemsetAsync(p.counter, 0, sizeof(int), s);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, kSmemLaunch, s>>>(tk, tv, tq, p);
  return cudaGetLastError();
}

template <int C>
static cudaError_t launch_c(int D, bool bf16, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& tq, const Params& p, cudaStream_t s) {
  if (D == 128) return bf16 ? launch<128, BF16, C>(tk, tv, tq, p, s)
                            : launch<128, F16, C>(tk, tv, tq, p, s);
  return bf16 ? launch<64, BF16, C>(tk, tv, tq, p, s) : launch<64, F16, C>(tk, tv, tq, p, s);
}

}  // namespace tcdec

static cudaError_t dispatch_copies(int D, bool bf16, int copies, const CUtensorMap& tk,
                                   const CUtensorMap& tv, const CUtensorMap& tq,
                                   const tcdec::Params& p, cudaStream_t s) {
  switch (copies) {
    case 1: return tcdec::launch_c<1>(D, bf16, tk, tv, tq, p, s);
    case 2: return tcdec::launch_c<2>(D, bf16, tk, tv, tq, p, s);
    default: return tcdec::launch_c<4>(D, bf16, tk, tv, tq, p, s);
  }
}

// From 32 heads per KV head on, reading each K/V byte once beats the
// warp-level path's re-reads (measured: 1.6x at 32, 2.6x at 64, 4.3x at 128
// heads; at 16 the warp-level path's two reads still win).
bool decode_tc_supported(int group, int head_size, int block_size, int partition_tokens) {
  return group >= 32 && tcdec::kRows % group == 0 && (head_size == 64 || head_size == 128) &&
         block_size >= 8 && partition_tokens % tcdec::kKeys == 0 &&
         partition_tokens / block_size + 2 <= tcdec::kMaxIds;
}

cudaError_t launch_decode_tc(const DecodeTcArgs& a, cudaStream_t s) {
  const int group = a.num_heads / a.num_kv_heads;
  const int box_rows = std::min(a.block_size, tcdec::kKeys);
  const int64_t slots = static_cast<int64_t>(a.num_blocks) * a.block_size;
  CUtensorMap tk, tv, tq;
  if (!encode_cache_map(&tk, a.k_cache, a.head_size, a.num_kv_heads, slots, box_rows,
                        kLineSwizzled) ||
      !encode_cache_map(&tv, a.v_cache, a.head_size, a.num_kv_heads, slots, box_rows,
                        kLineSwizzled) ||
      !encode_query_map(&tq, a.q, a.head_size, static_cast<int64_t>(a.num_seqs) * a.num_heads,
                        group))
    return cudaErrorInvalidValue;
  tcdec::Params p{};
  p.part_acc = a.part_acc;
  p.part_ml = a.part_ml;
  p.counter = a.counter;
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.err = a.err;
  p.num_seqs = a.num_seqs;
  p.num_heads = a.num_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = group;
  p.num_blocks = a.num_blocks;
  p.block_size = a.block_size;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.partition_tokens = a.partition_tokens;
  p.max_parts = a.max_parts;
  p.total_units = a.max_parts * a.num_seqs * a.num_kv_heads;
  p.box_rows = box_rows;
  p.q_scale = a.q_scale;
  p.wait_ns = a.wait_ns;
  p.stall_unit = a.stall_unit;
  return dispatch_copies(a.head_size, a.bf16, tcdec::kRows / group, tk, tv, tq, p, s);
}

}  // namespace pkv
