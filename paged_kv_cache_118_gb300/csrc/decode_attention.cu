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
//  * decode_reduce_kernel — one warp (four for rows of many partitions) per
//    (sequence, query head) merges the partition partials: M = max m_p,
//    Z = sum l_p 2^(m_p - M), o = sum acc_p 2^(m_p - M) / Z, rounded to the
//    output type, with several partitions' loads in flight at once.
// Every wait on an mbarrier has a time limit (see pkv_device.cuh); a block id
// or context length out of range is skipped and reported through err_flag.

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <type_traits>

#include "pagedkv.h"
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {

constexpr int kTile = 32;           // tokens per pipeline stage
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 2) * 32;   // + copy warp + scheduler warp
constexpr int kGroupLanes = 8;      // lanes that share one token row
constexpr int kGroups = kConsumerWarps * 32 / kGroupLanes;  // token groups per CTA (16)
constexpr float kRescaleThreshold = 8.0f;  // base-2 growth of the max that forces a rescale
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kCompactMaxSeqs = 1024;       // batches up to this size get a compact work list
constexpr int kMmaHeads = 8;                // query heads of one KV head a tensor-path CTA serves
constexpr int kMmaRows = 16;                // rows of its products: heads x sequences of a run
constexpr int kMaxRun = 8;                  // sequences one tensor-path unit serves at most
constexpr int kMaxGroupParts = 4095;        // group claims need F < 2^12 (packed with flags)
// The scheduler claims another unit whenever fewer than this many tiles of
// staged units are left to issue: enough to hide the claims (several short
// units may be staged at once), few enough to keep the end of the work list
// balanced across CTAs.
constexpr int kClaimAheadTiles = 2;
constexpr int kClaimAheadTilesMma = 16;
constexpr int kSchedSlots = 4;              // staged units (descriptor + table slice)

struct DecodeParams {
  float* part_acc;            // [rows][D], rows = num_seqs * num_heads * max_parts
  float2* part_ml;            // [rows] = (m in base-2 units, l)
  int* counter;               // work counter, zero at launch
  const uint16_t* q;          // [num_seqs][num_heads][D]
  const int32_t* block_tables;
  const int32_t* context_lens;
  int32_t* err;
  int num_seqs;
  int num_heads;
  int group;                  // query heads per KV head (num_heads / num_kv_heads)
  int subs;                   // CTAs' query-head slices per KV head
  int heads_per_cta;          // query heads one CTA serves (GS; at most 8 on the tensor path)
  int kv_slices;              // num_kv_heads * subs
  int num_blocks;
  int block_size;
  int max_blocks_per_seq;
  int partition_tokens;
  int max_parts;
  int total_units;            // max_parts * num_seqs * kv_slices
  int box_rows;               // rows per TMA copy: min(block_size, kTile)
  float q_scale;              // scale * log2(e)
};

// What the producer tells the consumers about the next unit of work.
struct UnitDesc {
  int seq;                    // -1: no more units; -2: the producer gave up (timeout)
  int head0;
  int part;
  int len;
  int nrun;                   // sequences seq .. seq+nrun-1 whose blocks for this
                              // partition are identical (shared prefix), served together
};

// The ring has 4 stages (5 on the tensor path, whose merge needs less room);
// on the tensor path GS is the row capacity (kMmaRows).
template <int D, int GS, bool kMma = false>
struct DecodeLayout {
  static constexpr int kStages = kMma ? 5 : 4;
  static constexpr int kRowBytes = D * 2;
  static constexpr int kTileBytes = kTile * kRowBytes;        // K (or V) of one stage
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kQBytes = GS * D * 2;                  // query rows of one unit (capacity)
  // merge area: per warp and row D + 2 floats; on the tensor path two warps'
  // fragments, (D/8 + 1) float4s per lane
  static constexpr int kCombineFloats =
      kMma ? 2 * (D / 8 + 1) * 32 * 4 : kConsumerWarps * GS * (D + 2);
  static constexpr int kChunks = D / 64;                      // 16-byte pieces per lane per row
  static constexpr int kE = 8 * kChunks;                      // elements per lane per row
  // offsets (bytes) from the 1024-aligned base
  static constexpr int kOffCombine = kRingBytes;
  static constexpr int kOffQ = kOffCombine + kCombineFloats * 4;
  static constexpr int kOffBars = kOffQ + kQBytes;            // 16-byte aligned
  // full, empty (ring); q_full, q_empty (one query buffer: the consumers
  // copy it to registers when a unit starts); merge; sched_full, sched_empty;
  // tree merge of the tensor path: x_full, x_free, y_full
  static constexpr int kNumBars = 2 * kStages + 1 + 1 + 2 + 2 * kSchedSlots + 3;
  static constexpr int kOffUnits = kOffBars + kNumBars * 8;    // units[1], then sched[]
  static constexpr int kOffFlag = kOffUnits + (1 + kSchedSlots) * sizeof(UnitDesc);
  static constexpr int kOffPref = (kOffFlag + 16 + 15) / 16 * 16;  // prefix of whole partitions per sequence
  static constexpr int kOffGroup = kOffPref + ((kCompactMaxSeqs + 1) * 4 + 15) / 16 * 16;
  // the sequences with a partial last partition, largest first (16-bit ids);
  // on the scalar paths, which form no groups, it takes the group info's place
  static constexpr int kOffOrder = kOffGroup + (kMma ? (kCompactMaxSeqs * 2 + 15) / 16 * 16 : 0);
  static constexpr int kOffSlice = kOffOrder + (kCompactMaxSeqs * 2 + 15) / 16 * 16;
  // table_slice: entries of one unit's block-table slice; kSchedSlots are staged
  static int smem_bytes(int table_slice) {
    return 1024 /*alignment slack*/ + kOffSlice + ((kSchedSlots * table_slice * 4 + 15) / 16) * 16;
  }
};

// Transposed reduction inside an 8-lane token group: every lane holds partial
// dot products for the GS heads over its 16 (or 8) elements; after three
// exchange steps each lane holds the full score of one head (lane pairs for
// GS=4, quads for GS=2), owners of a head agreeing bit for bit. It replaces
// GS separate butterflies (3*GS shuffles) by 4 (GS=4) or 3 shuffles.
template <int GS>
struct GroupHeads;
template <>
struct GroupHeads<2> {
  // lane j owns head (j >> 2) & 1
  static __device__ __forceinline__ int owner(int g) { return 4 * g; }
  static __device__ __forceinline__ float reduce(const float* s, int j, unsigned mask) {
    const bool hi = (j >> 2) & 1;
    const float send = hi ? s[0] : s[1];
    float x = hi ? s[1] : s[0];
    x += __shfl_xor_sync(mask, send, 4);
    x += __shfl_xor_sync(mask, x, 2);
    x += __shfl_xor_sync(mask, x, 1);
    return x;
  }
};
template <>
struct GroupHeads<4> {
  // lane j owns head 2 * ((j >> 2) & 1) + ((j >> 1) & 1)
  static __device__ __forceinline__ int owner(int g) { return 4 * (g >> 1) + 2 * (g & 1); }
  static __device__ __forceinline__ float reduce(const float* s, int j, unsigned mask) {
    const bool b2 = (j >> 2) & 1;
    const bool b1 = (j >> 1) & 1;
    const float send0 = b2 ? s[0] : s[2];
    const float send1 = b2 ? s[1] : s[3];
    float k0 = b2 ? s[2] : s[0];
    float k1 = b2 ? s[3] : s[1];
    k0 += __shfl_xor_sync(mask, send0, 4);
    k1 += __shfl_xor_sync(mask, send1, 4);
    const float send = b1 ? k0 : k1;
    float x = b1 ? k1 : k0;
    x += __shfl_xor_sync(mask, send, 2);
    x += __shfl_xor_sync(mask, x, 1);
    return x;
  }
};

__device__ __forceinline__ int ld_volatile(const int* p) { return *reinterpret_cast<const volatile int*>(p); }
__device__ __forceinline__ void st_volatile(int* p, int v) { *reinterpret_cast<volatile int*>(p) = v; }

// Per-lane state of one unit for one token group: scalar math for one query
// head (GS = 1), packed f32x2 math with the transposed reduction otherwise.
template <int D, int GS, typename T>
struct GroupState;

template <int D, typename T>
struct GroupState<D, 1, T> {
  static constexpr int E = DecodeLayout<D, 1>::kE;
  static constexpr int kChunks = DecodeLayout<D, 1>::kChunks;
  float q[E], acc[E], m, l;

  __device__ __forceinline__ void begin(const uint16_t* qs, int j, float q_scale) {
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      const uint4 raw = *reinterpret_cast<const uint4*>(qs + c * 64 + 8 * j);
      widen8<T>(raw, &q[c * 8]);
#pragma unroll
      for (int e = 0; e < 8; ++e) q[c * 8 + e] *= q_scale;
    }
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    m = -INFINITY;
    l = 0.f;
  }

  __device__ __forceinline__ void token(const uint16_t* krow, const uint16_t* vrow, int j,
                                        unsigned gmask, int) {
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      const uint4 raw = *reinterpret_cast<const uint4*>(krow + c * 64 + 8 * j);
      float kf[8];
      widen8<T>(raw, kf);
#pragma unroll
      for (int e = 0; e < 8; ++e) s = fmaf(q[c * 8 + e], kf[e], s);
    }
    s += __shfl_xor_sync(gmask, s, 1);
    s += __shfl_xor_sync(gmask, s, 2);
    s += __shfl_xor_sync(gmask, s, 4);
    if (s > m + kRescaleThreshold) {            // uniform in the group
      const float corr = ex2(m - s);
      l *= corr;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] *= corr;
      m = s;
    }
    const float pr = ex2(s - m);
    l += pr;
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      const uint4 raw = *reinterpret_cast<const uint4*>(vrow + c * 64 + 8 * j);
      float vf[8];
      widen8<T>(raw, vf);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[c * 8 + e] = fmaf(pr, vf[e], acc[c * 8 + e]);
    }
  }

  __device__ __forceinline__ float head_m(int, int) const { return m; }
  __device__ __forceinline__ float head_l(int, int) const { return l; }
  __device__ __forceinline__ void head_acc(int, int e, float& a, float& b) const {
    a = acc[2 * e];
    b = acc[2 * e + 1];
  }
};

template <int D, int GS, typename T>
struct GroupState {
  static constexpr int E = DecodeLayout<D, GS>::kE;
  static constexpr int P2 = E / 2;
  static constexpr int kChunks = DecodeLayout<D, GS>::kChunks;
  f32x2 q2[GS][P2], acc[GS][P2];
  float m, l;     // state of the head this lane owns (GroupHeads<GS>)

  __device__ __forceinline__ void begin(const uint16_t* qs, int j, float q_scale) {
    const f32x2 sc = pack2(q_scale, q_scale);
#pragma unroll
    for (int g = 0; g < GS; ++g)
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        const uint4 raw = *reinterpret_cast<const uint4*>(qs + g * D + c * 64 + 8 * j);
        q2[g][c * 4 + 0] = mul2(T::to_pair(raw.x), sc);
        q2[g][c * 4 + 1] = mul2(T::to_pair(raw.y), sc);
        q2[g][c * 4 + 2] = mul2(T::to_pair(raw.z), sc);
        q2[g][c * 4 + 3] = mul2(T::to_pair(raw.w), sc);
      }
#pragma unroll
    for (int g = 0; g < GS; ++g)
#pragma unroll
      for (int e = 0; e < P2; ++e) acc[g][e] = 0ull;
    m = -INFINITY;
    l = 0.f;
  }

  __device__ __forceinline__ void token(const uint16_t* krow, const uint16_t* vrow, int j,
                                        unsigned gmask, int base) {
    // q.k for the GS heads: one widening of each key pair serves all heads.
    f32x2 d2[GS];
#pragma unroll
    for (int g = 0; g < GS; ++g) d2[g] = 0ull;
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      const uint4 raw = *reinterpret_cast<const uint4*>(krow + c * 64 + 8 * j);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const f32x2 kp = T::to_pair(w[u]);
#pragma unroll
        for (int g = 0; g < GS; ++g) d2[g] = fma2(q2[g][c * 4 + u], kp, d2[g]);
      }
    }
    float s[GS];
#pragma unroll
    for (int g = 0; g < GS; ++g) {
      float a, b;
      unpack2(d2[g], a, b);
      s[g] = a + b;
    }
    const float sc = GroupHeads<GS>::reduce(s, j, gmask);
    // Online softmax of the owned head; the accumulators of every head are
    // rescaled only when some head's maximum grows by more than 2^8.
    const bool need = sc > m + kRescaleThreshold;
    if (__any_sync(gmask, need)) {
      const float mn = need ? sc : m;
      const float corr = need ? ex2(m - mn) : 1.f;
      m = mn;
      l *= corr;
#pragma unroll
      for (int g = 0; g < GS; ++g) {
        const float cg = __shfl_sync(gmask, corr, base + GroupHeads<GS>::owner(g));
        const f32x2 c2 = pack2(cg, cg);
#pragma unroll
        for (int e = 0; e < P2; ++e) acc[g][e] = mul2(acc[g][e], c2);
      }
    }
    const float pr = ex2(sc - m);
    l += pr;
    f32x2 pg[GS];
#pragma unroll
    for (int g = 0; g < GS; ++g) {
      const float x = __shfl_sync(gmask, pr, base + GroupHeads<GS>::owner(g));
      pg[g] = pack2(x, x);
    }
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      const uint4 raw = *reinterpret_cast<const uint4*>(vrow + c * 64 + 8 * j);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const f32x2 vp = T::to_pair(w[u]);
#pragma unroll
        for (int g = 0; g < GS; ++g) acc[g][c * 4 + u] = fma2(pg[g], vp, acc[g][c * 4 + u]);
      }
    }
  }

  __device__ __forceinline__ float head_m(int g, int base) const {
    return __shfl_sync(0xffffffffu, m, base + GroupHeads<GS>::owner(g));
  }
  __device__ __forceinline__ float head_l(int g, int base) const {
    return __shfl_sync(0xffffffffu, l, base + GroupHeads<GS>::owner(g));
  }
  __device__ __forceinline__ void head_acc(int g, int e, float& a, float& b) const {
    unpack2(acc[g][e], a, b);
  }
};

// Tensor-core state of one consumer warp (grouped query heads): the warp owns
// 8 tokens of every 32-token tile. q.k and p.v run as warp-level m16n8k16 /
// m16n8k8 products with fp32 accumulation; the 16 rows of A are the query
// heads of the unit's sequences (rows past them are zero). Lane
// (g = lane/4, t = lane%4) holds the scores of rows g and g+8 for tokens 2t,
// 2t+1 and their output columns 8j + 2t, 8j + 2t + 1. P is fed as two halves
// in the input format (p = hi + lo), which keeps p.v at close to fp32 accuracy.
// K and V tiles are stored by TMA with the 128-byte swizzle, each copy of R
// rows line-major (swizzled_chunk): the eight rows one ldmatrix reads sit in
// eight swizzle phases, so it meets no bank conflict, while one TMA box still
// moves whole rows of a block.
template <int D, typename T>
struct MmaState {
  static constexpr int KS = D / 16;               // k-steps of q.k
  static constexpr int NT = D / 8;                // 8-column tiles of the output
  static constexpr int NH = D / 64;               // 128-byte lines per token row
  // A fragments: [0] row g, k 2t..; [1] row g+8, k 2t..; [2] row g, k 2t+8..; [3] row g+8, k 2t+8..
  uint32_t qa[KS][4];
  float o[NT][4];                                 // [0..1] row g, [2..3] row g+8
  float mA, lA, mB, lB;                           // rows g and g+8

  // rows: query rows of the unit (sequences of the run x heads), at most 16
  __device__ __forceinline__ void begin(const uint16_t* qs, int rows, int lane) {
    const int g = lane >> 2, t = lane & 3;
    const bool ra = g < rows, rb = g + 8 < rows;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int c = 16 * ks + 2 * t;
      qa[ks][0] = ra ? *reinterpret_cast<const uint32_t*>(qs + g * D + c) : 0u;
      qa[ks][1] = rb ? *reinterpret_cast<const uint32_t*>(qs + (g + 8) * D + c) : 0u;
      qa[ks][2] = ra ? *reinterpret_cast<const uint32_t*>(qs + g * D + c + 8) : 0u;
      qa[ks][3] = rb ? *reinterpret_cast<const uint32_t*>(qs + (g + 8) * D + c + 8) : 0u;
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    mA = mB = -INFINITY;
    lA = lB = 0.f;
  }

  // kt, vt: the stage's K and V tiles, filled by copies of 2^rs rows; tok0:
  // first token of this warp in the tile; valid: tokens of the tile that exist.
  // kTwo: rows 8..15 hold query rows (a run of sequences); without them their
  // softmax is skipped and their products stay zero.
  template <bool kTwo>
  __device__ __forceinline__ void tile(const uint8_t* kt, const uint8_t* vt, int tok0, int valid,
                                       float q_scale, int lane, int rs) {
    const int t = lane & 3;
    const int r = lane & 7;                       // row this lane addresses in ldmatrix
    const int mat = lane >> 3;                    // matrix this lane addresses
    // two accumulators halve the dependent chain of products
    float s[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kp = 0; kp < KS / 2; ++kp) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(swizzled_chunk<NH>(kt, tok0 + r, 4 * kp + mat, rs), b0, b1, b2, b3);
      T::mma16816(s, qa[2 * kp][0], qa[2 * kp][1], qa[2 * kp][2], qa[2 * kp][3], b0, b1);
      T::mma16816(s2, qa[2 * kp + 1][0], qa[2 * kp + 1][1], qa[2 * kp + 1][2], qa[2 * kp + 1][3],
                  b2, b3);
    }
    const int tk = tok0 + 2 * t;
    const bool v0 = tk < valid, v1 = tk + 1 < valid;
    const float a0 = v0 ? (s[0] + s2[0]) * q_scale : -INFINITY;
    const float a1 = v1 ? (s[1] + s2[1]) * q_scale : -INFINITY;
    float tmA = fmaxf(a0, a1);
    tmA = fmaxf(tmA, __shfl_xor_sync(0xffffffffu, tmA, 1));
    tmA = fmaxf(tmA, __shfl_xor_sync(0xffffffffu, tmA, 2));
    const bool needA = tmA > mA + kRescaleThreshold;
    float b0s = -INFINITY, b1s = -INFINITY, tmB = -INFINITY;
    bool needB = false;
    if constexpr (kTwo) {
      b0s = v0 ? (s[2] + s2[2]) * q_scale : -INFINITY;
      b1s = v1 ? (s[3] + s2[3]) * q_scale : -INFINITY;
      tmB = fmaxf(b0s, b1s);
      tmB = fmaxf(tmB, __shfl_xor_sync(0xffffffffu, tmB, 1));
      tmB = fmaxf(tmB, __shfl_xor_sync(0xffffffffu, tmB, 2));
      needB = tmB > mB + kRescaleThreshold;
    }
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
    const float pa0 = a0 == -INFINITY ? 0.f : ex2(a0 - mA);
    const float pa1 = a1 == -INFINITY ? 0.f : ex2(a1 - mA);
    lA += pa0 + pa1;
    // P as two halves in the input format: p = hi + lo
    const uint32_t hA = T::pack(pa0, pa1);
    const float2 fA = T::to_float2(hA);
    const uint32_t lAo = T::pack(pa0 - fA.x, pa1 - fA.y);
    uint32_t hB = 0u, lBo = 0u;
    if constexpr (kTwo) {
      const float pb0 = b0s == -INFINITY ? 0.f : ex2(b0s - mB);
      const float pb1 = b1s == -INFINITY ? 0.f : ex2(b1s - mB);
      lB += pb0 + pb1;
      hB = T::pack(pb0, pb1);
      const float2 fB = T::to_float2(hB);
      lBo = T::pack(pb0 - fB.x, pb1 - fB.y);
    }
    // V rows of tokens past the tile's end may hold anything: zero their halves.
    const uint32_t keep = (v0 ? 0x0000ffffu : 0u) | (v1 ? 0xffff0000u : 0u);
#pragma unroll
    for (int nq = 0; nq < NT / 4; ++nq) {
      uint32_t b[4];
      ldsm_x4_t(swizzled_chunk<NH>(vt, tok0 + r, 4 * nq + mat, rs), b[0], b[1], b[2], b[3]);
#pragma unroll
      for (int i = 0; i < 4; ++i) b[i] &= keep;
#pragma unroll
      for (int i = 0; i < 4; ++i) T::mma1688(o[4 * nq + i], hA, hB, b[i]);
#pragma unroll
      for (int i = 0; i < 4; ++i) T::mma1688(o[4 * nq + i], lAo, lBo, b[i]);
    }
  }
};

// Builds the compact work list (see decode_partition_kernel) with all the
// CTA's threads: per chunk of 32 sequences (one warp each, every load in
// flight at once) the claims of whole partitions, the group info and the tile
// count of the partial last partition; then the prefix sums over the chunks,
// and a stable counting sort of the partial partitions by tile count, largest
// first, equal counts in sequence order. Every CTA builds the list on its own
// and claims index into it, so it must come out the same in every CTA: no
// step depends on the order of concurrent events. `scratch` is shared memory
// that no copy has reached yet (the ring); a proxy fence hands it back to the
// TMA copies. Ends with a block-wide barrier.
__device__ __forceinline__ void build_work_list(const DecodeParams& p, int max_ctx, bool grouping,
                                                int cap, int* scratch, int* pref, uint16_t* ginfo,
                                                uint16_t* porder, int& whole_units,
                                                int& partial_units) {
  constexpr int kWarps = kThreads / 32;
  constexpr int kChunks = kCompactMaxSeqs / 32;
  constexpr int kChunksPerWarp = (kChunks + kWarps - 1) / kWarps;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = p.num_seqs;
  const int nchunks = (n + 31) / 32;
  const int PT = p.partition_tokens;
  const int nbk = PT / kTile;                          // tile counts of partial partitions: 1 .. nbk
  // scratch: claims per chunk, then their offsets [32]; totals [2]; per tile
  // count its first place [nbk + 1]; per (tile count, chunk) the count, then
  // the place of the chunk's first one [(nbk + 1) * 32]; per sequence its
  // tile count and its rank among the chunk's equal counts [n] bytes each
  int* chunk_sum = scratch;
  int* totals = scratch + 32;
  int* base = scratch + 40;
  int* cnt = base + (nbk + 1);
  uint8_t* tiles_of = reinterpret_cast<uint8_t*>(cnt + (nbk + 1) * kChunks);
  uint8_t* rank_of = tiles_of + kCompactMaxSeqs;
  for (int i = tid; i < (nbk + 1) * kChunks; i += kThreads) cnt[i] = 0;
  int L[kChunksPerWarp], fb[kChunksPerWarp];
#pragma unroll
  for (int j = 0; j < kChunksPerWarp; ++j) {          // every load of this warp in flight at once
    const int s = (warp + j * kWarps) * 32 + lane;
    L[j] = s < n ? __ldg(p.context_lens + s) : 0;
    fb[j] = (grouping && s < n) ? __ldg(p.block_tables + static_cast<int64_t>(s) * p.max_blocks_per_seq) : -1;
  }
  __syncthreads();                                     // cnt is zero
#pragma unroll
  for (int j = 0; j < kChunksPerWarp; ++j) {
    const int ch = warp + j * kWarps;
    if (ch >= nchunks) break;
    const int s = ch * 32 + lane;
    const bool valid = s < n && L[j] >= 1 && L[j] <= max_ctx;
    if (s < n && !valid && blockIdx.x == 0) flag_error(p.err, PKV_DEVERR_CONTEXT);
    const int whole = valid ? L[j] / PT : 0;
    int c = whole;                                     // claims of this sequence's whole partitions
    if (grouping) {
      const int fb_prev = __shfl_up_sync(0xffffffffu, fb[j], 1);
      const int valid_prev = __shfl_up_sync(0xffffffffu, valid ? 1 : 0, 1);
      // windows never straddle the 32 lanes: cap divides 32
      const bool link = valid && valid_prev && (s & (cap - 1)) != 0 && fb[j] >= 0 && fb[j] == fb_prev;
      const unsigned starts = __ballot_sync(0xffffffffu, !link);
      const int hd = 31 - __clz(starts & (0xffffffffu >> (31 - lane)));   // group's first lane
      const int wb = lane & ~(cap - 1);
      const unsigned later = starts & ~(0xffffffffu >> (31 - hd));
      const int nx = later ? min(__ffs(later) - 1, wb + cap) : wb + cap;  // past the group
      int fmin = whole;
#pragma unroll
      for (int m = 0; m < kMaxRun; ++m) {
        const int v = __shfl_sync(0xffffffffu, whole, (wb + m) & 31);
        if (m < cap && wb + m >= hd && wb + m < nx) fmin = min(fmin, v);
      }
      uint16_t gi = 0;
      if (nx - hd > 1) {
        const bool member = lane != hd;
        if (member) c = whole - fmin;
        gi = static_cast<uint16_t>((fmin << 4) | ((nx - hd - 1) << 1) | (member ? 1 : 0));
      }
      if (s < n) ginfo[s] = gi;
    }
    int x = c;                                         // inclusive scan within the chunk
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (s < n) pref[s + 1] = x;
    if (lane == 31) chunk_sum[ch] = x;
    // the partial partition's tile count, and its rank among the chunk's
    // sequences with the same count (in lane order)
    const int r = valid ? L[j] % PT : 0;
    const int t = (r + kTile - 1) / kTile;           // 0: none; at most nbk <= 128
    const unsigned same = __match_any_sync(0xffffffffu, t);
    if (s < n) {
      tiles_of[s] = static_cast<uint8_t>(t);
      rank_of[s] = static_cast<uint8_t>(__popc(same & ((1u << lane) - 1u)));
    }
    if (t > 0 && lane == __ffs(same) - 1) cnt[t * kChunks + ch] = __popc(same);
  }
  __syncthreads();
  if (warp == 0) {                                     // chunk offsets of the claims (exclusive)
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
  // per tile count: its chunks' counts become places within the count
  for (int b = 1 + tid; b <= nbk; b += kThreads) {
    int acc = 0;
    for (int ch = 0; ch < nchunks; ++ch) {
      const int v = cnt[b * kChunks + ch];
      cnt[b * kChunks + ch] = acc;
      acc += v;
    }
    base[b] = acc;                                     // total of this count, for now
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
  fence_proxy_async_smem();                            // the ring goes back to the copies
  __syncthreads();
}

// Persistent: each CTA takes units of work — (context partition, sequence,
// KV-head slice), partition-major — from a global counter until none is
// left. The scheduler and copy warps fetch the next unit, its slice of the
// block table and its query rows while the consumers still work on the
// current one.
// kMma: grouped query heads on the tensor path (MmaState; K/V tiles stored
// with 128-byte swizzle by 64-element halves; GS is then the row capacity, 16:
// p.heads_per_cta heads of each of up to 16 / p.heads_per_cta sequences that
// share the partition's blocks). Otherwise GroupState.
template <int D, int GS, typename T, bool kMma>
__global__ void __launch_bounds__(kThreads, (GS >= 2 || kMma) ? 2 : 3)
    decode_partition_kernel(const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
  using Lay = DecodeLayout<D, GS, kMma>;
  constexpr int kStages = Lay::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* ring = smem;
  float* combine = reinterpret_cast<float*>(smem + Lay::kOffCombine);
  uint16_t* qbuf = reinterpret_cast<uint16_t*>(smem + Lay::kOffQ);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + Lay::kOffBars);
  uint64_t* empty_bar = full_bar + kStages;
  uint64_t* q_full = empty_bar + kStages;
  uint64_t* q_empty = q_full + 1;
  uint64_t* merge_bar = q_empty + 1;          // [0]: partials written, [1]: partials read
  uint64_t* sched_full = merge_bar + 2;       // scheduler -> copy warp, per staged unit
  uint64_t* sched_empty = sched_full + kSchedSlots;
  uint64_t* x_full = sched_empty + kSchedSlots;   // tensor path: warps 2, 3 -> warps 0, 1
  uint64_t* x_free = x_full + 1;
  uint64_t* y_full = x_free + 1;              // warp 1 -> warp 0
  UnitDesc* units = reinterpret_cast<UnitDesc*>(smem + Lay::kOffUnits);
  UnitDesc* sched = units + 1;
  int* abort_flag = reinterpret_cast<int*>(smem + Lay::kOffFlag);
  int* issued_tiles = abort_flag + 1;         // copy warp's tile count, read by the scheduler
  int* pref = reinterpret_cast<int*>(smem + Lay::kOffPref);
  uint16_t* ginfo = reinterpret_cast<uint16_t*>(smem + Lay::kOffGroup);
  uint16_t* porder = reinterpret_cast<uint16_t*>(smem + Lay::kOffOrder);
  int32_t* slice = reinterpret_cast<int32_t*>(smem + Lay::kOffSlice);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int B = p.block_size;
  const int max_ctx = p.max_blocks_per_seq * B;
  const int per_part = p.num_seqs * p.kv_slices;
  const int slice_cap = p.partition_tokens / B + 2;   // entries of one staged slice

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], kConsumerWarps);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, kConsumerWarps);
    for (int i = 0; i < 2; ++i) mbar_init(&merge_bar[i], kConsumerWarps);
    for (int i = 0; i < kSchedSlots; ++i) {
      mbar_init(&sched_full[i], 32);
      mbar_init(&sched_empty[i], 1);
    }
    mbar_init(x_full, 2);
    mbar_init(x_free, 1);
    mbar_init(y_full, 1);
    *abort_flag = 0;
    *issued_tiles = 0;
    fence_barrier_init();
  }
  __syncthreads();

  // The work list. For batches of up to kCompactMaxSeqs sequences only the
  // units that exist are numbered: first every whole partition,
  // sequence-major (a prefix sum of claims per sequence, then a binary search
  // per claim), then the partial last partitions, largest first, so that the
  // list ends with its shortest units and the CTAs finish close together.
  // Every warp helps build it before taking its role. Larger batches number
  // every (partition, sequence, slice) and skip the empty ones.
  //
  // Groups (tensor path): consecutive sequences of an aligned window of `cap`
  // (a power of two) whose first blocks are the same physical block (a shared
  // prefix) form a group. The partitions that are whole for every member, F
  // of them, are claimed once for the group by its first sequence; each member
  // claims only its own partitions from F on. A group claim checks the
  // members' table entries for that partition and serves the runs of identical
  // ones (normally one run: the whole group) as units.
  const bool compact = p.num_seqs <= kCompactMaxSeqs;
  int cap = 1;
  if (kMma) {
    const int c = min(kMmaRows / p.heads_per_cta, kMaxRun);
    cap = 1 << (31 - __clz(c));
  }
  const bool grouping = kMma && cap > 1 && compact && p.max_parts <= kMaxGroupParts;
  int whole_units = 0, partial_units = 0;
  if (compact)
    build_work_list(p, max_ctx, grouping, cap, reinterpret_cast<int*>(ring), pref, ginfo, porder,
                    whole_units, partial_units);

  // ------------------------------------------------------------ scheduler warp
  // Claims units from the global counter, resolves each one (sequence,
  // partition, head slice; on the tensor path the run of sequences that share
  // the partition's blocks) and stages its block-table slice ahead of the copy
  // warp, so that none of this latency falls between two units of the copy
  // stream.
  if (warp == kConsumerWarps + 1) {
    const int total = compact ? (whole_units + partial_units) * p.kv_slices : p.total_units;
    const int ahead = kMma ? kClaimAheadTilesMma : kClaimAheadTiles;
    bool ok = true;
    int staged = 0;                           // tiles of the units staged so far
    // runs of the last group claim still to be staged
    unsigned pend = 0, plink = 0;
    bool claimed = false;                     // the first unit is the CTA's index
    int pseq = 0, ppart = 0, pkvs = 0, pLm = 0, pgs = 0;
    for (int k = 0;; ++k) {
      if (k >= 1) {                           // wait until the staged backlog runs low
        int w = 1;
        if (lane == 0) {
          const uint64_t t0 = globaltimer_ns();
          while (staged - ld_volatile(issued_tiles) >= ahead) {
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
              w = 0;
              break;
            }
            __nanosleep(64);
          }
        }
        if (!__shfl_sync(0xffffffffu, w, 0)) {
          ok = false;
          break;
        }
      }
      const int sb = k % kSchedSlots;
      if (k >= kSchedSlots) {                 // the slot's previous unit has been issued
        int w = 1;
        if (lane == 0) w = mbar_wait(&sched_empty[sb], ((k / kSchedSlots) & 1) ^ 1);
        if (!__shfl_sync(0xffffffffu, w, 0) || ld_volatile(abort_flag)) {
          ok = false;
          break;
        }
      }
      int32_t* sl = slice + sb * slice_cap;
      // Writes this unit's slice (entries of `seq`'s table from jb0), checking ids.
      auto load_slice = [&](int seq, int jb0, int nb) {
        const int32_t* row = p.block_tables + static_cast<int64_t>(seq) * p.max_blocks_per_seq + jb0;
        for (int i = lane; i < nb; i += 32) {
          int32_t id = __ldg(row + i);
          if (id < 0 || id >= p.num_blocks) {
            flag_error(p.err, PKV_DEVERR_BLOCK_ID);
            id = 0;
          }
          sl[i] = id;
        }
      };
      UnitDesc d{-1, 0, 0, 0, 1};
      if (pend) {
        // the next run of the last group claim
        const int o = __ffs(pend) - 1;
        pend &= pend - 1;
        int e = o + 1;
        while (e < pgs && ((plink >> e) & 1u)) ++e;
        const int t_begin = ppart * p.partition_tokens;
        const int jb0 = t_begin / B;
        load_slice(pseq + o, jb0, (t_begin + p.partition_tokens - 1) / B - jb0 + 1);
        const int L = __shfl_sync(0xffffffffu, pLm, o);
        const int kvh = pkvs / p.subs;
        d = UnitDesc{pseq + o, kvh * p.group + (pkvs - kvh * p.subs) * p.heads_per_cta, ppart, L,
                     e - o};
        staged += p.partition_tokens / kTile;
      } else {
        while (true) {
          // the CTA's own index first (no round trip), then the shared counter
          int u = static_cast<int>(blockIdx.x);
          if (claimed) {
            if (lane == 0) u = static_cast<int>(gridDim.x) + atomicAdd(p.counter, 1);
            u = __shfl_sync(0xffffffffu, u, 0);
          }
          claimed = true;
          if (u >= total) break;
          int part, seq, kvs;
          int F = 0, gs = 1;
          bool member = false;
          if (compact && u >= whole_units * p.kv_slices) {
            // a partial last partition (its index follows from the length)
            const int w = u - whole_units * p.kv_slices;
            const int idx = w / p.kv_slices;
            kvs = w - idx * p.kv_slices;
            seq = porder[idx];
            part = -1;
          } else if (compact) {
            int lo = 0, hi = p.num_seqs;      // largest lo with pref[lo] * slices <= u
            while (hi - lo > 1) {
              const int mid = (lo + hi) >> 1;
              if (pref[mid] * p.kv_slices <= u) lo = mid; else hi = mid;
            }
            seq = lo;
            const int rem = u - pref[lo] * p.kv_slices;
            part = rem / p.kv_slices;
            kvs = rem - part * p.kv_slices;
            if (grouping) {
              const int gi = ginfo[seq];
              F = gi >> 4;
              gs = ((gi >> 1) & 7) + 1;
              member = gi & 1;
              if (member) part += F;
            }
          } else {
            part = u / per_part;
            const int rem = u - part * per_part;
            seq = rem / p.kv_slices;
            kvs = rem - seq * p.kv_slices;
          }
          int t_begin = part * p.partition_tokens;
          int need = t_begin + p.partition_tokens;    // end of a whole partition
          int jb0 = t_begin / B;
          const int kvh = kvs / p.subs;
          const int head0 = kvh * p.group + (kvs - kvh * p.subs) * p.heads_per_cta;
          if (!member && gs > 1 && part < F) {
            // Group claim: every member's partition is whole. One round of
            // loads: the members' lengths and table entries; the first run's
            // slice (the first member's entries) goes straight to the slot.
            const int nbw = (need - 1) / B - jb0 + 1;
            const int Lm = lane < gs ? __ldg(p.context_lens + seq + lane) : 0;
            unsigned same = 0xffffffffu;      // bit m: members m-1 and m name the same blocks
            for (int i = lane; i < nbw; i += 32) {
              int32_t id[kMaxRun];
#pragma unroll
              for (int m = 0; m < kMaxRun; ++m)
                id[m] = m < gs ? __ldg(p.block_tables +
                                       static_cast<int64_t>(seq + m) * p.max_blocks_per_seq + jb0 + i)
                               : -1;
              unsigned bits = 1u;
#pragma unroll
              for (int m = 1; m < kMaxRun; ++m) bits |= (id[m] == id[m - 1] ? 1u : 0u) << m;
              same &= bits;
              int32_t v = id[0];
              if (v < 0 || v >= p.num_blocks) {
                flag_error(p.err, PKV_DEVERR_BLOCK_ID);
                v = 0;
              }
              sl[i] = v;
            }
            same = __reduce_and_sync(0xffffffffu, same);
            const unsigned full =
                __ballot_sync(0xffffffffu, lane < gs && Lm >= need && Lm <= max_ctx);
            const unsigned link = same & full & (full << 1);
            int e = 1;
            while (e < gs && ((link >> e) & 1u)) ++e;
            // later runs start where the chain breaks
            pend = ~link & ((1u << gs) - 1u) & ~((1u << e) - 1u);
            plink = link;
            pseq = seq;
            ppart = part;
            pkvs = kvs;
            pLm = Lm;
            pgs = gs;
            d = UnitDesc{seq, head0, part, __shfl_sync(0xffffffffu, Lm, 0), e};
            staged += p.partition_tokens / kTile;
            break;
          }
          // A unit of one sequence.
          const int L = __ldg(p.context_lens + seq);
          if (L < 1 || L > max_ctx) {
            if (lane == 0 && part == 0 && kvs == 0) flag_error(p.err, PKV_DEVERR_CONTEXT);
            continue;
          }
          if (part < 0) {                     // the partial last partition
            part = L / p.partition_tokens;
            t_begin = part * p.partition_tokens;
            need = t_begin + p.partition_tokens;
            jb0 = t_begin / B;
          }
          if (t_begin >= L) continue;         // this sequence has no such partition
          const int t_end = min(L, need);
          load_slice(seq, jb0, (t_end - 1) / B - jb0 + 1);
          d = UnitDesc{seq, head0, part, L, 1};
          staged += (t_end - t_begin + kTile - 1) / kTile;
          break;
        }
      }
      if (lane == 0) sched[sb] = d;
      mbar_arrive(&sched_full[sb]);             // every lane: its slice entries are written
      if (d.seq < 0) break;
    }
    if (!ok && lane == 0) {
      flag_error(p.err, PKV_DEVERR_TIMEOUT);
      st_volatile(abort_flag, 1);
    }
    // No work is left to claim: the reduce kernel may be launched now (it
    // waits for this grid to finish).
    if (lane == 0) griddep_launch_dependents();
    return;
  }

  // ------------------------------------------------------------ copy warp
  // Publishes each staged unit to the consumers (its query rows by bulk copy)
  // and streams its K/V tiles through the ring. The lanes issue a tile's
  // copies (and a unit's query rows) together, each resolving its own block
  // id, so that issuing a tile costs a few dependent steps of the warp rather
  // than one thread's chain of every copy. Every lane waits on the barriers
  // itself (each then reads what the barrier published, or writes into the
  // space it freed); lane 0 makes the arrivals.
  if (warp == kConsumerWarps) {
    const uint64_t policy = l2_evict_first_policy();
    const uint32_t copy_bytes = static_cast<uint32_t>(p.box_rows) * Lay::kRowBytes;
    const int bshift = 31 - __clz(B);                 // block_size is a power of two
    if (lane == 0) {
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
    }
    int issued = 0;                           // tiles issued (ring position)
    int k = 0;                                // units published
    bool ok = true;
    while (true) {
      const int sb = k % kSchedSlots;
      if (!__all_sync(0xffffffffu, mbar_wait(&sched_full[sb], (k / kSchedSlots) & 1))) {
        ok = false;
        break;
      }
      const UnitDesc d = sched[sb];
      if (d.seq < 0) break;
      const int t_begin = d.part * p.partition_tokens;
      const int t_end = min(d.len, t_begin + p.partition_tokens);
      const int n_tiles = (t_end - t_begin + kTile - 1) / kTile;
      const int jb0 = t_begin >> bshift;
      const int kvh = d.head0 / p.group;
      const int32_t* sl = slice + sb * slice_cap;
      const int qb = 0;                       // one query buffer
      if (k >= 1 && !__all_sync(0xffffffffu, mbar_wait(&q_empty[qb], (k - 1) & 1))) {
        ok = false;
        break;
      }
      const uint32_t qbytes = static_cast<uint32_t>(p.heads_per_cta) * D * 2;
      if (lane == 0) {
        units[qb] = d;
        mbar_arrive_expect_tx(&q_full[qb], qbytes * d.nrun);
      }
      __syncwarp();
      if (lane < d.nrun)
        bulk_load(qbuf + qb * GS * D + lane * p.heads_per_cta * D,
                  p.q + (static_cast<int64_t>(d.seq + lane) * p.num_heads + d.head0) * D, qbytes,
                  &q_full[qb]);
      ++k;
      for (int i = 0; i < n_tiles; ++i, ++issued) {
        const int st = issued % kStages;
        if (issued >= kStages &&
            !__all_sync(0xffffffffu, mbar_wait(&empty_bar[st], ((issued / kStages) & 1) ^ 1))) {
          ok = false;
          break;
        }
        if (__shfl_sync(0xffffffffu, ld_volatile(abort_flag), 0)) {
          ok = false;
          break;
        }
        const int t0 = t_begin + i * kTile;
        const int valid = min(kTile, t_end - t0);
        const int copies = B >= kTile ? 1 : (valid + B - 1) >> bshift;
        uint8_t* kdst = ring + st * Lay::kStageBytes;
        if (lane == 0) mbar_arrive_expect_tx(&full_bar[st], 2u * copies * copy_bytes);
        __syncwarp();
        // copy j: K (j even) or V (j odd) of the tile's block j / 2
        for (int j = lane; j < 2 * copies; j += 32) {
          const int c = j >> 1;
          const int z = B >= kTile ? (sl[(t0 >> bshift) - jb0] << bshift) + (t0 & (B - 1))
                                   : sl[(t0 >> bshift) + c - jb0] << bshift;
          uint8_t* dst = kdst + (j & 1) * Lay::kTileBytes + c * copy_bytes;
          const CUtensorMap* map = (j & 1) ? &tm_v : &tm_k;
          if constexpr (kMma) {
            // 4-D view (64 elements, slot, head, D/64 lines): whole rows, swizzled
            tma_load_4d(dst, map, &full_bar[st], 0, z, kvh, 0, policy);
          } else {
            tma_load_3d(dst, map, &full_bar[st], 0, kvh, z, policy);
          }
        }
        if (lane == 0) st_volatile(issued_tiles, issued + 1);
      }
      if (!ok) break;
      __syncwarp();                           // every lane is done with the slice
      if (lane == 0) mbar_arrive(&sched_empty[sb]);
    }
    if (lane == 0) {
      // Publish the end of the work (or the abort) to the consumers.
      const int qb = 0;
      if (ok && k >= 1 && !mbar_wait(&q_empty[qb], (k - 1) & 1)) ok = false;
      if (!ok) {
        flag_error(p.err, PKV_DEVERR_TIMEOUT);
        st_volatile(abort_flag, 1);
      }
      units[qb].seq = ok ? -1 : -2;
      mbar_arrive(&q_full[qb]);
      if (!ok) {
        // Let the copies in flight (the last kStages tiles issued) land
        // before the CTA can retire.
        for (int g = max(0, issued - kStages); g < issued; ++g)
          mbar_wait(&full_bar[g % kStages], (g / kStages) & 1);
      }
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int grp = lane >> 3;                      // group within the warp
  const int gi = warp * 4 + grp;                  // group within the CTA (0..15)
  const int j = lane & 7;                         // lane within the group
  const int base = grp * 8;
  const unsigned gmask = 0xffu << base;
  const int heads = p.heads_per_cta;
  const int rows_shift = 31 - __clz(p.box_rows);  // rows per copy = 2^rows_shift
  using State = typename std::conditional<kMma, MmaState<D, T>, GroupState<D, GS, T>>::type;
  State gs;
  int consumed = 0;                               // tiles consumed (ring position)
  for (int k = 0;; ++k) {
    const int qb = 0;
    UnitDesc ud{-2, 0, 0, 0, 1};
    if (!ld_volatile(abort_flag) && mbar_wait(&q_full[qb], k & 1)) ud = units[qb];
    if (ud.seq == -1) break;                      // all work done
    if (ud.seq == -2) {                           // abort: nothing more is coming
      if (lane == 0) {
        flag_error(p.err, PKV_DEVERR_TIMEOUT);
        st_volatile(abort_flag, 1);
      }
      break;
    }
    const int rows = ud.nrun * heads;            // query rows of this unit
    if constexpr (kMma) {
      gs.begin(qbuf + qb * GS * D, rows, lane);
    } else {
      gs.begin(qbuf + qb * GS * D, j, p.q_scale);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&q_empty[qb]);

    const int t_begin = ud.part * p.partition_tokens;
    const int t_end = min(ud.len, t_begin + p.partition_tokens);
    const int n_tiles = (t_end - t_begin + kTile - 1) / kTile;
    for (int i = 0; i < n_tiles; ++i, ++consumed) {
      const int st = consumed % kStages;
      if (ld_volatile(abort_flag) || !mbar_wait(&full_bar[st], (consumed / kStages) & 1)) {
        if (lane == 0) st_volatile(abort_flag, 1);
        continue;                                 // keep the unit's control flow, skip work
      }
      const int valid = min(kTile, t_end - (t_begin + i * kTile));
      if constexpr (kMma) {
        const uint8_t* kt = ring + st * Lay::kStageBytes;
        if (warp * 8 < valid) {
          if (rows > 8)
            gs.template tile<true>(kt, kt + Lay::kTileBytes, warp * 8, valid, p.q_scale, lane,
                                   rows_shift);
          else
            gs.template tile<false>(kt, kt + Lay::kTileBytes, warp * 8, valid, p.q_scale, lane,
                                    rows_shift);
        }
      } else {
        const uint16_t* ks = reinterpret_cast<const uint16_t*>(ring + st * Lay::kStageBytes);
        const uint16_t* vs = ks + kTile * D;
#pragma unroll
        for (int r = 0; r < kTile / kGroups; ++r) {
          const int tk = gi + r * kGroups;
          if (tk < valid) gs.token(ks + tk * D, vs + tk * D, j, gmask, base);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[st]);
    }

    if constexpr (kMma) {
      // Tree merge of the four warps' states, fragment by fragment (every warp
      // holds the same rows and columns in the same registers): warps 2 and 3
      // hand theirs to warps 0 and 1 through two slots, warp 1 hands the sum
      // to warp 0 through its own slot, and warp 0 writes the unit's partials.
      using M = MmaState<D, T>;
      constexpr int kFrag4 = M::NT + 1;                 // float4s per lane: o, then (mA, mB, lA, lB)
      float4* xb = reinterpret_cast<float4*>(combine);  // [2][kFrag4][32]
      auto put = [&](float4* dst) {
#pragma unroll
        for (int jn = 0; jn < M::NT; ++jn)
          dst[jn * 32 + lane] = make_float4(gs.o[jn][0], gs.o[jn][1], gs.o[jn][2], gs.o[jn][3]);
        dst[M::NT * 32 + lane] = make_float4(gs.mA, gs.mB, gs.lA, gs.lB);
      };
      auto take = [&](const float4* src) {
        const float4 ml = src[M::NT * 32 + lane];
        const float MA = fmaxf(gs.mA, ml.x), MB = fmaxf(gs.mB, ml.y);
        const float fA = gs.mA == -INFINITY ? 0.f : ex2(gs.mA - MA);
        const float hA = ml.x == -INFINITY ? 0.f : ex2(ml.x - MA);
        const float fB = gs.mB == -INFINITY ? 0.f : ex2(gs.mB - MB);
        const float hB = ml.y == -INFINITY ? 0.f : ex2(ml.y - MB);
        gs.lA = fmaf(gs.lA, fA, ml.z * hA);
        gs.lB = fmaf(gs.lB, fB, ml.w * hB);
#pragma unroll
        for (int jn = 0; jn < M::NT; ++jn) {
          const float4 v = src[jn * 32 + lane];
          gs.o[jn][0] = fmaf(gs.o[jn][0], fA, v.x * hA);
          gs.o[jn][1] = fmaf(gs.o[jn][1], fA, v.y * hA);
          gs.o[jn][2] = fmaf(gs.o[jn][2], fB, v.z * hB);
          gs.o[jn][3] = fmaf(gs.o[jn][3], fB, v.w * hB);
        }
        gs.mA = MA;
        gs.mB = MB;
      };
      auto wait_or_abort = [&](uint64_t* bar, int parity) {
        if (!mbar_wait(bar, parity) && lane == 0) {
          flag_error(p.err, PKV_DEVERR_TIMEOUT);
          st_volatile(abort_flag, 1);
        }
      };
      if (warp >= 2) {
        if (k >= 1) wait_or_abort(x_free, (k - 1) & 1);    // both slots read by warp 0
        put(xb + (warp - 2) * kFrag4 * 32);
        __syncwarp();
        if (lane == 0) mbar_arrive(x_full);
      } else {
        wait_or_abort(x_full, k & 1);
        take(xb + warp * kFrag4 * 32);
        if (warp == 1) {
          put(xb + kFrag4 * 32);                  // each lane rewrites only what it read
          __syncwarp();
          if (lane == 0) mbar_arrive(y_full);
        } else {
          wait_or_abort(y_full, k & 1);
          take(xb + kFrag4 * 32);
          __syncwarp();
          if (lane == 0) mbar_arrive(x_free);
          const int g = lane >> 2, t = lane & 3;
          float lsA = gs.lA, lsB = gs.lB;
          lsA += __shfl_xor_sync(0xffffffffu, lsA, 1);
          lsA += __shfl_xor_sync(0xffffffffu, lsA, 2);
          lsB += __shfl_xor_sync(0xffffffffu, lsB, 1);
          lsB += __shfl_xor_sync(0xffffffffu, lsB, 2);
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int rw = g + 8 * half;          // sequence rw / heads of the run, head rw % heads
            if (rw < rows) {
              const int64_t row = ((static_cast<int64_t>(ud.seq) + rw / heads) * p.num_heads +
                                   ud.head0 + rw % heads) * p.max_parts + ud.part;
              float2* dst = reinterpret_cast<float2*>(p.part_acc + row * D);
#pragma unroll
              for (int jn = 0; jn < M::NT; ++jn)
                dst[4 * jn + t] = make_float2(gs.o[jn][2 * half], gs.o[jn][2 * half + 1]);
              if (t == 0) p.part_ml[row] = make_float2(half ? gs.mB : gs.mA, half ? lsB : lsA);
            }
          }
        }
      }
    } else {
      // Merge this warp's partial into shared memory (one row of D + 2 floats
      // per head: m, l, acc), then the four warps' rows into the unit's partial.
      // A wait that gives up flags the timeout and aborts the kernel; the merge
      // is then skipped (its shared rows may still be in use).
      auto merge_wait = [&](uint64_t* bar, int parity) {
        const bool w = __all_sync(0xffffffffu, mbar_wait(bar, parity));
        if (!w && lane == 0) {
          flag_error(p.err, PKV_DEVERR_TIMEOUT);
          st_volatile(abort_flag, 1);
        }
        return w;
      };
      const bool free_ok = k < 1 || merge_wait(&merge_bar[1], (k - 1) & 1);  // previous partials read
      // Lanes j, j+8, j+16, j+24 hold the same elements: merge the groups first.
#pragma unroll
      for (int g = 0; g < GS; ++g) {
        const float mg = gs.head_m(g, base);
        const float lg = gs.head_l(g, base);
        float mx = fmaxf(mg, __shfl_xor_sync(0xffffffffu, mg, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float f = (mx == -INFINITY) ? 0.f : ex2(mg - mx);
        float ls = lg * f;
        ls += __shfl_xor_sync(0xffffffffu, ls, 8);
        ls += __shfl_xor_sync(0xffffffffu, ls, 16);
        float* cw = combine + (warp * GS + g) * (D + 2);
#pragma unroll
        for (int e = 0; e < Lay::kE / 2; ++e) {
          float a, b;
          gs.head_acc(g, e, a, b);
          a *= f;
          b *= f;
          a += __shfl_xor_sync(0xffffffffu, a, 8);
          b += __shfl_xor_sync(0xffffffffu, b, 8);
          a += __shfl_xor_sync(0xffffffffu, a, 16);
          b += __shfl_xor_sync(0xffffffffu, b, 16);
          if (grp == 0 && free_ok) {
            const int el = (e / 4) * 64 + 8 * j + 2 * (e % 4);
            cw[2 + el] = a;
            cw[2 + el + 1] = b;
          }
        }
        if (grp == 0 && j == 0 && free_ok) {
          cw[0] = mx;
          cw[1] = ls;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&merge_bar[0]);
      const bool full_ok = merge_wait(&merge_bar[0], k & 1);

      for (int idx = threadIdx.x; free_ok && full_ok && idx < heads * D;
           idx += kConsumerWarps * 32) {
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
        const int64_t row =
            (static_cast<int64_t>(ud.seq) * p.num_heads + ud.head0 + g) * p.max_parts + ud.part;
        p.part_acc[row * D + e] = a;
        if (e == 0) p.part_ml[row] = make_float2(M, lsum);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&merge_bar[1]);
    }
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

// kWarps warps per row (1 for short contexts: four rows per CTA; 4 for long
// ones: the partitions of a row are split round-robin over the warps and the
// warps' sums are added in a fixed order). The order of the additions
// depends only on kWarps and the number of partitions.
template <int D, typename O, int kWarps>
__global__ void __launch_bounds__(128) decode_reduce_kernel(O* out, const ReduceParams p) {
  constexpr int PER = D / 32;                   // output elements per lane
  constexpr int kBatch = 4;                     // partitions whose loads a warp issues together
  __shared__ float part_o[kWarps][PER][32];
  __shared__ float part_z[kWarps];
  __shared__ float part_m[kWarps];
  // Launched as a programmatic dependent of the partition kernel: nothing is
  // read before that grid has completed.
  griddep_wait();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int wr = warp % kWarps;                 // warp within the row
  const int w = blockIdx.x * (4 / kWarps) + warp / kWarps;   // row: (sequence, query head)
  if (w >= p.num_seqs * p.num_heads) return;    // whole rows only: uniform across a row's warps
  const int seq = w / p.num_heads;
  O* dst = out + static_cast<int64_t>(w) * D + lane * PER;
  const int L = __ldg(p.context_lens + seq);
  if (L < 1 || L > p.max_context) {
    if (wr == 0) {
#pragma unroll
      for (int k = 0; k < PER; ++k) store_out<O>(dst + k, 0.f);
    }
    return;
  }
  const int np = (L + p.partition_tokens - 1) / p.partition_tokens;
  const int64_t row0 = static_cast<int64_t>(w) * p.max_parts;
  float M = -INFINITY;
  for (int i = wr * 32 + lane; i < np; i += kWarps * 32) M = fmaxf(M, p.part_ml[row0 + i].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if constexpr (kWarps > 1) {
    if (lane == 0) part_m[wr] = M;
    __syncthreads();
    M = part_m[0];
#pragma unroll
    for (int j = 1; j < kWarps; ++j) M = fmaxf(M, part_m[j]);
  }
  // This warp takes partitions wr, wr + kWarps, ... in order, kBatch of them
  // with their loads in flight together.
  float acc[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) acc[k] = 0.f;
  float Z = 0.f;
  for (int i0 = wr; i0 < np; i0 += kWarps * kBatch) {
    float2 ml[kBatch];
    float v[kBatch][PER];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int i = i0 + b * kWarps;
      ml[b] = i < np ? p.part_ml[row0 + i] : make_float2(-INFINITY, 0.f);
      const float* src = p.part_acc + (row0 + (i < np ? i : 0)) * D + lane * PER;
      if constexpr (PER == 4) {
        const float4 x = *reinterpret_cast<const float4*>(src);
        v[b][0] = x.x;
        v[b][1] = x.y;
        v[b][2] = x.z;
        v[b][3] = x.w;
      } else {
#pragma unroll
        for (int k = 0; k < PER; ++k) v[b][k] = src[k];
      }
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      if (i0 + b * kWarps < np) {
        const float wgt = ex2(ml[b].x - M);
        Z = fmaf(ml[b].y, wgt, Z);
#pragma unroll
        for (int k = 0; k < PER; ++k) acc[k] = fmaf(v[b][k], wgt, acc[k]);
      }
    }
  }
  if constexpr (kWarps == 1) {
#pragma unroll
    for (int k = 0; k < PER; ++k) store_out<O>(dst + k, acc[k] / Z);
  } else {
    if (lane == 0) part_z[wr] = Z;
#pragma unroll
    for (int k = 0; k < PER; ++k) part_o[wr][k][lane] = acc[k];
    __syncthreads();
    if (wr == 0) {
      float Zt = part_z[0];
#pragma unroll
      for (int j = 1; j < kWarps; ++j) Zt += part_z[j];
#pragma unroll
      for (int k = 0; k < PER; ++k) {
        float o = part_o[0][k][lane];
#pragma unroll
        for (int j = 1; j < kWarps; ++j) o += part_o[j][k][lane];
        store_out<O>(dst + k, o / Zt);
      }
    }
  }
}

// ---------------------------------------------------------------- host side

// Largest divisor of n that is at most cap.
static int largest_divisor_upto(int n, int cap) {
  for (int d = std::min(n, cap); d > 1; --d)
    if (n % d == 0) return d;
  return 1;
}

// Query heads per CTA on the packed-pair path: 4, 2 or 1, the largest that divides the group.
static int pick_group_slice(int group) {
  if (group % 4 == 0) return 4;
  if (group % 2 == 0) return 2;
  return 1;
}

template <int D, int GS, typename T, bool kMma>
static cudaError_t launch_partition(const CUtensorMap& tk, const CUtensorMap& tv,
                                    const DecodeParams& p, cudaStream_t stream) {
  auto kern = decode_partition_kernel<D, GS, T, kMma>;
  const int slice = p.partition_tokens / p.block_size + 2;
  const int smem = DecodeLayout<D, GS, kMma>::smem_bytes(slice);
  // attribute and occupancy: once per device and shared-memory size
  int per_sm = 0, sms = 0;
  cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), kThreads, smem, &per_sm);
  if (e != cudaSuccess) return e;
  e = device_sm_count(&sms);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const int grid = static_cast<int>(std::min<int64_t>(p.total_units,
                                                      static_cast<int64_t>(sms) * per_sm));
  e = cudaMemsetAsync(p.counter, 0, sizeof(int), stream);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, stream>>>(tk, tv, p);
  return cudaGetLastError();
}

template <int D, typename T>
static cudaError_t dispatch_gs(bool mma, int gs, const CUtensorMap& tk, const CUtensorMap& tv,
                               const DecodeParams& p, cudaStream_t s) {
  if (mma) return launch_partition<D, kMmaRows, T, true>(tk, tv, p, s);
  switch (gs) {
    case 1: return launch_partition<D, 1, T, false>(tk, tv, p, s);
    case 2: return launch_partition<D, 2, T, false>(tk, tv, p, s);
    default: return launch_partition<D, 4, T, false>(tk, tv, p, s);
  }
}

template <int D, int W>
static cudaError_t launch_reduce_as(void* out, int out_dtype, const ReduceParams& rp,
                                    cudaLaunchConfig_t& cfg) {
  switch (out_dtype) {
    case PKV_F32:
      return cudaLaunchKernelEx(&cfg, decode_reduce_kernel<D, float, W>, static_cast<float*>(out),
                                rp);
    case PKV_F16:
      return cudaLaunchKernelEx(&cfg, decode_reduce_kernel<D, __half, W>,
                                static_cast<__half*>(out), rp);
    default:
      return cudaLaunchKernelEx(&cfg, decode_reduce_kernel<D, __nv_bfloat16, W>,
                                static_cast<__nv_bfloat16*>(out), rp);
  }
}

template <int D>
static cudaError_t launch_reduce(void* out, int out_dtype, const ReduceParams& rp,
                                 cudaStream_t s) {
  const int rows = rp.num_seqs * rp.num_heads;
  // Programmatic dependent launch: the reduce grid is set up while the
  // partition grid drains and waits on it with griddepcontrol.wait.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(rows);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // four warps per row once rows have many partitions
  if (rp.max_parts > 16) return launch_reduce_as<D, 4>(out, out_dtype, rp, cfg);
  cfg.gridDim = dim3((rows + 3) / 4);
  return launch_reduce_as<D, 1>(out, out_dtype, rp, cfg);
}

}  // namespace pkv

using namespace pkv;

// The partition size a call uses. 0 picks 1024 tokens on the tensor paths
// when the batch has enough (sequence, KV head, 1024-token partition) units to
// keep every SM busy: kBigPartitionUnits on the warp-level path (query groups
// of 2 to 16 heads; two CTAs per SM), kBigPartitionUnitsTc on the tcgen05 path
// (groups of 32 or more; one CTA per SM). Each unit then carries twice the keys
// for one merge, one partial and one claim. Measured, fraction of the HBM copy
// rate: 0.82 against 0.80 on the 256-beam shared-prefix batch, 0.99 against
// 0.95 on the long-context one, 0.42 against 0.38 with 64 query heads on one KV
// head. On the tcgen05 path 2048 when even 2048-token units are that many
// (and a partition's blocks fit its id buffer): 0.44 against 0.42 with 64
// query heads on one KV head, back to back. Otherwise 512, or 1024 when the
// tables can hold 32K tokens or more.
constexpr int64_t kBigPartitionUnits = 1024;
constexpr int64_t kBigPartitionUnitsTc = 256;
static int effective_partition(int partition_tokens, int num_seqs, int num_heads,
                               int num_kv_heads, int head_size, int max_blocks_per_seq,
                               int block_size) {
  if (partition_tokens != 0) return partition_tokens;
  const int64_t max_ctx = static_cast<int64_t>(max_blocks_per_seq) * block_size;
  const int group = num_kv_heads >= 1 ? num_heads / num_kv_heads : 1;
  const int64_t units = static_cast<int64_t>(num_seqs) * num_kv_heads * ((max_ctx + 1023) / 1024);
  if (group >= 2 && decode_tc_supported(group, head_size, block_size, 1024)) {
    const int64_t units2 = static_cast<int64_t>(num_seqs) * num_kv_heads * ((max_ctx + 2047) / 2048);
    if (units2 >= kBigPartitionUnitsTc && decode_tc_supported(group, head_size, block_size, 2048))
      return 2048;
    return units >= kBigPartitionUnitsTc ? 1024 : (max_ctx >= 32768 ? 1024 : 512);
  }
  const bool warp_tensor = group >= 2 && block_size >= 8 &&
                           !decode_tc_supported(group, head_size, block_size, 512);
  if (warp_tensor && units >= kBigPartitionUnits) return 1024;
  return max_ctx >= 32768 ? 1024 : 512;
}

extern "C" int pkv_decode_partition_tokens(int num_seqs, int num_heads, int num_kv_heads,
                                           int head_size, int max_blocks_per_seq, int block_size,
                                           int partition_tokens) {
  return effective_partition(partition_tokens, num_seqs, num_heads, num_kv_heads, head_size,
                             max_blocks_per_seq, block_size);
}

// A 32-token tile is a whole number of blocks, or a whole number of tiles is a block.
static bool block_size_ok(int b) { return b >= 1 && b <= 256 && (b & (b - 1)) == 0; }

extern "C" size_t pkv_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads,
                                            int head_size, int max_blocks_per_seq, int block_size,
                                            int partition_tokens) {
  if (num_seqs < 0 || num_heads < 1 || num_kv_heads < 1 || head_size < 1 ||
      max_blocks_per_seq < 1 || block_size < 1)
    return 0;
  const int pt = effective_partition(partition_tokens, num_seqs, num_heads, num_kv_heads,
                                     head_size, max_blocks_per_seq, block_size);
  if (pt < 1) return 0;
  const int64_t parts = (static_cast<int64_t>(max_blocks_per_seq) * block_size + pt - 1) / pt;
  const int64_t rows = static_cast<int64_t>(num_seqs) * num_heads * parts;
  // partial accumulators, (m, l) pairs, then the work counter (16-byte aligned)
  return static_cast<size_t>(rows * head_size * 4 + ((rows * 8 + 15) / 16) * 16 + 16);
}

// The decode call. wait_ns limits every pipeline wait of the tensor-memory
// path and stall_unit (>= 0) makes its softmax warps wait out that unit; both
// exist for pkv_test_decode_wait_timeout, whose call must take that path
// (tc_only).
static pkv_status decode_impl(void* out, int out_dtype, const void* q, const void* k_cache,
                              const void* v_cache, int kv_dtype, const int32_t* block_tables,
                              const int32_t* context_lens, int num_seqs, int num_heads,
                              int num_kv_heads, int head_size, int num_blocks, int block_size,
                              int max_blocks_per_seq, float scale, int partition_tokens,
                              void* workspace, size_t workspace_bytes, int32_t* err_flag,
                              void* stream, uint64_t wait_ns, int stall_unit, bool tc_only) {
  if (num_seqs < 0 || num_seqs > 65535) return PKV_EINVAL;
  if (num_kv_heads < 1) return PKV_EINVAL;
  const int pt = effective_partition(partition_tokens, num_seqs, num_heads, num_kv_heads,
                                     head_size, max_blocks_per_seq, block_size);
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
  const size_t need = pkv_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_size,
                                                max_blocks_per_seq, block_size, pt);
  if (workspace_bytes < need) return PKV_EWORKSPACE;

  const int group = num_heads / num_kv_heads;
  const int64_t rows_all = static_cast<int64_t>(num_seqs) * num_heads * parts;
  float* part_acc = static_cast<float*>(workspace);
  float2* part_ml = reinterpret_cast<float2*>(part_acc + rows_all * head_size);
  int* counter = reinterpret_cast<int*>(static_cast<char*>(workspace) + rows_all * head_size * 4 +
                                        ((rows_all * 8 + 15) / 16) * 16);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ReduceParams rp{};
  rp.part_acc = part_acc;
  rp.part_ml = part_ml;
  rp.context_lens = context_lens;
  rp.num_seqs = num_seqs;
  rp.num_heads = num_heads;
  rp.max_parts = static_cast<int>(parts);
  rp.partition_tokens = pt;
  rp.max_context = static_cast<int>(max_ctx);
  if (decode_tc_supported(group, head_size, block_size, pt)) {
    // Large groups: all G heads of a KV head in one tensor-memory product.
    if (parts * num_seqs * num_kv_heads > INT32_MAX / 2) return PKV_EINVAL;
    DecodeTcArgs a{};
    a.part_acc = part_acc;
    a.part_ml = part_ml;
    a.counter = counter;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.err = err_flag;
    a.num_seqs = num_seqs;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_size = head_size;
    a.num_blocks = num_blocks;
    a.block_size = block_size;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.partition_tokens = pt;
    a.max_parts = static_cast<int>(parts);
    a.bf16 = kv_dtype == PKV_BF16;
    a.q_scale = scale * kLog2e;
    a.wait_ns = wait_ns;
    a.stall_unit = stall_unit;
    if (launch_decode_tc(a, st) != cudaSuccess) return PKV_ECUDA;
    const cudaError_t er = head_size == 128 ? launch_reduce<128>(out, out_dtype, rp, st)
                                            : launch_reduce<64>(out, out_dtype, rp, st);
    return er == cudaSuccess ? PKV_OK : PKV_ECUDA;
  }

  if (tc_only) return PKV_EINVAL;

  // Grouped query heads go to the warp-level tensor path when every TMA copy
  // lands on a 1 KB boundary of a tile half (block_size >= 8), else to the
  // packed-pair path.
  const bool mma = group >= 2 && block_size >= 8;
  const int box_rows = std::min(block_size, kTile);
  CUtensorMap tk, tv;
  const int64_t slots = static_cast<int64_t>(num_blocks) * block_size;
  const CacheView view = mma ? kRowsSwizzled : kRowsPlain;
  if (!encode_cache_map(&tk, k_cache, head_size, num_kv_heads, slots, box_rows, view) ||
      !encode_cache_map(&tv, v_cache, head_size, num_kv_heads, slots, box_rows, view))
    return PKV_ECUDA;

  const int64_t rows = static_cast<int64_t>(num_seqs) * num_heads * parts;
  const int gs = (num_heads / num_kv_heads >= 2 && block_size >= 8)
                     ? largest_divisor_upto(num_heads / num_kv_heads, kMmaHeads)
                     : pick_group_slice(num_heads / num_kv_heads);
  const int64_t kv_slices = static_cast<int64_t>(num_kv_heads) * (num_heads / num_kv_heads / gs);
  const int64_t total_units = parts * num_seqs * kv_slices;
  if (total_units > INT32_MAX / 2) return PKV_EINVAL;
  DecodeParams p{};
  p.part_acc = static_cast<float*>(workspace);
  p.part_ml = reinterpret_cast<float2*>(static_cast<float*>(workspace) + rows * head_size);
  p.counter = reinterpret_cast<int*>(static_cast<char*>(workspace) + rows * head_size * 4 +
                                     ((rows * 8 + 15) / 16) * 16);
  p.num_seqs = num_seqs;
  p.subs = num_heads / num_kv_heads / gs;
  p.heads_per_cta = gs;
  p.kv_slices = static_cast<int>(kv_slices);
  p.total_units = static_cast<int>(total_units);
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
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  cudaError_t e;
  if (head_size == 128) {
    e = kv_dtype == PKV_F16 ? dispatch_gs<128, F16>(mma, gs, tk, tv, p, s)
                            : dispatch_gs<128, BF16>(mma, gs, tk, tv, p, s);
  } else {
    e = kv_dtype == PKV_F16 ? dispatch_gs<64, F16>(mma, gs, tk, tv, p, s)
                            : dispatch_gs<64, BF16>(mma, gs, tk, tv, p, s);
  }
  if (e != cudaSuccess) return PKV_ECUDA;

  e = head_size == 128 ? launch_reduce<128>(out, out_dtype, rp, s)
                       : launch_reduce<64>(out, out_dtype, rp, s);
  return e == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

extern "C" pkv_status pkv_paged_attention_decode(
    void* out, int out_dtype, const void* q, const void* k_cache, const void* v_cache,
    int kv_dtype, const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
    int num_heads, int num_kv_heads, int head_size, int num_blocks, int block_size,
    int max_blocks_per_seq, float scale, int partition_tokens, void* workspace,
    size_t workspace_bytes, int32_t* err_flag, void* stream) {
  return decode_impl(out, out_dtype, q, k_cache, v_cache, kv_dtype, block_tables, context_lens,
                     num_seqs, num_heads, num_kv_heads, head_size, num_blocks, block_size,
                     max_blocks_per_seq, scale, partition_tokens, workspace, workspace_bytes,
                     err_flag, stream, kWaitLimitNs, -1, false);
}

extern "C" pkv_status pkv_test_decode_wait_timeout(
    void* out, int out_dtype, const void* q, const void* k_cache, const void* v_cache,
    int kv_dtype, const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
    int num_heads, int num_kv_heads, int head_size, int num_blocks, int block_size,
    int max_blocks_per_seq, float scale, int partition_tokens, void* workspace,
    size_t workspace_bytes, int32_t* err_flag, uint64_t wait_limit_ns, void* stream) {
  if (err_flag == nullptr || wait_limit_ns < 1000 || wait_limit_ns > kWaitLimitNs)
    return PKV_EINVAL;
  return decode_impl(out, out_dtype, q, k_cache, v_cache, kv_dtype, block_tables, context_lens,
                     num_seqs, num_heads, num_kv_heads, head_size, num_blocks, block_size,
                     max_blocks_per_seq, scale, partition_tokens, workspace, workspace_bytes,
                     err_flag, stream, wait_limit_ns, 0, true);
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
unsigned long long g_noalloc_ctx[kMaxDevices] = {};   // context the address belongs to
}  // namespace

// Device address of g_noalloc_scratch on the current device. Host code only
// sees a host-side stand-in under the array's name, so the address is looked
// up with the device current, once per device, and remembered together with
// the unique id of the context it was found in: after a cudaDeviceReset the
// device runs a new context (with the library's image loaded anew), whose
// first call looks the address up again instead of using a stale one.
static pkv_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ECUDA;
  unsigned long long ctx_id = 0;
  if (!current_context_id(&ctx_id)) return PKV_ECUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr || ctx_id == 0 || g_noalloc_ctx[dev] != ctx_id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return PKV_ECUDA;
    // the lookup makes the device's context current if none was
    if (ctx_id == 0 && !current_context_id(&ctx_id)) return PKV_ECUDA;
    g_noalloc_ptr[dev] = p;
    g_noalloc_ctx[dev] = ctx_id;
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
  const size_t need = pkv_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_size,
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
