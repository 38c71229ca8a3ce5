// Host block manager of the paged KV cache: free list, reference counts, fork,
// append with copy-on-write.
//
// Rules (see include/pagedkv.h for the sources): the free list starts as the
// caller's permutation (or 0..N-1) and hands blocks out from its end; a
// request fails with no side effect when too few blocks are free; a fork
// shares every block; a block returns to the list only when its count reaches
// zero; appending into a partly filled tail that another sequence still
// references first moves this sequence onto a fresh copy ("079｜vLLM 与
// PagedAttention", wq-win.github.io, §2 "共享与写时复制" and §3's algorithm box).

#include <algorithm>
#include <cstdint>
#include <list>
#include <unordered_map>
#include <vector>

#include "pagedkv.h"

namespace {

struct Sequence {
  std::vector<int32_t> table;  // logical block j -> physical block id
  int64_t len = 0;             // tokens stored
};

}  // namespace

struct pkv_bm {
  int num_blocks = 0;
  int block_size = 0;
  std::vector<int32_t> free_list;  // top of the stack is the back
  std::vector<int32_t> ref;
  std::unordered_map<int64_t, Sequence> seqs;
  // Prefix cache: registered full prompt blocks by chained hash. A registered
  // block whose count reaches zero keeps its contents and waits, oldest first,
  // in `evictable` until a fresh allocation finds the free list empty.
  std::unordered_map<uint64_t, int32_t> cached;
  std::unordered_map<int32_t, uint64_t> hash_of;
  std::list<int32_t> evictable;
  std::unordered_map<int32_t, std::list<int32_t>::iterator> evict_pos;

  int64_t blocks_for(int64_t tokens) const { return (tokens + block_size - 1) / block_size; }
  int64_t available() const {
    return static_cast<int64_t>(free_list.size() + evictable.size());
  }

  // A fresh block with count 1: from the free list, else the least recently
  // freed cached block (which leaves the cache).
  int32_t pop() {
    int32_t b;
    if (!free_list.empty()) {
      b = free_list.back();
      free_list.pop_back();
    } else {
      b = evictable.front();
      evictable.pop_front();
      evict_pos.erase(b);
      cached.erase(hash_of[b]);
      hash_of.erase(b);
    }
    ref[b] = 1;
    return b;
  }

  void release(int32_t b) {  // count reached zero
    if (hash_of.count(b)) {
      evictable.push_back(b);
      evict_pos[b] = std::prev(evictable.end());
    } else {
      free_list.push_back(b);
    }
  }
};

// 64-bit FNV-1a (offset basis 14695981039346656037, prime 1099511628211).
static uint64_t fnv1a64(const uint8_t* data, size_t n, uint64_t h) {
  for (size_t i = 0; i < n; ++i) {
    h ^= data[i];
    h *= 1099511628211ull;
  }
  return h;
}

// Chained hash of one full block: FNV-1a over the previous block's hash (8
// bytes, little-endian) and the block's token ids (4 bytes each, little-endian).
static uint64_t block_hash(uint64_t prev, const int32_t* tokens, int block_size) {
  uint8_t buf[8];
  for (int i = 0; i < 8; ++i) buf[i] = static_cast<uint8_t>(prev >> (8 * i));
  uint64_t h = fnv1a64(buf, 8, 14695981039346656037ull);
  for (int t = 0; t < block_size; ++t) {
    const uint32_t v = static_cast<uint32_t>(tokens[t]);
    uint8_t w[4] = {static_cast<uint8_t>(v), static_cast<uint8_t>(v >> 8),
                    static_cast<uint8_t>(v >> 16), static_cast<uint8_t>(v >> 24)};
    h = fnv1a64(w, 4, h);
  }
  return h;
}

extern "C" {

pkv_bm* pkv_bm_create(int num_blocks, int block_size, const int32_t* free_order) {
  if (num_blocks < 1 || block_size < 1) return nullptr;
  pkv_bm* bm = new pkv_bm;
  bm->num_blocks = num_blocks;
  bm->block_size = block_size;
  bm->ref.assign(num_blocks, 0);
  bm->free_list.resize(num_blocks);
  if (free_order == nullptr) {
    for (int i = 0; i < num_blocks; ++i) bm->free_list[i] = i;
  } else {
    std::vector<char> seen(num_blocks, 0);
    for (int i = 0; i < num_blocks; ++i) {
      int32_t b = free_order[i];
      if (b < 0 || b >= num_blocks || seen[b]) {
        delete bm;
        return nullptr;
      }
      seen[b] = 1;
      bm->free_list[i] = b;
    }
  }
  return bm;
}

void pkv_bm_destroy(pkv_bm* bm) { delete bm; }

pkv_status pkv_bm_allocate(pkv_bm* bm, int64_t seq, int64_t num_tokens) {
  if (bm == nullptr || num_tokens < 0) return PKV_EINVAL;
  if (bm->seqs.count(seq)) return PKV_ESTATE;
  int64_t need = bm->blocks_for(num_tokens);
  if (need > bm->available()) return PKV_ENOMEM;
  Sequence s;
  s.len = num_tokens;
  s.table.reserve(need);
  for (int64_t i = 0; i < need; ++i) s.table.push_back(bm->pop());
  bm->seqs.emplace(seq, std::move(s));
  return PKV_OK;
}

pkv_status pkv_bm_fork(pkv_bm* bm, int64_t parent, int64_t child) {
  if (bm == nullptr) return PKV_EINVAL;
  auto it = bm->seqs.find(parent);
  if (it == bm->seqs.end() || bm->seqs.count(child)) return PKV_ESTATE;
  Sequence c = it->second;
  for (int32_t b : c.table) bm->ref[b] += 1;
  bm->seqs.emplace(child, std::move(c));
  return PKV_OK;
}

// One append; the caller has checked that a free block exists when needed.
static void append_one(pkv_bm* bm, Sequence& s, int64_t* slot, int32_t* src, int32_t* dst) {
  const int64_t B = bm->block_size;
  const int64_t L = s.len;
  *src = -1;
  *dst = -1;
  if (L % B == 0) {
    s.table.push_back(bm->pop());
  } else {
    int32_t& tail = s.table[L / B];
    if (bm->ref[tail] > 1) {
      int32_t fresh = bm->pop();
      bm->ref[tail] -= 1;
      *src = tail;
      *dst = fresh;
      tail = fresh;
    }
  }
  *slot = static_cast<int64_t>(s.table[L / B]) * B + L % B;
  s.len = L + 1;
}

static bool append_needs_block(const pkv_bm* bm, const Sequence& s) {
  const int64_t L = s.len;
  if (L % bm->block_size == 0) return true;
  return bm->ref[s.table[L / bm->block_size]] > 1;
}

pkv_status pkv_bm_append_slot(pkv_bm* bm, int64_t seq, int64_t* slot, int32_t* cow_src,
                              int32_t* cow_dst) {
  if (bm == nullptr || slot == nullptr || cow_src == nullptr || cow_dst == nullptr)
    return PKV_EINVAL;
  auto it = bm->seqs.find(seq);
  if (it == bm->seqs.end()) return PKV_ESTATE;
  if (append_needs_block(bm, it->second) && bm->available() == 0) return PKV_ENOMEM;
  append_one(bm, it->second, slot, cow_src, cow_dst);
  return PKV_OK;
}

pkv_status pkv_bm_append_slots(pkv_bm* bm, const int64_t* seqs, int n, int64_t* slots,
                               int32_t* cow_pairs, int* num_cow) {
  if (bm == nullptr || n < 0 || (n > 0 && (seqs == nullptr || slots == nullptr ||
                                           cow_pairs == nullptr)))
    return PKV_EINVAL;
  // Dry run: count the blocks the batch takes, following the same order, so
  // that a shortage is reported before anything changes.
  std::unordered_map<int64_t, int64_t> len;       // simulated lengths
  std::unordered_map<int32_t, int32_t> dropped;   // simulated count decrements
  std::unordered_map<int64_t, bool> moved_tail;   // seq now sits on a fresh tail
  int64_t need = 0;
  const int64_t B = bm->block_size;
  for (int i = 0; i < n; ++i) {
    auto it = bm->seqs.find(seqs[i]);
    if (it == bm->seqs.end()) return PKV_ESTATE;
    const Sequence& s = it->second;
    auto li = len.find(seqs[i]);
    int64_t L = li == len.end() ? s.len : li->second;
    if (L % B == 0) {
      ++need;
      moved_tail[seqs[i]] = true;  // a new private tail block
    } else if (!moved_tail[seqs[i]]) {
      int32_t tail = s.table[L / B];
      if (bm->ref[tail] - dropped[tail] > 1) {
        ++need;
        dropped[tail] += 1;
        moved_tail[seqs[i]] = true;
      }
    }
    len[seqs[i]] = L + 1;
  }
  if (need > bm->available()) return PKV_ENOMEM;
  int k = 0;
  for (int i = 0; i < n; ++i) {
    int32_t src, dst;
    append_one(bm, bm->seqs[seqs[i]], &slots[i], &src, &dst);
    if (src >= 0) {
      cow_pairs[2 * k] = src;
      cow_pairs[2 * k + 1] = dst;
      ++k;
    }
  }
  if (num_cow) *num_cow = k;
  return PKV_OK;
}

pkv_status pkv_bm_free(pkv_bm* bm, int64_t seq) {
  if (bm == nullptr) return PKV_EINVAL;
  auto it = bm->seqs.find(seq);
  if (it == bm->seqs.end()) return PKV_ESTATE;
  for (int32_t b : it->second.table)
    if (bm->ref[b] < 1) return PKV_ESTATE;  // would underflow; leave state as is
  for (int32_t b : it->second.table) {
    bm->ref[b] -= 1;
    if (bm->ref[b] == 0) bm->release(b);
  }
  bm->seqs.erase(it);
  return PKV_OK;
}

pkv_status pkv_bm_allocate_prefix(pkv_bm* bm, int64_t seq, const int32_t* token_ids, int64_t n,
                                  int64_t* cached_tokens) {
  if (bm == nullptr || n < 0 || (n > 0 && token_ids == nullptr)) return PKV_EINVAL;
  if (bm->seqs.count(seq)) return PKV_ESTATE;
  const int B = bm->block_size;
  const int64_t full = n / B;
  std::vector<uint64_t> hashes(full);
  uint64_t prev = 0;
  for (int64_t j = 0; j < full; ++j) prev = hashes[j] = block_hash(prev, token_ids + j * B, B);
  std::vector<int32_t> hits;
  for (int64_t j = 0; j < full; ++j) {
    auto c = bm->cached.find(hashes[j]);
    if (c == bm->cached.end()) break;       // a later block needs every block before it
    hits.push_back(c->second);
  }
  int64_t revived = 0;
  for (int32_t b : hits) revived += bm->ref[b] == 0;
  const int64_t fresh = bm->blocks_for(n) - static_cast<int64_t>(hits.size());
  if (fresh > bm->available() - revived) return PKV_ENOMEM;
  for (int32_t b : hits) {
    if (bm->ref[b] == 0) {
      bm->evictable.erase(bm->evict_pos[b]);
      bm->evict_pos.erase(b);
    }
    bm->ref[b] += 1;
  }
  Sequence s;
  s.len = n;
  s.table = hits;
  for (int64_t j = static_cast<int64_t>(hits.size()); j < bm->blocks_for(n); ++j) {
    const int32_t b = bm->pop();
    if (j < full) {                          // full prompt block: registered for later hits
      bm->cached[hashes[j]] = b;
      bm->hash_of[b] = hashes[j];
    }
    s.table.push_back(b);
  }
  bm->seqs.emplace(seq, std::move(s));
  if (cached_tokens) *cached_tokens = static_cast<int64_t>(hits.size()) * B;
  return PKV_OK;
}

int pkv_bm_num_cached(const pkv_bm* bm) {
  return bm ? static_cast<int>(bm->cached.size()) : -1;
}

pkv_status pkv_bm_swap(pkv_bm* src, pkv_bm* dst, const int64_t* seqs, int n, int32_t* pairs,
                       int cap, int* num_pairs) {
  if (src == nullptr || dst == nullptr || src == dst || n < 0 || num_pairs == nullptr ||
      (n > 0 && seqs == nullptr) || src->block_size != dst->block_size)
    return PKV_EINVAL;
  // Validate the group, then count its distinct blocks in order of first reference.
  std::unordered_map<int64_t, int> seen_seq;
  for (int i = 0; i < n; ++i) {
    if (!src->seqs.count(seqs[i]) || dst->seqs.count(seqs[i]) || seen_seq.count(seqs[i]))
      return PKV_ESTATE;
    seen_seq[seqs[i]] = i;
  }
  std::vector<int32_t> distinct;
  std::unordered_map<int32_t, int32_t> mapping;
  for (int i = 0; i < n; ++i)
    for (int32_t b : src->seqs[seqs[i]].table)
      if (mapping.emplace(b, -1).second) distinct.push_back(b);
  *num_pairs = static_cast<int>(distinct.size());
  if (static_cast<int64_t>(distinct.size()) > cap || (cap > 0 && pairs == nullptr)) return PKV_ERANGE;
  if (static_cast<int64_t>(distinct.size()) > dst->available()) return PKV_ENOMEM;
  for (size_t i = 0; i < distinct.size(); ++i) {
    int32_t d = dst->pop();
    dst->ref[d] = 0;
    mapping[distinct[i]] = d;
    pairs[2 * i] = distinct[i];
    pairs[2 * i + 1] = d;
  }
  for (int i = 0; i < n; ++i) {
    Sequence moved = src->seqs[seqs[i]];
    for (int32_t& b : moved.table) {
      b = mapping[b];
      dst->ref[b] += 1;
    }
    dst->seqs.emplace(seqs[i], std::move(moved));
  }
  for (int i = 0; i < n; ++i) pkv_bm_free(src, seqs[i]);
  return PKV_OK;
}

int pkv_bm_num_free(const pkv_bm* bm) {
  return bm ? static_cast<int>(bm->available()) : -1;
}

int pkv_bm_refcount(const pkv_bm* bm, int32_t block) {
  if (bm == nullptr || block < 0 || block >= bm->num_blocks) return -1;
  return bm->ref[block];
}

int64_t pkv_bm_length(const pkv_bm* bm, int64_t seq) {
  if (bm == nullptr) return -1;
  auto it = bm->seqs.find(seq);
  return it == bm->seqs.end() ? -1 : it->second.len;
}

pkv_status pkv_bm_block_table(const pkv_bm* bm, int64_t seq, int32_t* out, int cap, int* n) {
  if (bm == nullptr || n == nullptr || (cap > 0 && out == nullptr)) return PKV_EINVAL;
  auto it = bm->seqs.find(seq);
  if (it == bm->seqs.end()) return PKV_ESTATE;
  const auto& t = it->second.table;
  *n = static_cast<int>(t.size());
  if (static_cast<int64_t>(t.size()) > cap) return PKV_ERANGE;
  std::copy(t.begin(), t.end(), out);
  return PKV_OK;
}

pkv_status pkv_bm_fill_tables(const pkv_bm* bm, const int64_t* seqs, int n, int32_t* out,
                              int width, int32_t* context_lens) {
  if (bm == nullptr || n < 0 || width < 0 || (n > 0 && (seqs == nullptr || out == nullptr)))
    return PKV_EINVAL;
  for (int i = 0; i < n; ++i) {
    auto it = bm->seqs.find(seqs[i]);
    if (it == bm->seqs.end()) return PKV_ESTATE;
    if (static_cast<int64_t>(it->second.table.size()) > width) return PKV_ERANGE;
  }
  for (int i = 0; i < n; ++i) {
    const Sequence& s = bm->seqs.find(seqs[i])->second;
    int32_t* row = out + static_cast<int64_t>(i) * width;
    std::copy(s.table.begin(), s.table.end(), row);
    std::fill(row + s.table.size(), row + width, -1);
    if (context_lens) context_lens[i] = static_cast<int32_t>(s.len);
  }
  return PKV_OK;
}

pkv_status pkv_bm_slots(const pkv_bm* bm, int64_t seq, int64_t first, int64_t count,
                        int64_t* out) {
  if (bm == nullptr || first < 0 || count < 0 || (count > 0 && out == nullptr)) return PKV_EINVAL;
  auto it = bm->seqs.find(seq);
  if (it == bm->seqs.end()) return PKV_ESTATE;
  const Sequence& s = it->second;
  if (first + count > s.len) return PKV_ERANGE;
  const int64_t B = bm->block_size;
  for (int64_t i = 0; i < count; ++i) {
    int64_t p = first + i;
    out[i] = static_cast<int64_t>(s.table[p / B]) * B + p % B;
  }
  return PKV_OK;
}

int pkv_bm_free_list(const pkv_bm* bm, int32_t* out, int cap) {
  if (bm == nullptr) return -1;
  int n = static_cast<int>(bm->free_list.size());
  if (out) std::copy(bm->free_list.begin(), bm->free_list.begin() + std::min(n, cap), out);
  return n;
}

}  // extern "C"
