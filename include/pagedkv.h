/*
 * pagedkv — paged KV-cache decode attention for NVIDIA GB300 (sm_103a).
 *
 * C ABI of libpagedkv.so. Plain pointers and sizes only; no CUDA or framework
 * types appear in the signatures. A CUDA stream is passed as `void*`
 * (a cudaStream_t; NULL is the legacy default stream).
 *
 * Sources of the operations (web pages on vLLM's PagedAttention):
 *  [R]  "079｜vLLM 与 PagedAttention：不改变模型，也能让更多请求同时运行",
 *       wq-win.github.io — review of Kwon et al., SOSP 2023.
 *  [G]  "vLLM 推理引擎：PagedAttention 与 KVCache 管理", gitcode.csdn.net.
 *  [D]  "PagedAttention 内存管理深度解析", deepinsea.top.
 *
 * Conventions shared by every call:
 *  - dtype codes: PKV_F16 = IEEE binary16, PKV_BF16 = bfloat16, PKV_F32 = binary32.
 *  - KV cache layout ([G] §3, PagedAttention.forward comments):
 *        k_cache, v_cache: [num_blocks][block_size][num_kv_heads][head_size]
 *    a "slot" is block * block_size + row; row-major, contiguous.
 *  - Device buffers are owned by the caller and must stay valid until the work
 *    queued on `stream` has finished. The library allocates no device memory;
 *    the decode call takes a caller-provided workspace.
 *  - Host-side validation is synchronous and happens before anything is queued:
 *    on an error status nothing was launched and nothing was written.
 *  - Device-side checks: a kernel that finds an out-of-range index in device
 *    data skips the access and ORs a PKV_DEVERR_* bit into *err_flag (a device
 *    int32 the caller zeroes and reads; may be NULL). Kernels never trap.
 *  - All GPU calls are asynchronous with respect to the host.
 */
#ifndef PAGEDKV_H_
#define PAGEDKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkv_status {
  PKV_OK = 0,
  PKV_EINVAL = 1,     /* null pointer, bad shape, unsupported size or dtype, misaligned pointer */
  PKV_ENOMEM = 2,     /* block manager: too few free blocks; nothing was changed */
  PKV_ERANGE = 3,     /* host-visible index out of range (block id, copy pair) */
  PKV_ECUDA = 4,      /* a CUDA runtime or launch error */
  PKV_ESTATE = 5,     /* block manager: unknown or duplicate sequence id, reference-count underflow */
  PKV_EWORKSPACE = 6  /* decode workspace smaller than pkv_decode_workspace_size() */
} pkv_status;

enum { PKV_F16 = 0, PKV_BF16 = 1, PKV_F32 = 2 };

/* Bits a kernel ORs into *err_flag. */
#define PKV_DEVERR_BLOCK_ID 0x1 /* block-table entry outside [0, num_blocks) */
#define PKV_DEVERR_CONTEXT 0x2  /* context length outside [1, max_blocks_per_seq * block_size] */
#define PKV_DEVERR_SLOT 0x4     /* slot_mapping entry >= num_blocks * block_size */
#define PKV_DEVERR_TIMEOUT 0x8  /* a pipeline wait gave up (the kernel returned early) */

/* Human-readable name of a status code; never NULL. */
const char* pkv_status_string(int status);
/* Library version string. */
const char* pkv_version(void);

/* ------------------------------------------------------------------------
 * Decode attention over the paged cache.
 *
 * Defines ([R] §2 "分块以后，注意力仍需对整个历史归一化"): for each sequence s
 * and query head h, with L = context_lens[s] tokens stored in the blocks
 * block_tables[s][0 .. ceil(L/B)-1] in position order,
 *     o[s][h] = sum_u exp(scale * q.k_u) v_u / sum_u exp(scale * q.k_u)
 * over all L positions u — one softmax denominator for the whole history, the
 * unfilled rows of the last block excluded. Query head h reads KV head
 * h / (num_heads / num_kv_heads).
 *
 * The context is processed in partitions of `partition_tokens` tokens (0 picks
 * a default, see pkv_decode_partition_tokens; otherwise a positive multiple of
 * 32, at most 4096): each (sequence, KV head, partition) produces an
 * unnormalised partial, and a second kernel merges the partials of each
 * (sequence, head) with the global denominator.
 *
 *   out          device, [num_seqs][num_heads][head_size] of out_dtype (F16, BF16 or F32)
 *   q            device, [num_seqs][num_heads][head_size] of kv_dtype
 *   k_cache,
 *   v_cache      device, [num_blocks][block_size][num_kv_heads][head_size] of kv_dtype
 *   kv_dtype     PKV_F16 or PKV_BF16
 *   block_tables device int32 [num_seqs][max_blocks_per_seq]; entries past
 *                ceil(L/B) are never read (pad with -1)
 *   context_lens device int32 [num_seqs]; 1 <= L <= max_blocks_per_seq * block_size
 *                (the newest token counts)
 *   head_size    64 or 128; num_heads a multiple of num_kv_heads
 *   block_size   a power of two from 1 to 256
 *   scale        multiplies q.k (typically 1/sqrt(head_size))
 *   workspace    device, >= pkv_decode_workspace_size(...) bytes, 16-byte aligned;
 *                scratch owned by the caller, contents on entry irrelevant
 *   err_flag     device int32 or NULL (see PKV_DEVERR_*); a sequence whose length
 *                is out of range gets an all-zero output row
 * q, out, k_cache and v_cache must be 16-byte aligned.
 * Errors: PKV_EINVAL (shape/dtype/alignment), PKV_EWORKSPACE, PKV_ECUDA.
 * ------------------------------------------------------------------------ */
/* Workspace bytes of a decode call with these arguments (the call's own
 * shape arguments); 0 for a shape no call accepts. */
size_t pkv_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_size,
                                 int max_blocks_per_seq, int block_size, int partition_tokens);

/* The partition size a decode call with these arguments uses: partition_tokens
 * itself when nonzero. Otherwise 1024 on the tensor paths when the batch has
 * enough units to keep every SM busy (each unit then carries twice the keys
 * per merge): units = num_seqs * num_kv_heads * ceil(max context / 1024) at
 * least 1024 for query groups of 2 to 16 heads per KV head (block_size >= 8),
 * at least 256 for groups of 32, 64 or 128 heads (the tensor-memory path),
 * where 2048 is taken instead when num_seqs * num_kv_heads * ceil(max
 * context / 2048) is at least 256 and 2048 / block_size is at most 254;
 * else 512, or 1024 when the tables can hold 32768 tokens or more (long
 * contexts then produce half as many partials). Never fails. */
int pkv_decode_partition_tokens(int num_seqs, int num_heads, int num_kv_heads, int head_size,
                                int max_blocks_per_seq, int block_size, int partition_tokens);

pkv_status pkv_paged_attention_decode(void* out, int out_dtype, const void* q,
                                      const void* k_cache, const void* v_cache, int kv_dtype,
                                      const int32_t* block_tables, const int32_t* context_lens,
                                      int num_seqs, int num_heads, int num_kv_heads, int head_size,
                                      int num_blocks, int block_size, int max_blocks_per_seq,
                                      float scale, int partition_tokens, void* workspace,
                                      size_t workspace_bytes, int32_t* err_flag, void* stream);

/* ------------------------------------------------------------------------
 * Test hook of the failure path (no counterpart on the pages): runs the
 * decode call's tensor-memory path (query groups of 32, 64 or 128 heads per
 * KV head; anything else gives PKV_EINVAL) with every pipeline wait limited to
 * wait_limit_ns (1000 .. 1e9) and the softmax warps of every CTA waiting, at
 * their first unit, on a barrier that no copy, product or thread completes.
 * That wait runs out, and then so do the waits of the threads that depended on
 * it: the kernel sets PKV_DEVERR_TIMEOUT in *err_flag (which must not be
 * NULL), lets its copies and products in flight finish, frees its tensor
 * memory and returns; the next call on the device runs normally. The outputs
 * of this call are undefined. Arguments otherwise as for
 * pkv_paged_attention_decode.
 * ------------------------------------------------------------------------ */
pkv_status pkv_test_decode_wait_timeout(void* out, int out_dtype, const void* q,
                                        const void* k_cache, const void* v_cache, int kv_dtype,
                                        const int32_t* block_tables, const int32_t* context_lens,
                                        int num_seqs, int num_heads, int num_kv_heads,
                                        int head_size, int num_blocks, int block_size,
                                        int max_blocks_per_seq, float scale, int partition_tokens,
                                        void* workspace, size_t workspace_bytes,
                                        int32_t* err_flag, uint64_t wait_limit_ns, void* stream);

/* ------------------------------------------------------------------------
 * Decode attention without a caller workspace.
 *
 * No counterpart on the pages: this is a convenience of this library. It is
 * for callers that cannot allocate device memory — a plugin that its host
 * application gives only input and output buffers, or a serving loop that
 * reserved all memory up front and must not call cudaMalloc (which can stall
 * the device) while decoding. It computes exactly what
 * pkv_paged_attention_decode computes, with the same arguments minus the
 * workspace; the partition partials go to a fixed array of
 * PKV_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that loads the
 * library keeps until the process exits. It allocates nothing.
 *
 *  - Limit: PKV_EWORKSPACE (nothing launched) when
 *    pkv_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_size,
 *    max_blocks_per_seq, block_size, partition_tokens) > PKV_NOALLOC_SCRATCH_BYTES.
 *  - The first call on a device looks up the array's device address (once per
 *    device, with that device current; host code cannot name device memory
 *    directly), and so does the first call after a cudaDeviceReset of that
 *    device, which unloads the array. Make that first call before any stream
 *    capture. A failed lookup returns PKV_ECUDA.
 *  - All calls share the one array and it keeps the last call's contents.
 *    Nothing in it needs to start at zero (each call writes every partial it
 *    reads), but calls whose GPU work overlaps — on different streams, or from
 *    different host threads — race on it and corrupt each other's outputs:
 *    issue them on one stream.
 * ------------------------------------------------------------------------ */
#define PKV_NOALLOC_SCRATCH_BYTES (8u << 20) /* 8 MiB */

pkv_status pkv_paged_attention_decode_noalloc(void* out, int out_dtype, const void* q,
                                              const void* k_cache, const void* v_cache,
                                              int kv_dtype, const int32_t* block_tables,
                                              const int32_t* context_lens, int num_seqs,
                                              int num_heads, int num_kv_heads, int head_size,
                                              int num_blocks, int block_size,
                                              int max_blocks_per_seq, float scale,
                                              int partition_tokens, int32_t* err_flag,
                                              void* stream);

/* ------------------------------------------------------------------------
 * Chunked prefill attention over the paged cache.
 *
 * Defines ([Z] §4 chunked prefill: a long prompt is processed in chunks whose
 * attention masks follow their position in the prompt, each attending to the
 * cache the earlier chunks left; [R] §2 for the one global denominator):
 * sequence s holds L = context_lens[s] tokens, the last C of which are its
 * query chunk, rows query_start[s] .. query_start[s+1]-1 of q; query i
 * (position L - C + i) attends over positions 0 .. L - C + i:
 *     o_i = sum_{u <= L-C+i} exp(scale * q_i.k_u) v_u / sum_{u <= L-C+i} exp(scale * q_i.k_u).
 * The chunk's keys and values must already be in the cache (reshape_and_cache).
 * C = 1 is a decode step; C = 0 leaves the sequence out.
 *
 *   out, q        device, [total_queries][num_heads][head_size] (out_dtype / kv_dtype)
 *   caches, tables, context_lens  as for pkv_paged_attention_decode
 *   query_start   device int32 [num_seqs + 1], non-decreasing, query_start[0] = 0
 *   max_query_len host int >= every C (sizes the work list)
 *   total_queries host int, rows of q and out
 *   head_size 64 or 128; block_size a power of two from 8 to 256;
 *   128 % (num_heads / num_kv_heads) == 0; scale > 0
 *   workspace     device, >= pkv_prefill_workspace_size() bytes, 16-byte
 *                 aligned, owned by the caller: holds the counter the
 *                 persistent CTAs claim work from (zeroed by the call on
 *                 `stream`); it must not be shared by calls that may run at
 *                 the same time
 * Work: one item per 256 query rows (chunk tokens x the KV head's query
 * heads), KV head and sequence; at most one CTA per SM takes items, those
 * with the most keys first.
 * Device checks: 0 <= C <= min(L, max_query_len), L <= max_blocks_per_seq *
 * block_size and query_start[s] + C <= total_queries, else the sequence is
 * skipped (its rows untouched) and PKV_DEVERR_CONTEXT set; bad block ids as
 * for decode.
 * Errors: PKV_EINVAL (also a missing, short or unaligned workspace),
 * PKV_ECUDA.
 * ------------------------------------------------------------------------ */
size_t pkv_prefill_workspace_size(void);
pkv_status pkv_paged_attention_prefill(void* out, int out_dtype, const void* q,
                                       const void* k_cache, const void* v_cache, int kv_dtype,
                                       const int32_t* block_tables, const int32_t* context_lens,
                                       const int32_t* query_start, int num_seqs, int num_heads,
                                       int num_kv_heads, int head_size, int num_blocks,
                                       int block_size, int max_blocks_per_seq, int max_query_len,
                                       int total_queries, float scale, void* workspace,
                                       size_t workspace_bytes, int32_t* err_flag, void* stream);

/* ------------------------------------------------------------------------
 * reshape_and_cache: write new tokens' keys and values into their slots.
 *
 * Defines ([R] §2 "共享与写时复制" and the §3 per-iteration algorithm box: the
 * new token goes into the sequence's tail block): for every token t with
 * slot = slot_mapping[t] >= 0,
 *     k_cache[slot / B][slot % B][h][:] = k[t][h][:]   (same for v), bitwise.
 * A negative slot means "skip". A slot >= num_blocks * B is skipped and sets
 * PKV_DEVERR_SLOT.
 *
 *   k, v          device, [num_tokens][num_kv_heads][head_size] of dtype
 *   k_cache, ...  device, layout above
 *   slot_mapping  device int64 [num_tokens]
 *   dtype         PKV_F16 or PKV_BF16; head_size * 2 a multiple of 16
 * All four data pointers 16-byte aligned. num_tokens == 0 is a no-op.
 * Two tokens with the same slot race (one of them wins).
 * ------------------------------------------------------------------------ */
pkv_status pkv_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                                 const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                 int head_size, int num_blocks, int block_size, int dtype,
                                 int32_t* err_flag, void* stream);

/* ------------------------------------------------------------------------
 * copy_blocks: copy-on-write block copies.
 *
 * Defines ([R] §2 "共享与写时复制" and "一次分叉什么时候真的要复制缓存块"):
 * before a branch writes into a block another branch still references, the
 * block is copied and only this branch is remapped. For every pair i,
 *     K[dst_i] = K[src_i], V[dst_i] = V[src_i]      (block_bytes bytes each).
 *
 *   src_dst_pairs  HOST int32 [num_pairs][2] = {src, dst}; read before the call
 *                  returns (the ids travel in the kernel's parameters, so the
 *                  host buffer may be reused at once)
 *   block_bytes    bytes of one block of one cache:
 *                  block_size * num_kv_heads * head_size * element size;
 *                  a multiple of 16; caches 16-byte aligned
 * Ids must lie in [0, num_blocks) (else PKV_ERANGE); destinations must be
 * distinct and no destination may also be a source (else PKV_EINVAL).
 * num_pairs == 0 is a no-op.
 * ------------------------------------------------------------------------ */
pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, const int32_t* src_dst_pairs,
                           int num_pairs, int num_blocks, size_t block_bytes, void* stream);

/* ------------------------------------------------------------------------
 * swap_blocks: copies between two block pools, one of which is typically in
 * pinned host memory (swap space).
 *
 * Defines ([R] §3 algorithm box: a preempted group's cache is swapped out and
 * later swapped back in; [D] "Swap 机制"): for every pair i,
 *     dst_K[dst_i] = src_K[src_i], dst_V[dst_i] = src_V[src_i]   (block_bytes each).
 *
 *   src_k, src_v, dst_k, dst_v  device memory, or pinned host memory the GPU can
 *                  address (cudaHostAlloc / cudaHostRegister); the kernel reads
 *                  and writes host memory directly over the CPU-GPU link
 *   src_dst_pairs  HOST int32 [num_pairs][2] = {src, dst}, read before the call returns
 *   src_blocks, dst_blocks  blocks in the two pools (ids must lie below them)
 *   block_bytes    as for copy_blocks
 * Distinct destinations required (PKV_EINVAL); ids out of range give
 * PKV_ERANGE; a pointer the GPU cannot address gives PKV_EINVAL.
 * num_pairs == 0 is a no-op.
 * ------------------------------------------------------------------------ */
pkv_status pkv_swap_blocks(void* dst_k, void* dst_v, const void* src_k, const void* src_v,
                           const int32_t* src_dst_pairs, int num_pairs, int src_blocks,
                           int dst_blocks, size_t block_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Host block manager: free list, reference counts, fork, copy-on-write.
 *
 * Defines: [D] "分页机制设计" (a free list of block ids; a request takes
 * ceil(n/B) blocks popped from the end of the list and fails with no side
 * effect when too few are free; released blocks are appended back) and [R] §2
 * "共享与写时复制" (per-block reference counts; a fork shares every block; a
 * block is reclaimed only when its count reaches zero; writing into a tail
 * block still shared copies it first), [R] §2 "一次分叉什么时候真的要复制缓存块"
 * (full blocks are never copied) and the §3 algorithm box (check whether the
 * next token needs a new block; copy-on-write a shared tail).
 *
 * The handle is owned by the library: create with pkv_bm_create, release with
 * pkv_bm_destroy. Not thread-safe: one thread at a time per handle.
 * Sequence ids are arbitrary int64 keys chosen by the caller.
 * ------------------------------------------------------------------------ */
typedef struct pkv_bm pkv_bm;

/* free_order: NULL, or a permutation of 0..num_blocks-1 that becomes the
 * initial free list (blocks are handed out from its end). NULL means the list
 * 0, 1, ..., num_blocks-1. Returns NULL on bad arguments. */
pkv_bm* pkv_bm_create(int num_blocks, int block_size, const int32_t* free_order);
void pkv_bm_destroy(pkv_bm* bm);

/* A new sequence holding num_tokens >= 0 tokens (ceil(n/B) blocks, count 1).
 * PKV_ESTATE if seq exists; PKV_ENOMEM (no change) if too few blocks are free. */
pkv_status pkv_bm_allocate(pkv_bm* bm, int64_t seq, int64_t num_tokens);
/* Automatic prefix caching ([Z] §2.2(5): every block is kept in a hash table
 * keyed by its tokens and all the tokens before it; a new request reuses the
 * cached blocks of its prefix). A new sequence holding the n prompt tokens
 * token_ids: for each full block j the chained hash h_j = FNV-1a-64(h_{j-1} as
 * 8 little-endian bytes, then the block's token ids as 4 little-endian bytes
 * each), h_{-1} = 0, is looked up; the blocks of the longest run of hits from
 * the start are shared (count + 1), the remaining blocks are fresh and the full
 * ones among them are registered. *cached_tokens (nullable) receives the
 * number of leading tokens whose keys/values are already in the pool — the
 * caller writes only the rest. A registered block whose count drops to zero
 * keeps its contents and is evictable (oldest first) when the free list runs
 * out. PKV_ESTATE if seq exists; PKV_ENOMEM (no change) if too few blocks. */
pkv_status pkv_bm_allocate_prefix(pkv_bm* bm, int64_t seq, const int32_t* token_ids, int64_t n,
                                  int64_t* cached_tokens);
/* Number of blocks registered in the prefix cache. */
int pkv_bm_num_cached(const pkv_bm* bm);

/* child shares all of parent's blocks (each count + 1) and its length. */
pkv_status pkv_bm_fork(pkv_bm* bm, int64_t parent, int64_t child);
/* Room for one more token of seq. *slot receives its slot. If the tail block
 * was shared, a fresh block replaces it in seq's table and (*cow_src, *cow_dst)
 * receive the pair to copy before writing; otherwise both are set to -1.
 * PKV_ENOMEM (no change) when a block is needed and none is free. */
pkv_status pkv_bm_append_slot(pkv_bm* bm, int64_t seq, int64_t* slot, int32_t* cow_src,
                              int32_t* cow_dst);
/* append_slot for n sequences in order, all or nothing: on PKV_ENOMEM /
 * PKV_ESTATE nothing changed. slots: int64 [n]; cow_pairs: int32 [n][2] (room
 * for n pairs); *num_cow receives the number of pairs written. */
pkv_status pkv_bm_append_slots(pkv_bm* bm, const int64_t* seqs, int n, int64_t* slots,
                               int32_t* cow_pairs, int* num_cow);
/* Drop seq; blocks whose count reaches zero return to the free list in the
 * sequence's logical order. */
pkv_status pkv_bm_free(pkv_bm* bm, int64_t seq);

/* Swap: move the sequence group seqs[0..n) from pool src to pool dst (for
 * instance GPU pool -> CPU pool on preemption and back on resumption; [R] §3
 * algorithm box, [Z] §3.3 swapped queue, [D] "Swap 机制"). Every distinct
 * block the group references gets one dst block, in order of first reference;
 * blocks shared inside the group stay shared; the sequences leave src (blocks
 * still referenced by other src sequences stay there). pairs[i] = {src block,
 * dst block} receives the copies to make (pkv_swap_blocks), *num_pairs their
 * number. All or nothing: PKV_ENOMEM if dst has too few free blocks,
 * PKV_ERANGE if cap < the number of pairs (*num_pairs still set),
 * PKV_ESTATE for an unknown, repeated or already-present sequence, PKV_EINVAL
 * if the block sizes differ. */
pkv_status pkv_bm_swap(pkv_bm* src, pkv_bm* dst, const int64_t* seqs, int n, int32_t* pairs,
                       int cap, int* num_pairs);

/* Queries. num_free counts the free list and evictable cached blocks. */
int pkv_bm_num_free(const pkv_bm* bm);
int pkv_bm_refcount(const pkv_bm* bm, int32_t block); /* -1 if out of range */
int64_t pkv_bm_length(const pkv_bm* bm, int64_t seq); /* -1 if unknown */
/* seq's table into out[0..cap); *n receives its length (PKV_ERANGE if > cap). */
pkv_status pkv_bm_block_table(const pkv_bm* bm, int64_t seq, int32_t* out, int cap, int* n);
/* Tables of n sequences into out[n][width], padded with -1, and their lengths
 * into context_lens[n] (may be NULL). PKV_ERANGE if a table is wider. */
pkv_status pkv_bm_fill_tables(const pkv_bm* bm, const int64_t* seqs, int n, int32_t* out,
                              int width, int32_t* context_lens);
/* Slots of positions first .. first+count-1 of seq into out[count]. */
pkv_status pkv_bm_slots(const pkv_bm* bm, int64_t seq, int64_t first, int64_t count,
                        int64_t* out);
/* The free list (without evictable cached blocks), bottom to top (the next
 * block handed out is the last one); returns its length, writes at most cap
 * entries. */
int pkv_bm_free_list(const pkv_bm* bm, int32_t* out, int cap);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H_ */
