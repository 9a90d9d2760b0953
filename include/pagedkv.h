/*
 * pagedkv.h -- C ABI of libpagedkv.so: single-token decode attention over a paged
 * KV cache, for NVIDIA GB300 (sm_103a).
 *
 * The operation: every request (sequence) keeps its keys and values in fixed-size
 * physical blocks of `block_size` tokens; a per-request block table maps logical
 * block j to a physical block id ("分页注意力" section of "大模型工程（五）：推理优化
 * 核心技法", chenk.top; section 2.2 of the gsyq.cn inference-optimisation page, which
 * recommends 16- or 32-token blocks). Each decode step appends the new token's K/V
 * into its slot and then attends one query per head over the whole cached context
 * ("两个特性截然不同的阶段" of the chenk.top page: decode reads the entire KV cache
 * every step and is memory-bound).
 *
 * Conventions shared by every entry point
 *   - All tensor arguments are DEVICE pointers on the current CUDA device, owned by
 *     the caller. The library never allocates, frees or synchronises; every call is
 *     asynchronous on `stream` (NULL = the legacy default stream).
 *   - Host-side validation happens before any launch; a failed check returns a
 *     negative pkv_status and launches nothing.
 *   - Layouts (row-major, contiguous):
 *       q, out          [num_seqs, num_q_heads, head_dim]            bf16
 *       k, v (new)      [num_tokens, num_kv_heads, head_dim]         bf16
 *       k_cache,v_cache [num_blocks, num_kv_heads, block_size, head_dim]  bf16, int8
 *                       or FP8 (E4M3 / E5M2) byte codes
 *       k_scale,v_scale [num_blocks, num_kv_heads, block_size]       fp32 (one-byte caches)
 *       block_tables    [num_seqs, max_blocks_per_seq]               int32
 *       context_lens    [num_seqs]                                   int32
 *       slot_mapping    [num_tokens]                                 int64
 *     A slot is physical_block * block_size + offset; a negative slot is skipped.
 *     Query head h reads KV head h / (num_q_heads / num_kv_heads).
 *     context_lens[s] counts every token sequence s attends to (the one appended
 *     this step included); entries of block_tables past ceil(context_len /
 *     block_size) are never read. A sequence with context_len 0 gets a zero output.
 *   - Every cache/q/out pointer must be 16-byte aligned.
 *   - Supported sizes: head_dim 64 or 128; block_size 16 or 32; any
 *     num_q_heads / num_kv_heads group size (groups of 4 and more run on the tensor
 *     cores, smaller ones on the CUDA cores).
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* pkv_stream_t;

typedef enum pkv_status {
  PKV_OK = 0,
  PKV_ERR_NULL = -1,         /* a required pointer is NULL */
  PKV_ERR_DTYPE = -2,        /* unknown KV dtype code */
  PKV_ERR_SHAPE = -3,        /* a size is non-positive or sizes disagree */
  PKV_ERR_UNSUPPORTED = -4,  /* head_dim / block_size / batch outside what is built */
  PKV_ERR_WORKSPACE = -5,    /* workspace NULL, too small or misaligned */
  PKV_ERR_CUDA = -6,         /* a CUDA runtime or driver call failed */
  PKV_ERR_ALIGNMENT = -7,    /* a device pointer is not 16-byte aligned */
  PKV_ERR_HOST_MEMORY = -8   /* a host buffer is not pinned (page-locked) host memory */
} pkv_status;

typedef enum pkv_kv_dtype {
  PKV_KV_BF16 = 0,
  PKV_KV_INT8 = 1,           /* int8 codes + one fp32 scale per (token, KV head) */
  PKV_KV_FP8_E4M3 = 2,       /* FP8 E4M3 codes (bias 7, max 448) + fp32 scales */
  PKV_KV_FP8_E5M2 = 3        /* FP8 E5M2 codes (bias 15, max 57344) + fp32 scales */
} pkv_kv_dtype;

typedef struct pkv_dims {
  int32_t num_seqs;            /* B: requests in the batch                      */
  int32_t num_q_heads;         /* Hq                                            */
  int32_t num_kv_heads;        /* Hkv; Hq must be a multiple of Hkv             */
  int32_t head_dim;            /* D: 64 or 128                                  */
  int32_t block_size;          /* tokens per physical block: 16 or 32           */
  int32_t num_blocks;          /* physical blocks in the pool (cache dim 0)     */
  int32_t max_blocks_per_seq;  /* row length of block_tables                    */
} pkv_dims;

/* Bits of the optional device status word (see pkv_decode_*). */
#define PKV_DEV_BAD_CONTEXT_LEN 0x1  /* context_len < 0 or > max_blocks_per_seq*block_size */
#define PKV_DEV_BAD_BLOCK_ID    0x2  /* a block id the context needs is outside [0, num_blocks) */
#define PKV_DEV_TIMEOUT         0x4  /* a shared-memory copy did not complete in time */
#define PKV_DEV_BAD_PREFIX      0x8  /* cascade: a table does not start with the shared prefix */

/* Human-readable name of a status code (static string, never NULL). */
const char* pkv_status_string(pkv_status status);

/* Library version as major*10000 + minor*100 + patch. */
int pkv_version(void);

/* Number of kernels this library has launched (or recorded into a CUDA graph being
 * captured) in this process since it was loaded, all devices and threads together.
 * Read it before and after a call to learn how many kernels the call launched. A
 * launch that fails is not counted. Host-side counter only: it never touches a
 * device. No counterpart on the pages; it exists to count the kernels of a timed
 * region. */
uint64_t pkv_kernel_launch_count(void);

/*
 * pkv_append_bf16 -- write each new token's K and V rows into its cache slot.
 * Block manager of the chenk.top page ("块管理器：分页如何运作"): a growing request
 * writes into the block its table appends.
 *   k, v          [num_tokens, Hkv, D] bf16, read.
 *   k_cache/v_cache  [num_blocks, Hkv, block_size, D] bf16, written at the slots.
 *   slot_mapping  [num_tokens] int64; slot < 0 skips the token; a slot at or past
 *                 num_blocks*block_size is also skipped (nothing is written).
 * num_tokens == 0 is a no-op returning PKV_OK. Bit-exact copy.
 */
pkv_status pkv_append_bf16(const void* k, const void* v, void* k_cache, void* v_cache,
                           const int64_t* slot_mapping, int32_t num_tokens,
                           const pkv_dims* dims, pkv_stream_t stream);

/*
 * pkv_append_int8 -- quantise each new token's K and V rows per KV head and write
 * codes and scales into the slot. INT8 KV of section 2.3 of the gsyq.cn page and
 * "KV 缓存量化" of the chenk.top page (per-token, per-head scales), with the
 * round(w / s) form of "INT8 仅权重量化" on the same page:
 *   s = absmax(row) / 127 (fp32, IEEE division); q = clamp(rint(x / s), -127, 127)
 *   (IEEE division, round half to even); absmax == 0 gives s = 0 and q = 0.
 *   k, v       [num_tokens, Hkv, D] bf16, read.
 *   k_cache, v_cache  int8 [num_blocks, Hkv, block_size, D], written.
 *   k_scale, v_scale  fp32 [num_blocks, Hkv, block_size], written.
 */
pkv_status pkv_append_int8(const void* k, const void* v, int8_t* k_cache, int8_t* v_cache,
                           float* k_scale, float* v_scale, const int64_t* slot_mapping,
                           int32_t num_tokens, const pkv_dims* dims, pkv_stream_t stream);

/*
 * pkv_decode_workspace_bytes -- size of the device workspace that pkv_decode_bf16 /
 * pkv_decode_int8 / pkv_decode_fp8 need for these dims and KV dtype on the CURRENT device (it
 * depends on the device's SM count). Host-only query; writes *bytes.
 */
pkv_status pkv_decode_workspace_bytes(const pkv_dims* dims, pkv_kv_dtype kv_dtype,
                                      size_t* bytes);

/*
 * pkv_decode_bf16 -- out[s, h, :] = softmax(scale * K_s q[s, h]) V_s, where K_s, V_s
 * are sequence s's first context_lens[s] cached rows of KV head h / g, gathered
 * through block_tables[s]. fp32 accumulation, bf16 output (round to nearest even).
 *   workspace  device scratch of at least pkv_decode_workspace_bytes() bytes,
 *              256-byte aligned, caller-owned; contents need no initialisation and
 *              are overwritten. Calls that share a workspace must not overlap.
 *   status     optional device int32 (NULL to skip the checks). When given, the
 *              call validates context_lens and the used block ids, ORs the
 *              PKV_DEV_* bits of what it finds into *status and writes a zero
 *              output for every sequence that failed. Without it, invalid ids are
 *              clamped into the pool (no fault) and those outputs are unspecified.
 * Long contexts are split over several workers and merged with an online-softmax
 * (max/sum) reduction in a second kernel of the same call.
 */
pkv_status pkv_decode_bf16(void* out, const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, const int32_t* context_lens,
                           float scale, const pkv_dims* dims, void* workspace,
                           size_t workspace_bytes, int32_t* status, pkv_stream_t stream);

/*
 * pkv_decode_int8 -- as pkv_decode_bf16 over an INT8 cache: the cached value of a
 * row is code * scale with the row's fp32 scale (k_scale for K, v_scale for V).
 * V scales must stay below 65504 (they are folded into fp16 softmax weights).
 */
pkv_status pkv_decode_int8(void* out, const void* q, const int8_t* k_cache,
                           const int8_t* v_cache, const float* k_scale, const float* v_scale,
                           const int32_t* block_tables, const int32_t* context_lens,
                           float scale, const pkv_dims* dims, void* workspace,
                           size_t workspace_bytes, int32_t* status, pkv_stream_t stream);

/*
 * pkv_append_fp8 -- as pkv_append_int8 with FP8 codes: the E4M3 or E5M2 KV cache of
 * "FP8（及 H100/H200 硬件路径）" (chenk.top page; E5M2 is the format it names for KV
 * caches) with the per-token, per-head scales of "KV 缓存量化" (same page), computed
 * from the row itself at append time:
 *   s = absmax(row) / FP8_MAX (FP8_MAX = 448 for E4M3, 57344 for E5M2; IEEE fp32
 *   division); code = x / s (IEEE division) rounded to the nearest FP8 value, ties to
 *   the even code, saturating at +-FP8_MAX; absmax == 0 gives s = 0 and zero codes.
 *   A value that rounds to zero from below keeps its sign bit (code 0x80).
 *   fp8_format  PKV_KV_FP8_E4M3 or PKV_KV_FP8_E5M2 (else PKV_ERR_DTYPE).
 *   k_cache, v_cache  uint8 codes [num_blocks, Hkv, block_size, D], written.
 *   k_scale, v_scale  fp32 [num_blocks, Hkv, block_size], written.
 */
pkv_status pkv_append_fp8(const void* k, const void* v, uint8_t* k_cache, uint8_t* v_cache,
                          float* k_scale, float* v_scale, const int64_t* slot_mapping,
                          int32_t num_tokens, pkv_kv_dtype fp8_format, const pkv_dims* dims,
                          pkv_stream_t stream);

/*
 * pkv_decode_fp8 -- as pkv_decode_bf16 over an FP8 cache: the cached value of a row
 * element is decode(code) * scale with the row's fp32 scale (k_scale for K, v_scale
 * for V); codes are widened exactly. The V side folds scale * 2^15 (E5M2) or
 * scale * 2^8 (E4M3) into fp16 softmax weights (undone on the output), so rows
 * written by pkv_append_fp8 must have absmax below about 1e5. NaN codes are not expected (the append never
 * writes them). Workspace as pkv_decode_workspace_bytes(dims, fp8_format).
 */
pkv_status pkv_decode_fp8(void* out, const void* q, const uint8_t* k_cache,
                          const uint8_t* v_cache, const float* k_scale, const float* v_scale,
                          const int32_t* block_tables, const int32_t* context_lens, float scale,
                          pkv_kv_dtype fp8_format, const pkv_dims* dims, void* workspace,
                          size_t workspace_bytes, int32_t* status, pkv_stream_t stream);

/*
 * Whole-block moves ("块管理器：分页如何运作", chenk.top page). One block of the cache
 * holds the rows of every KV head: Hkv * block_size * head_dim elements of K (and of
 * V), plus Hkv * block_size fp32 scales each for one-byte caches. kv_dtype selects
 * the element size (PKV_KV_BF16: 2 bytes, no scales; INT8 / FP8: 1 byte + scales);
 * the scale pointers are ignored (may be NULL) for bf16. Ids are device int32 arrays
 * checked against [0, num_blocks): a pair with a bad id is skipped and, when
 * `status` (optional device int32) is given, flagged PKV_DEV_BAD_BLOCK_ID. Moves are
 * bit-exact. num_blocks_moved == 0 is a no-op.
 *
 * pkv_copy_blocks -- copy-on-write: block dst_ids[i] := block src_ids[i] for every
 *   pair (K, V and scales). Before a request writes into a block that another request
 *   still shares (refcount > 1 after a fork for parallel sampling, beam search or a
 *   speculative rollback), the block manager moves it to a fresh block; this is that
 *   copy, batched. The pairs must not chain: no destination may also be a source or
 *   repeat (the copies run in parallel).
 */
pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                           const int32_t* src_ids, const int32_t* dst_ids, int32_t num_pairs,
                           pkv_kv_dtype kv_dtype, const pkv_dims* dims, int32_t* status,
                           pkv_stream_t stream);

/*
 * pkv_swap_out -- eviction to host memory: host_k[i] := block block_ids[i] of k_cache
 *   (likewise V and scales), i.e. the request's blocks packed densely in list order:
 *   host_k [num_blocks_moved, Hkv, block_size, D], host_k_scale [num_blocks_moved,
 *   Hkv, block_size]. The host buffers must be pinned host memory (cudaHostAlloc or
 *   cudaHostRegister; else PKV_ERR_HOST_MEMORY): the GPU writes them directly.
 * pkv_swap_in -- the reverse: block block_ids[i] := host_k[i] (block ids distinct).
 * Both are asynchronous on `stream`; the host buffer must not be touched until the
 * stream reaches the call.
 */
pkv_status pkv_swap_out(void* host_k, void* host_v, float* host_k_scale, float* host_v_scale,
                        const void* k_cache, const void* v_cache, const float* k_scale,
                        const float* v_scale, const int32_t* block_ids, int32_t num_blocks_moved,
                        pkv_kv_dtype kv_dtype, const pkv_dims* dims, int32_t* status,
                        pkv_stream_t stream);
pkv_status pkv_swap_in(void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                       const void* host_k, const void* host_v, const float* host_k_scale,
                       const float* host_v_scale, const int32_t* block_ids,
                       int32_t num_blocks_moved, pkv_kv_dtype kv_dtype, const pkv_dims* dims,
                       int32_t* status, pkv_stream_t stream);

/* Largest q_len of pkv_decode_multi_bf16. */
#define PKV_MAX_QUERY_LEN 256

/*
 * pkv_decode_multi_workspace_bytes -- workspace that pkv_decode_multi_bf16 needs for
 * these dims and q_len on the CURRENT device. Host-only query; writes *bytes.
 */
pkv_status pkv_decode_multi_workspace_bytes(const pkv_dims* dims, int32_t q_len,
                                            size_t* bytes);

/*
 * pkv_decode_multi_bf16 -- paged attention for q_len new tokens per sequence in one
 * call: the verification pass of speculative decoding ("推测解码", chenk.top page: the
 * target model scores the k drafted tokens and the next position, q_len = k + 1, in
 * one forward pass); also a chunk of chunked prefill ("Orca 的迭代级调度", same page:
 * a prompt's prefill split into chunks that run beside the decode steps). Every sequence's q_len newest tokens are already in the cache (appended
 * with pkv_append_bf16), so context_lens[s] counts them; new token i of sequence s
 * sits at position context_lens[s] - q_len + i and attends causally:
 *   out[s, i, h, :] = softmax(scale * K q[s, i, h]) V over positions 0 .. that position.
 *   q, out     [num_seqs, q_len, num_q_heads, head_dim] bf16.
 *   q_len      1 .. PKV_MAX_QUERY_LEN (else PKV_ERR_SHAPE); 1 is pkv_decode_bf16.
 *   workspace  at least pkv_decode_multi_workspace_bytes(dims, q_len) bytes, as for
 *              pkv_decode_bf16.
 *   status     as for pkv_decode_bf16; a sequence with 0 < context_len < q_len is
 *              also flagged PKV_DEV_BAD_CONTEXT_LEN (and zeroed). Without status,
 *              query tokens that see no position get zeros.
 * Rows are (token, head) pairs on the tensor cores for every group size: a KV head
 * with 48 or more rows (q_len * g) runs them as ceil(rows / 128) equal row tiles, each
 * in one M = 128 tcgen05 MMA per 128-token tile (the row tiles of a head run one after
 * the other, so their re-reads of its blocks come from L2); fewer rows run as 16-row
 * mma.sync subgroups sharing each block through shared memory. Every row tile reads
 * the head's whole context (positions a row may not see are masked, not skipped).
 */
pkv_status pkv_decode_multi_bf16(void* out, const void* q, const void* k_cache,
                                 const void* v_cache, const int32_t* block_tables,
                                 const int32_t* context_lens, int32_t q_len, float scale,
                                 const pkv_dims* dims, void* workspace, size_t workspace_bytes,
                                 int32_t* status, pkv_stream_t stream);

/*
 * pkv_decode_multi_q8 -- pkv_decode_multi_bf16 over a one-byte cache: INT8, FP8 E4M3 or
 * FP8 E5M2 codes with one fp32 scale per (token, KV head) for K and for V, as written
 * by pkv_append_int8 / pkv_append_fp8 (the quantised KV caches of "KV 缓存量化",
 * chenk.top page), for speculative verification or a prefill chunk over such a cache.
 * The cached value of a row element is decode(code) * scale; codes are widened exactly
 * and each K and V value is rounded once to bf16 (code x scale) before the same
 * tensor-core contraction as the bf16 path, for every row count (q_len * g).
 *   kv_dtype   PKV_KV_INT8, PKV_KV_FP8_E4M3 or PKV_KV_FP8_E5M2 (else PKV_ERR_DTYPE).
 *   k_cache, v_cache  one-byte codes [num_blocks, Hkv, block_size, D];
 *   k_scale, v_scale  fp32 [num_blocks, Hkv, block_size].
 *   workspace  at least pkv_decode_multi_q8_workspace_bytes(dims, q_len, kv_dtype).
 * Other arguments, layouts and the causal rule as for pkv_decode_multi_bf16; q_len 1 is
 * pkv_decode_int8 / pkv_decode_fp8.
 */
pkv_status pkv_decode_multi_q8_workspace_bytes(const pkv_dims* dims, int32_t q_len,
                                               pkv_kv_dtype kv_dtype, size_t* bytes);
pkv_status pkv_decode_multi_q8(void* out, const void* q, const void* k_cache,
                               const void* v_cache, const float* k_scale, const float* v_scale,
                               const int32_t* block_tables, const int32_t* context_lens,
                               int32_t q_len, float scale, pkv_kv_dtype kv_dtype,
                               const pkv_dims* dims, void* workspace, size_t workspace_bytes,
                               int32_t* status, pkv_stream_t stream);

/*
 * pkv_decode_cascade_bf16 -- pkv_decode_bf16 for a batch whose sequences all start
 * with the same `prefix_blocks` physical blocks (a shared system prompt or few-shot
 * prefix: the shared blocks of "分页注意力", chenk.top, and section 2.2 of the gsyq.cn
 * page). Precondition: block_tables[s, 0..prefix_blocks-1] equals row 0's entries and
 * context_lens[s] >= prefix_blocks * block_size for every s. The result is the same
 * attention as pkv_decode_bf16 over the whole table; the prefix part is computed once
 * per KV head for all sequences as one dense tensor-core contraction (query rows of
 * the batch x prefix tokens), the suffixes by the ordinary decode, then merged.
 *   workspace  at least pkv_decode_cascade_workspace_bytes() bytes, 256-byte
 *              aligned, no initialisation needed.
 *   status     optional; additionally flags PKV_DEV_BAD_PREFIX (and zeroes the
 *              output) for a sequence that breaks the precondition. Without it,
 *              such a sequence's output is unspecified.
 */
pkv_status pkv_decode_cascade_workspace_bytes(const pkv_dims* dims, int32_t prefix_blocks,
                                              size_t* bytes);

pkv_status pkv_decode_cascade_bf16(void* out, const void* q, const void* k_cache,
                                   const void* v_cache, const int32_t* block_tables,
                                   const int32_t* context_lens, int32_t prefix_blocks,
                                   float scale, const pkv_dims* dims, void* workspace,
                                   size_t workspace_bytes, int32_t* status, pkv_stream_t stream);

/*
 * pkv_decode_cascade_q8 -- pkv_decode_cascade_bf16 over a one-byte cache (INT8, FP8 E4M3
 * or E5M2 codes with one fp32 scale per (token, KV head) for K and for V): a shared
 * system prompt over the quantised caches of "KV 缓存量化" (chenk.top page). The
 * shared prefix runs on the tensor cores with the codes widened in shared memory (K
 * codes exactly, each score column times its K scale; V as fp16 code x scale), the
 * suffixes through the one-byte decode of pkv_decode_int8 / pkv_decode_fp8.
 *   kv_dtype   PKV_KV_INT8, PKV_KV_FP8_E4M3 or PKV_KV_FP8_E5M2 (else PKV_ERR_DTYPE).
 *   workspace  at least pkv_decode_cascade_q8_workspace_bytes(dims, prefix_blocks,
 *              kv_dtype) bytes.
 * Everything else as for pkv_decode_cascade_bf16.
 */
pkv_status pkv_decode_cascade_q8_workspace_bytes(const pkv_dims* dims, int32_t prefix_blocks,
                                                 pkv_kv_dtype kv_dtype, size_t* bytes);
pkv_status pkv_decode_cascade_q8(void* out, const void* q, const void* k_cache,
                                 const void* v_cache, const float* k_scale, const float* v_scale,
                                 const int32_t* block_tables, const int32_t* context_lens,
                                 int32_t prefix_blocks, float scale, pkv_kv_dtype kv_dtype,
                                 const pkv_dims* dims, void* workspace, size_t workspace_bytes,
                                 int32_t* status, pkv_stream_t stream);

/*
 * pkv_decode_bf16_noalloc -- pkv_decode_bf16 for callers that cannot allocate device
 * memory (code running inside another runtime's memory pool, plugins not allowed to
 * call cudaMalloc, or latency-critical paths where no allocation may happen). The pages
 * have no counterpart: this is a library convenience, not part of the method.
 *   Same arguments and result as pkv_decode_bf16, without workspace: the call uses a
 *   fixed scratch array of PKV_NOALLOC_SCRATCH_BYTES that the library keeps in device
 *   memory on every GPU that loads it, until the process exits. It allocates nothing
 *   (no cudaMalloc, no cudaFree, no allocating library routine).
 *   Limits: the first PKV_NOALLOC_MAX_SEQ_HEADS * 8 bytes of the array hold the
 *   counters of the split-KV fold, so num_seqs * num_kv_heads may be at most
 *   PKV_NOALLOC_MAX_SEQ_HEADS, and the workspace these dims need (see
 *   pkv_decode_workspace_bytes with PKV_KV_BF16) at most the rest of the array. A call
 *   beyond either limit returns PKV_ERR_WORKSPACE and launches nothing.
 *   The array's device address is looked up with cudaGetSymbolAddress the first time a
 *   call runs under a CUDA context (once per device, and again after a device reset or
 *   under another context made current on that device); make that first call before
 *   any stream capture.
 *   Every call on a device shares the one scratch array, which keeps the last call's
 *   contents (nothing in it needs to start at zero). Calls whose executions overlap
 *   on the GPU (different streams, or other threads) race on it: serialise them.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (16u << 20)
#define PKV_NOALLOC_MAX_SEQ_HEADS 65536

pkv_status pkv_decode_bf16_noalloc(void* out, const void* q, const void* k_cache,
                                   const void* v_cache, const int32_t* block_tables,
                                   const int32_t* context_lens, float scale,
                                   const pkv_dims* dims, int32_t* status, pkv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
