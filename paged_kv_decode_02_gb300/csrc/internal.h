// internal.h -- declarations shared by the library's translation units (not public).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <atomic>

#include "pagedkv.h"

namespace pkv {

// Parameters of one decode launch (device pointers; sizes as in pkv_dims).
struct DecodeParams {
  const void* q;               // [B, q_len, Hq, D] bf16
  void* out;                   // [B, q_len, Hq, D] bf16
  const float* k_scale;        // [NB, Hkv, BS] fp32 (one-byte caches only)
  const float* v_scale;
  const int32_t* block_tables; // [B, MBS]
  const int32_t* context_lens; // [B]
  float* part_o;               // [2W, GS, D] fp32 partial outputs (unnormalised)
  float* part_ml;              // [2W, GS, 2] fp32 (running max in log2 units, sum)
  int32_t* prefix_out;         // [B+1] blocks-per-sequence exclusive prefix (CTA 0 writes)
  int skip;                    // table entries skipped at the head of every sequence (cascade)
  int unit_slot0;              // >= 0: complete units write a partial to slot unit_slot0 + s*HU + u
                               //       instead of the output (cascade); -1: normal
  int32_t* status;             // optional device status word
  int B, Hq, Hkv, MBS, NB;
  int q_len;                   // new tokens per sequence (1: single-token decode)
  int beta;                    // tcgen05 kernel: ranges are cut in an order where every
                               //   non-empty KV head adds beta units after its tiles
  unsigned long long* fix_ctr; // [B, Hkv] counters of the in-kernel stream-K fixup
  int fixup;                   // fold cut units in the decode kernel (no merge kernel)
  int late_wait;               // wait for the previous grid only before exiting (cascade
                               //   suffix running beside the prefix kernel)
  int tma_out;                 // tcgen05 kernel: whole heads leave through TMA tensor stores
                               //   (boxes of g rows x 64 columns; needs g in {8, 16, 32})
  int g;                       // Hq / Hkv
  int gs;                      // query rows (token, head) handled per work unit
  int nsg;                     // work units per KV head (q_len * g / gs)
  int HU;                      // work units per sequence (Hkv * nsg)
  float scale_log2;            // softmax scale * log2(e)
  unsigned long long timeout_ns;
};

// Parameters of the shared-prefix (cascade) kernel: for KV head h, the B*g query rows
// (sequence s, group member i) attend the prefix blocks block_tables[0, 0..P-1].
struct PrefixParams {
  const void* q;               // [B, Hq, D] bf16
  const float* k_scale;        // [NB, Hkv, BS] fp32 (one-byte caches only)
  const float* v_scale;
  const int32_t* prefix_ids;   // [P] physical ids of the shared prefix (row 0 of the tables)
  float* pre_o;                // [nsplit, Hkv, R, D] unnormalised partial outputs
  float* pre_ml;               // [nsplit, Hkv, R, 2] (running max in log2 units, sum)
  int P, B, Hq, Hkv, g, R, NB;  // R = B * g query rows per KV head
  int nsplit, per_split;       // prefix blocks [z*per_split, min(P, (z+1)*per_split)) for split z
  int overlap;                 // let the next grid (the suffix decode, late_wait) start at once
  float scale_log2;
  unsigned long long timeout_ns;
  int32_t* status;
};

// Parameters of the cascade merge: prefix records plus suffix parts.
struct CascadeMergeParams {
  void* out;
  const float* part_o;         // decode partials: [2W + B*HU, gs, D]
  const float* part_ml;
  const float* pre_o;
  const float* pre_ml;
  const int32_t* prefix;       // suffix blocks-per-sequence prefix from the decode kernel
  const int32_t* block_tables;
  const int32_t* context_lens;
  int32_t* status;
  int B, Hq, Hkv, D, MBS, NB, BS, P;
  int g, gs, nsg, HU, R, nsplit;
  int W;                       // decode warps (whole-unit records start at slot 2W)
  int Wg;                      // decode workers (groups of nsg warps)
};

// The compiled prefix kernel for a (head_dim, block_size) and its launch shape.
struct PrefixKernelInfo {
  const void* fn;
  int smem;          // dynamic shared memory bytes
  int threads;       // threads per CTA
  int rows;          // query rows per CTA
  int tile_blocks;   // prefix blocks per tile (splits are cut at tile boundaries)
  int max_split_blocks;  // most prefix blocks one split may hold (a multiple of tile_blocks)
};
bool select_prefix_kernel(int D, int BS, int kvt, PrefixKernelInfo* info);
void launch_cascade_merge(const CascadeMergeParams& p, cudaStream_t stream);

// Parameters of the split-KV merge launch (units cut between decode workers).
struct MergeParams {
  void* out;
  const float* part_o;
  const float* part_ml;
  const int32_t* prefix;
  const int32_t* block_tables;
  const int32_t* context_lens;
  int32_t* status;
  int B, Hq, D, MBS, NB, BS;
  int q_len;                   // new tokens per sequence (rows map as in DecodeParams)
  int g, gs, nsg, HU;
  int W;                       // decode workers (groups of nsg warps, or tcgen05 CTAs)
  const int32_t* wprefix;      // beta > 0: per-sequence prefix of tiles + beta * [tiles > 0]
  int beta;                    // as in DecodeParams (0: workers cut the plain order)
};

void launch_merge(const MergeParams& p, cudaStream_t stream);

// Whole-block moves (copy-on-write copy, swap-out, swap-in): pair i moves chunk
// src_ids[i] (or i when src_ids is NULL: a dense host buffer) of every array to chunk
// dst_ids[i] (or i). Ids are checked against [0, NB): a bad pair is skipped and
// flagged PKV_DEV_BAD_BLOCK_ID.
struct MoveArray {
  const uint4* src;
  uint4* dst;
  int chunk16;                 // 16-byte words per block
};
struct MoveParams {
  MoveArray arrays[4];
  int narrays;
  const int32_t* src_ids;
  const int32_t* dst_ids;
  int n, NB;
  int32_t* status;
};

cudaError_t launch_block_move(const MoveParams& p, cudaStream_t stream);

// A compiled decode kernel and its static shape.
struct DecodeKernelInfo {
  const void* fn;
  int warps;         // warps per CTA (each warp is one independent worker)
  int stages;        // shared-memory pipeline depth per warp
  int warp_smem;     // shared-memory bytes per warp (1024-aligned)
  int mma;           // 1 = tensor-core path (groups >= 4), 0 = CUDA-core path
  int simt_heads;    // query heads per unit on the CUDA-core path
  int coop;          // 1: a worker is nsg warps sharing one ring (warp_smem per worker)
  int blk;           // physical blocks per work item (2: pairs of 16-token blocks)
  int tc;            // 1: the tcgen05 kernel (decode_tc.cu): one CTA per SM, all rows of a
                     //    KV head per MMA, warp_smem = fixed shared memory per CTA
  int fixup;         // 1: can fold cut units itself (DecodeParams::fixup)
};

// Kernel tables, one per translation unit. Return false if the shape is not built.
// pair: 16-token blocks in pairs on the tensor-core path (not with a skipped prefix)
bool select_decode_bf16(int D, int BS, int simt_heads, DecodeKernelInfo* info,
                        bool pair = false);
// q_len > 1: the causal multi-query variant of the bf16 tensor-core path, with
// workers of nsg warps sharing their shared-memory ring (CTA shape chosen for nsg)
bool select_decode_bf16_multi(int D, int BS, int nsg, DecodeKernelInfo* info);
// One-byte KV code formats.
enum : int { CODE_I8 = 0, CODE_E4M3 = 1, CODE_E5M2 = 2 };
// The tcgen05 decode kernel for a KV dtype (pkv_kv_dtype); row_tiles: the rows of a KV
// head run as several row tiles (more than 128 rows); split: a single tile of at most
// 64 rows, two softmax threads per row. The per-code tables live in decode_tc_int8.cu,
// decode_tc_e4m3.cu and decode_tc_e5m2.cu.
bool select_decode_tc(int D, int BS, bool row_tiles, bool split, int kvt,
                      DecodeKernelInfo* info);
bool select_decode_tc_int8(int D, int BS, bool row_tiles, bool split, DecodeKernelInfo* info);
bool select_decode_tc_e4m3(int D, int BS, bool row_tiles, bool split, DecodeKernelInfo* info);
bool select_decode_tc_e5m2(int D, int BS, bool row_tiles, bool split, DecodeKernelInfo* info);

bool select_decode_int8(int D, int BS, int simt_heads, DecodeKernelInfo* info,
                        bool pair = false);
bool select_decode_e4m3(int D, int BS, int simt_heads, DecodeKernelInfo* info,
                        bool pair = false);
bool select_decode_e5m2(int D, int BS, int simt_heads, DecodeKernelInfo* info,
                        bool pair = false);

// Launches with programmatic stream serialisation: the kernel may be scheduled while
// the previous kernel on the stream drains; every kernel of this library waits for its
// predecessor (griddepcontrol.wait) before touching global memory, so results are
// the same as with plain stream ordering.
// Kernels this library has launched in this process (launch_pdl is the only launch
// site); read through pkv_kernel_launch_count.
extern std::atomic<unsigned long long> g_kernel_launches;

inline cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, void** args, size_t smem,
                              cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t err = cudaLaunchKernelExC(&cfg, fn, args);
  if (err == cudaSuccess) g_kernel_launches.fetch_add(1, std::memory_order_relaxed);
  return err;
}

// pkv_decode_bf16 whose in-kernel fixup keeps its [B, Hkv] counter words at
// `counters` (at least B * Hkv 8-byte words, holding nothing but these counters)
// rather than in its region of the workspace.
pkv_status decode_bf16_fixed_counters(void* out, const void* q, const void* k_cache,
                                      const void* v_cache, const int32_t* block_tables,
                                      const int32_t* context_lens, float scale,
                                      const pkv_dims* dims, void* workspace,
                                      size_t workspace_bytes, unsigned long long* counters,
                                      size_t counter_words, int32_t* status,
                                      cudaStream_t stream);

cudaError_t launch_append_bf16(const void* k, const void* v, void* k_cache, void* v_cache,
                               const int64_t* slots, int T, int Hkv, int D, int BS, int NB,
                               cudaStream_t stream);
// code: CODE_I8, CODE_E4M3 or CODE_E5M2
cudaError_t launch_append_q8(int code, const void* k, const void* v, void* k_cache,
                             void* v_cache, float* k_scale, float* v_scale, const int64_t* slots,
                             int T, int Hkv, int D, int BS, int NB, cudaStream_t stream);

}  // namespace pkv
