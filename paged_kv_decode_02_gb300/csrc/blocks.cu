// blocks.cu -- whole-block moves of the paged KV cache.
//
// The block manager of "大模型工程（五）：推理优化核心技法" (chenk.top, section "块管理器：
// 分页如何运作") shares blocks between requests under copy-on-write: before a request
// writes into a block another request still references, the block is copied to a
// fresh one. Under memory pressure a victim request's blocks are copied to pinned host
// memory and freed, and copied back into (new) blocks when memory frees up.
//
// In the [num_blocks, Hkv, block_size, D] layout one block's rows of every KV head are
// one contiguous chunk (Hkv * block_size * D * elt bytes; Hkv * block_size * 4 bytes of
// scales), so every move is "chunk src_i -> chunk dst_i" over up to four arrays (K, V
// and, for one-byte caches, their scales). One kernel does all three moves: each CTA
// copies one 16 KiB slice of one chunk with 16-byte words, four loads in flight per
// thread, the array picked by blockIdx.y. Host buffers are pinned host memory that the
// GPU reads and writes directly (over NVLink-C2C on GB300), so a request moves in one
// launch instead of one copy call per scattered block.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace pkv {

constexpr int kMoveThreads = 256;
constexpr int kMoveUnroll = 4;
constexpr int kSliceWords = kMoveThreads * kMoveUnroll;  // 16 KiB per CTA

// CTA (x, y): slice x % slices of pair x / slices of array y.
__global__ void __launch_bounds__(kMoveThreads) paged_block_move_kernel(const MoveParams p) {
  pdl_wait_prior_grid();
  const MoveArray a = p.arrays[blockIdx.y];
  const int slices = (a.chunk16 + kSliceWords - 1) / kSliceWords;
  const int i = blockIdx.x / slices;
  if (i >= p.n) return;
  const int w0 = (blockIdx.x % slices) * kSliceWords;
  const int s = p.src_ids ? p.src_ids[i] : i;
  const int d = p.dst_ids ? p.dst_ids[i] : i;
  if ((p.src_ids && (s < 0 || s >= p.NB)) || (p.dst_ids && (d < 0 || d >= p.NB))) {
    if (p.status && threadIdx.x == 0 && w0 == 0 && blockIdx.y == 0)
      atomicOr(p.status, PKV_DEV_BAD_BLOCK_ID);
    return;
  }
  const uint4* src = a.src + (size_t)s * a.chunk16;
  uint4* dst = a.dst + (size_t)d * a.chunk16;
  uint4 v[kMoveUnroll];
#pragma unroll
  for (int k = 0; k < kMoveUnroll; ++k) {
    const int w = w0 + k * kMoveThreads + threadIdx.x;
    if (w < a.chunk16) v[k] = src[w];
  }
#pragma unroll
  for (int k = 0; k < kMoveUnroll; ++k) {
    const int w = w0 + k * kMoveThreads + threadIdx.x;
    if (w < a.chunk16) dst[w] = v[k];
  }
}

cudaError_t launch_block_move(const MoveParams& p, cudaStream_t stream) {
  if (p.n <= 0 || p.narrays <= 0) return cudaSuccess;
  long long gx = 0;
  for (int i = 0; i < p.narrays; ++i)
    gx = std::max(gx, (long long)p.n * ((p.arrays[i].chunk16 + kSliceWords - 1) / kSliceWords));
  if (gx >= (1ll << 31)) return cudaErrorInvalidValue;
  MoveParams copy = p;
  void* args[] = {&copy};
  return launch_pdl(reinterpret_cast<const void*>(&paged_block_move_kernel),
                    dim3(unsigned(gx), unsigned(p.narrays)), dim3(kMoveThreads), args, 0, stream);
}

}  // namespace pkv
