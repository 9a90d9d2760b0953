// merge.cu -- folds the partials of units cut between decode workers.
//
// A (sequence, unit) whose blocks were cut between several decode warps left one
// unnormalised partial per warp: o_w = sum_t 2^(x_t - m_w) v_t, l_w = sum_t
// 2^(x_t - m_w), m_w = max_t x_t (scores x_t in log2 units). The exact softmax output
// is recovered with the online-softmax rescaling
//   m = max_w m_w,  l = sum_w 2^(m_w - m) l_w,  out = sum_w 2^(m_w - m) o_w / l.
// One warp per (unit, group of query rows), one 16-byte output quad per lane: it
// zero-fills empty sequences and, when a status word is given, validates the
// sequence's context length and block ids (zeroing the output of a sequence that
// fails); units the decode kernel finished itself then leave at once. A lane folds
// its row's parts in chunks whose loads are all in flight together (fold.cuh).
#include "common.cuh"
#include "fold.cuh"
#include "internal.h"

namespace pkv {

constexpr int kMergeWarps = 8;  // one (unit, row group) per warp

__device__ __forceinline__ long long merge_worker_start(long long T, int w, int W) {
  return T * w / W;
}

// Largest worker w whose range [T*w/W, T*(w+1)/W) contains flat index x.
__device__ __forceinline__ int merge_worker_of(long long x, long long T, int W) {
  return int(((x + 1) * W + T - 1) / T) - 1;
}

__global__ void __launch_bounds__(kMergeWarps * 32, 3) paged_decode_merge_kernel(const MergeParams p) {
  pdl_wait_prior_grid();
  const int lane = threadIdx.x & 31;
  const int gs = p.gs, D = p.D, Q = D / 4;
  const int rpw = 32 / Q;                 // rows per warp: one output quad per lane
  const int ngrp = (gs + rpw - 1) / rpw;  // row groups per unit
  const int item = blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
  if (item >= p.B * p.HU * ngrp) return;
  const int unit = item / ngrp, r0 = (item % ngrp) * rpw;
  const int s = unit / p.HU, u = unit % p.HU;
  const int row = r0 + lane / Q, dq = lane % Q;
  // work items (blocks, or 128-token tiles for the tcgen05 kernel) of the sequence
  const int n = p.prefix[s + 1] - p.prefix[s];
  // output row of unit row r: (s * q_len + i) * Hq + kvh * g + j for the unit's query
  // row R = (u % nsg) * gs + r = i * g + j (with q_len = 1: head kvh * g + R)
  const int R = (u % p.nsg) * gs + row;
  // rows past q_len * g: the padding of a partial last row tile (tcgen05 kernel)
  const bool active = row < gs && R < p.q_len * p.g;
  uint2* out = reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.out) +
                                        ((size_t(s) * p.q_len + R / p.g) * p.Hq +
                                         (u / p.nsg) * p.g + R % p.g) * D) + dq;

  bool zero = (n == 0);
  if (p.status != nullptr) {
    int flags = 0;
    const int L = p.context_lens[s];
    if (lane == 0 && (L < 0 || L > p.MBS * p.BS || (L > 0 && L < p.q_len))) flags |= 0x1;
    const int nblk = L <= 0 ? 0 : min((L + p.BS - 1) / p.BS, p.MBS);
    for (int j = lane; j < nblk; j += 32) {
      const int id = p.block_tables[size_t(s) * p.MBS + j];
      if (id < 0 || id >= p.NB) flags |= 0x2;
    }
    flags = __reduce_or_sync(0xffffffffu, flags);
    if (flags) {
      if (lane == 0 && u == 0 && r0 == 0) atomicOr(p.status, flags);
      zero = true;
    }
  }
  if (zero) {
    if (active) *out = make_uint2(0u, 0u);
    return;
  }
  // The mma.sync kernels' flat order is (sequence, KV head, block) over W workers of nsg
  // warps each; this unit's parts come from warp worker * nsg + sg of each worker. The
  // tcgen05 kernel (beta > 0) orders (sequence, unit, tile) over W CTAs, every unit (a
  // row tile of a KV head) its own position in the order, and its parts are the CTAs'
  // slots; that order is weighted: every unit of a non-empty sequence takes n + beta
  // positions, its n tiles first, then beta that hold none.
  const int beta = p.beta;
  const bool tc = beta > 0;
  const int nsg = tc ? 1 : p.nsg, sg = tc ? 0 : u % p.nsg;
  const int ord = tc ? u : u / p.nsg;            // the unit's place within its sequence
  const int Hkv = tc ? p.HU : p.HU / p.nsg;      // places per sequence
  const int* pre = tc ? p.wprefix : p.prefix;
  const long long T = (long long)Hkv * pre[p.B];
  const long long A = (long long)Hkv * pre[s] + (long long)ord * (n + beta);
  const int W = p.W;
  const int w0 = merge_worker_of(A, T, W), w1 = merge_worker_of(A + n - 1, T, W);
  if (w0 == w1 || !active) return;  // one worker covered the whole unit: output written
  // T >= W: every worker range is non-empty and the parts are workers w0..w1;
  // otherwise ranges hold one position at most and part i is the worker of item A + i
  const bool dense = T >= W;
  const int nparts = dense ? (w1 - w0 + 1) : n;
  // the unit is not worker w0's first segment when w0 processed an item before it (the
  // previous unit's items end beta positions before A)
  const bool first_cut = A > 0 && merge_worker_start(T, w0, W) < A - beta;
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml);
  Fold f = fold_empty();
  fold_parts<8>(f, 0, 1, nparts, [&](int i, const float2*& pm, const float4*& po) {
    const size_t slot =
        dense ? size_t(2 * ((w0 + i) * nsg + sg) + ((i == 0 && first_cut) ? 1 : 0))
              : size_t(2 * (merge_worker_of(A + i, T, W) * nsg + sg));
    pm = ml + slot * gs + row;
    po = reinterpret_cast<const float4*>(p.part_o + (slot * gs + row) * D) + dq;
  });
  *out = fold_result(f);
}

void launch_merge(const MergeParams& p, cudaStream_t stream) {
  const int rpw = 32 / (p.D / 4);
  const long long items = (long long)p.B * p.HU * ((p.gs + rpw - 1) / rpw);
  if (items <= 0) return;
  const int grid = int((items + kMergeWarps - 1) / kMergeWarps);
  MergeParams copy = p;
  void* args[] = {&copy};
  launch_pdl(reinterpret_cast<const void*>(&paged_decode_merge_kernel), dim3(grid),
             dim3(kMergeWarps * 32), args, 0, stream);
}

}  // namespace pkv
