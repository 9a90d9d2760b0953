// decode.cuh -- paged-KV single-token decode attention kernels for sm_103a.
//
// What is computed: for every sequence s and query head h,
//   out[s,h,:] = softmax(scale * K_s q[s,h]) V_s
// over the first context_lens[s] cached tokens of KV head h/g, reached through the
// block table ("分页注意力" of "大模型工程（五）：推理优化核心技法", chenk.top). Decode
// reads every cached byte once per step and is bound by HBM bandwidth ("两个特性截然
// 不同的阶段", same page), so the design is built around streaming KV blocks:
//
// * Work split (stream-K over blocks): the (sequence, work-unit, logical block)
//   triples are laid out in one flat order and cut into W equal contiguous ranges,
//   one per warp of a persistent grid (W = warps per CTA x CTAs that fit x SMs).
//   Ragged lengths therefore cost nothing in balance. A warp whose range covers a
//   whole (sequence, unit) writes the final output; a cut unit leaves one
//   unnormalised partial (o, running max, sum) per warp, which the merge kernel
//   (merge.cu) folds with the online-softmax rescaling m = max m_w,
//   l = sum 2^(m_w - m) l_w, o = sum 2^(m_w - m) o_w / l. The merge kernel also
//   zero-fills empty sequences and, when asked, validates the tables.
// * Data movement: each warp owns a private ring of shared-memory stages. One lane
//   reads the block id from the table and issues TMA tensor copies of the block's K
//   and V tiles (128-byte swizzled, so that the tensor-core fragment loads below are
//   bank-conflict free) plus, for one-byte caches, 1-D bulk copies of the per-token scales, all
//   completing on that stage's mbarrier. Copies run `stages` blocks ahead of the math.
// * Math: groups of 4 or more query heads per KV head make q.K^T a small dense
//   contraction, done with m16n8k16 tensor-core MMAs (query heads on M, padded to 16;
//   tokens on N; fp32 accumulate); P.V reuses the score fragments as the A operand.
//   Smaller groups run on the CUDA cores with 16-byte shared loads and warp-shuffle
//   reductions. Online softmax in base 2 with a max subtraction keeps the weights
//   in [0, 1] ("softmax 数值稳定性" note of section 2.3 of the gsyq.cn page).
// * INT8 KV (section 2.3 of the gsyq.cn page; "KV 缓存量化" of the chenk.top page) and
//   FP8 KV, E4M3 or E5M2 ("FP8（及 H100/H200 硬件路径）", chenk.top): codes are widened
//   exactly to fp16 in registers (Code8 below); the K scale multiplies the fp32
//   score and the V scale is folded into the softmax weight before the P.V MMA.
#pragma once

#include "common.cuh"
#include "fold.cuh"
#include "internal.h"

namespace pkv {

// ---------------------------------------------------------------------------
// One-byte KV codes widened exactly to fp16 pairs in registers. pre() is applied
// once to each loaded 32-bit word of four codes; lo() then yields codes 0 and 1 of
// the word as an f16x2, hi() codes 2 and 3, equal to the codes' values.
//   INT8: the byte is placed under the fp16 exponent pattern of 1024 and 1152 is
//         subtracted (after the sign bit of the code is flipped) -- exact.
//   E5M2: an E5M2 code is the upper byte of the binary16 of the same value, so a
//         byte permute that puts it there with a zero lower byte is the conversion.
//   E4M3: the conversion instruction for packed E4M3 pairs (every E4M3 value is a
//         binary16 value, so it is exact). Measured on GB300 it costs the same as
//         the E5M2 permute, where moving the 7 magnitude bits under the sign with
//         integer operations (4 per pair) made the decode 44 % slower.
// ---------------------------------------------------------------------------
template <int CODE>
struct Code8;

template <>
struct Code8<CODE_I8> {
  __device__ static __forceinline__ uint32_t pre(uint32_t w) { return w ^ 0x80808080u; }
  __device__ static __forceinline__ uint32_t lo(uint32_t w) {
    return biased_bytes_to_f16x2(w, 0x4140u);
  }
  __device__ static __forceinline__ uint32_t hi(uint32_t w) {
    return biased_bytes_to_f16x2(w, 0x4342u);
  }
};

template <>
struct Code8<CODE_E5M2> {
  __device__ static __forceinline__ uint32_t pre(uint32_t w) { return w; }
  __device__ static __forceinline__ uint32_t lo(uint32_t w) { return prmt(w, 0u, 0x1404u); }
  __device__ static __forceinline__ uint32_t hi(uint32_t w) { return prmt(w, 0u, 0x3424u); }
};

template <>
struct Code8<CODE_E4M3> {
  __device__ static __forceinline__ uint32_t pre(uint32_t w) { return w; }
  __device__ static __forceinline__ uint32_t lo(uint32_t w) {
    uint32_t r;
    asm("{ .reg .b16 l, h; mov.b32 {l, h}, %1; cvt.rn.f16x2.e4m3x2 %0, l; }" : "=r"(r) : "r"(w));
    return r;
  }
  __device__ static __forceinline__ uint32_t hi(uint32_t w) {
    uint32_t r;
    asm("{ .reg .b16 l, h; mov.b32 {l, h}, %1; cvt.rn.f16x2.e4m3x2 %0, h; }" : "=r"(r) : "r"(w));
    return r;
  }
};

// ---------------------------------------------------------------------------
// Tile geometry: a K (or V) tile holds one physical block of one KV head,
// block_size rows of head_dim elements, landed by TMA as `halves` boxes of
// [BS rows x kSeg bytes], each swizzled in 128- (or 64-) byte rows.
// ---------------------------------------------------------------------------
template <bool Q8, int D, int BS>
struct TileGeom {
  static constexpr int kElt = Q8 ? 1 : 2;
  static constexpr int kRowBytes = D * kElt;
  static constexpr int kSeg = kRowBytes >= 128 ? 128 : 64;
  static constexpr int kHalves = kRowBytes / kSeg;
  static constexpr int kChunksPerSeg = kSeg / 16;
  static constexpr int kChunksPerRow = kRowBytes / 16;
  static constexpr int kTileBytes = BS * kRowBytes;
  static constexpr int kScaleBytes = Q8 ? BS * 4 : 0;
  static_assert(kTileBytes % 1024 == 0, "tiles must keep 1024-byte alignment");

  // Swizzled byte offset of 16-byte chunk `cc` of token row `t`.
  __device__ static __forceinline__ uint32_t off(int t, int cc) {
    const int half = cc / kChunksPerSeg, ci = cc % kChunksPerSeg;
    return swz<kSeg>(uint32_t((half * BS + t) * kSeg + ci * 16));
  }
};

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ float lds_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts128_zero(uint32_t addr) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
}

// First query head of work unit u (KV head u / nsg, subgroup u % nsg).
__device__ __forceinline__ int unit_head0(const DecodeParams& p, int u) {
  return (u / p.nsg) * p.g + (u % p.nsg) * p.gs;
}

// Query rows of a KV head are the q_len * g pairs (new token i, group member j),
// numbered R = i * g + j; work unit u takes rows (u % nsg) * gs .. + gs - 1. Row r of
// unit u of sequence s reads q / writes out row (s * q_len + i) * Hq + kvh * g + j.
// With q_len = 1 this is head unit_head0 + r of sequence s.
__device__ __forceinline__ size_t query_row(const DecodeParams& p, int s, int u, int r) {
  const int R = (u % p.nsg) * p.gs + r;
  return (size_t(s) * p.q_len + R / p.g) * p.Hq + (u / p.nsg) * p.g + R % p.g;
}

// Tokens of a unit's visible range that row r may not see: new token i sits at
// position L - q_len + i, so it sees all but the last q_len - 1 - i positions.
__device__ __forceinline__ int causal_hidden(const DecodeParams& p, int u, int r) {
  return p.q_len - 1 - ((u % p.nsg) * p.gs + r) / p.g;
}

// Where a warp leaves a cut unit: slot 2w for the unit its range starts in, 2w+1
// for the unit its range ends in (w = worker * nsg + row subgroup).
__device__ __forceinline__ size_t partial_slot(int w, bool first_segment) {
  return size_t(2 * w + (first_segment ? 0 : 1));
}

// Launch number of this grid within the context (differs between launches, graph
// replays included).
__device__ __forceinline__ unsigned long long grid_launch_id() {
  unsigned long long g;
  asm volatile("mov.u64 %0, %%gridid;" : "=l"(g));
  return g;
}

// 40-bit tag of this launch for the fixup counters: the launch number spread over all
// 40 bits by a multiplicative (Fibonacci) hash, never 0. Launch numbers are small
// integers, so unhashed tags would sit in the low bits, where stale data of another
// use of the workspace (floats such as +0.0 or small integers) often does; spread
// tags meet such a word by chance only (one in 2^40 per word).
__device__ __forceinline__ unsigned long long launch_tag() {
  const unsigned long long t = ((grid_launch_id() + 1ull) * 0x9E3779B97F4A7C15ull) >> 24;
  return t == 0ull ? 1ull : t;
}

// Stream-K fixup inside the decode kernel (single-token decode, one warp per unit row
// group, no status word): a warp that left a partial record for a cut unit adds the
// unit items it covered to the unit's counter; the warp whose addition completes the
// unit's n items folds every part (the same parts and slots the split-KV merge kernel
// would take) and writes the output. A counter word holds a launch tag (launch_tag: a
// 40-bit hash of the grid's launch number) over a 24-bit item count: a word with
// another tag counts as zero, so the workspace needs no clearing, and the completing
// warp resets it.
// Writers fence their records before the counter update, the completing warp fences
// after it and reads the records through L2.
template <int D>
__device__ __forceinline__ void fixup_cut_unit(const DecodeParams& p, const int* s_prefix,
                                               int s, int kvh, int n, int mine,
                                               long long T, int W, int lane) {
  __threadfence();
  __syncwarp();
  int last = 0;
  if (lane == 0) {
    const unsigned long long tag = launch_tag();
    unsigned long long* ctr = p.fix_ctr + size_t(s) * p.Hkv + kvh;
    unsigned long long cur = *reinterpret_cast<volatile unsigned long long*>(ctr);
    for (;;) {
      const unsigned long long base = (cur >> 24) == tag ? (cur & 0xffffffull) : 0ull;
      const unsigned long long want = (tag << 24) | (base + unsigned(mine));
      const unsigned long long seen = atomicCAS(ctr, cur, want);
      if (seen == cur) {
        last = int(base) + mine == n;
        break;
      }
      cur = seen;
    }
    if (last) atomicExch(ctr, 0ull);
  }
  if (!__shfl_sync(0xffffffffu, last, 0)) return;
  __threadfence();
  // the unit's parts, as in the split-KV merge kernel
  const long long A = (long long)p.Hkv * s_prefix[s] + (long long)kvh * n;
  auto worker_of = [&](long long x) { return int(((x + 1) * W + T - 1) / T) - 1; };
  const int w0 = worker_of(A), w1 = worker_of(A + n - 1);
  const bool dense = T >= W;
  const int nparts = dense ? (w1 - w0 + 1) : n;
  const bool first_cut = A > 0 && (T * w0 / W) < A;
  constexpr int Q = D / 4;
  const int gs = p.gs, items = gs * Q;
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml);
  constexpr int kRows = 1;  // one item per lane at a time: few registers beside the main loop
  for (int k0 = lane; k0 < items; k0 += 32 * kRows) {
    const int live = min(kRows, (items - k0 + 31) / 32);
    Fold f[kRows];
#pragma unroll
    for (int j = 0; j < kRows; ++j) f[j] = fold_empty();
    fold_rows<kRows, 2, true>(f, live, nparts, [&](int i, int j, const float2*& pm,
                                                   const float4*& po) {
      const int k = k0 + 32 * j, r = k / Q, dq = k % Q;
      const size_t slot =
          dense ? size_t(2 * (w0 + i) + ((i == 0 && first_cut) ? 1 : 0))
                : size_t(2 * worker_of(A + i));
      pm = ml + slot * gs + r;
      po = reinterpret_cast<const float4*>(p.part_o + (slot * gs + r) * D) + dq;
    });
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      if (j >= live) break;
      const int k = k0 + 32 * j, r = k / Q, dq = k % Q;
      reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.out) +
                               (size_t(s) * p.Hq + size_t(kvh) * p.g + r) * D)[dq] =
          fold_result(f[j]);
    }
  }
}

// ===========================================================================
// CUDA-core path (groups of 1..3 query heads per KV head)
//
// Eight lanes share a token row (four rows per round); a lane owns one or two
// 16-byte chunks of head_dim and keeps q for them in registers. Dot products use
// packed fp32x2 FMAs and a 3-step shuffle reduction over the row's lanes; P.V
// accumulates each lane's chunks in fp32x2 registers, combined across the four row
// groups once per work unit.
// ===========================================================================
template <bool Q8, int D, int BS, int G, int CODE = CODE_I8>
struct SimtPath {
  // cut units are folded in the decode kernel (fixup_cut_unit) where that leaves the
  // kernel's occupancy as it was: bf16 caches, head_dim 128, one query head per KV head
  static constexpr bool kFixup = !Q8 && D == 128 && G == 1;
  using Geo = TileGeom<Q8, D, BS>;
  using Codec = Code8<CODE>;
  static constexpr int kChunks = Geo::kChunksPerRow;          // 16-byte chunks per row
  static constexpr int kLPR = kChunks < 8 ? kChunks : 8;      // lanes per token row
  static constexpr int kCPL = kChunks / kLPR;                 // chunks per lane
  static constexpr int kRPR = 32 / kLPR;                      // token rows per round
  static constexpr int kRounds = BS / kRPR;
  static constexpr int kEPC = 16 / Geo::kElt;                 // elements per chunk
  static constexpr int kEPL = kCPL * kEPC;                    // elements per lane
  static_assert(kRounds >= 1 && kEPL % 2 == 0, "row geometry");

  int lane, c, r0, head0, s;
  float2 q2[G][kEPL / 2];
  float2 o2[G][kEPL / 2];
  float m[G], l[G];

  // lane chunk k covers elements [(c + k*kLPR) * kEPC, +kEPC)
  __device__ __forceinline__ int chunk_of(int k) const { return c + k * kLPR; }

  __device__ __forceinline__ void init(int lane_) {
    lane = lane_;
    c = lane % kLPR;
    r0 = lane / kLPR;
  }

  __device__ __forceinline__ void begin(const DecodeParams& p, int s_, int u) {
    s = s_;
    head0 = unit_head0(p, u);
    const __nv_bfloat16* qb = reinterpret_cast<const __nv_bfloat16*>(p.q);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const __nv_bfloat16* row = qb + (size_t(s) * p.Hq + head0 + h) * D;
#pragma unroll
      for (int k = 0; k < kCPL; ++k) {
#pragma unroll
        for (int v = 0; v < kEPC / 8; ++v) {
          const uint4 raw =
              __ldg(reinterpret_cast<const uint4*>(row + chunk_of(k) * kEPC) + v);
          const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = unpack_bf16x2(w[e]);
            q2[h][(k * kEPC + v * 8) / 2 + e] =
                make_float2(f.x * p.scale_log2, f.y * p.scale_log2);
          }
        }
      }
      m[h] = -INFINITY;
      l[h] = 0.f;
#pragma unroll
      for (int e = 0; e < kEPL / 2; ++e) o2[h][e] = make_float2(0.f, 0.f);
    }
  }

  // kEPL/2 fp32 pairs of one token row (bf16 and one-byte codes exactly widened).
  __device__ __forceinline__ void load_row(uint32_t tile, int row, float2 (&f)[kEPL / 2]) const {
#pragma unroll
    for (int k = 0; k < kCPL; ++k) {
      const uint4 raw = lds128(tile + Geo::off(row, chunk_of(k)));
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
      if constexpr (Q8) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t b = Codec::pre(w[e]);
          f[k * 8 + 2 * e] = unpack_f16x2(Codec::lo(b));
          f[k * 8 + 2 * e + 1] = unpack_f16x2(Codec::hi(b));
        }
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) f[k * 4 + e] = unpack_bf16x2(w[e]);
      }
    }
  }

  __device__ __forceinline__ void block(const DecodeParams&, uint32_t sK, uint32_t sV,
                                        uint32_t sKs, uint32_t sVs, int nvalid) {
    float sc[G][kRounds];
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
      const int row = r * kRPR + r0;
      float2 kf[kEPL / 2];
      load_row(sK, row, kf);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < kEPL / 2; ++e) acc = __ffma2_rn(q2[h][e], kf[e], acc);
        float a = acc.x + acc.y;
#pragma unroll
        for (int off = kLPR / 2; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
        if constexpr (Q8) a *= lds_f32(sKs + 4 * row);
        sc[h][r] = (row < nvalid) ? a : -INFINITY;
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float mx = sc[h][0];
#pragma unroll
      for (int r = 1; r < kRounds; ++r) mx = fmaxf(mx, sc[h][r]);
#pragma unroll
      for (int off = kLPR; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mn = fmaxf(m[h], mx);
      const float alpha = fast_exp2(m[h] - mn);
      m[h] = mn;
      l[h] *= alpha;
      const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
      for (int e = 0; e < kEPL / 2; ++e) o2[h][e] = __fmul2_rn(o2[h][e], a2);
#pragma unroll
      for (int r = 0; r < kRounds; ++r) sc[h][r] = fast_exp2(sc[h][r] - mn);
    }
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
      const int row = r * kRPR + r0;
      if (row < nvalid) {
        float2 vf[kEPL / 2];
        load_row(sV, row, vf);
        float vsc = 1.f;
        if constexpr (Q8) vsc = lds_f32(sVs + 4 * row);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          l[h] += sc[h][r];
          const float pw = sc[h][r] * vsc;
          const float2 p2 = make_float2(pw, pw);
#pragma unroll
          for (int e = 0; e < kEPL / 2; ++e) o2[h][e] = __ffma2_rn(p2, vf[e], o2[h][e]);
        }
      }
    }
  }

  __device__ __forceinline__ void finish(const DecodeParams& p, bool complete, size_t slot) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
      for (int off = kLPR; off < 32; off <<= 1) {
        l[h] += __shfl_xor_sync(0xffffffffu, l[h], off);
#pragma unroll
        for (int e = 0; e < kEPL / 2; ++e) {
          o2[h][e].x += __shfl_xor_sync(0xffffffffu, o2[h][e].x, off);
          o2[h][e].y += __shfl_xor_sync(0xffffffffu, o2[h][e].y, off);
        }
      }
    }
    if (r0 != 0) return;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      if (complete) {
        const float inv = 1.f / l[h];
        __nv_bfloat16* row =
            reinterpret_cast<__nv_bfloat16*>(p.out) + (size_t(s) * p.Hq + head0 + h) * D;
#pragma unroll
        for (int k = 0; k < kCPL; ++k) {
#pragma unroll
          for (int v = 0; v < kEPC / 8; ++v) {
            const float2* f = &o2[h][(k * kEPC + v * 8) / 2];
            uint4 pk;
            pk.x = pack_bf16x2(f[0].x * inv, f[0].y * inv);
            pk.y = pack_bf16x2(f[1].x * inv, f[1].y * inv);
            pk.z = pack_bf16x2(f[2].x * inv, f[2].y * inv);
            pk.w = pack_bf16x2(f[3].x * inv, f[3].y * inv);
            reinterpret_cast<uint4*>(row + chunk_of(k) * kEPC)[v] = pk;
          }
        }
      } else {
        float* row = p.part_o + (slot * p.gs + h) * D;
#pragma unroll
        for (int k = 0; k < kCPL; ++k) {
#pragma unroll
          for (int v = 0; v < kEPC / 4; ++v) {
            const float2* f = &o2[h][(k * kEPC + v * 4) / 2];
            reinterpret_cast<float4*>(row + chunk_of(k) * kEPC)[v] =
                make_float4(f[0].x, f[0].y, f[1].x, f[1].y);
          }
        }
        if (c == 0)
          reinterpret_cast<float2*>(p.part_ml)[slot * p.gs + h] = make_float2(m[h], l[h]);
      }
    }
  }
};

// ===========================================================================
// Tensor-core path, bf16 cache (groups of 4..16 query heads per work unit)
//
// kCausal: the multi-query variant (q_len new tokens per sequence; rows are (token,
// head) pairs, see query_row). Each row hides the positions after its own token, a
// row may then see no token of a block (its softmax state stays empty: m = -inf,
// l = 0, handled without NaNs), and a row that sees nothing at all outputs zeros.
// ===========================================================================
template <int D, int BS, bool kCausal = false>
struct MmaPathBf16 {
  static constexpr bool kFixup = false;  // cut units go to the merge kernel
  using Geo = TileGeom<false, D, BS>;
  static constexpr int kKS = D / 16;  // k-steps of q.K^T
  static constexpr int kNT = BS / 8;  // token n-tiles
  static constexpr int kND = D / 8;   // head_dim n-tiles of P.V
  static constexpr int kKK = BS / 16; // token k-steps of P.V

  int lane, gid, cq, head0, s, gs;
  int u, hide0, hide1;                // kCausal: unit, hidden trailing tokens of both rows
  uint32_t qa[kKS][4];
  float o[kND][4];
  float m0, m1, l0, l1;

  __device__ __forceinline__ void init(int lane_) {
    lane = lane_;
    gid = lane >> 2;
    cq = lane & 3;
  }

  __device__ __forceinline__ void begin(const DecodeParams& p, int s_, int u_) {
    s = s_;
    gs = p.gs;
    const uint32_t* qw = reinterpret_cast<const uint32_t*>(p.q);
    if constexpr (kCausal) {
      u = u_;
      const bool v0 = gid < gs, v1 = gid + 8 < gs;
      hide0 = v0 ? causal_hidden(p, u, gid) : 0;
      hide1 = v1 ? causal_hidden(p, u, gid + 8) : 0;
      load_q(qw + (v0 ? query_row(p, s, u, gid) : 0) * (D / 2),
             qw + (v1 ? query_row(p, s, u, gid + 8) : 0) * (D / 2), v0, v1);
    } else {
      head0 = unit_head0(p, u_);
      const size_t row0 = (size_t(s) * p.Hq + head0 + gid) * (D / 2);
      load_q(qw + row0, qw + row0 + 8 * (D / 2), gid < gs, gid + 8 < gs);
    }
  }

  // Q fragments from the rows of this lane's two M rows (gid, gid + 8; absent rows are
  // zero), and a fresh softmax state.
  __device__ __forceinline__ void load_q(const uint32_t* r0, const uint32_t* r1, bool v0,
                                         bool v1) {
#pragma unroll
    for (int ks = 0; ks < kKS; ++ks) {
      const int w = 8 * ks + cq;  // 32-bit word index of elements 16ks + 2cq
      qa[ks][0] = v0 ? __ldg(r0 + w) : 0u;
      qa[ks][1] = v1 ? __ldg(r1 + w) : 0u;
      qa[ks][2] = v0 ? __ldg(r0 + w + 4) : 0u;
      qa[ks][3] = v1 ? __ldg(r1 + w + 4) : 0u;
    }
#pragma unroll
    for (int nd = 0; nd < kND; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
  }

  // Unnormalised (o, m, l) of the lane's two rows to explicit row addresses.
  __device__ __forceinline__ void store_rows(float* o_r0, float* o_r1, float2* ml_r0,
                                             float2* ml_r1, bool v0, bool v1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
#pragma unroll
    for (int nd = 0; nd < kND; ++nd) {
      if (v0) reinterpret_cast<float2*>(o_r0)[4 * nd + cq] = make_float2(o[nd][0], o[nd][1]);
      if (v1) reinterpret_cast<float2*>(o_r1)[4 * nd + cq] = make_float2(o[nd][2], o[nd][3]);
    }
    if (cq == 0) {
      if (v0) *ml_r0 = make_float2(m0, l0);
      if (v1) *ml_r1 = make_float2(m1, l1);
    }
  }

  __device__ __forceinline__ void block(const DecodeParams& p, uint32_t sK, uint32_t sV, uint32_t,
                                        uint32_t, int nvalid) {
    const int r8 = lane & 7, mi = lane >> 3;
    float sacc[kNT][4];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
    for (int np = 0; np < kNT / 2; ++np) {
#pragma unroll
      for (int ks = 0; ks < kKS; ++ks) {
        uint32_t b[4];
        ldmatrix_x4(b, sK + Geo::off(np * 16 + ((mi >> 1) << 3) + r8, 2 * ks + (mi & 1)));
        mma_bf16_16816(sacc[2 * np], qa[ks], b[0], b[1]);
        mma_bf16_16816(sacc[2 * np + 1], qa[ks], b[2], b[3]);
      }
    }
    // scale, mask the tokens past the context, row maxima
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tok = nt * 8 + 2 * cq + (e & 1);
        int lim = nvalid;
        if constexpr (kCausal) lim -= (e < 2) ? hide0 : hide1;
        const float x = tok < lim ? sacc[nt][e] * p.scale_log2 : -INFINITY;
        sacc[nt][e] = x;
      }
      mx0 = fmaxf(mx0, fmaxf(sacc[nt][0], sacc[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(sacc[nt][2], sacc[nt][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float mp0 = m0, mp1 = m1;
    m0 = mn0;
    m1 = mn1;
    if constexpr (kCausal) {  // a row with nothing visible yet: subtract 0, not -inf
      mn0 = mn0 == -INFINITY ? 0.f : mn0;
      mn1 = mn1 == -INFINITY ? 0.f : mn1;
    }
    const float a0 = fast_exp2(mp0 - mn0), a1 = fast_exp2(mp1 - mn1);
    l0 *= a0;
    l1 *= a1;
#pragma unroll
    for (int nd = 0; nd < kND; ++nd) {
      o[nd][0] *= a0;
      o[nd][1] *= a0;
      o[nd][2] *= a1;
      o[nd][3] *= a1;
    }
    // weights -> bf16 A fragments; the sums use the rounded weights
    uint32_t pa[kKK][4];
#pragma unroll
    for (int kk = 0; kk < kKK; ++kk) {
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) {
        const int nt = 2 * kk + hlf;
        const uint32_t w0 =
            pack_bf16x2(fast_exp2(sacc[nt][0] - mn0), fast_exp2(sacc[nt][1] - mn0));
        const uint32_t w1 =
            pack_bf16x2(fast_exp2(sacc[nt][2] - mn1), fast_exp2(sacc[nt][3] - mn1));
        pa[kk][2 * hlf] = w0;
        pa[kk][2 * hlf + 1] = w1;
        const float2 f0 = unpack_bf16x2(w0), f1 = unpack_bf16x2(w1);
        l0 += f0.x + f0.y;
        l1 += f1.x + f1.y;
      }
    }
    // rows past the context may hold anything (even NaN): zero them before P.V
    if (nvalid < BS) {
      for (int idx = lane; idx < (BS - nvalid) * Geo::kChunksPerRow; idx += 32)
        sts128_zero(sV + Geo::off(nvalid + idx / Geo::kChunksPerRow, idx % Geo::kChunksPerRow));
      __syncwarp();
    }
#pragma unroll
    for (int kk = 0; kk < kKK; ++kk) {
#pragma unroll
      for (int nd2 = 0; nd2 < kND / 2; ++nd2) {
        uint32_t b[4];
        ldmatrix_x4_trans(b, sV + Geo::off(16 * kk + ((mi & 1) << 3) + r8, 2 * nd2 + (mi >> 1)));
        mma_bf16_16816(o[2 * nd2], pa[kk], b[0], b[1]);
        mma_bf16_16816(o[2 * nd2 + 1], pa[kk], b[2], b[3]);
      }
    }
  }

  __device__ __forceinline__ void finish(const DecodeParams& p, bool complete, size_t slot) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const bool v0 = gid < gs, v1 = gid + 8 < gs;
    if (complete) {
      float i0 = 1.f / l0, i1 = 1.f / l1;
      uint32_t* out = reinterpret_cast<uint32_t*>(p.out);
      size_t row0, row1;
      if constexpr (kCausal) {
        i0 = l0 > 0.f ? i0 : 0.f;
        i1 = l1 > 0.f ? i1 : 0.f;
        row0 = (v0 ? query_row(p, s, u, gid) : 0) * (D / 2);
        row1 = (v1 ? query_row(p, s, u, gid + 8) : 0) * (D / 2);
      } else {
        row0 = (size_t(s) * p.Hq + head0 + gid) * (D / 2);
        row1 = row0 + 8 * (D / 2);
      }
#pragma unroll
      for (int nd = 0; nd < kND; ++nd) {
        if (v0) out[row0 + 4 * nd + cq] = pack_bf16x2(o[nd][0] * i0, o[nd][1] * i0);
        if (v1) out[row1 + 4 * nd + cq] = pack_bf16x2(o[nd][2] * i1, o[nd][3] * i1);
      }
    } else {
      float2* po = reinterpret_cast<float2*>(p.part_o);
      const size_t row0 = (slot * p.gs + gid) * (D / 2);
      const size_t row1 = row0 + 8 * (D / 2);
#pragma unroll
      for (int nd = 0; nd < kND; ++nd) {
        if (v0) po[row0 + 4 * nd + cq] = make_float2(o[nd][0], o[nd][1]);
        if (v1) po[row1 + 4 * nd + cq] = make_float2(o[nd][2], o[nd][3]);
      }
      if (cq == 0) {
        float2* ml = reinterpret_cast<float2*>(p.part_ml);
        if (v0) ml[slot * p.gs + gid] = make_float2(m0, l0);
        if (v1) ml[slot * p.gs + gid + 8] = make_float2(m1, l1);
      }
    }
  }
};

// ===========================================================================
// Tensor-core path, one-byte caches (fp16 MMAs on exactly widened codes)
//
// The softmax weight w in [0, 1] times the V scale becomes the fp16 A operand of
// P.V. FP8 scales are absmax/448 or absmax/57344, which would leave most weights
// in fp16's subnormal range, so the weight also carries a power of two kVUp (2^8
// for E4M3, 2^15 for E5M2: about w * absmax(v) * 0.57), undone on the output. Rows
// whose absmax exceeds about 1e5 would overflow fp16 here. INT8 keeps w * scale.
// ===========================================================================
template <int D, int BS, int CODE = CODE_I8>
struct MmaPathInt8 {
  static constexpr bool kFixup = false;  // cut units go to the merge kernel
  using Geo = TileGeom<true, D, BS>;
  using Codec = Code8<CODE>;
  static constexpr float kVUp = CODE == CODE_E5M2 ? 32768.f : CODE == CODE_E4M3 ? 256.f : 1.f;
  static constexpr float kOutScale = 1.f / kVUp;
  static constexpr int kKS = D / 16;
  static constexpr int kNT = BS / 8;
  static constexpr int kND = D / 8;
  static constexpr int kKK = BS / 16;
  static constexpr int kQB = D / 4;       // bytes of a K row each lane reads
  static constexpr int kQC = kQB / 16;    // ... as 16-byte chunks

  int lane, gid, cq, head0, s, gs;
  uint32_t qa[kKS][4];
  float o[kND][4];
  float m0, m1, l0, l1, rs0, rs1, qb0, qb1;

  __device__ __forceinline__ void init(int lane_) {
    lane = lane_;
    gid = lane >> 2;
    cq = lane & 3;
  }

  // Query rows are scaled by a power of two so that their largest entry sits near
  // 2^14 before the (then exact) narrowing from bf16 to fp16; the score scale undoes it.
  __device__ __forceinline__ void begin(const DecodeParams& p, int s_, int u) {
    s = s_;
    gs = p.gs;
    head0 = unit_head0(p, u);
    const bool v0 = gid < gs, v1 = gid + 8 < gs;
    const uint2* qd = reinterpret_cast<const uint2*>(p.q);  // 4 bf16 per uint2
    const size_t row0 = (size_t(s) * p.Hq + head0 + gid) * (D / 4);
    const size_t row1 = row0 + 8 * (D / 4);
    float f0[kKS][4], f1[kKS][4];
    float mx0 = 0.f, mx1 = 0.f;
#pragma unroll
    for (int ks = 0; ks < kKS; ++ks) {
      const int w = (kQB / 4) * cq + ks;  // elements kQB*cq + 4ks .. +3
      const uint2 a = v0 ? __ldg(qd + row0 + w) : make_uint2(0u, 0u);
      const uint2 b = v1 ? __ldg(qd + row1 + w) : make_uint2(0u, 0u);
      const float2 a01 = unpack_bf16x2(a.x), a23 = unpack_bf16x2(a.y);
      const float2 b01 = unpack_bf16x2(b.x), b23 = unpack_bf16x2(b.y);
      f0[ks][0] = a01.x; f0[ks][1] = a01.y; f0[ks][2] = a23.x; f0[ks][3] = a23.y;
      f1[ks][0] = b01.x; f1[ks][1] = b01.y; f1[ks][2] = b23.x; f1[ks][3] = b23.y;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        mx0 = fmaxf(mx0, fabsf(f0[ks][e]));
        mx1 = fmaxf(mx1, fabsf(f1[ks][e]));
      }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    int e0 = 0, e1 = 0;
    if (mx0 > 0.f) { frexpf(mx0, &e0); e0 = 14 - e0; }
    if (mx1 > 0.f) { frexpf(mx1, &e1); e1 = 14 - e1; }
    const float sc0 = ldexpf(1.f, e0), sc1 = ldexpf(1.f, e1);
    rs0 = p.scale_log2 * ldexpf(1.f, -e0);
    rs1 = p.scale_log2 * ldexpf(1.f, -e1);
#pragma unroll
    for (int ks = 0; ks < kKS; ++ks) {
      qa[ks][0] = pack_f16x2(f0[ks][0] * sc0, f0[ks][1] * sc0);
      qa[ks][1] = pack_f16x2(f1[ks][0] * sc1, f1[ks][1] * sc1);
      qa[ks][2] = pack_f16x2(f0[ks][2] * sc0, f0[ks][3] * sc0);
      qa[ks][3] = pack_f16x2(f1[ks][2] * sc1, f1[ks][3] * sc1);
    }
    // INT8 K codes enter the score MMA as c + 1152 (the biased fp16 pattern without
    // its subtraction); 1152 * sum(q row), of the fp16 q the MMA sees, comes off the
    // fp32 score instead.
    qb0 = qb1 = 0.f;
    if constexpr (CODE == CODE_I8) {
      float t0 = 0.f, t1 = 0.f;
#pragma unroll
      for (int ks = 0; ks < kKS; ++ks) {
        const float2 a = unpack_f16x2(qa[ks][0]), b = unpack_f16x2(qa[ks][2]);
        const float2 c = unpack_f16x2(qa[ks][1]), d = unpack_f16x2(qa[ks][3]);
        t0 += (a.x + a.y) + (b.x + b.y);
        t1 += (c.x + c.y) + (d.x + d.y);
      }
      t0 += __shfl_xor_sync(0xffffffffu, t0, 1);
      t0 += __shfl_xor_sync(0xffffffffu, t0, 2);
      t1 += __shfl_xor_sync(0xffffffffu, t1, 1);
      t1 += __shfl_xor_sync(0xffffffffu, t1, 2);
      qb0 = 1152.f * t0;
      qb1 = 1152.f * t1;
    }
#pragma unroll
    for (int nd = 0; nd < kND; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
  }

  __device__ __forceinline__ void block(const DecodeParams& p, uint32_t sK, uint32_t sV,
                                        uint32_t sKs, uint32_t sVs, int nvalid) {
    float sacc[kNT][4];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
      sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
      const int row = nt * 8 + gid;
#pragma unroll
      for (int ch = 0; ch < kQC; ++ch) {
        const uint4 raw = lds128(sK + Geo::off(row, kQC * cq + ch));
        const uint32_t w[4] = {Codec::pre(raw.x), Codec::pre(raw.y), Codec::pre(raw.z),
                               Codec::pre(raw.w)};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int ks = 4 * ch + k;
          if constexpr (CODE == CODE_I8)
            mma_f16_16816(sacc[nt], qa[ks], prmt(w[k], 0x64646464u, 0x4140u),
                          prmt(w[k], 0x64646464u, 0x4342u));
          else
            mma_f16_16816(sacc[nt], qa[ks], Codec::lo(w[k]), Codec::hi(w[k]));
        }
      }
    }
    float mx0 = -INFINITY, mx1 = -INFINITY;
    float kscl[kNT][2];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int tok = nt * 8 + 2 * cq + e;
        kscl[nt][e] = lds_f32(sKs + 4 * tok);
        const bool ok = tok < nvalid;
        sacc[nt][e] = ok ? (sacc[nt][e] - qb0) * kscl[nt][e] * rs0 : -INFINITY;
        sacc[nt][e + 2] = ok ? (sacc[nt][e + 2] - qb1) * kscl[nt][e] * rs1 : -INFINITY;
      }
      mx0 = fmaxf(mx0, fmaxf(sacc[nt][0], sacc[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(sacc[nt][2], sacc[nt][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float a0 = fast_exp2(m0 - mn0), a1 = fast_exp2(m1 - mn1);
    m0 = mn0;
    m1 = mn1;
    l0 *= a0;
    l1 *= a1;
#pragma unroll
    for (int nd = 0; nd < kND; ++nd) {
      o[nd][0] *= a0;
      o[nd][1] *= a0;
      o[nd][2] *= a1;
      o[nd][3] *= a1;
    }
    // weights times the V scale -> fp16 A fragments (a token past the context gets 0)
    uint32_t pa[kKK][4];
#pragma unroll
    for (int kk = 0; kk < kKK; ++kk) {
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) {
        const int nt = 2 * kk + hlf;
        float w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = fast_exp2(sacc[nt][e] - ((e < 2) ? mn0 : mn1));
        l0 += w[0] + w[1];
        l1 += w[2] + w[3];
        float vs[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int tok = nt * 8 + 2 * cq + e;
          vs[e] = tok < nvalid ? lds_f32(sVs + 4 * tok) * kVUp : 0.f;
        }
        pa[kk][2 * hlf] = pack_f16x2(w[0] * vs[0], w[1] * vs[1]);
        pa[kk][2 * hlf + 1] = pack_f16x2(w[2] * vs[0], w[3] * vs[1]);
      }
    }
#pragma unroll
    for (int kk = 0; kk < kKK; ++kk) {
      const int ta = 16 * kk + 2 * cq;
#pragma unroll
      for (int qg = 0; qg < D / 32; ++qg) {
        const int bo = 32 * qg + 4 * gid;
        const int ch = bo >> 4, wi = bo & 15;
        const uint32_t w0 = Codec::pre(lds32(sV + Geo::off(ta, ch) + wi));
        const uint32_t w1 = Codec::pre(lds32(sV + Geo::off(ta + 1, ch) + wi));
        const uint32_t w2 = Codec::pre(lds32(sV + Geo::off(ta + 8, ch) + wi));
        const uint32_t w3 = Codec::pre(lds32(sV + Geo::off(ta + 9, ch) + wi));
        const uint32_t x01 = prmt(w0, w1, 0x5140u), x23 = prmt(w0, w1, 0x7362u);
        const uint32_t y01 = prmt(w2, w3, 0x5140u), y23 = prmt(w2, w3, 0x7362u);
        mma_f16_16816(o[4 * qg + 0], pa[kk], Codec::lo(x01), Codec::lo(y01));
        mma_f16_16816(o[4 * qg + 1], pa[kk], Codec::hi(x01), Codec::hi(y01));
        mma_f16_16816(o[4 * qg + 2], pa[kk], Codec::lo(x23), Codec::lo(y23));
        mma_f16_16816(o[4 * qg + 3], pa[kk], Codec::hi(x23), Codec::hi(y23));
      }
    }
  }

  // n-tile 4qg+i, column n holds head_dim index 32qg + 4n + i, so a lane's c0 values
  // over i = 0..3 are the 4 consecutive elements 32qg + 8cq + i and its c1 values
  // the next 4.
  __device__ __forceinline__ void finish(const DecodeParams& p, bool complete, size_t slot) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const bool v0 = gid < gs, v1 = gid + 8 < gs;
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      if (!(rr == 0 ? v0 : v1)) continue;
      const int e0 = 2 * rr;
      const float lsum = rr == 0 ? l0 : l1;
      const int hrow = gid + 8 * rr;
#pragma unroll
      for (int qg = 0; qg < D / 32; ++qg) {
        float vals[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          vals[i] = o[4 * qg + i][e0];
          vals[4 + i] = o[4 * qg + i][e0 + 1];
        }
        if constexpr (kOutScale != 1.f) {
#pragma unroll
          for (int i = 0; i < 8; ++i) vals[i] *= kOutScale;
        }
        const int d0 = 32 * qg + 8 * cq;
        if (complete) {
          const float inv = 1.f / lsum;
          uint4 pk;
          pk.x = pack_bf16x2(vals[0] * inv, vals[1] * inv);
          pk.y = pack_bf16x2(vals[2] * inv, vals[3] * inv);
          pk.z = pack_bf16x2(vals[4] * inv, vals[5] * inv);
          pk.w = pack_bf16x2(vals[6] * inv, vals[7] * inv);
          __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.out) +
                               (size_t(s) * p.Hq + head0 + hrow) * D + d0;
          *reinterpret_cast<uint4*>(dst) = pk;
        } else {
          float* dst = p.part_o + (slot * p.gs + hrow) * D + d0;
          reinterpret_cast<float4*>(dst)[0] = make_float4(vals[0], vals[1], vals[2], vals[3]);
          reinterpret_cast<float4*>(dst)[1] = make_float4(vals[4], vals[5], vals[6], vals[7]);
        }
      }
      if (!complete && cq == 0)
        reinterpret_cast<float2*>(p.part_ml)[slot * p.gs + hrow] =
            make_float2(rr == 0 ? m0 : m1, lsum);
    }
  }
};

// ===========================================================================
// Work cursor over the flat (sequence, unit, block) order.
// ===========================================================================
struct Cursor {
  int s, u, j, n;  // sequence, unit of the sequence (U per sequence), block, blocks of s
};

__device__ __forceinline__ void cursor_locate(Cursor& c, long long f, const int* prefix, int B,
                                              int U) {
  int lo = 0, hi = B;  // U*prefix[lo] <= f < U*prefix[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if ((long long)U * prefix[mid] <= f) lo = mid; else hi = mid;
  }
  c.s = lo;
  c.n = prefix[lo + 1] - prefix[lo];
  const long long rem = f - (long long)U * prefix[lo];
  c.u = int(rem / c.n);
  c.j = int(rem % c.n);
}

__device__ __forceinline__ void cursor_next(Cursor& c, const int* prefix, int B, int U) {
  if (++c.j < c.n) return;
  c.j = 0;
  if (++c.u < U) return;
  c.u = 0;
  do { ++c.s; } while (c.s < B && prefix[c.s + 1] == prefix[c.s]);
  c.n = c.s < B ? prefix[c.s + 1] - prefix[c.s] : 0;
}

// ===========================================================================
// The kernel
// ===========================================================================
// kCoop = false: every warp is a worker with its own ring of stages, filled by its own
// lane 0. kCoop = true (multi-query decode): a worker is nsg warps of one CTA, one per
// row subgroup of a KV head; they share one ring, filled once per block by the first
// warp of the worker (the leader) and released by all nsg warps through an "empty"
// mbarrier per stage, so a block crosses from L2 into shared memory once per worker
// rather than once per warp.
// kBlk = 2 (16-token caches, tensor-core paths): a work item is two consecutive blocks
// of one KV head, landed by two boxes into one 32-token stage and processed as one
// tile, so per-item costs (waits, fragment set-up, row maxima, rescaling) are paid
// once per 32 tokens.
template <bool Q8, int D, int BS, class Path, int kWarps, int kStages, bool kCoop = false,
          int kBlk = 1>
struct DecodeKernel {
  using Geo = TileGeom<Q8, D, BS * kBlk>;
  static constexpr int kTile = Geo::kTileBytes;
  static constexpr int kScaleBytes = Geo::kScaleBytes;
  // per-ring shared memory: K tiles, V tiles, K/V scales, mbarriers (full[kStages],
  // then empty[kStages] for a shared ring)
  static constexpr int kOffV = kStages * kTile;
  static constexpr int kOffScale = 2 * kStages * kTile;
  static constexpr int kOffBar = kOffScale + kStages * 2 * kScaleBytes;
  static constexpr int kWarpBytes =
      ((kOffBar + (kCoop ? 2 : 1) * kStages * 8) + 1023) / 1024 * 1024;
  static constexpr uint32_t kTxBytes = 2 * kTile + 2 * kScaleBytes;
};

template <bool Q8, int D, int BS, class Path, int kWarps, int kStages, bool kCoop = false,
          int kBlk = 1>
__global__ void __launch_bounds__(kWarps * 32)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv, const DecodeParams p) {
  using K = DecodeKernel<Q8, D, BS, Path, kWarps, kStages, kCoop, kBlk>;
  constexpr int BSI = BS * kBlk;  // tokens per work item
  using Geo = typename K::Geo;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem_gen = smem_raw + (smem_base - smem_u32(smem_raw));
  const int nsg = p.nsg;
  const int wpc = kCoop ? kWarps / nsg : kWarps;  // rings (workers or warps) per CTA
  int* s_prefix = reinterpret_cast<int*>(smem_gen + wpc * K::kWarpBytes);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = p.B;
  // late_wait: the previous grid (the cascade prefix kernel, which waited for its own
  // predecessor before letting this grid start) writes nothing read here; this grid
  // only must not complete before it, so every thread waits on the way out
  const PdlWaitOnExit wait_on_exit{p.late_wait != 0};
  if (!p.late_wait) pdl_wait_prior_grid();
  if constexpr (kCoop) {  // shared rings: barriers ready before the CTA-wide sync below
    if (tid < wpc * kStages) {
      const uint32_t rb = smem_base + (tid / kStages) * K::kWarpBytes + K::kOffBar;
      mbar_init(rb + (tid % kStages) * 8, 1);
      mbar_init(rb + (kStages + tid % kStages) * 8, uint32_t(nsg));
    }
    fence_mbar_init();
  }

  // ---- blocks per sequence and their exclusive prefix (every CTA computes it) ----
  {
    const int nthr = kWarps * 32;
    const int per = (B + nthr - 1) / nthr;
    const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
    int sum = 0;
    for (int i = b0; i < b1; ++i) {
      const int L = __ldg(p.context_lens + i);
      sum += (max(0, (L <= 0 ? 0 : min((L + BS - 1) / BS, p.MBS)) - p.skip) + kBlk - 1) / kBlk;
    }
    // inclusive warp scan, then across warps
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    __shared__ int warp_tot[kWarps];
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w2 = 0; w2 < warp; ++w2) base += warp_tot[w2];
    int run = base + incl - sum;
    for (int i = b0; i < b1; ++i) {
      const int L = __ldg(p.context_lens + i);
      run += (max(0, (L <= 0 ? 0 : min((L + BS - 1) / BS, p.MBS)) - p.skip) + kBlk - 1) / kBlk;
      s_prefix[i + 1] = run;
    }
    if (tid == 0) s_prefix[0] = 0;
    __syncthreads();
    if (blockIdx.x == 0)
      for (int i = tid; i <= B; i += nthr) p.prefix_out[i] = s_prefix[i];
  }
  if (Path::kFixup && p.fixup) {  // no merge kernel follows: empty sequences get zeros here
    constexpr int Q = D / 4;
    for (int s = blockIdx.x; s < B; s += gridDim.x) {
      if (s_prefix[s + 1] != s_prefix[s]) continue;
      uint2* row = reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.out) +
                                            size_t(s) * p.Hq * D);
      for (int k = tid; k < p.Hq * Q; k += kWarps * 32) row[k] = make_uint2(0u, 0u);
    }
  }

  // Flat order (sequence, KV head, block), cut into Wg equal ranges. A worker is nsg
  // consecutive warps, one per row subgroup of the KV head: they stream the same blocks
  // at the same time, so all but the first read of a block hit L2.
  const int Hkv = p.Hkv;
  const long long T = (long long)Hkv * s_prefix[B];
  int Wg, wk, sg, ring;
  if constexpr (kCoop) {
    if (warp >= wpc * nsg) return;  // warps left over when nsg does not divide kWarps
    Wg = gridDim.x * wpc;
    wk = blockIdx.x * wpc + warp / nsg;
    sg = warp % nsg;
    ring = warp / nsg;
  } else {
    Wg = (gridDim.x * kWarps) / nsg;
    wk = (blockIdx.x * kWarps + warp) / nsg;
    sg = (blockIdx.x * kWarps + warp) % nsg;
    ring = warp;
  }
  const int w = wk * nsg + sg;  // partial slots 2w, 2w + 1
  if (wk >= Wg) return;
  const long long a = T * wk / Wg, b = T * (wk + 1) / Wg;
  if (a >= b) return;
  const int nblk = int(b - a);

  const uint32_t wbase = smem_base + ring * K::kWarpBytes;
  const bool leader = !kCoop || sg == 0;  // fills the ring
  auto sK = [&](int st) { return wbase + st * K::kTile; };
  auto sV = [&](int st) { return wbase + K::kOffV + st * K::kTile; };
  auto sKs = [&](int st) { return wbase + K::kOffScale + st * 2 * K::kScaleBytes; };
  auto sVs = [&](int st) { return sKs(st) + K::kScaleBytes; };
  auto bar = [&](int st) { return wbase + K::kOffBar + st * 8; };
  auto empty_bar = [&](int st) { return wbase + K::kOffBar + (kStages + st) * 8; };

  if (lane == 0) {
    if constexpr (!kCoop) {
      for (int st = 0; st < kStages; ++st) mbar_init(bar(st), 1);
      fence_mbar_init();
    }
    if (leader) {
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
    }
  }
  __syncwarp();

  Cursor pc, cc;  // u: the KV head
  cursor_locate(pc, a, s_prefix, B, Hkv);
  cc = pc;

  // lane 0 of the leader issues the copies of the item at the producer cursor into
  // stage st. The item's physical block ids were loaded one refill earlier (fetch_id
  // right after the cursor moved), so no table read sits on the warp's critical path.
  // A pair's second block past its sequence is an all-zero box (and, for one-byte
  // caches, takes the first block's scales: its weights are 0 but must stay finite).
  int pid[kBlk];
  int pc_s = -1, pc_nb = 0;  // sequence at the producer cursor and its blocks (pairs)
  auto fetch_id = [&]() {
    if (lane == 0 && leader && pc.s < B) {
      if constexpr (kBlk > 1) {
        if (pc.s != pc_s) {
          pc_s = pc.s;
          const int L = __ldg(p.context_lens + pc.s);
          pc_nb = (L <= 0 ? 0 : min((L + BS - 1) / BS, p.MBS)) - p.skip;
        }
      }
#pragma unroll
      for (int b = 0; b < kBlk; ++b) {
        const int blk = pc.j * kBlk + b;
        pid[b] = (kBlk == 1 || blk < pc_nb)
                     ? __ldg(p.block_tables + size_t(pc.s) * p.MBS + p.skip + blk)
                     : -1;
      }
    }
  };
  const int rows_total = p.NB * p.Hkv * BS;  // a box at this row is all zero fill
  auto issue = [&](int st) {
    if (lane == 0 && leader) {
      mbar_arrive_expect_tx(bar(st), K::kTxBytes);
      int row0 = 0;
#pragma unroll
      for (int b = 0; b < kBlk; ++b) {
        int row = rows_total;
        if (b == 0 || pid[b] >= 0) {
          const int phys = (pid[b] < 0 || pid[b] >= p.NB) ? 0 : pid[b];  // stay in the pool
          row = (phys * p.Hkv + pc.u) * BS;
        }
        if (b == 0) row0 = row;
#pragma unroll
        for (int hf = 0; hf < Geo::kHalves; ++hf) {
          const int x = hf * (Geo::kSeg / Geo::kElt);
          tma_load_2d(sK(st) + (hf * BSI + b * BS) * Geo::kSeg, &tmk, bar(st), x, row);
          tma_load_2d(sV(st) + (hf * BSI + b * BS) * Geo::kSeg, &tmv, bar(st), x, row);
        }
        if constexpr (Q8) {
          const int srow = row == rows_total ? row0 : row;
          bulk_load(sKs(st) + b * BS * 4, p.k_scale + size_t(srow), BS * 4, bar(st));
          bulk_load(sVs(st) + b * BS * 4, p.v_scale + size_t(srow), BS * 4, bar(st));
        }
      }
    }
  };

  const int npro = min(kStages, nblk);
  fetch_id();
  for (int i = 0; i < npro; ++i) {
    issue(i);
    cursor_next(pc, s_prefix, B, Hkv);
    fetch_id();
  }

  Path path;
  path.init(lane);
  path.begin(p, cc.s, cc.u * nsg + sg);
  int seg_j0 = cc.j;
  bool first_seg = true;
  int Lc = min(__ldg(p.context_lens + cc.s), p.MBS * BS);

  for (int i = 0; i < nblk; ++i) {  // nblk: work items (blocks, or pairs of blocks)
    const int st = i % kStages;
    const uint32_t par = uint32_t(i / kStages) & 1u;
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(st), par, p.timeout_ns));
    if (!ok) {
      if (lane == 0 && p.status) atomicOr(p.status, 0x4);
      // let every copy in flight land before the warp leaves its shared memory: the
      // stage that timed out (it is still owed its bytes) and the ones issued after it,
      // each with a wait of its own, also bounded
      if (leader) {
        const int issued = min(nblk, i + kStages);
        for (int k2 = i; k2 < issued; ++k2)
          mbar_wait_bounded(bar(k2 % kStages), uint32_t(k2 / kStages) & 1u, p.timeout_ns);
      }
      return;
    }
    path.block(p, sK(st), sV(st), sKs(st), sVs(st), Lc - (p.skip + cc.j * kBlk) * BS);
    __syncwarp();
    if (i + kStages < nblk) {
      fence_proxy_async_smem();  // this warp's reads of the stage before its refill
      if constexpr (kCoop) {
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(st));
        // the leader refills once every warp of the worker has released the stage
        if (leader &&
            !__all_sync(0xffffffffu, mbar_wait_bounded(empty_bar(st), par, p.timeout_ns))) {
          if (lane == 0 && p.status) atomicOr(p.status, 0x4);
          const int issued = min(nblk, i + kStages);
          for (int k2 = i + 1; k2 < issued; ++k2)
            mbar_wait_bounded(bar(k2 % kStages), uint32_t(k2 / kStages) & 1u, p.timeout_ns);
          return;
        }
      }
      issue(st);
      cursor_next(pc, s_prefix, B, Hkv);
      fetch_id();
    }
    const bool seg_end = (cc.j == cc.n - 1) || (i == nblk - 1);
    if (seg_end) {
      const bool complete = (seg_j0 == 0) && (cc.j == cc.n - 1);
      if (complete && p.unit_slot0 >= 0)  // cascade: the suffix result is one more part
        path.finish(p, false,
                    size_t(p.unit_slot0) + size_t(cc.s) * p.HU + size_t(cc.u) * nsg + sg);
      else {
        path.finish(p, complete, partial_slot(w, first_seg));
        if constexpr (Path::kFixup) {
          if (!complete && p.fixup)
            fixup_cut_unit<D>(p, s_prefix, cc.s, cc.u, cc.n, cc.j - seg_j0 + 1, T, Wg, lane);
        }
      }
      first_seg = false;
    }
    cursor_next(cc, s_prefix, B, Hkv);
    if (seg_end && i + 1 < nblk) {
      seg_j0 = cc.j;
      Lc = min(__ldg(p.context_lens + cc.s), p.MBS * BS);
      path.begin(p, cc.s, cc.u * nsg + sg);
    }
  }
}

template <bool Q8, int D, int BS, class Path, int kWarps, int kStages, bool kCoop = false,
          int kBlk = 1>
DecodeKernelInfo make_decode_info(int mma, int simt_heads) {
  DecodeKernelInfo info{};
  info.fn = reinterpret_cast<const void*>(
      &paged_decode_kernel<Q8, D, BS, Path, kWarps, kStages, kCoop, kBlk>);
  info.warps = kWarps;
  info.stages = kStages;
  info.warp_smem = DecodeKernel<Q8, D, BS, Path, kWarps, kStages, kCoop, kBlk>::kWarpBytes;
  info.blk = kBlk;
  info.mma = mma;
  info.simt_heads = simt_heads;
  info.coop = kCoop ? 1 : 0;
  info.tc = 0;
  info.fixup = Path::kFixup ? 1 : 0;
  return info;
}

}  // namespace pkv
