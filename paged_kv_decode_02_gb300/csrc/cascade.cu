// cascade.cu -- decode with a prefix shared by every sequence of the batch.
//
// Requests that share a prefix (a system prompt, few-shot examples: the prefix
// sharing of "分页注意力" in "大模型工程（五）：推理优化核心技法", chenk.top, and of
// section 2.2 of the gsyq.cn page) hold the same physical blocks at the head of their
// block tables. Every query row of a KV head then attends the same prefix keys, so for
// the prefix the B*g query rows of a KV head form a real dense contraction:
//   S = Q_rows (B*g x D) . K_prefix^T (D x P*bs),  O = softmax-weighted V_prefix.
// paged_prefix_kernel computes it once per KV head on the fifth-generation tensor cores
// (tcgen05 MMAs with operands in shared memory and accumulators in tensor memory, 128
// query rows per CTA), leaving unnormalised partials per query row. The private suffixes go
// through the ordinary decode kernel (skipping the prefix entries of the tables), and
// paged_cascade_merge_kernel folds prefix and suffix partials with the online-softmax
// rescaling. The result equals decode attention over the whole table.
#include "convert.cuh"
#include "decode.cuh"
#include "fold.cuh"
#include "tcgen05.cuh"

namespace pkv {

// ---------------------------------------------------------------------------
// Prefix kernel on the fifth-generation tensor cores. One CTA takes 128 query rows
// of one KV head and one split of the prefix, in tiles of 128 prefix tokens:
//   S_j = Q K_j^T          (tcgen05 MMA, M 128 x N 128 x K D, fp32 in TMEM, two buffers)
//   P_j = 2^(S_j*scale*log2e - m)   (softmax warps, one row per thread, bf16 to TMEM)
//   O  += P_j V_j          (tcgen05 MMA, A = P from TMEM, M 128 x N D x K 128, fp32 in TMEM)
// Roles: warps 0 and 6 issue the TMA copies of the K and the V tiles (128 tokens as
// boxes of one block x 64 columns, 128-byte swizzled; lane b copies block b, so the
// small copies of a tile leave in parallel and a score MMA never waits behind a V
// tile); warp 1 allocates TMEM and one of its threads issues every MMA; warps 2..5
// (TMEM lane quarters 2, 3, 0, 1) run the online softmax. The running reference max m
// of a row moves only when a tile's max exceeds it by more than 8 (log2 units); O in
// TMEM is then rescaled by 2^(m_old - m_new) before the next P.V accumulates, so
// weights stay below 2^8 and most tiles skip the rescale. Each split leaves per row the unnormalised (o, m, l) record that
// the cascade merge folds.
// The row sums l of the bf16 weights come from the tensor cores too (P times a tile
// of ones, issued beside P.V and rescaled with O), so the normalisation uses exactly
// the weights P.V used and the softmax warps add nothing up.
// Shared memory (1024-byte aligned): Q [D/64 slabs][128 rows x 128 B], K and V
// tiles x2 [D/64 slabs][128 tokens x 128 B], the ones tile (4 KiB), then the
// mbarriers, the TMEM address word and the split's block ids. TMEM columns: S x2
// [0, 256), O [256, 256 + D), P (bf16 pairs) [384, 448), l [448, 464).
// One-byte caches (INT8 / FP8 codes with per-(token, KV head) scales): as in the
// tcgen05 decode kernel, the producers land codes and scales, four converter warps
// (7..10) widen K codes exactly to bf16 and V to fp16 code x scale (convert.cuh), the
// softmax multiplies each score column by its K scale, and P.V runs on fp16 weights.
// ---------------------------------------------------------------------------
template <int D, int BS, bool Q8 = false>
struct PrefixTc {
  static constexpr int kM = 128;                      // query rows per CTA
  static constexpr int kN = 128;                      // prefix tokens per tile
  static constexpr int kBlocks = kN / BS;             // blocks per tile
  static constexpr int kSlabs = D / 64;               // 128-byte column slabs of a row
  static constexpr int kSlab = kN * 128;              // one slab of a K or V tile
  static constexpr int kQSlab = kM * 128;
  static constexpr int kTile = kSlabs * kSlab;        // a K or V tile
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kSlabs * kQSlab;
  static constexpr int kOffV = kOffK + 2 * kTile;
  // all-ones B operand (16 x 128 tokens, K-major) of the MMA that sums the rows of P
  static constexpr int kOffOnes = kOffV + 2 * kTile;
  // one-byte caches: codes in the last kCodeTile bytes of a tile's buffer; scales in kN
  // fp32 slots, K scales of tile j in slot j % 4, V scales in slot 4 + j % 2
  static constexpr int kCodeTile = kN * D;
  static constexpr int kCodeOff = kTile - kCodeTile;
  static constexpr int kScaleBytes = kN * 4;
  static constexpr int kOffScales = kOffOnes + 4096;
  static constexpr int kOffBar = kOffScales + (Q8 ? 6 * kScaleBytes : 0);
  // mbarriers: kfull[2] kempty[2] vfull[2] vempty[2] sfull[2] pfull ofull mdone
  // (+ one-byte caches: kstage[2] vstage[2] kscale[4])
  static constexpr int kNumBars = Q8 ? 21 : 13;
  static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kMaxIds = 2048;                // prefix blocks per split (planner cap)
  static constexpr int kOffIds = kOffAbort + 4;
  static constexpr int kSmem = kOffIds + 4 * kMaxIds + 1024;  // + slack for 1024-byte alignment
  // warps: 0 K copies, 1 MMA, 2..5 softmax, 6 V copies (+ 7..10 converters)
  static constexpr int kThreads = Q8 ? 352 : 224;
  static constexpr uint32_t kTmemCols = 512;          // power of two
  // S x2, O, P (bf16 pairs), l (row sums of P, fp32; 16 columns written by its MMA)
  static constexpr int kColS = 0, kColO = 2 * kN, kColP = 2 * kN + 128, kColL = kColP + kN / 2;
  static_assert(kColL + 16 <= int(kTmemCols) && kColO + D <= kColP, "TMEM columns");
  static_assert(kOffOnes % 1024 == 0, "swizzle atom alignment");
  static_assert(kSmem <= 227 * 1024, "shared memory");
  static_assert(kN % BS == 0 && D % 64 == 0, "tile shape");
  static_assert(kQSlab == kSlab, "Q, K and P slabs share one stride");
  static_assert(kMaxIds % kBlocks == 0, "split cap in whole tiles");
};

// CODE: -1 for bf16 caches, else the one-byte code format.
template <int D, int BS, int CODE = -1>
__global__ void __launch_bounds__(PrefixTc<D, BS, (CODE >= 0)>::kThreads, 1)
    paged_prefix_kernel(const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv, const PrefixParams pp) {
  constexpr bool kQ8 = CODE >= 0;
  using K = PrefixTc<D, BS, kQ8>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  volatile int* abort_flag =
      reinterpret_cast<volatile int*>(smem_raw + (base - raw) + K::kOffAbort);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.y, z = blockIdx.z;
  const int row0 = blockIdx.x * K::kM;
  const int b0 = z * pp.per_split, b1 = min(pp.P, b0 + pp.per_split);
  const int nb = max(0, b1 - b0);
  const int ntiles = (nb + K::kBlocks - 1) / K::kBlocks;
  auto bar = [&](int i) { return base + K::kOffBar + 8 * i; };
  auto kfull = [&](int st) { return bar(st); };
  auto kempty = [&](int st) { return bar(2 + st); };
  auto vfull = [&](int st) { return bar(4 + st); };
  auto vempty = [&](int st) { return bar(6 + st); };
  auto sfull = [&](int st) { return bar(8 + st); };
  const uint32_t pfull = bar(10), ofull = bar(11), mdone = bar(12);
  auto kstage = [&](int st) { return bar(13 + st); };
  auto vstage = [&](int st) { return bar(15 + st); };
  auto kscale = [&](int j) { return bar(17 + (j & 3)); };
  auto scale_area = [&](bool is_k, int j) {
    return base + K::kOffScales + uint32_t(is_k ? (j & 3) : 4 + (j & 1)) * K::kScaleBytes;
  };
  const uint32_t tmem_slot = base + K::kOffTmemSlot;

  pdl_wait_prior_grid();
  // the suffix decode reads nothing this kernel writes: with its late wait it may start
  // now, on the SMs this grid leaves free
  if (pp.overlap) pdl_allow_next_grid();
  if (tid == 0) {
    for (int i = 0; i < 10; ++i) mbar_init(bar(i), 1);
    mbar_init(pfull, 4 * 32);
    mbar_init(ofull, 1);
    mbar_init(mdone, 1);
    if constexpr (kQ8)
      for (int i = 13; i < 21; ++i) mbar_init(bar(i), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, K::kTmemCols);
  for (int k = tid; k < 4096 / 16; k += K::kThreads)  // 1.0 everywhere (bf16, or fp16)
    tc::sts128(base + K::kOffOnes + 16 * k,
               kQ8 ? make_uint4(0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u)
                   : make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u));

  // this split's physical block ids -> shared memory (the producer's copies then need
  // no dependent global load)
  int* s_ids = reinterpret_cast<int*>(smem_raw + (base - raw) + K::kOffIds);
  for (int i = tid; i < min(nb, K::kMaxIds); i += K::kThreads)
    s_ids[i] = __ldg(pp.prefix_ids + b0 + i);
  // Q rows of this CTA -> shared memory as the K-major A operand (zero rows past R);
  // every load is issued before the first store
  {
    const uint4* q = reinterpret_cast<const uint4*>(pp.q);
    constexpr int kChunks = D / 8;  // 16-byte chunks per row
    constexpr int kIters = (K::kM * kChunks + K::kThreads - 1) / K::kThreads;
    uint4 v[kIters];
#pragma unroll
    for (int it = 0; it < kIters; ++it) {
      const int c = tid + it * K::kThreads;
      const int r = c / kChunks, cc = c % kChunks;
      const int gr = row0 + r;
      v[it] = make_uint4(0u, 0u, 0u, 0u);
      if (c < K::kM * kChunks && gr < pp.R) {
        const int s = gr / pp.g, i = gr % pp.g;
        v[it] = __ldg(q + (size_t(s) * pp.Hq + h * pp.g + i) * kChunks + cc);
      }
    }
#pragma unroll
    for (int it = 0; it < kIters; ++it) {
      const int c = tid + it * K::kThreads;
      const int r = c / kChunks, cc = c % kChunks;
      if (c < K::kM * kChunks)
        tc::sts128(base + K::kOffQ + (cc >> 3) * K::kQSlab + r * 128 + (((cc & 7) ^ (r & 7)) << 4),
               v[it]);
    }
  }
  fence_proxy_async_smem();  // Q (generic-proxy writes) before the MMAs read it
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem_raw + (base - raw) +
                                                             K::kOffTmemSlot);

  if (warp == 0 || warp == 6) {
    // ---------------- TMA producers: warp 0 streams K, warp 6 streams V ----------------
    // lane b issues the copies of block b of a tile, so a tile's copies leave together
    const bool is_k = warp == 0;
    const CUtensorMap* map = is_k ? &tmk : &tmv;
    const uint32_t region = base + (is_k ? K::kOffK : K::kOffV);
    const int rows_total = pp.NB * pp.Hkv * BS;  // a box at this row is all zero fill
    int issued = 0;
    // the barrier a tile's copies complete on: the tile itself (bf16), or the staged
    // codes and scales the converters wait for (one-byte caches)
    auto copy_bar = [&](int st) {
      return kQ8 ? (is_k ? kstage(st) : vstage(st)) : (is_k ? kfull(st) : vfull(st));
    };
    for (int j = 0; j < ntiles; ++j) {
      const int st = j & 1;
      const uint32_t fb = copy_bar(st);
      if (j >= 2 &&
          !__all_sync(0xffffffffu, tc::wait_or_abort(is_k ? kempty(st) : vempty(st),
                                               uint32_t((j >> 1) - 1) & 1u, pp.timeout_ns,
                                               abort_flag)))
        break;
      if (lane == 0) mbar_arrive_expect_tx(fb, kQ8 ? K::kCodeTile + K::kScaleBytes : K::kTile);
      __syncwarp();
      int row = rows_total;
      if (lane < K::kBlocks) {
        const int i = j * K::kBlocks + lane;  // block of the split
        if (i < nb) {
          int phys = s_ids[i];
          phys = (phys < 0 || phys >= pp.NB) ? 0 : phys;  // never copy outside the pool
          row = (phys * pp.Hkv + h) * BS;
        }
      }
      if constexpr (kQ8) {
        // a block past the split copies zero-filled codes and block 0's scales
        const int row0 = __shfl_sync(0xffffffffu, row, 0);
        if (lane < K::kBlocks) {
          tma_load_2d(region + st * K::kTile + K::kCodeOff + lane * BS * D, map, fb, 0, row);
          bulk_load(scale_area(is_k, j) + lane * BS * 4,
                    (is_k ? pp.k_scale : pp.v_scale) + size_t(row == rows_total ? row0 : row),
                    BS * 4, fb);
        }
      } else if (lane < K::kBlocks) {
        const uint32_t dst = region + st * K::kTile + lane * BS * 128;
#pragma unroll
        for (int sl = 0; sl < K::kSlabs; ++sl)
          tma_load_2d(dst + sl * K::kSlab, map, fb, sl * 64, row);
      }
      issued = j + 1;
    }
    // every copy issued must have landed before the CTA may exit
    if (lane == 0)
      for (int j = max(0, issued - 2); j < issued; ++j)
        mbar_wait_bounded(copy_bar(j & 1), uint32_t(j >> 1) & 1u, pp.timeout_ns);
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t kIdS = tc::idesc_bf16<128, K::kN, false>();
      // P.V and the row sums run on fp16 weights and values for one-byte caches
      constexpr uint32_t kIdO =
          kQ8 ? tc::idesc_f16<128, D, true>() : tc::idesc_bf16<128, D, true>();
      constexpr uint32_t kIdL =
          kQ8 ? tc::idesc_f16<128, 16, false>() : tc::idesc_bf16<128, 16, false>();
      // shared-memory descriptors built once and advanced by offset / 16 (the start
      // address field, as in the tcgen05 decode kernel)
      constexpr uint32_t kTileDesc = K::kTile >> 4, kSlabDesc = K::kSlab >> 4;
      const uint64_t desc_q = tc::sdesc_sw128(base + K::kOffQ, 16, 1024);
      const uint64_t desc_k = tc::sdesc_sw128(base + K::kOffK, 16, 1024);
      const uint64_t desc_v = tc::sdesc_sw128(base + K::kOffV, K::kSlab, 1024);
      const uint64_t desc_ones = tc::sdesc_sw128(base + K::kOffOnes, 16, 1024);
      auto mma_s = [&](int j) {
        const int st = j & 1;
        tc::fence_after_sync();
        const uint64_t kd = desc_k + st * kTileDesc;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ko = (kk >> 2) * kSlabDesc + (kk & 3) * 2;  // kQSlab == kSlab
          tc::mma_bf16(tmem + K::kColS + st * K::kN, desc_q + ko, kd + ko, kIdS, kk > 0 ? 1u : 0u);
        }
        tc::commit(sfull(st));
        tc::commit(kempty(st));
      };
      auto mma_pv = [&](int j) {
        const int st = j & 1;
        tc::fence_after_sync();
        const uint64_t vd = desc_v + st * kTileDesc;
#pragma unroll
        for (int kk = 0; kk < K::kN / 16; ++kk) {
          // A = P in TMEM (8 columns per 16 tokens), B = V (MN-major: D contiguous,
          // tokens as rows)
          tc::mma_bf16_tmem_a(tmem + K::kColO, tmem + K::kColP + kk * 8, vd + kk * 128, kIdO,
                              (j > 0 || kk > 0) ? 1u : 0u);
          // the row sums of the bf16 weights this P.V used (P times the ones tile)
          tc::mma_bf16_tmem_a(tmem + K::kColL, tmem + K::kColP + kk * 8,
                              desc_ones + (kk >> 2) * 128 + (kk & 3) * 2, kIdL,
                              (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc::commit(vempty(st));
        tc::commit(ofull);
      };
      // MMAs go out in the order their inputs become ready (as in the tcgen05 decode
      // kernel): S_ns once K_ns has landed and softmax pass ns - 2 is observed (its score
      // buffer free), PV_np once pass np is observed and V_np has landed. Pass i + 1
      // cannot complete before PV_i, so no barrier runs two phases past the one polled.
      int ns = 0, np = 0, pdone = 0;
      uint32_t idle = 0;
      uint64_t t_idle = 0;
      while (np < ntiles) {
        bool prog = false;
        if (pdone < ns && mbar_test_wait(pfull, uint32_t(pdone) & 1u)) {
          ++pdone;
          prog = true;
        }
        if (np < pdone && mbar_test_wait(vfull(np & 1), uint32_t(np >> 1) & 1u)) {
          mma_pv(np);
          ++np;
          prog = true;
        }
        if (ns < ntiles && pdone + 1 >= ns &&
            mbar_test_wait(kfull(ns & 1), uint32_t(ns >> 1) & 1u)) {
          mma_s(ns);
          ++ns;
          prog = true;
        }
        if (prog) {
          idle = 0;
        } else {  // bounded like every other wait: give up on a timeout or another abort
          if (idle == 0) t_idle = global_timer_ns();
          if ((++idle & 63u) == 0u) {
            if (*abort_flag) break;
            if (global_timer_ns() - t_idle > pp.timeout_ns) {
              *abort_flag = 1;
              break;
            }
          }
        }
      }
      // every MMA issued must have completed before TMEM is freed
      tc::commit(mdone);
      mbar_wait_bounded(mdone, 0u, pp.timeout_ns);
    }
    __syncwarp();
  } else if (warp >= 2 && warp <= 5) {
    // ---------------- softmax warps (2..5): one query row per thread ----------------
    const int quarter = warp & 3;  // warps 2, 3, 4, 5 own TMEM lanes 64.., 96.., 0.., 32..
    const int r = quarter * 32 + lane;
    const uint32_t trow = tmem + (uint32_t(quarter * 32) << 16);
    const float sl = pp.scale_log2;
    float m_ref = -INFINITY;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int st = j & 1;
      if (!__all_sync(0xffffffffu,
                      tc::wait_or_abort(sfull(st), uint32_t(j >> 1) & 1u, pp.timeout_ns,
                                        abort_flag))) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      uint32_t s[K::kN];
      tc::tmem_ld128(trow + K::kColS + st * K::kN, s);
      if constexpr (kQ8) {  // one-byte caches: each column times its K scale
        if (!__all_sync(0xffffffffu, tc::wait_or_abort(kscale(j), uint32_t(j >> 2) & 1u,
                                                       pp.timeout_ns, abort_flag))) {
          ok = false;
          break;
        }
        const uint32_t ks = scale_area(true, j);
#pragma unroll
        for (int t = 0; t < K::kN; t += 4) {
          const uint4 k4 = lds128(ks + 4 * t);  // the same address in every lane
          s[t] = __float_as_uint(__uint_as_float(s[t]) * __uint_as_float(k4.x));
          s[t + 1] = __float_as_uint(__uint_as_float(s[t + 1]) * __uint_as_float(k4.y));
          s[t + 2] = __float_as_uint(__uint_as_float(s[t + 2]) * __uint_as_float(k4.z));
          s[t + 3] = __float_as_uint(__uint_as_float(s[t + 3]) * __uint_as_float(k4.w));
        }
      }
      // scores of masked columns (past the split, zero-filled K) never count; a
      // negative scale is carried by flipping the scores' signs (warp-uniform branches,
      // taken only on a split's last tile or with scale < 0)
      const int valid = min(K::kBlocks, nb - j * K::kBlocks) * BS;
      if (sl < 0.f) {
#pragma unroll
        for (int t = 0; t < K::kN; ++t) s[t] ^= 0x80000000u;
      }
      if (valid < K::kN) {
#pragma unroll
        for (int t = 0; t < K::kN; ++t)
          if (t >= valid) s[t] = 0xff800000u;  // -inf
      }
      const float asl = fabsf(sl);
      // tile maximum: three-input max over eight independent chains
      float mx[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx[e] = __uint_as_float(s[e]);
#pragma unroll
      for (int u = 0; u < (K::kN - 8) / 2; ++u)
        mx[u & 7] = fmax3(mx[u & 7], __uint_as_float(s[8 + 2 * u]), __uint_as_float(s[9 + 2 * u]));
      const float mt = asl * fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                   fmaxf(mx[6], mx[7]));
      float alpha = 1.f;
      bool rescale = false;
      if (mt > m_ref + 8.f) {
        alpha = fast_exp2(m_ref - mt);  // 0 on the first tile
        m_ref = mt;
        rescale = j > 0;
      }
      // weights 2^(scale * s - m) (packed fp32x2 FMAs), bf16 pairs; their row sums come
      // from the tensor cores (P times the ones tile, beside P.V)
      uint32_t pk[K::kN / 2];
      const float2 asl2 = make_float2(asl, asl), nm2 = make_float2(-m_ref, -m_ref);
      if (valid == K::kN) {
#pragma unroll
        for (int t = 0; t < K::kN; t += 2) {
          const float2 x = __ffma2_rn(make_float2(__uint_as_float(s[t]), __uint_as_float(s[t + 1])),
                                      asl2, nm2);
          pk[t / 2] = kQ8 ? pack_f16x2(fast_exp2(x.x), fast_exp2(x.y))
                          : pack_bf16x2(fast_exp2(x.x), fast_exp2(x.y));
        }
      } else {
#pragma unroll
        for (int t = 0; t < K::kN; t += 2) {
          const float2 x = __ffma2_rn(make_float2(__uint_as_float(s[t]), __uint_as_float(s[t + 1])),
                                      asl2, nm2);
          const float w0 = t < valid ? fast_exp2(x.x) : 0.f;
          const float w1 = t + 1 < valid ? fast_exp2(x.y) : 0.f;
          pk[t / 2] = kQ8 ? pack_f16x2(w0, w1) : pack_bf16x2(w0, w1);
        }
      }
      // P.V of the previous tile must be complete before P is overwritten or O rescaled
      if (j > 0 && !__all_sync(0xffffffffu, tc::wait_or_abort(ofull, uint32_t(j - 1) & 1u,
                                                        pp.timeout_ns, abort_flag))) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tc::tmem_ld32(trow + K::kColO + c, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tc::tmem_st32(trow + K::kColO + c, o);
        }
        tc::tmem_st1(trow + K::kColL,
                     __float_as_uint(__uint_as_float(tc::tmem_ld1(trow + K::kColL)) * alpha));
      }
      // P row -> TMEM (bf16 pairs of consecutive tokens), the A operand of P.V
#pragma unroll
      for (int c = 0; c < K::kN / 2; c += 32) {
        uint32_t w[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) w[e] = pk[c + e];
        tc::tmem_st32(trow + K::kColP + c, w);
      }
      tc::fence_before_sync();
      mbar_arrive(pfull);
    }
    if (ok && ntiles > 0 &&
        !__all_sync(0xffffffffu, tc::wait_or_abort(ofull, uint32_t(ntiles - 1) & 1u, pp.timeout_ns,
                                             abort_flag)))
      ok = false;
    tc::fence_after_sync();
    const int gr = row0 + r;
    const size_t rec = size_t(z * pp.Hkv + h) * pp.R + gr;
    float4* dst = reinterpret_cast<float4*>(pp.pre_o + rec * D);
#pragma unroll
    for (int c = 0; c < D; c += 32) {
      uint32_t o[32];
      if (ok && ntiles > 0) {
        tc::tmem_ld32(trow + K::kColO + c, o);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0u;
      }
      if (gr < pp.R) {
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          dst[(c + e) / 4] = make_float4(__uint_as_float(o[e]), __uint_as_float(o[e + 1]),
                                         __uint_as_float(o[e + 2]), __uint_as_float(o[e + 3]));
      }
    }
    const float l = (ok && ntiles > 0) ? __uint_as_float(tc::tmem_ld1(trow + K::kColL)) : 0.f;
    if (gr < pp.R)
      reinterpret_cast<float2*>(pp.pre_ml)[rec] =
          (ok && ntiles > 0) ? make_float2(m_ref, l) : make_float2(-INFINITY, 0.f);
    tc::fence_before_sync();
  } else if (kQ8) {
    // ---------------- converters (7..10): one-byte codes -> 16-bit values ----------------
    const int ct = tid - 7 * 32;
    for (int j = 0; j < ntiles; ++j) {
      const int st = j & 1;
      const uint32_t par = uint32_t(j >> 1) & 1u;
      const int valid = min(K::kBlocks, nb - j * K::kBlocks) * BS;  // tokens of the split
      bool go = true;
      for (int kv = 0; kv < 2; ++kv) {
        // every converter takes part in every barrier: they agree on going on first
        const bool landed = __all_sync(
            0xffffffffu,
            tc::wait_or_abort(kv == 0 ? kstage(st) : vstage(st), par, pp.timeout_ns, abort_flag));
        if (!converters_all(landed)) {
          go = false;
          break;
        }
        // K: the codes themselves as bf16 (exact; the softmax applies the K scales);
        // V: code x scale as fp16
        if constexpr (kQ8) {
          const uint32_t tile = base + (kv == 0 ? K::kOffK : K::kOffV) + st * K::kTile;
          if (kv == 0) {
            convert_codes<D, (kQ8 ? CODE : 0), false, false>(tile, scale_area(true, j), valid,
                                                             ct);
            if (ct >= valid) tc::sts32(scale_area(true, j) + 4 * ct, 0u);
          } else {
            convert_codes<D, (kQ8 ? CODE : 0), true, true>(tile, scale_area(false, j), valid,
                                                           ct);
          }
        }
        fence_proxy_async_smem();  // the 16-bit values, for the MMAs (async proxy)
        converters_sync();
        if (ct == 0) {
          mbar_arrive(kv == 0 ? kfull(st) : vfull(st));
          if (kv == 0) mbar_arrive(kscale(j));
        }
      }
      if (!go) break;
    }
  }
  __syncthreads();
  if (*abort_flag && tid == 0 && pp.status) atomicOr(pp.status, 0x4);
  if (warp == 1) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, K::kTmemCols);
  }
}

template <int D, int BS, int CODE>
void prefix_info(PrefixKernelInfo* info) {
  using K = PrefixTc<D, BS, (CODE >= 0)>;
  info->fn = reinterpret_cast<const void*>(&paged_prefix_kernel<D, BS, CODE>);
  info->smem = K::kSmem;
  info->threads = K::kThreads;
  info->rows = K::kM;
  info->tile_blocks = K::kBlocks;
  info->max_split_blocks = K::kMaxIds;
}

template <int CODE>
bool select_prefix_code(int D, int BS, PrefixKernelInfo* info) {
  if (D == 128 && BS == 16) prefix_info<128, 16, CODE>(info);
  else if (D == 128 && BS == 32) prefix_info<128, 32, CODE>(info);
  else if (D == 64 && BS == 16) prefix_info<64, 16, CODE>(info);
  else if (D == 64 && BS == 32) prefix_info<64, 32, CODE>(info);
  else return false;
  return true;
}

bool select_prefix_kernel(int D, int BS, int kvt, PrefixKernelInfo* info) {
  switch (kvt) {
    case PKV_KV_BF16: return select_prefix_code<-1>(D, BS, info);
    case PKV_KV_INT8: return select_prefix_code<CODE_I8>(D, BS, info);
    case PKV_KV_FP8_E4M3: return select_prefix_code<CODE_E4M3>(D, BS, info);
    case PKV_KV_FP8_E5M2: return select_prefix_code<CODE_E5M2>(D, BS, info);
    default: return false;
  }
}

// ---------------------------------------------------------------------------
// Cascade merge: one warp per (sequence, unit), one 16-byte output quad per lane and
// row, folds the nsplit prefix partials of the unit's rows and the suffix parts (the
// unit's own record when one decode worker covered the whole suffix, else the cut
// workers' slots). With a status word it first validates the sequence:
// context length in [prefix, max_blocks*block_size], block ids in the pool, and the
// table's head equal to the shared prefix (row 0); a sequence that fails gets a zero
// output.
// ---------------------------------------------------------------------------
constexpr int kCascadeWarps = 8;  // one (sequence, unit) per warp

__global__ void __launch_bounds__(kCascadeWarps * 32)
    paged_cascade_merge_kernel(const CascadeMergeParams p) {
  pdl_wait_prior_grid();
  const int lane = threadIdx.x & 31;
  const int gs = p.gs, D = p.D, Q = D / 4;
  const int rpw = 32 / Q;                    // rows per warp step: one quad per lane
  const int nsteps = (gs + rpw - 1) / rpw;   // steps over the unit's rows
  const int unit = blockIdx.x * kCascadeWarps + (threadIdx.x >> 5);
  if (unit >= p.B * p.HU) return;
  const int s = unit / p.HU, u = unit % p.HU;
  const int h = u / p.nsg, sg = u % p.nsg;
  const int dq = lane % Q;
  auto out_quad = [&](int row) {
    return reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.out) +
                                    (size_t(s) * p.Hq + h * p.g + sg * gs + row) * D) +
           dq;
  };

  if (p.status != nullptr) {
    int flags = 0;
    const int L = p.context_lens[s];
    if (lane == 0 && (L < p.P * p.BS || L > p.MBS * p.BS)) flags |= (L < p.P * p.BS) ? 0x8 : 0x1;
    const int n = L <= 0 ? 0 : min((L + p.BS - 1) / p.BS, p.MBS);
    for (int j = lane; j < n; j += 32) {
      const int id = p.block_tables[size_t(s) * p.MBS + j];
      if (id < 0 || id >= p.NB) flags |= 0x2;
      if (j < p.P && id != p.block_tables[j]) flags |= 0x8;
    }
    flags = __reduce_or_sync(0xffffffffu, flags);
    if (flags) {
      if (lane == 0 && u == 0) atomicOr(p.status, flags);
      for (int k = 0; k < nsteps; ++k) {
        const int row = k * rpw + lane / Q;
        if (row < gs) *out_quad(row) = make_uint2(0u, 0u);
      }
      return;
    }
  }

  // the parts: nsplit prefix records, then the suffix parts
  // suffix parts: the decode kernel's flat order is (sequence, KV head, block) over Wg
  // workers of nsg warps; this unit's parts come from warp worker * nsg + sg
  const int n = p.prefix[s + 1] - p.prefix[s];
  const long long T = (long long)p.Hkv * p.prefix[p.B];
  const int Wg = p.Wg;
  int nsuf = 0, w0 = 0;
  bool dense = true, first_cut = false, whole = false;
  long long A = 0;
  if (n > 0) {
    A = (long long)p.Hkv * p.prefix[s] + (long long)h * n;
    w0 = int(((A + 1) * Wg + T - 1) / T) - 1;
    const int w1 = int(((A + n) * Wg + T - 1) / T) - 1;
    whole = (w0 == w1);
    dense = T >= Wg;
    nsuf = whole ? 1 : (dense ? (w1 - w0 + 1) : n);
    first_cut = (T * w0 / Wg) != A;
  }
  const int nparts = p.nsplit + nsuf;
  const float2* pre_ml = reinterpret_cast<const float2*>(p.pre_ml);
  const float2* part_ml = reinterpret_cast<const float2*>(p.part_ml);
  // up to four row steps at a time, every load of a chunk in flight together
  constexpr int kRows = 4;
  for (int k0 = 0; k0 < nsteps; k0 += kRows) {
    const int kn = min(kRows, nsteps - k0);
    Fold f[kRows];
#pragma unroll
    for (int k = 0; k < kRows; ++k) f[k] = fold_empty();
    fold_rows<kRows, 2>(f, kn, nparts, [&](int i, int k, const float2*& pm, const float4*& po) {
      const int row = min((k0 + k) * rpw + lane / Q, gs - 1);  // rows past gs: not stored
      if (i < p.nsplit) {
        const size_t rec = size_t(i * p.Hkv + h) * p.R + size_t(s) * p.g + size_t(sg) * gs + row;
        pm = pre_ml + rec;
        po = reinterpret_cast<const float4*>(p.pre_o + rec * D) + dq;
        return;
      }
      const int kk = i - p.nsplit;
      size_t slot;
      if (whole) slot = size_t(2 * p.W) + size_t(s) * p.HU + u;
      else if (dense)
        slot = size_t(2 * ((w0 + kk) * p.nsg + sg) + ((kk == 0 && first_cut) ? 1 : 0));
      else slot = size_t(2 * ((int(((A + kk + 1) * Wg + T - 1) / T) - 1) * p.nsg + sg));
      pm = part_ml + slot * gs + row;
      po = reinterpret_cast<const float4*>(p.part_o + (slot * gs + row) * D) + dq;
    });
#pragma unroll
    for (int k = 0; k < kRows; ++k) {
      const int row = (k0 + k) * rpw + lane / Q;
      if (k < kn && row < gs) *out_quad(row) = fold_result(f[k]);
    }
  }
}

void launch_cascade_merge(const CascadeMergeParams& p, cudaStream_t stream) {
  const long long units = (long long)p.B * p.HU;
  if (units <= 0) return;
  const int grid = int((units + kCascadeWarps - 1) / kCascadeWarps);
  CascadeMergeParams copy = p;
  void* args[] = {&copy};
  launch_pdl(reinterpret_cast<const void*>(&paged_cascade_merge_kernel), dim3(grid),
             dim3(kCascadeWarps * 32), args, 0, stream);
}

}  // namespace pkv
