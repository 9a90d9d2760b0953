// fold.cuh -- online-softmax folding of unnormalised partial results.
//
// A part covering some of a row's tokens holds m = max_t x_t (scores in log2 units),
// l = sum_t 2^(x_t - m) and o = sum_t 2^(x_t - m) v_t. Parts fold with the
// online-softmax rescaling: with M the largest m so far, l = sum 2^(m_i - M) l_i and
// o = sum 2^(m_i - M) o_i; the row's result is o / l. A part that saw no token has
// m = -inf and adds nothing; a row no part saw gives zeros.
#pragma once

#include "common.cuh"

namespace pkv {

struct Fold {
  float m, l;
  float4 o;
};

__device__ __forceinline__ Fold fold_empty() {
  return Fold{-INFINITY, 0.f, make_float4(0.f, 0.f, 0.f, 0.f)};
}

__device__ __forceinline__ void fold_scale(Fold& f, float r) {
  f.l *= r;
  f.o.x *= r;
  f.o.y *= r;
  f.o.z *= r;
  f.o.w *= r;
}

// Folds parts first, first + stride, ... (< nparts) of one output quad. part(i)
// returns the part's (m, l) pointer and its output quad pointer. Up to kChunk parts
// are loaded before any is used, so their loads are in flight together; the running
// maximum moves once per chunk.
template <int kChunk, class PartFn>
__device__ __forceinline__ void fold_parts(Fold& f, int first, int stride, int nparts,
                                           PartFn part) {
  for (int i0 = first; i0 < nparts; i0 += kChunk * stride) {
    float2 v[kChunk];
    float4 x[kChunk];
#pragma unroll
    for (int k = 0; k < kChunk; ++k) {
      const int i = i0 + k * stride;
      v[k] = make_float2(-INFINITY, 0.f);
      x[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < nparts) {
        const float2* ml;
        const float4* o;
        part(i, ml, o);
        v[k] = *ml;
        x[k] = *o;
      }
    }
    float cm = v[0].x;
#pragma unroll
    for (int k = 1; k < kChunk; ++k) cm = fmaxf(cm, v[k].x);
    if (cm > f.m) {
      fold_scale(f, fast_exp2(f.m - cm));  // 0 while nothing was folded in
      f.m = cm;
    }
#pragma unroll
    for (int k = 0; k < kChunk; ++k) {
      const float e = v[k].x > -INFINITY ? fast_exp2(v[k].x - f.m) : 0.f;
      f.l = fmaf(e, v[k].y, f.l);
      f.o.x = fmaf(e, x[k].x, f.o.x);
      f.o.y = fmaf(e, x[k].y, f.o.y);
      f.o.z = fmaf(e, x[k].z, f.o.z);
      f.o.w = fmaf(e, x[k].w, f.o.w);
    }
  }
}

// fold_parts for up to kRows rows at once (nrows of them live): the chunk's loads of
// every row are issued before any is used. part(i, k) returns part i of row k.
// kL2: load through L2 only (parts other CTAs wrote during the same launch).
template <int kRows, int kChunk, bool kL2 = false, class PartFn>
__device__ __forceinline__ void fold_rows(Fold (&f)[kRows], int nrows, int nparts,
                                          PartFn part) {
  for (int i0 = 0; i0 < nparts; i0 += kChunk) {
    float2 v[kRows][kChunk];
    float4 x[kRows][kChunk];
#pragma unroll
    for (int k = 0; k < kRows; ++k) {
#pragma unroll
      for (int c = 0; c < kChunk; ++c) {
        const int i = i0 + c;
        v[k][c] = make_float2(-INFINITY, 0.f);
        x[k][c] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (k < nrows && i < nparts) {
          const float2* ml;
          const float4* o;
          part(i, k, ml, o);
          v[k][c] = kL2 ? __ldcg(ml) : *ml;
          x[k][c] = kL2 ? __ldcg(o) : *o;
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kRows; ++k) {
      float cm = v[k][0].x;
#pragma unroll
      for (int c = 1; c < kChunk; ++c) cm = fmaxf(cm, v[k][c].x);
      if (cm > f[k].m) {
        fold_scale(f[k], fast_exp2(f[k].m - cm));
        f[k].m = cm;
      }
#pragma unroll
      for (int c = 0; c < kChunk; ++c) {
        const float e = v[k][c].x > -INFINITY ? fast_exp2(v[k][c].x - f[k].m) : 0.f;
        f[k].l = fmaf(e, v[k][c].y, f[k].l);
        f[k].o.x = fmaf(e, x[k][c].x, f[k].o.x);
        f[k].o.y = fmaf(e, x[k][c].y, f[k].o.y);
        f[k].o.z = fmaf(e, x[k][c].z, f[k].o.z);
        f[k].o.w = fmaf(e, x[k][c].w, f[k].o.w);
      }
    }
  }
}

// Adds another running fold.
__device__ __forceinline__ void fold_merge(Fold& f, const Fold& g) {
  if (!(g.m > -INFINITY)) return;
  if (g.m > f.m) {
    fold_scale(f, fast_exp2(f.m - g.m));
    f.m = g.m;
  }
  const float e = fast_exp2(g.m - f.m);
  f.l = fmaf(e, g.l, f.l);
  f.o.x = fmaf(e, g.o.x, f.o.x);
  f.o.y = fmaf(e, g.o.y, f.o.y);
  f.o.z = fmaf(e, g.o.z, f.o.z);
  f.o.w = fmaf(e, g.o.w, f.o.w);
}

// bf16 quad o / l (zeros for a row that saw no token).
__device__ __forceinline__ uint2 fold_result(const Fold& f) {
  const float inv = f.l > 0.f ? 1.f / f.l : 0.f;
  uint2 pk;
  pk.x = pack_bf16x2(f.o.x * inv, f.o.y * inv);
  pk.y = pack_bf16x2(f.o.z * inv, f.o.w * inv);
  return pk;
}

}  // namespace pkv
