// numerics.cuh -- the one definition of every floating-point step that must
// give the same bits in every kernel: the block state of one query row
// against one global KV block, and the canonical fold of states.
//
// The state of a row against global block b is
//   state_b = (o_b, lse_b, b)
// ("WS2 Attention PR5 Drift Benchmark", Transformer Engine Reuse).  The fused
// prefill, the state producer, the merge and the paged decode all call the
// functions below, so a state produced by one kernel and merged by another
// has exactly the bits the fused kernel folds on chip.  All of it is FP32
// with one explicit rounding per operation (the library is compiled with
// -fmad=false as well); the only downcast is the final BF16 write
// ("[WS2][Attention] H100 validation and reproduction guide", Status: FP32
// accumulation, fixed global_block_index merge, downcast at final write).
#pragma once
#include <cstdint>

namespace rlk {

constexpr float kLn2f = 0.693147182464599609375f;  // nearest float to ln 2

// 2^x by the hardware's ex2 instruction (flush-to-zero; ex2(-inf) = +0).
__device__ __forceinline__ float ex2_hw(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Pack two floats into a bf16x2 word (round to nearest even): lo in bits
// 0..15, hi in bits 16..31.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float bf16_lo_as_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi_as_f32(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Block softmax of one row, in the canonical order every kernel follows.
//   m   = max of the raw scores S_c over the visible keys
//   mc  = m * scale_log2                     (one rounding; log2 domain)
//   p_c = 2^fma(S_c, scale_log2, -mc)        for visible keys, 0 otherwise
//   l   = canonical row sum of p (below)
//   lse_b = fma(mc, ln2, ln l)  (natural log),  rcp = 1/l (IEEE-rounded)
// A row with no visible key has no state: p = 0, lse_b = -inf.
// (scale_log2 > 0, so the maximum of the raw scores scaled once is also the
// maximum of the scaled scores.)
//
// Canonical row sum: the block's keys are split into two halves of B/2; in
// each half, key c goes to partial c mod 16 (the keys of a partial added in
// ascending order) and the 16 partials are combined by the fixed tree
// a[t] <- a[t] + a[t + off] for off = 8, 4, 2, 1 -- the association an xor
// butterfly over 16 lanes produces, so a kernel with keys on lanes
// reproduces it; the block sum is half 0 + half 1.  (The halves let two
// warps share a row, each reading its half of S once; 16 partials keep a
// half row's softmax within 128 registers.)
__device__ __forceinline__ float prob(float s, float scale_log2, float neg_mc) {
  return ex2_hw(__fmaf_rn(s, scale_log2, neg_mc));
}
__device__ __forceinline__ float partial_tree(float (&a)[16]) {
#pragma unroll
  for (int off = 8; off >= 1; off >>= 1) {
#pragma unroll
    for (int t = 0; t < off; ++t) a[t] = __fadd_rn(a[t], a[t + off]);
  }
  return a[0];
}
__device__ __forceinline__ void block_stats(float mc, float l, float& lse_b, float& rcp) {
  lse_b = __fmaf_rn(mc, kLn2f, logf(l));
  rcp = __frcp_rn(l);
}

// Split p into BF16 hi + lo (p_hi = bf16(p), p_lo = bf16(p - p_hi)) packed
// two keys per word, key 2k in the low half.
__device__ __forceinline__ void split_pair(float p0, float p1, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16x2(p0, p1);
  const float r0 = __fsub_rn(p0, bf16_lo_as_f32(hi));
  const float r1 = __fsub_rn(p1, bf16_hi_as_f32(hi));
  lo = pack_bf16x2(r0, r1);
}

// Packed FP32x2 forms (sm_100-class): each lane is one IEEE round-to-nearest
// operation, bit-identical to the scalar __fmaf_rn / __fadd_rn / __fsub_rn /
// __fmul_rn on that lane, so kernels may use either form for the same step.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 fsub2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
// max of three (exact, so any grouping gives the same maximum)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Split a pair of probabilities into packed BF16 hi and lo words (the same
// values as split_pair).  The residual p - hi is exact in FP32 and is formed
// by one mixed-precision fma per element (hi * -1 + p, hi read as BF16
// straight from its half of the packed word), so lo = bf16_rn(p - hi) without
// widening hi first; an exact zero residual is +0, as __fsub_rn gives.
__device__ __forceinline__ void split_pair2(float2 p, uint32_t& hi, uint32_t& lo) {
  asm("{\n\t.reg .b16 h0, h1, m1;\n\t.reg .f32 r0, r1;\n\t"
      "cvt.rn.bf16x2.f32 %0, %3, %2;\n\t"
      "mov.b32 {h0, h1}, %0;\n\t"
      "mov.b16 m1, 0xBF80;\n\t"  // BF16 -1.0
      "fma.rn.f32.bf16 r0, h0, m1, %2;\n\t"
      "fma.rn.f32.bf16 r1, h1, m1, %3;\n\t"
      "cvt.rn.bf16x2.f32 %1, r1, r0;\n\t}"
      : "=r"(hi), "=r"(lo)
      : "f"(p.x), "f"(p.y));
}

// Block output element: o = PV * (1/l).
__device__ __forceinline__ float state_elem(float pv, float rcp) { return __fmul_rn(pv, rcp); }

// Canonical fold of running (O, L) with state (o_b, lse_b):
//   M = max(L, lse_b), mn = min(L, lse_b)
//   L' = M + log1p(exp(mn - M))
//   alpha = exp(L - L'), beta = exp(lse_b - L')
//   O  = fma(o_b, beta, O * alpha)
__device__ __forceinline__ void fold_coeffs(float L, float lb, float& Lp, float& alpha,
                                            float& beta) {
  const float M = fmaxf(L, lb);
  const float mn = fminf(L, lb);
  Lp = __fadd_rn(M, log1pf(expf(__fsub_rn(mn, M))));
  alpha = expf(__fsub_rn(L, Lp));
  beta = expf(__fsub_rn(lb, Lp));
}
__device__ __forceinline__ float fold_elem(float O, float o, float alpha, float beta) {
  return __fmaf_rn(o, beta, __fmul_rn(O, alpha));
}

// RoPE of one rotate-half pair (x0 = element i, x1 = element i + 64) with
// the table's FP32 cos / sin of its position and frequency, in the one FP32
// form every RoPE path of the library uses (the products rounded to FP32 on
// their own, then one fma each):
//   y0 = fma(x0, c, -(x1 * s)),  y1 = fma(x1, c, x0 * s)
__device__ __forceinline__ void rope_pair(float x0, float x1, float c, float s, float& y0, float& y1) {
  y0 = __fmaf_rn(x0, c, -__fmul_rn(x1, s));
  y1 = __fmaf_rn(x1, c, __fmul_rn(x0, s));
}
// Rotate 8 pairs held as packed BF16: a holds elements i..i+7, b elements
// i+64..i+71; c[e], s[e] belong to pair e.  Results rounded once to BF16.
__device__ __forceinline__ void rope_words8(uint4& a, uint4& b, const float (&c)[8], const float (&s)[8]) {
  const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
  uint32_t ra[4], rb[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    float ya0, yb0, ya1, yb1;
    rope_pair(bf16_lo_as_f32(wa[w]), bf16_lo_as_f32(wb[w]), c[2 * w], s[2 * w], ya0, yb0);
    rope_pair(bf16_hi_as_f32(wa[w]), bf16_hi_as_f32(wb[w]), c[2 * w + 1], s[2 * w + 1], ya1, yb1);
    ra[w] = pack_bf16x2(ya0, ya1);
    rb[w] = pack_bf16x2(yb0, yb1);
  }
  a = make_uint4(ra[0], ra[1], ra[2], ra[3]);
  b = make_uint4(rb[0], rb[1], rb[2], rb[3]);
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float x) {
  uint32_t w;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(0.0f), "f"(x));
  return static_cast<uint16_t>(w & 0xFFFFu);
}

}  // namespace rlk
