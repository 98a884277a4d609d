// Tensor-core score body (fp16 or q8_0 keys, head_dim a multiple of 64),
// shared by the score stage (k_score_tc) and the fused pass (k_pass).
//
// [Worklog] "TriAttention Native C++ Worklog", Phase 9 (the score is taken on
// the stored rotated keys: the calibrated mean query times the conjugate key,
// the rotation applied on the query side only, plus a norm term on the keys'
// magnitudes) and 2026-04-18 (phases from the absolute decode position).
//
// Per row r and query head h of the segment's group:
//   raw_h(r) = sum_f  Wr_{h,f} K[r][f] + Wi_{h,f} K[r][f+fc] + M_{h,f} |k_f|
// with W = qbar E_f e^{i w_f p} and M = q_abs - |qbar|.
//
// The phase term sum_f Wr K[f] + Wi K[f+fc] is a contraction of the key rows
// with a [head_dim x heads] weight matrix, and the keys are exact in fp16: it
// runs as m16n8k16 MMAs (fp32 accumulation) against W split into an fp16 high
// part and an fp16 remainder, scaled per head by a power of two so that both
// parts are normal. The magnitude term sum_f M |k_f| is formed in fp32 from
// the same key fragments and contracted with M by m16n8k8 tf32 MMAs, again on
// a high part and its remainder. The columns of one n-tile are [high parts of
// the G heads, remainders of the G heads], so a head's score is the sum of two
// accumulator columns: fp32-level accuracy from half-precision operands.
//
// A warp computes 16 rows (one m-tile) at a time. Lane (g, q) = (lane / 4,
// lane % 4) reads 16-byte granule q of the 64-byte step s of rows g and g + 8;
// the MMA k-slots are mapped to the granule's elements (the same map in A and
// B, which a contraction is free to permute), so no transposing load is
// needed. Real and imaginary parts of a frequency sit in steps s and
// s + S/2 at the same lane and register position.
//
// Heads with non-rotary dims (the last nonrot of head_dim are never rotated;
// the first rot = head_dim - nonrot are NEOX pairs (f, f + rot/2)): the
// statistics loader extends the rot/2 rotary pairs with nonrot/2 "content
// pairs" (rot + e, rot + nonrot/2 + e) of frequency 0 and norm weight 0, whose
// phase term is exactly the mean non-rotary query's dot product with those
// dims. With rot a multiple of 64, pair step s (32 pairs) is all rotary for
// s < hr = rot/64 (real parts in step s, imaginary in step s + hr) and all
// content otherwise (steps s + hr and s + S/2); the norm term runs on the
// rotary pair steps only.
#pragma once

#include "tria_internal.cuh"

namespace tria {

__device__ __forceinline__ float sqrt_approx(float x) {
  float y;
  asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The high part of x for a tf32 hi / remainder split: x with its low 13
// mantissa bits cleared (one logic op). x - hi is exact in fp32 and below
// 2^-10 |x|, so the remainder's own truncation to tf32 costs < 2^-20 |x|.
__device__ __forceinline__ uint32_t tf32_hi(float x) { return __float_as_uint(x) & 0xFFFFE000u; }

__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t y;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Four signed 8-bit values (one 32-bit word) as two fp16 pairs, exactly: with
// u = x + 128 in a byte, the fp16 bit pattern 0x6400 | u is 1024 + u, and
// subtracting 1152 leaves x (both steps exact in fp16).
__device__ __forceinline__ void i8x4_to_h2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140u);
  const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342u);
  const __half2 bias = __halves2half2(__ushort_as_half((unsigned short)0x6480u), __ushort_as_half((unsigned short)0x6480u));
  const __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
  const __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
  lo = *reinterpret_cast<const uint32_t*>(&ha);
  hi = *reinterpret_cast<const uint32_t*>(&hb);
}

// Products of fp16 values in fp32 without converting them first: the
// mixed-precision fma (fp16 sources, fp32 addend and result) forms the
// product exactly and rounds once after the add.
__device__ __forceinline__ float2 mul_h2_h(uint32_t pair, unsigned short s) {   // (pair.lo * s, pair.hi * s)
  float lo, hi;
  asm("{.reg .f16 a, b, c;\n"
      " mov.b32 {a, b}, %2;\n"
      " mov.b16 c, %3;\n"
      " fma.rn.f32.f16 %0, a, c, 0f00000000;\n"
      " fma.rn.f32.f16 %1, b, c, 0f00000000;\n}"
      : "=f"(lo), "=f"(hi)
      : "r"(pair), "h"(s));
  return make_float2(lo, hi);
}

__device__ __forceinline__ float2 sumsq_h2(uint32_t re, uint32_t im) {   // re^2 + im^2 per half, in fp32
  float lo, hi;
  asm("{.reg .f16 a, b, c, d;\n"
      " .reg .f32 t, u;\n"
      " mov.b32 {a, b}, %2;\n"
      " mov.b32 {c, d}, %3;\n"
      " fma.rn.f32.f16 t, a, a, 0f00000000;\n"
      " fma.rn.f32.f16 u, b, b, 0f00000000;\n"
      " fma.rn.f32.f16 %0, c, c, t;\n"
      " fma.rn.f32.f16 %1, d, d, u;\n}"
      : "=f"(lo), "=f"(hi)
      : "r"(re), "r"(im));
  return make_float2(lo, hi);
}

// |k| of 8 frequencies from fp16 pairs of block values times their fp16
// scales: real parts r * dr, imaginary parts i * di (products exact in fp32)
__device__ __forceinline__ void q8_mag(const uint32_t* r, const uint32_t* i, unsigned short dr, unsigned short di,
                                       float* m) {
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const float2 a = mul_h2_h(r[t], dr);
    const float2 b = mul_h2_h(i[t], di);
    const float2 sq = __ffma2_rn(b, b, __fmul2_rn(a, a));
    m[2 * t] = sqrt_approx(sq.x);
    m[2 * t + 1] = sqrt_approx(sq.y);
  }
}

// |k| of the 8 frequencies of one granule: real parts r, imaginary parts i
// (the squares exact in fp32, one rounding for their sum)
__device__ __forceinline__ void granule_mag(const uint4& r, const uint4& i, float* m) {
  const uint32_t rr[4] = {r.x, r.y, r.z, r.w}, ii[4] = {i.x, i.y, i.z, i.w};
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const float2 sq = sumsq_h2(rr[t], ii[t]);
    m[2 * t] = sqrt_approx(sq.x);
    m[2 * t + 1] = sqrt_approx(sq.y);
  }
}

template <int G, int S>
struct TcShape {
  static constexpr int NT = (2 * G + 7) / 8;   // n-tiles: G high-part columns, then G remainder columns
  static constexpr bool kOk = S % 2 == 0 && NT * S <= 8;
};

// One warp's tensor-core scorer: the B fragments of the current segment, the
// per-head unscaling factors, and the running moments of the rows scored
// since the last flush. Lane (g, q) writes heads (oh, oh + 1) (one head when
// G == 1) of one row per m-tile (two rows when G == 8); with G <= 2 only
// lanes q < 2 write.
template <int KT, int G, int S>
struct TcBody {
  static_assert(KT == TRIA_F16 || KT == TRIA_Q8_0, "fp16 or q8_0 keys");
  static constexpr bool kQ8 = KT == TRIA_Q8_0;
  using SH = TcShape<G, S>;
  static constexpr int NT = SH::NT;
  static constexpr int FC = 16 * S;   // frequency pairs (head_dim / 2)
  static constexpr int kHeads = G >= 2 ? 2 : 1;
  static constexpr int kWriters = G == 8 ? 4 : (G == 4 ? 2 : 1);
  static_assert(SH::kOk, "tensor-core body shape");

  int g, q, oh, hl;
  int hr;                           // rotary pair steps (S / 2 when every dim is rotary)
  bool owriter;
  uint32_t bp[S][NT][4];            // phase weights, fp16 pairs
  uint32_t bm[S / 2][NT][4][2];     // magnitude weights, tf32
  float unscale[kHeads];
  Mom run[kHeads];

  // fcr: rotary frequency pairs of the head (a multiple of 32)
  __device__ __forceinline__ void init(int lane, int fcr) {
    hr = fcr / 32;
    g = lane >> 2;
    q = lane & 3;
    oh = G == 8 ? 2 * q : (G == 4 ? 2 * (q & 1) : 0);
    owriter = G >= 4 || q < 2;
    hl = g < 2 * G ? g % G : 0;   // lane (g, q) builds column g of every n-tile, which belongs to head hl
#pragma unroll
    for (int k = 0; k < kHeads; ++k) run[k] = Mom{0.f, 0.f, 0.f};
  }

  // B fragments of one segment: qe / mw point at the segment's KV head
  // ([G][FC] each), turns at the FC turn factors (shared memory), pos is the
  // absolute decode position.
  __device__ __forceinline__ void load_consts(const float2* qe_g, const float* mw_g, const unsigned long long* turns,
                                              unsigned long long pos) {
    const float2* qe = qe_g + (size_t)hl * FC;
    const float* mw = mw_g + (size_t)hl * FC;
    // inputs of this lane's frequencies f = 32 s + 8 q + j (s < S / 2) of head
    // hl, all loaded up front
    float2 a[S / 2][8];
    float m[S / 2][8];
#pragma unroll
    for (int s2 = 0; s2 < S / 2; ++s2)
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int f = 32 * s2 + 8 * q + j;
        a[s2][j] = qe[f];
        m[s2][j] = mw[f];
      }
    // scale 2^e with max(|qbar E|, |M|) of the head (a bound of every weight,
    // since |Wr|, |Wi| <= |qbar E|) in [2^14, 2^15): both fp16 parts stay
    // normal; the four lanes of a column cover all frequencies
    float amax = 0.f;
#pragma unroll
    for (int s2 = 0; s2 < S / 2; ++s2)
#pragma unroll
      for (int j = 0; j < 8; ++j)
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(a[s2][j].x), fabsf(a[s2][j].y)), fabsf(m[s2][j])));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    int e = 0;
    if (amax > 0.f && amax < INFINITY) e = 14 - ilogbf(amax);
    e = max(-120, min(120, e));
    const float scale = __int_as_float((127 + e) << 23);
#pragma unroll
    for (int s2 = 0; s2 < S / 2; ++s2) {
      float wre_hi[8], wre_lo[8], wim_hi[8], wim_lo[8], wm_hi[8], wm_lo[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const unsigned long long x = turns[32 * s2 + 8 * q + j] * pos;   // exact turn fraction of w_f * p
        float sn, cs;
        sincospif((float)(int)(x >> 32) * 0x1p-31f, &sn, &cs);
        const float wr = (a[s2][j].x * cs - a[s2][j].y * sn) * scale;
        const float wi = (a[s2][j].x * sn + a[s2][j].y * cs) * scale;
        const float ms = m[s2][j] * scale;
        wre_hi[j] = __half2float(__float2half_rn(wr));
        wre_lo[j] = wr - wre_hi[j];
        wim_hi[j] = __half2float(__float2half_rn(wi));
        wim_lo[j] = wi - wim_hi[j];
        wm_hi[j] = __uint_as_float(to_tf32(ms));
        wm_lo[j] = ms - wm_hi[j];
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int c = 8 * nt + g;
        const bool live = c < 2 * G, rem = c >= G;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float r0 = !live ? 0.f : (rem ? wre_lo[2 * t] : wre_hi[2 * t]);
          const float r1 = !live ? 0.f : (rem ? wre_lo[2 * t + 1] : wre_hi[2 * t + 1]);
          const float i0 = !live ? 0.f : (rem ? wim_lo[2 * t] : wim_hi[2 * t]);
          const float i1 = !live ? 0.f : (rem ? wim_lo[2 * t + 1] : wim_hi[2 * t + 1]);
          const float m0 = !live ? 0.f : (rem ? wm_lo[2 * t] : wm_hi[2 * t]);
          const float m1 = !live ? 0.f : (rem ? wm_lo[2 * t + 1] : wm_hi[2 * t + 1]);
          bp[s2][nt][t] = pack_f16x2(r0, r1);
          bp[s2 + S / 2][nt][t] = pack_f16x2(i0, i1);
          bm[s2][nt][t][0] = __float_as_uint(m0);
          bm[s2][nt][t][1] = __float_as_uint(m1);
        }
      }
    }
    // unscaling factors of the heads this lane writes: lane 4 h holds the
    // exponent of head h (column h of n-tile 0)
#pragma unroll
    for (int k = 0; k < kHeads; ++k) {
      const int eh = __shfl_sync(0xffffffffu, e, 4 * (oh + k));
      unscale[k] = __int_as_float((127 - eh) << 23);
    }
  }

  // Scores `rows` key rows staged in shared memory at buf (k_rb bytes each;
  // q8_0: their block scales at scb, ks_rb bytes each), writes the raw scores
  // to out[row * G + head] and adds the rows to the running moments.
  __device__ __forceinline__ void piece(const uint8_t* buf, const uint8_t* scb, int rows, int k_rb, int ks_rb,
                                        float* out) {
    if (hr == S / 2) piece_t<S / 2>(buf, scb, rows, k_rb, ks_rb, out);
    else piece_t<-1>(buf, scb, rows, k_rb, ks_rb, out);
  }

  // The body for HR rotary pair steps (-1: the runtime hr); HR = S / 2 is the
  // all-rotary head with every step offset a constant.
  template <int HR>
  __device__ __forceinline__ void piece_t(const uint8_t* buf, const uint8_t* scb, int rows, int k_rb, int ks_rb,
                                          float* out) {
    const int hr_ = HR >= 0 ? HR : hr;
    // shifted sums of this piece for my output heads
    float shift[kHeads], m1[kHeads], m2[kHeads], cnt[kHeads];
#pragma unroll
    for (int k = 0; k < kHeads; ++k) shift[k] = m1[k] = m2[k] = cnt[k] = 0.f;
    auto emit = [&](int rr, const float (&x)[kHeads]) {
      if (rr >= rows) return;
      float y[kHeads];
#pragma unroll
      for (int k = 0; k < kHeads; ++k) y[k] = x[k] * unscale[k];
      float* dst = out + (size_t)rr * G + oh;
      if constexpr (kHeads == 2) *reinterpret_cast<float2*>(dst) = make_float2(y[0], y[1]);
      else *dst = y[0];
#pragma unroll
      for (int k = 0; k < kHeads; ++k) {
        if (cnt[k] == 0.f) shift[k] = y[k];
        const float d = y[k] - shift[k];
        m1[k] += d;
        m2[k] = fmaf(d, d, m2[k]);
        cnt[k] += 1.f;
      }
    };
    for (int mt = 0; 16 * mt < rows; ++mt) {
      // independent accumulator chains, summed at the end: real, imaginary,
      // |k| high part, |k| remainder (two chains for head_dim > 128, where
      // registers are short and the chains are long enough anyway)
      constexpr bool kFour = S <= 4;
      float acc[NT][4], acc_i[NT][4], acc_mh[NT][4], acc_ml[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int t = 0; t < 4; ++t) acc[nt][t] = acc_i[nt][t] = acc_mh[nt][t] = acc_ml[nt][t] = 0.f;
      if constexpr (!kQ8) {
        const uint8_t* rg = buf + (size_t)(16 * mt + g) * k_rb + 16 * q;
        const uint8_t* rg8 = rg + (size_t)8 * k_rb;
#pragma unroll
        for (int s2 = 0; s2 < S / 2; ++s2) {
          const bool rotary = s2 < hr_;
          const int sr = rotary ? s2 : s2 + hr_, si = rotary ? s2 + hr_ : s2 + S / 2;   // real / imaginary steps
          const uint4 kr0 = *reinterpret_cast<const uint4*>(rg + 64 * sr);
          const uint4 kr8 = *reinterpret_cast<const uint4*>(rg8 + 64 * sr);
          const uint4 ki0 = *reinterpret_cast<const uint4*>(rg + 64 * si);
          const uint4 ki8 = *reinterpret_cast<const uint4*>(rg8 + 64 * si);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma_f16(acc[nt], kr0.x, kr8.x, kr0.y, kr8.y, bp[s2][nt][0], bp[s2][nt][1]);
            float(&di)[4] = kFour ? acc_i[nt] : acc[nt];
            mma_f16(di, ki0.x, ki8.x, ki0.y, ki8.y, bp[s2 + S / 2][nt][0], bp[s2 + S / 2][nt][1]);
            mma_f16(acc[nt], kr0.z, kr8.z, kr0.w, kr8.w, bp[s2][nt][2], bp[s2][nt][3]);
            mma_f16(di, ki0.z, ki8.z, ki0.w, ki8.w, bp[s2 + S / 2][nt][2], bp[s2 + S / 2][nt][3]);
          }
          if (!rotary) continue;   // content pairs: no norm term
          float mg0[8], mg8[8];
          granule_mag(kr0, ki0, mg0);
          granule_mag(kr8, ki8, mg8);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t h0 = tf32_hi(mg0[2 * u]), h1 = tf32_hi(mg8[2 * u]);
            const uint32_t h2 = tf32_hi(mg0[2 * u + 1]), h3 = tf32_hi(mg8[2 * u + 1]);
            const uint32_t l0 = __float_as_uint(mg0[2 * u] - __uint_as_float(h0));
            const uint32_t l1 = __float_as_uint(mg8[2 * u] - __uint_as_float(h1));
            const uint32_t l2 = __float_as_uint(mg0[2 * u + 1] - __uint_as_float(h2));
            const uint32_t l3 = __float_as_uint(mg8[2 * u + 1] - __uint_as_float(h3));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              mma_tf32(acc_mh[nt], h0, h1, h2, h3, bm[s2][nt][u][0], bm[s2][nt][u][1]);
              float(&dl)[4] = kFour ? acc_ml[nt] : acc_mh[nt];
              mma_tf32(dl, l0, l1, l2, l3, bm[s2][nt][u][0], bm[s2][nt][u][1]);
            }
          }
        }
      } else {
        // q8_0: a 32-value block is one step s (bytes 32 s .. 32 s + 32 of the
        // row); its two MMAs go to a fresh accumulator scaled by the block's
        // scale of each row, and |k| uses the scaled values
        const uint8_t* rg = buf + (size_t)(16 * mt + g) * k_rb + 8 * q;
        const uint8_t* rg8 = rg + (size_t)8 * k_rb;
        const __half* sg0 = reinterpret_cast<const __half*>(scb + (size_t)(16 * mt + g) * ks_rb);
        const __half* sg8 = reinterpret_cast<const __half*>(scb + (size_t)(16 * mt + g + 8) * ks_rb);
#pragma unroll
        for (int s2 = 0; s2 < S / 2; ++s2) {
          const bool rotary = s2 < hr_;
          const int sr = rotary ? s2 : s2 + hr_, si = rotary ? s2 + hr_ : s2 + S / 2;   // real / imaginary blocks
          const uint2 wr0 = *reinterpret_cast<const uint2*>(rg + 32 * sr);
          const uint2 wr8 = *reinterpret_cast<const uint2*>(rg8 + 32 * sr);
          const uint2 wi0 = *reinterpret_cast<const uint2*>(rg + 32 * si);
          const uint2 wi8 = *reinterpret_cast<const uint2*>(rg8 + 32 * si);
          const float dr0 = __half2float(sg0[sr]), dr8 = __half2float(sg8[sr]);
          const float di0 = __half2float(sg0[si]), di8 = __half2float(sg8[si]);
          uint32_t ar0[4], ar8[4], ai0[4], ai8[4];
          i8x4_to_h2x2(wr0.x, ar0[0], ar0[1]);
          i8x4_to_h2x2(wr0.y, ar0[2], ar0[3]);
          i8x4_to_h2x2(wr8.x, ar8[0], ar8[1]);
          i8x4_to_h2x2(wr8.y, ar8[2], ar8[3]);
          i8x4_to_h2x2(wi0.x, ai0[0], ai0[1]);
          i8x4_to_h2x2(wi0.y, ai0[2], ai0[3]);
          i8x4_to_h2x2(wi8.x, ai8[0], ai8[1]);
          i8x4_to_h2x2(wi8.y, ai8[2], ai8[3]);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            float tr[4] = {0.f, 0.f, 0.f, 0.f}, ti[4] = {0.f, 0.f, 0.f, 0.f};
            mma_f16(tr, ar0[0], ar8[0], ar0[1], ar8[1], bp[s2][nt][0], bp[s2][nt][1]);
            mma_f16(ti, ai0[0], ai8[0], ai0[1], ai8[1], bp[s2 + S / 2][nt][0], bp[s2 + S / 2][nt][1]);
            mma_f16(tr, ar0[2], ar8[2], ar0[3], ar8[3], bp[s2][nt][2], bp[s2][nt][3]);
            mma_f16(ti, ai0[2], ai8[2], ai0[3], ai8[3], bp[s2 + S / 2][nt][2], bp[s2 + S / 2][nt][3]);
            acc[nt][0] = fmaf(tr[0], dr0, fmaf(ti[0], di0, acc[nt][0]));
            acc[nt][1] = fmaf(tr[1], dr0, fmaf(ti[1], di0, acc[nt][1]));
            acc[nt][2] = fmaf(tr[2], dr8, fmaf(ti[2], di8, acc[nt][2]));
            acc[nt][3] = fmaf(tr[3], dr8, fmaf(ti[3], di8, acc[nt][3]));
          }
          if (!rotary) continue;   // content pairs: no norm term
          float mg0[8], mg8[8];
          q8_mag(ar0, ai0, __half_as_ushort(sg0[sr]), __half_as_ushort(sg0[si]), mg0);
          q8_mag(ar8, ai8, __half_as_ushort(sg8[sr]), __half_as_ushort(sg8[si]), mg8);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t h0 = tf32_hi(mg0[2 * u]), h1 = tf32_hi(mg8[2 * u]);
            const uint32_t h2 = tf32_hi(mg0[2 * u + 1]), h3 = tf32_hi(mg8[2 * u + 1]);
            const uint32_t l0 = __float_as_uint(mg0[2 * u] - __uint_as_float(h0));
            const uint32_t l1 = __float_as_uint(mg8[2 * u] - __uint_as_float(h1));
            const uint32_t l2 = __float_as_uint(mg0[2 * u + 1] - __uint_as_float(h2));
            const uint32_t l3 = __float_as_uint(mg8[2 * u + 1] - __uint_as_float(h3));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              mma_tf32(acc_mh[nt], h0, h1, h2, h3, bm[s2][nt][u][0], bm[s2][nt][u][1]);
              float(&dl)[4] = kFour ? acc_ml[nt] : acc_mh[nt];
              mma_tf32(dl, l0, l1, l2, l3, bm[s2][nt][u][0], bm[s2][nt][u][1]);
            }
          }
        }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int t = 0; t < 4; ++t)
          acc[nt][t] = kFour ? (acc[nt][t] + acc_i[nt][t]) + (acc_mh[nt][t] + acc_ml[nt][t]) : acc[nt][t] + acc_mh[nt][t];
      // column pairs (high part, remainder) -> head scores
      if constexpr (G == 8) {
        emit(16 * mt + g, {acc[0][0] + acc[1][0], acc[0][1] + acc[1][1]});
        emit(16 * mt + g + 8, {acc[0][2] + acc[1][2], acc[0][3] + acc[1][3]});
      } else if constexpr (G == 4) {
        float v[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) v[t] = acc[0][t] + __shfl_xor_sync(0xffffffffu, acc[0][t], 2);
        if (q & 2) emit(16 * mt + g + 8, {v[2], v[3]});
        else emit(16 * mt + g, {v[0], v[1]});
      } else if constexpr (G == 2) {
        float v[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) v[t] = acc[0][t] + __shfl_xor_sync(0xffffffffu, acc[0][t], 1);
        if (q == 0) emit(16 * mt + g, {v[0], v[1]});
        else if (q == 1) emit(16 * mt + g + 8, {v[2], v[3]});
      } else {
        const float a = acc[0][0] + acc[0][1], b = acc[0][2] + acc[0][3];
        const float b_from0 = __shfl_xor_sync(0xffffffffu, b, 1);
        if (q == 0) emit(16 * mt + g, {a});
        else if (q == 1) emit(16 * mt + g + 8, {b_from0});
      }
    }
    // this piece's moments -> the running moments
#pragma unroll
    for (int k = 0; k < kHeads; ++k) {
      Mom b;
      b.n = cnt[k];
      const float mean_d = cnt[k] > 0.f ? __fdividef(m1[k], cnt[k]) : 0.f;
      b.mean = shift[k] + mean_d;
      b.m2 = fmaxf(m2[k] - m1[k] * mean_d, 0.f);
      run[k] = mom_merge(run[k], b);
    }
  }

  // Merges the running moments over the lanes that carry the same heads
  // (lanes without output carry zero counts), in a fixed order
  // (deterministic), and restarts them. Afterwards the lanes with g == 0 and
  // q < kWriters hold the merged moments of heads (oh, oh + 1) in out.
  __device__ __forceinline__ void flush(Mom (&out)[kHeads]) {
#pragma unroll
    for (int k = 0; k < kHeads; ++k) {
      Mom m = owriter ? run[k] : Mom{0.f, 0.f, 0.f};
#pragma unroll
      for (int mask = 1; mask < 32; mask <<= 1) {
        const bool same_heads = G == 8 ? mask >= 4 : (G == 4 ? mask >= 2 : true);
        if (same_heads) m = mom_merge(m, mom_shfl(m, mask));
      }
      out[k] = m;
      run[k] = Mom{0.f, 0.f, 0.f};
    }
  }

  __device__ __forceinline__ bool flush_writer() const { return g == 0 && q < kWriters; }
};

}  // namespace tria
