// Device side of the numeric contract "rlk-linlogp-v1": the library's own
// exp, log and rsqrt, and the (max, sum-exp) merge operator.
//
// The pages require the primitives to be fixed, not which ones ("vLLM
// RL-Kernel v0.1.0: ROCm 上でのビット単位のトレーニング-ロールアウト一貫性",
// section 数値実行契約, item 6: exp, log, ... FMA; the Chinese report "ROCm上
// 实现训练与推理logprob逐位对齐", section 技术路径, "数学原语").  Vendor exp/log
// may differ in the last place between implementations, so the contract
// defines its own from textbook methods and writes every operation with an
// explicit IEEE round-to-nearest intrinsic: no compiler contraction, no
// fast-math reassociation can change a bit.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <math_constants.h>

namespace rlk {

// exp(x) for x <= 0 (the only arguments the contract forms: logit - max and
// max differences).  Cody-Waite reduction x = n ln2 + r, |r| <= ln2/2, with
// n the nearest integer to x log2(e) (taken from the rounding of an fma
// against 1.5 * 2^23), r in two fma steps against a two-part ln 2; e^r by its
// degree-7 Taylor polynomial (coefficients 1/k! rounded to fp32) in Horner
// form; then an exact scaling by 2^n.  Arguments below -86 give +0, which
// keeps 2^n a normal number; their true value is below 2^-124 and vanishes
// next to the tile maximum's exp(0) = 1 in every sum the contract forms.
// Accuracy: under 1 ulp over [-86, 0] (checked exhaustively on the CPU).
__device__ __forceinline__ float contract_exp(float x) {
    const float kLog2e = 0x1.715476p+0f;
    const float kShift = 0x1.8p+23f;
    const float kLn2Hi = 0x1.62e430p-1f;
    const float kLn2Lo = -0x1.05c610p-29f;
    const float t = __fmaf_rn(x, kLog2e, kShift);
    const float n = __fsub_rn(t, kShift);
    const int ni = __float_as_int(t) - __float_as_int(kShift);
    float r = __fmaf_rn(-n, kLn2Hi, x);
    r = __fmaf_rn(-n, kLn2Lo, r);
    float p = 0x1.a01a02p-13f;             // 1/7!
    p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);  // 1/6!
    p = __fmaf_rn(p, r, 0x1.111112p-7f);   // 1/5!
    p = __fmaf_rn(p, r, 0x1.555556p-5f);   // 1/4!
    p = __fmaf_rn(p, r, 0x1.555556p-3f);   // 1/3!
    p = __fmaf_rn(p, r, 0.5f);             // 1/2!
    p = __fmaf_rn(p, r, 1.0f);             // 1/1!
    p = __fmaf_rn(p, r, 1.0f);             // 1/0!
    const float y = __fmul_rn(p, __int_as_float((ni + 127) << 23));
    return (x < -86.0f) ? 0.0f : y;
}

// log(s) for positive normal s (the contract only takes the log of a root
// sum, which lies in [1, 2^21]).  s = 2^e f with f in [sqrt(1/2), sqrt(2)];
// log f = 2 atanh(u), u = (f - 1)/(f + 1), by the odd series through u^11;
// log s = e ln2 + log f with the same two-part ln 2.  Accuracy: within 2 ulp
// on [1, 2^21] (checked exhaustively on the CPU).
__device__ __forceinline__ float contract_log(float s) {
    const float kLn2Hi = 0x1.62e430p-1f;
    const float kLn2Lo = -0x1.05c610p-29f;
    const int bits = __float_as_int(s);
    int e = (bits >> 23) - 127;
    float f = __int_as_float((bits & 0x007FFFFF) | 0x3F800000);
    if (f > 0x1.6a09e6p+0f) {  // sqrt(2) rounded to fp32
        f = __fmul_rn(f, 0.5f);
        e += 1;
    }
    const float u = __fdiv_rn(__fsub_rn(f, 1.0f), __fadd_rn(f, 1.0f));
    const float u2 = __fmul_rn(u, u);
    float p = 0x1.745d18p-3f;             // 2/11
    p = __fmaf_rn(p, u2, 0x1.c71c72p-3f);  // 2/9
    p = __fmaf_rn(p, u2, 0x1.24924ap-2f);  // 2/7
    p = __fmaf_rn(p, u2, 0x1.99999ap-2f);  // 2/5
    p = __fmaf_rn(p, u2, 0x1.555556p-1f);  // 2/3
    const float logf_ = __fmaf_rn(p, __fmul_rn(u, u2), __fmul_rn(2.0f, u));
    const float ef = __int2float_rn(e);
    return __fmaf_rn(ef, kLn2Hi, __fmaf_rn(ef, kLn2Lo, logf_));
}

// ---------------------------------------------------------------- two lanes
// Blackwell's packed fp32 instructions (fma/add/mul .rn .f32x2) round each of
// their two lanes exactly like the scalar instruction, so the contract's
// arithmetic can run two values per instruction with unchanged bits.  A
// pair's low 32 bits are its first value.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t p, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(p));
}
__device__ __forceinline__ uint64_t f2_splat(float x) { return f2_pack(x, x); }
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// contract_exp on both lanes, each lane bit for bit the scalar function:
// fma(-n, c, x) is written fma(n, -c, x) (the exact product only changes
// sign), t - shift as t + (-shift), and the scale 2^n is formed from the
// low bits of t directly: with t = 1.5 * 2^23 + n exactly, the scalar's
// (bits(t) - bits(1.5 * 2^23) + 127) << 23 equals bits(t) * 2^23 + bits(1.0f)
// modulo 2^32, because bits(1.5 * 2^23) * 2^23 vanishes modulo 2^32.
// kUnderflow = false is for arguments known to lie in [-86, 0] (numbers, not
// NaN): no select is needed, and since p is a normal number in [0.7, 1.5]
// and n >= -124, p * 2^n is normal and exact, i.e. n added to p's exponent
// field -- bits(p) + bits(t) * 2^23 modulo 2^32 (same reasoning as for the
// scale) -- an integer shift and add instead of forming 2^n and
// multiplying.  The shift is a funnel shift, which runs on the integer ALU
// rather than on the FMA pipe that bounds the exp (1.3 % faster in the bf16
// materialised-logits kernel than a multiply-add by 2^23).
template <bool kUnderflow = true>
__device__ __forceinline__ uint64_t contract_exp_x2(uint64_t x) {
    const uint64_t t = f2_fma(x, f2_splat(0x1.715476p+0f), f2_splat(0x1.8p+23f));
    const uint64_t n = f2_add(t, f2_splat(-0x1.8p+23f));
    uint64_t r = f2_fma(n, f2_splat(-0x1.62e430p-1f), x);
    r = f2_fma(n, f2_splat(0x1.05c610p-29f), r);
    uint64_t p = f2_fma(f2_splat(0x1.a01a02p-13f), r, f2_splat(0x1.6c16c2p-10f));
    p = f2_fma(p, r, f2_splat(0x1.111112p-7f));
    p = f2_fma(p, r, f2_splat(0x1.555556p-5f));
    p = f2_fma(p, r, f2_splat(0x1.555556p-3f));
    p = f2_fma(p, r, f2_splat(0.5f));
    p = f2_fma(p, r, f2_splat(1.0f));
    p = f2_fma(p, r, f2_splat(1.0f));
    float tl, th;
    f2_unpack(t, tl, th);
    if (!kUnderflow) {
        float pl, ph;
        f2_unpack(p, pl, ph);
        return f2_pack(__uint_as_float(__float_as_uint(pl) + __funnelshift_l(0u, __float_as_uint(tl), 23)),
                       __uint_as_float(__float_as_uint(ph) + __funnelshift_l(0u, __float_as_uint(th), 23)));
    }
    const uint64_t scale = f2_pack(__uint_as_float(__float_as_uint(tl) * 8388608u + 0x3F800000u),
                                   __uint_as_float(__float_as_uint(th) * 8388608u + 0x3F800000u));
    float yl, yh, xl, xh;
    f2_unpack(f2_mul(p, scale), yl, yh);
    f2_unpack(x, xl, xh);
    return f2_pack(xl < -86.0f ? 0.0f : yl, xh < -86.0f ? 0.0f : yh);
}

// Two columns of the logit gradient G = bf16_RN(RN(g * d)), d = RN(1 - p) at
// the target and -p elsewhere, p = contract_exp(RN(l - lse)), from the fp32
// logits (l0, l1) as one packed pair; neg_lse = (-lse, -lse), g2 = (g, g).
// Returns the two bf16 values, the first in the low half.  Rows that take no
// part pass valid = false and get zeros.
__device__ __forceinline__ uint32_t contract_grad_x2(uint64_t l01, uint64_t neg_lse, uint64_t g2,
                                                     bool tgt0, bool tgt1, bool valid) {
    float p0, p1;
    f2_unpack(contract_exp_x2(f2_add(l01, neg_lse)), p0, p1);
    const float d0 = tgt0 ? __fsub_rn(1.0f, p0) : -p0;
    const float d1 = tgt1 ? __fsub_rn(1.0f, p1) : -p1;
    float g0, g1;
    f2_unpack(f2_mul(g2, f2_pack(d0, d1)), g0, g1);
    if (!valid) g0 = g1 = 0.0f;
    const __nv_bfloat162 b = __floats2bfloat162_rn(g0, g1);  // round each to nearest
    return static_cast<uint32_t>(__bfloat16_as_ushort(b.x)) |
           (static_cast<uint32_t>(__bfloat16_as_ushort(b.y)) << 16);
}

// rsqrt(a) for positive normal a: Lomont's seed for the bit-level inverse
// square-root estimate, two Newton steps, then one in correction form.
// Under 0.86 ulp over [2^-40, 2^40] (checked exhaustively on the CPU).
__device__ __forceinline__ float contract_rsqrt(float a) {
    float y = __uint_as_float(0x5f375a86u - (__float_as_uint(a) >> 1));
    const float h = __fmul_rn(0.5f, a);
#pragma unroll
    for (int k = 0; k < 2; ++k) y = __fmul_rn(y, __fmaf_rn(-h, __fmul_rn(y, y), 1.5f));
    const float e = __fmaf_rn(-h, __fmul_rn(y, y), 0.5f);
    return __fmaf_rn(y, e, y);
}

// A (max, sum of exp(x - max)) pair.
struct MaxSum {
    float m;
    float s;
};

// The contract's merge: the operand with the larger max is kept ("hi"; the
// left operand on a tie), the other's sum is scaled by exp(lo.m - hi.m) and
// added with one fused rounding.  On a tie exp(0) = 1 exactly, so the result
// is RN(s_left + s_right) whichever side is left.
//
// Padding slots of the GPU's power-of-two tree carry m = -inf, s = 0; the
// contract's own tree never forms them, and a padding operand must pass the
// other one through unchanged, which the final select guarantees (it also
// keeps -inf - -inf from producing a NaN).
__device__ __forceinline__ MaxSum contract_merge(MaxSum left, MaxSum right) {
    const bool right_hi = right.m > left.m;
    const float mh = right_hi ? right.m : left.m;
    const float sh = right_hi ? right.s : left.s;
    const float ml = right_hi ? left.m : right.m;
    const float sl = right_hi ? left.s : right.s;
    const float scaled = __fmaf_rn(sl, contract_exp(__fsub_rn(ml, mh)), sh);
    MaxSum out;
    out.m = mh;
    out.s = (ml == -CUDART_INF_F) ? sh : scaled;
    return out;
}

// The contract's 128-column tile reduction on values held as 64 pairs,
// P[k] = (v[2k], v[2k+1]); padding columns must already be -inf.  Returns
// (max, sum) with the bits of the scalar evaluation: the max is exact, each
// exp is contract_exp of RN(v - max), and the sum is the pairwise tree over
// the column index.  Level 1 adds the two lanes of each pair, giving s_j =
// e_2j + e_2j+1; the level-1 sums are packed as X_j = (s_j, s_j+32), so each
// packed add of neighbours X_2i + X_2i+1 forms the next level's nodes of
// both 64-column halves at once, left node plus right node in each lane;
// levels 2-6 run this way and level 7 adds the two halves.  The packed
// levels are evaluated as a binary counter over j (a node is formed as soon
// as both children exist), which keeps few partial sums live.
struct TreeX2 {
    uint64_t pending[5];  // pending[L]: a finished left node of packed level L + 2
    uint64_t x = 0;
    // the exps of pairs j and j + 32 (columns 2j, 2j+1 and 64+2j, 64+2j+1), in
    // order j = 0..31; j must be a compile-time constant after unrolling
    __device__ __forceinline__ void push(int j, uint64_t e_lo, uint64_t e_hi) {
        float a, b, c, d;
        f2_unpack(e_lo, a, b);
        f2_unpack(e_hi, c, d);
        push_node(j, f2_pack(__fadd_rn(a, b), __fadd_rn(c, d)));
    }
    // the level-1 node X_j = (s_j, s_j+32) itself, in order j = 0..31; with the
    // exps formed on (column 2j, column 64+2j) and (2j+1, 64+2j+1) pairs, X_j
    // is one packed add of the two
    __device__ __forceinline__ void push_node(int j, uint64_t X) {
        x = X;
        int level = 0;
#pragma unroll
        for (; level < 5; ++level) {
            if (!(j & (1 << level))) break;
            x = f2_add(pending[level], x);  // left sibling + this node
        }
        if (level < 5) pending[level] = x;
    }
    __device__ __forceinline__ float total() const {
        float z0, z1;
        f2_unpack(x, z0, z1);  // the two 64-column halves
        return __fadd_rn(z0, z1);
    }
};

__device__ __forceinline__ MaxSum tile_reduce_x2(uint64_t (&P)[64]) {
    float m0, m1, m2, m3;
    f2_unpack(P[0], m0, m1);
    f2_unpack(P[1], m2, m3);
#pragma unroll
    for (int k = 2; k < 64; k += 2) {
        float a, b, c, d;
        f2_unpack(P[k], a, b);
        f2_unpack(P[k + 1], c, d);
        m0 = fmaxf(m0, a);
        m1 = fmaxf(m1, b);
        m2 = fmaxf(m2, c);
        m3 = fmaxf(m3, d);
    }
    const float m = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
    const uint64_t neg_m = f2_splat(-m);
    TreeX2 tree;
#pragma unroll
    for (int j = 0; j < 32; ++j)
        tree.push(j, contract_exp_x2(f2_add(P[j], neg_m)), contract_exp_x2(f2_add(P[j + 32], neg_m)));
    MaxSum out;
    out.m = m;
    out.s = tree.total();
    return out;
}

}  // namespace rlk
