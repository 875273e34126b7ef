// exact.cuh -- the nearest-centroid rule the clustering is defined by, and the fp32
// certificate that lets most decisions skip it.
//
// The nearest centroid is the one with the smallest D(x, c) = sum_j (x_j - c_j)^2 evaluated
// in fp64 in index order, lowest index on ties.  An fp32 evaluation (difference, then fused
// square-accumulate, in any order) is within (d + 2) 2^-24 D of D, since every term is
// non-negative; a best centroid whose fp32 runner-up is farther than that bound on both
// values (with a safety factor) is the exact argmin.
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace mog {

// relative error bound of the fp32 distance, with a safety factor of ~3 over (d+2)*2^-24
constexpr float kCertRel = 2.5e-5f;

__device__ __forceinline__ bool certified(float b1, float b2) {
    // true minimum is b1's centroid for every rounding within the bound
    return b2 - b1 > kCertRel * (b1 + b2);
}

// exact rule: fp64, index order, no contraction
__device__ __forceinline__ double exact_dist(const uint16_t *x, const float *c) {
    double acc = 0.0;
    for (int j = 0; j < MOG_D; ++j) {
        double diff = __dsub_rn((double)bf1(x[j]), (double)c[j]);
        acc = __dadd_rn(acc, __dmul_rn(diff, diff));
    }
    return acc;
}

// A double-float evaluation of D(x, c) (x fp32 values of bf16 keys, c fp32): each
// difference is split exactly into hi + lo (two-sum), its square into the exact product
// dh^2 (the fused multiply-add's residual) plus 2 dh dl (dl^2 < 2^-48 dh^2 is dropped), and
// the terms are summed in a (hi, lo) pair.  The low word gathers at most 4 * 2^-24 of
// each term; its own rounding is at most 2^9 * 2^-48 of D a step, so over d = 128 terms
// the pair is within 2^-31 D of the exact sum (kDfRel carries a safety factor of 20 over
// that).  The fp64 rule of D sums exact squares (the differences of fp32 values and
// their squares fit in 53 bits) with 127 roundings, within 2^-46 D of the exact sum: a
// best candidate whose double-float value is below every other by more than both bounds
// is the fp64 argmin.
constexpr double kDfRel = 1e-8;

__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

__device__ __forceinline__ double df_dist(const float *x, const float *c) {
    float sh = 0.f, sl = 0.f;
    for (int j = 0; j < MOG_D; ++j) {
        float dh, dl;
        two_sum(x[j], -c[j], dh, dl);
        const float ph = __fmul_rn(dh, dh);
        float pl = __fmaf_rn(dh, dh, -ph);
        pl = __fmaf_rn(__fmul_rn(2.f, dh), dl, pl);
        float s, e;
        two_sum(sh, ph, s, e);
        sh = s;
        sl = __fadd_rn(sl, __fadd_rn(e, pl));
    }
    return __dadd_rn((double)sh, (double)sl);
}

}  // namespace mog
