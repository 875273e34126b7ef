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

}  // namespace mog
