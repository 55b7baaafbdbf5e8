// softcap.cuh -- the softcap score modifier, s -> c tanh(s / c), for pairs of scores.
//
// softcap_tanh2 returns tanh(u), u = scale * s / c (the logit divided by c), so the caller
// folds c into the factor that turns scores into exponents.  It uses tanh u = 1 - 2 / (e^(2u) + 1)
// with a hardware exp2 and a hardware reciprocal: e^(2u) overflowing to +inf gives 1 and
// underflowing to 0 gives -1, and the absolute error in tanh is a few fp32 ulps of 1.
#pragma once

#include "ptx.cuh"

namespace attn {

// The factor from a raw score to 2 log2(e) u, u = scale s / c.
__host__ __device__ __forceinline__ float softcap_ku(float scale, float softcap) {
    return 2.f * 1.44269504088896340736f * scale / softcap;
}

// s0, s1: raw scores in, tanh(u) out; ku2 = (ku, ku) from softcap_ku.
__device__ __forceinline__ void softcap_tanh2(float& s0, float& s1, uint64_t ku2) {
    float y0, y1, d0, d1;
    f2_split(f2_mul(f2_make(s0, s1), ku2), y0, y1);
    f2_split(f2_add(f2_make(ex2_approx(y0), ex2_approx(y1)), f2_make(1.f, 1.f)), d0, d1);
    f2_split(f2_fma(f2_make(rcp_approx(d0), rcp_approx(d1)), f2_make(-2.f, -2.f), f2_make(1.f, 1.f)),
             s0, s1);
}

}  // namespace attn
