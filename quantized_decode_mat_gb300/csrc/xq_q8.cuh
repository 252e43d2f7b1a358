// One warp quantises one 256-value activation block to the q8 layout ("25 -
// Writing XPU Kernels" 25.2: 256 int8 values, eight sub-block sums, one f32
// scale).  Used by the standalone quantiser (to global memory) and by the
// fused quantise + mat-vec kernels (to shared memory), so both produce the
// same bytes.
//
// Rule (one f32 rounding per operation, no contraction):
//   amax = max|x|; iscale = 127/amax; q = clamp(rint(x*iscale), -127, 127)
//   (round half to even; a NaN product gives 0); d = amax/127; an all-zero
//   block has d = 0 and q = 0.  Sub-block sums are exact int32.
#pragma once

#include <stdint.h>

namespace xq {

struct Q8Lane {
    uint32_t w0, w1;  // this lane's eight int8 values (values 8*lane .. 8*lane+7)
    int sum;          // its sub-block's sum (sub-block lane/4), in every lane
    float d;          // the block scale, in every lane
};

// vals: values 8*lane .. 8*lane+7 of the block.  All 32 lanes must call.
__device__ __forceinline__ Q8Lane q8_quantize_lane(const float (&vals)[8]) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float t = fabsf(vals[i]);
        amax = t > amax ? t : amax;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, amax, off);
        amax = o > amax ? o : amax;
    }
    int q[8];
    if (amax == 0.0f) {
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = 0;
    } else {
        const float iscale = __fdiv_rn(127.0f, amax);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float t = __fmul_rn(vals[i], iscale);
            int r;
            if (t != t)
                r = 0;
            else if (t >= 127.0f)
                r = 127;
            else if (t <= -127.0f)
                r = -127;
            else
                r = __float2int_rn(t);  // round half to even
            q[i] = r;
        }
    }
    Q8Lane out;
    out.w0 = out.w1 = 0;
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        out.w0 |= (uint32_t)(q[i] & 0xFF) << (8 * i);
        out.w1 |= (uint32_t)(q[4 + i] & 0xFF) << (8 * i);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) sum += q[i];
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    out.sum = sum;
    out.d = (amax == 0.0f) ? 0.0f : __fdiv_rn(amax, 127.0f);
    return out;
}

}  // namespace xq
