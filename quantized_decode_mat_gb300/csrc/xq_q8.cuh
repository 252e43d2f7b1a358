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

// N blocks at once, one warp: vals[j] holds values 8*lane .. 8*lane+7 of
// block j.  All 32 lanes must call.  The steps of the N blocks are
// interleaved and nothing branches: an all-zero block (amax = 0) gets
// iscale = 127/0 = inf, so each of its products is 0*inf = NaN and quantises
// to 0, and d = 0/127 = 0, as the rule asks.  A product is rounded by one
// saturating conversion (NaN -> 0, +-inf -> 127 / -128) and raised to -127:
// a finite product stays below 127.5 in magnitude, and an iscale that
// overflowed to inf on a tiny amax still gives +-127.  With N >= 2 lane j
// takes block j's two divisions and the others read them by shuffle: one
// division pass for all N blocks.
// SAT: each product rounded by one saturating conversion (below); false: by
// an explicit clamp, a rounding and a NaN select (the same bytes; the form
// the raw codebook kernel's register assignment measured faster with).
template <int N, bool SAT = true>
__device__ __forceinline__ void q8_quantize_lanes(const float (&vals)[N][8], Q8Lane (&out)[N],
                                                  int lane) {
    static_assert(N >= 1 && N <= 32, "one block a lane at most");
    float amax[N];
#pragma unroll
    for (int j = 0; j < N; ++j) {
        amax[j] = 0.0f;  // fmaxf keeps the non-NaN operand: NaN values do not count
#pragma unroll
        for (int i = 0; i < 8; ++i) amax[j] = fmaxf(amax[j], fabsf(vals[j][i]));
    }
    // across the warp: a non-negative float (never NaN here) orders as its
    // bits do, so one integer max reduction gives the block's amax exactly
#pragma unroll
    for (int j = 0; j < N; ++j)
        amax[j] = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(amax[j])));
    float iscale[N], d[N];
    if constexpr (N == 1) {
        iscale[0] = __fdiv_rn(127.0f, amax[0]);
        d[0] = __fdiv_rn(amax[0], 127.0f);
    } else {
        float a = amax[0];
#pragma unroll
        for (int j = 1; j < N; ++j) a = lane == j ? amax[j] : a;
        const float is = __fdiv_rn(127.0f, a), dd = __fdiv_rn(a, 127.0f);
#pragma unroll
        for (int j = 0; j < N; ++j) {
            iscale[j] = __shfl_sync(0xffffffffu, is, j);
            d[j] = __shfl_sync(0xffffffffu, dd, j);
        }
    }
    int sum[N];
#pragma unroll
    for (int j = 0; j < N; ++j) {
        int q[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            // round half to even, saturating to [-128, 127] with NaN -> 0;
            // a finite product is below 127.5 in magnitude (|x| <= amax), so
            // only -inf (iscale overflowed) reaches -128, raised to -127
            const float t = __fmul_rn(vals[j][i], iscale[j]);
            if constexpr (SAT) {
                int r;
                asm("cvt.rni.sat.s8.f32 %0, %1;" : "=r"(r) : "f"(t));
                q[i] = max(r, -127);
            } else {
                const int r = __float2int_rn(fminf(fmaxf(t, -127.0f), 127.0f));
                q[i] = t != t ? 0 : r;
            }
        }
        out[j].w0 = __byte_perm(__byte_perm((uint32_t)q[0], (uint32_t)q[1], 0x0040u),
                                __byte_perm((uint32_t)q[2], (uint32_t)q[3], 0x0040u), 0x5410u);
        out[j].w1 = __byte_perm(__byte_perm((uint32_t)q[4], (uint32_t)q[5], 0x0040u),
                                __byte_perm((uint32_t)q[6], (uint32_t)q[7], 0x0040u), 0x5410u);
        if constexpr (SAT) {  // the lane's sum: its eight signed bytes dotted with ones
            sum[j] = __dp4a((int)out[j].w1, 0x01010101, __dp4a((int)out[j].w0, 0x01010101, 0));
        } else {
            sum[j] = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) sum[j] += q[i];
        }
        out[j].d = d[j];
    }
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1)
#pragma unroll
        for (int j = 0; j < N; ++j) sum[j] += __shfl_xor_sync(0xffffffffu, sum[j], off);
#pragma unroll
    for (int j = 0; j < N; ++j) out[j].sum = sum[j];
}

// One block: vals holds values 8*lane .. 8*lane+7.  All 32 lanes must call.
__device__ __forceinline__ Q8Lane q8_quantize_lane(const float (&vals)[8]) {
    float v[1][8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[0][i] = vals[i];
    Q8Lane out[1];
    q8_quantize_lanes<1>(v, out, 0);
    return out[0];
}

}  // namespace xq
