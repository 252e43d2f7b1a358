// Persistent, asynchronously staged decode mat-vec for sm_103a, templated on
// the weight format, the batch (1..8), whether it also emits the exact
// integer dots, and whether it quantises the f32 activation itself (the
// fused quantise + mat-vec) or reads q8 blocks.
//
// Arithmetic: integer dots with dp4a, reduced to the super-block exactly in
// int32 ("reduce first, then scale once", "25 - Writing XPU Kernels" 25.2),
// then an f32 epilogue with an error-free compensation term (TwoProduct /
// TwoSum), so the float result is within a few f32 ulps of the exact one.
#pragma once

#include "xq_internal.h"
#include "xq_ptx.cuh"
#include "xq_norm.cuh"
#include "xq_q8.cuh"

namespace xq {

// ---- activation views ----------------------------------------------------------------
// A staged q8 block (one chunk of one activation vector) in shared memory,
// kActStride bytes apart per chunk and nb*kActStride apart per vector:
//   [0,256) int8 values   [256,288) int32 sums   [288,292) f32 scale
//   [304,320) the eight sums split into bytes: low bytes of sums 0..3, of
//   4..7 (unsigned), then high bytes (sum >> 8, signed) of 0..3, of 4..7.
struct ActSmem {
    const uint8_t *p;
    int64_t bstride;
    __device__ __forceinline__ uint4 q16(int b, int i) const {  // values 16i..16i+15
        return reinterpret_cast<const uint4 *>(p + b * bstride)[i];
    }
    __device__ __forceinline__ float xs(int b) const {
        return *reinterpret_cast<const float *>(p + b * bstride + kQ8ScaleAt);
    }
    __device__ __forceinline__ uint4 split(int b) const {
        return *reinterpret_cast<const uint4 *>(p + b * bstride + kActSplitAt);
    }
};

// The eight sub-block sums (each |s| <= 127*32) as unsigned low bytes and
// signed high bytes, so that sum_j m_j*s_j is four dp4a: s = 256*hi + lo.
__device__ __forceinline__ uint4 split_sums(uint4 s0, uint4 s1) {
    const uint32_t s[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    uint32_t l0 = 0, l1 = 0, h0 = 0, h1 = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        l0 |= (s[j] & 0xFFu) << (8 * j);
        l1 |= (s[j + 4] & 0xFFu) << (8 * j);
        h0 |= (((uint32_t)((int)s[j] >> 8)) & 0xFFu) << (8 * j);
        h1 |= (((uint32_t)((int)s[j + 4] >> 8)) & 0xFFu) << (8 * j);
    }
    return make_uint4(l0, l1, h0, h1);
}

// ---- shared epilogue --------------------------------------------------------
// Adds xs*(d*S1 - dmin*S2) to (hi, lo).  S1, S2 exact integers, |S1| < 2^25,
// |S2| < 2^24.  The inner difference is formed first as an unevaluated pair
// D + Dl (TwoProduct of each scale with its exact integer, then TwoSum of
// the two products), then scaled by xs (one TwoProduct), so the term reaches
// (hi, lo) with an error of the order of 2^-44 of its magnitude.  S1 is split
// into its f32 rounding and an exact residual (0 unless |S1| > 2^24).
// first: (hi, lo) holds nothing yet, so the term is assigned to it.
__device__ __forceinline__ void q4k_epilogue(float xs, float d, float dmin, int S1, int S2,
                                             float &hi, float &lo, bool first) {
    const float f1 = __int2float_rn(S1);
    const float r1 = __int2float_rn(S1 - __float2int_rn(f1));  // exact, |r1| <= 1
    const float f2 = __int2float_rn(S2);                       // exact
    float a, ae, b, be, D, De;
    two_prod(d, f1, a, ae);          // d*f1 = a + ae exactly
    ae = __fmaf_rn(d, r1, ae);       // + d*r1 (second order)
    two_prod(dmin, f2, b, be);       // dmin*S2 = b + be exactly
    two_sum(a, -b, D, De);           // a - b = D + De exactly
    const float Dl = __fadd_rn(__fsub_rn(ae, be), De);
    float t, te;
    two_prod(xs, D, t, te);          // xs*D = t + te exactly
    const float tl = __fmaf_rn(xs, Dl, te);
    if (first) {
        hi = t;
        lo = tl;
    } else {
        acc_add(hi, lo, t, tl);
    }
}

__device__ __forceinline__ int byte_of(uint32_t x, int k) {
    return (int)__byte_perm(x, 0u, 0x4440u | (uint32_t)k);
}

// ---- Q4_K chunk ---------------------------------------------------------------------
// w: this lane's 144-byte super-block in shared memory; act: its q8 blocks.
template <int B, bool DOTS, class Act>
__device__ __forceinline__ void q4k_chunk(const uint8_t *__restrict__ w, const Act &act,
                                          float (&hi)[B], float (&lo)[B], int32_t *dots,
                                          int64_t dots_bstride, bool first) {
    const uint4 h = *reinterpret_cast<const uint4 *>(w);
    uint32_t q[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint4 v = *reinterpret_cast<const uint4 *>(w + 16 + 16 * i);
        q[4 * i + 0] = v.x;
        q[4 * i + 1] = v.y;
        q[4 * i + 2] = v.z;
        q[4 * i + 3] = v.w;
    }
    const float d = f16_bits_to_f32(h.x);
    const float dmin = f16_bits_to_f32(h.x >> 16);
    // six-bit scales and mins, one byte each: bytes 4..7 (h.y), 8..11 (h.z), 12..15 (h.w)
    const uint32_t sc_lo = h.y & 0x3F3F3F3Fu;
    const uint32_t m_lo = h.z & 0x3F3F3F3Fu;
    const uint32_t sc_hi = (h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u);
    const uint32_t m_hi = ((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u);
    int sc[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        sc[j] = byte_of(sc_lo, j);
        sc[j + 4] = byte_of(sc_hi, j);
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
        int dot[8];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            // sub-block 2g: values 64g..64g+31 (low nibbles of group g);
            // sub-block 2g+1: values 64g+32..64g+63 (high nibbles of group g)
            const uint4 a0 = act.q16(b, 4 * g + 0), a1 = act.q16(b, 4 * g + 1);
            const uint4 a2 = act.q16(b, 4 * g + 2), a3 = act.q16(b, 4 * g + 3);
            const uint32_t alo[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const uint32_t ahi[8] = {a2.x, a2.y, a2.z, a2.w, a3.x, a3.y, a3.z, a3.w};
            // High nibbles are used in place (x16): an unsigned byte 16*q times
            // a signed byte; the sum is a multiple of 16, so >> 4 is exact.
            int d0 = 0, d1 = 0;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t word = q[8 * g + k];
                d0 = dp4a(word & 0x0F0F0F0Fu, alo[k], d0);
                d1 = dp4a_us(word & 0xF0F0F0F0u, ahi[k], d1);
            }
            dot[2 * g] = d0;
            dot[2 * g + 1] = d1 >> 4;
        }
        int S1 = 0;
#pragma unroll
        for (int s = 0; s < 8; ++s) S1 += sc[s] * dot[s];
        const uint4 sp = act.split(b);  // sum_j m_j * bsum_j as four byte dots
        const int S2 = dp4a_uu(m_hi, sp.y, dp4a_uu(m_lo, sp.x, 0)) +
                       256 * dp4a_us(m_hi, sp.w, dp4a_us(m_lo, sp.z, 0));
        q4k_epilogue(act.xs(b), d, dmin, S1, S2, hi[b], lo[b], first);
        if (DOTS && dots != nullptr) {
            int4 *o = reinterpret_cast<int4 *>(dots + b * dots_bstride);
            o[0] = make_int4(dot[0], dot[1], dot[2], dot[3]);
            o[1] = make_int4(dot[4], dot[5], dot[6], dot[7]);
        }
    }
}

// ---- Q4_K, M row groups at once --------------------------------------------------------
// The same arithmetic as q4k_chunk for M chunks that share one column (lane
// l's chunk in each of M row groups): every activation load from shared
// memory is used against M chunks instead of one.  The loop runs over the four
// 64-value groups, then the vectors, then the chunks.  S1 is an exact
// integer and each (chunk, vector) epilogue is the single-chunk one, so y is
// bit-for-bit that of the one-chunk form.
//
// The high-nibble dots are used in place (x16), so the low sub-block's scale
// is taken x16 and the sum is 16*S1, shifted once per chunk and vector
// (|16*S1| <= 16 * 8 * 63 * 32 * 15 * 127 < 2^29).  Chunks of rows that do not
// exist were zero-filled when staged (d = dmin = 0, no scales, mins or values)
// and add exact zeros, so no lane branches around its epilogue; ok[m] gates
// only the dots export.  FIRST: this is the row's first chunk of the lane (one
// segment per row), so the epilogue assigns (hi, lo) instead of adding to it.
template <int B, int M, bool DOTS, bool FIRST, class Act>
__device__ __forceinline__ void q4k_chunks(const uint8_t *const (&w)[M], const bool (&ok)[M],
                                           const Act &act, float (&hi)[M][B], float (&lo)[M][B],
                                           int32_t *const (&dots)[M], int64_t dots_bstride) {
    float d[M], dmin[M];
    uint32_t sc_lo[M], sc_hi[M], m_lo[M], m_hi[M];
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const uint4 h = *reinterpret_cast<const uint4 *>(w[m]);
        d[m] = f16_bits_to_f32(h.x);
        dmin[m] = f16_bits_to_f32(h.x >> 16);
        sc_lo[m] = h.y & 0x3F3F3F3Fu;
        m_lo[m] = h.z & 0x3F3F3F3Fu;
        sc_hi[m] = (h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u);
        m_hi[m] = ((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u);
    }
    int S16[M][B];  // 16 * S1
#pragma unroll
    for (int m = 0; m < M; ++m)
#pragma unroll
        for (int b = 0; b < B; ++b) S16[m][b] = 0;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        // sub-block 2g: low nibbles of group g; sub-block 2g+1: its high nibbles
        uint32_t ql[M][8], qh[M][8];
        int s0x16[M], s1[M];
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const uint4 v0 = *reinterpret_cast<const uint4 *>(w[m] + 16 + 32 * g);
            const uint4 v1 = *reinterpret_cast<const uint4 *>(w[m] + 32 + 32 * g);
            const uint32_t q[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                ql[m][k] = q[k] & 0x0F0F0F0Fu;
                qh[m][k] = q[k] & 0xF0F0F0F0u;
            }
            const uint32_t scw = g < 2 ? sc_lo[m] : sc_hi[m];
            s0x16[m] = byte_of(scw, 2 * (g & 1)) << 4;
            s1[m] = byte_of(scw, 2 * (g & 1) + 1);
        }
#pragma unroll
        for (int b = 0; b < B; ++b) {
            const uint4 a0 = act.q16(b, 4 * g + 0), a1 = act.q16(b, 4 * g + 1);
            const uint4 a2 = act.q16(b, 4 * g + 2), a3 = act.q16(b, 4 * g + 3);
            const uint32_t alo[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const uint32_t ahi[8] = {a2.x, a2.y, a2.z, a2.w, a3.x, a3.y, a3.z, a3.w};
#pragma unroll
            for (int m = 0; m < M; ++m) {
                int d0 = 0, d1 = 0;  // d1: 16 * the high sub-block's dot
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    d0 = dp4a(ql[m][k], alo[k], d0);
                    d1 = dp4a_us(qh[m][k], ahi[k], d1);
                }
                S16[m][b] += s0x16[m] * d0 + s1[m] * d1;
                if (DOTS && ok[m])
                    *reinterpret_cast<int2 *>(dots[m] + b * dots_bstride + 2 * g) =
                        make_int2(d0, d1 >> 4);
            }
        }
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
        const uint4 sp = act.split(b);  // sum_j m_j * bsum_j as four byte dots
        const float xs = act.xs(b);
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const int S2 = dp4a_uu(m_hi[m], sp.y, dp4a_uu(m_lo[m], sp.x, 0)) +
                           256 * dp4a_us(m_hi[m], sp.w, dp4a_us(m_lo[m], sp.z, 0));
            q4k_epilogue(xs, d[m], dmin[m], S16[m][b] >> 4, S2, hi[m][b], lo[m][b], FIRST);
        }
    }
}

// ---- codebook chunk -----------------------------------------------------------------
// The codebook kernels stage each 32-value sub-block of the activation
// interleaved: word 2i holds values (4i, 4i+16, 4i+1, 4i+17) and word 2i+1
// values (4i+2, 4i+18, 4i+3, 4i+19), i = 0..3 -- the order in which the
// nibbles of payload word i sit (byte j: low nibble = element 4i+j, high
// nibble = element 4i+j+16).  A decoded payload word then dots with two
// activation words as it is.  (Sums are order-free, so the dots are those of
// the natural order.)
__device__ __forceinline__ uint32_t interleave_lo(uint32_t a, uint32_t b) {
    return __byte_perm(a, b, 0x5140u);  // a.0 b.0 a.1 b.1
}
__device__ __forceinline__ uint32_t interleave_hi(uint32_t a, uint32_t b) {
    return __byte_perm(a, b, 0x7362u);  // a.2 b.2 a.3 b.3
}

// Eight nibbles of a payload word -> two words of int8 codebook values in
// nibble order: F0 = kv of nibbles 0..3 (L0, H0, L1, H1), F1 = of nibbles
// 4..7.  The table is four registers.  prmt looks up 8 entries at a time,
// so each nibble is looked up in both half tables with its low three bits,
// and a byte mask made from its bit 3 (prmt's sign-replicate mode on the
// byte whose top bit it is) selects the half.  Exact by construction.
__device__ __forceinline__ void cb4_decode(uint32_t q, const uint32_t (&T)[4], uint32_t &F0,
                                           uint32_t &F1) {
    const uint32_t s = q & 0x77777777u;  // entry index within a half table
    const uint32_t sh = s >> 16;
    const uint32_t a0 = prmt(T[0], T[1], s);   // kv[0..7] for nibbles 0..3
    const uint32_t a1 = prmt(T[0], T[1], sh);  // ... nibbles 4..7
    const uint32_t b0 = prmt(T[2], T[3], s);   // kv[8..15]
    const uint32_t b1 = prmt(T[2], T[3], sh);
    // bit 3 of an even nibble is the top bit of its byte in q << 4, of an
    // odd nibble the top bit of its byte in q; selector 8+j replicates it
    const uint32_t q4 = q << 4;
    const uint32_t m0 = prmt(q4, q, 0xD9C8u);  // nibbles 0..3
    const uint32_t m1 = prmt(q4, q, 0xFBEAu);  // nibbles 4..7
    F0 = (a0 & ~m0) | (b0 & m0);
    F1 = (a1 & ~m1) | (b1 & m1);
}

// The dot of a payload word q (eight nibbles) with the two activation words
// in its nibble order, from a table split in two: kv[n] = L[n] + H[n] (signed
// bytes), where one lookup of the whole nibble in (S[0], S[1]) gives L -- an
// entry for n < 8, and for n >= 8 prmt's sign replication of byte n - 8,
// 0 or -1 -- and one lookup of n ^ 8 in (S[2], S[3]) gives H the other way
// round (the host finds the bytes; split_table in the API).  Four lookups
// and four dp4a, no select: seven operations of decode a word against the
// eleven of cb4_decode, for one vector (with more vectors the select form
// does fewer operations, as its decoded words are shared).
__device__ __forceinline__ int cb4_dot_split(uint32_t q, const uint32_t (&S)[4], uint32_t a0,
                                             uint32_t a1, int acc) {
    const uint32_t qx = q ^ 0x88888888u;
    const uint32_t l0 = prmt(S[0], S[1], q);          // nibbles 0..3
    const uint32_t h0 = prmt(S[2], S[3], qx);
    const uint32_t l1 = prmt(S[0], S[1], q >> 16);    // nibbles 4..7
    const uint32_t h1 = prmt(S[2], S[3], qx >> 16);
    acc = dp4a(l0, a0, acc);
    acc = dp4a(h0, a0, acc);
    acc = dp4a(l1, a1, acc);
    return dp4a(h1, a1, acc);
}

// Eight codebook blocks of one chunk: scales dk[k] and payload words P[k][0..3]
// (block k's 16 payload bytes, little-endian), against the interleaved q8
// block `act`.  Block by block: decode, then its dot with every vector; per
// vector the compensated sum over the blocks runs in block order.  T: the
// table as sixteen bytes, or with SPLIT (one vector only) as the two lookup
// tables of cb4_dot_split; either gives the same integer dots.
template <int B, bool DOTS, bool FIRST, bool SPLIT, class Act>
__device__ __forceinline__ void cb4_blocks(const float (&dk)[8], const uint32_t (&P)[8][4],
                                           const Act &act, const uint32_t (&T)[4], float (&hi)[B],
                                           float (&lo)[B], int32_t *dots, int64_t dots_bstride) {
    static_assert(!SPLIT || B == 1, "the split table serves one vector");
    float ch[B], cl[B];  // sum_k d_k * dot_k per vector, compensated
#pragma unroll
    for (int b = 0; b < B; ++b) ch[b] = cl[b] = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        uint32_t F[8];
        if constexpr (!SPLIT) {
#pragma unroll
            for (int i = 0; i < 4; ++i) cb4_decode(P[k][i], T, F[2 * i], F[2 * i + 1]);
        }
#pragma unroll
        for (int b = 0; b < B; ++b) {
            const uint4 a0 = act.q16(b, 2 * k), a1 = act.q16(b, 2 * k + 1);
            int dt = 0;
            if constexpr (SPLIT) {
                dt = cb4_dot_split(P[k][0], T, a0.x, a0.y, dt);
                dt = cb4_dot_split(P[k][1], T, a0.z, a0.w, dt);
                dt = cb4_dot_split(P[k][2], T, a1.x, a1.y, dt);
                dt = cb4_dot_split(P[k][3], T, a1.z, a1.w, dt);
            } else {
                dt = dp4a(F[0], a0.x, dt);
                dt = dp4a(F[1], a0.y, dt);
                dt = dp4a(F[2], a0.z, dt);
                dt = dp4a(F[3], a0.w, dt);
                dt = dp4a(F[4], a1.x, dt);
                dt = dp4a(F[5], a1.y, dt);
                dt = dp4a(F[6], a1.z, dt);
                dt = dp4a(F[7], a1.w, dt);
            }
            float p, e;
            two_prod(dk[k], __int2float_rn(dt), p, e);  // |dt| < 2^20: exact in f32
            if (k == 0) {  // an exact add to zero is an assignment
                ch[b] = p;
                cl[b] = e;
            } else {
                acc_add(ch[b], cl[b], p, e);
            }
            if (DOTS && dots != nullptr) dots[b * dots_bstride + k] = dt;
        }
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
        const float xs = act.xs(b);
        float t, te;
        two_prod(ch[b], xs, t, te);
        if (FIRST) {  // the lane's first chunk of the row: (hi, lo) holds nothing yet
            hi[b] = t;
            lo[b] = __fmaf_rn(cl[b], xs, te);
        } else {
            acc_add(hi[b], lo[b], t, __fmaf_rn(cl[b], xs, te));
        }
    }
}

// Raw layout: w is this lane's 144-byte chunk (eight 18-byte blocks) in
// shared memory.
template <int B, bool DOTS, bool FIRST, bool SPLIT, class Act>
__device__ __forceinline__ void cb4_chunk(const uint8_t *__restrict__ w, const Act &act,
                                          const uint32_t (&T)[4], float (&hi)[B], float (&lo)[B],
                                          int32_t *dots, int64_t dots_bstride) {
    uint32_t v[36];
#pragma unroll
    for (int i = 0; i < 9; ++i) {
        const uint4 t = *reinterpret_cast<const uint4 *>(w + 16 * i);
        v[4 * i + 0] = t.x;
        v[4 * i + 1] = t.y;
        v[4 * i + 2] = t.z;
        v[4 * i + 3] = t.w;
    }
    // Block pair p (blocks 2p, 2p+1) is the 36 bytes at 36p: words 9p..9p+8.
    // Block 2p: scale = low half of word 9p, payload = bytes 2..17 of the pair
    // (realigned by 16-bit funnel shifts); block 2p+1: scale = high half of
    // word 9p+4, payload = words 9p+5..9p+8.
    float dk[8];
    uint32_t P[8][4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        dk[2 * p] = f16_bits_to_f32(v[9 * p]);
        dk[2 * p + 1] = f16_bits_to_f32(v[9 * p + 4] >> 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            P[2 * p][i] = __funnelshift_r(v[9 * p + i], v[9 * p + i + 1], 16);
            P[2 * p + 1][i] = v[9 * p + 5 + i];
        }
    }
    cb4_blocks<B, DOTS, FIRST, SPLIT>(dk, P, act, T, hi, lo, dots, dots_bstride);
}

// ---- resident codebook rows: the staged layout ----------------------------------------
// A box of resident rows (32 chunks, 4608 bytes) is staged as 32 payload
// slots of 128 bytes -- slot l holds the eight 16-byte payloads of the chunk
// lane l takes, payload i at 16-byte position i ^ (l & 7) -- followed by 32
// scale slots of 16 bytes at 4096 + 16 l.  A warp's copy instruction moves 32
// consecutive 16-byte pieces of a row, which land in four whole 128-byte
// payload slots (or in the contiguous scale slots), so each copy is written
// as four shared-memory wavefronts; the position swizzle puts the payloads
// that eight lanes read at once on distinct 4-bank groups.  (A slot of the
// chunk's scales followed by its payloads, 144 bytes, left every 128-byte run
// unaligned: 12.9 wavefronts a copy instruction, and each line fetched from
// L2 about 1.55 times.)
__device__ __forceinline__ uint32_t cb4r_scale_slot(int slot) {
    return 4096u + 16u * (uint32_t)slot;
}
__device__ __forceinline__ uint32_t cb4r_payload_slot(int slot, int i) {
    return 128u * (uint32_t)slot + 16u * (uint32_t)(i ^ (slot & 7));
}

// stage: the staged box; slot: the chunk this lane takes.
template <int B, bool DOTS, bool FIRST, bool SPLIT, class Act>
__device__ __forceinline__ void cb4r_chunk(const uint8_t *__restrict__ stage, int slot,
                                           const Act &act, const uint32_t (&T)[4], float (&hi)[B],
                                           float (&lo)[B], int32_t *dots, int64_t dots_bstride) {
    const uint4 sc = *reinterpret_cast<const uint4 *>(stage + cb4r_scale_slot(slot));
    const uint32_t sw[4] = {sc.x, sc.y, sc.z, sc.w};
    const uint8_t *pay = stage + 128 * slot;
    const int key = slot & 7;
    float dk[8];
    uint32_t P[8][4];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        dk[k] = f16_bits_to_f32(sw[k >> 1] >> (16 * (k & 1)));
        const uint4 t = *reinterpret_cast<const uint4 *>(pay + 16 * (k ^ key));
        P[k][0] = t.x;
        P[k][1] = t.y;
        P[k][2] = t.z;
        P[k][3] = t.w;
    }
    cb4_blocks<B, DOTS, FIRST, SPLIT>(dk, P, act, T, hi, lo, dots, dots_bstride);
}

// ---- reduction of a row's partial sums -------------------------------------------------
// Recursive halving over the aligned group of `width` lanes that share a row
// (width a power of two): at offset o, a lane keeps the lower or upper half of
// its batch values (by its lane bit o), sends the other half to lane ^ o and
// adds the received half, compensated (acc_add).  log2(P) such steps leave
// one value a lane, summed over 2^steps lanes; the remaining offsets are a
// plain xor butterfly on that value.  With batch 1 this is the butterfly
// alone.  Compared with a butterfly of every value, it moves and adds
// B/2 + B/4 + ... values a lane instead of B*log2(width).  On return,
// h[i], l[i] (i < nlive) hold vector base + i of the row, complete in the
// lanes whose bits below `keep` are zero.
// a compile-time int as a value (for generic lambdas)
template <int N>
struct IntTag {
    static constexpr int value = N;
};

template <int B>
struct Pow2Ceil {
    static constexpr int v = B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : 8;
};

template <int P>
__device__ __forceinline__ void halving_reduce(float (&h)[P], float (&l)[P], int width, int lane,
                                               int &base, int &nlive, int &keep) {
    base = 0;
    nlive = P;
    int off = width >> 1;
#pragma unroll
    for (int s = 0; (P >> s) >= 2; ++s) {
        if (off == 0) break;
        const int n = P >> s;
        const bool up = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float kh = up ? h[n / 2 + i] : h[i], kl = up ? l[n / 2 + i] : l[i];
            const float sh = up ? h[i] : h[n / 2 + i], sl = up ? l[i] : l[n / 2 + i];
            const float rh = __shfl_xor_sync(0xffffffffu, sh, off);
            const float rl = __shfl_xor_sync(0xffffffffu, sl, off);
            float a = kh, c = kl;
            acc_add(a, c, rh, rl);
            h[i] = a;
            l[i] = c;
        }
        if (up) base += n / 2;
        nlive = n / 2;
        off >>= 1;
    }
    keep = off ? 2 * off - 1 : 0;
    for (; off > 0; off >>= 1) {  // nlive == 1 here
        const float oh = __shfl_xor_sync(0xffffffffu, h[0], off);
        const float ol = __shfl_xor_sync(0xffffffffu, l[0], off);
        acc_add(h[0], l[0], oh, ol);
    }
}

// ---- work-unit descriptor ---------------------------------------------------------------
// Row group g of a launch: where its rows start in W, how many exist, where
// their outputs go and which staged activation vector they use.  In the
// grouped-expert form (ID), the launch's rows are `used` slots of
// rows_per_expert rows each; slot kk reads expert sel[kk]'s rows from the
// slab and writes output rows kk*rows_per_expert.. ("25 - Writing XPU
// Kernels" 25.2.2); a group never straddles two slots.
struct GroupInfo {
    int64_t row0;   // first row in W
    int64_t out0;   // first output row
    int valid;      // rows of the group that exist (0..R)
    int vec;        // staged activation vector
    bool bad;       // ID form: sel[kk] outside [0, n_experts)
};

template <bool ID>
__device__ __forceinline__ GroupInfo group_info(const MatvecArgs &a, int64_t g, int R) {
    GroupInfo gi;
    if (!ID) {
        gi.row0 = g * R;
        gi.out0 = gi.row0;
        const int64_t rr = a.rows - gi.row0;
        gi.valid = (int)(rr < R ? rr : R);
        gi.vec = 0;
        gi.bad = false;
    } else {
        const int64_t gps = a.groups_per_slot;
        const int64_t kk = g / gps;
        const int64_t r0 = (g - kk * gps) * R;  // first row within the slot
        const int e = __ldg(a.sel + kk);
        gi.bad = e < 0 || e >= a.n_experts;
        gi.row0 = (int64_t)(gi.bad ? 0 : e) * a.rows_per_expert + r0;
        gi.out0 = kk * a.rows_per_expert + r0;
        const int64_t rr = a.rows_per_expert - r0;
        gi.valid = (int)(rr < R ? rr : R);
        gi.vec = a.act_vectors > 1 ? (int)kk : 0;
    }
    return gi;
}

// ---- transposed reduction for rows of 16 chunks ----------------------------------------
// Whole rows of 16 chunks in a box (4096 columns): lane l holds chunk l % 16 of
// row l / 16 of each of the unit's M row groups, for B vectors.  The lanes
// write their partial sums (M * P pairs, P = B rounded up to a power of two)
// to a warp-private scratch -- the stage the unit was just read from -- and
// read them back transposed: lane t then holds the 16 chunks of one (row
// group, row, vector) and adds them with the pairing tree of the shuffle
// reductions (chunks 8 apart, then 4, 2, 1).  acc_add is symmetric, so the
// bits are those of every other reduction form, at a fraction of the
// instructions and none of the shuffle latency.  The row stride of
// (M * P + 1) * 8 bytes puts the writes of 16 lanes, and the reads of one
// scratch row, on distinct banks.
template <int M, int B>
__device__ __forceinline__ void reduce_rows16_store(const float (&hi)[M][B], const float (&lo)[M][B],
                                                    uint8_t *scratch, int lane,
                                                    const GroupInfo (&gi)[M], float *y,
                                                    int64_t rows) {
    constexpr int P = Pow2Ceil<B>::v;
    constexpr int kStride = (M * P + 1) * 8;
    static_assert(M * 2 * P <= 32, "one output a lane at most");
    static_assert(M == 1 || M == 2, "row groups are picked by a select");
    float2 *mine = reinterpret_cast<float2 *>(scratch + lane * kStride);
#pragma unroll
    for (int m = 0; m < M; ++m)
#pragma unroll
        for (int b = 0; b < B; ++b) mine[m * P + b] = make_float2(hi[m][b], lo[m][b]);
    __syncwarp();
    if constexpr (M * 2 * P == 16) {
        // sixteen outputs: two lanes an output, lane half h taking the chunks
        // of parity h (the tree's first three levels pair chunks of equal
        // parity), then one exchange for the last level
        const int o = lane & 15, h = lane >> 4;
        const int b = o % P, m = (o / P) % M, rig = o / (P * M);
        float hh[8], ll[8];
        const uint8_t *src = scratch + rig * 16 * kStride + (m * P + b) * 8 + h * kStride;
#pragma unroll
        for (int j = 0; j < 8; ++j) {  // chunk 2j + h
            const float2 v = *reinterpret_cast<const float2 *>(src + 2 * j * kStride);
            hh[j] = v.x;
            ll[j] = v.y;
        }
#pragma unroll
        for (int lvl = 0; lvl < 3; ++lvl) {
            const int off = 4 >> lvl;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (j < off) acc_add(hh[j], ll[j], hh[j + off], ll[j + off]);
        }
        const float ph = __shfl_xor_sync(0xffffffffu, hh[0], 16);
        const float pl = __shfl_xor_sync(0xffffffffu, ll[0], 16);
        acc_add(hh[0], ll[0], ph, pl);
        const int valid = m == 0 ? gi[0].valid : gi[M - 1].valid;
        const int64_t out0 = m == 0 ? gi[0].out0 : gi[M - 1].out0;
        if (h == 0 && b < B && rig < valid) y[(int64_t)b * rows + out0 + rig] = __fadd_rn(hh[0], ll[0]);
        __syncwarp();  // the scratch is read before the stage is refilled
        return;
    }
    const int b = lane % P, m = (lane / P) % M, rig = lane / (P * M);
    if (lane < M * 2 * P && b < B) {
        float h[16], l[16];
        const uint8_t *src = scratch + rig * 16 * kStride + (m * P + b) * 8;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const float2 v = *reinterpret_cast<const float2 *>(src + c * kStride);
            h[c] = v.x;
            l[c] = v.y;
        }
        // levels with pairs 8, 4, 2, 1 apart (constant trip counts, so the
        // arrays stay in registers)
#pragma unroll
        for (int lvl = 0; lvl < 4; ++lvl) {
            const int off = 8 >> lvl;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (i < off) acc_add(h[i], l[i], h[i + off], l[i + off]);
        }
        // this lane's row group by selects, not an index into gi (a run-time
        // index would put gi in local memory)
        const int valid = m == 0 ? gi[0].valid : gi[M - 1].valid;
        const int64_t out0 = m == 0 ? gi[0].out0 : gi[M - 1].out0;
        if (rig < valid) y[(int64_t)b * rows + out0 + rig] = __fadd_rn(h[0], l[0]);
    }
    __syncwarp();  // the scratch is read before the stage is refilled
}

// ---- the kernel ------------------------------------------------------------------------
// Row group: R rows.  When nb (256-weight chunks per row) is a power of two
// below 32, R = 32/nb and the group is one contiguous 4608-byte box;
// otherwise R = 1 and the row is streamed as ceil(nb/32) contiguous segments
// of up to 32 chunks.  Lane l of the warp takes chunk l of the box ("one wave
// per row, consecutive lanes read consecutive bytes", 25.2).  Work unit: M
// consecutive row groups, processed together (lane l holds chunk l of each).
// Global warp g (warp-major over CTAs) takes units g, g + TW, ...
//
// Shared memory: the batch's q8 blocks, staged once per CTA at kActStride
// bytes per chunk | [W][S] stages of M boxes of 4608 bytes.  Each warp fills
// its stages with coalesced 16-byte cp.async copies (copy p moves bytes
// 16p..16p+15 of a box to shared offset 16p; lane l's chunk lands at 144*l),
// keeping S-1 stages in flight (none with S = 1: the warp waits for its own
// copies and the CTA's other warps cover them).  (Requesting all S stages
// before the activation is staged measured slower.)  The act stride puts the
// chunks that one instruction reads on distinct bank groups.
template <int FMT, int B, int FUSE, bool DOTS = false>
constexpr int max_threads() { return warps_limit(FMT, B, FUSE, DOTS) * 32; }

// The launch bound a build is compiled for.  The row-blocked whole-row builds
// are compiled for 12 warps (at most 168 registers a thread) although the plan
// runs them with 8 beside the batch's activation: the tighter register budget
// schedules faster (128256 x 4096 batch 8: 107.3 -> 106.0 us, 14336 x 4096
// batch 8: 15.69 -> 15.59 us) and still spills nothing.
template <int FMT, int B, int FUSE, int M, int WR, bool DOTS>
constexpr int bound_threads() {
    return (M == 2 && WR && max_threads<FMT, B, FUSE, DOTS>() < 384)
               ? 384
               : max_threads<FMT, B, FUSE, DOTS>();
}

// M: row groups a warp works on at once (a work unit).  Two for Q4_K with
// several activation vectors, where the activation loads from shared memory
// are the limit; one otherwise.  WR: 0 for the general build; 16 for a build
// for rows of exactly 16 chunks (4096 columns: two whole rows a box), where
// the row width, the rows a box and the segment bookkeeping are known at
// compile time; the row-blocked launches and the batch-1 codebook launches
// take it for such rows (has_whole_row_build).
template <int FMT, int B, bool DOTS, int FUSE, bool ID, int M, int WR = 0, bool VP = false,
          bool KS = false>
__global__ void __launch_bounds__(VP ? kVpWarps * 32 : bound_threads<FMT, B, FUSE, M, WR, DOTS>(), 1)
    xq_matvec_kernel(const MatvecArgs a) {
    static_assert(!KS || (FMT != kQ4K && B == 1), "KS: the codebook table split, one vector");
    static_assert(!ID || (B == 1 && !DOTS && FUSE == 0), "the grouped form is batch 1 on q8 input");
    static_assert(!VP || (FMT == kQ4K && M == 2 && WR == 16 && !DOTS && !ID && FUSE == 0 &&
                          B == 8),
                  "warp pairs: the row-blocked Q4_K form for rows of 16 chunks, on q8 input");
    // BW: the vectors this warp computes (VP: a warp pair shares each unit and
    // its stages, each warp taking half of the vectors)
    constexpr int BW = VP ? B / 2 : B;
    static_assert(M == 1 || (M == 2 && FMT == kQ4K && !ID), "row blocking is a Q4_K form");
    static_assert(FUSE >= 0 && FUSE <= 2, "FUSE: 0 q8 input, 1 quantise x, 2 RMSNorm then quantise");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    const int W = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int half = VP ? (warp & 1) : 0;        // which half of the vectors
    const int uwarp = VP ? (warp >> 1) : warp;   // the unit stream (a pair in VP)
    const int WU = VP ? (W >> 1) : W;
    const int S = a.stages;
    static_assert(WR == 0 || WR == 16, "the whole-row build is for rows of 16 chunks");
    const int nb = WR ? WR : a.nb;
    const int R = WR ? kTileRows / WR : a.rows_per_group;
    const bool whole = WR || R > 1;  // whole rows in a box (WR: known at compile time)
    const int spr = WR ? 1 : a.segments;
    const int64_t rows = a.rows;
    const int64_t ngroups = a.groups;
    const int64_t row_bytes = (int64_t)nb * kChunkBytes;
    const int64_t act_bstride = (int64_t)nb * kActStride;
    const int nvec = ID ? a.act_vectors : B;  // staged activation vectors
    const int act_bytes = (int)((nvec * act_bstride + 127) & ~(int64_t)127);
    const uint32_t unit_bytes = (uint32_t)M * kStageBytes;  // one stage: M boxes
    uint8_t *act = smem;
    uint8_t *stage0 = smem + act_bytes + (size_t)uwarp * S * unit_bytes;
    const uint32_t stage0_u32 = smem_u32(stage0);

    // the codebook table (KS: its two split lookup tables)
    uint32_t T[4] = {a.kv[0], a.kv[1], a.kv[2], a.kv[3]};

    // 1. this warp's work units (M consecutive row groups) and their boxes;
    //    the first S-1 stages are requested before the activation is staged,
    //    so the two overlap
    const int G = gridDim.x;
    const int64_t gw = (int64_t)uwarp * G + blockIdx.x;
    const int64_t TW = (int64_t)G * WU;
    const int64_t nunits = (ngroups + M - 1) / M;
    const int64_t my_units = gw < nunits ? (nunits - 1 - gw) / TW + 1 : 0;
    const int nitems = (int)(my_units * spr);

    int64_t pu = gw;  // producer cursor: unit, segment, stage
    int ps = 0, p_stage = 0, issued = 0;
    // Resident rows: where each of this lane's nine 16-byte copies of a box
    // lands in the stage (the same for every box of the launch).  With whole
    // rows in the box (R > 1), copy k moves piece q = lane + 32k of the
    // contiguous box; with row segments (R == 1), copy 0 moves the scales of
    // chunk c0 + lane and copy k >= 1 payload piece 32(k-1) + lane of the
    // segment's 32 chunks.
    uint32_t dmap[9];
    if (FMT == kCB4R) {
#pragma unroll
        for (int k = 0; k < 9; ++k) {
            if (whole) {
                // pieces per resident row: 9 * nb, nb a power of two here
                const int q = lane + 32 * k, rp = 9 * nb;
                const int rig = (q >> (31 - __clz(nb))) / 9, r = q - rig * rp;
                dmap[k] = r < nb ? cb4r_scale_slot(rig * nb + r)
                                 : cb4r_payload_slot(rig * nb + ((r - nb) >> 3), (r - nb) & 7);
            } else {
                const int pp = 32 * (k - 1) + lane;
                dmap[k] = k == 0 ? cb4r_scale_slot(lane) : cb4r_payload_slot(pp >> 3, pp & 7);
            }
        }
    }
    // one box: row group pg, segment ps, into the stage bytes at dst_stage
    auto issue_box = [&](int64_t pg, uint32_t dst_stage) {
        const GroupInfo gi = group_info<ID>(a, pg, R);
        if (FMT == kCB4R) {
            const uint8_t *rowp = a.W + gi.row0 * row_bytes;
            if (gi.bad) {
                // an invalid expert id reads nothing
            } else if (whole) {
                const int valid = gi.valid * (int)row_bytes;
                if (valid == kStageBytes) {  // a full box: no per-copy test
#pragma unroll
                    for (int k = 0; k < 9; ++k)
                        cp_async_16(dst_stage + dmap[k], rowp + 16 * (lane + 32 * k));
                } else {
#pragma unroll
                    for (int k = 0; k < 9; ++k)
                        if (16 * (lane + 32 * k) < valid)
                            cp_async_16(dst_stage + dmap[k], rowp + 16 * (lane + 32 * k));
                }
            } else {
                const int c0 = ps * 32;
                const int n = nb - c0 < 32 ? nb - c0 : 32;  // chunks of this segment
                if (lane < n) cp_async_16(dst_stage + dmap[0], rowp + 16 * (c0 + lane));
                const uint8_t *pay = rowp + 16 * nb + 128 * c0;
#pragma unroll
                for (int k = 1; k < 9; ++k) {
                    const int pp = 32 * (k - 1) + lane;
                    if ((pp >> 3) < n) cp_async_16(dst_stage + dmap[k], pay + 16 * pp);
                }
            }
        } else {
            const uint8_t *src0;
            int valid;  // bytes of the box that exist in W
            if (whole) {
                src0 = a.W + gi.row0 * row_bytes;
                valid = gi.valid * (int)row_bytes;
            } else {
                const int c0 = ps * 32;
                src0 = a.W + gi.row0 * row_bytes + c0 * kChunkBytes;
                valid = (nb - c0 < 32 ? nb - c0 : 32) * kChunkBytes;
            }
            if (gi.bad) valid = 0;  // an invalid expert id reads nothing
            const uint8_t *src = src0 + 16 * lane;
            const uint32_t dst = dst_stage + 16u * lane;
            if (valid == kStageBytes) {
#pragma unroll
                for (int k = 0; k < 9; ++k) cp_async_16(dst + 512u * k, src + 512 * k);
            } else if (M > 1) {
                // bytes past the rows' end are zero-filled (no global read): the
                // row-blocked arithmetic runs over them unconditionally
#pragma unroll
                for (int k = 0; k < 9; ++k) {
                    const bool in = 16 * (lane + 32 * k) < valid;
                    cp_async_16_zfill(dst + 512u * k, in ? src + 512 * k : a.W, in ? 16u : 0u);
                }
            } else {
#pragma unroll
                for (int k = 0; k < 9; ++k)
                    if (16 * (lane + 32 * k) < valid) cp_async_16(dst + 512u * k, src + 512 * k);
            }
        }
    };
    auto issue_next = [&]() {
        const uint32_t dst_stage = stage0_u32 + (uint32_t)p_stage * unit_bytes;
#pragma unroll
        for (int m = 0; m < M; ++m) {
            if (VP && m != half) continue;  // the partner warp copies the other box
            if (pu * M + m < ngroups) {
                issue_box(pu * M + m, dst_stage + (uint32_t)m * kStageBytes);
            } else if (M > 1) {  // the unit's missing last group: zeros
#pragma unroll
                for (int k = 0; k < 9; ++k)
                    cp_async_16_zfill(dst_stage + (uint32_t)m * kStageBytes + 16u * lane + 512u * k,
                                      a.W, 0u);
            }
        }
        if (++ps == spr) {
            ps = 0;
            pu += TW;
        }
        if (++p_stage == S) p_stage = 0;
        ++issued;
    };

    // The weights are the one input no earlier kernel on the stream writes, so
    // their first boxes are requested before waiting for that kernel (under
    // an overlapped launch); the expert ids of the grouped form are not.
    if (ID) grid_dependency_wait();
    for (int j = 0; j < S - 1; ++j) {  // prologue: S-1 boxes in flight
        if (issued < nitems) issue_next();
        cp_async_commit();
    }
    grid_dependency_wait();     // x, q8 blocks and y belong to the stream's order
    grid_dependency_trigger();  // the next launch may start its own prologue

    // 2. the activation (a different region of shared memory than the stages)
    if (FUSE == 1 || FUSE == 2) {
        // quantise x (FUSE == 2: y = x * scale) here: warp w takes blocks w,
        // w+W, ... (vector-major) with the standalone producers' arithmetic,
        // so the same bytes.  The values of QG blocks are loaded before any
        // of them is processed: one L2 round trip per group.
        const int nblk = B * nb;
        constexpr int QG = B >= 2 ? 2 * kQuantGroup : kQuantGroup;
        // blocks quantised together (a divisor of QG).  The codebook forms
        // take one at a time: the grouped form's registers cost their main
        // loop more than it saves here (128256 x 4096 resident rows: 47.0
        // against 45.7 us a step)
        constexpr int QN = FMT == kQ4K ? 4 : 1;
        static_assert(QG % QN == 0, "whole sub-groups");
        float4 u[QG], v[QG];
        auto load_group = [&](int k0) {
#pragma unroll
            for (int j = 0; j < QG; ++j) {
                const int blk = k0 + j * W;
                if (blk < nblk) {
                    const float4 *src = reinterpret_cast<const float4 *>(a.x + (int64_t)blk * 256 + lane * 8);
                    u[j] = __ldg(src);
                    v[j] = __ldg(src + 1);
                }
            }
        };
        load_group(warp);  // in flight while the RMSNorm scale is taken
        // FUSE == 2: the RMSNorm scale of each vector (warp w takes vectors
        // w, w+W, ...; one vector with eight warps or more, warps 0..7
        // together) is parked in bytes 320..335 of the vector's first staged
        // block (stride padding that nothing else reads or writes)
        if (FUSE == 2) {
            if (B == 1 && W >= 8) {
                // one vector and eight warps or more: warps 0..7 are the
                // workgroup (rms_scale_block: one L2 round trip per 32 rows
                // instead of per 8); its wave partials meet in warp 0's last
                // stage, to which no copy is issued before the main loop
                if (warp < 8) {
                    float *s_wave = reinterpret_cast<float *>(smem + act_bytes + (S - 1) * unit_bytes);
                    const float sc = rms_scale_block(a.x, (int64_t)nb * 256, s_wave, true);
                    if (threadIdx.x == 0) *reinterpret_cast<float *>(act + kActNormAt) = sc;
                }
            } else {
                for (int b = warp; b < B; b += W) {
                    const float sc = rms_scale_warp(a.x + (int64_t)b * nb * 256, (int64_t)nb * 256, lane);
                    if (lane == 0) *reinterpret_cast<float *>(act + b * act_bstride + kActNormAt) = sc;
                }
            }
            __syncthreads();
        }
        // The round's blocks are quantised QN at a time (q8_quantize_lanes:
        // their steps interleaved, one division pass); a round with one block
        // for this warp takes the one-block form.  Values, sums and scale go to
        // the staged block; the Q4_K split sums are formed afterwards from the
        // staged sums, one block a thread.
        auto quantise_round = [&](int k0, int j0, auto tag) {
            constexpr int N = decltype(tag)::value;
            float vals[N][8];
#pragma unroll
            for (int jj = 0; jj < N; ++jj) {
                const int j = j0 + jj, blk = k0 + j * W;
                const bool in = N == 1 || blk < nblk;  // one block: always in range (warp-uniform)
                vals[jj][0] = in ? u[j].x : 0.0f;
                vals[jj][1] = in ? u[j].y : 0.0f;
                vals[jj][2] = in ? u[j].z : 0.0f;
                vals[jj][3] = in ? u[j].w : 0.0f;
                vals[jj][4] = in ? v[j].x : 0.0f;
                vals[jj][5] = in ? v[j].y : 0.0f;
                vals[jj][6] = in ? v[j].z : 0.0f;
                vals[jj][7] = in ? v[j].w : 0.0f;
                if (FUSE == 2 && in) {
                    const int b = blk / nb;
                    const float ns = *reinterpret_cast<const float *>(act + b * act_bstride + kActNormAt);
#pragma unroll
                    for (int i = 0; i < 8; ++i) vals[jj][i] = __fmul_rn(vals[jj][i], ns);
                }
            }
            Q8Lane r[N];
            q8_quantize_lanes<N, FMT == kQ4K>(vals, r, lane);  // the codebook builds: the clamp form
#pragma unroll
            for (int jj = 0; jj < N; ++jj) {
                const int blk = k0 + (j0 + jj) * W;
                if (blk >= nblk) break;  // warp-uniform
                uint8_t *dst = act + blk * kActStride;
                const Q8Lane &q = r[jj];
                if (FMT == kQ4K) {
                    *reinterpret_cast<uint2 *>(dst + lane * 8) = make_uint2(q.w0, q.w1);
                } else {
                    // interleaved order: lane 4k+i writes words 2i, 2i+1 of
                    // sub-block k, made of its words i and i+4 (lanes 4k + i/2
                    // and 4k + 2 + i/2 hold them)
                    const int i = lane & 3, src = (lane & ~3) + (i >> 1);
                    const uint32_t v0 = __shfl_sync(0xffffffffu, q.w0, src);
                    const uint32_t v1 = __shfl_sync(0xffffffffu, q.w1, src);
                    const uint32_t u0 = __shfl_sync(0xffffffffu, q.w0, src + 2);
                    const uint32_t u1 = __shfl_sync(0xffffffffu, q.w1, src + 2);
                    const uint32_t wa = (i & 1) ? v1 : v0, wb = (i & 1) ? u1 : u0;
                    *reinterpret_cast<uint2 *>(dst + lane * 8) =
                        make_uint2(interleave_lo(wa, wb), interleave_hi(wa, wb));
                }
                if ((lane & 3) == 0) *reinterpret_cast<int *>(dst + kQ8SumAt + (lane >> 2) * 4) = q.sum;
                if (lane == 0) *reinterpret_cast<float *>(dst + kQ8ScaleAt) = q.d;
            }
        };
        for (int k0 = warp; k0 < nblk; k0 += QG * W) {
            if (k0 != warp) load_group(k0);
            if constexpr (FMT == kCB4) {
                // one call site a block: in the raw codebook build this form
                // left the main loop at 688 warp-instructions a box against
                // 735 with the two call sites below (128256 x 4096: 45.8
                // against 46.2 us a step); the resident-row build measured the
                // other way (46.8 against 45.6 us), the Q4_K builds alike
#pragma unroll
                for (int j = 0; j < QG; ++j) {
                    if (k0 + j * W >= nblk) break;  // warp-uniform
                    quantise_round(k0, j, IntTag<1>{});
                }
            } else if (k0 + W >= nblk) {
                quantise_round(k0, 0, IntTag<1>{});
            } else {
#pragma unroll
                for (int j0 = 0; j0 < QG; j0 += QN)
                    if (k0 + j0 * W < nblk) quantise_round(k0, j0, IntTag<QN>{});  // warp-uniform
            }
        }
        if (FMT == kQ4K) {
            __syncthreads();  // every block's sums are staged
            for (int blk = threadIdx.x; blk < nblk; blk += blockDim.x) {
                const uint4 *sums = reinterpret_cast<const uint4 *>(act + blk * kActStride + kQ8SumAt);
                *reinterpret_cast<uint4 *>(act + blk * kActStride + kActSplitAt) = split_sums(sums[0], sums[1]);
            }
        }
    } else if (FMT == kQ4K && nvec * nb >= kStageAsyncBlocks) {
        // Many q8 blocks: bytes 0..303 of every block by asynchronous copies,
        // all in flight at once (one commit group after the prologue's weight
        // boxes, so waiting for it waits for those too), then each block's
        // split sums from its staged int32 sums.
        const int nblk = nvec * nb;
        const uint32_t act_u32 = smem_u32(act);
        for (int i = threadIdx.x; i < nblk * 19; i += blockDim.x) {
            const int blk = i / 19, piece = i - 19 * blk;
            cp_async_16(act_u32 + (uint32_t)(blk * kActStride + 16 * piece),
                        a.xq + (int64_t)blk * kQ8Bytes + 16 * piece);
        }
        cp_async_commit();
        cp_async_wait_pending(0);
        __syncthreads();
        for (int blk = threadIdx.x; blk < nblk; blk += blockDim.x) {
            const uint4 *sums = reinterpret_cast<const uint4 *>(act + blk * kActStride + kQ8SumAt);
            const uint4 sp = split_sums(sums[0], sums[1]);
            *reinterpret_cast<uint4 *>(act + blk * kActStride + kActSplitAt) = sp;
        }
    } else if (FMT == kQ4K) {
        // Few q8 blocks: bytes 0..303 of every block, then its split sums
        // (item 19 of the block, from its int32 sums), by loads and stores:
        // each thread issues the loads of kStageItems items before it stores
        // any, one L2 round trip per group of items, and the weight boxes
        // already in flight are not waited for here.
        const int n = nvec * nb * 20;
        for (int i0 = threadIdx.x; i0 < n; i0 += kStageItems * blockDim.x) {
            uint4 u[kStageItems], v[kStageItems];
#pragma unroll
            for (int j = 0; j < kStageItems; ++j) {
                const int i = i0 + j * blockDim.x;
                v[j] = make_uint4(0u, 0u, 0u, 0u);
                if (i < n) {
                    const int blk = i / 20, piece = i - 20 * blk;
                    const uint4 *src = reinterpret_cast<const uint4 *>(a.xq + (int64_t)blk * kQ8Bytes);
                    u[j] = __ldg(src + (piece < 19 ? piece : 16));
                    if (piece == 19) v[j] = __ldg(src + 17);
                }
            }
#pragma unroll
            for (int j = 0; j < kStageItems; ++j) {
                const int i = i0 + j * blockDim.x;
                if (i < n) {
                    const int blk = i / 20, piece = i - 20 * blk;
                    *reinterpret_cast<uint4 *>(act + blk * kActStride + 16 * piece) =
                        piece < 19 ? u[j] : split_sums(u[j], v[j]);
                }
            }
        }
    } else {
        // The values of every q8 block in interleaved order (one 32-value
        // sub-block an item), then bytes 256..303 (three items of one piece),
        // loads issued kStageItems items at a time as above.
        const int n = nvec * nb * 11;
        for (int i0 = threadIdx.x; i0 < n; i0 += kStageItems * blockDim.x) {
            uint4 u[kStageItems], v[kStageItems];
#pragma unroll
            for (int j = 0; j < kStageItems; ++j) {
                const int i = i0 + j * blockDim.x;
                v[j] = make_uint4(0u, 0u, 0u, 0u);
                if (i < n) {
                    const int blk = i / 11, part = i - 11 * blk;
                    const uint4 *src = reinterpret_cast<const uint4 *>(a.xq + (int64_t)blk * kQ8Bytes);
                    u[j] = __ldg(src + (part < 8 ? 2 * part : 8 + part));
                    if (part < 8) v[j] = __ldg(src + 2 * part + 1);
                }
            }
#pragma unroll
            for (int j = 0; j < kStageItems; ++j) {
                const int i = i0 + j * blockDim.x;
                if (i < n) {
                    const int blk = i / 11, part = i - 11 * blk;
                    uint4 *dst = reinterpret_cast<uint4 *>(act + blk * kActStride);
                    if (part < 8) {
                        const uint32_t in[8] = {u[j].x, u[j].y, u[j].z, u[j].w,
                                                v[j].x, v[j].y, v[j].z, v[j].w};
                        dst[2 * part] =
                            make_uint4(interleave_lo(in[0], in[4]), interleave_hi(in[0], in[4]),
                                       interleave_lo(in[1], in[5]), interleave_hi(in[1], in[5]));
                        dst[2 * part + 1] =
                            make_uint4(interleave_lo(in[2], in[6]), interleave_hi(in[2], in[6]),
                                       interleave_lo(in[3], in[7]), interleave_hi(in[3], in[7]));
                    } else {
                        dst[8 + part] = u[j];  // pieces 16..18
                    }
                }
            }
        }
    }
    __syncthreads();

    const int64_t dots_row = (int64_t)nb * 8;
    const int64_t dots_bstride = rows * dots_row;
    const int width = whole ? nb : 32;  // lanes that share a row
    const int rig = whole ? lane / nb : 0;  // this lane's row within a group
    int c_stage = 0;
    for (int64_t u = gw; u < nunits; u += TW) {
        GroupInfo gi[M];
#pragma unroll
        for (int m = 0; m < M; ++m) {
            if (u * M + m < ngroups) {
                gi[m] = group_info<ID>(a, u * M + m, R);
            } else {
                gi[m].row0 = gi[m].out0 = 0;
                gi[m].valid = 0;
                gi[m].vec = 0;
                gi[m].bad = false;
            }
        }
        float hi[M][BW], lo[M][BW];
#pragma unroll
        for (int m = 0; m < M; ++m)
#pragma unroll
            for (int b = 0; b < BW; ++b) hi[m][b] = lo[m][b] = 0.0f;
        for (int s = 0; s < spr; ++s) {
            if constexpr (VP) {
                // the unit's copies were issued one unit ahead, half by each warp
                // of the pair: wait for this warp's, then meet the partner, after
                // which both have landed and both warps are done with the stage
                // read in the previous unit, which is refilled next (S >= 2)
                cp_async_wait_pending(S - 2);
                __syncwarp();
                pair_barrier(uwarp);
                if (issued < nitems) issue_next();
                cp_async_commit();
            } else {
                if (issued < nitems) issue_next();
                cp_async_commit();
                cp_async_wait_pending(S - 1);  // this lane's copies of the stage landed
                __syncwarp();                  // ... and every other lane's
            }
            const int c = whole ? (lane & (nb - 1)) : s * 32 + lane;
            const uint8_t *st = stage0 + c_stage * unit_bytes + lane * kChunkBytes;
            // (M > 1 reads the activation of chunks past the row's end too, and
            // multiplies it by zero-filled weights: a real block keeps it finite)
            const int ca = M > 1 && c >= nb ? nb - 1 : c;
            const ActSmem as{act + (gi[0].vec + half * BW) * act_bstride + ca * kActStride,
                             act_bstride};
            if (M > 1) {
                const uint8_t *w[M];
                bool ok[M];
                int32_t *dp[M];
                bool any = false;
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    w[m] = st + m * kStageBytes;
                    ok[m] = rig < gi[m].valid && c < nb;
                    any |= ok[m];
                    dp[m] = DOTS && ok[m] ? a.dots + (gi[m].row0 + rig) * dots_row + c * 8 : nullptr;
                }
                if (any) {
                    if (spr == 1)  // one segment a row: every chunk is its lane's first
                        q4k_chunks<BW, M, DOTS, true>(w, ok, as, hi, lo, dp, dots_bstride);
                    else  // (hi, lo) start at zero, to which an exact add is an assignment
                        q4k_chunks<BW, M, DOTS, false>(w, ok, as, hi, lo, dp, dots_bstride);
                }
            } else {
                const bool ok = rig < gi[0].valid && c < nb && !gi[0].bad;
                if (ok) {
                    int32_t *dp = DOTS ? a.dots + (gi[0].row0 + rig) * dots_row + c * 8 : nullptr;
                    if (FMT == kQ4K)
                        q4k_chunk<BW, DOTS>(st, as, hi[0], lo[0], dp, dots_bstride, s == 0);
                    else if (FMT == kCB4 && spr == 1)  // one segment a row: the lane's first chunk
                        cb4_chunk<BW, DOTS, true, KS>(st, as, T, hi[0], lo[0], dp, dots_bstride);
                    else if (FMT == kCB4)
                        cb4_chunk<BW, DOTS, false, KS>(st, as, T, hi[0], lo[0], dp, dots_bstride);
                    else if (spr == 1)
                        cb4r_chunk<BW, DOTS, true, KS>(st - lane * kChunkBytes, lane, as, T,
                                                       hi[0], lo[0], dp, dots_bstride);
                    else
                        cb4r_chunk<BW, DOTS, false, KS>(st - lane * kChunkBytes, lane, as, T,
                                                        hi[0], lo[0], dp, dots_bstride);
                }
            }
            __syncwarp();
            if (++c_stage == S) c_stage = 0;
        }
        bool stored = false;
        // rows of 16 chunks, three vectors or more: the transposed reduction
        // (with one or two vectors it leaves most lanes without an output, and
        // the shuffle reduction is faster: 14336 x 4096 batch 2, 8.64 against
        // 8.37 us)
        if constexpr (M == 2 && WR == 16 && !DOTS && BW >= 3) {
            // scratch: the stage just read, or with warp pairs (whose stages are
            // shared) this warp's own region after all the stages
            const int used = c_stage == 0 ? S - 1 : c_stage - 1;
            uint8_t *scratch = VP ? smem + act_bytes + (size_t)WU * S * unit_bytes +
                                        (size_t)warp * kVpScratchBytes
                                  : stage0 + used * unit_bytes;
            reduce_rows16_store<M, BW>(hi, lo, scratch, lane, gi, a.y + (int64_t)half * BW * rows,
                                       rows);
            stored = true;
        }
        if (!DOTS && !stored) {
            constexpr int P = Pow2Ceil<BW>::v;
#pragma unroll
            for (int m = 0; m < M; ++m) {
                float h[P], l[P];
#pragma unroll
                for (int b = 0; b < P; ++b) {
                    h[b] = b < BW ? hi[m][b] : 0.0f;
                    l[b] = b < BW ? lo[m][b] : 0.0f;
                }
                int base, nlive, keep;
                halving_reduce<P>(h, l, width, lane, base, nlive, keep);
                if ((lane & keep) == 0 && rig < gi[m].valid) {
                    float *yb = a.y + (int64_t)(half * BW + base) * rows + gi[m].out0 + rig;
                    const float nan = __int_as_float(0x7FC00000);
                    if (P == 1 || nlive == 1) {  // rows of P lanes or more: one value a lane
                        if (base < BW) yb[0] = gi[m].bad ? nan : __fadd_rn(h[0], l[0]);
                    } else {
#pragma unroll
                        for (int i = 0; i < P; ++i)
                            if (i < nlive && base + i < BW)
                                yb[(int64_t)i * rows] = gi[m].bad ? nan : __fadd_rn(h[i], l[i]);
                    }
                    if (ID && gi[m].bad && rig == 0 && (lane & (width - 1)) == 0)
                        atomicOr(a.status, kStatusBadExpertId);
                }
            }
        }
    }
    cp_async_wait_all();  // only empty groups can remain; keeps the exit clean
}

// Builds for rows of 16 chunks (WR = 16): the row-blocked Q4_K kernels, and
// the batch-1 codebook kernels (raw or resident rows; 128256 x 4096: 56.7 ->
// 51.8 us, 11008 x 4096: 7.33 -> 6.80 us).  The batch-1 Q4_K kernel is
// HBM-bound and measured no faster with a whole-row build.
template <int FMT, int B, bool DOTS, int FUSE, bool ID, int M>
constexpr bool has_whole_row_build() {
    return M == 2 || (M == 1 && FMT != kQ4K && B == 1 && !DOTS && !ID);
}

// Builds for warp pairs (VP): the row-blocked Q4_K mat-vec on q8 blocks for
// rows of 16 chunks at 8 vectors, launched when the plan asks for them.
template <int FMT, int B, bool DOTS, int FUSE, bool ID, int M>
constexpr bool has_vector_pair_build() {
    return FMT == kQ4K && M == 2 && !DOTS && !ID && FUSE == 0 && B == 8;
}

template <int FMT, int B, bool DOTS, int FUSE, bool ID = false, int M = 1>
inline cudaError_t launch_matvec_t(const MatvecArgs &a, dim3 grid, dim3 block, size_t smem,
                                   cudaStream_t s) {
    if constexpr (FMT != kQ4K && B == 1) {  // one vector: the split codebook table, if it splits
        if (a.kv_split) {
            if constexpr (has_whole_row_build<FMT, B, DOTS, FUSE, ID, M>()) {
                if (a.nb == 16)
                    return launch_kernel(xq_matvec_kernel<FMT, B, DOTS, FUSE, ID, M, 16, false, true>,
                                         grid, block, smem, s, a.overlap != 0, a);
            }
            return launch_kernel(xq_matvec_kernel<FMT, B, DOTS, FUSE, ID, M, 0, false, true>, grid,
                                 block, smem, s, a.overlap != 0, a);
        }
    }
    if constexpr (has_vector_pair_build<FMT, B, DOTS, FUSE, ID, M>()) {
        if (a.vector_pairs && a.nb == 16)
            return launch_kernel(xq_matvec_kernel<FMT, B, DOTS, FUSE, ID, M, 16, true>, grid, block,
                                 smem, s, a.overlap != 0, a);
    }
    if constexpr (has_whole_row_build<FMT, B, DOTS, FUSE, ID, M>()) {
        if (a.nb == 16)
            return launch_kernel(xq_matvec_kernel<FMT, B, DOTS, FUSE, ID, M, 16>, grid, block,
                                 smem, s, a.overlap != 0, a);
    }
    return launch_kernel(xq_matvec_kernel<FMT, B, DOTS, FUSE, ID, M>, grid, block, smem, s,
                         a.overlap != 0, a);
}

template <int FMT, int B, bool DOTS, int FUSE, bool ID = false, int M = 1>
inline cudaError_t configure_t(int smem_optin) {
    if constexpr (FMT != kQ4K && B == 1) {
        if constexpr (has_whole_row_build<FMT, B, DOTS, FUSE, ID, M>()) {
            const cudaError_t e = cudaFuncSetAttribute(
                xq_matvec_kernel<FMT, B, DOTS, FUSE, ID, M, 16, false, true>,
                cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
            if (e != cudaSuccess) return e;
        }
        const cudaError_t e = cudaFuncSetAttribute(
            xq_matvec_kernel<FMT, B, DOTS, FUSE, ID, M, 0, false, true>,
            cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
        if (e != cudaSuccess) return e;
    }
    if constexpr (has_vector_pair_build<FMT, B, DOTS, FUSE, ID, M>()) {
        const cudaError_t e = cudaFuncSetAttribute(
            xq_matvec_kernel<FMT, B, DOTS, FUSE, ID, M, 16, true>,
            cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
        if (e != cudaSuccess) return e;
    }
    if constexpr (has_whole_row_build<FMT, B, DOTS, FUSE, ID, M>()) {
        const cudaError_t e = cudaFuncSetAttribute(xq_matvec_kernel<FMT, B, DOTS, FUSE, ID, M, 16>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   smem_optin);
        if (e != cudaSuccess) return e;
    }
    return cudaFuncSetAttribute(xq_matvec_kernel<FMT, B, DOTS, FUSE, ID, M>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
}

// kind: 0 = mat-vec on q8 blocks, 1 = the same with the exact dots,
// 2 = fused quantise + mat-vec, 3 = grouped experts (batch 1, q8 input),
// 4 = fused RMSNorm + quantise + mat-vec.  M: row groups per work unit
// (batch 1 always takes M = 1).
template <int FMT, int M>
inline cudaError_t launch_matvec_fmt(const MatvecArgs &a, int batch, int kind, dim3 grid,
                                     dim3 block, size_t smem, cudaStream_t s) {
    if constexpr (M == 1) {
        if (kind == 3)
            return batch == 1 ? launch_matvec_t<FMT, 1, false, 0, true>(a, grid, block, smem, s)
                              : cudaErrorInvalidValue;
        if (batch == 1)
            return kind == 1   ? launch_matvec_t<FMT, 1, true, 0>(a, grid, block, smem, s)
                   : kind == 2 ? launch_matvec_t<FMT, 1, false, 1>(a, grid, block, smem, s)
                   : kind == 4 ? launch_matvec_t<FMT, 1, false, 2>(a, grid, block, smem, s)
                               : launch_matvec_t<FMT, 1, false, 0>(a, grid, block, smem, s);
    } else {
        if (kind == 3 || batch == 1) return cudaErrorInvalidValue;
    }
#define XQ_CASE(BB, MM)                                                                         \
    case BB:                                                                                    \
        return kind == 1   ? launch_matvec_t<FMT, BB, true, 0, false, MM>(a, grid, block, smem, s)  \
               : kind == 2 ? launch_matvec_t<FMT, BB, false, 1, false, MM>(a, grid, block, smem, s) \
               : kind == 4 ? launch_matvec_t<FMT, BB, false, 2, false, MM>(a, grid, block, smem, s) \
                           : launch_matvec_t<FMT, BB, false, 0, false, MM>(a, grid, block, smem, s);
    switch (batch) {
        XQ_CASE(2, M)
        XQ_CASE(3, M)
        XQ_CASE(4, M)
        XQ_CASE(5, M)
        XQ_CASE(6, M)
        XQ_CASE(7, M)
        XQ_CASE(8, M)
        default:
            return cudaErrorInvalidValue;
    }
#undef XQ_CASE
}

template <int FMT, int M>
inline cudaError_t configure_fmt(int smem_optin) {
    cudaError_t e = cudaSuccess;
#define XQ_CFG(BB, MM)                                                                  \
    if (e == cudaSuccess) e = configure_t<FMT, BB, false, 0, false, MM>(smem_optin); \
    if (e == cudaSuccess) e = configure_t<FMT, BB, true, 0, false, MM>(smem_optin);  \
    if (e == cudaSuccess) e = configure_t<FMT, BB, false, 1, false, MM>(smem_optin); \
    if (e == cudaSuccess) e = configure_t<FMT, BB, false, 2, false, MM>(smem_optin);
    if constexpr (M == 1) {
        XQ_CFG(1, 1)
        if (e == cudaSuccess) e = configure_t<FMT, 1, false, 0, true>(smem_optin);
    }
    XQ_CFG(2, M)
    XQ_CFG(3, M)
    XQ_CFG(4, M)
    XQ_CFG(5, M)
    XQ_CFG(6, M)
    XQ_CFG(7, M)
    XQ_CFG(8, M)
#undef XQ_CFG
    return e;
}

}  // namespace xq
