// Q4_K mat-vec on the fifth-generation tensor cores (tcgen05): rows of 16
// chunks (4096 columns), 5..8 vectors on q8 blocks.
//
// The integer sub-block dots ("25 -- Writing XPU Kernels" 25.2: dot the
// quantised values, scale once per super-block) are a dense product of the
// 4-bit codes with the int8 activations, so at 5..8 vectors they are taken by
// tcgen05.mma (kind::f16, f32 accumulators in tensor memory) instead of dp4a.
// They stay exact integers: a code q is made the f16 value 1024 + q (a high
// nibble 1024 + 16q: a mask and an OR put the nibble under the f16 exponent
// of 1024), then one fused multiply-add by the sub-block's six-bit scale sc
// and -1024 * sc (sc/16 and -64 * sc) gives the exact f16 q * sc (at most
// 945); an activation value enters as itself.  Sub-blocks 0..3 and 4..7 each
// accumulate in one f32 accumulator, whose partial sums are integers below
// 4 * 32 * 945 * 127 < 2^24, so f32 holds them exactly and cvt.rni reads
// them back: their sum is S1.  From there the arithmetic is the dp4a
// kernel's: the same integers S1 and S2, the same epilogue, and the same
// pairing tree over a row's 16 chunk terms, so y has the same bits.
//
// A CTA of seventeen warps owns tiles of 128 rows (one tensor-memory lane a
// row; the warps of a quarter share lanes 32(w%4) .. 32(w%4)+31 and their 32
// rows).  The roles run side by side, paced only by mbarriers:
//   - decoders (warps 0-7, two a quarter): the quarter's two stage its 32
//     rows' 144-byte chunks by cp.async (three stages) and meet on a named
//     barrier; warp w unpacks groups 2(w/4), 2(w/4)+1 of its rows' codes to
//     f16 pairs and writes them to tensor memory (tcgen05.st, the A operand,
//     128 x 256), then arrives on A-full;
//   - the issuer (warp 16) waits for A-full and for the accumulators to be
//     free, issues 16 tcgen05.mma (two K=16 slices a sub-block, sub-blocks
//     0..3 into one accumulator and 4..7 into another, M = 128, N = 16: the
//     8 vectors twice, the B descriptor's N-group stride being 0) and
//     commits to D-full;
//   - epilogue warps (8-15, two a quarter): warp w waits for D-full, reads
//     vectors 4((w-8)/4) .. +3 of its rows' two accumulators (tcgen05.ld),
//     arrives on D-empty and forms the chunk's terms, with the rows' scales
//     read from global memory one step ahead.
// A and the accumulators are double-buffered (A in columns 0..255, the
// accumulators in 256..319 of the 512 allocated).
// The activation is the B operand, staged once per CTA as f16 in the
// canonical K-major layout without swizzle: core matrices of 8 vectors x 8
// values (16 bytes a vector), the next 8 values of K 128 bytes on.
//
// Chunk order and the tree: chunks are taken in the order 0, 8, 4, 12, 2, 10,
// 6, 14, 1, 9, 5, 13, 3, 11, 7, 15 (the bit reversal of the step), so the
// tree's first level (chunks 8 apart) pairs consecutive steps and every
// upper level (4, 2, 1 apart) consecutive pairs: a binary counter over the
// steps, with one pending partial sum a level.
//
// Fragment order: within a K=16 slice (16 payload bytes of one group, low or
// high nibbles), column 2i of the slice holds the codes of bytes 4i and
// 4i + 2, column 2i + 1 those of bytes 4i + 1 and 4i + 3 (a mask of the word,
// or of the word >> 8); the activation is staged in the same order.  (Which
// K index a value takes inside a product does not change the sum.)
#pragma once

#include "xq_matvec.cuh"

namespace xq {

// ---- tcgen05 / mbarrier wrappers (inline PTX, sm_100 family) --------------------------
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// 32 lanes x 16 columns of 32 bits from registers into this warp's lanes
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}
// 32 lanes x 4 columns of 32 bits into registers
__device__ __forceinline__ void tc_ld4(uint32_t taddr, uint32_t (&v)[4]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
                 : "r"(taddr)
                 : "memory");
}
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// D (tensor memory) = A (tensor memory) x B (shared memory descriptor), or +=
__device__ __forceinline__ void tc_mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive on the mbarrier once every tcgen05 operation this thread issued is done
__device__ __forceinline__ void tc_commit(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t mbar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(mbar), "r"(parity)
        : "memory");
    return done != 0;
}

// four int8 values (a q8 word) -> two f16 pairs: (x0, x2) and (x1, x3), exact
__device__ __forceinline__ uint2 q8_word_to_f16_tc(uint32_t w) {
    const uint32_t u = w ^ 0x80808080u;                   // x + 128, unsigned
    const uint32_t p02 = prmt(u, 0x64646464u, 0x4240u);  // f16 1024 + u0, 1024 + u2
    const uint32_t p13 = prmt(u, 0x64646464u, 0x4341u);
    const __half2 off = __float2half2_rn(1152.0f);
    const __half2 r02 = __hsub2(*reinterpret_cast<const __half2 *>(&p02), off);
    const __half2 r13 = __hsub2(*reinterpret_cast<const __half2 *>(&p13), off);
    return make_uint2(*reinterpret_cast<const uint32_t *>(&r02),
                      *reinterpret_cast<const uint32_t *>(&r13));
}

// the chunk taken at step s of a tile: the bit reversal of s (four bits)
__device__ __forceinline__ constexpr int tc_step_chunk(int s) {
    return ((s & 1) << 3) | ((s & 2) << 1) | ((s >> 1) & 2) | ((s >> 3) & 1);
}

// The shared-memory descriptor of K=16 slice `slice` of chunk `c` of the
// staged activation: canonical K-major, no swizzle; leading (K) byte offset
// 128 (the next 8 values), stride (N-group) byte offset 0 (N = 16 reads the 8
// vectors twice), descriptor version 1.
__device__ __forceinline__ uint64_t tc_act_desc(uint32_t act_u32, int c, int slice) {
    const uint32_t addr = act_u32 + (uint32_t)(c * 16 + slice) * 256u;
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)(128u >> 4) << 16) | (1ull << 46);
}

// instruction descriptor: f32 accumulate, f16 A and B, both K-major, N = 16, M = 128
constexpr uint32_t kTcIdesc = (1u << 4) | ((16u >> 3) << 17) | ((128u >> 4) << 24);

// bounded wait on an mbarrier phase; false when it ran out
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t mbar, uint32_t parity) {
    for (uint32_t spins = 0; spins < kTcSpinLimit; ++spins)
        if (mbar_try_wait(mbar, parity)) return true;
    return false;
}
__device__ __forceinline__ void mbar_arrive(uint32_t mbar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(mbar) : "memory");
}
// named barrier of a quarter's two decoder warps (ids 1..4; 0 is __syncthreads)
__device__ __forceinline__ void decoder_barrier(int quarter) {
    asm volatile("bar.sync %0, 64;" ::"r"(1 + quarter) : "memory");
}

template <int B>
__global__ void __maxnreg__(kTcMaxRegs) xq_tc_q4k_kernel(const MatvecArgs a) {
    static_assert(B >= 1 && B <= 8, "up to eight vectors (the N = 16 product holds them twice)");
    constexpr int nb = kTcChunks;
    constexpr int64_t kRowBytes = (int64_t)nb * kChunkBytes;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const bool issuer = warp == kTcWorkWarps;  // warp 16: issues the products
    const bool decoder = warp < 8;             // warps 0-7; 8-15 the epilogue
    const int quarter = warp & 3, half = (warp >> 2) & 1;  // lanes 32*quarter..; groups / vectors
    const int qtid = half * 32 + lane;  // 0..63 among the quarter's decoders
    const int S = a.stages;
    const int64_t rows = a.rows;
    const int64_t ntiles = (rows + kTcRows - 1) / kTcRows;
    const int64_t my_tiles = blockIdx.x < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int nitems = (int)(my_tiles * nb);  // steps: (tile, chunk)
    uint8_t *act = smem;  // the B operand
    const uint32_t act_u32 = smem_u32(act);
    const float *xs_tab = reinterpret_cast<const float *>(smem + kTcXsAt);
    const uint4 *split_tab = reinterpret_cast<const uint4 *>(smem + kTcSplitAt);
    // this quarter's stages: 32 rows x 144 bytes each
    uint8_t *qstage0 = smem + kTcStagesAt + (size_t)quarter * S * kTcQStageBytes;
    const uint32_t qstage0_u32 = smem_u32(qstage0);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kTcStagesAt + 4 * S * kTcQStageBytes);
    // a give-up flag, then mbarriers: A-full[2] (8 decoder arrivals), D-full[2]
    // (the commit), D-empty[2] (8 epilogue arrivals)
    volatile uint32_t *abort_flag = tmem_slot + 1;
    const uint32_t bar0 = smem_u32(tmem_slot + 2);
    const uint32_t a_full = bar0, d_full = bar0 + 16, d_empty = bar0 + 32;

    if (warp == 0) {  // tensor memory: A0 0..127, A1 128..255, D0 256..287, D1 288..319
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"((uint32_t)kTcTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        *abort_flag = 0u;
        for (int b = 0; b < 2; ++b) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a_full + 8 * b), "r"(8u) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(d_full + 8 * b), "r"(1u) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(d_empty + 8 * b), "r"(8u) : "memory");
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }

    // producer (each quarter's two decoders for its 32 rows): step ps of tile
    // pt into stage p_stage; piece p = qtid + 64k (< 288) is byte 16(p % 9) of
    // the chunk of row p / 9 (rows past the end zero-filled)
    int64_t pt = blockIdx.x;
    int ps = 0, p_stage = 0, issued = 0;
    auto issue_next = [&]() {
        const int c = tc_step_chunk(ps);
        const int64_t row0 = pt * kTcRows + 32 * quarter;
        const uint8_t *base = a.W + row0 * kRowBytes + c * kChunkBytes;
        const int64_t rows_left = rows - row0;
        const uint32_t dst = qstage0_u32 + (uint32_t)p_stage * kTcQStageBytes;
#pragma unroll
        for (int k = 0; k < 5; ++k) {
            const int p = qtid + 64 * k;
            if (p < 32 * 9) {
                const int r = p / 9, q = p - 9 * r;
                const bool in = r < rows_left;
                cp_async_16_zfill(dst + 16u * p, in ? base + r * kRowBytes + 16 * q : a.W, in ? 16u : 0u);
            }
        }
        if (++ps == nb) {
            ps = 0;
            pt += gridDim.x;
        }
        if (++p_stage == S) p_stage = 0;
        ++issued;
    };
    if (decoder) {
        for (int j = 0; j < S - 1; ++j) {  // the weights are read by nothing before this grid
            if (issued < nitems) issue_next();
            cp_async_commit();
        }
    }
    grid_dependency_wait();

    // the activation: values as f16, per chunk 16 slices of 256 bytes (slice
    // gq*4 + part*2 + h: values 64gq + 32part + 16h .. +15, the two 8-value
    // halves 128 bytes apart, each vector's 8 values 16 bytes); vectors past
    // B are zeros; every thread's loads in flight together
    {
        constexpr int kN = 8 * nb * 16;  // 16-byte pieces
        constexpr int kPer = (kN + kTcThreads - 1) / kTcThreads;
        uint4 w4[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int i = tid + kTcThreads * k, v = i / (nb * 16), c = (i / 16) % nb, qd = i % 16;
            w4[k] = make_uint4(0u, 0u, 0u, 0u);
            if (i < kN && v < B)
                w4[k] = __ldg(reinterpret_cast<const uint4 *>(a.xq + ((int64_t)v * nb + c) * kQ8Bytes) + qd);
        }
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int i = tid + kTcThreads * k, v = i / (nb * 16), c = (i / 16) % nb, qd = i % 16;
            if (i >= kN) break;
            const uint32_t ww[4] = {w4[k].x, w4[k].y, w4[k].z, w4[k].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int w = 4 * qd + e, slice = w >> 2, i4 = w & 3;  // q8 word w: values 4w..4w+3
                *reinterpret_cast<uint2 *>(act + (c * 16 + slice) * 256 + (i4 >> 1) * 128 + v * 16 + (i4 & 1) * 8) =
                    q8_word_to_f16_tc(ww[e]);
            }
        }
    }
    if (tid < nb * 8) {  // per (chunk, vector): the scale and the split sums
        const int c = tid >> 3, v = tid & 7;
        uint4 s0 = make_uint4(0u, 0u, 0u, 0u), s1 = s0;
        float xs = 0.0f;
        if (v < B) {
            const uint8_t *blk = a.xq + ((int64_t)v * nb + c) * kQ8Bytes;
            s0 = __ldg(reinterpret_cast<const uint4 *>(blk + kQ8SumAt));
            s1 = __ldg(reinterpret_cast<const uint4 *>(blk + kQ8SumAt + 16));
            xs = __ldg(reinterpret_cast<const float *>(blk + kQ8ScaleAt));
        }
        reinterpret_cast<float *>(smem + kTcXsAt)[c * 8 + v] = xs;
        reinterpret_cast<uint4 *>(smem + kTcSplitAt)[c * 8 + v] = split_sums(s0, s1);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor cores
    grid_dependency_trigger();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // A wait that runs out sets the flag and the status bit; from then on no
    // warp waits or issues products (the issuer waits, bounded, for the
    // products it already issued); every warp still runs to the end, where
    // the copies are drained and the tensor memory freed.
    auto give_up = [&]() {
        *abort_flag = 1u;
        atomicOr(a.status, kStatusTensorTimeout);
    };

    if (issuer) {
        // warp 16: the products of every step, in order
        if (lane == 0) {
            int last = -1;  // the last step whose products were issued
            for (int u = 0; u < nitems && *abort_flag == 0u; ++u) {
                const uint32_t b = (uint32_t)(u & 1), par = (uint32_t)(u >> 1) & 1u;
                if (!mbar_wait_bounded(a_full + 8 * b, par) ||
                    (u >= 2 && !mbar_wait_bounded(d_empty + 8 * b, par ^ 1u))) {
                    give_up();
                    break;
                }
                tc_fence_after();
                const int c = tc_step_chunk(u % nb);
                const uint32_t a_t = tmem + b * 128u, d_t = tmem + 256u + b * 32u;
#pragma unroll
                for (int j = 0; j < 8; ++j) {  // sub-block j = 2gq + part: slices gq*4 + part*2 + {0, 1}
                    // sub-blocks 0..3 into the first accumulator, 4..7 into the second
                    const int s0 = (j >> 1) * 4 + (j & 1) * 2;
                    const uint32_t acc = d_t + 16u * (uint32_t)(j >> 2);
                    tc_mma_f16_ts(acc, a_t + 8 * s0, tc_act_desc(act_u32, c, s0), kTcIdesc, (j & 3) ? 1u : 0u);
                    tc_mma_f16_ts(acc, a_t + 8 * (s0 + 1), tc_act_desc(act_u32, c, s0 + 1), kTcIdesc, 1u);
                }
                tc_commit(d_full + 8 * b);
                last = u;
            }
            // after a give-up nobody may wait for the last products: wait for
            // them here (bounded) so the tensor memory is not freed under them
            if (last >= 0 && *abort_flag != 0u)
                (void)mbar_wait_bounded(d_full + 8 * (uint32_t)(last & 1), (uint32_t)(last >> 1) & 1u);
        }
        __syncwarp();
    } else if (decoder) {
        const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;  // this warp's 32 lanes
        // the step's stage: this thread's copies, then the quarter decoders'
        auto stage_ready = [&]() {
            cp_async_wait_pending(S - 2);
            decoder_barrier(quarter);
        };
        for (int g = 0; g < nitems; ++g) {
            stage_ready();  // step g landed; both decoders are past step g - 1
            // step g + S - 1 into the stage of step g - 1
            if (issued < nitems) issue_next();
            cp_async_commit();
            // A[g & 1] is free once the products of step g - 2 are done
            if (g >= 2 && !__any_sync(0xffffffffu, *abort_flag != 0u)) {
                const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(d_full + 8 * (uint32_t)(g & 1),
                                                                         (uint32_t)((g - 2) >> 1) & 1u));
                if (!ok && lane == 0) give_up();
            }
            const uint8_t *row_chunk = qstage0 + (g % S) * kTcQStageBytes + lane * kChunkBytes;
            const uint4 h = *reinterpret_cast<const uint4 *>(row_chunk);
            const uint32_t sc_lo = h.y & 0x3F3F3F3Fu;  // six-bit scales of sub-blocks 0..3, 4..7
            const uint32_t sc_hi = (h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u);
            const uint32_t a_cols = tmem + lane_base + (uint32_t)(g & 1) * 128u;
#pragma unroll
            for (int gg = 0; gg < 2; ++gg) {  // group gq: slices 4gq + h (low), 4gq + 2 + h (high)
                const int gq = 2 * half + gg;
                const uint4 u0 = *reinterpret_cast<const uint4 *>(row_chunk + 16 + 32 * gq);
                const uint4 u1 = *reinterpret_cast<const uint4 *>(row_chunk + 32 + 32 * gq);
                const uint32_t q[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
                const uint32_t scw = gq < 2 ? sc_lo : sc_hi;
#pragma unroll
                for (int part = 0; part < 2; ++part) {
                    // sub-block 2gq + part: (1024 + q) * sc - 1024 * sc, or for a
                    // high nibble (1024 + 16q) * sc/16 - 64 * sc: the exact f16
                    // q * sc (<= 945) by one fused multiply-add
                    const float sc = (float)byte_of(scw, 2 * (gq & 1) + part);
                    const __half2 mul = __float2half2_rn(part ? sc * 0.0625f : sc);
                    const __half2 add = __float2half2_rn(part ? -64.0f * sc : -1024.0f * sc);
                    const uint32_t mask = part ? 0x00F000F0u : 0x000F000Fu;
                    uint32_t f[16];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t b0 = (q[i] & mask) | 0x64006400u;
                        const uint32_t b1 = ((q[i] >> 8) & mask) | 0x64006400u;
                        const __half2 r0 = __hfma2(*reinterpret_cast<const __half2 *>(&b0), mul, add);
                        const __half2 r1 = __hfma2(*reinterpret_cast<const __half2 *>(&b1), mul, add);
                        f[2 * i] = *reinterpret_cast<const uint32_t *>(&r0);
                        f[2 * i + 1] = *reinterpret_cast<const uint32_t *>(&r1);
                    }
                    tc_st16(a_cols + 32u * gq + 16u * part, f);
                }
            }
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(a_full + 8 * (uint32_t)(g & 1));
        }
    } else {
        // epilogue warps (8-15): vectors 4half .. 4half + 3 of this warp's 32 rows
        const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
        float xh[4][4], xl[4][4];  // the binary counter of the pairing tree, four vectors
        // this row's 16-byte header of step g, from global memory
        auto header = [&](int g) -> uint4 {
            const int64_t tile = blockIdx.x + (int64_t)(g / nb) * gridDim.x;
            const int64_t row = tile * kTcRows + 32 * quarter + lane;
            if (g >= nitems || row >= rows) return make_uint4(0u, 0u, 0u, 0u);
            return __ldg(reinterpret_cast<const uint4 *>(a.W + row * kRowBytes +
                                                         tc_step_chunk(g % nb) * kChunkBytes));
        };
        uint4 h_next = header(0);
        int g = 0;
        for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
            const int64_t row = tile * kTcRows + 32 * quarter + lane;
#pragma unroll
            for (int s = 0; s < nb; ++s, ++g) {
                const uint4 h = h_next;
                h_next = header(g + 1);  // in flight during this step
                const uint32_t b = (uint32_t)(g & 1);
                bool ok = *abort_flag == 0u && mbar_wait_bounded(d_full + 8 * b, (uint32_t)(g >> 1) & 1u);
                ok = __all_sync(0xffffffffu, ok);  // warp-uniform: tcgen05.ld is warp-wide
                if (!ok && lane == 0) give_up();
                tc_fence_after();
                uint32_t dv[2][4];
                const uint32_t d_t = tmem + lane_base + 256u + b * 32u + 4u * half;
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    dv[k][0] = dv[k][1] = dv[k][2] = dv[k][3] = 0u;
                    if (ok) tc_ld4(d_t + 16 * k, dv[k]);
                }
                tc_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(d_empty + 8 * b);
                const int c = tc_step_chunk(s);
                const float d = f16_bits_to_f32(h.x);
                const float dmin = f16_bits_to_f32(h.x >> 16);
                const uint32_t m_lo = h.z & 0x3F3F3F3Fu;
                const uint32_t m_hi = ((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u);
#pragma unroll
                for (int vv = 0; vv < 4; ++vv) {
                    const int v = 4 * half + vv;
                    // S1 = sum of sc * dot over the eight sub-blocks: the two
                    // accumulators' exact integers
                    const int S1 = __float2int_rn(__uint_as_float(dv[0][vv])) +
                                   __float2int_rn(__uint_as_float(dv[1][vv]));
                    const uint4 sp = split_tab[c * 8 + v];
                    const int S2 = dp4a_uu(m_hi, sp.y, dp4a_uu(m_lo, sp.x, 0)) +
                                   256 * dp4a_us(m_hi, sp.w, dp4a_us(m_lo, sp.z, 0));
                    float th, tl;
                    q4k_epilogue(xs_tab[c * 8 + v], d, dmin, S1, S2, th, tl, true);
                    // the binary counter: level l pending after step s iff bit l of s is 0
#pragma unroll
                    for (int l = 0; l < 4; ++l) {
                        if (((s >> l) & 1) == 0) {
                            xh[l][vv] = th;
                            xl[l][vv] = tl;
                            break;
                        }
                        acc_add(th, tl, xh[l][vv], xl[l][vv]);
                    }
                    if (s == nb - 1 && v < B && row < rows && *abort_flag == 0u)  // all levels merged
                        a.y[(int64_t)v * rows + row] = __fadd_rn(th, tl);
                }
            }
        }
    }
    cp_async_wait_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"((uint32_t)kTcTmemCols)
                     : "memory");
    }
}

}  // namespace xq
