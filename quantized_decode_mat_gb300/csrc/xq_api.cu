// C ABI of the decode mat-vec library: argument checks, per-device set-up,
// launch planning, and the q8 activation quantiser.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "xq_internal.h"
#include "xq_ptx.cuh"
#include "xq_norm.cuh"
#include "xq_q8.cuh"

namespace xq {

// Device status word for kernel-side errors reported without trapping (bit 1:
// a grouped mat-vec met an expert id outside [0, n_experts)).
__device__ uint32_t g_status_word;

// ---- q8 activation quantiser ------------------------------------------------------
// One warp per 256-value block (the arithmetic is q8_quantize_lane, shared with
// the fused kernels); lane l holds values 8l..8l+7, so lanes 4s..4s+3 hold
// sub-block s.  Layout: values @0, int32 sums @256, f32 scale @288, zero
// bytes 292..319.
__global__ void __launch_bounds__(256) q8_quantize_kernel(const float *__restrict__ x,
                                                          uint8_t *__restrict__ xq,
                                                          int64_t nblocks) {
    grid_dependency_wait();  // x may come from the kernel before on the stream
    grid_dependency_trigger();
    const int64_t blk = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (blk >= nblocks) return;  // whole warps leave together
    const float4 *src = reinterpret_cast<const float4 *>(x + blk * 256 + lane * 8);
    const float4 u = __ldg(src), v = __ldg(src + 1);
    const float vals[8] = {u.x, u.y, u.z, u.w, v.x, v.y, v.z, v.w};
    const Q8Lane r = q8_quantize_lane(vals);
    uint8_t *out = xq + blk * kQ8Bytes;
    *reinterpret_cast<uint2 *>(out + lane * 8) = make_uint2(r.w0, r.w1);
    if ((lane & 3) == 0) *reinterpret_cast<int *>(out + kQ8SumAt + (lane >> 2) * 4) = r.sum;
    if (lane == 0)
        *reinterpret_cast<float *>(out + kQ8ScaleAt) = r.d;
    else if (lane < 8)
        *reinterpret_cast<uint32_t *>(out + kQ8ScaleAt + 4 * lane) = 0u;  // bytes 292..319
}

// ---- RMSNorm + q8 pack -------------------------------------------------------------
// Grid (ceil(nb/8), batch), 256 threads: block (c, b) owns q8 blocks 8c ..
// 8c+7 of vector b, one per warp.  Each warp loads its block's values, the
// block's 256 threads take the scale in the fixed order (rms_scale_block,
// the workgroup itself; every CTA of the vector gets the same bits), then
// each warp writes y = x * scale (when y is non-null) and its q8 block via
// q8_quantize_lane.
__global__ void __launch_bounds__(256) rmsnorm_q8_kernel(const float *__restrict__ x,
                                                         uint8_t *__restrict__ xq,
                                                         float *__restrict__ y, int64_t cols) {
    __shared__ float s_wave[8];
    grid_dependency_wait();  // x may come from the kernel before on the stream
    grid_dependency_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nb = cols / 256;
    const int64_t k = (int64_t)blockIdx.x * 8 + warp;  // this warp's q8 block
    const float *xv = x + (int64_t)blockIdx.y * cols;
    float4 u = make_float4(0.f, 0.f, 0.f, 0.f), v = u;
    if (k < nb) {
        const float4 *src = reinterpret_cast<const float4 *>(xv + k * 256 + lane * 8);
        u = __ldg(src);
        v = __ldg(src + 1);
    }
    const float scale = rms_scale_block(xv, cols, s_wave);
    if (k >= nb) return;  // whole warps
    float vals[8] = {u.x, u.y, u.z, u.w, v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) vals[i] = __fmul_rn(vals[i], scale);
    if (y) {
        float4 *dy = reinterpret_cast<float4 *>(y + (int64_t)blockIdx.y * cols + k * 256 + lane * 8);
        dy[0] = make_float4(vals[0], vals[1], vals[2], vals[3]);
        dy[1] = make_float4(vals[4], vals[5], vals[6], vals[7]);
    }
    const Q8Lane r = q8_quantize_lane(vals);
    uint8_t *out = xq + ((int64_t)blockIdx.y * nb + k) * kQ8Bytes;
    *reinterpret_cast<uint2 *>(out + lane * 8) = make_uint2(r.w0, r.w1);
    if ((lane & 3) == 0) *reinterpret_cast<int *>(out + kQ8SumAt + (lane >> 2) * 4) = r.sum;
    if (lane == 0)
        *reinterpret_cast<float *>(out + kQ8ScaleAt) = r.d;
    else if (lane < 8)
        *reinterpret_cast<uint32_t *>(out + kQ8ScaleAt + 4 * lane) = 0u;  // bytes 292..319
}

// ---- resident repack of codebook blocks ---------------------------------------------
// CTA t (256 threads) takes blocks 256t .. 256t+255 of the chunk.  The tile's
// raw bytes are read with coalesced loads into shared memory (16-byte loads
// when the source is 16-byte aligned, byte loads otherwise); then thread i
// writes block i's f16 scale into its row's prefix and its 16 payload bytes
// as one 16-byte store into the row's payload run, so consecutive threads
// store consecutive bytes of a row.  The scale and payload of a block move in
// the same pass ("25 - Writing XPU Kernels" 25.4: a separate pass over the
// scales pulls a line per block for two useful bytes).
__global__ void __launch_bounds__(256) repack_cb4_kernel(const uint8_t *__restrict__ src,
                                                         uint8_t *__restrict__ Wr,
                                                         int64_t block_base, int64_t n_blocks,
                                                         int64_t bpr, int64_t prefix,
                                                         int64_t row_bytes, int src_vec16) {
    __shared__ __align__(16) uint8_t tile[256 * kCb4Bytes];
    const int64_t b0 = (int64_t)blockIdx.x * 256;
    const int64_t left = n_blocks - b0;
    const int nblk = left < 256 ? (int)left : 256;
    const int nbytes = nblk * kCb4Bytes;
    const uint8_t *s = src + b0 * kCb4Bytes;
    int done = 0;
    if (src_vec16) {  // s is 16-byte aligned: 4608 * blockIdx.x is a multiple of 16
        const int n16 = nbytes >> 4;
        for (int i = threadIdx.x; i < n16; i += 256)
            reinterpret_cast<uint4 *>(tile)[i] = __ldg(reinterpret_cast<const uint4 *>(s) + i);
        done = n16 << 4;
    }
    for (int i = done + threadIdx.x; i < nbytes; i += 256) tile[i] = __ldg(s + i);
    __syncthreads();
    const int t = threadIdx.x;
    if (t >= nblk) return;
    const int64_t g = block_base + b0 + t;
    const int64_t row = g / bpr, j = g - row * bpr;
    uint8_t *rp = Wr + row * row_bytes;
    const uint16_t *h = reinterpret_cast<const uint16_t *>(tile + t * kCb4Bytes);  // even offset
    reinterpret_cast<uint16_t *>(rp)[j] = h[0];
    uint4 p;
    p.x = (uint32_t)h[1] | ((uint32_t)h[2] << 16);
    p.y = (uint32_t)h[3] | ((uint32_t)h[4] << 16);
    p.z = (uint32_t)h[5] | ((uint32_t)h[6] << 16);
    p.w = (uint32_t)h[7] | ((uint32_t)h[8] << 16);
    *reinterpret_cast<uint4 *>(rp + prefix + 16 * j) = p;
}

namespace {

thread_local std::string t_error;
thread_local xq_plan t_last_plan;
thread_local bool t_have_plan = false;
std::atomic<uint64_t> g_counts[XQ_COUNT_N];
std::atomic<int32_t> g_override_warps{0};
std::atomic<int32_t> g_override_stages{0};
std::atomic<int32_t> g_override_row_block{0};
std::atomic<int32_t> g_override_quantise_once{0};
std::atomic<int32_t> g_override_vector_pairs{0};
std::atomic<int32_t> g_override_tensor{0};
std::atomic<int32_t> g_overlap{0};
// The decode step with a workspace quantises the activation once, in a
// launch of its own, when a launch's batch has at least this many q8 blocks;
// below that every CTA of the one fused launch quantises it for itself.
// Measured on GB300 over Q4_K and codebook rows of 4096 and 14336 and 2048 to
// 14336 columns at batch 1 to 8: up to 32 blocks the fused launch was faster
// in 21 of 24 shapes (by up to a third; the others by at most 2.4 %), from 48
// blocks the launch of its own in most.
constexpr int64_t kQuantOnceMinBlocks = 33;
// Whether the planner picks warp pairs by itself (the override can force
// them either way).
constexpr bool kVectorPairsAuto = true;
constexpr int64_t kVpMinUnits = 16;
// Whether the planner picks the tensor-core kernel by itself.
constexpr bool kTensorAuto = false;

xq_status fail(xq_status s, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
xq_status fail(xq_status s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_error = buf;
    return s;
}

xq_status cuda_fail(cudaError_t e, const char *what) {
    return fail(XQ_ELAUNCH, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool overlap(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return na && nb && a0 < b0 + nb && b0 < a0 + na;
}

xq_status check_shape(int64_t rows, int64_t cols, int64_t batch, bool need_rows) {
    if (cols <= 0 || cols % 256 != 0)
        return fail(XQ_ESHAPE, "cols=%lld must be a positive multiple of 256", (long long)cols);
    if (cols > (int64_t)1 << 24)
        return fail(XQ_ESHAPE, "cols=%lld exceeds 2^24", (long long)cols);
    if (batch < 1 || batch > 8)
        return fail(XQ_ESHAPE, "batch=%lld must be in 1..8", (long long)batch);
    if (need_rows && (rows < 1 || rows > 0x7FFFFFFFLL))
        return fail(XQ_ESHAPE, "rows=%lld must be in 1..2^31-1", (long long)rows);
    return XQ_OK;
}

struct DeviceState {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    const char *what = "";
    int sm_count = 0;
    int smem_optin = 0;
    uint32_t *status = nullptr;
};
constexpr int kMaxDevices = 64;
DeviceState g_dev[kMaxDevices];

// Per-device set-up on the first call with that device current: device
// attributes, the status word's device address, and the kernels' dynamic
// shared memory limit.
xq_status device_state(DeviceState **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(XQ_ELAUNCH, "device %d out of range", dev);
    DeviceState &st = g_dev[dev];
    std::call_once(st.once, [&st, dev]() {
        auto step = [&st](cudaError_t r, const char *what) {
            if (st.err == cudaSuccess && r != cudaSuccess) {
                st.err = r;
                st.what = what;
            }
        };
        step(cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev),
             "cudaDeviceGetAttribute(MultiProcessorCount)");
        step(cudaDeviceGetAttribute(&st.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev),
             "cudaDeviceGetAttribute(MaxSharedMemoryPerBlockOptin)");
        void *p = nullptr;
        step(cudaGetSymbolAddress(&p, g_status_word), "cudaGetSymbolAddress(status word)");
        st.status = static_cast<uint32_t *>(p);
        if (st.err == cudaSuccess) step(configure_matvec_q4k(st.smem_optin), "configure Q4_K kernels");
        if (st.err == cudaSuccess) step(configure_matvec_cb4(st.smem_optin), "configure codebook kernels");
        if (st.err == cudaSuccess)
            step(configure_matvec_cb4r(st.smem_optin), "configure resident codebook kernels");
        if (st.err == cudaSuccess)
            step(configure_matvec_q4k_tc(st.smem_optin), "configure tensor-core Q4_K kernels");

    });
    if (st.err != cudaSuccess) return cuda_fail(st.err, st.what);
    *out = &st;
    return XQ_OK;
}

int64_t align128(int64_t v) { return (v + 127) & ~(int64_t)127; }

// Row groups: 32/nb rows (one contiguous 4608-byte box) when nb is a power
// of two below 32, else one row streamed in ceil(nb/32) boxes.  A warp's work
// unit is row_block consecutive row groups (see the kernel).  The batch's q8
// blocks are staged in shared memory; when they do not fit beside two stages,
// the batch is split across launches (each re-reads W).  Grid: one CTA per
// SM, at most one per work unit.  Warps: enough to cover the work units,
// within the instantiation's register budget.  Stages: 2 (measured best),
// fewer warps if even that does not fit.  slots > 0 plans the grouped-expert
// form: `rows` rows per expert, `slots` selected experts, each group inside
// one slot, and `batch` staged activation vectors (1 shared, or one per slot).
// fused: the launch is the fused decode step (xq_linear_*), whose kernel
// quantises x itself unless the plan quantises once into a workspace.
xq_status make_plan(int fmt, int64_t rows, int64_t cols, int64_t batch, int32_t sm_count,
                    int64_t smem_optin, xq_plan *p, int64_t slots = 0, bool have_ws = false,
                    int fuse = 0, bool dots = false, bool fused = false) {
    const int32_t nb = (int32_t)(cols / 256);
    const int32_t R = (nb < 32 && 32 % nb == 0) ? 32 / nb : 1;
    const int32_t spr = R > 1 ? 1 : (nb + 31) / 32;
    const int64_t groups = slots > 0 ? slots * ((rows + R - 1) / R) : (rows + R - 1) / R;
    int32_t bl = (int32_t)batch;
    while (bl > 0 && align128((int64_t)bl * nb * kActStride) + 2LL * kStageBytes + 128 > smem_optin)
        --bl;
    if (bl < 1)
        return fail(XQ_ESHAPE, "cols=%lld: one q8 vector does not fit in shared memory",
                    (long long)cols);
    const int64_t act = align128((int64_t)bl * nb * kActStride);
    if (slots > 0 && bl != batch)
        return fail(XQ_ESHAPE, "the per-slot activations do not fit in shared memory");
    const int32_t wmax = warps_limit(fmt, slots > 0 ? 1 : bl, fuse, dots);
    const int32_t ow = g_override_warps.load(), os = g_override_stages.load();
    const int32_t om = g_override_row_block.load();
    // Two stages (one box in flight per warp while the other is consumed) read
    // fastest on GB300: the warps of the GPU then stream one contiguous window.
    const int32_t S0 = os > 0 ? (os > kMaxStages ? kMaxStages : os) : 2;
    // Row groups per warp unit: two for Q4_K with two or more vectors.  When
    // the instantiation's full warp count of two-box stages does not fit in
    // shared memory beside the activations, a single stage a warp (the warps
    // overlap one another's copies) measured faster than fewer warps or one
    // row group (4096 x 14336 at batch 8: 23.5 against 26.5 us); if even that
    // does not fit, one row group.
    int32_t M = (fmt == kQ4K && bl >= 2 && slots == 0) ? 2 : 1;
    if (om > 0) M = (om >= 2 && M == 2) ? 2 : 1;
    auto bytes = [&](int32_t w, int32_t st, int32_t m) {
        return act + (int64_t)w * st * m * kStageBytes + 128;
    };
    if (M == 2 && om <= 0 && bytes(wmax, 1, 2) > smem_optin) M = 1;
    const int32_t Smin = M == 2 ? 1 : 2;  // the fewest stages the planner lowers to
    const int64_t units = (groups + M - 1) / M;
    const int32_t grid = (int32_t)(units < sm_count ? units : sm_count);
    const int64_t per_cta = (units + grid - 1) / grid;
    const int32_t oq = g_override_quantise_once.load();
    const bool qonce = have_ws && (oq == 2 || (oq == 0 && (int64_t)bl * nb >= kQuantOnceMinBlocks));
    // Batch 1: 16 warps, the fastest for Q4_K boxes of whole rows (20: 46.1
    // against 44.6 us on 128256 x 4096) and for the fused RMSNorm form; 20 for
    // the mat-vec behind a quantise launch (4096 x 14336 step: 8.23 against
    // 9.15 us) and for the codebook (11008 x 4096 step: 7.42 against 7.63 us,
    // resident rows 8.88 against 9.08 us)
    const bool wide1 = slots == 0 && (qonce || fmt != kQ4K);
    const int32_t wpref = bl == 1 && !wide1 && wmax > 16 ? 16 : wmax;
    int32_t W = (int32_t)(per_cta < wpref ? per_cta : wpref);
    if (ow > 0) W = ow < wmax ? ow : wmax;
    // above 8 warps, whole warps a scheduler (12, 16, 20) with two stages each;
    // where those do not fit, the next such count down
    if (ow <= 0)
        while (W > kMaxWarps && bytes(W, S0, M) > smem_optin) W = (W - 1) / 4 * 4;
    int32_t S = S0;
    while (bytes(W, S, M) > smem_optin) {
        if (S > Smin)
            --S;
        else if (W > 1)
            --W;
        else
            break;
    }
    if (bytes(W, S, M) > smem_optin)
        return fail(XQ_ESHAPE, "plan needs %lld bytes of shared memory, device allows %lld",
                    (long long)bytes(W, S, M), (long long)smem_optin);
    const int64_t tw = (int64_t)grid * W;
    if (((units + tw - 1) / tw) * spr > 0x7FFFFFFFLL)
        return fail(XQ_ESHAPE, "too many boxes per warp");
    p->warps = W;
    p->stages = S;
    p->grid = grid;
    p->rows_per_group = R;
    p->segments = spr;
    p->chunks_per_row = nb;
    p->groups = groups;
    p->batch_per_launch = bl;
    p->launches = (int32_t)((batch + bl - 1) / bl);
    p->smem_bytes = bytes(W, S, M);
    p->row_block = M;
    p->quantise_once = qonce;
    p->vector_pairs = 0;
    p->tensor = 0;
    // Warp pairs: the row-blocked mat-vec on q8 blocks (the plain mat-vec, or
    // the decode step when it quantises once) for rows of 16 chunks at 8
    // vectors, on matrices that give every pair at least kVpMinUnits units,
    // when no warp or stage override is set: 16 warps (eight pairs, four warps
    // a scheduler) share two stages of two boxes a pair (128256 x 4096: 106.3
    // against 99.1 us, 99.8 with 12 warps; slower on 14336 x 4096, 15.7
    // against 18.0 us, and at 6 vectors, 79.6 against 86.2 us with 12 warps).
    // Only those kernels have a warp-pair build.  Forced on (override 2), the
    // warp and stage overrides size it.
    const int32_t ovp = g_override_vector_pairs.load();
    const bool q8_input = fuse == 0 && !dots && (!fused || qonce);
    if (fmt == kQ4K && M == 2 && nb == 16 && bl == 8 && slots == 0 && q8_input && ovp != 1) {
        int32_t vw = kVpWarps, vs = kVpStages;
        if (ovp == 2 && ow > 0) vw = ow & ~1;
        if (ovp == 2 && os > 0) vs = os;
        const bool want = ovp == 2 || (kVectorPairsAuto && ow <= 0 && os <= 0 &&
                                       units >= (int64_t)kVpMinUnits * grid * (vw / 2));
        const int64_t vp_bytes = act + (int64_t)(vw / 2) * vs * M * kStageBytes +
                                 (int64_t)vw * kVpScratchBytes + 128;
        if (want && vw >= 2 && vw <= kVpWarps && vs >= 2 && vs <= kMaxStages &&
            vp_bytes <= smem_optin) {
            p->warps = vw;
            p->stages = vs;
            p->smem_bytes = vp_bytes;
            p->vector_pairs = 1;
        }
    }
    // The tensor-core kernel: the Q4_K mat-vec on q8 blocks for rows of 16
    // chunks at 5..8 vectors; one CTA of seventeen warps an SM on tiles of 128
    // rows (it holds all 512 columns of tensor memory), three stages.  Forced
    // on (override 2), a stage override (two or more) sizes it.
    const int32_t otc = g_override_tensor.load();
    if (fmt == kQ4K && nb == kTcChunks && bl >= 5 && bl <= 8 && slots == 0 && q8_input &&
        otc != 1 && (otc == 2 || (kTensorAuto && ow <= 0 && os <= 0))) {
        const int32_t ts = otc == 2 && os >= 2 ? os : kTcStages;
        const int64_t tiles = (rows + kTcRows - 1) / kTcRows;
        const int64_t t_bytes = tc_smem_bytes(ts);
        if (ts <= kMaxStages && t_bytes <= smem_optin) {
            p->warps = kTcThreads / 32;
            p->stages = ts;
            p->grid = (int32_t)(tiles < sm_count ? tiles : sm_count);
            p->rows_per_group = kTcRows;
            p->segments = kTcChunks;
            p->groups = tiles;
            p->row_block = 1;
            p->smem_bytes = t_bytes;
            p->vector_pairs = 0;
            p->tensor = 1;
        }
    }
    return XQ_OK;
}

// When every CTA quantises the activation itself, its warps share that work
// one q8 block each; a plan with fewer warps than blocks (few rows a CTA) gets
// more warps, which find no row group of their own and only quantise.
void widen_for_quantise(xq_plan *p, int fmt, int fuse, int64_t nb, int64_t smem_optin) {
    const int64_t nblk = (int64_t)p->batch_per_launch * nb;
    const int32_t wmax = warps_limit(fmt, p->batch_per_launch, fuse);
    int32_t W = p->warps;
    const int64_t want = nblk < wmax ? nblk : wmax;
    if (W >= want) return;
    const int64_t act = align128((int64_t)p->batch_per_launch * nb * kActStride);
    const int64_t per_warp = (int64_t)p->stages * p->row_block * kStageBytes;
    while (W < want && act + (int64_t)(W + 1) * per_warp + 128 <= smem_optin) ++W;
    p->warps = W;
    p->smem_bytes = act + (int64_t)W * per_warp + 128;
}

enum class Kind { kMatvec, kDots, kLinear, kNormLinear };

struct OpInfo {
    int fmt;    // kQ4K, kCB4 or kCB4R
    Kind kind;
    int count;  // launch counter
};

cudaError_t launch_fmt(int fmt, const MatvecArgs &a, int batch, int kind, dim3 grid, dim3 block,
                       size_t smem, cudaStream_t s) {
    return fmt == kQ4K   ? launch_matvec_q4k(a, batch, kind, grid, block, smem, s)
           : fmt == kCB4 ? launch_matvec_cb4(a, batch, kind, grid, block, smem, s)
                         : launch_matvec_cb4r(a, batch, kind, grid, block, smem, s);
}

void pack_table(const int8_t *table, uint32_t (&kv)[4]) {
    for (int i = 0; i < 4; ++i) {
        uint32_t w = 0;
        for (int j = 0; j < 4; ++j) w |= (uint32_t)(uint8_t)table[4 * i + j] << (8 * j);
        kv[i] = w;
    }
}

// The two lookup tables of the one-vector codebook dot (cb4_dot_split): bytes
// L[0..7] in kv[0..1] and H[0..7] in kv[2..3] with, for i = 0..7,
//   kv[i]     = L[i] + rep(H[i])      (rep: 0 for a byte >= 0, -1 below 0)
//   kv[i + 8] = rep(L[i]) + H[i]
// since prmt returns byte n of a table for an index n < 8 and rep of byte
// n - 8 for n >= 8.  Per i the signs s = rep(H[i]), t = rep(L[i]) must agree
// with the bytes they produce; one of the two choices of s works unless an
// entry is 127 where its partner needs one more (then false: the select
// decode is used).
bool split_table(const int8_t *table, uint32_t (&kv)[4]) {
    uint8_t L[8], H[8];
    for (int i = 0; i < 8; ++i) {
        bool found = false;
        for (int s = 0; s <= 1 && !found; ++s) {  // s = 1: H[i] < 0, so rep(H[i]) = -1
            const int l = table[i] + s;
            const int t = l < 0 ? 1 : 0;
            const int h = table[i + 8] + t;
            if (l > 127 || h > 127 || h < -128 || (h < 0 ? 1 : 0) != s) continue;
            L[i] = (uint8_t)(int8_t)l;
            H[i] = (uint8_t)(int8_t)h;
            found = true;
        }
        if (!found) return false;
    }
    for (int w = 0; w < 2; ++w) {
        kv[w] = kv[w + 2] = 0;
        for (int j = 0; j < 4; ++j) {
            kv[w] |= (uint32_t)L[4 * w + j] << (8 * j);
            kv[w + 2] |= (uint32_t)H[4 * w + j] << (8 * j);
        }
    }
    return true;
}

// in: q8 blocks (mat-vec and sub-dots) or f32 x (the fused linear ops).
// ws (the fused linear ops only): a workspace of linear_ws_bytes(cols,
// batch) bytes for the quantise-once form (the q8 blocks), or null.
size_t linear_ws_bytes(int64_t cols, int64_t batch) {
    return (size_t)batch * (cols / 256) * kQ8Bytes;
}

xq_status run_matvec(OpInfo op, const void *W, const int8_t *table, const void *in, void *out,
                     int64_t rows, int64_t cols, int64_t batch, void *stream,
                     void *ws = nullptr, size_t ws_bytes = 0, bool want_ws = false) {
    const bool cb4 = op.fmt != kQ4K;
    const bool dots = op.kind == Kind::kDots;
    const bool norm = op.kind == Kind::kNormLinear;
    const bool fused = norm || op.kind == Kind::kLinear;
    t_error.clear();
    if (!W || !in || !out)
        return fail(XQ_EINVAL, fused ? "null device pointer (x, W or y)"
                                     : "null device pointer (W, xq or output)");
    if (cb4 && !table) return fail(XQ_EINVAL, "null codebook table");
    if (xq_status s = check_shape(rows, cols, batch, true)) return s;
    if (!aligned(W, 16)) return fail(XQ_EALIGN, "W must be 16-byte aligned");
    if (!aligned(in, 16)) return fail(XQ_EALIGN, fused ? "x must be 16-byte aligned"
                                                         : "xq must be 16-byte aligned");
    if (!aligned(out, dots ? 16 : 4))
        return fail(XQ_EALIGN, dots ? "dots must be 16-byte aligned" : "y must be 4-byte aligned");
    const int64_t nb = cols / 256;
    const size_t w_bytes = (size_t)rows * nb * kChunkBytes;
    const size_t in_bytes = fused ? (size_t)batch * cols * 4 : (size_t)batch * nb * kQ8Bytes;
    const size_t o_bytes = (size_t)batch * rows * (dots ? nb * 8 * 4 : 4);
    if (overlap(out, o_bytes, W, w_bytes) || overlap(out, o_bytes, in, in_bytes))
        return fail(XQ_EINVAL, "output overlaps an input");
    if (want_ws) {
        const size_t need = linear_ws_bytes(cols, batch);
        if (!ws) return fail(XQ_EINVAL, "null workspace");
        if (!aligned(ws, 16)) return fail(XQ_EALIGN, "workspace must be 16-byte aligned");
        if (ws_bytes < need)
            return fail(XQ_EINVAL, "workspace of %zu bytes is too small: %zu needed", ws_bytes, need);
        if (overlap(ws, need, W, w_bytes) || overlap(ws, need, in, in_bytes) ||
            overlap(ws, need, out, o_bytes))
            return fail(XQ_EINVAL, "workspace overlaps x, W or y");
    }

    DeviceState *dev = nullptr;
    if (xq_status s = device_state(&dev)) return s;
    xq_plan plan;
    if (xq_status s = make_plan(op.fmt, rows, cols, batch, dev->sm_count, dev->smem_optin, &plan,
                                0, want_ws && op.kind == Kind::kLinear, norm ? 2 : 0, dots, fused))
        return s;
    MatvecArgs a;
    memset(&a, 0, sizeof a);
    a.W = static_cast<const uint8_t *>(W);
    a.rows = rows;
    a.groups = plan.groups;
    a.nb = (int32_t)nb;
    a.rows_per_group = plan.rows_per_group;
    a.segments = plan.segments;
    a.stages = plan.stages;
    a.row_block = plan.row_block;
    a.vector_pairs = plan.vector_pairs;
    a.tensor = plan.tensor;
    a.status = dev->status;
    a.overlap = g_overlap.load();
    if (cb4) {
        a.kv_split = plan.batch_per_launch == 1 && split_table(table, a.kv);
        if (!a.kv_split) pack_table(table, a.kv);
    }
    // quantise once: q8 blocks into the workspace, then the mat-vec on them
    const bool once = plan.quantise_once != 0;
    if (fused && !once && g_override_warps.load() == 0)  // an override is kept as given
        widen_for_quantise(&plan, op.fmt, norm ? 2 : 1, nb, dev->smem_optin);
    const dim3 grid(plan.grid), block(plan.warps * 32);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int kind = dots ? 1 : norm ? 4 : (fused && !once) ? 2 : 0;
    // only the row-blocked Q4_K mat-vec on q8 blocks has a warp-pair build
    if (plan.vector_pairs && !(kind == 0 && op.fmt == kQ4K && plan.row_block == 2 && nb == 16 &&
                               plan.launches == 1 && plan.warps % 2 == 0 &&
                               plan.warps <= kVpWarps && plan.stages >= 2 &&
                               plan.batch_per_launch == 8))
        return fail(XQ_ELAUNCH, "internal: a warp-pair plan for a kernel without that build");
    if (plan.tensor && !(kind == 0 && op.fmt == kQ4K && nb == kTcChunks && plan.launches == 1 &&
                         plan.batch_per_launch >= 5 && plan.batch_per_launch <= 8 &&
                         plan.warps * 32 == kTcThreads && plan.stages >= 2 &&
                         plan.smem_bytes == tc_smem_bytes(plan.stages)))
        return fail(XQ_ELAUNCH, "internal: a tensor-core plan for a kernel without that build");
    for (int64_t b0 = 0; b0 < batch; b0 += plan.batch_per_launch) {
        const int64_t bc = batch - b0 < plan.batch_per_launch ? batch - b0 : plan.batch_per_launch;
        if (once) {
            const int64_t nblk = bc * nb;
            const cudaError_t e = launch_kernel(
                q8_quantize_kernel, dim3((unsigned)((nblk + 7) / 8)), dim3(256), 0, s, a.overlap != 0,
                static_cast<const float *>(in) + b0 * cols, static_cast<uint8_t *>(ws), nblk);
            if (e != cudaSuccess) return cuda_fail(e, "quantise launch");
            a.xq = static_cast<const uint8_t *>(ws);
        } else if (fused) {
            a.x = static_cast<const float *>(in) + b0 * cols;
        } else {
            a.xq = static_cast<const uint8_t *>(in) + b0 * nb * kQ8Bytes;
        }
        a.y = dots ? nullptr : static_cast<float *>(out) + b0 * rows;
        a.dots = dots ? static_cast<int32_t *>(out) + b0 * rows * nb * 8 : nullptr;
        cudaError_t e = plan.tensor ? launch_matvec_q4k_tc(a, (int)bc, grid, block,
                                                          (size_t)plan.smem_bytes, s)
                                    : launch_fmt(op.fmt, a, (int)bc, kind, grid, block,
                                                 (size_t)plan.smem_bytes, s);
        if (e != cudaSuccess) return cuda_fail(e, "mat-vec launch");
        g_counts[op.count].fetch_add(1, std::memory_order_relaxed);
        if (once) g_counts[XQ_COUNT_QUANTISE_ONCE].fetch_add(1, std::memory_order_relaxed);
    }
    t_last_plan = plan;
    t_have_plan = true;
    return XQ_OK;
}

xq_status run_matvec_id(int fmt, const void *W, const int8_t *table, const int32_t *sel,
                        const void *xq_in, float *y, int64_t rpe, int64_t cols,
                        int64_t n_experts, int64_t used, int32_t x_per_slot, void *stream) {
    const bool cb4 = fmt != kQ4K;
    t_error.clear();
    if (!W || !sel || !xq_in || !y) return fail(XQ_EINVAL, "null device pointer (W, sel, xq or y)");
    if (cb4 && !table) return fail(XQ_EINVAL, "null codebook table");
    if (xq_status s = check_shape(rpe, cols, 1, true)) return s;
    if (n_experts < 1 || n_experts > 0x7FFFFFFFLL || rpe * n_experts > 0x7FFFFFFFLL)
        return fail(XQ_ESHAPE, "n_experts=%lld out of range", (long long)n_experts);
    if (used < 1 || used > (1 << 20)) return fail(XQ_ESHAPE, "used=%lld out of range", (long long)used);
    if (x_per_slot && used > 8) return fail(XQ_ESHAPE, "per-slot activations: used must be <= 8");
    if (!aligned(W, 16)) return fail(XQ_EALIGN, "W must be 16-byte aligned");
    if (!aligned(xq_in, 16)) return fail(XQ_EALIGN, "xq must be 16-byte aligned");
    if (!aligned(sel, 4)) return fail(XQ_EALIGN, "sel must be 4-byte aligned");
    if (!aligned(y, 4)) return fail(XQ_EALIGN, "y must be 4-byte aligned");
    const int64_t nb = cols / 256;
    const int64_t nvec = x_per_slot ? used : 1;
    const size_t o_bytes = (size_t)used * rpe * 4;
    if (overlap(y, o_bytes, W, (size_t)n_experts * rpe * nb * kChunkBytes) ||
        overlap(y, o_bytes, xq_in, (size_t)nvec * nb * kQ8Bytes) ||
        overlap(y, o_bytes, sel, (size_t)used * 4))
        return fail(XQ_EINVAL, "output overlaps an input");
    DeviceState *dev = nullptr;
    if (xq_status s = device_state(&dev)) return s;
    xq_plan plan;
    if (xq_status s = make_plan(fmt, rpe, cols, nvec, dev->sm_count, dev->smem_optin, &plan, used))
        return s;
    MatvecArgs a;
    memset(&a, 0, sizeof a);
    a.W = static_cast<const uint8_t *>(W);
    a.xq = static_cast<const uint8_t *>(xq_in);
    a.y = y;
    a.rows = used * rpe;
    a.groups = plan.groups;
    a.nb = (int32_t)nb;
    a.rows_per_group = plan.rows_per_group;
    a.segments = plan.segments;
    a.stages = plan.stages;
    a.row_block = plan.row_block;
    a.overlap = g_overlap.load();
    a.sel = sel;
    a.rows_per_expert = rpe;
    a.n_experts = (int32_t)n_experts;
    a.groups_per_slot = (int32_t)(plan.groups / used);
    a.act_vectors = (int32_t)nvec;
    a.status = dev->status;
    if (cb4) {  // one vector a slot
        a.kv_split = split_table(table, a.kv);
        if (!a.kv_split) pack_table(table, a.kv);
    }
    const dim3 grid(plan.grid), block(plan.warps * 32);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_fmt(fmt, a, 1, 3, grid, block, (size_t)plan.smem_bytes, s);
    if (e != cudaSuccess) return cuda_fail(e, "grouped mat-vec launch");
    const int which = fmt == kQ4K   ? XQ_COUNT_MATVEC_ID_Q4K
                      : fmt == kCB4 ? XQ_COUNT_MATVEC_ID_CB4
                                    : XQ_COUNT_MATVEC_ID_CB4R;
    g_counts[which].fetch_add(1, std::memory_order_relaxed);
    t_last_plan = plan;
    t_have_plan = true;
    return XQ_OK;
}

// ---- fixed scratch for callers that cannot allocate ---------------------------------------
// Scratch of xq_linear_q4k_static: the q8 blocks of the activation, when the
// plan quantises it once.  A file-scope device array: every GPU that loads the
// library holds it until the process exits.  Host code may use its name only
// to look up its device address (cudaGetSymbolAddress), never as a pointer.
constexpr size_t kStaticScratchBytes = 256 * 1024;

// The scratch's device address per device, kept once a lookup has succeeded;
// a failed lookup is not kept, so the next call tries again.
std::mutex g_static_scratch_mutex;
void *g_static_scratch_ptr[kMaxDevices];

}  // namespace
}  // namespace xq

static __device__ __align__(256) uint8_t g_static_scratch[xq::kStaticScratchBytes];

namespace xq {
namespace {

// Device address of g_static_scratch on the current device, looked up on the
// first call with that device current that gets this far (that call should
// come before any stream capture) and kept from then on.
xq_status static_scratch(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(XQ_ELAUNCH, "device %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_static_scratch_mutex);
    if (!g_static_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
        g_static_scratch_ptr[dev] = p;
    }
    *out = g_static_scratch_ptr[dev];
    return XQ_OK;
}

}  // namespace
}  // namespace xq

using namespace xq;

extern "C" {

size_t xq_q8_bytes(int64_t cols, int64_t batch) {
    if (cols <= 0 || cols % 256 || batch < 1) return 0;
    return (size_t)batch * (size_t)(cols / 256) * kQ8Bytes;
}

size_t xq_q4k_bytes(int64_t rows, int64_t cols) {
    if (cols <= 0 || cols % 256 || rows < 0) return 0;
    return (size_t)rows * (size_t)(cols / 256) * kQ4kBytes;
}

size_t xq_cb4_bytes(int64_t rows, int64_t cols) {
    if (cols <= 0 || cols % 256 || rows < 0) return 0;
    return (size_t)rows * (size_t)(cols / 32) * kCb4Bytes;
}

xq_status xq_quantize_q8(const float *x, void *xq_out, int64_t cols, int64_t batch, void *stream) {
    t_error.clear();
    if (!x || !xq_out) return fail(XQ_EINVAL, "null device pointer (x or xq)");
    if (xq_status s = check_shape(0, cols, batch, false)) return s;
    if (!aligned(x, 16)) return fail(XQ_EALIGN, "x must be 16-byte aligned");
    if (!aligned(xq_out, 16)) return fail(XQ_EALIGN, "xq must be 16-byte aligned");
    const int64_t nblocks = batch * (cols / 256);
    if (overlap(xq_out, (size_t)nblocks * kQ8Bytes, x, (size_t)batch * cols * 4))
        return fail(XQ_EINVAL, "xq overlaps x");
    DeviceState *dev = nullptr;
    if (xq_status s = device_state(&dev)) return s;
    const unsigned grid = (unsigned)((nblocks + 7) / 8);
    const cudaError_t e =
        launch_kernel(q8_quantize_kernel, dim3(grid), dim3(256), 0, static_cast<cudaStream_t>(stream),
                      g_overlap.load() != 0, x, static_cast<uint8_t *>(xq_out), nblocks);
    if (e != cudaSuccess) return cuda_fail(e, "quantise launch");
    g_counts[XQ_COUNT_QUANTIZE].fetch_add(1, std::memory_order_relaxed);
    return XQ_OK;
}

xq_status xq_rmsnorm_q8(const float *x, void *xq_out, float *y, int64_t cols, int64_t batch,
                        void *stream) {
    t_error.clear();
    if (!x || !xq_out) return fail(XQ_EINVAL, "null device pointer (x or xq)");
    if (xq_status s = check_shape(0, cols, batch, false)) return s;
    if (!aligned(x, 16)) return fail(XQ_EALIGN, "x must be 16-byte aligned");
    if (!aligned(xq_out, 16)) return fail(XQ_EALIGN, "xq must be 16-byte aligned");
    if (y && !aligned(y, 16)) return fail(XQ_EALIGN, "y must be 16-byte aligned");
    const size_t x_bytes = (size_t)batch * cols * 4;
    const size_t q_bytes = (size_t)batch * (cols / 256) * kQ8Bytes;
    if (overlap(xq_out, q_bytes, x, x_bytes) || (y && overlap(y, x_bytes, x, x_bytes)) ||
        (y && overlap(y, x_bytes, xq_out, q_bytes)))
        return fail(XQ_EINVAL, "outputs overlap each other or x");
    DeviceState *dev = nullptr;
    if (xq_status s = device_state(&dev)) return s;
    const dim3 grid((unsigned)((cols / 256 + 7) / 8), (unsigned)batch);
    const cudaError_t e =
        launch_kernel(rmsnorm_q8_kernel, grid, dim3(256), 0, static_cast<cudaStream_t>(stream),
                      g_overlap.load() != 0, x, static_cast<uint8_t *>(xq_out), y, cols);
    if (e != cudaSuccess) return cuda_fail(e, "RMSNorm launch");
    g_counts[XQ_COUNT_RMSNORM_Q8].fetch_add(1, std::memory_order_relaxed);
    return XQ_OK;
}

xq_status xq_matvec_q4k(const void *W, const void *xq_in, float *y, int64_t rows, int64_t cols,
                        int64_t batch, void *stream) {
    return run_matvec({kQ4K, Kind::kMatvec, XQ_COUNT_MATVEC_Q4K}, W, nullptr, xq_in, y, rows, cols, batch, stream);
}

xq_status xq_matvec_cb4(const void *W, const int8_t *table, const void *xq_in, float *y,
                        int64_t rows, int64_t cols, int64_t batch, void *stream) {
    return run_matvec({kCB4, Kind::kMatvec, XQ_COUNT_MATVEC_CB4}, W, table, xq_in, y, rows, cols, batch, stream);
}

xq_status xq_linear_q4k(const float *x, const void *W, float *y, int64_t rows, int64_t cols,
                        int64_t batch, void *stream) {
    return run_matvec({kQ4K, Kind::kLinear, XQ_COUNT_LINEAR_Q4K}, W, nullptr, x, y, rows, cols, batch, stream);
}

xq_status xq_linear_cb4(const float *x, const void *W, const int8_t *table, float *y,
                        int64_t rows, int64_t cols, int64_t batch, void *stream) {
    return run_matvec({kCB4, Kind::kLinear, XQ_COUNT_LINEAR_CB4}, W, table, x, y, rows, cols, batch, stream);
}

size_t xq_linear_workspace_bytes(int64_t cols, int64_t batch) {
    if (cols <= 0 || cols % 256 || batch < 1 || batch > 8) return 0;
    return linear_ws_bytes(cols, batch);
}

xq_status xq_linear_q4k_ws(const float *x, const void *W, float *y, int64_t rows, int64_t cols,
                           int64_t batch, void *ws, size_t ws_bytes, void *stream) {
    return run_matvec({kQ4K, Kind::kLinear, XQ_COUNT_LINEAR_Q4K}, W, nullptr, x, y, rows, cols,
                      batch, stream, ws, ws_bytes, true);
}

// Some callers cannot allocate device memory where they run the decode
// step: a host framework that owns all device memory through its own pool and
// allows no allocation outside it, or a latency-bound serving loop that may
// not call cudaMalloc (which can synchronise the device).  This variant of
// xq_linear_q4k_ws takes its workspace from the library's fixed device array
// instead of from the caller, and allocates nothing.
xq_status xq_linear_q4k_static(const float *x, const void *W, float *y, int64_t rows, int64_t cols,
                               int64_t batch, void *stream) {
    t_error.clear();
    // the caller's arguments first: a bad call makes no CUDA call at all
    if (!x || !W || !y) return fail(XQ_EINVAL, "null device pointer (x, W or y)");
    if (xq_status s = check_shape(rows, cols, batch, true)) return s;
    const size_t need = xq_linear_workspace_bytes(cols, batch);
    if (need > kStaticScratchBytes)
        return fail(XQ_ESHAPE,
                    "batch %lld x cols %lld needs %zu bytes of scratch; the fixed scratch holds %zu "
                    "(batch * cols <= %zu)",
                    (long long)batch, (long long)cols, need, kStaticScratchBytes,
                    kStaticScratchBytes / kQ8Bytes * 256);
    void *ws = nullptr;
    if (xq_status st = static_scratch(&ws)) return st;
    return run_matvec({kQ4K, Kind::kLinear, XQ_COUNT_LINEAR_Q4K}, W, nullptr, x, y, rows, cols,
                      batch, stream, ws, kStaticScratchBytes, true);
}

xq_status xq_linear_cb4_ws(const float *x, const void *W, const int8_t *table, float *y,
                           int64_t rows, int64_t cols, int64_t batch, void *ws, size_t ws_bytes,
                           void *stream) {
    return run_matvec({kCB4, Kind::kLinear, XQ_COUNT_LINEAR_CB4}, W, table, x, y, rows, cols,
                      batch, stream, ws, ws_bytes, true);
}

xq_status xq_linear_cb4r_ws(const float *x, const void *Wr, const int8_t *table, float *y,
                            int64_t rows, int64_t cols, int64_t batch, void *ws, size_t ws_bytes,
                            void *stream) {
    return run_matvec({kCB4R, Kind::kLinear, XQ_COUNT_LINEAR_CB4R}, Wr, table, x, y, rows, cols,
                      batch, stream, ws, ws_bytes, true);
}

xq_status xq_norm_linear_q4k(const float *x, const void *W, float *y, int64_t rows, int64_t cols,
                             int64_t batch, void *stream) {
    return run_matvec({kQ4K, Kind::kNormLinear, XQ_COUNT_NORM_LINEAR_Q4K}, W, nullptr, x, y, rows, cols, batch, stream);
}

xq_status xq_norm_linear_cb4(const float *x, const void *W, const int8_t *table, float *y,
                             int64_t rows, int64_t cols, int64_t batch, void *stream) {
    return run_matvec({kCB4, Kind::kNormLinear, XQ_COUNT_NORM_LINEAR_CB4}, W, table, x, y, rows, cols, batch, stream);
}

xq_status xq_matvec_q4k_id(const void *W, const int32_t *sel, const void *xq_in, float *y,
                           int64_t rows_per_expert, int64_t cols, int64_t n_experts, int64_t used,
                           int32_t x_per_slot, void *stream) {
    return run_matvec_id(kQ4K, W, nullptr, sel, xq_in, y, rows_per_expert, cols, n_experts, used,
                         x_per_slot, stream);
}

xq_status xq_matvec_cb4_id(const void *W, const int8_t *table, const int32_t *sel,
                           const void *xq_in, float *y, int64_t rows_per_expert, int64_t cols,
                           int64_t n_experts, int64_t used, int32_t x_per_slot, void *stream) {
    return run_matvec_id(kCB4, W, table, sel, xq_in, y, rows_per_expert, cols, n_experts, used,
                         x_per_slot, stream);
}

xq_status xq_subdots_q4k(const void *W, const void *xq_in, int32_t *dots, int64_t rows,
                         int64_t cols, int64_t batch, void *stream) {
    return run_matvec({kQ4K, Kind::kDots, XQ_COUNT_SUBDOTS_Q4K}, W, nullptr, xq_in, dots, rows, cols, batch, stream);
}

xq_status xq_subdots_cb4(const void *W, const int8_t *table, const void *xq_in, int32_t *dots,
                         int64_t rows, int64_t cols, int64_t batch, void *stream) {
    return run_matvec({kCB4, Kind::kDots, XQ_COUNT_SUBDOTS_CB4}, W, table, xq_in, dots, rows, cols, batch, stream);
}

size_t xq_cb4r_bytes(int64_t rows, int64_t cols) { return xq_cb4_bytes(rows, cols); }

xq_status xq_repack_cb4(const void *src, void *Wr, int64_t block_base, int64_t n_blocks,
                        int64_t rows, int64_t cols, void *stream) {
    t_error.clear();
    if (!src || !Wr) return fail(XQ_EINVAL, "null device pointer (src or Wr)");
    if (xq_status s = check_shape(rows, cols, 1, true)) return s;
    if (!aligned(Wr, 16)) return fail(XQ_EALIGN, "Wr must be 16-byte aligned");
    const int64_t bpr = cols / 32;
    if (block_base < 0 || n_blocks < 0 || block_base > rows * bpr ||
        n_blocks > rows * bpr - block_base)
        return fail(XQ_ESHAPE, "blocks %lld..%lld+%lld outside the matrix's %lld blocks",
                    (long long)block_base, (long long)block_base, (long long)n_blocks,
                    (long long)(rows * bpr));
    if ((n_blocks + 255) / 256 > 0x7FFFFFFFLL) return fail(XQ_ESHAPE, "chunk too large");
    const int64_t prefix = ((2 * bpr + 3) / 4) * 4, row_bytes = prefix + 16 * bpr;
    if (overlap(src, (size_t)n_blocks * kCb4Bytes, Wr, (size_t)(rows * row_bytes)))
        return fail(XQ_EINVAL, "src overlaps Wr");
    if (n_blocks == 0) return XQ_OK;
    DeviceState *dev = nullptr;
    if (xq_status s = device_state(&dev)) return s;
    const unsigned grid = (unsigned)((n_blocks + 255) / 256);
    repack_cb4_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t *>(src), static_cast<uint8_t *>(Wr), block_base, n_blocks, bpr,
        prefix, row_bytes, aligned(src, 16) ? 1 : 0);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "repack launch");
    g_counts[XQ_COUNT_REPACK_CB4].fetch_add(1, std::memory_order_relaxed);
    return XQ_OK;
}

xq_status xq_matvec_cb4r(const void *Wr, const int8_t *table, const void *xq_in, float *y,
                         int64_t rows, int64_t cols, int64_t batch, void *stream) {
    return run_matvec({kCB4R, Kind::kMatvec, XQ_COUNT_MATVEC_CB4R}, Wr, table, xq_in, y, rows,
                      cols, batch, stream);
}

xq_status xq_linear_cb4r(const float *x, const void *Wr, const int8_t *table, float *y,
                         int64_t rows, int64_t cols, int64_t batch, void *stream) {
    return run_matvec({kCB4R, Kind::kLinear, XQ_COUNT_LINEAR_CB4R}, Wr, table, x, y, rows, cols,
                      batch, stream);
}

xq_status xq_norm_linear_cb4r(const float *x, const void *Wr, const int8_t *table, float *y,
                              int64_t rows, int64_t cols, int64_t batch, void *stream) {
    return run_matvec({kCB4R, Kind::kNormLinear, XQ_COUNT_NORM_LINEAR_CB4R}, Wr, table, x, y,
                      rows, cols, batch, stream);
}

xq_status xq_matvec_cb4r_id(const void *Wr, const int8_t *table, const int32_t *sel,
                            const void *xq_in, float *y, int64_t rows_per_expert, int64_t cols,
                            int64_t n_experts, int64_t used, int32_t x_per_slot, void *stream) {
    return run_matvec_id(kCB4R, Wr, table, sel, xq_in, y, rows_per_expert, cols, n_experts, used,
                         x_per_slot, stream);
}

xq_status xq_subdots_cb4r(const void *Wr, const int8_t *table, const void *xq_in, int32_t *dots,
                          int64_t rows, int64_t cols, int64_t batch, void *stream) {
    return run_matvec({kCB4R, Kind::kDots, XQ_COUNT_SUBDOTS_CB4R}, Wr, table, xq_in, dots, rows,
                      cols, batch, stream);
}

xq_status xq_plan_matvec(int32_t format, int64_t rows, int64_t cols, int64_t batch,
                         int32_t sm_count, int64_t smem_optin_bytes, xq_plan *plan) {
    t_error.clear();
    if (!plan) return fail(XQ_EINVAL, "null plan");
    if (format != XQ_FORMAT_Q4K && format != XQ_FORMAT_CB4 && format != XQ_FORMAT_CB4R)
        return fail(XQ_EINVAL, "format must be XQ_FORMAT_Q4K, XQ_FORMAT_CB4 or XQ_FORMAT_CB4R");
    if (xq_status s = check_shape(rows, cols, batch, true)) return s;
    if (sm_count < 1) return fail(XQ_EINVAL, "sm_count must be positive");
    return make_plan(format == XQ_FORMAT_Q4K ? kQ4K : format == XQ_FORMAT_CB4 ? kCB4 : kCB4R, rows,
                     cols, batch, sm_count, smem_optin_bytes, plan, 0, true, 0, false, true);
}

void xq_set_plan_override(int32_t warps, int32_t stages) {
    g_override_warps.store(warps < 0 ? 0 : warps);
    g_override_stages.store(stages < 0 ? 0 : stages);
}

void xq_set_row_block_override(int32_t row_block) {
    g_override_row_block.store(row_block < 0 ? 0 : row_block);
}

void xq_set_overlap_launches(int32_t enable) { g_overlap.store(enable ? 1 : 0); }

int32_t xq_overlap_launches(void) { return g_overlap.load(); }

void xq_set_quantise_once_override(int32_t mode) {
    g_override_quantise_once.store(mode < 0 || mode > 2 ? 0 : mode);
}

void xq_set_tensor_override(int32_t mode) {
    g_override_tensor.store(mode < 0 || mode > 2 ? 0 : mode);
}

int32_t xq_codebook_split_table(const int8_t *table, uint32_t *out) {
    if (!table || !out) return 0;
    uint32_t kv[4];
    if (!split_table(table, kv)) return 0;
    for (int i = 0; i < 4; ++i) out[i] = kv[i];
    return 1;
}

void xq_set_vector_pairs_override(int32_t mode) {
    g_override_vector_pairs.store(mode < 0 || mode > 2 ? 0 : mode);
}

xq_status xq_last_plan(xq_plan *plan) {
    if (!plan) return fail(XQ_EINVAL, "null plan");
    if (!t_have_plan) return fail(XQ_EINVAL, "no mat-vec launched on this thread yet");
    *plan = t_last_plan;
    return XQ_OK;
}

uint64_t xq_launch_count(int32_t which) {
    if (which < 0 || which >= XQ_COUNT_N) return 0;
    return g_counts[which].load(std::memory_order_relaxed);
}

xq_status xq_device_status(uint32_t *out, int32_t clear, void *stream) {
    t_error.clear();
    if (!out) return fail(XQ_EINVAL, "null output");
    DeviceState *dev = nullptr;
    if (xq_status s = device_state(&dev)) return s;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(out, dev->status, sizeof(uint32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess && clear) e = cudaMemsetAsync(dev->status, 0, sizeof(uint32_t), s);
    if (e == cudaSuccess && clear) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
    return *out ? XQ_EDEVICE : XQ_OK;
}

const char *xq_status_string(xq_status s) {
    switch (s) {
        case XQ_OK: return "XQ_OK";
        case XQ_EINVAL: return "XQ_EINVAL: invalid argument";
        case XQ_EALIGN: return "XQ_EALIGN: misaligned base address";
        case XQ_ESHAPE: return "XQ_ESHAPE: shape out of range";
        case XQ_ELAUNCH: return "XQ_ELAUNCH: CUDA runtime error";
        case XQ_EDEVICE: return "XQ_EDEVICE: device status word set";
    }
    return "unknown xq_status";
}

const char *xq_last_error(void) { return t_error.c_str(); }

int32_t xq_version(void) { return 3; }

}  // extern "C"
