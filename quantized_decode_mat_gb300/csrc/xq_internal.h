// Internal declarations shared by the library's translation units (host and
// device).  Not part of the public ABI (that is include/xq.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "xq.h"

namespace xq {

// Layout constants of the formats (see include/xq.h).
constexpr int kQ8Bytes = 320;       // q8 block: 256 int8, 8 int32 sums, f32 scale, pad
constexpr int kQ8SumAt = 256;
constexpr int kQ8ScaleAt = 288;
constexpr int kQ4kBytes = 144;      // Q4_K super-block
constexpr int kCb4Bytes = 18;       // codebook block
// A 256-weight chunk of a row is 144 bytes in both formats: one Q4_K
// super-block, or eight codebook blocks (8 * 18).  It pairs with exactly one
// q8 activation block.
constexpr int kChunkBytes = 144;
constexpr int kTileRows = 32;                       // lanes (chunks) per box
constexpr int kStageBytes = kTileRows * kChunkBytes;  // one staged box: 4608 B
// Shared-memory stride of a staged q8 block: bytes 0..303 of the block, then
// its split sums at 304..319; 336 = 84 words puts 8 consecutive chunks on
// distinct 4-bank groups.  Bytes 320..335 are padding; the fused RMSNorm
// kernels park a vector's scale there, in its first block.
constexpr int kActStride = 336;
constexpr int kActSplitAt = 304;
constexpr int kActNormAt = 320;
// q8 blocks whose activation values one warp loads at once in the fused
// kernels at batch 1 (one L2 round trip per group; twice as many above).
constexpr int kQuantGroup = 4;
// Staging of q8 blocks into shared memory: from kStageAsyncBlocks blocks up
// (Q4_K), asynchronous copies all in flight at once (4096 x 14336 at batch 8:
// 23.5 against 31.4 us for one load a thread at a time); below, and for the
// codebook (whose reordering pass then runs after the copies and measured
// slower), loads issued kStageItems items (16 or 32 bytes each) at a time
// before any store (4 and 8 measured alike; 4 keeps the registers low).
constexpr int kStageAsyncBlocks = 64;
constexpr int kStageItems = 4;
constexpr int kMaxWarps = 8;
// Warp pairs (the row-blocked Q4_K form for rows of 16 chunks, 8 vectors):
// each unit of two row groups and its stages are shared by two warps, each
// computing half of the vectors; 16 warps a CTA (8 pairs, 128 registers a
// thread), and each warp's reduction scratch (32 lanes x (2 x 4 + 1) pairs of
// floats) after the stages.
constexpr int kVpWarps = 16;
constexpr int kVpStages = 2;
constexpr int kVpScratchBytes = (2 * 4 + 1) * 8 * 32;
constexpr int kMaxStages = 8;
// Tensor-core form (xq_tc.cuh): Q4_K rows of 16 chunks, 5..8 vectors on q8
// blocks.  A CTA of eight decoding, eight epilogue and one issuing warp owns
// tiles of 128 rows; shared memory: the activation as the f16 B operand (16 chunks x
// 16 slices x 256 bytes), the q8 scales and split sums per (chunk, vector),
// each lane quarter's weight stages (32 rows x one chunk), the tensor-memory
// address and six mbarriers; tensor memory (all 512 columns): A twice in 128
// columns, the eight sub-block accumulators (16 columns each) twice in 128.
constexpr int kTcWorkWarps = 16;
// registers a thread: five of the 17 warps on one scheduler share its 16384
constexpr int kTcMaxRegs = 96;
constexpr int kTcThreads = (kTcWorkWarps + 1) * 32;
constexpr int kTcRows = 128;
constexpr int kTcChunks = 16;
constexpr int kTcTmemCols = 512;
constexpr int kTcXsAt = kTcChunks * 16 * 256;
constexpr int kTcSplitAt = kTcXsAt + kTcChunks * 8 * 4;
constexpr int kTcStagesAt = kTcSplitAt + kTcChunks * 8 * 16;
constexpr int kTcQStageBytes = 32 * kChunkBytes;
constexpr int kTcStageBytes = 4 * kTcQStageBytes;  // the four quarters' stages of one step
constexpr int kTcStages = 3;
constexpr uint32_t kTcSpinLimit = 1u << 20;
// shared memory of a launch with S stages (1024 bytes of alignment slack)
constexpr int64_t tc_smem_bytes(int S) { return (int64_t)kTcStagesAt + (int64_t)S * kTcStageBytes + 64 + 1024; }
static_assert(kTcStagesAt % 128 == 0 && kTcStageBytes % 128 == 0, "128-byte aligned regions");

// kCB4R: codebook blocks in resident rows (scale prefix, then 16-byte
// payloads).  A 256-weight chunk is then 16 bytes of scales in the prefix and
// 128 bytes of payloads, 144 bytes in all, as in the raw layout.
enum Format { kQ4K = 0, kCB4 = 1, kCB4R = 2 };

// Largest warps per CTA of an instantiation (format, batch), which its
// register budget allows no more.  Each of the SM's four schedulers has a
// quarter of the register file, so the cap is set by the warps a scheduler
// holds: 20 warps (5 a scheduler) allow 96 registers a thread, 16 allow 128,
// 12 allow 168, 8 allow 255.  Batch 1: 20 (72-95 registers), but 16 for
// the fused RMSNorm form (fuse 2), whose one-warp norm pass ran slower in 96
// registers.  Q4_K: 12 at batch 2, 8 above (its row-blocked kernels need up
// to 211).  Codebook: 16 up to batch 4 (98-128 registers), 8 above (12
// measured slower there).  Warp counts that split unevenly over the
// schedulers measured slower.  The exact-dots builds (a test export) of two
// vectors or more take 8, so that writing the dots never spills.  The planner
// may use fewer (see make_plan).
constexpr int warps_limit(int fmt, int64_t batch, int fuse = 0, bool dots = false) {
    return batch == 1 ? (fuse == 2 ? 16 : 20)
           : dots     ? kMaxWarps
           : fmt == kQ4K ? (batch == 2 ? 12 : kMaxWarps) : (batch <= 4 ? 16 : kMaxWarps);
}

struct MatvecArgs {
    const uint8_t *W;       // [rows][nb][144]
    const uint8_t *xq;      // [batch][nb][320] (q8 input)
    const float *x;         // [batch][cols] (fused quantise + mat-vec input)
    float *y;               // [batch][rows]
    int32_t *dots;          // [batch][rows][nb*8] (sub-dot launches only)
    int64_t rows;
    int64_t groups;         // ceil(rows / rows_per_group)
    int32_t nb;             // 256-weight chunks per row
    int32_t rows_per_group; // 32/nb if nb is a power of two below 32, else 1
    int32_t segments;       // boxes per group: 1, or ceil(nb/32) when rows_per_group == 1
    int32_t stages;         // shared-memory stages per warp (2..8)
    int32_t row_block;      // row groups a warp works on at once (1, or 2 for Q4_K at batch >= 2)
    int32_t vector_pairs;   // 1: warp pairs share each unit, half of the vectors each
    int32_t tensor;         // 1: the tensor-core kernel (xq_tc.cuh)
    uint32_t kv[4];         // codebook bytes kv[0..15], little-endian words (or, with
                            // kv_split, the two lookup tables whose sum is kv)
    int32_t kv_split;       // 1: kv holds the split tables (one-vector launches)
    // grouped-expert form
    const int32_t *sel;     // [used] expert ids (device)
    int64_t rows_per_expert;
    int32_t n_experts;
    int32_t groups_per_slot;
    int32_t act_vectors;    // 1: every slot reads vector 0; used: slot kk reads vector kk
    uint32_t *status;       // device status word
    int32_t overlap;        // host side: launch with programmatic stream serialization
};

// Launch a kernel, with programmatic stream serialization when `overlap`: the
// grid may start while the one before it on the stream finishes (its kernels
// call grid_dependency_wait before touching anything but the weights).
template <class... P, class... A>
inline cudaError_t launch_kernel(void (*kern)(P...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t s, bool overlap, A... args) {
    if (!overlap) {
        kern<<<grid, block, smem, s>>>(args...);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Status word bits (see xq_device_status).
constexpr uint32_t kStatusBadExpertId = 2u;
constexpr uint32_t kStatusTensorTimeout = 4u;

// Launch entry points implemented per format (xq_matvec_q4k.cu / _cb4.cu).
// kind: 0 = mat-vec on q8 blocks, 1 = the same with the exact dots,
// 2 = fused quantise + mat-vec on f32 x, 3 = grouped experts, 4 = fused
// RMSNorm + quantise + mat-vec.
cudaError_t launch_matvec_q4k(const MatvecArgs &a, int batch, int kind, dim3 grid, dim3 block,
                              size_t smem, cudaStream_t s);
cudaError_t launch_matvec_cb4(const MatvecArgs &a, int batch, int kind, dim3 grid, dim3 block,
                              size_t smem, cudaStream_t s);
// Raise the dynamic shared memory limit of every instantiation of a format.
cudaError_t configure_matvec_q4k(int smem_optin);
cudaError_t configure_matvec_cb4(int smem_optin);
cudaError_t launch_matvec_q4k_rb2(const MatvecArgs &a, int batch, int kind, dim3 grid,
                                  dim3 block, size_t smem, cudaStream_t s);
cudaError_t configure_matvec_q4k_rb2(int smem_optin);
cudaError_t launch_matvec_cb4r(const MatvecArgs &a, int batch, int kind, dim3 grid, dim3 block,
                               size_t smem, cudaStream_t s);
cudaError_t configure_matvec_cb4r(int smem_optin);
// The tensor-core Q4_K mat-vec on q8 blocks (xq_matvec_q4k_tc.cu): rows of 16
// chunks, batch 5..8.
cudaError_t launch_matvec_q4k_tc(const MatvecArgs &a, int batch, dim3 grid, dim3 block,
                                 size_t smem, cudaStream_t s);
cudaError_t configure_matvec_q4k_tc(int smem_optin);

}  // namespace xq
