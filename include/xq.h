/*
 * xq.h -- C ABI of the GB300 (sm_103a) 4-bit decode mat-vec library.
 *
 * y = W . x for one to eight activation vectors, with W block-quantised to 4
 * bits and x quantised once per call to q8 blocks, so that every block's dot
 * product is integer arithmetic and is scaled to float afterwards.  Two
 * weight formats:
 *
 *   Q4_K super-block, 144 bytes per 256 weights (row-major, rows contiguous):
 *     +0  f16 d            +2  f16 dmin
 *     +4  12 bytes: eight 6-bit scales sc_s and eight 6-bit mins m_s
 *         (bytes 0..3: sc_0..3 in the low 6 bits, the top 2 bits of
 *          sc_4..7; bytes 4..7: m_0..3 likewise with m_4..7; bytes 8..11:
 *          low nibble = low 4 bits of sc_4..7, high nibble = of m_4..7)
 *     +16 128 nibble bytes: group g (0..3) = bytes 16+32g..16+32g+31; the
 *         low nibbles are sub-block 2g, the high nibbles sub-block 2g+1
 *     weight value w = d*sc_s*q - dmin*m_s (never formed on this route)
 *     Source: super-block stride 144 and group offset 16+32g, "cajeta.xpu -
 *     one kernel, any device" section 2.3; the field layout is the Q4_K
 *     block of the decode workload.
 *
 *   Nonlinear 4-bit codebook block, 18 bytes per 32 weights:
 *     +0 f16 d, +2 16 payload bytes; element j < 16 is kv[qs[j] & 15],
 *     element j >= 16 is kv[qs[j-16] >> 4]; kv is a 16-entry int8 table.
 *     Source: "25 - Writing XPU Kernels" section 25.2.1.
 *
 *   q8 activation block, 320 bytes per 256 values ("25 - Writing XPU
 *   Kernels" section 25.2): +0 int8 q[256], +256 int32 sums of each
 *   32-value sub-block, +288 f32 scale, +292..319 zero.
 *
 * Conventions for every entry point
 *   - Pointers named W, xq, x, y, dots are DEVICE pointers owned by the
 *     caller; `table` is a HOST pointer read during the call (copied by
 *     value into the launch).  The library allocates no device memory and
 *     keeps no state beyond launch counters, the last launch plan of the
 *     calling thread, a per-device status word and per-thread error text.
 *   - Layouts are row-major; x is [batch][cols] f32, xq is
 *     [batch][cols/256][320 B], y is [batch][rows] f32, fully overwritten.
 *   - Preconditions, all checked on the host before any CUDA call:
 *     cols > 0 and cols % 256 == 0; 1 <= rows <= 2^31-1; 1 <= batch <= 8;
 *     the mat-vec kernels also need one q8 vector to fit in shared memory
 *     beside two weight stages: cols <= 169984 on GB300 (232448 bytes of
 *     shared memory a CTA), else XQ_ESHAPE;
 *     W, xq, x and dots 16-byte aligned; y 4-byte aligned; outputs must not
 *     overlap inputs.  A violation returns XQ_EINVAL / XQ_EALIGN / XQ_ESHAPE
 *     and launches nothing.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *     compute entry point is asynchronous on it: the return code covers
 *     argument checks and the launch only.  Nothing here synchronises except
 *     xq_device_status.  No kernel traps or asserts; the one wait in a kernel
 *     on its own tensor-core operations is bounded and, if it runs out,
 *     sets bit 2 of the device status word.
 *   - The first call on a device configures the kernels for that device;
 *     make one call per device before capturing a stream into a CUDA graph.
 */
#ifndef XQ_H
#define XQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    XQ_OK = 0,
    XQ_EINVAL = 1,  /* null pointer, overlapping buffers, bad argument      */
    XQ_EALIGN = 2,  /* a base address is not aligned as required          */
    XQ_ESHAPE = 3,  /* rows, cols or batch out of range                     */
    XQ_ELAUNCH = 4, /* the CUDA runtime refused a query or the launch       */
    XQ_EDEVICE = 5  /* the device status word reports a kernel-side error   */
} xq_status;

/* Bytes of the q8 blocks for `batch` vectors of `cols` values; 0 if the
 * shape is invalid.  = batch * (cols/256) * 320. */
size_t xq_q8_bytes(int64_t cols, int64_t batch);
/* Bytes of a Q4_K matrix: rows * (cols/256) * 144; 0 if invalid. */
size_t xq_q4k_bytes(int64_t rows, int64_t cols);
/* Bytes of a codebook matrix: rows * (cols/32) * 18; 0 if invalid. */
size_t xq_cb4_bytes(int64_t rows, int64_t cols);

/* Quantise x ([batch][cols] f32, device) into q8 blocks xq (device,
 * xq_q8_bytes(cols, batch) bytes), one 256-value block at a time:
 * amax = max|x|; d = amax/127; q = round-half-even(x * (127/amax)) clamped
 * to [-127, 127] (all in f32 with one rounding per operation); an all-zero
 * block gets d = 0, q = 0; the eight 32-value sums are stored exactly.
 * Source: "25 - Writing XPU Kernels" section 25.2 (the q8_K block: quantise
 * the activation once, 256 int8 values, eight sums, one f32 scale); the
 * scale and rounding rule are this library's reading (the page names no
 * rule). */
xq_status xq_quantize_q8(const float *x, void *xq, int64_t cols, int64_t batch, void *stream);

/* y[b][r] = sum over super-blocks k of xs_{b,k} * (d_{r,k} * sum_s sc_s*dot_s
 *           - dmin_{r,k} * sum_s m_s*bsum_{b,k,s}),
 * dot_s = sum of 32 (unsigned nibble x signed int8) products, exact.
 * W: Q4_K rows (device, xq_q4k_bytes(rows, cols)), xq: q8 blocks of the
 * batch, y: [batch][rows] f32.  Integer dots are exact; the float epilogue
 * carries a compensation term so y is within a few f32 ulps of the exact
 * value.  Source: "25 - Writing XPU Kernels" sections 25.2 (integer route,
 * reduce first then scale once) and 25.5 (the Q4_K mat-vec as 16-byte
 * vector loads and dp4a); "cajeta.xpu - one kernel, any device" 2.3. */
xq_status xq_matvec_q4k(const void *W, const void *xq, float *y, int64_t rows, int64_t cols,
                        int64_t batch, void *stream);

/* y[b][r] = sum over blocks k of d_{r,k} * xs_{b,k/8} * dot_k,
 * dot_k = sum_j kv[nibble_j] * xq_{b, 32k+j} (signed x signed, exact).
 * table: HOST pointer to the 16 int8 codebook values, read during the call.
 * Source: "25 - Writing XPU Kernels" section 25.2.1 (the integer codebook
 * decode wave: the codebook maps a nibble to int8, one float multiply per
 * block after the integer dot). */
xq_status xq_matvec_cb4(const void *W, const int8_t *table, const void *xq, float *y,
                        int64_t rows, int64_t cols, int64_t batch, void *stream);

/* The fused decode step: quantise x ([batch][cols] f32, device) to q8 blocks
 * exactly as xq_quantize_q8 does, and compute y = W . x as xq_matvec_q4k /
 * xq_matvec_cb4 do, in one launch and without a q8 buffer: every CTA
 * quantises the activation into its own shared memory.  y is bit-identical
 * to the two-call path.  x must be 16-byte aligned.  Source: the fused tail
 * of "25 - Writing XPU Kernels" 25.5 (chained launches cost round trips; a
 * fused tail removes the gaps as well as the launches). */
xq_status xq_linear_q4k(const float *x, const void *W, float *y, int64_t rows, int64_t cols,
                        int64_t batch, void *stream);
xq_status xq_linear_cb4(const float *x, const void *W, const int8_t *table, float *y,
                        int64_t rows, int64_t cols, int64_t batch, void *stream);

/* The decode step with a caller workspace.  It computes what xq_linear_q4k /
 * _cb4 / _cb4r compute, bit for bit, and picks how by the shape
 * (xq_plan.quantise_once):
 *   - small activations: the one fused launch, where every CTA quantises the
 *     activation into its own shared memory (the workspace is not touched);
 *   - wide or batched activations (more than 32 q8 blocks a launch): the
 *     activation is quantised once, by xq_quantize_q8's kernel, into the
 *     workspace, and the mat-vec reads those q8 blocks.  Every CTA
 *     re-quantising the whole activation costs more than the second launch
 *     there (measured on GB300: 4096 x 14336 at batch 4, 16.8 us fused against
 *     13.9 us).
 * ws: DEVICE scratch of at least xq_linear_workspace_bytes(cols, batch) bytes
 * (= xq_q8_bytes(cols, batch)), 16-byte aligned, not overlapping x, W or y;
 * its contents on entry do not matter; on return it holds the q8 blocks of
 * the last launch's vectors or is untouched.  Calls that share a workspace
 * must not overlap on the GPU.  Source: "25 - Writing XPU Kernels" 25.2
 * (quantise the activation once per call) and 25.5 (fuse where it removes
 * work, not only launches). */
size_t xq_linear_workspace_bytes(int64_t cols, int64_t batch);
xq_status xq_linear_q4k_ws(const float *x, const void *W, float *y, int64_t rows, int64_t cols,
                           int64_t batch, void *ws, size_t ws_bytes, void *stream);
xq_status xq_linear_cb4_ws(const float *x, const void *W, const int8_t *table, float *y,
                           int64_t rows, int64_t cols, int64_t batch, void *ws, size_t ws_bytes,
                           void *stream);
xq_status xq_linear_cb4r_ws(const float *x, const void *Wr, const int8_t *table, float *y,
                            int64_t rows, int64_t cols, int64_t batch, void *ws, size_t ws_bytes,
                            void *stream);

/* xq_linear_q4k_ws without a caller workspace, for callers that cannot
 * allocate device memory where they run the decode step (a framework that
 * owns all device memory and allows no allocation outside its pool, or a
 * serving loop that may not call cudaMalloc, which can synchronise the
 * device).  The scratch is a fixed device array of 256 KiB inside the library
 * (every GPU that loads the library holds it until the process exits), so a
 * call may need at most 819 q8 blocks (xq_linear_workspace_bytes(cols, batch)
 * <= 262144, i.e. batch * cols <= 209664); larger shapes return XQ_ESHAPE and
 * launch nothing.  The call
 * allocates nothing.  Null pointers and bad shapes are refused before any
 * CUDA call.  The first call on a device that passes those checks looks up
 * the array's device address (cudaGetSymbolAddress) for that device and keeps
 * it (a failed lookup is not kept: the next call tries again), so make that
 * first call before any stream capture.  Nothing in the array needs clearing: the
 * q8 blocks are written before they are read.  Every call shares the one
 * array, which keeps the last call's contents, so calls that may overlap on
 * the GPU (other streams, other threads) race; order them on one stream.
 * Arguments, results and other errors as xq_linear_q4k_ws.  The pages have no
 * counterpart to this entry point. */
xq_status xq_linear_q4k_static(const float *x, const void *W, float *y, int64_t rows, int64_t cols,
                               int64_t batch, void *stream);

/* RMSNorm + q8 pack, the producer of the next layer's activation blocks:
 * for each of the batch vectors x_b ([batch][cols] f32, device),
 *   scale_b = 1 / sqrt(sum_i x_{b,i}^2 / cols + 1e-5),  y_b = x_b * scale_b,
 * and xq receives the q8 blocks of y_b exactly as xq_quantize_q8 would write
 * them.  The f32 sum of squares is taken in one fixed order, that of a
 * workgroup of 256 items in eight waves of 32: item t adds x_t^2,
 * x_{t+256}^2, ... in turn, each wave combines its items by an xor
 * butterfly over lane offsets 16, 8, 4, 2, 1, and the eight wave sums are
 * added from wave 0 upward; every f32 operation rounds once.  So the scale
 * and the q8 codes are one defined value, not merely close.  y (device,
 * [batch][cols] f32, 16-byte aligned) receives y_b when it is non-null.
 * Shapes as for xq_quantize_q8.  Source: "25 - Writing XPU Kernels" 25.2.3
 * (a sum across the whole workgroup; the RMSNorm kernel) and 25.5 (a fused
 * tail ends with the next layer's norm and pack). */
xq_status xq_rmsnorm_q8(const float *x, void *xq, float *y, int64_t cols, int64_t batch,
                        void *stream);

/* The fused decode step behind an RMSNorm: y = W . q8(x_b * scale_b), with
 * scale_b as in xq_rmsnorm_q8, in one launch (every CTA computes the scale
 * in the same fixed order and quantises into its own shared memory).  y is
 * bit-identical to xq_rmsnorm_q8 followed by xq_matvec_q4k / xq_matvec_cb4.
 * x must be 16-byte aligned. */
xq_status xq_norm_linear_q4k(const float *x, const void *W, float *y, int64_t rows, int64_t cols,
                             int64_t batch, void *stream);
xq_status xq_norm_linear_cb4(const float *x, const void *W, const int8_t *table, float *y,
                             int64_t rows, int64_t cols, int64_t batch, void *stream);

/* Grouped experts ("25 - Writing XPU Kernels" 25.2.2, the mul_mat_vec_id
 * shape): W is a slab of n_experts experts of rows_per_expert rows each,
 * contiguous; sel (DEVICE int32[used]) selects the experts.  One launch
 * computes, for every slot kk < used,
 *   y[kk*rows_per_expert + r] = (row r of expert sel[kk]) . x_kk,
 * where x_kk is q8 vector 0 of xq when x_per_slot == 0 (every slot reads the
 * one decoded token) and q8 vector kk when x_per_slot != 0 (used <= 8).  y is
 * slot-major, [used][rows_per_expert], and bit-identical to one dense
 * xq_matvec_* launch per slot.  A slot whose id lies outside [0, n_experts)
 * reads nothing, gets NaN rows and sets bit 1 of the device status word. */
xq_status xq_matvec_q4k_id(const void *W, const int32_t *sel, const void *xq, float *y,
                           int64_t rows_per_expert, int64_t cols, int64_t n_experts, int64_t used,
                           int32_t x_per_slot, void *stream);
xq_status xq_matvec_cb4_id(const void *W, const int8_t *table, const int32_t *sel, const void *xq,
                           float *y, int64_t rows_per_expert, int64_t cols, int64_t n_experts,
                           int64_t used, int32_t x_per_slot, void *stream);

/* ---- Resident codebook rows ("25 - Writing XPU Kernels" 25.4, one resident
 * layout read by every kernel, and the 25.2.1 kernel that walks it) --------
 * A resident row of a codebook matrix holds the f16 scales of its
 * bpr = cols/32 blocks first (block j's at byte 2j), padded to a whole dword,
 * then the blocks' 16-byte payloads (block j's at prefix + 16j), so every
 * payload is a 16-byte aligned run:
 *   prefix = ceil(2*bpr / 4) * 4 bytes,  row bytes = prefix + 16*bpr.
 * With cols % 256 == 0 (this library's shapes) prefix = cols/16 and a row is
 * 144*cols/256 bytes, the size of the raw row, and both are multiples of 16.
 * The payload bytes are the raw block's bytes 2..17 unchanged.
 *
 * Bytes of a resident matrix: rows * (prefix + 16*bpr); 0 if invalid. */
size_t xq_cb4r_bytes(int64_t rows, int64_t cols);

/* Repack raw codebook blocks into resident rows: src (DEVICE, any alignment)
 * holds n_blocks consecutive raw 18-byte blocks, blocks block_base ..
 * block_base + n_blocks - 1 of the row-major raw matrix (block g is block
 * g % bpr of row g / bpr); each is written into the resident matrix Wr
 * (DEVICE, 16-byte aligned, xq_cb4r_bytes(rows, cols) bytes): its scale to
 * the row's prefix, its payload to the row's payload run.  A chunk may start
 * and end anywhere, including mid-row; bytes of Wr that the chunk does not
 * cover are left as they are, so chunks can be repacked in any order.  One
 * launch moves the scales and the payloads together (the page's separate
 * scale pass re-reads every block's line for two bytes).  n_blocks == 0 is a
 * no-op that launches nothing.  Preconditions (host-checked): cols as for
 * the mat-vec; 0 <= block_base, block_base + n_blocks <= rows*cols/32; src
 * and Wr do not overlap. */
xq_status xq_repack_cb4(const void *src, void *Wr, int64_t block_base, int64_t n_blocks,
                        int64_t rows, int64_t cols, void *stream);

/* The codebook entry points on resident rows Wr (same arguments, results and
 * preconditions as their raw-layout twins above; y is bit-identical to the
 * twin's on the same weights, because only the staging of the bytes
 * differs). */
xq_status xq_matvec_cb4r(const void *Wr, const int8_t *table, const void *xq, float *y,
                         int64_t rows, int64_t cols, int64_t batch, void *stream);
xq_status xq_linear_cb4r(const float *x, const void *Wr, const int8_t *table, float *y,
                         int64_t rows, int64_t cols, int64_t batch, void *stream);
xq_status xq_norm_linear_cb4r(const float *x, const void *Wr, const int8_t *table, float *y,
                              int64_t rows, int64_t cols, int64_t batch, void *stream);
xq_status xq_matvec_cb4r_id(const void *Wr, const int8_t *table, const int32_t *sel,
                            const void *xq, float *y, int64_t rows_per_expert, int64_t cols,
                            int64_t n_experts, int64_t used, int32_t x_per_slot, void *stream);
xq_status xq_subdots_cb4r(const void *Wr, const int8_t *table, const void *xq, int32_t *dots,
                          int64_t rows, int64_t cols, int64_t batch, void *stream);

/* Test exports: the exact per-sub-block integer dots of the same kernels.
 * dots: [batch][rows][cols/32] int32 (device).  Q4_K: dots[b][r][8k+s] is
 * dot_s of super-block k; codebook: dots[b][r][k] is dot_k of block k. */
xq_status xq_subdots_q4k(const void *W, const void *xq, int32_t *dots, int64_t rows,
                         int64_t cols, int64_t batch, void *stream);
xq_status xq_subdots_cb4(const void *W, const int8_t *table, const void *xq, int32_t *dots,
                         int64_t rows, int64_t cols, int64_t batch, void *stream);

/* Weight formats, for xq_plan_matvec. */
enum { XQ_FORMAT_Q4K = 0, XQ_FORMAT_CB4 = 1, XQ_FORMAT_CB4R = 2 };

/* Launch plan of the mat-vec kernels (pure host computation; needs no GPU).
 * format: XQ_FORMAT_Q4K, XQ_FORMAT_CB4 or XQ_FORMAT_CB4R.  sm_count and
 * smem_optin_bytes describe the device (for GB300: 152 SMs, 232448 bytes).
 * A work unit (row group) is rows_per_group rows read as `segments`
 * contiguous boxes of at most 32 chunks of 256 weights (4608 bytes); lane l
 * of a warp takes chunk l of a box.  A warp works on row_block row groups at
 * once (2 for Q4_K with two or more activation vectors: each activation load
 * then serves two chunks of one column), one stage holding row_block boxes.
 * Each of the `warps` warps of the `grid` persistent CTAs keeps stages-1
 * stages in flight (with one stage, the warp waits for its own copies and the
 * other warps' work covers them).  The batch's q8 blocks are staged in shared memory; if
 * they do not fit, each call makes `launches` launches of batch_per_launch
 * vectors (each re-reads W).  quantise_once: 1 if the decode step with a
 * workspace (xq_linear_q4k_ws) quantises the activation once, in a launch of
 * its own, 0 if every CTA of the fused launch quantises it for itself;
 * xq_plan_matvec reports that step's choice, and the other entry points
 * ignore the field.  vector_pairs: 1 if each unit of work (two row groups)
 * and its stages are shared by a pair of warps that compute half of the
 * vectors each (the Q4_K mat-vec on q8 blocks with rows of 16 chunks at 8
 * vectors, on matrices large enough to give each pair many units; then
 * warps = 16 by default, stages counts the stages of a pair, and smem_bytes
 * includes each warp's reduction scratch).  tensor: 1 if the dots are
 * taken on the tensor cores (tcgen05; the Q4_K mat-vec on q8 blocks with
 * rows of 16 chunks at 5..8 vectors): one CTA of seventeen warps an SM then
 * owns tiles of 128 rows (groups = tiles, rows_per_group = 128, segments =
 * 16 chunks a tile), and smem_bytes includes the activation staged as
 * f16. */
typedef struct {
    int32_t warps;
    int32_t stages;
    int32_t grid;
    int32_t rows_per_group;
    int32_t segments;
    int32_t chunks_per_row;
    int64_t groups;
    int32_t batch_per_launch;
    int32_t launches;
    int64_t smem_bytes;
    int32_t row_block;
    int32_t quantise_once;
    int32_t vector_pairs;
    int32_t tensor;
} xq_plan;

xq_status xq_plan_matvec(int32_t format, int64_t rows, int64_t cols, int64_t batch,
                         int32_t sm_count, int64_t smem_optin_bytes, xq_plan *plan);
/* Override the automatic plan for sweeps: warps (up to the kernel's limit:
 * 20 at batch 1, 16 for the fused RMSNorm form there; Q4_K 12 at batch 2, 8
 * above; codebook 16 up to batch 4, 8 above) and stages (1..8), 0 =
 * automatic.  Process-wide; not for concurrent
 * use with launches. */
void xq_set_plan_override(int32_t warps, int32_t stages);
/* Override the row groups a warp works on at once: 1, or 2 where the
 * automatic plan would use 2 (Q4_K at batch >= 2); 0 = automatic.
 * Process-wide, for sweeps and tests, like xq_set_plan_override. */
void xq_set_row_block_override(int32_t row_block);
/* Override the choice of the decode step with a workspace: 1 = every CTA
 * quantises the activation, 2 = quantise once into the workspace, 0 =
 * automatic.  Process-wide, for sweeps and tests. */
void xq_set_quantise_once_override(int32_t mode);
/* Override the use of warp pairs (xq_plan.vector_pairs): 1 = never, 2 =
 * wherever they apply (the Q4_K mat-vec on q8 blocks, rows of 16 chunks, 8
 * vectors, any matrix size), 0 = automatic (not beside a warp or stage
 * override).  When forced, a warp override (rounded down to even, 2..16) and
 * a stage override (2..8) size the pairs if they fit in shared memory.
 * Process-wide, for sweeps and tests; the results are bit-identical either
 * way. */
void xq_set_vector_pairs_override(int32_t mode);
/* Override the use of the tensor cores (xq_plan.tensor): 1 = never, 2 =
 * wherever they apply (the Q4_K mat-vec on q8 blocks, rows of 16 chunks, 5..8
 * vectors), 0 = automatic.  When forced, a stage override (2..8) sizes the
 * plan if it fits in shared memory.  Process-wide, for sweeps and tests; the
 * results are bit-identical either way. */
void xq_set_tensor_override(int32_t mode);
/* The codebook table as the one-vector launches use it, when it splits: four
 * words, bytes L[0..7] then H[0..7], with kv[n] = L[n] + rep(H[n]) and
 * kv[n + 8] = rep(L[n]) + H[n] for n = 0..7 (signed bytes; rep(v) = -1 if
 * v < 0, else 0), which a byte permute in its sign-replicating mode reads as
 * two lookups whose sum is kv.  Returns 1 and writes out[0..3], or 0 when no
 * such split exists (an entry of 127 next to one that needs a larger
 * partner), in which case those launches decode with the sixteen-byte table.
 * Host only; for tests. */
int32_t xq_codebook_split_table(const int8_t *table, uint32_t *out);
/* Plan used by the calling thread's last mat-vec or sub-dot launch. */
xq_status xq_last_plan(xq_plan *plan);

/* Overlapped launches (process-wide; default off).  When on, the mat-vec,
 * quantise and RMSNorm entry points launch their kernels with programmatic
 * stream serialization: a launch may start while the kernel before it on the
 * stream is still finishing.  Such a kernel first requests its first weight
 * boxes (it reads W and nothing else), then waits until the earlier kernel has
 * completed and its writes are visible before it reads x, q8 blocks or expert
 * ids and before it writes anything.  So the kernel just before a mat-vec on
 * the stream must not write that mat-vec's W (for instance xq_repack_cb4 into
 * the rows it then reads): separate the two with an event or a stream
 * synchronisation, or keep overlap off.  Constant weights, the decode case,
 * are safe.  With overlap on, consecutive launches hide each other's start-up
 * and tail. */
void xq_set_overlap_launches(int32_t enable);
int32_t xq_overlap_launches(void);

/* Launch counters (process-wide, monotonic) per kernel family. */
enum {
    XQ_COUNT_QUANTIZE = 0,
    XQ_COUNT_MATVEC_Q4K = 1,
    XQ_COUNT_MATVEC_CB4 = 2,
    XQ_COUNT_SUBDOTS_Q4K = 3,
    XQ_COUNT_SUBDOTS_CB4 = 4,
    XQ_COUNT_LINEAR_Q4K = 5,
    XQ_COUNT_LINEAR_CB4 = 6,
    XQ_COUNT_MATVEC_ID_Q4K = 7,
    XQ_COUNT_MATVEC_ID_CB4 = 8,
    XQ_COUNT_RMSNORM_Q8 = 9,
    XQ_COUNT_NORM_LINEAR_Q4K = 10,
    XQ_COUNT_NORM_LINEAR_CB4 = 11,
    XQ_COUNT_REPACK_CB4 = 12,
    XQ_COUNT_MATVEC_CB4R = 13,
    XQ_COUNT_SUBDOTS_CB4R = 14,
    XQ_COUNT_LINEAR_CB4R = 15,
    XQ_COUNT_NORM_LINEAR_CB4R = 16,
    XQ_COUNT_MATVEC_ID_CB4R = 17,
    XQ_COUNT_QUANTISE_ONCE = 18,
    XQ_COUNT_N = 19
};
uint64_t xq_launch_count(int32_t which);

/* Read (and optionally clear) the current device's status word, where
 * kernels report errors without trapping: bit 1 = a grouped mat-vec met an
 * expert id outside [0, n_experts); bit 2 = a tensor-core mat-vec gave up
 * waiting for its own products (its outputs are then not written).  Returns
 * XQ_EDEVICE when it is non-zero.
 * SYNCHRONISES `stream` (device-to-host copy of 4 bytes, and a clear). */
xq_status xq_device_status(uint32_t *out, int32_t clear, void *stream);

const char *xq_status_string(xq_status s);
/* Detail text of the calling thread's last failed call ("" if none). */
const char *xq_last_error(void);
/* ABI version: 2 (the plan struct gained row_block and quantise_once). */
int32_t xq_version(void);

#ifdef __cplusplus
}
#endif
#endif /* XQ_H */
