// Instantiations of the mat-vec kernel on resident codebook rows (scale
// prefix, then 16-byte payloads): batch 1..8; on q8 blocks, with the exact
// sub-dot export, fused with the quantiser or with RMSNorm + quantiser; and
// the grouped-expert form.
#include "xq_matvec.cuh"

namespace xq {

cudaError_t launch_matvec_cb4r(const MatvecArgs &a, int batch, int kind, dim3 grid, dim3 block,
                               size_t smem, cudaStream_t s) {
    return launch_matvec_fmt<kCB4R, 1>(a, batch, kind, grid, block, smem, s);
}

cudaError_t configure_matvec_cb4r(int smem_optin) { return configure_fmt<kCB4R, 1>(smem_optin); }

}  // namespace xq
