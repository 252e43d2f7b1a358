// Codebook instantiations of the mat-vec kernel (batch 1..8; on q8 blocks,
// with the exact sub-dot export, and fused with the activation quantiser).
#include "xq_matvec.cuh"

namespace xq {

cudaError_t launch_matvec_cb4(const MatvecArgs &a, int batch, int kind, dim3 grid, dim3 block,
                              size_t smem, cudaStream_t s) {
    return launch_matvec_fmt<kCB4, 1>(a, batch, kind, grid, block, smem, s);
}

cudaError_t configure_matvec_cb4(int smem_optin) { return configure_fmt<kCB4, 1>(smem_optin); }

}  // namespace xq
