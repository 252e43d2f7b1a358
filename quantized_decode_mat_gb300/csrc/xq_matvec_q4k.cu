// Q4_K instantiations of the mat-vec kernel (batch 1..8; on q8 blocks, with
// the exact sub-dot export, and fused with the activation quantiser).
#include "xq_matvec.cuh"

namespace xq {

cudaError_t launch_matvec_q4k(const MatvecArgs &a, int batch, int kind, dim3 grid, dim3 block,
                              size_t smem, cudaStream_t s) {
    return launch_matvec_fmt<kQ4K>(a, batch, kind, grid, block, smem, s);
}

cudaError_t configure_matvec_q4k(int smem_optin) { return configure_fmt<kQ4K>(smem_optin); }

}  // namespace xq
