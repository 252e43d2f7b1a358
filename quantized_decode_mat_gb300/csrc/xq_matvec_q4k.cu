// Q4_K instantiations of the mat-vec kernel with one row group per warp unit
// (batch 1..8; on q8 blocks, with the exact sub-dot export, fused with the
// quantiser or with RMSNorm + quantiser; and the grouped-expert form).  Launches
// planned with two row groups per unit go to xq_matvec_q4k_rb2.cu.
#include "xq_matvec.cuh"

namespace xq {

cudaError_t launch_matvec_q4k(const MatvecArgs &a, int batch, int kind, dim3 grid, dim3 block,
                              size_t smem, cudaStream_t s) {
    if (a.row_block == 2 && batch >= 2 && kind != 3)
        return launch_matvec_q4k_rb2(a, batch, kind, grid, block, smem, s);
    return launch_matvec_fmt<kQ4K, 1>(a, batch, kind, grid, block, smem, s);
}

cudaError_t configure_matvec_q4k(int smem_optin) {
    const cudaError_t e = configure_fmt<kQ4K, 1>(smem_optin);
    return e == cudaSuccess ? configure_matvec_q4k_rb2(smem_optin) : e;
}

}  // namespace xq
