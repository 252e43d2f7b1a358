// Q4_K instantiations with two row groups per warp unit (batch 2..8): each
// activation load from shared memory then serves two chunks of one column.
#include "xq_matvec.cuh"

namespace xq {

cudaError_t launch_matvec_q4k_rb2(const MatvecArgs &a, int batch, int kind, dim3 grid,
                                  dim3 block, size_t smem, cudaStream_t s) {
    return launch_matvec_fmt<kQ4K, 2>(a, batch, kind, grid, block, smem, s);
}

cudaError_t configure_matvec_q4k_rb2(int smem_optin) { return configure_fmt<kQ4K, 2>(smem_optin); }

}  // namespace xq
