// The tensor-core Q4_K mat-vec (xq_tc.cuh): rows of 16 chunks, 5..8 vectors on
// q8 blocks.
#include "xq_tc.cuh"

namespace xq {

cudaError_t launch_matvec_q4k_tc(const MatvecArgs &a, int batch, dim3 grid, dim3 block,
                                 size_t smem, cudaStream_t s) {
    const bool ov = a.overlap != 0;
    switch (batch) {
        case 5: return launch_kernel(xq_tc_q4k_kernel<5>, grid, block, smem, s, ov, a);
        case 6: return launch_kernel(xq_tc_q4k_kernel<6>, grid, block, smem, s, ov, a);
        case 7: return launch_kernel(xq_tc_q4k_kernel<7>, grid, block, smem, s, ov, a);
        case 8: return launch_kernel(xq_tc_q4k_kernel<8>, grid, block, smem, s, ov, a);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t configure_matvec_q4k_tc(int smem_optin) {
    const void *k[4] = {(const void *)xq_tc_q4k_kernel<5>, (const void *)xq_tc_q4k_kernel<6>,
                        (const void *)xq_tc_q4k_kernel<7>, (const void *)xq_tc_q4k_kernel<8>};
    for (const void *f : k) {
        const cudaError_t e =
            cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace xq
