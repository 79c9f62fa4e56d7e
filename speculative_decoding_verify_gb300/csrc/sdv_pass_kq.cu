// sdv_pass_kq.cu - the one-launch verify pass over a K-quant stack (Q4_K projections, Q4_K or Q6_K down
// projections, Q8_0 head) with greedy acceptance, compiled in its own translation unit.
#include "sdv_qmatmul.cuh"

namespace sdv {

cudaError_t pass_launch_kq(const QmmArgs *phases, int n_phases, uint32_t *ctr, uint64_t *trace, int nt, size_t smem,
                           int grid, cudaStream_t s) {
    return pass_launch_kernel(nt == 1 ? pass_kernel<1, false, true> : pass_kernel<2, false, true>, phases, n_phases,
                              ctr, trace, smem, grid, s);
}

}  // namespace sdv
