// sdv_pass_sample.cu - the one-launch verify pass ending in rejection-sampling acceptance (its own
// translation unit, compiled in parallel with the greedy pass).
#include "sdv_qmatmul.cuh"

namespace sdv {

cudaError_t pass_launch_sampling(const QmmArgs *phases, int n_phases, uint32_t *ctr, uint64_t *trace, int nt,
                                 size_t smem, int grid, cudaStream_t s) {
    return pass_launch_kernel(nt == 1 ? pass_kernel<1, true> : pass_kernel<2, true>, phases, n_phases, ctr, trace,
                              smem, grid, s);
}

}  // namespace sdv
