// sdv_qmm_q4kp.cu - instantiation of the multi-position matmul for qtype SD_Q4_K, gate|up pairing 1
// (one translation unit per variant so the build compiles them in parallel).
#include "sdv_qmatmul.cuh"

namespace sdv {

template cudaError_t qmm_dispatch<SD_Q4_K, 1>(QmmArgs, QmmPlan &, cudaStream_t);

}  // namespace sdv
