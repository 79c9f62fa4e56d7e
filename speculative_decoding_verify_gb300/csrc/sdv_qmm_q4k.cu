// sdv_qmm_q4k.cu - instantiation of the multi-position matmul for qtype SD_Q4_K, gate|up pairing 0
// (one translation unit per variant so the build compiles them in parallel).
#include "sdv_qmatmul.cuh"

namespace sdv {

template cudaError_t qmm_dispatch<SD_Q4_K, 0>(QmmArgs, QmmPlan &, cudaStream_t);

}  // namespace sdv
