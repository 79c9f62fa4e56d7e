// sdv_qmm_q4.cu - instantiations of the multi-position matmul for
// qtype SD_Q4_32, gate|up pairing 0 (one translation unit per variant so
// the build compiles them in parallel).
#include "sdv_qmatmul.cuh"

namespace sdv {

template <>
cudaError_t qmm_dispatch<SD_Q4_32, 0>(QmmArgs a, QmmPlan &p, cudaStream_t s) {
    const int NT = a.M <= 8 ? 1 : 2;
    uint32_t o_ring, o_act, o_meta, o_red, o_tmp;
    const size_t smem = plan_smem(p, NT, 0 != 0, o_ring, o_act, o_meta, o_red, o_tmp);
    a.SB = p.SB;
    a.NS = p.NS;
    a.off_ring = o_ring;
    a.off_act = o_act;
    a.off_meta = o_meta;
    a.off_red = o_red;
    a.off_tmp = o_tmp;
    a.stage_stride = static_cast<uint32_t>(p.SB) * p.step_bytes;
    a.kind = KIND_MATMUL;
    return NT == 1 ? qmm_launch<SD_Q4_32, 0, 1>(a, smem, s) : qmm_launch<SD_Q4_32, 0, 2>(a, smem, s);
}

}  // namespace sdv
