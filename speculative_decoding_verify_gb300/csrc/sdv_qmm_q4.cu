// sdv_qmm_q4.cu - instantiations of the multi-position matmul for
// qtype SD_Q4_32, gate|up pairing 0 (one translation unit per variant so
// the build compiles them in parallel).
#include "sdv_qmatmul.cuh"

namespace sdv {

template <>
cudaError_t qmm_dispatch<SD_Q4_32, 0>(QmmArgs a, QmmPlan &p, cudaStream_t s) {
    const int MT = a.M <= 8 ? a.M : 16;
    uint32_t o_ring, o_act, o_meta, o_red;
    const size_t smem = plan_smem(p, MT, 0 != 0, o_ring, o_act, o_meta, o_red);
    a.SB = p.SB;
    a.NS = p.NS;
    a.off_ring = o_ring;
    a.off_act = o_act;
    a.off_meta = o_meta;
    a.off_red = o_red;
    switch (a.M) {
        case 1: return qmm_launch<SD_Q4_32, 0, 1, true>(a, smem, s);
        case 2: return qmm_launch<SD_Q4_32, 0, 2, true>(a, smem, s);
        case 3: return qmm_launch<SD_Q4_32, 0, 3, true>(a, smem, s);
        case 4: return qmm_launch<SD_Q4_32, 0, 4, true>(a, smem, s);
        case 5: return qmm_launch<SD_Q4_32, 0, 5, true>(a, smem, s);
        case 6: return qmm_launch<SD_Q4_32, 0, 6, true>(a, smem, s);
        case 7: return qmm_launch<SD_Q4_32, 0, 7, true>(a, smem, s);
        case 8: return qmm_launch<SD_Q4_32, 0, 8, true>(a, smem, s);
        default: return qmm_launch<SD_Q4_32, 0, 16, false>(a, smem, s);
    }
}

}  // namespace sdv
