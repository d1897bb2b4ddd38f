// gemm_tc_f16.cu -- the tcgen05 GEMM with IEEE-half operands and outputs (the
// fp16 mixed-precision step of the dl-scratch page, 3.4): the kernel of
// gemm_tc_kernel.cuh instantiated with F16, which sets the MMA instruction
// descriptor's operand format to f16 and converts the epilogue's loads and
// stores through half; accumulation stays fp32.  Kept in its own translation
// unit so that both sets of instantiations compile in parallel.
#include "gemm_tc_kernel.cuh"

namespace tt {
namespace tc {

bool launch_tc_f16(int BN, bool a_mn, bool b_mn, bool pair, const Launch& L, const Plan& pl,
                   const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& md, const CUtensorMap& mx) {
#define TCH(BN_, AM_, BM_)                                                     \
    (pair ? launch_tc<BN_, AM_, BM_, true, true>(L, pl, ma, mb, md, mx)        \
          : launch_tc<BN_, AM_, BM_, false, true>(L, pl, ma, mb, md, mx))
    if (BN == 256) {
        if (!a_mn && !b_mn) return TCH(256, false, false);
        if (!a_mn) return TCH(256, false, true);
        return TCH(256, true, true);
    }
    if (BN == 192) return a_mn && b_mn && !pair && launch_tc<192, true, true, false, true>(L, pl, ma, mb, md, mx);
    if (!a_mn && !b_mn) return TCH(128, false, false);
    if (!a_mn) return TCH(128, false, true);
    return TCH(128, true, true);
#undef TCH
}

}  // namespace tc
}  // namespace tt
