// qmm_gemm_affine.cu -- instances of the tensor-core GEMM for the affine
// variant (group 64; weight operand in tensor or shared memory).
#include "qmm_gemm.cuh"

namespace qmm {

cudaError_t launch_gemm_affine(const LaunchCtx& c, const CUtensorMap& map, const GemmShape& sh,
                               const uint8_t* blob, const float* gsum, float* Y, bool a_in_smem)
{
    const int half = sh.m_tile / 2;
    if (a_in_smem) {
        if (half <= 16) return run_gemm<1, 64, false, false, 32, 8>(c, map, sh, blob, gsum, Y, nullptr);
        if (half <= 32) return run_gemm<1, 64, false, false, 32>(c, map, sh, blob, gsum, Y, nullptr);
        if (half <= 48) return run_gemm<1, 64, false, false, 48>(c, map, sh, blob, gsum, Y, nullptr);
        return run_gemm<1, 64, false, false, 64>(c, map, sh, blob, gsum, Y, nullptr);
    }
    if (half <= 16) return run_gemm<1, 64, true, false, 32, 8>(c, map, sh, blob, gsum, Y, nullptr);
    if (half <= 32) return run_gemm<1, 64, true, false, 32>(c, map, sh, blob, gsum, Y, nullptr);
    if (half <= 48) return run_gemm<1, 64, true, false, 48>(c, map, sh, blob, gsum, Y, nullptr);
    return run_gemm<1, 64, true, false, 64>(c, map, sh, blob, gsum, Y, nullptr);
}

}  // namespace qmm
