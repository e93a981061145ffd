// qmm_gemm_cq4.cu -- instances of the tensor-core GEMM for codebook 4-bit
// (CQ4) weights (group 64 and 128, weight operand in tensor or shared memory,
// result or raw-partials epilogue). Same tiles as the symmetric variant; the
// expand warps look the indices up in the matrix's 16 levels.
#include "qmm_gemm.cuh"

namespace qmm {

template <int GROUP>
static cudaError_t dispatch(const LaunchCtx& c, const CUtensorMap& map, const GemmShape& sh, const uint8_t* blob,
                            const float* sx, float* Y, int32_t* P, bool a_in_smem)
{
    const int half = sh.m_tile / 2;
    if (P) {
        if (a_in_smem) return run_gemm<2, GROUP, false, true, 64>(c, map, sh, blob, sx, Y, P);
        return run_gemm<2, GROUP, true, true, 64>(c, map, sh, blob, sx, Y, P);
    }
    if (a_in_smem) {
        if (half <= 16) return run_gemm<2, GROUP, false, false, 32, 8>(c, map, sh, blob, sx, Y, P);
        if (half <= 32) return run_gemm<2, GROUP, false, false, 32>(c, map, sh, blob, sx, Y, P);
        if (half <= 48) return run_gemm<2, GROUP, false, false, 48>(c, map, sh, blob, sx, Y, P);
        return run_gemm<2, GROUP, false, false, 64>(c, map, sh, blob, sx, Y, P);
    }
    if (half <= 16) return run_gemm<2, GROUP, true, false, 32, 8>(c, map, sh, blob, sx, Y, P);
    if (half <= 32) return run_gemm<2, GROUP, true, false, 32>(c, map, sh, blob, sx, Y, P);
    if (half <= 48) return run_gemm<2, GROUP, true, false, 48>(c, map, sh, blob, sx, Y, P);
    return run_gemm<2, GROUP, true, false, 64>(c, map, sh, blob, sx, Y, P);
}

cudaError_t launch_gemm_cq4(const LaunchCtx& c, int group, const CUtensorMap& map, const GemmShape& sh,
                            const uint8_t* blob, const float* sx, float* Y, int32_t* P, bool a_in_smem)
{
    if (group == 64) return dispatch<64>(c, map, sh, blob, sx, Y, P, a_in_smem);
    if (group == 128) return dispatch<128>(c, map, sh, blob, sx, Y, P, a_in_smem);
    return cudaErrorInvalidValue;
}

}  // namespace qmm
