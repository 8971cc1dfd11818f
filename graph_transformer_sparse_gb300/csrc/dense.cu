// dense.cu -- dense-block attention path (placeholder until the tensor-core
// kernel lands: reports no support, so complete blocks take the row kernels).
#include "dense.cuh"

namespace gt {

bool dense_supported(int, int, gtattn_dtype, const void*, const void*, const void*, const void*) {
    return false;
}

gtattn_status launch_dense(const int2*, int, const void*, const void*, const void*, void*, int, int,
                           float, cudaStream_t) {
    return GTATTN_ERR_UNSUPPORTED;
}

}  // namespace gt
