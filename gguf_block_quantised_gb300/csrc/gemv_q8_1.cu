// gemv_q8_1.cu -- decode matvec and expert matvec kernels for Q8_1 weights (one translation unit
// per format so the kernels compile in parallel).
#include "gemv_launch.cuh"

QMV_GEMV_INSTANTIATE(QMV_Q8_1, qmv_gemv_q8_1)
QMV_MOE_INSTANTIATE(QMV_Q8_1, qmv_moe_q8_1)
