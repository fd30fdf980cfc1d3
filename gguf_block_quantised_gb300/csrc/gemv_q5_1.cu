// gemv_q5_1.cu -- decode matvec and expert matvec kernels for Q5_1 weights (one translation unit
// per format so the kernels compile in parallel).
#include "gemv_launch.cuh"

QMV_GEMV_INSTANTIATE(QMV_Q5_1, qmv_gemv_q5_1)
QMV_MOE_INSTANTIATE(QMV_Q5_1, qmv_moe_q5_1)
