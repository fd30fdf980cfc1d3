// gemv_q5_0.cu -- decode matvec and expert matvec kernels for Q5_0 weights (one translation unit
// per format so the kernels compile in parallel).
#include "gemv_launch.cuh"

QMV_GEMV_INSTANTIATE(QMV_Q5_0, qmv_gemv_q5_0)
QMV_MOE_INSTANTIATE(QMV_Q5_0, qmv_moe_q5_0)
