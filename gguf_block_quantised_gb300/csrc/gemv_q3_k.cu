// gemv_q3_k.cu -- decode matvec and expert matvec kernels for Q3_K weights (one translation unit
// per format so the kernels compile in parallel).
#include "gemv_launch.cuh"

QMV_GEMV_INSTANTIATE(QMV_Q3_K, qmv_gemv_q3_k)
QMV_MOE_INSTANTIATE(QMV_Q3_K, qmv_moe_q3_k)
