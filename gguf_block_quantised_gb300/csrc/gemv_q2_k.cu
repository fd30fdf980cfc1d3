// gemv_q2_k.cu -- decode matvec and expert matvec kernels for Q2_K weights (one translation unit
// per format so the kernels compile in parallel).
#include "gemv_launch.cuh"

QMV_GEMV_INSTANTIATE(QMV_Q2_K, qmv_gemv_q2_k)
QMV_MOE_INSTANTIATE(QMV_Q2_K, qmv_moe_q2_k)
