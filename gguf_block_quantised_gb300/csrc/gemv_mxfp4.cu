// gemv_mxfp4.cu -- decode matvec and expert matvec kernels for MXFP4 weights (one translation unit
// per format so the kernels compile in parallel).
#include "gemv_launch.cuh"

QMV_GEMV_INSTANTIATE(QMV_MXFP4, qmv_gemv_mxfp4)
QMV_MOE_INSTANTIATE(QMV_MXFP4, qmv_moe_mxfp4)
