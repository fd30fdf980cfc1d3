// gemv_mxfp4.cu -- decode matvec kernels for MXFP4 weights (one translation unit
// per format so the kernels compile in parallel).
#include "gemv_launch.cuh"

QMV_GEMV_INSTANTIATE(QMV_MXFP4, qmv_gemv_mxfp4)
