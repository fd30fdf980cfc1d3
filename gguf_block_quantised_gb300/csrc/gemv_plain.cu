// gemv_plain.cu -- decode matvec and expert matvec kernels for plain F32, F16 and BF16 weights
// (fp32 activations only).
#include "gemv_launch.cuh"

QMV_GEMV_INSTANTIATE(QMV_F32, qmv_gemv_f32)
QMV_MOE_INSTANTIATE(QMV_F32, qmv_moe_f32)
QMV_GEMV_INSTANTIATE(QMV_F16, qmv_gemv_f16)
QMV_MOE_INSTANTIATE(QMV_F16, qmv_moe_f16)
QMV_GEMV_INSTANTIATE(QMV_BF16, qmv_gemv_bf16)
QMV_MOE_INSTANTIATE(QMV_BF16, qmv_moe_bf16)
