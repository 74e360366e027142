// qmm_lib.cu -- the single translation unit of libqmm.so (the kernels share
// the device error word, so they are compiled together).
#include "qmm_api.cu"
#include "quantize.cu"
#include "gemv.cu"
#include "gemv_rows.cu"
#include "gemm.cu"
#include "q6k.cu"
#include "fp8.cu"
#include "kquant.cu"
#include "sbrows.cu"
#include "static_scratch.cu"
