// gemv_cb3.cu - grouped GEMV kernels for the MOE_CB3 weight format (one translation unit per format so
// the formats compile in parallel).
#include "gemv.cuh"

MOE_FORMAT_TU(cb3, MOE_CB3)
