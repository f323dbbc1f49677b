// gemv_cb2.cu - grouped GEMV kernels for the MOE_CB2 weight format (one translation unit per format so
// the formats compile in parallel).
#include "gemv.cuh"

MOE_FORMAT_TU(cb2, MOE_CB2)
