// gemv_q8_0.cu - grouped GEMV kernels for the MOE_Q8_0 weight format (one translation unit per format so
// the formats compile in parallel).
#include "gemv.cuh"

MOE_FORMAT_TU(q8_0, MOE_Q8_0)
