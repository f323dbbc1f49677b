// gemv_q4b.cu - grouped GEMV kernels for the MOE_Q4B weight format (one translation unit per format so
// the formats compile in parallel).
#include "gemv.cuh"

MOE_FORMAT_TU(q4b, MOE_Q4B)
