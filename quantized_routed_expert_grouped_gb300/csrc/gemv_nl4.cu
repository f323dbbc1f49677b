// gemv_nl4.cu - grouped GEMV kernels for the MOE_NL4 weight format (one translation unit per format so
// the formats compile in parallel).
#include "gemv.cuh"

MOE_FORMAT_TU(nl4, MOE_NL4)
