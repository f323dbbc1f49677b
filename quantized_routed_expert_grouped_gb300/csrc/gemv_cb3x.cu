// gemv_cb3x.cu - grouped GEMV kernels for the MOE_CB3X transcoded slot layout (one translation unit per
// format so the formats compile in parallel).
#include "gemv.cuh"

MOE_FORMAT_TU(cb3x, MOE_CB3X)
