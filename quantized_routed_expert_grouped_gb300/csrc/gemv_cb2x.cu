// gemv_cb2x.cu - grouped GEMV kernels for the MOE_CB2X transcoded slot layout (one translation unit per
// format so the formats compile in parallel).
#include "gemv.cuh"

MOE_FORMAT_TU(cb2x, MOE_CB2X)
