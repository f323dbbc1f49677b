// Fused layer kernel, cb3x gate/up weights (down NL4 or Q8_0).
#include "layer.cuh"

MOE_LAYER_TU(cb3x, MOE_CB3X)
