// Fused layer kernel, cb2x gate/up weights (down NL4 or Q8_0).
#include "layer.cuh"

MOE_LAYER_TU(cb2x, MOE_CB2X)
