// Fused layer kernel, cb3 gate/up weights (down NL4 or Q8_0).
#include "layer.cuh"

MOE_LAYER_TU(cb3, MOE_CB3)
