// Fused layer kernel, cb2 gate/up weights (down NL4 or Q8_0).
#include "layer.cuh"

MOE_LAYER_TU(cb2, MOE_CB2)
