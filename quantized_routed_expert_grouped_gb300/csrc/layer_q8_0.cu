// Fused layer kernel, q8_0 gate/up weights (down NL4 or Q8_0).
#include "layer.cuh"

MOE_LAYER_TU(q8_0, MOE_Q8_0)
