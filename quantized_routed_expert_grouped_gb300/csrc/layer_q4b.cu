// Fused layer kernel, q4b gate/up weights (down NL4 or Q8_0).
#include "layer.cuh"

MOE_LAYER_TU(q4b, MOE_Q4B)
