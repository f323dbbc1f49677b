// Fused layer kernel, nl4 gate/up weights (down NL4 or Q8_0).
#include "layer.cuh"

MOE_LAYER_TU(nl4, MOE_NL4)
