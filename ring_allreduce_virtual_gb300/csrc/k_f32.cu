// Kernels of element type float: 4 reductions x 3 protocols.
#include "vr_ring_generic.cuh"

VR_INSTANTIATE_GENERIC(vrGetGeneric_f32, float)
