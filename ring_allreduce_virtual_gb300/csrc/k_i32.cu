// Kernels of element type int32_t: 4 reductions x 3 protocols.
#include "vr_ring_generic.cuh"

VR_INSTANTIATE_GENERIC(vrGetGeneric_i32, int32_t)
