// Kernels of element type uint8_t: 4 reductions x 3 protocols.
#include "vr_ring_generic.cuh"

VR_INSTANTIATE_GENERIC(vrGetGeneric_u8, uint8_t)
