// Kernels of element type int64_t: 4 reductions x 3 protocols.
#include "vr_ring_generic.cuh"

VR_INSTANTIATE_GENERIC(vrGetGeneric_i64, int64_t)
