// Kernels of element type double: 4 reductions x 3 protocols.
#include "vr_ring_generic.cuh"

VR_INSTANTIATE_GENERIC(vrGetGeneric_f64, double)
