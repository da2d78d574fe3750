// Kernels of element type __nv_bfloat16: 4 reductions x 3 protocols.
#include "vr_ring_generic.cuh"

VR_INSTANTIATE_GENERIC(vrGetGeneric_bf16, __nv_bfloat16)
