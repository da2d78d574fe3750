// Latency kernels of element type __nv_bfloat16: the warp rings for calls that fit
// one pass of their rings (4 reductions x Simple and LL, one CTA or a cluster
// per ring), and for Simple calls of several passes on rings in one CTA.
#include "vr_ring_lat.cuh"

VR_INSTANTIATE_LAT(vrGetLat_bf16, __nv_bfloat16)
