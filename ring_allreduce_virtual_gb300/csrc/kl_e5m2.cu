// Latency kernels of element type vr::vr_fp8_e5m2: the warp rings for calls that fit
// one pass of their rings (4 reductions x Simple and LL, one CTA or a cluster
// per ring), and for Simple calls of several passes on rings in one CTA.
#include "vr_ring_lat.cuh"

VR_INSTANTIATE_LAT(vrGetLat_e5m2, vr::vr_fp8_e5m2)
