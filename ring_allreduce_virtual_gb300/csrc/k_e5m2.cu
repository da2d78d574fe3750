// Kernels of the 8-bit floating type E5M2: global-memory FIFOs and warp rings
// (4 reductions x 3 protocols), cluster rings (4 reductions, Simple
// protocol), the double-binary-tree AllReduce and the ring-walk calibration
// fold (4 reductions each).
#include "vr_ring_generic.cuh"
#include "vr_ring_walk.cuh"
#include "vr_ring_warp.cuh"
#include "vr_tree_warp.cuh"

VR_INSTANTIATE_GENERIC(vrGetGeneric_e5m2, vr::vr_fp8_e5m2)
VR_INSTANTIATE_WARP(vrGetWarp_e5m2, vr::vr_fp8_e5m2)
VR_INSTANTIATE_WALK(vrGetWalk_e5m2, vr::vr_fp8_e5m2)
VR_INSTANTIATE_TREE(vrGetTree_e5m2, vr::vr_fp8_e5m2)
