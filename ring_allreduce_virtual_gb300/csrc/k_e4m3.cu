// Kernels of the 8-bit floating type E4M3: global-memory FIFOs and warp rings
// (4 reductions x 3 protocols), cluster rings (4 reductions, Simple
// protocol), the double-binary-tree AllReduce and the ring-walk calibration
// fold (4 reductions each).
#include "vr_ring_generic.cuh"
#include "vr_ring_walk.cuh"
#include "vr_ring_warp.cuh"
#include "vr_tree_warp.cuh"

VR_INSTANTIATE_GENERIC(vrGetGeneric_e4m3, vr::vr_fp8_e4m3)
VR_INSTANTIATE_WARP(vrGetWarp_e4m3, vr::vr_fp8_e4m3)
VR_INSTANTIATE_WALK(vrGetWalk_e4m3, vr::vr_fp8_e4m3)
VR_INSTANTIATE_TREE(vrGetTree_e4m3, vr::vr_fp8_e4m3)
