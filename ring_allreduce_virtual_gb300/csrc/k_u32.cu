// Kernels of element type uint32_t: global-memory FIFOs and warp rings (4
// reductions x 3 protocols), the double-binary-tree AllReduce and the
// ring-walk calibration fold (4 reductions each).
#include "vr_ring_generic.cuh"
#include "vr_ring_walk.cuh"
#include "vr_ring_warp.cuh"
#include "vr_tree_warp.cuh"

VR_INSTANTIATE_GENERIC(vrGetGeneric_u32, uint32_t)
VR_INSTANTIATE_WARP(vrGetWarp_u32, uint32_t)
VR_INSTANTIATE_WALK(vrGetWalk_u32, uint32_t)
VR_INSTANTIATE_TREE(vrGetTree_u32, uint32_t)
