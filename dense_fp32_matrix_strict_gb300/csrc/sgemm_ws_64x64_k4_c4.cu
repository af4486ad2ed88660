// The 64 x 64 tile in four k-groups with its CTAs in thread-block clusters
// of 4 (Cfg::CS): the 4 CTAs of a cluster share one tile, each taking 1/4
// of its k-tiles, and the partial sums meet in the first CTA's shared
// memory (distributed shared memory) instead of global memory and a second
// kernel. "auto" takes it for problems whose tiles x 4 still fit in one
// wave, so that more SMs work on a few tiles.
#include "kernels.h"

namespace sg {

static const KernelFamily kFamily = SG_FAMILY_KC("ws_64x64x32_s4_k4_c4", 64, 64, 4, 4, 4);

const KernelFamily* family_64x64_k4_c4() { return &kFamily; }

}  // namespace sg
