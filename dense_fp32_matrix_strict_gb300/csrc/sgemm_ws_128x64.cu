// The 128 x 128 x 32 kernel's 128 x 64 CTA-tile sibling (4 consumer warps,
// 4-stage ring, 64 KB of shared memory, two CTAs per SM): "auto" takes it,
// with whole tiles only, for problems whose 128 x 64 grid fits in about one
// wave while the 128 x 128 grid would leave SMs idle.
#include "kernels.h"

namespace sg {

static const KernelFamily kFamily = SG_FAMILY("ws_128x64x32_s4", 128, 64, 4, 3, 1, 0);

const KernelFamily* family_128x64() { return &kFamily; }

}  // namespace sg
