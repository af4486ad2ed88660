// The 128 x 128 x 32 CTA-tile family (8 consumer warps, 4-stage ring,
// 128 KB of shared memory, packed FFMA2 outer product with the column pairs
// outer, early probe of the next stage): the kernel for every problem with
// enough work to fill the GPU. It also has the mode that makes the transposed
// copy of a row-major A itself (Cfg::FUSED).
#include "kernels.h"

namespace sg {

static const KernelFamily kFamily = SG_FAMILY_FUSED("ws_128x128x32_s4", 128, 128, 4, 3, 1, 0);

const KernelFamily* family_128x128() { return &kFamily; }

}  // namespace sg
