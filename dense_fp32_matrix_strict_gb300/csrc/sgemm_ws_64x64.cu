// The 64 x 64 x 32 CTA-tile family (2 consumer warps, 4-stage ring, 64 KB of
// shared memory, the same outer product and stage probe as 128 x 128), for
// problems too small to give every SM a 128 x 128 tile.
#include "kernels.h"

namespace sg {

static const KernelFamily kFamily = SG_FAMILY("ws_64x64x32_s4", 64, 64, 4, 3, 1, 0);

const KernelFamily* family_64x64() { return &kFamily; }

}  // namespace sg
