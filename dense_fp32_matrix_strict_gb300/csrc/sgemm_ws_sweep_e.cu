// Tuning alternative: the default 128 x 128 x 32 kernel with a
// 6-stage ring (192 KB of shared memory).
#include "kernels.h"

namespace sg {

static const KernelFamily kFamily = SG_FAMILY("ws_128x128x32_s6", 128, 128, 6, 3, 1, 0);

const KernelFamily* sweep_family_e() { return &kFamily; }

}  // namespace sg
