// Tuning alternative: the default 128 x 128 x 32 kernel with a
// 3-stage ring (96 KB of shared memory).
#include "kernels.h"

namespace sg {

static const KernelFamily kFamily = SG_FAMILY("ws_128x128x32_s3", 128, 128, 3, 3, 1, 0);

const KernelFamily* sweep_family_d() { return &kFamily; }

}  // namespace sg
