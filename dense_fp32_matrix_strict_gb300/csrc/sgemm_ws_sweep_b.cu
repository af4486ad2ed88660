// Tuning alternative of the 128 x 128 x 32 family: a 6-stage ring (192 KB).
#include "kernels.h"

namespace sg {

static const KernelFamily kFamily = SG_FAMILY("ws_128x128x32_s6", 128, 128, 6, 2);

const KernelFamily* sweep_family_b() { return &kFamily; }

}  // namespace sg
