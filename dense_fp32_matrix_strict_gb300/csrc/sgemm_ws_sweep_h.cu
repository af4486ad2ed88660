// Tuning alternative: the default 128 x 128 x 32 kernel reading a lane's
// row-major A values one float per row and k-step (ALOAD 1 in Cfg).
#include "kernels.h"

namespace sg {

static const KernelFamily kFamily = SG_FAMILY_A("ws_128x128x32_s4_a1", 128, 128, 4, 3, 1, 0, 1);

const KernelFamily* sweep_family_h() { return &kFamily; }

}  // namespace sg
