// Tuning alternative: the default 128 x 128 x 32 kernel reading a lane's
// row-major A values as float2 pairs of k-steps (ALOAD 2 in Cfg).
#include "kernels.h"

namespace sg {

static const KernelFamily kFamily = SG_FAMILY_A("ws_128x128x32_s4_a2", 128, 128, 4, 3, 1, 0, 2);

const KernelFamily* sweep_family_i() { return &kFamily; }

}  // namespace sg
