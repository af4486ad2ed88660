// Tuning alternative of the 128 x 128 x 32 family: 6 stages, lane map 0,
// cross-stage fragment prefetch 0, FMA form 2 (see Cfg).
#include "kernels.h"

namespace sg {

static const KernelFamily kFamily =
    SG_FAMILY("ws_128x128x32_s6_x0_f2", 128, 128, 6, 0, 0, 2, 0);

const KernelFamily* sweep_family_b() { return &kFamily; }

}  // namespace sg
