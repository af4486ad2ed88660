// Tuning alternative of the 128 x 128 x 32 family: 4 stages, lane map 0,
// cross-stage fragment prefetch 0, FMA form 0 (see Cfg).
#include "kernels.h"

namespace sg {

static const KernelFamily kFamily =
    SG_FAMILY("ws_128x128x32_s4_x0_f0", 128, 128, 4, 0, 0, 0, 0);

const KernelFamily* sweep_family_a() { return &kFamily; }

}  // namespace sg
