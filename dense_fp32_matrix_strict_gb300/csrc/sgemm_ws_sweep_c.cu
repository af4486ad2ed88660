// Tuning alternative of the 128 x 128 x 32 family: lane map 1 (see Cfg) with
// the default outer product and stage probe.
#include "kernels.h"

namespace sg {

static const KernelFamily kFamily = SG_FAMILY("ws_128x128x32_s4_l1", 128, 128, 4, 3, 1, 1);

const KernelFamily* sweep_family_c() { return &kFamily; }

}  // namespace sg
