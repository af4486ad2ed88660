// Tuning alternative of the 128 x 128 x 32 family: FFMA2 with the rows outer
// and no early stage probe (FORDER 2, EARLY 0 in Cfg).
#include "kernels.h"

namespace sg {

static const KernelFamily kFamily = SG_FAMILY("ws_128x128x32_s4_f2", 128, 128, 4, 2, 0, 0);

const KernelFamily* sweep_family_b() { return &kFamily; }

}  // namespace sg
