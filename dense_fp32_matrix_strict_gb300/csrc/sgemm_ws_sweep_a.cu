// Tuning alternative of the 128 x 128 x 32 family: scalar FFMA outer product
// (the packed FFMA2 form is the default).
#include "kernels.h"

namespace sg {

static const KernelFamily kFamily = SG_FAMILY("ws_128x128x32_s4_ffma", 128, 128, 4, 0, 0, 0);

const KernelFamily* sweep_family_a() { return &kFamily; }

}  // namespace sg
