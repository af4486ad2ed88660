// Tuning alternative: a 64 x 128 CTA tile (4 consumer warps), sized
// for two CTAs per SM.
#include "kernels.h"

namespace sg {

static const KernelFamily kFamily = SG_FAMILY("ws_64x128x32_s4", 64, 128, 4, 3, 1, 0);

const KernelFamily* sweep_family_g() { return &kFamily; }

}  // namespace sg
