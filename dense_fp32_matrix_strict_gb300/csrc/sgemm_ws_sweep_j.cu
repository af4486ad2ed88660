// Tuning alternative: a 128 x 128 x 32 CTA tile with four consumer warps of
// 32 x 128 (8 x 16 outputs a lane, twice the multiply-adds per shared load;
// one consumer warp per scheduler, up to 255 registers).
#include "kernels.h"

namespace sg {

static const KernelFamily kFamily = SG_FAMILY_T("ws_128x128x32_s4_w4", 128, 128, 4, 3, 1, 0, 16);

const KernelFamily* sweep_family_j() { return &kFamily; }

}  // namespace sg
