// Tuning alternative: a 64 x 64 CTA tile with four k-groups of two consumer warps (KSPLIT in Cfg): more warps per SM for problems
// with few tiles, the k-groups' sums added in group order.
#include "kernels.h"

namespace sg {

static const KernelFamily kFamily = SG_FAMILY_K("ws_64x64x32_s4_k4", 64, 64, 4, 4);

const KernelFamily* sweep_family_m() { return &kFamily; }

}  // namespace sg
