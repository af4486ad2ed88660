// Tuning alternative: a 128 x 64 CTA tile with two k-groups of four consumer warps (KSPLIT in Cfg): more warps per SM for problems
// with few tiles, the k-groups' sums added in group order.
#include "kernels.h"

namespace sg {

static const KernelFamily kFamily = SG_FAMILY_K("ws_128x64x32_s4_k2", 128, 64, 4, 2);

const KernelFamily* sweep_family_k() { return &kFamily; }

}  // namespace sg
