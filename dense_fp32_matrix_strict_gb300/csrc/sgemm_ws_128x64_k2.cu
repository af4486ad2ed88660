// A 128 x 64 CTA tile whose eight consumer warps form two k-groups of four
// (KSPLIT in Cfg): each group takes half of every stage's k, and the groups'
// sums are added in group order before the epilogue. One CTA per SM. "auto"
// takes it, with whole tiles, for problems whose 128 x 64 grid fills about
// one wave (1024^3 on GB300: 47.1 us against 51.2 us for the two-CTA 128 x 64
// tile).
#include "kernels.h"

namespace sg {

static const KernelFamily kFamily = SG_FAMILY_K("ws_128x64x32_s4_k2", 128, 64, 4, 2);

const KernelFamily* family_128x64_k2() { return &kFamily; }

}  // namespace sg
