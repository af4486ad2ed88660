// A 64 x 64 CTA tile whose eight consumer warps form four k-groups of two
// (KSPLIT in Cfg): each group takes a quarter of every stage's k, and the
// groups' sums are added in group order before the epilogue. One CTA per SM.
// "auto" takes it for problems with few 128 x 128 tiles (256^3 on GB300:
// 12.9 us against 18.4 us for the plain 64 x 64 tile), with the stream-K
// tail when K is deep enough to pay for it.
#include "kernels.h"

namespace sg {

static const KernelFamily kFamily = SG_FAMILY_K("ws_64x64x32_s4_k4", 64, 64, 4, 4);

const KernelFamily* family_64x64_k4() { return &kFamily; }

}  // namespace sg
