// The list of tuning alternatives (one translation unit each).
#include "kernels.h"

namespace sg {

const KernelFamily* sweep_family_a();
const KernelFamily* sweep_family_b();
const KernelFamily* sweep_family_c();
const KernelFamily* sweep_family_d();
const KernelFamily* sweep_family_e();
const KernelFamily* sweep_family_g();
const KernelFamily* sweep_family_h();
const KernelFamily* sweep_family_i();
const KernelFamily* sweep_family_j();
const KernelFamily* sweep_family_l();

const KernelFamily* const* sweep_families(int* count) {
#ifdef SGEMM_DEBUG
    // The debug build compiles only the families "auto" chooses between.
    *count = 0;
    return nullptr;
#endif
    static const KernelFamily* const list[] = {sweep_family_a(), sweep_family_b(), sweep_family_c(),
                                               sweep_family_d(), sweep_family_e(), sweep_family_g(),
                                               sweep_family_h(), sweep_family_i(),
                                               sweep_family_j(), sweep_family_l()};
    *count = static_cast<int>(sizeof(list) / sizeof(list[0]));
    return list;
}

}  // namespace sg
