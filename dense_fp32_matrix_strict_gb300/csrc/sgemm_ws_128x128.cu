// Instantiations of the warp-specialised kernel with a 128 x 128 x 32 CTA tile
// (8 consumer warps) and a 4-stage ring (128 KB of shared memory).
#include "kernels.h"

namespace sg {

static const KernelEntry kTable[4] = {
    SG_WS_ENTRY("ws_128x128x32_s4_Atma_Btma", 128, 128, 4, LOAD_TMA, LOAD_TMA),
    SG_WS_ENTRY("ws_128x128x32_s4_Acp_Btma", 128, 128, 4, LOAD_CPASYNC, LOAD_TMA),
    SG_WS_ENTRY("ws_128x128x32_s4_Atma_Bcp", 128, 128, 4, LOAD_TMA, LOAD_CPASYNC),
    SG_WS_ENTRY("ws_128x128x32_s4_Acp_Bcp", 128, 128, 4, LOAD_CPASYNC, LOAD_CPASYNC),
};

const KernelEntry* ws_kernels_128x128() { return kTable; }

}  // namespace sg
