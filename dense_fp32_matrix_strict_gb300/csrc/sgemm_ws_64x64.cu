// Instantiations of the warp-specialised kernel with a 64 x 64 x 32 CTA tile
// (2 consumer warps) and a 4-stage ring (64 KB of shared memory), for
// problems too small to give every SM a 128 x 128 tile.
#include "kernels.h"

namespace sg {

static const KernelEntry kTable[4] = {
    SG_WS_ENTRY("ws_64x64x32_s4_Atma_Btma", 64, 64, 4, LOAD_TMA, LOAD_TMA),
    SG_WS_ENTRY("ws_64x64x32_s4_Acp_Btma", 64, 64, 4, LOAD_CPASYNC, LOAD_TMA),
    SG_WS_ENTRY("ws_64x64x32_s4_Atma_Bcp", 64, 64, 4, LOAD_TMA, LOAD_CPASYNC),
    SG_WS_ENTRY("ws_64x64x32_s4_Acp_Bcp", 64, 64, 4, LOAD_CPASYNC, LOAD_CPASYNC),
};

const KernelEntry* ws_kernels_64x64() { return kTable; }

}  // namespace sg
