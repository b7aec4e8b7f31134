// sweep_variants_a.cu -- configurations of the persistent TMA/FFMA kernel kept
// for tile-configuration sweeps and as evidence for the design choices:
// variant 2 (the thread-0 issuer), 4 (48-deep slabs in three stages), 5 and 6
// (128x192 tiles with a producer warpgroup, or with the thread-0 issuer).
// Compiled on its own so the library's translation units build in parallel.
#include "variant.cuh"

namespace {

using sg::ISSUE_LAST_WARP;
using sg::ISSUE_PRODUCER_WG;
using sg::ISSUE_THREAD0;
using sg::MICRO_FFMA2;
using sgv::make_variant;

const sgv::Variant kTable[] = {
    // variant 2
    make_variant<sg::TileConfig<256, 128, 64, 2, 8, 2, 8, 8, MICRO_FFMA2, ISSUE_THREAD0>>(
        "ffma2 tile=256x128x64 stages=2 warps=16 issuer=thread0 thread=8x8 stream_k", true),
    // variant 4
    make_variant<sg::TileConfig<256, 128, 48, 3, 8, 2, 8, 8, MICRO_FFMA2, ISSUE_LAST_WARP>>(
        "ffma2 tile=256x128x48 stages=3 warps=16 issuer=last_warp thread=8x8 stream_k", true),
    // variant 5
    make_variant<sg::TileConfig<128, 192, 64, 2, 4, 3, 8, 8, MICRO_FFMA2, ISSUE_PRODUCER_WG>>(
        "ffma2 tile=128x192x64 stages=2 warps=12+producer_wg thread=8x8 stream_k", true),
    // variant 6
    make_variant<sg::TileConfig<128, 192, 64, 2, 4, 3, 8, 8, MICRO_FFMA2, ISSUE_THREAD0>>(
        "ffma2 tile=128x192x64 stages=2 warps=12 issuer=thread0 thread=8x8 stream_k", true),
};

cudaError_t error_word(unsigned *v, bool clear) { return sgv::unit_error_word(v, clear); }

}  // namespace

sgv::VariantTable sgv::sweep_variants_a() {
    return {kTable, int(sizeof(kTable) / sizeof(kTable[0])), &error_word};
}
