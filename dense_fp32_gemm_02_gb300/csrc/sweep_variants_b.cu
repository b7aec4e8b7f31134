// sweep_variants_b.cu -- configurations of the persistent TMA/FFMA kernel kept
// for tile-configuration sweeps and as evidence for the design choices:
// variant 7 (128x192 tiles, last-warp issuer), 8 (192x128 with a producer
// warpgroup), 9 and 10 (128x128x48 with a producer warpgroup, packed FP32x2
// or scalar FMA) and 11 (a 16x8 thread tile).  Compiled on its own so the
// library's translation units build in parallel.
#include "variant.cuh"

namespace {

using sg::ISSUE_LAST_WARP;
using sg::ISSUE_PRODUCER_WG;
using sg::MICRO_FFMA;
using sg::MICRO_FFMA2;
using sgv::make_variant;

const sgv::Variant kTable[] = {
    // variant 7
    make_variant<sg::TileConfig<128, 192, 64, 2, 4, 3, 8, 8, MICRO_FFMA2, ISSUE_LAST_WARP>>(
        "ffma2 tile=128x192x64 stages=2 warps=12 issuer=last_warp thread=8x8 stream_k", true),
    // variant 8
    make_variant<sg::TileConfig<192, 128, 64, 2, 6, 2, 8, 8, MICRO_FFMA2, ISSUE_PRODUCER_WG>>(
        "ffma2 tile=192x128x64 stages=2 warps=12+producer_wg thread=8x8 stream_k", true),
    // variant 9
    make_variant<sg::TileConfig<128, 128, 48, 4, 4, 2, 8, 8, MICRO_FFMA2, ISSUE_PRODUCER_WG>>(
        "ffma2 tile=128x128x48 stages=4 warps=8+producer_wg thread=8x8 stream_k", true),
    // variant 10
    make_variant<sg::TileConfig<128, 128, 48, 4, 4, 2, 8, 8, MICRO_FFMA, ISSUE_PRODUCER_WG>>(
        "ffma tile=128x128x48 stages=4 warps=8+producer_wg thread=8x8 stream_k", true),
    // variant 11
    make_variant<sg::TileConfig<256, 128, 32, 4, 4, 2, 16, 8, MICRO_FFMA2, ISSUE_PRODUCER_WG>>(
        "ffma2 tile=256x128x32 stages=4 warps=8+producer_wg thread=16x8 stream_k", true),
};

cudaError_t error_word(unsigned *v, bool clear) { return sgv::unit_error_word(v, clear); }

}  // namespace

sgv::VariantTable sgv::sweep_variants_b() {
    return {kTable, int(sizeof(kTable) / sizeof(kTable[0])), &error_word};
}
