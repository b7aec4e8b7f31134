// sweep_variants_c.cu -- configurations of the persistent TMA/FFMA kernel with
// two CTAs per SM (TwoPerSMConfig): variant 12 (128x128 tiles, 48-deep slabs
// in two stages) and 13 (128x128, 32-deep slabs in three stages), 8 consumer
// warps each.  The two CTAs of an SM run their tiles independently, so one's
// epilogue overlaps the other's main loop.  Compiled on its own so the
// library's translation units build in parallel.
#include "variant.cuh"

namespace {

using sg::ISSUE_LAST_WARP;
using sg::MICRO_FFMA2;
using sgv::make_variant;

const sgv::Variant kTable[] = {
    // variant 12
    make_variant<sg::TwoPerSMConfig<
        sg::TileConfig<128, 128, 48, 2, 4, 2, 8, 8, MICRO_FFMA2, ISSUE_LAST_WARP>>>(
        "ffma2 tile=128x128x48 stages=2 warps=8 issuer=last_warp thread=8x8 stream_k ctas_per_sm=2",
        true),
    // variant 13
    make_variant<sg::TwoPerSMConfig<
        sg::TileConfig<128, 128, 32, 3, 4, 2, 8, 8, MICRO_FFMA2, ISSUE_LAST_WARP>>>(
        "ffma2 tile=128x128x32 stages=3 warps=8 issuer=last_warp thread=8x8 stream_k ctas_per_sm=2",
        true),
};

cudaError_t error_word(unsigned *v, bool clear) { return sgv::unit_error_word(v, clear); }

}  // namespace

sgv::VariantTable sgv::sweep_variants_c() {
    return {kTable, int(sizeof(kTable) / sizeof(kTable[0])), &error_word};
}
