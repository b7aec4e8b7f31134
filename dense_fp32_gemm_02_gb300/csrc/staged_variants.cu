// staged_variants.cu -- the two default tile configurations of the persistent
// TMA/FFMA kernel (256x128 and 128x256) compiled with the staged epilogue
// (StagedEpilogueConfig): sgemm() takes them when the rows of C do not all
// start 16-byte aligned (ldc % 4 != 0, or C itself not 16-byte aligned), C_in
// is read and K is short (plain_variant in sgemm.cu).
// Compiled on its own so the library's translation units build in parallel.
#include "variant.cuh"

namespace {

using sg::ISSUE_LAST_WARP;
using sg::MICRO_FFMA2;
using sgv::make_variant;

const sgv::Variant kTable[] = {
    // STAGED_256x128: variant 0 with the staged epilogue
    make_variant<sg::StagedEpilogueConfig<
        sg::TileConfig<256, 128, 64, 2, 8, 2, 8, 8, MICRO_FFMA2, ISSUE_LAST_WARP>>>(
        "ffma2 tile=256x128x64 stages=2 warps=16 issuer=last_warp thread=8x8 stream_k "
        "staged_epilogue",
        true),
    // STAGED_128x256: variant 1 with the staged epilogue
    make_variant<sg::StagedEpilogueConfig<
        sg::TileConfig<128, 256, 64, 2, 4, 4, 8, 8, MICRO_FFMA2, ISSUE_LAST_WARP>>>(
        "ffma2 tile=128x256x64 stages=2 warps=16 issuer=last_warp thread=8x8 stream_k "
        "staged_epilogue",
        true),
};

cudaError_t error_word(unsigned *v, bool clear) { return sgv::unit_error_word(v, clear); }

}  // namespace

sgv::VariantTable sgv::staged_variants() {
    return {kTable, int(sizeof(kTable) / sizeof(kTable[0])), &error_word};
}
