// extra_variants.cu -- the default 256x128x64 configuration of the persistent
// TMA/FFMA kernel compiled three more times: with the batch coordinate (3-D
// tensor maps) and the fused bias/activation epilogue, for batched calls of
// sgemm_ex; with the fused epilogue alone (2-D maps), for one GEMM with a bias
// or an activation, which keeps the plain kernel's register count; and with
// one release left out on purpose (AbortTestConfig), for the failure-detection
// test switch.  Compiled on its own so the library's translation units build
// in parallel.
#include "variant.cuh"

namespace {

using Tile = sg::TileConfig<256, 128, 64, 2, 8, 2, 8, 8, sg::MICRO_FFMA2, sg::ISSUE_LAST_WARP>;

const sgv::Variant kTable[] = {
    // EXTRA_BATCHED
    sgv::make_variant<sg::ExConfig<Tile>>(
        "ffma2 tile=256x128x64 stages=2 warps=16 issuer=last_warp thread=8x8 stream_k "
        "batched+epilogue",
        true),
    // EXTRA_FUSED
    sgv::make_variant<sg::FusedConfig<Tile>>(
        "ffma2 tile=256x128x64 stages=2 warps=16 issuer=last_warp thread=8x8 stream_k epilogue",
        true),
    // EXTRA_DROP_RELEASE
    sgv::make_variant<sg::AbortTestConfig<Tile>>(
        "ffma2 tile=256x128x64 stages=2 warps=16 issuer=last_warp thread=8x8 stream_k "
        "drop_release_test",
        true),
};

cudaError_t error_word(unsigned *v, bool clear) { return sgv::unit_error_word(v, clear); }

}  // namespace

sgv::VariantTable sgv::extra_variants() {
    return {kTable, int(sizeof(kTable) / sizeof(kTable[0])), &error_word};
}
