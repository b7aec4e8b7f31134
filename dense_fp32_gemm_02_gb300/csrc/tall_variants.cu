// tall_variants.cu -- the default 256x128x64 configuration of the persistent
// TMA/FFMA kernel compiled as TallBatchConfig: a strided batch of GEMMs with
// no bias or activation whose batches hold whole tiles (M a multiple of 256,
// K of 64) and whose C batches lie one under the other runs as one tall GEMM
// through the plain kernel's epilogue (tall_batch_call in sgemm.cu).
// Compiled on its own so the library's translation units build in parallel.
#include "variant.cuh"

namespace {

const sgv::Variant kTable[] = {
    sgv::make_variant<sg::TallBatchConfig<
        sg::TileConfig<256, 128, 64, 2, 8, 2, 8, 8, sg::MICRO_FFMA2, sg::ISSUE_LAST_WARP>>>(
        "ffma2 tile=256x128x64 stages=2 warps=16 issuer=last_warp thread=8x8 stream_k "
        "tall_batch",
        true),
};

cudaError_t error_word(unsigned *v, bool clear) { return sgv::unit_error_word(v, clear); }

}  // namespace

sgv::VariantTable sgv::tall_variants() {
    return {kTable, int(sizeof(kTable) / sizeof(kTable[0])), &error_word};
}
