// variant.cuh -- a compiled configuration of the persistent TMA/FFMA kernel as
// the host sees it (tile sizes, work split, launch and attribute functions),
// and the tables of configurations that other translation units compile.
//
// The library is built from several translation units compiled in parallel:
// sgemm.cu (host code, the default configurations, the 3xTF32 kernels),
// extra_variants.cu (the batched and fused-epilogue kernels, the
// failure-detection test kernel), staged_variants.cu (the default tiles with
// the staged epilogue), tall_variants.cu (a batch run as one tall GEMM) and
// sweep_variants_a.cu / sweep_variants_b.cu / sweep_variants_c.cu
// (configurations kept for tile-configuration sweeps).  They are linked without relocatable device
// code, so each unit has its own copy of the device error word (kernels.cuh);
// every table carries the function that reads and clears its unit's copy.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "kernels.cuh"

namespace sgv {

struct Variant {
    const char *name;
    int bm, bn, bk;
    bool stream_k;
    int group_m;
    int ctas_per_sm;   // resident CTAs per SM: the persistent grid is ctas_per_sm x SMs
    cudaError_t (*set_attr)();
    void (*launch)(int grid, cudaStream_t s, const CUtensorMap &a, const CUtensorMap &b,
                   const sg::MainParams &p, const sg::ExParams &x);
};

template <class Cfg>
cudaError_t set_attr_t() {
    return cudaFuncSetAttribute(sg::sgemm_tma_ffma_kernel<Cfg>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, int(Cfg::SMEM_BYTES));
}

template <class Cfg>
void launch_t(int grid, cudaStream_t s, const CUtensorMap &a, const CUtensorMap &b,
              const sg::MainParams &p, const sg::ExParams &x) {
    sg::sgemm_tma_ffma_kernel<Cfg><<<grid, Cfg::THREADS, Cfg::SMEM_BYTES, s>>>(a, b, p, x);
}

template <class Cfg>
constexpr Variant make_variant(const char *name, bool stream_k, int group_m = 8) {
    return Variant{name,      Cfg::BM,          Cfg::BN,          Cfg::BK, stream_k, group_m,
                   Cfg::CTAS_PER_SM, &set_attr_t<Cfg>, &launch_t<Cfg>};
}

// Reads this translation unit's device error word into *v (current device),
// and clears it when `clear` is set and the word is not zero.  Internal
// linkage, like the word itself: every unit gets its own function.
static cudaError_t unit_error_word(unsigned *v, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(v, sg::g_error_word, sizeof(unsigned));
    if (e != cudaSuccess || !clear || *v == 0) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(sg::g_error_word, &zero, sizeof(unsigned));
}

// Configurations compiled in another translation unit: `count` entries in
// variant-number order, and that unit's error-word access.
struct VariantTable {
    const Variant *entries;
    int count;
    cudaError_t (*error_word)(unsigned *v, bool clear);
};

VariantTable sweep_variants_a();
VariantTable sweep_variants_b();
VariantTable sweep_variants_c();

// extra_variants.cu: the default tile for batched calls with the fused
// epilogue, for one GEMM with the fused epilogue, and the failure-detection
// test kernel, at these indices.
enum { EXTRA_BATCHED = 0, EXTRA_FUSED = 1, EXTRA_DROP_RELEASE = 2 };
VariantTable extra_variants();

// staged_variants.cu: variants 0 and 1 (in that order) with the staged
// epilogue, for C whose rows do not all start 16-byte aligned.
VariantTable staged_variants();

// tall_variants.cu: the default tile for a batch run as one tall GEMM
// (TallBatchConfig).
VariantTable tall_variants();

}  // namespace sgv
