// sgemm.cu -- host side of libsgemm.so: the C ABI declared in include/sgemm.h,
// argument checks, per-device state, the stream-ordered workspace pool, TMA
// descriptor encoding, kernel selection and launch, and benchmark timing hooks.
//
// Path of one sgemm() call (all on the caller's stream, no host sync):
//   1. pack_a_transpose_kernel: A (M x K, any lda) -> At (K x roundup(M, 4))
//   2. B re-pitched, only when B's address or row pitch is not 16-byte aligned
//      as the TMA requires: one pack_ab_kernel does steps 1 and 2 together
//   3. sgemm_tma_ffma_kernel: persistent CTAs, TMA ring, FFMA micro-tiles,
//      alpha/beta epilogue straight to C
//   4. the workspace goes back to the pool, ordered after step 3.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "../../include/sgemm.h"
#include "aux_kernels.cuh"
#include "kernels.cuh"
#include "tf32x3.cuh"
#include "tf32x3_pair.cuh"
#include "variant.cuh"

#define SGEMM_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr int kVersion = 1 * 10000 + 0 * 100 + 0;
constexpr int kMaxDevices = 64;

thread_local int t_last_cuda_error = 0;
// Configuration text of the last main kernel this thread's calls launched
// (sgemm_last_kernel): a variant's name or one of the fixed texts below.
thread_local const char *t_last_kernel = "";
constexpr const char *kSmallKernel32 = "direct small-problem kernel, 32x32 tiles";
constexpr const char *kSmallKernel64 = "direct small-problem kernel, 64x64 tiles";
constexpr const char *kSmallSplitK = "direct small-problem kernel, 32x32 tiles, k split over a cluster";
constexpr const char *kScaleOnly = "scale only (C = beta * C)";
constexpr const char *kSkinny = "skinny-M kernel (B read once, k split over the grid)";
constexpr const char *kSkinnyN = "skinny-N kernel (A read once, k split over the grid)";
constexpr const char *kT3Pair = "3xtf32 tcgen05 cta_group::2, 256x256 pair tiles";
constexpr const char *kT3Single = "3xtf32 tcgen05, 128x256 tiles";

// ------------------------------------------------------------------ kernel variants
// Every variant is the same persistent TMA/FFMA kernel with other tile sizes or
// micro-kernel.  The default is chosen per shape by pick_variant(); a specific
// one can be forced for tile-configuration sweeps with sgemm_set_variant().
using sgv::make_variant;
using sgv::Variant;
using sg::MICRO_FFMA2;
using sg::ISSUE_LAST_WARP;
// Variant 0 is the default: it was the fastest or within 1% of the fastest on
// every measured workload.  Its 16 consumer warps (four per scheduler) hide
// the shared-memory latency of the fragment loads better than 12 warps plus a
// producer warpgroup (16 consumer warps at 128 registers fill the register
// file, so the two do not fit together), and the warp that releases a stage
// last refills it, so no warp waits for the others.  Variant 1, the same tile
// turned, takes the shapes that it pads less (pick_variant).  Variant 3 is
// variant 0's kernel with whole tiles only (no stream-K tail).  The others,
// compiled in sweep_variants_a.cu and sweep_variants_b.cu, stay for sweeps
// and as evidence for the design choices (issuer, tile shape, warp
// specialisation, packed FP32x2 FMA, thread-tile size, k depth of a stage).
using DefaultTile = sg::TileConfig<256, 128, 64, 2, 8, 2, 8, 8, MICRO_FFMA2, ISSUE_LAST_WARP>;
const Variant kMainVariants[] = {
    make_variant<DefaultTile>(
        "ffma2 tile=256x128x64 stages=2 warps=16 issuer=last_warp thread=8x8 stream_k", true),
    make_variant<sg::TileConfig<128, 256, 64, 2, 4, 4, 8, 8, MICRO_FFMA2, ISSUE_LAST_WARP>>(
        "ffma2 tile=128x256x64 stages=2 warps=16 issuer=last_warp thread=8x8 stream_k", true),
    make_variant<DefaultTile>(
        "ffma2 tile=256x128x64 stages=2 warps=16 issuer=last_warp thread=8x8 no_stream_k", false),
};

// All variants in variant-number order: 0, 1 and 3 from this file, 2 and 4-6
// from sweep_variants_a.cu, 7-11 from sweep_variants_b.cu, 12-13 from
// sweep_variants_c.cu.
struct VariantIndex {
    const Variant *v[32];
    int n = 0;
    VariantIndex() {
        const sgv::VariantTable a = sgv::sweep_variants_a(), b = sgv::sweep_variants_b();
        const sgv::VariantTable c = sgv::sweep_variants_c();
        v[n++] = &kMainVariants[0];
        v[n++] = &kMainVariants[1];
        v[n++] = &a.entries[0];
        v[n++] = &kMainVariants[2];
        for (int i = 1; i < a.count; ++i) v[n++] = &a.entries[i];
        for (int i = 0; i < b.count; ++i) v[n++] = &b.entries[i];
        for (int i = 0; i < c.count; ++i) v[n++] = &c.entries[i];
    }
};
const VariantIndex &variant_index() {
    static const VariantIndex idx;
    return idx;
}
int variant_count() { return variant_index().n; }
const Variant &variant_at(int id) { return *variant_index().v[id]; }

// Batched calls run the default configuration compiled with the batch
// coordinate (3-D tensor maps) and the fused epilogue; unbatched calls with a
// bias or an activation run it with the fused epilogue alone (2-D maps), which
// keeps the plain kernel's 123 registers (the batched one needs 128).  Both,
// and the failure-detection test kernel, are compiled in extra_variants.cu.
const Variant &ex_variant() { return sgv::extra_variants().entries[sgv::EXTRA_BATCHED]; }
const Variant &fused_variant() { return sgv::extra_variants().entries[sgv::EXTRA_FUSED]; }
const Variant &abort_test_variant() { return sgv::extra_variants().entries[sgv::EXTRA_DROP_RELEASE]; }
// A batch that tall_batch_call() accepts runs as one tall GEMM through the
// plain kernel's epilogue (tall_variants.cu).
const Variant &tall_variant() { return sgv::tall_variants().entries[0]; }
std::atomic<int> g_forced_variant{-1};
std::atomic<int> g_drop_release{0};
// 3xTF32 main kernel: -1 = chosen per shape (t3_use_pair), 0 = the single-CTA
// kernel, 1 = the CTA pair
std::atomic<int> g_t3_pair{-1};

// Shape heuristic between the two orientations of the default tile, 256x128
// (variant 0) and 128x256 (variant 1): same kernel, same speed where both fit
// the shape, so the one that pads C less wins; variant 0 on a tie.  Padding is
// the FMA work spent on the rows and columns past M and N in edge tiles (M =
// 4097: 17 tile rows of 256 or 33 of 128).
long long padded_area(const Variant &v, int M, int N) {
    return ((M + v.bm - 1LL) / v.bm) * v.bm * (((N + v.bn - 1LL) / v.bn) * v.bn);
}

// Stream-K is worth its fix-up (partial sums written and read back, a second
// pass over them before the epilogue) only while whole tiles alone would
// leave a noticeable share of the SMs' slots idle in their last wave.  Below
// 1 % it is left out: 16384x16384x512 (8192 tiles of 256x128 in 54 waves of
// 152, 0.2 % idle) measured 86.4 % of the FFMA peak with whole tiles only
// against 86.1 % with the stream-K tail; 8192^3 (2048 tiles, 3.8 % idle)
// keeps it.
bool stream_k_pays(long long tiles, int sms) {
    const long long waves = (tiles + sms - 1) / sms;
    return double(waves * sms - tiles) >= 0.01 * double(waves * sms);
}

// Few tiles: when the chosen orientation of the default tile makes fewer
// tiles than a quarter of the SMs, stream-K splits every tile over more than
// four CTAs, and the CTA that completes a tile reads back all its pieces
// (128 KB each) before the epilogue.  The 128x128x48 tile of variant 9 (four
// stages fed by a producer warpgroup) makes twice the tiles with half-size
// pieces.  Same box, pre-pass + main kernel: 1024^3 0.066 ms against 0.073,
// 768^3 0.049 against 0.065, 1024x1024x4096 0.164 against 0.172,
// 128x4096x4096 0.101 against 0.115, 512x512x2048 0.065 against 0.084,
// 128x3001x1023 0.068 against 0.070; 256x3001x1023 (24 tiles, no padding in
// M for the 256-row tile) 0.073 against 0.071 is the one loss seen.  48 tiles
// and more stay on the default tile (512x3001x1023: 0.090 against 0.095).
// `sms` 0 (no device known) leaves this rule out.
constexpr int kFewTilesVariant = 9;

// Rows up to which a GEMM that is not a small problem takes the skinny-M
// kernel (launch_skinny) instead of the persistent one.  Same box, main kernel
// against the 128x128 tile the few-tiles rule would give: 1 x 8192 x 8192
// 0.052 ms against 0.279, 16 x 8192 x 8192 0.104 against 0.276, 32 x 8192 x
// 8192 0.216 against 0.278, 16 x 16384 x 2048 0.061 against 0.149, 32 x 3001
// x 1023 0.029 against 0.055.  At 32 rows the margin at 8192^2 x 8192 is down
// to 22 %, so the persistent kernel keeps 33 rows and more.
constexpr int kSkinnyRows = sg::SKINNY_ROWS;
// Columns up to which such a GEMM takes the skinny-N kernel (launch_skinny_n).
constexpr int kSkinnyCols = sg::SKINNY_COLS_MAX;

int pick_variant(int M, int N, int K, int sms) {
    const int forced = g_forced_variant.load();
    if (forced >= 0 && forced < variant_count()) return forced;
    (void)K;
    const int id = padded_area(variant_at(1), M, N) < padded_area(variant_at(0), M, N) ? 1 : 0;
    const Variant &v = variant_at(id);
    const long long tiles = ((M + v.bm - 1LL) / v.bm) * ((N + v.bn - 1LL) / v.bn);
    return (sms > 0 && 4 * tiles < sms) ? kFewTilesVariant : id;
}

struct DeviceState {
    bool ready = false;
    int status = SGEMM_OK;
    int sm_count = 0;
    cudaMemPool_t pool = nullptr;
};

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;
std::atomic<unsigned long long> g_timeout_ns{2000000000ull};
std::atomic<long long> g_launches{0};

// ------------------------------------------------------------------ profiling
// One interval timed by a pair of events: a call's pre-pass kernels, or its
// main kernel.  `owns_*`: the event goes back to the free list when the
// record is collected (an event shared by two records belongs to one).
struct ProfRecord {
    cudaEvent_t start, stop;
    bool is_main, owns_start, owns_stop;
};
std::mutex g_prof_mutex;
std::atomic<int> g_prof_on{0};
std::vector<ProfRecord> g_prof_used;
std::vector<cudaEvent_t> g_prof_free;

cudaEvent_t prof_event() {
    // caller holds g_prof_mutex
    if (!g_prof_free.empty()) {
        cudaEvent_t e = g_prof_free.back();
        g_prof_free.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

// Kernel timing of one call while profiling is on: an event before its
// pre-pass kernels, one between them and its main kernel, one after the main
// kernel.  The pre-pass's end and the main kernel's start share an event:
// each event record between two kernels keeps the GPU from overlapping the
// second one's launch with the first one's end (measured: 4 records per call
// cost about 9 us per call more than none).
struct ProfCall {
    cudaStream_t stream;
    bool on;
    cudaEvent_t pre = nullptr, mid = nullptr, end = nullptr;

    explicit ProfCall(cudaStream_t s) : stream(s), on(g_prof_on.load() != 0) {}
    cudaEvent_t record() {
        cudaEvent_t e;
        {
            std::lock_guard<std::mutex> lk(g_prof_mutex);
            e = prof_event();
        }
        if (e) cudaEventRecord(e, stream);
        return e;
    }
    void pre_begin() {   // before the first pre-pass kernel (later calls: no-op)
        if (on && !pre && !mid) pre = record();
    }
    void main_begin() {
        if (on && !mid) mid = record();
    }
    void main_end() {
        if (on && mid && !end) end = record();
    }
    ~ProfCall() {
        if (!on) return;
        std::lock_guard<std::mutex> lk(g_prof_mutex);
        if (pre && mid) {
            g_prof_used.push_back({pre, mid, false, true, end == nullptr});
        } else if (pre) {
            g_prof_free.push_back(pre);
        }
        if (mid && end) {
            g_prof_used.push_back({mid, end, true, true, true});
        } else if (mid && !pre) {
            g_prof_free.push_back(mid);
        }
    }
};

// ------------------------------------------------------------------ helpers
int cuda_fail(cudaError_t e) {
    t_last_cuda_error = int(e);
    return (e == cudaErrorMemoryAllocation) ? SGEMM_ERR_ALLOC : SGEMM_ERR_CUDA;
}

bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Largest M, N or K accepted: the kernels round sizes up to whole tiles and
// k steps in 32-bit arithmetic, so 2^16 below 2^31 leaves them room.
constexpr int kMaxDim = 0x7fffffff - 0xffff;

int checked_args(int M, int N, int K, const float *A, int lda, const float *B, int ldb,
                 const float *C, int ldc, float alpha, float beta) {
    if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_ARG;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return SGEMM_ERR_TOO_LARGE;
    if (lda < std::max(1, K) || ldb < std::max(1, N) || ldc < std::max(1, N))
        return SGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return SGEMM_OK;
    if (!C || !aligned4(C)) return SGEMM_ERR_INVALID_ARG;
    if (K > 0 && alpha != 0.0f) {
        if (!A || !B || !aligned4(A) || !aligned4(B)) return SGEMM_ERR_INVALID_ARG;
    }
    (void)beta;
    return SGEMM_OK;
}

// Lazily initialise per-device state for the current device.
int device_state(DeviceState **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return SGEMM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lk(g_mutex);
    DeviceState &d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e);
        if (major != 10 || minor != 3) {
            d.status = SGEMM_ERR_UNSUPPORTED_DEVICE;
        } else {
            if (!g_encode_tiled) {
                void *fn = nullptr;
                cudaDriverEntryPointQueryResult q;
                e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
                if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
                    return cuda_fail(e != cudaSuccess ? e : cudaErrorNotSupported);
                g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
            }
            cudaMemPoolProps props;
            std::memset(&props, 0, sizeof(props));
            props.allocType = cudaMemAllocationTypePinned;
            props.handleTypes = cudaMemHandleTypeNone;
            props.location.type = cudaMemLocationTypeDevice;
            props.location.id = dev;
            if ((e = cudaMemPoolCreate(&d.pool, &props)) != cudaSuccess) return cuda_fail(e);
            // keep up to 4 GiB of released workspace cached for reuse
            cuuint64_t keep = 4ull << 30;
            cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep);
            for (int i = 0; i < variant_count(); ++i)
                if ((e = variant_at(i).set_attr()) != cudaSuccess) return cuda_fail(e);
            if ((e = ex_variant().set_attr()) != cudaSuccess) return cuda_fail(e);
            if ((e = fused_variant().set_attr()) != cudaSuccess) return cuda_fail(e);
            if ((e = abort_test_variant().set_attr()) != cudaSuccess) return cuda_fail(e);
            if ((e = tall_variant().set_attr()) != cudaSuccess) return cuda_fail(e);
            for (int i = 0; i < sgv::staged_variants().count; ++i)
                if ((e = sgv::staged_variants().entries[i].set_attr()) != cudaSuccess)
                    return cuda_fail(e);
            if ((e = cudaFuncSetAttribute(sg::t3::sgemm_3xtf32_pair_kernel,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          int(sg::t3::P_SMEM_BYTES))) != cudaSuccess)
                return cuda_fail(e);
            e = cudaFuncSetAttribute(sg::t3::sgemm_3xtf32_kernel,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     int(sg::t3::SMEM_BYTES));
            if (e != cudaSuccess) return cuda_fail(e);
            d.status = SGEMM_OK;
        }
        d.ready = true;
    }
    *out = &d;
    return d.status;
}

int encode_2d(CUtensorMap *map, const float *ptr, uint64_t inner, uint64_t outer,
              uint64_t row_pitch_elems, uint32_t box_inner, uint32_t box_outer,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_pitch_elems * sizeof(float)};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(ptr),
                                dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        t_last_cuda_error = int(r);
        return SGEMM_ERR_CUDA;
    }
    return SGEMM_OK;
}

// 3-D tensor map over `planes` row-major matrices of outer x inner floats,
// rows row_pitch floats apart and planes plane_pitch floats apart; box
// box_inner x box_outer x 1.
int encode_3d(CUtensorMap *map, const float *ptr, uint64_t inner, uint64_t outer, uint64_t planes,
              uint64_t row_pitch_elems, uint64_t plane_pitch_elems, uint32_t box_inner,
              uint32_t box_outer) {
    cuuint64_t dims[3] = {inner, outer, planes};
    cuuint64_t strides[2] = {row_pitch_elems * sizeof(float), plane_pitch_elems * sizeof(float)};
    cuuint32_t box[3] = {box_inner, box_outer, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(ptr),
                                dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        t_last_cuda_error = int(r);
        return SGEMM_ERR_CUDA;
    }
    return SGEMM_OK;
}

long long round_up(long long x, long long m) { return (x + m - 1) / m * m; }

// One call of the FFMA path: `batch` GEMMs with strided operands and the
// fused epilogue.  sgemm() is batch 1 without bias or activation.
struct GemmCall {
    int M, N, K;
    float alpha;
    const float *A;
    int lda;
    long long stride_a;
    const float *B;
    int ldb;
    long long stride_b;
    float beta;
    float *C;
    int ldc;
    long long stride_c;
    int batch;
    const float *bias;
    long long stride_bias;
    int act;
};

GemmCall plain_call(int M, int N, int K, float alpha, const float *A, int lda, const float *B,
                    int ldb, float beta, float *C, int ldc) {
    return GemmCall{M, N, K, alpha, A, lda, 0, B, ldb, 0, beta, C, ldc, 0, 1, nullptr, 0,
                    sg::ACT_NONE};
}

// Argument checks of a batched call (the single-GEMM checks plus batch,
// strides, bias and activation).  Batches of C must not overlap.
int checked_call(const GemmCall &g) {
    if (g.batch < 0 || g.stride_a < 0 || g.stride_b < 0 || g.stride_c < 0 || g.stride_bias < 0)
        return SGEMM_ERR_INVALID_ARG;
    if (g.act < sg::ACT_NONE || g.act > sg::ACT_GELU) return SGEMM_ERR_INVALID_ARG;
    // an empty batch, like an empty matrix, reads and writes nothing
    const bool empty = g.batch == 0;
    int st = checked_args(g.M, empty ? 0 : g.N, g.K, g.A, g.lda, g.B, g.ldb, g.C,
                          empty ? std::max(g.ldc, 1) : g.ldc, g.alpha, g.beta);
    if (st != SGEMM_OK) return st;
    if (g.M == 0 || g.N == 0 || empty) return SGEMM_OK;
    if (g.bias && !aligned4(g.bias)) return SGEMM_ERR_INVALID_ARG;
    if (g.batch > 1 && g.stride_c < (long long)(g.M - 1) * g.ldc + g.N) return SGEMM_ERR_INVALID_ARG;
    return SGEMM_OK;
}

// The pre-pass of one GEMM whose B must be re-pitched, in one launch
// (pack_ab_kernel): up to 16 blocks per SM for each of the A transpose (64x64
// tiles) and the B copy (16 x 256 strips), each part walking its own work.
void launch_pack_ab(const float *A, long long lda, int M, int K, float *At, long long ldat,
                    const float *B, long long ldb, int N, float *Bp, long long ldbp, int *zero,
                    int zero_count, int sms, cudaStream_t stream) {
    const long long cap = 16LL * sms;
    const long long a_tiles = ((K + 63LL) / 64) * ((M + 63LL) / 64);
    const long long b_strips = ((N + 255LL) / 256) * ((K + 15LL) / 16);
    const int a_blocks = int(std::min(a_tiles, cap)), b_blocks = int(std::min(b_strips, cap));
    sg::pack_ab_kernel<<<a_blocks + b_blocks, 256, 0, stream>>>(A, lda, M, K, At, ldat, B, ldb, N,
                                                                Bp, ldbp, a_blocks, zero,
                                                                zero_count);
    g_launches.fetch_add(1);
}

int launch_scale(cudaStream_t stream, const GemmCall &g, int sms) {
    const long long total = (long long)g.M * g.N * g.batch;
    const int blocks = int(std::min<long long>((total + 255) / 256, (long long)sms * 8));
    sg::scale_c_kernel<<<blocks, 256, 0, stream>>>(g.C, g.ldc, g.stride_c, g.M, g.N, g.batch,
                                                   g.beta, g.bias, g.stride_bias, g.act);
    g_launches.fetch_add(1);
    t_last_kernel = kScaleOnly;
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SGEMM_OK : cuda_fail(e);
}

// Epilogue and batch parameters of the batched / fused kernel.
sg::ExParams ex_params(const GemmCall &g, int a_planes, int b_planes) {
    sg::ExParams x;
    x.batch = g.batch;
    x.stride_c = g.stride_c;
    x.a_planes = a_planes;
    x.b_planes = b_planes;
    x.bias = g.bias;
    x.stride_bias = g.stride_bias;
    x.bias_vec4 = (g.bias && aligned16(g.bias) && g.stride_bias % 4 == 0) ? 1 : 0;
    x.act = g.act;
    x.tall_b_rows = 0;
    return x;
}

// The kernel of a plain GEMM: the variant pick_variant() names, or the same
// tile with the staged epilogue (store_tile_staged) when that pays: it is one
// of the two default tiles, the rows of C do not all start 16-byte aligned,
// C_in is read (beta != 0) and K is short (at most 2048: 32 slabs per tile).
// There the staged epilogue's loads of C_in (128 contiguous bytes per warp
// access, instead of four times the sectors they use) outweigh its main loop,
// which runs about 2 % slower at the staged kernel's register allocation
// (same box: 4097x3001x1023 with beta 1 0.430 ms against 0.458; with beta 0
// 0.420 against 0.416; 4096x3001x4096 equal; 8192x8191x8192 15.84 against
// 15.54).
const Variant &plain_variant(int M, int N, int K, float beta, const float *C, int ldc, int sms) {
    const int id = pick_variant(M, N, K, sms);
    const bool rows_aligned = aligned16(C) && ldc % 4 == 0;
    if (id <= 1 && !rows_aligned && beta != 0.0f && K <= 2048)
        return sgv::staged_variants().entries[id];
    return variant_at(id);
}

// True when a strided batch can run as one tall GEMM (TallBatchConfig): no
// bias or activation, one A per batch, every batch whole tiles of the default
// 256x128x64 tile (M a multiple of 256, K of 64) and at most 16 tile rows (the
// raster groups are the batches, and a group of 16 rows is twice the default
// 8), the batches of C one under the other (stride_c = M * ldc), and B either
// shared (stride_b = 0), its batches one under the other (stride_b = K * ldb),
// or re-pitched anyway (rows that break the TMA's 16-byte rule).  Batch b's
// rows of C are then rows b*M .. b*M+M-1 of one (batch*M) x N matrix, its
// transposed A columns b*M .. of one K x (batch*M) matrix, and its B rows
// b*K .. of one (batch*K) x N matrix.  The batched kernel (ExConfig) takes the
// rest: its 3-D tensor maps read B with any plane pitch, but its main loop
// runs 2 % slower (same box: 64 x 1024^3 2.026 ms against 1.989).
bool tall_batch_call(const GemmCall &g) {
    if (g.batch <= 1 || g.bias != nullptr || g.act != sg::ACT_NONE || g.stride_a == 0) return false;
    if (g.M % 256 != 0 || g.M > 16 * 256 || g.K % 64 != 0) return false;
    if (g.stride_c != (long long)g.M * g.ldc) return false;
    if ((long long)g.batch * g.M > kMaxDim || (long long)g.batch * g.K > kMaxDim) return false;
    const bool b_tma = aligned16(g.B) && g.ldb % 4 == 0;
    return !b_tma || g.stride_b == 0 || g.stride_b == (long long)g.K * g.ldb;
}

// True when the default 256x128x64 tiling offers fewer slabs of work than
// there are SMs: the persistent kernel would run a handful of CTAs, each
// through a pre-pass, a slab and a stream-K fix-up.  Such GEMMs take the
// direct small-problem kernel.
bool small_problem(int M, int N, int K, int sms) {
    const long long tiles = ((M + 255LL) / 256) * ((N + 127LL) / 128);
    return tiles * ((K + 63LL) / 64) < sms;
}

// The small-problem kernel's configuration: 64x64 tiles when they fill at
// least the SMs, else 32x32 tiles; with 32x32 tiles that fill at most half
// the SMs, the k range of a tile is split over the CTAs of a cluster (S <= 8,
// at least two k steps of 32 each): 256^3 runs 64 tiles x 4 CTAs instead of
// 64 CTAs walking all of K.
struct SmallSplit {
    int tile, S, kchunk;
};
SmallSplit small_split(int M, int N, int K, int sms) {
    const long long t64 = ((M + 63LL) / 64) * ((N + 63LL) / 64);
    const long long t32 = ((M + 31LL) / 32) * ((N + 31LL) / 32);
    SmallSplit r{t64 < sms ? 32 : 64, 1, K};
    if (t64 < sms && 2 * t32 <= sms) {
        const int by_sms = int(std::min<long long>(8, (2LL * sms) / t32));
        const int by_k = (K + 2 * sg::SMALL_BK - 1) / (2 * sg::SMALL_BK);
        r.S = std::max(1, std::min(by_sms, by_k));
        if (r.S > 1) {
            r.kchunk = int(round_up((K + r.S - 1) / r.S, sg::SMALL_BK));
            r.S = (K + r.kchunk - 1) / r.kchunk;
        }
    }
    return r;
}

const char *small_kernel_text(const SmallSplit &sp) {
    return sp.S > 1 ? kSmallSplitK : sp.tile == 32 ? kSmallKernel32 : kSmallKernel64;
}

int launch_small(const GemmCall &g, cudaStream_t stream, int sms) {
    ProfCall prof(stream);
    prof.main_begin();
    const SmallSplit sp = small_split(g.M, g.N, g.K, sms);
    const int S = sp.S, kchunk = sp.kchunk;
    if (S > 1) {
        cudaLaunchConfig_t cfg;
        std::memset(&cfg, 0, sizeof(cfg));
        cfg.gridDim = dim3(unsigned((g.N + 31) / 32), unsigned((g.M + 31) / 32), unsigned(S));
        cfg.blockDim = dim3(256);
        cfg.stream = stream;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 1;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = unsigned(S);
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        t_last_kernel = kSmallSplitK;
        cudaLaunchKernelEx(&cfg, sg::sgemm_small_splitk_kernel<32>, g.M, g.N, g.K, kchunk, g.alpha,
                           g.A, (long long)g.lda, g.B, (long long)g.ldb, g.beta, g.C,
                           (long long)g.ldc);
    } else if (sp.tile == 32) {
        dim3 grid(unsigned((g.N + 31) / 32), unsigned((g.M + 31) / 32));
        t_last_kernel = kSmallKernel32;
        sg::sgemm_small_kernel<32><<<grid, 256, 0, stream>>>(g.M, g.N, g.K, g.alpha, g.A, g.lda, g.B,
                                                            g.ldb, g.beta, g.C, g.ldc);
    } else {
        dim3 grid(unsigned((g.N + 63) / 64), unsigned((g.M + 63) / 64));
        t_last_kernel = kSmallKernel64;
        sg::sgemm_small_kernel<64><<<grid, 256, 0, stream>>>(g.M, g.N, g.K, g.alpha, g.A, g.lda, g.B,
                                                            g.ldb, g.beta, g.C, g.ldc);
    }
    prof.main_end();
    g_launches.fetch_add(1);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SGEMM_OK : cuda_fail(e);
}

// One instantiation of the skinny kernel: rows, columns per thread, blocks per
// SM (the register budget: 65536 / (256 x MINB) per thread) and k steps
// unrolled.  Chosen per row count by a sweep of 25 instantiations over
// 4096^2 x 4096, 8192^2 x 8192, 16384 x 2048 x N and 3001 x 1023 x N shapes
// (same box): M = 1 runs at 4.2-5.1 TB/s of B at the larger shapes.
struct SkinnyConfig {
    int rows, cols;
    void (*kernel)(int, int, int, int, float, const float *, long long, const float *, long long,
                   float, float *, long long, float *);
};
template <int MR, int COLS, int MINB, int UNR>
constexpr SkinnyConfig skinny_config() {
    return {MR, COLS, &sg::sgemm_skinny_kernel<MR, COLS, MINB, UNR>};
}
constexpr SkinnyConfig kSkinnyConfigs[] = {
    skinny_config<1, 4, 4, 8>(), skinny_config<2, 4, 4, 4>(), skinny_config<4, 2, 4, 8>(),
    skinny_config<8, 2, 4, 8>(), skinny_config<16, 2, 2, 8>(), skinny_config<32, 2, 1, 8>(),
};
// k-range split: about this many blocks per SM (skinny-M blocks of 256
// threads, skinny-N blocks of 128)
constexpr int kSkinnyBlocksPerSM = 4;
constexpr int kSkinnyNBlocksPerSM = 8;

// The split-K launch shared by the skinny kernels: `blocks` blocks along the
// grid's x dimension, K cut into S ranges of whole `step`-deep steps along y so
// that about `per_sm` blocks per SM run; with S > 1 the kernel writes S
// partial sums per output to pool memory and skinny_reduce_kernel adds them in
// range order and applies alpha and beta.  launch(grid, kchunk, P) issues the
// kernel on `stream`.
template <class Launch>
int run_split_k(const GemmCall &g, cudaStream_t stream, DeviceState *dev, long long blocks,
                int step, int per_sm, const char *text, Launch &&launch) {
    const int M = g.M, N = g.N, K = g.K;
    const long long steps = (K + step - 1LL) / step;
    const long long want = (long long)per_sm * dev->sm_count;
    long long S = std::max(1LL, std::min(steps, (want + blocks - 1) / blocks));
    const int kchunk = int(((steps + S - 1) / S) * step);
    S = (K + kchunk - 1LL) / kchunk;
    if (blocks > 0x7fffffffLL || S > 65535) return SGEMM_ERR_TOO_LARGE;
    float *P = nullptr;
    if (S > 1) {
        cudaError_t e = cudaMallocFromPoolAsync(reinterpret_cast<void **>(&P),
                                                size_t(S) * M * N * 4, dev->pool, stream);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    ProfCall prof(stream);
    prof.main_begin();
    launch(dim3(static_cast<unsigned>(blocks), static_cast<unsigned>(S)), kchunk, P);
    g_launches.fetch_add(1);
    t_last_kernel = text;
    if (S > 1) {
        const long long total = (long long)M * N;
        const int rblocks = int(std::min<long long>((total + 255) / 256, (long long)dev->sm_count * 8));
        sg::skinny_reduce_kernel<<<rblocks, 256, 0, stream>>>(M, N, int(S), P, g.alpha, g.beta,
                                                              g.C, g.ldc);
        g_launches.fetch_add(1);
    }
    prof.main_end();
    cudaError_t e = cudaGetLastError();
    cudaError_t ef = S > 1 ? cudaFreeAsync(P, stream) : cudaSuccess;
    if (e != cudaSuccess) return cuda_fail(e);
    if (ef != cudaSuccess) return cuda_fail(ef);
    return SGEMM_OK;
}

// GEMMs of at most SKINNY_ROWS rows that are not small problems: B streamed
// once by sgemm_skinny_kernel, the k range split so that about
// kSkinnyBlocksPerSM blocks per SM run (whole 128-deep sub-ranges), partial
// sums added in order by skinny_reduce_kernel.
int launch_skinny(const GemmCall &g, cudaStream_t stream, DeviceState *dev) {
    const SkinnyConfig *cfg = &kSkinnyConfigs[0];
    while (cfg->rows < g.M) ++cfg;
    const long long block_cols = (long long)sg::SKINNY_THREADS * cfg->cols;
    return run_split_k(g, stream, dev, (g.N + block_cols - 1) / block_cols, sg::SKINNY_KSUB,
                       kSkinnyBlocksPerSM, kSkinny, [&](dim3 grid, int kchunk, float *P) {
                           cfg->kernel<<<grid, sg::SKINNY_THREADS, 0, stream>>>(
                               g.M, g.N, g.K, kchunk, g.alpha, g.A, g.lda, g.B, g.ldb, g.beta,
                               g.C, g.ldc, P);
                       });
}

// GEMMs of at most SKINNY_COLS_MAX columns that are not small problems (nor
// skinny in M): A streamed once by sgemm_skinny_n_kernel, 128 rows per block,
// the k range split so that about kSkinnyNBlocksPerSM blocks per SM run,
// partial sums added in order by skinny_reduce_kernel.
int launch_skinny_n(const GemmCall &g, cudaStream_t stream, DeviceState *dev) {
    auto kernel = g.N <= 4    ? &sg::sgemm_skinny_n_kernel<4>
                  : g.N <= 8  ? &sg::sgemm_skinny_n_kernel<8>
                  : g.N <= 16 ? &sg::sgemm_skinny_n_kernel<16>
                              : &sg::sgemm_skinny_n_kernel<32>;
    return run_split_k(g, stream, dev, (g.M + sg::SKINNY_N_ROWS - 1LL) / sg::SKINNY_N_ROWS,
                       sg::SKINNY_N_KC, kSkinnyNBlocksPerSM, kSkinnyN,
                       [&](dim3 grid, int kchunk, float *P) {
                           kernel<<<grid, sg::SKINNY_N_ROWS, 0, stream>>>(
                               g.M, g.N, g.K, kchunk, g.alpha, g.A, g.lda, g.B, g.ldb, g.beta,
                               g.C, g.ldc, P);
                       });
}

int gemm_device(const GemmCall &g, cudaStream_t stream) {
    int st = checked_call(g);
    if (st != SGEMM_OK || g.M == 0 || g.N == 0 || g.batch == 0) return st;
    DeviceState *dev = nullptr;
    if ((st = device_state(&dev)) != SGEMM_OK) return st;

    if (g.K == 0 || g.alpha == 0.0f) return launch_scale(stream, g, dev->sm_count);

    const int M = g.M, N = g.N, K = g.K;
    const bool batched = g.batch > 1;
    const bool extended = batched || g.bias != nullptr || g.act != sg::ACT_NONE;
    const bool drop_test = !extended && g_drop_release.load() != 0;
    if (!extended && !drop_test && g_forced_variant.load() < 0) {
        if (small_problem(M, N, K, dev->sm_count)) return launch_small(g, stream, dev->sm_count);
        if (M <= kSkinnyRows) return launch_skinny(g, stream, dev);
        if (N <= kSkinnyCols) return launch_skinny_n(g, stream, dev);
    }
    const bool tall = tall_batch_call(g);
    const Variant &var = tall ? tall_variant()
                         : batched ? ex_variant()
                         : extended ? fused_variant()
                         : drop_test ? abort_test_variant()
                                     : plain_variant(M, N, K, g.beta, g.C, g.ldc, dev->sm_count);
    // A and B enter as one plane per batch, or one plane for all batches when
    // their stride is 0
    const int a_planes = (g.batch > 1 && g.stride_a != 0) ? g.batch : 1;
    const int b_planes = (g.batch > 1 && g.stride_b != 0) ? g.batch : 1;
    // the rows and batches the kernel walks: a tall batch is one GEMM of
    // batch * M rows
    const long long m_rows = tall ? (long long)g.batch * M : M;
    const int k_batch = tall ? 1 : g.batch;
    // ---- work split: whole-tile waves, then the leftover tiles' k-slabs spread
    // evenly over all CTAs (stream-K) so the last wave is not partly idle
    const long long tiles_m = (m_rows + var.bm - 1) / var.bm, tiles_n = (N + var.bn - 1) / var.bn;
    const long long tiles = tiles_m * tiles_n * k_batch;
    const long long k_tiles = (K + var.bk - 1) / var.bk;
    const int slots = dev->sm_count * var.ctas_per_sm;   // persistent CTAs
    const bool sk = var.stream_k && stream_k_pays(tiles, slots);
    const int grid = sk ? int(std::min<long long>(slots, tiles * k_tiles))
                        : int(std::min<long long>(slots, tiles));
    const long long dp_tiles = sk ? (tiles / grid) * grid : tiles;
    const long long sk_tiles = tiles - dp_tiles;
    const long long sk_slabs = sk_tiles * k_tiles;
    if (tiles > (1LL << 30)) return SGEMM_ERR_TOO_LARGE;

    // ---- workspace: transposed A, a re-pitched B if needed, stream-K partial
    // sums and tile counters.  A transposed: one K x ldat plane per batch
    // (256-byte aligned planes), or for a tall batch one K x (batch*M) matrix
    // with batch b's columns at b*M.
    const long long ldat = tall ? m_rows : round_up(M, 4);
    const long long at_plane = tall ? M : round_up((long long)K * ldat, 64);
    // B is read in place when the TMA can address it: 16-byte base and row
    // pitch, and (several planes) a 16-byte plane pitch that is at least a
    // whole matrix
    const bool b_direct = aligned16(g.B) && (g.ldb % 4 == 0) &&
                          (b_planes == 1 || (g.stride_b % 4 == 0 && g.stride_b >= (long long)K * g.ldb));
    // (a tall batch's re-pitched B planes lie one under the other)
    const long long ldbp = b_direct ? g.ldb : round_up(N, 4);
    const long long bp_plane = b_direct ? g.stride_b
                               : tall   ? (long long)K * ldbp
                                        : round_up((long long)K * ldbp, 64);
    const size_t at_bytes = tall ? size_t(round_up((long long)K * ldat, 64)) * 4
                                 : size_t(at_plane) * a_planes * 4;
    const size_t bp_bytes = b_direct ? 0 : size_t(bp_plane) * b_planes * 4;
    const size_t part_bytes = sk_slabs ? size_t(2) * grid * var.bm * var.bn * 4 : 0;
    const size_t cnt_bytes = size_t(sk_tiles) * 4;
    const size_t ws_bytes = at_bytes + bp_bytes + part_bytes + cnt_bytes;

    void *ws = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, ws_bytes, dev->pool, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    char *wsb = static_cast<char *>(ws);
    float *At = reinterpret_cast<float *>(wsb);
    float *Bp = b_direct ? const_cast<float *>(g.B) : reinterpret_cast<float *>(wsb + at_bytes);
    float *partials = sk_slabs ? reinterpret_cast<float *>(wsb + at_bytes + bp_bytes) : nullptr;
    int *counters = sk_slabs ? reinterpret_cast<int *>(wsb + at_bytes + bp_bytes + part_bytes) : nullptr;

    ProfCall prof(stream);
    {
        prof.pre_begin();
        if (a_planes == 1 && b_planes == 1 && !b_direct) {
            launch_pack_ab(g.A, g.lda, M, K, At, ldat, g.B, g.ldb, N, Bp, ldbp, counters,
                           int(sk_tiles), dev->sm_count, stream);
        } else if (a_planes == 1) {
            dim3 pgrid(unsigned(std::min<long long>((K + 63) / 64, 1LL << 20)),
                       unsigned(std::min<long long>((M + 63) / 64, 65535)));
            sg::pack_a_transpose_kernel<<<pgrid, 256, 0, stream>>>(g.A, g.lda, M, K, At, ldat,
                                                                   counters, int(sk_tiles));
            g_launches.fetch_add(1);
        }
        for (int z0 = 0; a_planes > 1 && z0 < a_planes; z0 += 65535) {
            const int nz = std::min(a_planes - z0, 65535);
            dim3 pgrid(unsigned(std::min<long long>((K + 63) / 64, 1LL << 20)),
                       unsigned(std::min<long long>((M + 63) / 64, 65535)), unsigned(nz));
            sg::pack_a_transpose_batched_kernel<<<pgrid, 256, 0, stream>>>(
                g.A + (long long)z0 * g.stride_a, g.lda, g.stride_a, M, K,
                At + (long long)z0 * at_plane, ldat, at_plane, z0 == 0 ? counters : nullptr,
                z0 == 0 ? int(sk_tiles) : 0);
            g_launches.fetch_add(1);
        }
        if (!b_direct && !(a_planes == 1 && b_planes == 1)) {
            dim3 bgrid(unsigned(std::min<long long>((N + 255) / 256, 64)),
                       unsigned(std::min<long long>(K, 65535)),
                       unsigned(std::min(b_planes, 65535)));
            sg::pack_b_copy_kernel<<<bgrid, 256, 0, stream>>>(g.B, g.ldb, g.stride_b, K, N, Bp,
                                                              ldbp, bp_plane, b_planes);
            g_launches.fetch_add(1);
        }
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) {
        cudaFreeAsync(ws, stream);
        return cuda_fail(e);
    }

    // the batched kernel takes 3-D tensor maps, the others 2-D maps (a tall
    // batch's B: batch*K rows, or K when every batch shares it)
    CUtensorMap tmA, tmB;
    if (tall) {
        const long long b_rows = b_planes > 1 ? (long long)g.batch * K : K;
        if ((st = encode_2d(&tmA, At, m_rows, K, ldat, var.bm, var.bk)) == SGEMM_OK)
            st = encode_2d(&tmB, Bp, N, b_rows, ldbp, var.bn, var.bk);
    } else if (batched) {
        if ((st = encode_3d(&tmA, At, M, K, a_planes, ldat, at_plane, var.bm, var.bk)) == SGEMM_OK)
            st = encode_3d(&tmB, Bp, N, K, b_planes, ldbp, b_planes > 1 ? bp_plane : K * ldbp,
                           var.bn, var.bk);
    } else {
        if ((st = encode_2d(&tmA, At, M, K, ldat, var.bm, var.bk)) == SGEMM_OK)
            st = encode_2d(&tmB, Bp, N, K, ldbp, var.bn, var.bk);
    }
    if (st != SGEMM_OK) {
        cudaFreeAsync(ws, stream);
        return st;
    }

    sg::MainParams p;
    p.C = g.C;
    p.ldc = g.ldc;
    p.M = int(m_rows);
    p.N = N;
    p.K = K;
    p.alpha = g.alpha;
    p.beta = g.beta;
    p.tiles_m = int(tiles_m);
    p.tiles_n = int(tiles_n);
    // a tall batch's raster groups are its batches (TallBatchConfig)
    p.group_m = tall ? M / var.bm : var.group_m;
    p.c_vec4 = aligned16(g.C) ? 1 : 0;
    p.timeout_ns = g_timeout_ns.load();
    p.dp_tiles = int(dp_tiles);
    p.sk_slabs = sk_slabs;
    p.partials = partials;
    p.counters = counters;
    sg::ExParams x = ex_params(g, a_planes, b_planes);
    if (tall) {
        x.batch = 1;
        x.a_planes = 1;
        x.b_planes = 1;
        x.tall_b_rows = b_planes > 1 ? K : 0;
    }
    prof.main_begin();
    var.launch(grid, stream, tmA, tmB, p, x);
    t_last_kernel = var.name;
    prof.main_end();
    g_launches.fetch_add(1);
    e = cudaGetLastError();
    cudaError_t ef = cudaFreeAsync(ws, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    if (ef != cudaSuccess) return cuda_fail(ef);
    return SGEMM_OK;
}

int sgemm_device(int M, int N, int K, float alpha, const float *A, int lda, const float *B,
                 int ldb, float beta, float *C, int ldc, cudaStream_t stream) {
    return gemm_device(plain_call(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc), stream);
}

// ------------------------------------------------------------------ 3xTF32 path
// Split A and B into tf32 hi/lo parts (B transposed, both K-major), then one
// persistent CTA per SM runs three TF32 MMAs per k step (tf32x3.cuh).

// Bh, Bl (N x ldk each): B split and transposed.
int t3_split_b(int N, int K, const float *B, int ldb, float *Bh, float *Bl, long long ldk,
               cudaStream_t stream) {
    dim3 gb(unsigned(std::min<long long>((N + 63) / 64, 1LL << 20)),
            unsigned(std::min<long long>((K + 63) / 64, 65535)));
    sg::t3::split_bt_kernel<<<gb, 256, 0, stream>>>(B, ldb, K, N, Bh, Bl, ldk);
    g_launches.fetch_add(1);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SGEMM_OK : cuda_fail(e);
}

// C = alpha*A*B + beta*C with B already split (Bh, Bl); Ah, Al: M x ldk scratch.
// Waves of `tiles` equal tiles over `slots` CTAs (or CTA pairs), counting a
// last partial wave of at most half the slots as half a wave (it runs as
// half-width tiles).
double t3_waves(long long tiles, long long slots) {
    const long long w = tiles / slots, r = tiles % slots;
    return double(w) + (r == 0 ? 0.0 : (2 * r <= slots ? 0.5 : 1.0));
}

// The CTA-pair kernel (256 x 256 tiles on 2 SMs) against the single-CTA one
// (128 x 256 tiles): the same work per SM and tile, so the waves decide, with
// the pair's faster main loop (about 5 % at 4096^3 and 8192^3, 13 % at
// 16384x16384x512, same box) as the tie-break.  M = 2432, N = 2048 (152
// single tiles, one wave; 80 pair tiles) stays on the single kernel.
bool t3_use_pair(int M, int N, int sms) {
    const long long ts = ((M + 127LL) / 128) * ((N + 255LL) / 256);
    const long long tp = ((M + 255LL) / 256) * ((N + 255LL) / 256);
    return 0.95 * t3_waves(tp, sms / 2) < t3_waves(ts, sms);
}

int t3_run(int M, int N, int K, float alpha, const float *A, int lda, const float *Bh,
           const float *Bl, long long ldk, float beta, float *C, int ldc, float *Ah, float *Al,
           int sm_count, cudaStream_t stream, ProfCall &prof) {
    namespace t3 = sg::t3;
    int st;
    {
        const int vec4 = (aligned16(A) && lda % 4 == 0 && K % 4 == 0) ? 1 : 0;
        dim3 ga(unsigned(std::min<long long>((K + 4095) / 4096, 64)), unsigned(std::min(M, 65535)));
        prof.pre_begin();
        t3::split_a_kernel<<<ga, 256, 0, stream>>>(A, lda, M, K, Ah, Al, ldk, vec4);
        g_launches.fetch_add(1);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    const int forced = g_t3_pair.load();
    const bool pair = sm_count >= 2 && (forced >= 0 ? forced == 1 : t3_use_pair(M, N, sm_count));
    // B boxes: the rows of B^T one CTA copies for a whole tile, and half that
    // for the half-width tiles of the last wave (*2)
    const int b_rows = pair ? t3::P_BN / 2 : t3::BN;
    CUtensorMap mAh, mAl, mBh, mBl, mBh2, mBl2;
    const auto sw = t3::ROW_BYTES == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    if ((st = encode_2d(&mAh, Ah, K, M, ldk, t3::BK, t3::BM, sw)) != SGEMM_OK ||
        (st = encode_2d(&mAl, Al, K, M, ldk, t3::BK, t3::BM, sw)) != SGEMM_OK ||
        (st = encode_2d(&mBh, Bh, K, N, ldk, t3::BK, b_rows, sw)) != SGEMM_OK ||
        (st = encode_2d(&mBl, Bl, K, N, ldk, t3::BK, b_rows, sw)) != SGEMM_OK ||
        (st = encode_2d(&mBh2, Bh, K, N, ldk, t3::BK, b_rows / 2, sw)) != SGEMM_OK ||
        (st = encode_2d(&mBl2, Bl, K, N, ldk, t3::BK, b_rows / 2, sw)) != SGEMM_OK)
        return st;
    t3::Params p;
    p.C = C;
    p.ldc = ldc;
    p.M = M;
    p.N = N;
    p.K = K;
    p.alpha = alpha;
    p.beta = beta;
    const int tile_m = pair ? t3::P_BM : t3::BM, tile_n = pair ? t3::P_BN : t3::BN;
    p.tiles_m = int((M + tile_m - 1) / tile_m);
    p.tiles_n = int((N + tile_n - 1) / tile_n);
    // 2048 rows of C per raster group (16 rows of 128-row tiles, 8 of the
    // pair's 256-row tiles): a wave then covers the fewest distinct A and B
    // panels; measured at 8192^3 on the single-CTA kernel: group 4 3.28 ms,
    // 8 3.18, 12 3.11, 16 3.07, 20 3.10, 32 3.18
    p.group_m = 2048 / tile_m;
    p.timeout_ns = g_timeout_ns.load();
    const long long tiles = (long long)p.tiles_m * p.tiles_n;
    if (tiles > 0x7fffffffLL) return SGEMM_ERR_INVALID_ARG;
    prof.main_begin();
    if (pair) {
        const unsigned pairs = unsigned(std::min<long long>(tiles, sm_count / 2));
        t3::sgemm_3xtf32_pair_kernel<<<2 * pairs, t3::THREADS, t3::P_SMEM_BYTES, stream>>>(
            mAh, mAl, mBh, mBl, mBh2, mBl2, p);
        t_last_kernel = kT3Pair;
    } else {
        const unsigned grid = unsigned(std::min<long long>(tiles, sm_count));
        t3::sgemm_3xtf32_kernel<<<grid, t3::THREADS, t3::SMEM_BYTES, stream>>>(
            mAh, mAl, mBh, mBl, mBh2, mBl2, p);
        t_last_kernel = kT3Single;
    }
    prof.main_end();
    g_launches.fetch_add(1);
    e = cudaGetLastError();
    return e == cudaSuccess ? SGEMM_OK : cuda_fail(e);
}

int sgemm_device_3xtf32(int M, int N, int K, float alpha, const float *A, int lda,
                        const float *B, int ldb, float beta, float *C, int ldc,
                        cudaStream_t stream) {
    int st = checked_args(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta);
    if (st != SGEMM_OK || M == 0 || N == 0) return st;
    DeviceState *dev = nullptr;
    if ((st = device_state(&dev)) != SGEMM_OK) return st;
    if (K == 0 || alpha == 0.0f) return launch_scale(stream, plain_call(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc),
                            dev->sm_count);

    const long long ldk = round_up(K, 4);
    const size_t a_bytes = round_up((long long)M * ldk * 4, 256);
    const size_t b_bytes = round_up((long long)N * ldk * 4, 256);
    void *ws = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, 2 * a_bytes + 2 * b_bytes, dev->pool, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    char *w = static_cast<char *>(ws);
    float *Ah = reinterpret_cast<float *>(w);
    float *Al = reinterpret_cast<float *>(w + a_bytes);
    float *Bh = reinterpret_cast<float *>(w + 2 * a_bytes);
    float *Bl = reinterpret_cast<float *>(w + 2 * a_bytes + b_bytes);
    ProfCall prof(stream);
    prof.pre_begin();
    st = t3_split_b(N, K, B, ldb, Bh, Bl, ldk, stream);
    if (st == SGEMM_OK)
        st = t3_run(M, N, K, alpha, A, lda, Bh, Bl, ldk, beta, C, ldc, Ah, Al, dev->sm_count,
                    stream, prof);
    cudaError_t ef = cudaFreeAsync(ws, stream);
    if (st != SGEMM_OK) return st;
    if (ef != cudaSuccess) return cuda_fail(ef);
    return SGEMM_OK;
}

// ------------------------------------------------------------------ host buffers
// Copy streams of a device, created on first use: one for host->device copies,
// one for device->host copies, so both directions of the host link and the
// GEMM on the caller's stream run at the same time.
struct CopyStreams {
    cudaStream_t h2d = nullptr, d2h = nullptr;
};
CopyStreams g_copy_streams[kMaxDevices];

int copy_streams(CopyStreams **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return SGEMM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lk(g_mutex);
    CopyStreams &c = g_copy_streams[dev];
    if (!c.h2d) {
        if ((e = cudaStreamCreateWithFlags(&c.h2d, cudaStreamNonBlocking)) != cudaSuccess)
            return cuda_fail(e);
        if ((e = cudaStreamCreateWithFlags(&c.d2h, cudaStreamNonBlocking)) != cudaSuccess)
            return cuda_fail(e);
    }
    *out = &c;
    return SGEMM_OK;
}

struct EventSet {
    std::vector<cudaEvent_t> ev;
    cudaEvent_t make() {
        cudaEvent_t e = nullptr;
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return nullptr;
        ev.push_back(e);
        return e;
    }
    ~EventSet() {
        for (cudaEvent_t e : ev) cudaEventDestroy(e);
    }
};

// Row blocks of the host-buffer pipeline: a first block of kEdgeRows rows (the
// first multiply waits only for its own operands), a last one of kLastRows (the
// copy back after the last multiply is short) and blocks of about kMidRows rows
// between them (fewer launches); `uniform`: equal blocks of at least kEdgeRows
// rows, at most 8.  One block when M < 2 * kEdgeRows or when nothing is
// multiplied.  Returns (first row, rows) per block.
constexpr int kEdgeRows = 1024, kMidRows = 2048, kLastRows = 512;
std::vector<std::pair<int, int>> host_row_blocks(int M, bool multiply, bool uniform) {
    std::vector<std::pair<int, int>> b;
    if (!multiply || M < 2 * kEdgeRows) {
        b.emplace_back(0, M);
        return b;
    }
    if (uniform) {
        // equal blocks of at least kEdgeRows rows, at most 8
        const int n = std::min(8, M / kEdgeRows), per = (M + n - 1) / n;
        for (int r0 = 0; r0 < M; r0 += per) b.emplace_back(r0, std::min(per, M - r0));
        return b;
    }
    b.emplace_back(0, kEdgeRows);
    const int rest = M - kEdgeRows;
    if (rest <= kMidRows) {
        b.emplace_back(kEdgeRows, rest);
        return b;
    }
    const int mid = rest - kLastRows;
    const int nmid = (mid + kMidRows - 1) / kMidRows;
    // block starts on multiples of 128 rows, so only the last block can leave
    // a partly filled tile row
    for (int i = 0; i < nmid; ++i) {
        const int r0 = kEdgeRows + int((long long)mid * i / nmid) / 128 * 128;
        const int r1 = i + 1 == nmid ? M - kLastRows
                                     : kEdgeRows + int((long long)mid * (i + 1) / nmid) / 128 * 128;
        b.emplace_back(r0, r1 - r0);
    }
    b.emplace_back(M - kLastRows, kLastRows);
    return b;
}

// The host-buffer GEMM, pipelined over row blocks of A and C (host_row_blocks):
// block i of A (and of C when beta != 0) is copied in on the h2d stream,
// multiplied on the caller's stream while block i+1 is copied in, and copied
// back on the d2h stream while block i+1 is multiplied.  Block 0 is multiplied
// in k-chunks as the matching columns of A and rows of B arrive (B follows
// block 0 chunk by chunk), so the first multiply waits for a quarter of B
// rather than for all of it and for none of C: the first chunk runs with
// beta = 0, later ones accumulate (beta = 1), and beta * C_in is added once
// block 0's C_in has arrived.  `tensor` selects the 3xTF32 path (B is split
// chunk by chunk, each block of A with its GEMM).
int host_gemm(int M, int N, int K, float alpha, const float *A, int lda, const float *B, int ldb,
              float beta, float *C, int ldc, cudaStream_t stream, bool tensor) {
    int st = checked_args(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta);
    if (st != SGEMM_OK || M == 0 || N == 0) return st;
    DeviceState *dev = nullptr;
    if ((st = device_state(&dev)) != SGEMM_OK) return st;
    CopyStreams *cs = nullptr;
    if ((st = copy_streams(&cs)) != SGEMM_OK) return st;

    const bool need_ab = (K > 0 && alpha != 0.0f);
    const bool need_c_in = (beta != 0.0f);
    const long long ldk = round_up(std::max(K, 1), 4);
    const std::vector<std::pair<int, int>> blocks = host_row_blocks(M, need_ab, tensor);
    int max_rows = 0;
    for (const auto &b : blocks) max_rows = std::max(max_rows, b.second);
    // Block 0 in k-chunks when K is long enough for the copies of B to matter.
    // 3xTF32: four equal chunks.  FFMA: a first chunk of K/8 (the first
    // multiply waits only for it) and chunks growing by half after it: a
    // chunk's multiply takes longer than the copy of the next one (at 8192^3
    // 0.28 us against 0.18 us of host link per k), so the copies stay ahead.
    // K = 8192: 1024, 1536, 2304, 3328.
    std::vector<std::pair<int, int>> chunks;   // (k0, kn)
    if (need_ab && K >= 4096 && !tensor) {
        int k0 = 0, kn = int(round_up((K + 7) / 8, 64));
        while (k0 < K) {
            if (K - k0 - kn < kn / 2) kn = K - k0;   // no short last chunk
            chunks.emplace_back(k0, kn);
            k0 += kn;
            kn = int(round_up(kn + kn / 2, 64));
        }
    } else if (need_ab && K >= 4096) {
        const int kc = int(round_up((K + 3) / 4, 64));
        for (int k0 = 0; k0 < K; k0 += kc) chunks.emplace_back(k0, std::min(kc, K - k0));
    } else if (need_ab) {
        chunks.emplace_back(0, K);
    }
    const int kchunks = int(chunks.size());
    // The 3xTF32 path is bound by the host link, not by its first multiply:
    // it keeps equal row blocks and C_in in front of B (the deferred add and
    // the unequal blocks measured 0.4-1.3 % slower there, 2.2 % faster on the
    // FFMA path at 8192^3).
    const bool defer_c_in = kchunks > 1 && need_c_in && !tensor;

    const size_t a_bytes = need_ab ? round_up((long long)M * K * 4, 256) : 0;
    const size_t b_bytes = need_ab ? round_up((long long)K * N * 4, 256) : 0;
    const size_t c_bytes = round_up((long long)M * N * 4, 256);
    // block 0's C_in while its chunks accumulate
    const size_t cin_bytes = defer_c_in ? round_up((long long)blocks[0].second * N * 4, 256) : 0;
    // 3xTF32: split parts of B (2 x N x ldk) and of the largest block of A
    const size_t bs_bytes = (need_ab && tensor) ? round_up((long long)N * ldk * 4, 256) : 0;
    const size_t as_bytes = (need_ab && tensor) ? round_up((long long)max_rows * ldk * 4, 256) : 0;
    const size_t total = a_bytes + b_bytes + c_bytes + cin_bytes + 2 * bs_bytes + 2 * as_bytes;
    void *buf = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&buf, total, dev->pool, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    char *base = static_cast<char *>(buf);
    float *dA = reinterpret_cast<float *>(base);
    float *dB = reinterpret_cast<float *>(base + a_bytes);
    float *dC = reinterpret_cast<float *>(base + a_bytes + b_bytes);
    float *dCin = reinterpret_cast<float *>(base + a_bytes + b_bytes + c_bytes);
    float *Bh = reinterpret_cast<float *>(base + a_bytes + b_bytes + c_bytes + cin_bytes);
    float *Bl = Bh + bs_bytes / 4;
    float *Ah = reinterpret_cast<float *>(base + a_bytes + b_bytes + c_bytes + cin_bytes + 2 * bs_bytes);
    float *Al = Ah + as_bytes / 4;

    EventSet evs;
    auto fail = [&](int code) {
        cudaStreamSynchronize(cs->h2d);
        cudaStreamSynchronize(cs->d2h);
        cudaFreeAsync(buf, stream);
        cudaStreamSynchronize(stream);
        return code;
    };
    cudaEvent_t allocated = evs.make(), done = evs.make();
    if (!allocated || !done) return fail(SGEMM_ERR_CUDA);
    // the copy streams may touch the buffer only after its allocation on `stream`
    if ((e = cudaEventRecord(allocated, stream)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(cs->h2d, allocated, 0)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(cs->d2h, allocated, 0)) != cudaSuccess)
        return fail(cuda_fail(e));
    // copy in on the h2d stream, then make `stream` wait for it
    auto arrive = [&](cudaEvent_t ev) {
        cudaError_t r = cudaEventRecord(ev, cs->h2d);
        return r == cudaSuccess ? cudaStreamWaitEvent(stream, ev, 0) : r;
    };
    auto gemm = [&](int rows, int k, const float *a, const float *b, float *Bhi, float *Blo,
                    float beta_x, float *c) {
        if (!tensor) return sgemm_device(rows, N, k, alpha, a, K, b, N, beta_x, c, N, stream);
        ProfCall prof(stream);
        return t3_run(rows, N, k, alpha, a, K, Bhi, Blo, ldk, beta_x, c, N, Ah, Al,
                      dev->sm_count, stream, prof);
    };
    for (size_t bi = 0; bi < blocks.size(); ++bi) {
        const int r0 = blocks[bi].first, rows = blocks[bi].second;
        cudaEvent_t in = evs.make(), out = evs.make();
        if (!in || !out) return fail(SGEMM_ERR_CUDA);
        const float *a_blk = need_ab ? dA + (size_t)r0 * K : nullptr;
        float *c_blk = dC + (size_t)r0 * N;
        if (bi == 0 && need_ab) {
            // block 0: copy order A_0 chunk, (C_0 unless deferred), B chunk, ...
            for (int c = 0; c < kchunks; ++c) {
                const int k0 = chunks[c].first, kn = chunks[c].second;
                cudaEvent_t chunk = evs.make();
                if (!chunk) return fail(SGEMM_ERR_CUDA);
                e = cudaMemcpy2DAsync(dA + k0, size_t(K) * 4, A + k0, size_t(lda) * 4,
                                      size_t(kn) * 4, size_t(rows), cudaMemcpyHostToDevice, cs->h2d);
                if (e == cudaSuccess && c == 0 && need_c_in && !defer_c_in)
                    e = cudaMemcpy2DAsync(c_blk, size_t(N) * 4, C, size_t(ldc) * 4, size_t(N) * 4,
                                          size_t(rows), cudaMemcpyHostToDevice, cs->h2d);
                if (e == cudaSuccess)
                    e = cudaMemcpy2DAsync(dB + (size_t)k0 * N, size_t(N) * 4, B + (size_t)k0 * ldb,
                                          size_t(ldb) * 4, size_t(N) * 4, size_t(kn),
                                          cudaMemcpyHostToDevice, cs->h2d);
                if (e == cudaSuccess) e = arrive(chunk);
                if (e != cudaSuccess) return fail(cuda_fail(e));
                if (tensor && (st = t3_split_b(N, kn, dB + (size_t)k0 * N, N, Bh + k0, Bl + k0,
                                               ldk, stream)) != SGEMM_OK)
                    return fail(st);
                const float beta_c = c > 0 ? 1.0f : (defer_c_in ? 0.0f : beta);
                if ((st = gemm(rows, kn, a_blk + k0, dB + (size_t)k0 * N, Bh + k0, Bl + k0,
                               beta_c, c_blk)) != SGEMM_OK)
                    return fail(st);
            }
            if (defer_c_in) {
                e = cudaMemcpy2DAsync(dCin, size_t(N) * 4, C, size_t(ldc) * 4, size_t(N) * 4,
                                      size_t(rows), cudaMemcpyHostToDevice, cs->h2d);
                if (e == cudaSuccess) e = arrive(in);
                if (e != cudaSuccess) return fail(cuda_fail(e));
                const long long n = (long long)rows * N;
                const int grid = int(std::min<long long>((n + 255) / 256, (long long)dev->sm_count * 8));
                sg::add_scaled_kernel<<<grid, 256, 0, stream>>>(c_blk, N, dCin, N, rows, N, beta);
                g_launches.fetch_add(1);
                if ((e = cudaGetLastError()) != cudaSuccess) return fail(cuda_fail(e));
            }
        } else {
            // later blocks (all of B already copied) and the no-multiply case
            e = cudaSuccess;
            if (need_ab)
                e = cudaMemcpy2DAsync(dA + (size_t)r0 * K, size_t(K) * 4, A + (size_t)r0 * lda,
                                      size_t(lda) * 4, size_t(K) * 4, size_t(rows),
                                      cudaMemcpyHostToDevice, cs->h2d);
            if (e == cudaSuccess && need_c_in)
                e = cudaMemcpy2DAsync(c_blk, size_t(N) * 4, C + (size_t)r0 * ldc, size_t(ldc) * 4,
                                      size_t(N) * 4, size_t(rows), cudaMemcpyHostToDevice, cs->h2d);
            if (e == cudaSuccess) e = arrive(in);
            if (e != cudaSuccess) return fail(cuda_fail(e));
            st = need_ab ? gemm(rows, K, a_blk, dB, Bh, Bl, beta, c_blk)
                         : sgemm_device(rows, N, K, alpha, nullptr, std::max(1, K), nullptr,
                                        std::max(1, N), beta, c_blk, N, stream);
            if (st != SGEMM_OK) return fail(st);
        }
        e = cudaEventRecord(out, stream);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(cs->d2h, out, 0);
        if (e == cudaSuccess)
            e = cudaMemcpy2DAsync(C + (size_t)r0 * ldc, size_t(ldc) * 4, c_blk, size_t(N) * 4,
                                  size_t(N) * 4, size_t(rows), cudaMemcpyDeviceToHost, cs->d2h);
        if (e != cudaSuccess) return fail(cuda_fail(e));
    }
    // the buffer is freed only after the last copy back
    if ((e = cudaEventRecord(done, cs->d2h)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(stream, done, 0)) != cudaSuccess)
        return fail(cuda_fail(e));
    cudaFreeAsync(buf, stream);
    e = cudaStreamSynchronize(stream);
    return e == cudaSuccess ? SGEMM_OK : cuda_fail(e);
}

// Synchronises `stream`, then reads and clears the device error word of every
// translation unit (each has its own copy, variant.cuh) on the current device.
int read_and_clear_error_word(cudaStream_t stream) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e);
    cudaError_t (*const units[])(unsigned *, bool) = {
        &sgv::unit_error_word, sgv::extra_variants().error_word,
        sgv::staged_variants().error_word, sgv::sweep_variants_a().error_word,
        sgv::sweep_variants_b().error_word, sgv::sweep_variants_c().error_word,
        sgv::tall_variants().error_word};
    unsigned any = 0;
    for (auto word : units) {
        unsigned v = 0;
        if ((e = word(&v, true)) != cudaSuccess) return cuda_fail(e);
        any |= v;
    }
    if (any & sg::ERR_BOUNDS) return SGEMM_ERR_BOUNDS;
    return any ? SGEMM_ERR_TIMEOUT : SGEMM_OK;
}

// ------------------------------------------------------------------ no-allocation path
// Scratch of sgemm_noalloc(): a fixed device array instead of pool memory.  It
// holds the transposed copy of A and, when B does not meet the TMA's 16-byte
// rule, the re-pitched copy of B.  Every device that loads this library keeps
// it (32 MiB) until the process exits.
constexpr size_t kNoAllocScratchFloats = size_t(8) << 20;
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];

struct NoAllocState {
    bool ready = false;
    int status = SGEMM_OK;
    int sm_count = 0;
    float *scratch = nullptr;   // device address of g_noalloc_scratch on this device
};
NoAllocState g_noalloc[kMaxDevices];

// Per-device set-up of the no-allocation path, done on the first call on each
// device with that device current: device checks, kernel attributes and the
// device address of the scratch array.  Allocates nothing.
int noalloc_state(NoAllocState **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return SGEMM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lk(g_mutex);
    NoAllocState &d = g_noalloc[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e);
        if (major != 10 || minor != 3) {
            d.status = SGEMM_ERR_UNSUPPORTED_DEVICE;
        } else {
            if (!g_encode_tiled) {
                void *fn = nullptr;
                cudaDriverEntryPointQueryResult q;
                e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
                if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
                    return cuda_fail(e != cudaSuccess ? e : cudaErrorNotSupported);
                g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
            }
            for (int i = 0; i < variant_count(); ++i)
                if ((e = variant_at(i).set_attr()) != cudaSuccess) return cuda_fail(e);
            for (int i = 0; i < sgv::staged_variants().count; ++i)
                if ((e = sgv::staged_variants().entries[i].set_attr()) != cudaSuccess)
                    return cuda_fail(e);
            // In host code the array's name is only a host-side stand-in: the
            // kernels must be given its device address.
            void *ptr = nullptr;
            if ((e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch)) != cudaSuccess)
                return cuda_fail(e);
            d.scratch = static_cast<float *>(ptr);
            d.status = SGEMM_OK;
        }
        d.ready = true;
    }
    *out = &d;
    return d.status;
}

int sgemm_device_noalloc(int M, int N, int K, float alpha, const float *A, int lda,
                         const float *B, int ldb, float beta, float *C, int ldc,
                         cudaStream_t stream) {
    int st = checked_args(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta);
    if (st != SGEMM_OK || M == 0 || N == 0) return st;
    NoAllocState *dev = nullptr;
    if ((st = noalloc_state(&dev)) != SGEMM_OK) return st;

    if (K == 0 || alpha == 0.0f)
        return launch_scale(stream, plain_call(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc),
                            dev->sm_count);

    const Variant &var = plain_variant(M, N, K, beta, C, ldc, dev->sm_count);
    const long long ldat = round_up(M, 4);
    const bool b_direct = aligned16(B) && (ldb % 4 == 0);
    const long long ldbp = b_direct ? ldb : round_up(N, 4);
    const long long at_floats = round_up((long long)K * ldat, 64);   // 256-byte aligned
    const long long bp_floats = b_direct ? 0 : (long long)K * ldbp;
    if ((unsigned long long)(at_floats + bp_floats) > kNoAllocScratchFloats)
        return SGEMM_ERR_TOO_LARGE;
    float *At = dev->scratch;
    float *Bp = b_direct ? const_cast<float *>(B) : dev->scratch + at_floats;

    if (!b_direct) {
        launch_pack_ab(A, lda, M, K, At, ldat, B, ldb, N, Bp, ldbp, nullptr, 0, dev->sm_count,
                       stream);
    } else {
        dim3 grid(unsigned(std::min<long long>((K + 63) / 64, 1LL << 20)),
                  unsigned(std::min<long long>((M + 63) / 64, 65535)));
        sg::pack_a_transpose_kernel<<<grid, 256, 0, stream>>>(A, lda, M, K, At, ldat, nullptr, 0);
        g_launches.fetch_add(1);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);

    CUtensorMap tmA, tmB;
    if ((st = encode_2d(&tmA, At, M, K, ldat, var.bm, var.bk)) != SGEMM_OK ||
        (st = encode_2d(&tmB, Bp, N, K, ldbp, var.bn, var.bk)) != SGEMM_OK)
        return st;

    sg::MainParams p;
    p.C = C;
    p.ldc = ldc;
    p.M = M;
    p.N = N;
    p.K = K;
    p.alpha = alpha;
    p.beta = beta;
    p.tiles_m = int((M + var.bm - 1) / var.bm);
    p.tiles_n = int((N + var.bn - 1) / var.bn);
    p.group_m = var.group_m;
    p.c_vec4 = aligned16(C) ? 1 : 0;
    p.timeout_ns = g_timeout_ns.load();
    const long long tiles = (long long)p.tiles_m * p.tiles_n;
    const int grid_main = int(std::min<long long>(tiles, (long long)dev->sm_count * var.ctas_per_sm));
    p.dp_tiles = int(tiles);     // whole tiles only: no partial-sum scratch needed
    p.sk_slabs = 0;
    p.partials = nullptr;
    p.counters = nullptr;
    t_last_kernel = var.name;
    var.launch(grid_main, stream, tmA, tmB, p,
               ex_params(plain_call(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc), 1, 1));
    g_launches.fetch_add(1);
    e = cudaGetLastError();
    return e == cudaSuccess ? SGEMM_OK : cuda_fail(e);
}

}  // namespace

// ==================================================================== C ABI
SGEMM_API int sgemm(int M, int N, int K, float alpha, const float *A, int lda, const float *B,
                    int ldb, float beta, float *C, int ldc, sgemm_stream_t stream) {
    return sgemm_device(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                        reinterpret_cast<cudaStream_t>(stream));
}

SGEMM_API int sgemm_ex(int M, int N, int K, float alpha, const float *A, int lda,
                       long long stride_a, const float *B, int ldb, long long stride_b, float beta,
                       float *C, int ldc, long long stride_c, int batch, const float *bias,
                       long long stride_bias, int act, sgemm_stream_t stream) {
    const GemmCall g{M, N, K, alpha, A, lda, stride_a, B, ldb, stride_b, beta, C, ldc, stride_c,
                     batch, bias, stride_bias, act};
    return gemm_device(g, reinterpret_cast<cudaStream_t>(stream));
}

SGEMM_API int sgemm_host(int M, int N, int K, float alpha, const float *A, int lda,
                         const float *B, int ldb, float beta, float *C, int ldc,
                         sgemm_stream_t stream) {
    return host_gemm(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                     reinterpret_cast<cudaStream_t>(stream), false);
}

SGEMM_API int sgemm_host_3xtf32(int M, int N, int K, float alpha, const float *A, int lda,
                                const float *B, int ldb, float beta, float *C, int ldc,
                                sgemm_stream_t stream) {
    return host_gemm(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                     reinterpret_cast<cudaStream_t>(stream), true);
}

SGEMM_API const char *sgemm_status_string(int status) {
    switch (status) {
        case SGEMM_OK: return "SGEMM_OK: success";
        case SGEMM_ERR_INVALID_ARG: return "SGEMM_ERR_INVALID_ARG: invalid size, leading dimension or pointer";
        case SGEMM_ERR_UNSUPPORTED_DEVICE: return "SGEMM_ERR_UNSUPPORTED_DEVICE: the current device is not sm_103";
        case SGEMM_ERR_CUDA: return "SGEMM_ERR_CUDA: a CUDA call failed (see sgemm_last_cuda_error)";
        case SGEMM_ERR_TIMEOUT: return "SGEMM_ERR_TIMEOUT: a bounded in-kernel wait expired";
        case SGEMM_ERR_ALLOC: return "SGEMM_ERR_ALLOC: workspace allocation failed";
        case SGEMM_ERR_TOO_LARGE:
            return "SGEMM_ERR_TOO_LARGE: a size past 2^31 - 65536, or the problem needs more scratch "
                   "than the fixed array of sgemm_noalloc holds";
        case SGEMM_ERR_BOUNDS: return "SGEMM_ERR_BOUNDS: the range-checked build found an index out of range (the access was skipped)";
        default: return "unknown sgemm status";
    }
}

SGEMM_API int sgemm_version(void) { return kVersion; }

SGEMM_API int sgemm_last_cuda_error(void) { return t_last_cuda_error; }

SGEMM_API const char *sgemm_last_kernel(void) { return t_last_kernel; }

SGEMM_API int sgemm_device_status(sgemm_stream_t stream) {
    DeviceState *dev = nullptr;
    int st = device_state(&dev);
    if (st != SGEMM_OK) return st;
    return read_and_clear_error_word(reinterpret_cast<cudaStream_t>(stream));
}

SGEMM_API int sgemm_set_wait_timeout_ns(unsigned long long ns) {
    if (ns < 1000ull) return SGEMM_ERR_INVALID_ARG;
    g_timeout_ns.store(ns);
    return SGEMM_OK;
}

SGEMM_API int sgemm_selftest_wait_timeout(unsigned long long ns, sgemm_stream_t stream_) {
    if (ns < 1000ull || ns > 10000000000ull) return SGEMM_ERR_INVALID_ARG;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    DeviceState *dev = nullptr;
    int st = device_state(&dev);
    if (st != SGEMM_OK) return st;
    // start from a clear error word so the result reflects this launch only
    st = read_and_clear_error_word(stream);
    if (st == SGEMM_ERR_CUDA) return st;
    sg::wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(ns);
    g_launches.fetch_add(1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    return read_and_clear_error_word(stream);
}

SGEMM_API int sgemm_profile_enable(int on) {
    g_prof_on.store(on ? 1 : 0);
    return SGEMM_OK;
}

SGEMM_API int sgemm_profile_collect(double *main_ms, long long *main_launches, double *pack_ms,
                                    long long *pack_launches) {
    std::lock_guard<std::mutex> lk(g_prof_mutex);
    double mm = 0.0, pm = 0.0;
    long long mn = 0, pn = 0;
    int st = SGEMM_OK;
    for (auto &r : g_prof_used) {
        float ms = 0.0f;
        cudaError_t e = cudaEventSynchronize(r.stop);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.start, r.stop);
        if (e != cudaSuccess) {
            st = cuda_fail(e);
        } else if (r.is_main) {
            mm += ms;
            ++mn;
        } else {
            pm += ms;
            ++pn;
        }
        if (r.owns_start) g_prof_free.push_back(r.start);
        if (r.owns_stop) g_prof_free.push_back(r.stop);
    }
    g_prof_used.clear();
    if (main_ms) *main_ms = mm;
    if (main_launches) *main_launches = mn;
    if (pack_ms) *pack_ms = pm;
    if (pack_launches) *pack_launches = pn;
    return st;
}

SGEMM_API long long sgemm_kernel_launch_count(void) { return g_launches.load(); }

SGEMM_API const char *sgemm_config_string(int M, int N, int K) {
    // with a device, its SM count decides between the direct kernels and the
    // tiled ones (as sgemm() does), picks the tile for few-tile shapes, and the
    // text says when the work split leaves the stream-K tail out
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();   // the failure just caused here (no device) is not kept
        sms = 0;
    }
    if (sms > 0 && g_forced_variant.load() < 0 && M > 0 && N > 0 && K > 0) {
        if (small_problem(M, N, K, sms)) return small_kernel_text(small_split(M, N, K, sms));
        if (M <= kSkinnyRows) return kSkinny;
        if (N <= kSkinnyCols) return kSkinnyN;
    }
    const Variant &v = variant_at(pick_variant(M, N, K, sms));
    if (!v.stream_k || M <= 0 || N <= 0) return v.name;
    const long long tiles = ((M + v.bm - 1LL) / v.bm) * ((N + v.bn - 1LL) / v.bn);
    if (sms <= 0 || stream_k_pays(tiles, sms)) return v.name;
    thread_local std::string text;
    text = std::string(v.name) + " (whole tiles only on this device)";
    return text.c_str();
}

SGEMM_API int sgemm_variant_count(void) { return variant_count(); }

SGEMM_API const char *sgemm_variant_name(int id) {
    if (id < 0 || id >= variant_count()) return "";
    return variant_at(id).name;
}

SGEMM_API int sgemm_set_variant(int id) {
    if (id < -1 || id >= variant_count()) return SGEMM_ERR_INVALID_ARG;
    g_forced_variant.store(id);
    return SGEMM_OK;
}

SGEMM_API int sgemm_debug_bounds_checks(void) {
#ifdef SGEMM_DEBUG_BOUNDS
    return 1;
#else
    return 0;
#endif
}

SGEMM_API int sgemm_debug_drop_release(int on) {
    if (on != 0 && on != 1) return SGEMM_ERR_INVALID_ARG;
    g_drop_release.store(on);
    return SGEMM_OK;
}

SGEMM_API int sgemm_set_3xtf32_kernel(int pair) {
    if (pair < -1 || pair > 1) return SGEMM_ERR_INVALID_ARG;
    g_t3_pair.store(pair);
    return SGEMM_OK;
}

SGEMM_API int sgemm_noalloc(int M, int N, int K, float alpha, const float *A, int lda,
                            const float *B, int ldb, float beta, float *C, int ldc,
                            sgemm_stream_t stream) {
    return sgemm_device_noalloc(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                                reinterpret_cast<cudaStream_t>(stream));
}

SGEMM_API int sgemm_3xtf32(int M, int N, int K, float alpha, const float *A, int lda,
                           const float *B, int ldb, float beta, float *C, int ldc,
                           sgemm_stream_t stream) {
    return sgemm_device_3xtf32(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                               reinterpret_cast<cudaStream_t>(stream));
}
