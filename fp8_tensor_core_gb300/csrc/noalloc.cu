// fp8_gemm_nt_noalloc: the small-token SwapAB stream-K GEMM with its scratch
// in a fixed, file-scope device array instead of library-allocated memory.
//
// Some callers cannot let a library call cudaMalloc: a framework whose
// caching allocator must own every device byte (it accounts, pools and
// reuses memory and would be bypassed), or a serving loop that must not take
// cudaMalloc's implicit device-wide synchronisation on its latency path.
// fp8_gemm_nt may allocate its stream-K workspace on first use; this entry
// point never allocates.  It launches the same k_gemm_swap kernel as
// fp8_gemm_nt's SwapAB path, pointing the kernel's stream-K partial tiles
// and arrival counters at g_noalloc_scratch.
// Its configuration differs in one respect: every CTA takes a whole SM (all
// of its shared memory and 512 TMEM columns), while fp8_gemm_nt lets two
// launches share an SM for problems of up to 16 tokens.
//
// The scratch array is FP8G_NOALLOC_SCRATCH_BYTES long and every GPU that
// loads this library holds it until the process exits.  All calls on a
// device share it and it keeps the last call's contents, so each call clears
// the arrival counters (the only part that must start at zero) on its
// stream before the launch; calls that overlap on the GPU (different
// streams, no ordering between them) race on the array and give wrong
// results.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "fp8g.h"
#include "kernels.cuh"

namespace fp8g {
namespace {

static_assert(FP8G_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size must keep 256-byte alignment");

// The scratch itself.  In host code this name is only a stand-in for the
// device symbol; its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FP8G_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDev = 64;
constexpr int64_t kMaxTokens = 256;
constexpr int64_t kDimLimit = (int64_t(1) << 31) - 1;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // bounded-wait limit of these launches (2 s)

std::mutex g_mu;
void *g_scratch_dev[kMaxDev];   // device address of g_noalloc_scratch, per device
int g_sms[kMaxDev];
int g_smem[kMaxDev];

// Once per device, with that device current: look up the scratch array's
// device address and the launch limits.
int setup_device(int dev, void **scratch, int *sms, int *smem)
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_dev[dev]) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&g_sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&g_smem[dev], cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess)
            return FP8G_ERR_CUDA;
        if (major != 10 || minor != 3)
            return FP8G_ERR_UNSUPPORTED;
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
            return FP8G_ERR_CUDA;
        g_scratch_dev[dev] = p;
    }
    *scratch = g_scratch_dev[dev];
    *sms = g_sms[dev];
    *smem = g_smem[dev];
    return FP8G_OK;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                              CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                              CUtensorMapFloatOOBfill);

EncodeFn encoder()
{
    static EncodeFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(p);
    });
    return fn;
}

// [1, rows, k] bytes, box {128, box_rows, 1}, 128-byte swizzle, zero fill.
bool encode(CUtensorMap *m, const void *base, int64_t k, int64_t rows, uint32_t box_rows)
{
    EncodeFn enc = encoder();
    if (!enc)
        return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(rows), 1};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(k),
                                   static_cast<cuuint64_t>(rows) * static_cast<cuuint64_t>(k)};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(kBlockK), box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    std::memset(m, 0, sizeof(*m));
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace fp8g

using namespace fp8g;

extern "C" int fp8_gemm_nt_noalloc(const void *A, const void *B, void *D, int64_t M, int64_t N,
                                   int64_t K, int a_dtype, int b_dtype, cudaStream_t stream)
{
    if (!A || !B || !D)
        return FP8G_ERR_INVALID_ARG;
    if (M <= 0 || N <= 0 || K <= 0 || N > kDimLimit || K > kDimLimit || K % 16 != 0 || N % 8 != 0)
        return FP8G_ERR_INVALID_ARG;
    if ((a_dtype != FP8G_E4M3 && a_dtype != FP8G_E5M2) || (b_dtype != FP8G_E4M3 && b_dtype != FP8G_E5M2))
        return FP8G_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(D)) &
        15u)
        return FP8G_ERR_MISALIGNED;
    if (M > kMaxTokens)
        return FP8G_ERR_UNSUPPORTED;

    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess || count <= 0) {
        cudaGetLastError();
        return FP8G_ERR_NO_DEVICE;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev)
        return FP8G_ERR_CUDA;
    void *scratch = nullptr;
    int sms = 0, smem = 0;
    int st = setup_device(dev, &scratch, &sms, &smem);
    if (st != FP8G_OK)
        return st;

    const int num_kb = static_cast<int>(cdiv(K, kBlockK));
    const int64_t cap = cdiv(M, 16) * 16;             // tokens per chunk (M <= 256: one chunk)
    const int64_t tiles = cdiv(N, kTileM);
    const int grid = static_cast<int>(std::min<int64_t>(sms, tiles * num_kb));
    // Scratch layout: arrival counters (two int32 per epilogue warp, so 8
    // = 32 bytes per 128-row tile), then the stream-K partial tiles (2 per
    // CTA).
    const size_t counter_bytes = swap_counter_bytes(tiles);
    const size_t counter_span = (counter_bytes + 255) & ~static_cast<size_t>(255);
    const size_t ws_bytes = swap_partials_bytes(grid, static_cast<int>(cap));
    if (counter_span + ws_bytes > static_cast<size_t>(FP8G_NOALLOC_SCRATCH_BYTES))
        return FP8G_ERR_UNSUPPORTED;                  // needs more scratch than the fixed array holds

    GemmArgs args;
    std::memset(&args, 0, sizeof(args));
    args.rows_a = static_cast<int32_t>(M);
    args.n = static_cast<int32_t>(N);
    args.k = static_cast<int32_t>(K);
    args.groups = 1;
    args.num_kb = num_kb;
    args.masked_m = nullptr;
    args.d = D;
    args.tile_n = static_cast<int32_t>(cap);
    args.stage_bytes = static_cast<int32_t>(kTileM * kBlockK + cap * kBlockK);
    const int budget = smem - ctl_bytes_for(1) - kSmemAlignPad;
    args.stages = std::max(1, std::min(kMaxStages, budget / args.stage_bytes));
    args.k_splits = 0;                                // stream-K, as fp8_gemm_nt's SwapAB path
    args.tmem_cols = 512;
    args.raster_band = 1;
    args.a_fmt = static_cast<uint32_t>(a_dtype);
    args.b_fmt = static_cast<uint32_t>(b_dtype);
    args.flags = 0;
    args.timeout_ns = kWaitLimitNs;
    unsigned char *base = static_cast<unsigned char *>(scratch);
    args.counters = reinterpret_cast<int32_t *>(base);
    args.workspace = reinterpret_cast<float *>(base + counter_span);

    CUtensorMap tm_w, tm_t;
    args.tok_box = static_cast<int32_t>(M);   // one box of exactly the tokens, as fp8_gemm_nt's SwapAB path
    if (!encode(&tm_w, B, K, N, kTileM) || !encode(&tm_t, A, K, M, static_cast<uint32_t>(args.tok_box)))
        return FP8G_ERR_CUDA;
    args.prefetch_kb = early_prefetch_kb(kTileM * kBlockK, false);
    if (cudaMemsetAsync(args.counters, 0, counter_bytes, stream) != cudaSuccess)
        return FP8G_ERR_CUDA;
    return launch_gemm_swap(tm_w, tm_t, tm_w, tm_t, args, grid, static_cast<size_t>(smem), stream) == cudaSuccess
               ? FP8G_OK
               : FP8G_ERR_CUDA;
}
