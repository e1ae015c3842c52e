// Tensor-core instruction costs on this GPU, measured with the library's own
// PTX wrappers: how often one thread can issue tcgen05.mma (plain
// kind::f8f6f4 and kind::mxf8f6f4.block_scale) on operands resident in shared
// memory, with one or two issuing warps, with and without the stage handshake
// the GEMM kernels run around every K block (wait on a full barrier, fence,
// four MMAs, commit to an empty barrier), for one SM (cta_group::1) and for an
// SM pair (cta_group::2); and how long four warps take to write one block-scale
// set into TMEM.  Every SM runs one CTA (or one CTA of a pair), as the kernels
// do.  The handshake cases can also stream bytes from L2 into shared memory
// with bulk copies completing on the full barriers, as the kernels' operand
// loads do (the MMAs still read the resident operands), to show what that
// traffic costs the MMA stream.  All waits are bounded; a wait that runs out
// sets an error flag.
//
// Build and run (bench.py --mma-microbench does both):
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 \
//        -I fp8_tensor_core_gb300/csrc -o bench_mma bench_mma.cu && ./bench_mma
// Output: one JSON object per line.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

#include "ptx.cuh"

using namespace fp8g;

namespace {

constexpr int kStages = 4;                  // handshake ring (all on the same resident operands)
constexpr int kCopyStages = 3;              // ... with copy traffic (one buffer per stage)
constexpr int kCopyMax = 48 * 1024;         // copy bytes per stage at most
constexpr int kSetCol = 448;                // TMEM column of the scale set (A side 4, B side 8 columns)
constexpr uint64_t kLimitNs = 2000000000ull;  // bound on every wait
constexpr int kThreads = 256;   // warps 0-3 the roles below, warps 4-7 optional scale-set writers

enum Mode : int {
    kPlain = 0,        // one issuer, back-to-back plain MMAs, a commit every 4
    kBlockScaled = 1,  // the same with block-scaled MMAs on a resident scale set
    kPlain2 = 2,       // two issuing warps, each its own accumulator
    kBlockScaled2 = 3,
    kPlainHs = 4,      // one issuer with the stage handshake
    kBlockScaledHs = 5,
    kScaleSetWrite = 6,  // four warps write one scale set (12 columns) into TMEM, repeatedly
};

struct Smem {
    uint8_t a[128 * 128];   // A: 128 rows x 128 bytes of K, 128-byte swizzle atoms
    uint8_t b[256 * 128];   // B: up to 256 rows
    uint8_t copy[kCopyStages][kCopyMax];   // bulk-copy targets (traffic only)
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t commit_sink;   // per-K-block commits nobody waits for
    uint64_t done[2];       // per issuer: all its MMAs completed
    uint64_t set_done;      // scale-set writes: one arrival per warp
    uint32_t tmem_base;
    volatile int stop;      // handshake cases: the MMAs are done (stops the scale-set writers)
};

// %globaltimer with a memory clobber, so that the compiler keeps each read
// in place relative to the barriers around it.
__device__ __forceinline__ uint64_t stamp_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)::"memory");
    return t;
}

__device__ bool warp_wait_bounded(uint32_t bar, uint32_t parity, uint64_t t0, int *flag)
{
    bool ok = true;
    for (;;) {
        const bool got = __all_sync(0xffffffffu, mbar_try_wait(bar, parity) != 0);
        if (got)
            break;
        if (stamp_ns() - t0 > kLimitNs) {
            ok = false;
            break;
        }
    }
    if (!ok && (threadIdx.x & 31) == 0)
        atomicExch(flag, 1);
    return ok;
}

// Bulk copy global -> this CTA's shared memory, completing on an mbarrier.
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ void fill_operands(Smem &s)
{
    // E4M3 1.0 everywhere: values do not change the timing.
    for (int i = threadIdx.x; i < static_cast<int>((sizeof(s.a) + sizeof(s.b)) / 16); i += blockDim.x)
        reinterpret_cast<uint4 *>(s.a)[i] = make_uint4(0x38383838u, 0x38383838u, 0x38383838u, 0x38383838u);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Each warp writes its own lane quadrant of the scale set: A side (4 columns)
// and B side (8 columns), UE8M0 127 (= 1.0) in every byte.
__device__ void write_scale_set(uint32_t tmem_base, uint32_t col)
{
    const uint32_t q = static_cast<uint32_t>((threadIdx.x >> 5) & 3) * 32u;
    const uint32_t t = tmem_base + (q << 16) + col;
    const uint32_t one = 0x7F7F7F7Fu;
    tmem_st_32x32b_x4(t, one, one, one, one);
    tmem_st_32x32b_x4(t + 4, one, one, one, one);
    tmem_st_32x32b_x4(t + 8, one, one, one, one);
}

// Four MMAs covering one 128-element K block (K = 32 each), as the kernels
// issue them; `first` zeroes the accumulator.
template <bool kBS>
__device__ __forceinline__ void issue_kblock(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t sets, int kb, bool first)
{
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t acc = (first && k == 0) ? 0u : 1u;
        if constexpr (kBS) {
            const uint32_t id = static_cast<uint32_t>(kb & 3);
            mma_f8f6f4_bs(d, adesc + 2u * k, bdesc + 2u * k, idesc | (id << 4) | (id << 29), sets, sets + 4u, acc);
        } else {
            mma_f8f6f4(d, adesc + 2u * k, bdesc + 2u * k, idesc, acc);
        }
    }
}

template <bool kBS>
__device__ __forceinline__ void issue_kblock_pair(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                  uint32_t sets, int kb, bool first)
{
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t acc = (first && k == 0) ? 0u : 1u;
        if constexpr (kBS) {
            const uint32_t id = static_cast<uint32_t>(kb & 3);
            mma_f8f6f4_bs_pair(d, adesc + 2u * k, bdesc + 2u * k, idesc | (id << 4) | (id << 29), sets, sets + 4u,
                               acc);
        } else {
            mma_f8f6f4_pair(d, adesc + 2u * k, bdesc + 2u * k, idesc, acc);
        }
    }
}

__device__ Smem &carve()
{
    extern __shared__ uint8_t raw[];
    return *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~static_cast<uintptr_t>(1023));
}

// One SM per CTA.  Returns per CTA the nanoseconds from the common start to
// the completion of every MMA (or of every scale-set write).
__global__ void __launch_bounds__(kThreads, 1) k_single(int mode, int n, int iters, int copy_bytes,
                                                        const uint8_t *copy_src, int write_gap_ns, int cols,
                                                        unsigned long long *ns_out, int *flag)
{
    Smem &s = carve();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    fill_operands(s);
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_addr(&s.full[i]), 1);
            mbar_init(smem_addr(&s.empty[i]), 1);
        }
        mbar_init(smem_addr(&s.commit_sink), 1);
        mbar_init(smem_addr(&s.done[0]), 1);
        mbar_init(smem_addr(&s.done[1]), 1);
        mbar_init(smem_addr(&s.set_done), 4);
        s.stop = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 0) {
        tmem_alloc(smem_addr(&s.tmem_base), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = s.tmem_base;
    write_scale_set(tb, kSetCol);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const bool bs = mode == kBlockScaled || mode == kBlockScaled2 || mode == kBlockScaledHs;
    const int issuers = (mode == kPlain2 || mode == kBlockScaled2) ? 2 : 1;
    const uint32_t idesc = bs ? make_idesc_bs(0, 0, 128, static_cast<uint32_t>(n), 0)
                              : make_idesc(0, 0, 128, static_cast<uint32_t>(n));
    const uint64_t adesc = smem_desc_k_sw128(smem_addr(s.a));
    const uint64_t bdesc = smem_desc_k_sw128(smem_addr(s.b));
    // handshake cases: accumulator and scale-set columns (cols = acc << 16 | set; 0: 0 and kSetCol)
    const uint32_t acc_col = static_cast<uint32_t>(cols) >> 16;
    const uint32_t set_col = (cols & 0xFFFF) ? static_cast<uint32_t>(cols & 0xFFFF) : static_cast<uint32_t>(kSetCol);
    if (set_col != kSetCol) {
        write_scale_set(tb, set_col);
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    const uint32_t sets = tb + set_col;
    __shared__ unsigned long long t_start;
    if (threadIdx.x == 0)
        t_start = stamp_ns();
    __syncthreads();
    const uint64_t t0 = t_start;

    if (mode == kScaleSetWrite && warp < 4) {
        // Each round: every warp writes its quadrant (tcgen05.st + wait::st),
        // orders it before the arrive and arrives; all four then wait for the
        // round's four arrivals, as an MMA issuer waiting for the set would.
        for (int i = 0; i < iters; ++i) {
            write_scale_set(tb, kSetCol + static_cast<uint32_t>((i & 1) * 16));
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_addr(&s.set_done));
            if (!warp_wait_bounded(smem_addr(&s.set_done), static_cast<uint32_t>(i & 1), t0, flag))
                break;
        }
    } else if (mode == kPlainHs || mode == kBlockScaledHs) {
        const int stages = copy_bytes > 0 ? kCopyStages : kStages;
        if (warp == 0) {
            // producer: passes each stage on once the MMAs released it, after
            // copying copy_bytes from L2 into the stage's buffer (if any)
            int st = 0;
            uint32_t ph = 0;
            const uint8_t *src = copy_src + static_cast<size_t>(blockIdx.x % 16) * kCopyMax * kCopyStages;
            for (int i = 0; i < iters; ++i) {
                if (!warp_wait_bounded(smem_addr(&s.empty[st]), ph ^ 1u, t0, flag))
                    break;
                if (lane == 0) {
                    const uint32_t fb = smem_addr(&s.full[st]);
                    if (copy_bytes > 0) {
                        mbar_arrive_expect_tx(fb, static_cast<uint32_t>(copy_bytes));
                        for (int off = 0; off < copy_bytes; off += 16384) {
                            const int len = copy_bytes - off < 16384 ? copy_bytes - off : 16384;
                            bulk_copy(smem_addr(s.copy[st] + off), src + static_cast<size_t>(st) * kCopyMax + off,
                                      static_cast<uint32_t>(len), fb);
                        }
                    } else {
                        mbar_arrive(fb);
                    }
                }
                __syncwarp();
                if (++st == stages) {
                    st = 0;
                    ph ^= 1u;
                }
            }
        } else if (warp == 1) {
            int st = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int i = 0; i < iters && ok; ++i) {
                ok = warp_wait_bounded(smem_addr(&s.full[st]), ph, t0, flag);
                if (!ok)
                    break;
                tc_fence_after();
                if (lane == 0) {
                    if (bs)
                        issue_kblock<true>(tb + acc_col, adesc, bdesc, idesc, sets, i, i == 0);
                    else
                        issue_kblock<false>(tb + acc_col, adesc, bdesc, idesc, sets, i, i == 0);
                    mma_commit(smem_addr(&s.empty[st]));
                }
                __syncwarp();
                if (++st == stages) {
                    st = 0;
                    ph ^= 1u;
                }
            }
            if (lane == 0)
                mma_commit(smem_addr(&s.done[0]));
            __syncwarp();
            warp_wait_bounded(smem_addr(&s.done[0]), 0, t0, flag);
            if (lane == 0)
                s.stop = 1;
        } else if (warp >= 4 && write_gap_ns > 0) {
            // scale-set writers: every write_gap_ns a set (12 columns per lane
            // quadrant) into TMEM columns the MMAs do not read, as staging
            // warps do beside the MMA stream, until the MMAs are done
            for (int i = 0; i < 1000000 && !s.stop; ++i) {
                write_scale_set(tb, kSetCol + 16u + static_cast<uint32_t>((i & 1) * 16));
                __nanosleep(static_cast<unsigned>(write_gap_ns));
                if (stamp_ns() - t0 > kLimitNs)
                    break;
            }
        }
    } else if (warp >= 1 && warp <= issuers) {
        const int me = warp - 1;
        const uint32_t d = tb + static_cast<uint32_t>(me) * (bs ? 224u : 256u);
        const int mine = iters / issuers;
        if (lane == 0) {
            for (int i = 0; i < mine; ++i) {
                if (bs)
                    issue_kblock<true>(d, adesc, bdesc, idesc, sets, i, i == 0);
                else
                    issue_kblock<false>(d, adesc, bdesc, idesc, sets, i, i == 0);
                mma_commit(smem_addr(&s.commit_sink));
            }
            mma_commit(smem_addr(&s.done[me]));
        }
        __syncwarp();
        warp_wait_bounded(smem_addr(&s.done[me]), 0, t0, flag);
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0)
        ns_out[blockIdx.x] = stamp_ns() - t0;
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tb, 512);
    }
}

// SM pairs: the even CTA's warp 1 issues cta_group::2 MMAs (M = 256) that
// read A and half of B from each CTA and write each CTA's TMEM.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    k_pair(int bs, int n, int iters, unsigned long long *ns_out, int *flag)
{
    Smem &s = carve();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool leader = cluster_ctarank() == 0;
    fill_operands(s);
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&s.commit_sink), 1);
        mbar_init(smem_addr(&s.done[0]), 1);
        fence_mbar_init();
    }
    cluster_sync_all();
    if (warp == 0) {
        tmem_alloc_pair(smem_addr(&s.tmem_base), 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = s.tmem_base;
    write_scale_set(tb, kSetCol);
    tc_fence_before();
    cluster_sync_all();   // both CTAs' scale sets written before any pair MMA reads them
    tc_fence_after();
    __shared__ unsigned long long t_start;
    if (threadIdx.x == 0)
        t_start = stamp_ns();
    __syncthreads();
    const uint64_t t0 = t_start;
    if (leader && warp == 1) {
        const uint32_t idesc = bs ? make_idesc_bs(0, 0, 256, static_cast<uint32_t>(n), 0)
                                  : make_idesc(0, 0, 256, static_cast<uint32_t>(n));
        const uint64_t adesc = smem_desc_k_sw128(smem_addr(s.a));
        const uint64_t bdesc = smem_desc_k_sw128(smem_addr(s.b));
        if (lane == 0) {
            for (int i = 0; i < iters; ++i) {
                if (bs)
                    issue_kblock_pair<true>(tb, adesc, bdesc, idesc, tb + kSetCol, i, i == 0);
                else
                    issue_kblock_pair<false>(tb, adesc, bdesc, idesc, tb + kSetCol, i, i == 0);
                mma_commit_pair_mc(smem_addr(&s.commit_sink), 0x3);
            }
            mma_commit_pair_mc(smem_addr(&s.done[0]), 0x3);
        }
        __syncwarp();
    }
    // Both CTAs see the pair's MMAs complete before either releases TMEM or
    // exits; each CTA's warp 1 records when it saw them complete.
    if (warp == 1) {
        warp_wait_bounded(smem_addr(&s.done[0]), 0, t0, flag);
        if (lane == 0)
            ns_out[blockIdx.x] = stamp_ns() - t0;
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc_pair(tb, 512);
    }
}

int check(cudaError_t e, const char *what)
{
    if (e != cudaSuccess) {
        std::fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
        return 1;
    }
    return 0;
}

}  // namespace

int main()
{
    int dev = 0, sms = 0, clk_khz = 0;
    if (check(cudaGetDevice(&dev), "device") || check(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "sms"))
        return 1;
    cudaDeviceGetAttribute(&clk_khz, cudaDevAttrClockRate, dev);
    // Room for the operands, but requested at 200 KB so that no two CTAs
    // share an SM (as in the GEMM kernels, which take it all).
    const size_t smem = 200 * 1024;
    static_assert(sizeof(Smem) + 1024 <= 200 * 1024, "shared memory layout");
    if (check(cudaFuncSetAttribute(k_single, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)),
              "smem") ||
        check(cudaFuncSetAttribute(k_pair, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)),
              "smem"))
        return 1;
    const int grid = sms & ~1;
    unsigned long long *d_ns = nullptr;
    int *d_flag = nullptr;
    uint8_t *d_copy = nullptr;   // L2-resident copy source: 16 CTA slots of kCopyStages x kCopyMax bytes
    if (check(cudaMalloc(&d_ns, sizeof(unsigned long long) * grid), "malloc") ||
        check(cudaMalloc(&d_flag, sizeof(int)), "malloc") || check(cudaMemset(d_flag, 0, sizeof(int)), "memset") ||
        check(cudaMalloc(&d_copy, static_cast<size_t>(16) * kCopyStages * kCopyMax), "malloc") ||
        check(cudaMemset(d_copy, 0x38, static_cast<size_t>(16) * kCopyStages * kCopyMax), "memset"))
        return 1;
    const int iters = 4096;   // K blocks: 16384 MMAs per issuing CTA
    const char *names[] = {"plain", "block_scaled", "plain", "block_scaled", "plain", "block_scaled", "scale_set_write"};

    auto report = [&](const char *kind, int cta_group, int issuers, bool handshake, int n, long long units,
                      const char *unit, int copy_bytes = 0, int write_gap = 0, int cols = 0) -> int {
        if (check(cudaDeviceSynchronize(), kind))
            return 1;
        unsigned long long h[512] = {};
        int flag = 0;
        cudaMemcpy(h, d_ns, sizeof(unsigned long long) * grid, cudaMemcpyDeviceToHost);
        cudaMemcpy(&flag, d_flag, sizeof(int), cudaMemcpyDeviceToHost);
        unsigned long long worst = 0;
        for (int i = 0; i < grid; ++i)
            worst = h[i] > worst ? h[i] : worst;
        std::printf("{\"op\": \"%s\", \"cta_group\": %d, \"issuers\": %d, \"handshake\": %s, \"n\": %d, "
                    "\"copy_bytes_per_kblock\": %d, \"set_write_gap_ns\": %d, \"acc_col\": %d, \"set_col\": %d, "
                    "\"ns_per_%s\": %.2f, \"ctas\": %d, \"timed_out\": %s}\n",
                    kind, cta_group, issuers, handshake ? "true" : "false", n, copy_bytes, write_gap, cols >> 16,
                    (cols & 0xFFFF) ? (cols & 0xFFFF) : kSetCol, unit,
                    static_cast<double>(worst) / static_cast<double>(units), grid, flag ? "true" : "false");
        std::fflush(stdout);
        return flag;
    };

    // one SM per CTA
    // copy bytes per K block with the handshake: 0, an SM pair's per-SM operand
    // bytes (256 x 256 tile: 16 KB + 16 KB), and a single SM's at 224 / 256
    // columns (16 KB + 28 KB / 32 KB)
    struct Case { int mode, n, copy, write_gap = 0, cols = 0; };
    const Case cases[] = {
        {kPlain, 32, 0}, {kPlain, 128, 0}, {kPlain, 224, 0}, {kPlain, 256, 0},
        {kBlockScaled, 32, 0}, {kBlockScaled, 128, 0}, {kBlockScaled, 224, 0}, {kBlockScaled, 256, 0},
        {kPlain2, 128, 0}, {kPlain2, 224, 0}, {kBlockScaled2, 128, 0}, {kBlockScaled2, 224, 0},
        {kPlainHs, 224, 0}, {kPlainHs, 256, 0}, {kBlockScaledHs, 224, 0}, {kBlockScaledHs, 256, 0},
        {kPlainHs, 256, 32768}, {kPlainHs, 224, 45056}, {kPlainHs, 256, 49152},
        {kBlockScaledHs, 224, 45056}, {kBlockScaledHs, 256, 49152},
        // with four warps writing a scale set into other TMEM columns every ~1 us
        {kPlainHs, 224, 0, 1000}, {kBlockScaledHs, 224, 0, 1000}, {kBlockScaledHs, 224, 0, 250},
        // TMEM placement: accumulator at column 224, scale set at 460 / 472 (the tile kernel's)
        {kBlockScaledHs, 224, 0, 0, (224 << 16) | 448}, {kBlockScaledHs, 224, 0, 0, 460},
        {kBlockScaledHs, 224, 0, 0, 472}, {kBlockScaledHs, 224, 0, 0, (224 << 16) | 460},
        {kPlainHs, 224, 0, 0, (224 << 16) | 448},
    };
    for (const Case &c : cases) {
        for (int rep = 0; rep < 2; ++rep) {   // the first run warms up
            k_single<<<grid, kThreads, smem>>>(c.mode, c.n, iters, c.copy, d_copy, c.write_gap, c.cols, d_ns, d_flag);
            if (check(cudaGetLastError(), "launch"))
                return 1;
            if (rep == 0) {
                if (check(cudaDeviceSynchronize(), "warm-up"))
                    return 1;
                continue;
            }
            const int issuers = (c.mode == kPlain2 || c.mode == kBlockScaled2) ? 2 : 1;
            const bool hs = c.mode == kPlainHs || c.mode == kBlockScaledHs;
            if (report(names[c.mode], 1, issuers, hs, c.n, 4LL * iters, "mma", c.copy, c.write_gap, c.cols))
                return 2;
        }
    }
    for (int rep = 0; rep < 2; ++rep) {
        k_single<<<grid, kThreads, smem>>>(kScaleSetWrite, 0, iters, 0, d_copy, 0, 0, d_ns, d_flag);
        if (check(cudaGetLastError(), "launch"))
            return 1;
        if (rep == 1 && report(names[kScaleSetWrite], 1, 4, true, 0, iters, "set"))
            return 2;
        if (rep == 0 && check(cudaDeviceSynchronize(), "warm-up"))
            return 1;
    }
    // SM pairs
    for (int bs = 0; bs < 2; ++bs) {
        for (int n : {128, 224, 256}) {
            for (int rep = 0; rep < 2; ++rep) {
                k_pair<<<grid, kThreads, smem>>>(bs, n, iters, d_ns, d_flag);
                if (check(cudaGetLastError(), "launch"))
                    return 1;
                if (rep == 0) {
                    if (check(cudaDeviceSynchronize(), "warm-up"))
                        return 1;
                    continue;
                }
                if (report(bs ? "block_scaled" : "plain", 2, 1, false, n, 4LL * iters, "mma"))
                    return 2;
            }
        }
    }
    std::printf("{\"sm_clock_mhz_attr\": %d}\n", clk_khz / 1000);
    cudaFree(d_copy);
    cudaFree(d_ns);
    cudaFree(d_flag);
    return 0;
}
