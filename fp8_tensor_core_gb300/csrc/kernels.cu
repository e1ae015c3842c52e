// FP8 GEMM kernels for sm_103a (GB300).
//
// All three kernels are persistent (one CTA, or CTA pair, per SM, looping
// over work units) and warp-specialised:
//   warp 0      loader: TMA copies of 128-byte K slices into a ring of
//               shared-memory stages (full/empty mbarrier pairs);
//   warp 1      MMA issuer: one thread issues tcgen05.mma kind::f8f6f4 into
//               a TMEM accumulator (two accumulators, so the epilogue of one
//               unit overlaps the main loop of the next);
//   warps 2-5   epilogue: tcgen05.ld TMEM -> registers, FP32 -> BF16 (round
//               to nearest even, or the fused epilogue), stores to D;
// and, in the block-scaled instantiations (kind::mxf8f6f4 with UE8M0 scale
// factors in TMEM),
//   warp 6      a second MMA issuer taking alternate K blocks into its own
//               accumulator, where TMEM has room;
//   warps 7-10  scale staging: each writes the scale sets into its TMEM lane
//               quadrant with tcgen05.st.
//
// k_gemm_mn    tokens (A) on the MMA M side (128-row tiles), weights (B) on
//              N (tile_n columns).  Dense, or grouped with a valid-row count
//              per group (masked or contiguous layout).
// k_gemm_mn2   dense, 256-row tiles on an SM pair (tcgen05 cta_group::2).
// k_gemm_swap  SwapAB: weights (B) on the M side (128 weight rows), tokens
//              (A) on N with a per-unit runtime N = valid tokens rounded up
//              to 16, written into the instruction descriptor.  Stream-K
//              work split with a deterministic K-ordered reduction of the
//              partial tiles.
//
// Sources: "DeepGEMM：基于 Hopper Tensor Core 的 FP8 矩阵乘法内核优化实践"
// (sheratonhq.com/news/187119) §3.3 (producer/consumer warp roles), §4.3
// (multi-stage ring), §6.2-6.4 (K tails clipped exactly, no wrap-around);
// "一次“转置”，半张算力：DeepSeek SwapAB 漂流史" (hwcomputing.csdn.net)
// §1.1 (TMEM 128 lanes x 512 columns, lane m holds row m; M in {64,128} for
// one CTA, N a multiple of 8 up to 256 and writable at run time), §3.2
// (swap operand roles), §3.3 (instruction-descriptor N set to the valid
// tokens; the first MMA of a tile does not accumulate), §3.5 (epilogue
// walks TMEM columns = tokens).
//
// Every barrier wait is bounded (GemmArgs::timeout_ns).  When a wait runs
// out the block records FP8G_ERR_TIMEOUT, every role leaves its loop, the
// loader waits (bounded) for the copies it issued, the MMA issuer waits
// (bounded) for its tensor-core work, TMEM is freed and the block returns.
#include <atomic>

#include <cuda_bf16.h>

#include "fp8g.h"
#include "kernels.cuh"
#include "ptx.cuh"

namespace fp8g {

// Per-device status word: {code, block, role, detail}.  First error wins.
__device__ int32_t g_status[4];

__device__ __forceinline__ void record_status(int32_t code, int32_t role, int32_t detail)
{
    if (atomicCAS(&g_status[0], 0, code) == 0) {
        g_status[1] = static_cast<int32_t>(blockIdx.x);
        g_status[2] = role;
        g_status[3] = detail;
        __threadfence();
    }
}

struct alignas(16) SmemCtl {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint64_t pair_exit;   // CTA-pair kernel: the peer's "done" arrival
    uint64_t sffull[kMaxStages];    // this CTA's scale bytes of stage s (or of ring slot s) landed
    uint64_t sffree[kMaxSfSets];    // TMEM scale set no longer read by any MMA
    uint64_t sfset_ready[kMaxSfSets];   // scale set written into TMEM by the staging warps
    uint64_t sfslot_free[kSfRingSlots];  // scale ring slot read by the staging warps (single-SM tiles)
    uint64_t drain2;                // SwapAB: completion of the second issuer's tensor-core work
    uint64_t peer_done;             // CTA-pair kernel (even CTA): the odd CTA's loader has stopped
    volatile int32_t peer_issued;   // ... after issuing this many stage fills
    uint32_t tmem_base;
    volatile int32_t abort;
    int32_t units_total;
    int32_t pad_;
    int32_t *group_prefix;   // [groups + 1] work units before group g (after this struct)
    int32_t *group_m;        // [groups] valid token rows of group g, clamped
    int32_t *group_row0;     // [groups] output row of group g's first token row
};
static_assert(sizeof(SmemCtl) <= kCtlFixedBytes, "control block too large");
static_assert(kSfRingSlots <= kMaxStages && kSfRingSlots <= 32, "scale ring barriers and slot masks");

// Warp-uniform bounded wait on an mbarrier phase.  Returns false when the
// block is aborting (another role timed out) or this wait ran out.
// kCluster: acquire at cluster scope (the phase is completed by the peer CTA).
template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, SmemCtl &ctl,
                                          uint64_t timeout_ns, int role, int detail)
{
    auto test = [&]() { return kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
    if (__all_sync(0xffffffffu, test()))
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (__all_sync(0xffffffffu, test()))
            return true;
        if ((it & 15u) == 0) {
            int stop = 0;
            if ((threadIdx.x & 31) == 0) {
                if (ctl.abort) {
                    stop = 1;
                } else if (globaltimer_ns() - t0 > timeout_ns) {
                    stop = 1;
                    ctl.abort = 1;
                    record_status(FP8G_ERR_TIMEOUT, role, detail);
                }
            }
            if (__shfl_sync(0xffffffffu, stop, 0))
                return false;
        }
    }
}

// Single thread: poll a global counter (acquire) until it reaches `target`;
// false if that takes longer than timeout_ns.
__device__ __forceinline__ bool wait_count_at_least(const int32_t *p, int target, uint64_t timeout_ns)
{
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        int v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
        if (v >= target)
            return true;
        if (globaltimer_ns() - t0 > timeout_ns)
            return false;
    }
}

// Bounded wait that ignores the abort flag (used while draining).
// kCluster: acquire at cluster scope (the phase is completed by the peer CTA).
template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait_drain(uint32_t bar, uint32_t parity, uint64_t timeout_ns)
{
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (__all_sync(0xffffffffu, kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)))
            return true;
        int late = 0;
        if ((threadIdx.x & 31) == 0)
            late = (globaltimer_ns() - t0 > timeout_ns) ? 1 : 0;
        if (__shfl_sync(0xffffffffu, late, 0))
            return false;
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo_bits, uint32_t hi_bits)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
    return *reinterpret_cast<uint32_t *>(&v);
}

// ---- output scales -------------------------------------------------------------
// D = bf16(sa * sb * acc): "the scale is computed beforehand and multiplied
// back at the output" (DeepGEMM page, §3.1), per tensor or per channel
// (§5.2).  In FP32: (acc * row_factor) * column_factor.

// Factor that is constant along an output row of the token operand (output
// row grow, in group g): sa(grow) or sa(g), times sb(g) when B's scale is per
// tensor.
__device__ __forceinline__ float row_factor(const GemmArgs &a, int g, int64_t grow)
{
    float f = 1.0f;
    if (a.scale_a)
        f = __ldg(a.scale_a + (a.sa_per_row ? grow : static_cast<int64_t>(g)));
    if (a.scale_b && !a.sb_per_col)
        f *= __ldg(a.scale_b + g);
    return f;
}

// Eight accumulator values (bits) of columns col..col+7, times `rf` and, with
// per-column B scales, times sb(g, col + i); packed to eight BF16.
__device__ __forceinline__ uint4 scale_pack8(const GemmArgs &a, const uint32_t *v, float rf, int g, int col)
{
    float f[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        f[i] = __uint_as_float(v[i]) * rf;
    if (a.scale_b && a.sb_per_col) {
        const float4 *p = reinterpret_cast<const float4 *>(a.scale_b + static_cast<int64_t>(g) * a.n + col);
        const float4 x = __ldg(p), y = __ldg(p + 1);
        f[0] *= x.x;
        f[1] *= x.y;
        f[2] *= x.z;
        f[3] *= x.w;
        f[4] *= y.x;
        f[5] *= y.y;
        f[6] *= y.z;
        f[7] *= y.w;
    }
    uint4 o;
    o.x = pack_bf16x2(__float_as_uint(f[0]), __float_as_uint(f[1]));
    o.y = pack_bf16x2(__float_as_uint(f[2]), __float_as_uint(f[3]));
    o.z = pack_bf16x2(__float_as_uint(f[4]), __float_as_uint(f[5]));
    o.w = pack_bf16x2(__float_as_uint(f[6]), __float_as_uint(f[7]));
    return o;
}

// ---- fused epilogue ---------------------------------------------------------------
// "DeepGEMM：基于 Hopper Tensor Core 的 FP8 矩阵乘法内核优化实践" §3.3: alpha * AB
// + beta * C + per-channel bias and an optional ReLU inside the GEMM's
// epilogue, with a choice of rounding for the final conversion.

__device__ __forceinline__ uint16_t bf16_bits_rounded(float x, int mode)
{
    __nv_bfloat16 h;
    switch (mode) {
    case 1: h = __float2bfloat16_rz(x); break;
    case 2: h = __float2bfloat16_ru(x); break;
    case 3: h = __float2bfloat16_rd(x); break;
    default: h = __float2bfloat16_rn(x); break;
    }
    return __bfloat16_as_ushort(h);
}

__device__ __forceinline__ float epi_value(const GemmArgs &a, float v, float c, float b)
{
    float x = fmaf(a.alpha, v, fmaf(a.beta, c, b));
    if (a.relu && x < 0.0f)
        x = 0.0f;
    return x;
}

// Eight scaled products of output row `row` (row of the [groups * rows_a]
// output), columns col..col+7 of group g, through the fused epilogue.
__device__ __forceinline__ uint4 epi_pack8(const GemmArgs &a, const float *f, int g, int64_t row, int col)
{
    float c[8], b[8];
    if (a.c_in) {
        const uint4 cv = *reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(a.c_in) +
                                                          row * a.n + col);
        const uint32_t w[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            c[2 * i] = __uint_as_float(w[i] << 16);
            c[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            c[i] = 0.0f;
    }
    if (a.bias) {
        const float4 *p = reinterpret_cast<const float4 *>(a.bias + static_cast<int64_t>(g) * a.n + col);
        const float4 x = __ldg(p), y = __ldg(p + 1);
        b[0] = x.x; b[1] = x.y; b[2] = x.z; b[3] = x.w;
        b[4] = y.x; b[5] = y.y; b[6] = y.z; b[7] = y.w;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            b[i] = 0.0f;
    }
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        o[i] = static_cast<uint32_t>(bf16_bits_rounded(epi_value(a, f[2 * i], c[2 * i], b[2 * i]), a.round_mode)) |
               (static_cast<uint32_t>(bf16_bits_rounded(epi_value(a, f[2 * i + 1], c[2 * i + 1], b[2 * i + 1]),
                                                        a.round_mode))
                << 16);
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Output of eight accumulator values (bits) of output row `grow` (group g) at
// columns col..col+7: output scales, then the fused epilogue or a plain
// round-to-nearest-even.
__device__ __forceinline__ uint4 out_pack8(const GemmArgs &a, const uint32_t *v, float rf, int g, int64_t grow,
                                           int col)
{
    if (!a.epi)
        return scale_pack8(a, v, rf, g, col);
    float f[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        f[i] = __uint_as_float(v[i]) * rf;
    if (a.scale_b && a.sb_per_col) {
        const float4 *p = reinterpret_cast<const float4 *>(a.scale_b + static_cast<int64_t>(g) * a.n + col);
        const float4 x = __ldg(p), y = __ldg(p + 1);
        f[0] *= x.x; f[1] *= x.y; f[2] *= x.z; f[3] *= x.w;
        f[4] *= y.x; f[5] *= y.y; f[6] *= y.z; f[7] *= y.w;
    }
    return epi_pack8(a, f, g, grow, col);
}

// Eight FP32 accumulator values (bits) rounded to nearest even and packed.
__device__ __forceinline__ uint4 plain_pack8(const uint32_t *v)
{
    return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                      pack_bf16x2(v[6], v[7]));
}

// Kernels are instantiated with and without the scale / fused-epilogue store
// path, so that the plain GEMM carries none of its code.
template <bool kEpi>
__device__ __forceinline__ uint4 store_pack8(const GemmArgs &a, const uint32_t *v, float rf, int g, int64_t grow,
                                             int col)
{
    if constexpr (kEpi)
        return out_pack8(a, v, rf, g, grow, col);
    else
        return plain_pack8(v);
}

// Transpose the 8x8 blocks held by each group of 8 lanes: lane 8g+t holds
// x[i] = row t, column i of its group's block on entry and x[i] = row i,
// column t on return.  Three butterfly stages of shuffles, each exchanging
// the off-diagonal halves at one bit of the lane index.
__device__ __forceinline__ void transpose8x8(uint32_t (&x)[8])
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int m = 4; m >= 1; m >>= 1) {
        const bool hi = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if ((i & m) == 0) {
                const uint32_t send = hi ? x[i] : x[i | m];
                const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, m);
                if (hi)
                    x[i] = recv;
                else
                    x[i | m] = recv;
            }
        }
    }
}

// Tile epilogue stores.  A warp of the tile kernels holds one output row
// per lane (TMEM lane = row), so 16-byte stores straight from registers
// touch 32 rows per instruction.  Instead each lane packs its row's four
// 8-column groups, and each group of 4 lanes transposes its 4x4 block of
// 16-byte groups: lane 4h+t then holds column group t of the rows of lanes
// 4h..4h+3, and one store instruction writes 8 rows x 64 contiguous bytes.
__device__ __forceinline__ void transpose4x4_u4(uint4 (&x)[4])
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int m = 2; m >= 1; m >>= 1) {
        const bool hi = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if ((i & m) == 0) {
                const uint4 send = hi ? x[i] : x[i | m];
                uint4 recv;
                recv.x = __shfl_xor_sync(0xffffffffu, send.x, m);
                recv.y = __shfl_xor_sync(0xffffffffu, send.y, m);
                recv.z = __shfl_xor_sync(0xffffffffu, send.z, m);
                recv.w = __shfl_xor_sync(0xffffffffu, send.w, m);
                if (hi)
                    x[i] = recv;
                else
                    x[i | m] = recv;
            }
        }
    }
}

// Where lane 4h+t stores: the row start (element offset into D) and
// validity of each row of its group of 4 lanes, gathered once per tile.
struct RowTargets {
    int64_t off[4];
    bool ok[4];
};

__device__ __forceinline__ RowTargets row_targets(int64_t my_off, bool my_ok)
{
    const int base = (threadIdx.x & 31) & ~3;
    RowTargets t;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        t.off[j] = __shfl_sync(0xffffffffu, static_cast<long long>(my_off), base + j);
        t.ok[j] = __shfl_sync(0xffffffffu, my_ok ? 1 : 0, base + j) != 0;
    }
    return t;
}

// All lanes: 32 accumulator columns (bits) v of this lane's row `grow`
// (valid if row_ok), columns col0 .. col0 + 31 of the output.
template <bool kEpi>
__device__ __forceinline__ void store_rows32(const GemmArgs &a, __nv_bfloat16 *dout, const uint32_t *v, float rf,
                                             int g, int64_t grow, bool row_ok, int col0, const RowTargets &t)
{
    const int lane = threadIdx.x & 31;
    uint4 p[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int col = col0 + 8 * j;
        p[j] = (row_ok && col < a.n) ? store_pack8<kEpi>(a, v + 8 * j, rf, g, grow, col) : make_uint4(0u, 0u, 0u, 0u);
    }
    transpose4x4_u4(p);
    const int col = col0 + 8 * (lane & 3);
    if (col < a.n) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (t.ok[j])
                *reinterpret_cast<uint4 *>(dout + t.off[j] + col) = p[j];
    }
}

// SwapAB output of 16 tokens: on entry lane `lane` of the warp holds
// accumulator values (bits) v[j] of weight row (= output column) col_base +
// lane for tokens tok0+j, j < 16.  Two in-warp 8x8 transposes give lane 8g+t
// the columns col_base + 8g .. +7 of tokens tok0 + t and tok0 + 8 + t, which
// it writes as two 16-byte stores through out_pack8 (scales, fused
// epilogue): 2 store instructions per lane instead of 16 scalar ones.
template <bool kEpi>
__device__ __forceinline__ void swap_store16(const GemmArgs &a, __nv_bfloat16 *dout, const uint32_t (&v)[16],
                                             int g, int64_t grow_tok0, int n_valid, int col_base)
{
    const int lane = threadIdx.x & 31;
    const int t = lane & 7;
    const int col = col_base + 8 * (lane >> 3);
    uint32_t lo[8], hi[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        lo[i] = v[i];
        hi[i] = v[8 + i];
    }
    transpose8x8(lo);
    transpose8x8(hi);
    if (col < a.n) {
        if (t < n_valid) {
            const int64_t grow = grow_tok0 + t;
            *reinterpret_cast<uint4 *>(dout + grow * a.n + col) =
                store_pack8<kEpi>(a, lo, kEpi ? row_factor(a, g, grow) : 1.0f, g, grow, col);
        }
        if (8 + t < n_valid) {
            const int64_t grow = grow_tok0 + 8 + t;
            *reinterpret_cast<uint4 *>(dout + grow * a.n + col) =
                store_pack8<kEpi>(a, hi, kEpi ? row_factor(a, g, grow) : 1.0f, g, grow, col);
        }
    }
}

// ---- block scales --------------------------------------------------------------
// Per-group scales of the K dimension ("DeepGEMM：基于 Hopper Tensor Core 的 FP8
// 矩阵乘法内核优化实践" §5.2, groups of 128 elements) applied by the tensor core
// itself: kind::mxf8f6f4 with one UE8M0 scale factor per row per 32 K
// elements, read from TMEM ("一次“转置”，半张算力：DeepSeek SwapAB 漂流史" §5:
// UE8M0 scales on SM100; §3.4: the A- and B-side scale-factor columns).

// A scale load brings four K groups per row (TMA box {rows, 4}), as bytes
// [group][row].  With 128-element groups (sf_k = 1) one load serves four K
// blocks: it rides with the stage of K block kb when kb is a multiple of 4 or
// the first block of a run, and covers groups (kb & ~3) .. +3; the MMA of
// block kb picks byte kb & 3.  With 32-element groups (sf_k = 4) every K block
// loads groups 4kb .. 4kb+3 and its k-th MMA picks byte k.
__device__ __forceinline__ bool sf_load_at(int kb, int kb_first, int sf_k)
{
    return kb == kb_first || sf_k == 4 || (kb & 3) == 0;
}
__device__ __forceinline__ int sf_first_group(int kb, int sf_k) { return sf_k == 1 ? (kb & ~3) : 4 * kb; }

// ---- block scales written into TMEM by staging warps ---------------------------------
// (All three kernels.)  The scale sets are written by four staging warps
// (tcgen05.st, one TMEM lane quadrant each), which also turn the copied
// bytes into the TMEM layout, and announced on sfset_ready[set] (four
// arrivals); the MMA issuers only wait for a set and retire it.

// Staging warp, all lanes, for scale load j (raw: its bytes, [4][128] of
// side A then [4][box_b] of side B, whose full barrier has passed): build
// one 32-bit word per row (byte g = K group g of the load); if slot_free is
// given, release the bytes' buffer there (one arrival per staging warp);
// wait until every issuer has retired the set's previous contents, write
// the set into this warp's lane quadrant -- row r of side A at lane r % 32,
// column r / 32; side B from column 4 likewise -- and arrive (kPair: on the
// even CTA's barrier, which counts both CTAs' staging warps).  box_b <= 256.
// Returns false when a wait gave up.
// (The set and the retire parity given: TMEM set `set`, waiting for the
// retire phase of parity free_par first if wait_free.)
template <bool kPair = false>
__device__ __forceinline__ bool sf_stage_tmem_set(SmemCtl &ctl, const GemmArgs &a, const uint8_t *raw, int box_b,
                                                  int set, bool wait_free, uint32_t free_par, uint32_t sets_q,
                                                  int set_cols, uint64_t *slot_free = nullptr)
{
    const int lane = threadIdx.x & 31;
    auto word = [](const uint8_t *raw, int box, int r) {
        return static_cast<uint32_t>(raw[r]) | (static_cast<uint32_t>(raw[box + r]) << 8) |
               (static_cast<uint32_t>(raw[2 * box + r]) << 16) | (static_cast<uint32_t>(raw[3 * box + r]) << 24);
    };
    const uint8_t *raw_a = raw;                 // [4][128]
    const uint8_t *raw_b = raw_a + 4 * kTileM;  // [4][box_b]
    uint32_t wa[4], wb[8];
#pragma unroll
    for (int c = 0; c < 4; ++c)
        wa[c] = word(raw_a, kTileM, 32 * c + lane);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const int r = 32 * c + lane;
        wb[c] = r < box_b ? word(raw_b, box_b, r) : 0u;
    }
    if (slot_free) {
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_addr(slot_free));
    }
    if (wait_free && !warp_wait(smem_addr(&ctl.sffree[set]), free_par, ctl, a.timeout_ns, kRoleScales, 400 + set))
        return false;
    tc_fence_after();
    const uint32_t t = sets_q + static_cast<uint32_t>(set * set_cols);
    tmem_st_32x32b_x4(t, wa[0], wa[1], wa[2], wa[3]);
    tmem_st_32x32b_x4(t + 4u, wb[0], wb[1], wb[2], wb[3]);
    if (box_b > 128)
        tmem_st_32x32b_x4(t + 8u, wb[4], wb[5], wb[6], wb[7]);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
        if constexpr (kPair)
            mbar_arrive_cluster(mapa_shared(smem_addr(&ctl.sfset_ready[set]), 0));
        else
            mbar_arrive(smem_addr(&ctl.sfset_ready[set]));
    }
    return true;
}

// Scale load j into TMEM set j % sf_sets.
template <bool kPair = false>
__device__ __forceinline__ bool sf_stage_tmem(SmemCtl &ctl, const GemmArgs &a, const uint8_t *raw, int box_b,
                                              int j, uint32_t sets_q, int set_cols, uint64_t *slot_free = nullptr)
{
    const int R = a.sf_sets;
    return sf_stage_tmem_set<kPair>(ctl, a, raw, box_b, j % R, j >= R, static_cast<uint32_t>((j / R - 1) & 1), sets_q,
                                    set_cols, slot_free);
}

// MMA issuer warp, all lanes, at scale load j + 1: retire set j (a commit
// that arrives once this thread's MMAs so far are done; kPair: in both
// CTAs), wait for set j + 1 and point set_tmem at it.  Returns false when
// the wait gave up.
template <bool kPair = false>
__device__ __forceinline__ bool sf_next_set(SmemCtl &ctl, const GemmArgs &a, int &j, uint32_t sets_tmem,
                                            int set_cols, uint32_t &set_tmem)
{
    const int R = a.sf_sets;
    if (j >= 0 && (threadIdx.x & 31) == 0) {
        if constexpr (kPair)
            mma_commit_pair_mc(smem_addr(&ctl.sffree[j % R]), 0x3);
        else
            mma_commit(smem_addr(&ctl.sffree[j % R]));
    }
    __syncwarp();
    ++j;
    const int set = j % R;
    if (!warp_wait<kPair>(smem_addr(&ctl.sfset_ready[set]), static_cast<uint32_t>((j / R) & 1), ctl, a.timeout_ns,
                          kRoleMma, 300 + set))
        return false;
    tc_fence_after();
    set_tmem = sets_tmem + static_cast<uint32_t>(set * set_cols);
    return true;
}

// Group table: valid rows per group (clamped to [0, rows_a]) and the
// exclusive prefix of work units.  Run by one warp.
template <typename UnitsFn>
__device__ void build_group_table(SmemCtl &ctl, const GemmArgs &a, UnitsFn units_of)
{
    const int lane = threadIdx.x & 31;
    int running = 0;
    for (int base = 0; base < a.groups; base += 32) {
        const int g = base + lane;
        int cnt = 0;
        if (g < a.groups) {
            int m, r0;
            if (a.group_offsets) {
                // Contiguous layout: rows offsets[g] .. offsets[g+1]-1; a group
                // whose extent is not inside [0, rows_a] is flagged and skipped.
                const int lo = __ldg(a.group_offsets + g), hi = __ldg(a.group_offsets + g + 1);
                if (lo < 0 || hi < lo || hi > a.rows_a) {
                    if (blockIdx.x == 0)
                        record_status(FP8G_ERR_MASKED_M_RANGE, kRoleScheduler, g);
                    m = 0;
                    r0 = 0;
                } else {
                    m = hi - lo;
                    r0 = lo;
                }
            } else {
                m = a.masked_m ? __ldg(a.masked_m + g) : a.rows_a;
                if (m < 0 || m > a.rows_a) {
                    if (blockIdx.x == 0)
                        record_status(FP8G_ERR_MASKED_M_RANGE, kRoleScheduler, g);
                    m = m < 0 ? 0 : a.rows_a;
                }
                r0 = g * a.rows_a;
            }
            ctl.group_m[g] = m;
            ctl.group_row0[g] = r0;
            cnt = units_of(m);
        }
        int x = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o)
                x += y;
        }
        if (g < a.groups)
            ctl.group_prefix[g] = running + x - cnt;
        running += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) {
        ctl.group_prefix[a.groups] = running;
        ctl.units_total = running;
    }
}

// TMA coordinates (row, group) of token row m of group g in A: the 3-D
// [groups, rows_a, k] map, or the contiguous layout's [1, rows_a, k] map.
__device__ __forceinline__ int a_row(const GemmArgs &a, const SmemCtl &ctl, int g, int m)
{
    return a.group_offsets ? ctl.group_row0[g] + m : m;
}
__device__ __forceinline__ int a_grp(const GemmArgs &a, int g) { return a.group_offsets ? 0 : g; }

// Group g with prefix[g] <= u < prefix[g+1].
__device__ __forceinline__ int find_group(const SmemCtl &ctl, int groups, int u)
{
    int lo = 0, hi = groups;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (ctl.group_prefix[mid] <= u)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Shared-memory carve-up common to the kernels: `stages` stages of
// `stage_bytes` starting at a 1024-byte aligned base, the scale ring (if
// any), then the control block.
struct Smem {
    uint8_t *stages;
    uint8_t *sf_ring;
    SmemCtl *ctl;
};

__device__ __forceinline__ Smem carve(uint8_t *raw, const GemmArgs &a)
{
    const uint32_t base = smem_addr(raw);
    const uint32_t pad = (1024u - (base & 1023u)) & 1023u;
    Smem s;
    s.stages = raw + pad;
    s.sf_ring = s.stages + static_cast<size_t>(a.stages) * a.stage_bytes;
    s.ctl = reinterpret_cast<SmemCtl *>(s.sf_ring + static_cast<size_t>(a.sf_ring) * a.sf_slot_bytes);
    int32_t *tables = reinterpret_cast<int32_t *>(reinterpret_cast<uint8_t *>(s.ctl) + kCtlFixedBytes);
    s.ctl->group_prefix = tables;
    s.ctl->group_m = tables + a.groups + 1;
    s.ctl->group_row0 = tables + 2 * a.groups + 1;
    return s;
}

// `issuers`: MMA-issuing threads that each commit to tfull and sffree (1 or 2).
__device__ __forceinline__ void init_barriers(SmemCtl &ctl, int stages, uint32_t issuers = 1)
{
    for (int s = 0; s < stages; ++s) {
        mbar_init(smem_addr(&ctl.full[s]), 1);
        mbar_init(smem_addr(&ctl.empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
        mbar_init(smem_addr(&ctl.tfull[b]), issuers);
        mbar_init(smem_addr(&ctl.tempty[b]), 4 * 32);
    }
    mbar_init(smem_addr(&ctl.drain), 1);
    mbar_init(smem_addr(&ctl.drain2), 1);
    // Scale-byte barriers: one per stage, or per ring slot (single-SM tiles,
    // whatever the stage count).
    const int sf_bars = stages > kSfRingSlots ? stages : kSfRingSlots;
    for (int s = 0; s < sf_bars; ++s)
        mbar_init(smem_addr(&ctl.sffull[s]), 1);
    for (int i = 0; i < kMaxSfSets; ++i) {
        mbar_init(smem_addr(&ctl.sffree[i]), issuers);
        mbar_init(smem_addr(&ctl.sfset_ready[i]), 4);   // one arrival per staging warp
    }
    for (int i = 0; i < kSfRingSlots; ++i)
        mbar_init(smem_addr(&ctl.sfslot_free[i]), 4);   // one arrival per staging warp
    ctl.abort = 0;
    fence_mbar_init();
}

// Loader epilogue: after the last issue, wait until the consumer has
// released every stage (so no tensor-core arrive is still headed for this
// block's shared memory).  When aborting, instead wait for the copies
// still in flight.
__device__ __forceinline__ void loader_tail(SmemCtl &ctl, const GemmArgs &a, int stage,
                                            uint32_t phase, long long issued, bool aborted,
                                            bool dropped_first)
{
    if (!aborted) {
        int st = stage;
        uint32_t ph = phase;
        bool ok = true;
        for (int i = 0; i < a.stages; ++i) {
            if (!warp_wait(smem_addr(&ctl.empty[st]), ph ^ 1u, ctl, a.timeout_ns, kRoleLoader, st)) {
                ok = false;
                break;
            }
            if (++st == a.stages) {
                st = 0;
                ph ^= 1u;
            }
        }
        if (ok)
            return;
        // Another role aborted while copies may still be landing: drain.
    }
    // Aborting: stage s was last filled in the current phase if s < stage,
    // else in the previous one.
    const long long n = issued < a.stages ? issued : a.stages;
    for (int s = 0; s < a.stages; ++s) {
        if (issued <= s && n < a.stages)
            continue;                       // never filled
        if (dropped_first && issued <= a.stages && s == 0)
            continue;                       // its only fill was skipped on purpose
        const uint32_t par = (s < stage) ? phase : (phase ^ 1u);
        warp_wait_drain(smem_addr(&ctl.full[s]), par, a.timeout_ns);
    }
}

// Loader (all lanes), block-scaled kernels: scale bytes complete on their
// own barriers sffull[s], one per stage (SM-pair and SwapAB kernels) or per
// ring slot (single-SM tiles), n_bars of them.  `par` holds, per barrier,
// the parity of the number of scale fills posted, `used` which ever had
// one; wait (bounded) until the last fill of each has landed.  Without an
// abort they all have (the staging warps consumed them).
__device__ __forceinline__ void sf_loader_drain(SmemCtl &ctl, const GemmArgs &a, uint32_t par, uint32_t used,
                                                int n_bars)
{
    for (int s = 0; s < n_bars; ++s)
        if ((used >> s) & 1u)
            warp_wait_drain(smem_addr(&ctl.sffull[s]), ((par >> s) & 1u) ^ 1u, a.timeout_ns);
}

// MMA issuer tail: wait until every tensor-core operation it issued has
// completed, so TMEM can be freed.
__device__ __forceinline__ void mma_drain(SmemCtl &ctl, const GemmArgs &a, bool issued_any,
                                          uint64_t *bar = nullptr)
{
    if (!issued_any)
        return;
    const uint32_t b = smem_addr(bar ? bar : &ctl.drain);
    if ((threadIdx.x & 31) == 0)
        mma_commit(b);
    __syncwarp();
    warp_wait_drain(b, 0, a.timeout_ns);
}

// =====================================================================================
// k_gemm_mn: tokens on M, weights on N.
// =====================================================================================
template <bool kBS, bool kEpi>
__global__ void __launch_bounds__(kBS ? kThreadsTmemScaled : kThreads, 1)
    k_gemm_mn(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
              const __grid_constant__ CUtensorMap tm_sa, const __grid_constant__ CUtensorMap tm_sb,
              const GemmArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    // The tensor maps are kernel parameters, never written by an earlier
    // launch: fetch their descriptors now, while programmatic dependent
    // launch may still hold this CTA before griddepcontrol.wait.
    if (threadIdx.x == 0) {
        tma_prefetch_map(&tm_a);
        tma_prefetch_map(&tm_b);
        if constexpr (kBS) {
            tma_prefetch_map(&tm_sa);
            tma_prefetch_map(&tm_sb);
        }
    }
    const Smem sm = carve(smem_raw, a);
    SmemCtl &ctl = *sm.ctl;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_tiles = ceil_div(a.n, a.tile_n);
    const uint32_t a_bytes = kTileM * kBlockK;                  // 16 KB A box
    // A dense problem of fewer than 128 tokens loads only its rows (a box
    // reaching past the tensor costs the copy engine time for every row it
    // fills); the MMA's other A rows read stale stage bytes and feed only
    // accumulator rows that are never stored.
    const uint32_t a_box_bytes = a.a_box_rows ? static_cast<uint32_t>(a.a_box_rows) * kBlockK : a_bytes;
    const uint32_t tx_bytes = a_box_bytes + static_cast<uint32_t>(a.tile_n) * kBlockK;
    const uint32_t sf_bytes = 4u * static_cast<uint32_t>(kTileM + a.tile_n);
    // Accumulator spacing in TMEM: 256 columns, or tile_n when the block-scale
    // sets follow the accumulators.  With block scales and two MMA issuers,
    // issuer i's accumulator of buffer b sits at column (acc_step * b + i) *
    // tile_n.  With one buffer per issuer (four do not fit, or 256-wide
    // block-scaled tiles) the epilogue of a tile holds the issuers back
    // until it has read it.
    const int acc_stride = kBS ? a.tile_n : kAccStride;
    const int acc_step = (kBS && a.dual_mma) ? 2 : 1;
    const int n_bufs = (kBS && a.acc_bufs == 1) ? 1 : 2;
    const int set_cols = sf_set_cols(a.tile_n);

    if (threadIdx.x == 0)
        init_barriers(ctl, a.stages, static_cast<uint32_t>(acc_step));
    if (warp == 0) {
        // A dense problem's table reads nothing from global memory.
        if (a.prefetch_kb == 0)
            grid_dep_wait();
        build_group_table(ctl, a, [&](int m) { return ceil_div(m, kTileM) * n_tiles; });
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&ctl.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl.tmem_base;
    const int total = ctl.units_total;

    // Unit u -> (group, first row, first column).  Inside a group, bands of
    // raster_band M tiles are walked M-fastest so concurrent CTAs share the
    // same weight tiles and a bounded set of token tiles in L2.
    auto decode = [&](int u, int &g, int &m0, int &n0, int &m_valid) {
        g = find_group(ctl, a.groups, u);
        const int local = u - ctl.group_prefix[g];
        m_valid = ctl.group_m[g];
        const int m_tiles = ceil_div(m_valid, kTileM);
        const int band_units = a.raster_band * n_tiles;
        const int band = local / band_units;
        const int in_band = local - band * band_units;
        const int rows_left = m_tiles - band * a.raster_band;
        const int gm = rows_left < a.raster_band ? rows_left : a.raster_band;
        m0 = (band * a.raster_band + in_band % gm) * kTileM;
        n0 = (in_band / gm) * a.tile_n;
    };

    // Dense problems: fetch the first prefetch_kb K blocks of this CTA's
    // weight tiles into L2 while the previous launch may still run.
    if (a.prefetch_kb > 0 && warp == 2 && lane == 0 && static_cast<int>(blockIdx.x) < a.spare_ctas) {
        // A CTA that may start on an SM this launch leaves idle, while the
        // previous launch still streams: fetch all K blocks of the weight
        // tiles of CTAs blockIdx.x, + spare_ctas, ... into L2, so that the
        // CTAs starting later find their weights there.  (L2 is the point of
        // coherence: the loads after griddepcontrol.wait still see whatever
        // the previous launch wrote.)
        for (int b = blockIdx.x; b < static_cast<int>(gridDim.x); b += a.spare_ctas)
            for (int u = b; u < total; u += gridDim.x) {
                int g, m0, n0, mv;
                decode(u, g, m0, n0, mv);
                for (int kb = 0; kb < a.num_kb; ++kb)
                    tma_prefetch_l2_3d(&tm_b, kb * kBlockK, n0, g);
            }
    } else if (a.prefetch_kb > 0 && warp == 2 && lane == 0) {
        int left = a.prefetch_kb;
        for (int u = blockIdx.x; u < total && left > 0; u += gridDim.x) {
            int g, m0, n0, mv;
            decode(u, g, m0, n0, mv);
            for (int kb = 0; kb < a.num_kb && left > 0; ++kb, --left)
                tma_prefetch_l2_3d(&tm_b, kb * kBlockK, n0, g);
        }
    }
    grid_dep_wait();   // inputs may come from the previous launch in the stream
    if (threadIdx.x == 0)
        grid_dep_launch_dependents();

    // Block scales, two ways.  With a ring (a.sf_ring > 0, 128-element
    // groups) the scale loads form their own sequence, one per scale set --
    // K blocks 0, 4, 8, ... of each of this CTA's tiles -- into a ring of
    // a.sf_ring slots, kept one set ahead of the operands so that the staging
    // warps have written a set into TMEM before its first MMA.  Without one
    // (32-element groups: a set per K block) each K block's scale bytes ride
    // in its stage.
    const bool sf_ring = kBS && a.sf_ring > 0;
    const int sf_step = a.sf_k == 4 ? 1 : 4;
    const int sf_ahead = 1;
    auto sf_advance = [&](int &u, int &kb) {
        kb += sf_step;
        if (kb >= a.num_kb) {
            kb = 0;
            u += gridDim.x;
        }
    };

    if (warp == 0) {
        // ------------------------------- loader -------------------------------
        int stage = 0;
        uint32_t phase = 0;
        long long issued = 0;
        bool aborted = false;
        const bool drop = (a.flags & FP8G_DEBUG_DROP_FIRST_LOAD) && blockIdx.x == 0;
        uint32_t sf_par = 0, sf_used = 0;   // per ring slot (or stage): parity of scale fills posted, any posted
        int sf_u = blockIdx.x, sf_kb = 0;   // next scale load (its tile and first K block)
        int sf_posted = 0, sf_reached = 0;  // scale loads posted; scale sets whose first K block was reached
        int sf_du = -1, sf_g = 0, sf_m0 = 0, sf_n0 = 0;   // the last tile decoded for scale loads
        // Post the next scale load into slot sf_posted % sf_ring, once the
        // staging warps have read that slot's previous load.
        auto sf_post = [&]() -> bool {
            const int slot = sf_posted % a.sf_ring;
            if (sf_posted >= a.sf_ring &&
                !warp_wait(smem_addr(&ctl.sfslot_free[slot]), static_cast<uint32_t>((sf_posted / a.sf_ring - 1) & 1),
                           ctl, a.timeout_ns, kRoleLoader, 600 + slot))
                return false;
            if (sf_u != sf_du) {
                int mv;
                decode(sf_u, sf_g, sf_m0, sf_n0, mv);
                sf_du = sf_u;
            }
            if (lane == 0) {
                const int g = sf_g, m0 = sf_m0, n0 = sf_n0;
                uint8_t *dst = sm.sf_ring + static_cast<size_t>(slot) * a.sf_slot_bytes;
                const uint32_t sb = smem_addr(&ctl.sffull[slot]);
                const int y = sf_first_group(sf_kb, a.sf_k);
                mbar_arrive_expect_tx(sb, sf_bytes);
                tma_load_3d(smem_addr(dst), &tm_sa, sb, m0, y, g);
                tma_load_3d(smem_addr(dst + 4 * kTileM), &tm_sb, sb, n0, y, g);
            }
            __syncwarp();
            sf_par ^= 1u << slot;
            sf_used |= 1u << slot;
            ++sf_posted;
            sf_advance(sf_u, sf_kb);
            return true;
        };
        for (int u = blockIdx.x; u < total && !aborted; u += gridDim.x) {
            int g, m0, n0, mv;
            decode(u, g, m0, n0, mv);
            for (int kb = 0; kb < a.num_kb; ++kb) {
                if (sf_ring && sf_load_at(kb, 0, a.sf_k)) {
                    ++sf_reached;
                    while (sf_posted < sf_reached + sf_ahead && sf_u < total) {
                        if (!sf_post()) {
                            aborted = true;
                            break;
                        }
                    }
                    if (aborted)
                        break;
                }
                if (!warp_wait(smem_addr(&ctl.empty[stage]), phase ^ 1u, ctl, a.timeout_ns,
                               kRoleLoader, stage)) {
                    aborted = true;
                    break;
                }
                const bool sf = kBS && !sf_ring && sf_load_at(kb, 0, a.sf_k) && !(drop && issued == 0);
                if (lane == 0 && !(drop && issued == 0)) {
                    uint8_t *sa = sm.stages + static_cast<size_t>(stage) * a.stage_bytes;
                    const uint32_t fb = smem_addr(&ctl.full[stage]);
                    mbar_arrive_expect_tx(fb, tx_bytes);
                    tma_load_3d(smem_addr(sa), &tm_a, fb, kb * kBlockK, a_row(a, ctl, g, m0), a_grp(a, g));
                    tma_load_3d(smem_addr(sa + a_bytes), &tm_b, fb, kb * kBlockK, n0, g);
                    if (sf) {
                        const uint32_t sb = smem_addr(&ctl.sffull[stage]);
                        const int y = sf_first_group(kb, a.sf_k);
                        mbar_arrive_expect_tx(sb, sf_bytes);
                        tma_load_3d(smem_addr(sa + a.sf_off), &tm_sa, sb, m0, y, g);
                        tma_load_3d(smem_addr(sa + a.sf_off + 4 * kTileM), &tm_sb, sb, n0, y, g);
                    }
                }
                if (sf) {
                    sf_par ^= 1u << stage;
                    sf_used |= 1u << stage;
                }
                __syncwarp();
                ++issued;
                if (++stage == a.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        loader_tail(ctl, a, stage, phase, issued, aborted, drop);
        if constexpr (kBS)
            sf_loader_drain(ctl, a, sf_par, sf_used, sf_ring ? a.sf_ring : a.stages);
    } else if (warp == 1 && !kBS) {
        // ----------------------------- MMA issuer -----------------------------
        const uint32_t idesc = make_idesc(a.a_fmt, a.b_fmt, kTileM, a.tile_n);
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool issued_any = false;
        for (int u = blockIdx.x; u < total; u += gridDim.x) {
            if (!warp_wait(smem_addr(&ctl.tempty[acc]), acc_phase ^ 1u, ctl, a.timeout_ns, kRoleMma,
                           100 + acc))
                break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * acc_stride);
            bool ok = true;
            for (int kb = 0; kb < a.num_kb; ++kb) {
                if (!warp_wait(smem_addr(&ctl.full[stage]), phase, ctl, a.timeout_ns, kRoleMma,
                               stage)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t sa = smem_addr(sm.stages + static_cast<size_t>(stage) * a.stage_bytes);
                    const uint64_t adesc = smem_desc_k_sw128(sa);
                    const uint64_t bdesc = smem_desc_k_sw128(sa + a_bytes);
#pragma unroll
                    for (int k = 0; k < kBlockK / 32; ++k) {
                        // +32 bytes of K per instruction = +2 in the address field
                        mma_f8f6f4(d_tmem, adesc + 2u * k, bdesc + 2u * k, idesc,
                                   (kb | k) != 0 ? 1u : 0u);
                    }
                    mma_commit(smem_addr(&ctl.empty[stage]));
                }
                __syncwarp();
                issued_any = true;
                if (++stage == a.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok)
                break;
            if (lane == 0)
                mma_commit(smem_addr(&ctl.tfull[acc]));
            __syncwarp();
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        mma_drain(ctl, a, issued_any);
    } else if (kBS && (warp == 1 || (warp == 6 && a.dual_mma))) {
        // ---------------------- MMA issuers, block-scaled ----------------------
        // As in the SwapAB kernel: one or two issuing threads (warps 1 and
        // 6); with two, issuer i takes the K blocks whose running index in
        // this CTA is i mod 2, into its own accumulator, and the epilogue
        // adds the two.  Scale sets come from the staging warps.
        const int me = warp == 1 ? 0 : 1;
        const uint32_t idesc_bs = make_idesc_bs(a.a_fmt, a.b_fmt, kTileM, a.tile_n, 0);
        const uint32_t sets_tmem = tmem_base + static_cast<uint32_t>(a.sf_col0);
        uint32_t set_tmem = sets_tmem;
        int j = -1;   // scale loads passed
        int stage = 0;
        uint32_t phase = 0;
        uint32_t par = 0;   // running K-block index mod 2
        int acc = 0;
        uint32_t acc_phase = 0;
        bool issued_any = false;
        bool ok = true;
        const bool lean = acc_step == 1 && a.sf_k == 1;
        if (lean) {
            // One issuer, 128-element groups: a scale set covers four K
            // blocks.  The loop is kept as short as the plain kernel's: at a
            // set switch the retire commit, then the waits for the new set
            // and for the operands behind one tensor fence, the set's TMEM
            // slot and phase kept by increment (no division).
            const int R = a.sf_sets;
            int cur = -1;            // TMEM scale set in use
            int nxt = 0;             // the next one
            uint32_t rpar = 0;       // parity of its ready phase
            for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
                if (!warp_wait(smem_addr(&ctl.tempty[acc]), acc_phase ^ 1u, ctl, a.timeout_ns, kRoleMma,
                               100 + acc))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * acc_stride);
                for (int kb = 0; kb < a.num_kb; ++kb) {
                    if ((kb & 3) == 0) {
                        if (cur >= 0 && lane == 0)
                            mma_commit(smem_addr(&ctl.sffree[cur]));
                        cur = nxt;
                        if (!warp_wait(smem_addr(&ctl.sfset_ready[cur]), rpar, ctl, a.timeout_ns, kRoleMma,
                                       300 + cur)) {
                            ok = false;
                            break;
                        }
                        if (++nxt == R) {
                            nxt = 0;
                            rpar ^= 1u;
                        }
                        set_tmem = sets_tmem + static_cast<uint32_t>(cur * set_cols);
                    }
                    if (!warp_wait(smem_addr(&ctl.full[stage]), phase, ctl, a.timeout_ns, kRoleMma, stage)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t sa = smem_addr(sm.stages + static_cast<size_t>(stage) * a.stage_bytes);
                        const uint64_t adesc = smem_desc_k_sw128(sa);
                        const uint64_t bdesc = smem_desc_k_sw128(sa + a_bytes);
                        const uint32_t id = static_cast<uint32_t>(kb & 3);
                        const uint32_t idesc = idesc_bs | (id << 4) | (id << 29);
#pragma unroll
                        for (int k = 0; k < kBlockK / 32; ++k)
                            mma_f8f6f4_bs(d_tmem, adesc + 2u * k, bdesc + 2u * k, idesc, set_tmem, set_tmem + 4u,
                                          (kb | k) != 0 ? 1u : 0u);
                        mma_commit(smem_addr(&ctl.empty[stage]));
                    }
                    __syncwarp();
                    issued_any = true;
                    if (++stage == a.stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                if (lane == 0)
                    mma_commit(smem_addr(&ctl.tfull[acc]));
                __syncwarp();
                if (++acc == n_bufs) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
        }
        for (int u = blockIdx.x; !lean && u < total && ok; u += gridDim.x) {
            if (!warp_wait(smem_addr(&ctl.tempty[acc]), acc_phase ^ 1u, ctl, a.timeout_ns, kRoleMma,
                           100 + acc))
                break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>((acc * acc_step + me) * acc_stride);
            bool first = true;
            for (int kb = 0; kb < a.num_kb; ++kb) {
                if (sf_load_at(kb, 0, a.sf_k) && !sf_next_set(ctl, a, j, sets_tmem, set_cols, set_tmem)) {
                    ok = false;
                    break;
                }
                if (acc_step == 1 || static_cast<int>(par) == me) {
                    if (!warp_wait(smem_addr(&ctl.full[stage]), phase, ctl, a.timeout_ns, kRoleMma, stage)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t sa = smem_addr(sm.stages + static_cast<size_t>(stage) * a.stage_bytes);
                        const uint64_t adesc = smem_desc_k_sw128(sa);
                        const uint64_t bdesc = smem_desc_k_sw128(sa + a_bytes);
#pragma unroll
                        for (int k = 0; k < kBlockK / 32; ++k) {
                            const uint32_t id = a.sf_k == 1 ? static_cast<uint32_t>(kb & 3) : static_cast<uint32_t>(k);
                            mma_f8f6f4_bs(d_tmem, adesc + 2u * k, bdesc + 2u * k, idesc_bs | (id << 4) | (id << 29),
                                          set_tmem, set_tmem + 4u, (!first || k != 0) ? 1u : 0u);
                        }
                        mma_commit(smem_addr(&ctl.empty[stage]));
                    }
                    __syncwarp();
                    first = false;
                    issued_any = true;
                }
                par ^= 1u;
                if (++stage == a.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok)
                break;
            if (lane == 0)
                mma_commit(smem_addr(&ctl.tfull[acc]));
            __syncwarp();
            if (++acc == n_bufs) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        mma_drain(ctl, a, issued_any, me == 0 ? &ctl.drain : &ctl.drain2);
    } else if (kBS && warp >= 7) {
        // --------------------- block-scale staging into TMEM ---------------------
        // Warps 7-10, one per TMEM lane quadrant: scale load j becomes TMEM
        // scale set j (sf_stage_tmem).  From a ring slot (j % sf_ring),
        // released as soon as its bytes are in registers; else from the stage
        // of the set's K block.
        if constexpr (kBS) {
            const uint32_t sets_q = tmem_base + static_cast<uint32_t>(a.sf_col0) +
                                    (static_cast<uint32_t>((warp & 3) * 32) << 16);
            int su = blockIdx.x, skb = 0;
            int stage = 0;
            uint32_t st_par = 0;   // per stage: parity of the next scale fill to wait for
            // Load j's ring slot (j % sf_ring) with its fill parity, and its
            // TMEM set (j % sf_sets) with j / sf_sets, kept by increment.
            int slot = 0, set = 0;
            uint32_t slot_par = 0, gen = 0;
            for (int j = 0; su < total; ++j) {
                if (sf_ring) {
                    if (!warp_wait(smem_addr(&ctl.sffull[slot]), slot_par, ctl, a.timeout_ns, kRoleScales,
                                   700 + slot) ||
                        !sf_stage_tmem_set(ctl, a, sm.sf_ring + static_cast<size_t>(slot) * a.sf_slot_bytes, a.tile_n,
                                           set, gen > 0, (gen & 1u) ^ 1u, sets_q, set_cols, &ctl.sfslot_free[slot]))
                        break;
                    if (++slot == a.sf_ring) {
                        slot = 0;
                        slot_par ^= 1u;
                    }
                } else {
                    // every K block carries a scale load (32-element groups):
                    // the sets follow the stages one to one
                    if (!warp_wait(smem_addr(&ctl.sffull[stage]), (st_par >> stage) & 1u, ctl, a.timeout_ns,
                                   kRoleScales, stage) ||
                        !sf_stage_tmem_set(ctl, a, sm.stages + static_cast<size_t>(stage) * a.stage_bytes + a.sf_off,
                                           a.tile_n, set, gen > 0, (gen & 1u) ^ 1u, sets_q, set_cols))
                        break;
                    st_par ^= 1u << stage;
                    if (++stage == a.stages)
                        stage = 0;
                }
                if (++set == a.sf_sets) {
                    set = 0;
                    ++gen;
                }
                sf_advance(su, skb);
            }
        }
    } else if (warp >= 2 && warp <= 5) {
        // ------------------------------ epilogue ------------------------------
        const int q = warp & 3;  // TMEM lane quadrant this warp may read
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t par = 0;   // running K-block index mod 2 (which issuer took a tile's first K block)
        __nv_bfloat16 *dout = static_cast<__nv_bfloat16 *>(a.d);
        for (int u = blockIdx.x; u < total; u += gridDim.x) {
            int g, m0, n0, mv;
            decode(u, g, m0, n0, mv);
            if (!warp_wait(smem_addr(&ctl.tfull[acc]), acc_phase, ctl, a.timeout_ns, kRoleEpilogue,
                           200 + acc))
                break;
            tc_fence_after();
            const int row = m0 + q * 32 + lane;
            const bool row_ok = row < mv;
            const int64_t grow = static_cast<int64_t>(ctl.group_row0[g]) + row;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(acc * acc_step * acc_stride);
            const uint32_t t_first = t_row + par * static_cast<uint32_t>(acc_stride);
            const uint32_t t_second = t_row + (par ^ 1u) * static_cast<uint32_t>(acc_stride);
            const bool both = acc_step == 2 && a.num_kb >= 2;
            if (acc_step == 2)
                par ^= static_cast<uint32_t>(a.num_kb & 1);
            const float rf = (kEpi && row_ok) ? row_factor(a, g, grow) : 1.0f;
            const RowTargets tg = row_targets(grow * static_cast<int64_t>(a.n), row_ok);
            for (int c = 0; c < a.tile_n; c += 32) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_first + static_cast<uint32_t>(c), r);
                if constexpr (kBS) {
                    if (both) {
                        uint32_t r2[32];
                        tmem_ld_32x32b_x32(t_second + static_cast<uint32_t>(c), r2);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            r[i] = __float_as_uint(__uint_as_float(r[i]) + __uint_as_float(r2[i]));
                    }
                }
                store_rows32<kEpi>(a, dout, r, rf, g, grow, row_ok, n0 + c, tg);
            }
            tc_fence_before();
            mbar_arrive(smem_addr(&ctl.tempty[acc]));
            if (++acc == n_bufs) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// =====================================================================================
// k_gemm_mn2: dense, tokens on M, two SMs per tile (tcgen05 cta_group::2).
//
// A cluster of two CTAs computes 256 x tile_n output tiles.  Each CTA loads
// its own 128 token rows and half of the tile's weight rows into its shared
// memory; the even CTA issues one 256-row MMA that reads A from both CTAs and
// B from both halves, so each weight byte is read from shared memory once
// for two SMs' worth of tensor-core work.  Each CTA's TMEM holds its own 128
// output rows and its own epilogue writes them.
//
// Work split: whole tiles round-robin over the pairs (so concurrent pairs
// work on neighbouring tiles and share operands in L2).  With k_splits != 1
// only the complete waves go that way; the tiles of the last, partial wave
// are split stream-K: their K blocks are laid end to end and every pair
// takes an equal contiguous range.  A partial segment publishes FP32
// partials (each CTA its own 128 rows) and the contributor completing a tile
// sums them in K order and writes BF16.
//
// Barriers: full[s] lives in the even CTA (both CTAs' copies complete on it,
// the even CTA's producer posts the byte count for both); empty[s] and
// tfull[b] receive multicast commits in both CTAs; tempty[b] (even CTA)
// counts the four epilogue warps of both CTAs.
// =====================================================================================
struct PairSeg {
    int tile, m0, n0, kb0, kb1;
    int kind;   // 0: first segment of the pair's range, 1: a later one
    int g, mv;  // group and its valid rows (dense: 0 and M)
};

template <bool kBS, bool kEpi>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kBS ? kThreadsTmemScaled : kThreads, 1)
    k_gemm_mn2(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
               const __grid_constant__ CUtensorMap tm_sa, const __grid_constant__ CUtensorMap tm_sb,
               const GemmArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    // The tensor maps are kernel parameters, never written by an earlier
    // launch: fetch their descriptors now, while programmatic dependent
    // launch may still hold this CTA before griddepcontrol.wait.
    if (threadIdx.x == 0) {
        tma_prefetch_map(&tm_a);
        tma_prefetch_map(&tm_b);
        if constexpr (kBS) {
            tma_prefetch_map(&tm_sa);
            tma_prefetch_map(&tm_sb);
        }
    }
    const Smem sm = carve(smem_raw, a);
    SmemCtl &ctl = *sm.ctl;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int half_n = a.tile_n / 2;
    const int n_tiles = ceil_div(a.n, a.tile_n);
    const int m_tiles = ceil_div(a.rows_a, 2 * kTileM);
    // Grouped problems (masked or contiguous layout): 256-row tiles inside
    // each group, counted by the group table built on the device; whole
    // tiles only.
    const bool grouped = a.groups > 1 || a.masked_m != nullptr || a.group_offsets != nullptr;
    int total = m_tiles * n_tiles;
    const int num_kb = a.num_kb;
    const bool stream_k = a.k_splits != 1;
    const uint32_t a_bytes = kTileM * kBlockK;                          // own 128 token rows
    const uint32_t tx_pair = 2u * (a_bytes + static_cast<uint32_t>(half_n) * kBlockK);
    // Block scales: each CTA loads its own 128 rows' A-side scales and the
    // whole tile's B-side scales (each CTA's tensor core scales all N
    // columns), completing on its own sffull barrier.  Accumulators are then
    // tile_n columns apart, followed by the scale sets.
    const uint32_t sf_bytes = 4u * static_cast<uint32_t>(kTileM + a.tile_n);
    const int acc_stride = kBS ? a.tile_n : kAccStride;
    // Two MMA issuers in the even CTA (warps 1 and 6, alternate K blocks,
    // one accumulator each; one buffer each when four do not fit in TMEM).
    const int acc_step = (kBS && a.dual_mma) ? 2 : 1;
    const int n_bufs = (kBS && a.acc_bufs == 1) ? 1 : 2;
    const int set_cols = sf_set_cols(a.tile_n);
    const int cid = blockIdx.x >> 1;
    const int ncl = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(smem_addr(&ctl.full[s]), 1);
            mbar_init(smem_addr(&ctl.empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_addr(&ctl.tfull[b]), static_cast<uint32_t>(acc_step));
            mbar_init(smem_addr(&ctl.tempty[b]), 2 * 4);
        }
        mbar_init(smem_addr(&ctl.drain), 1);
        mbar_init(smem_addr(&ctl.drain2), 1);
        mbar_init(smem_addr(&ctl.pair_exit), 1);
        mbar_init(smem_addr(&ctl.peer_done), 1);
        ctl.peer_issued = 0;
        if constexpr (kBS) {
            for (int s = 0; s < a.stages; ++s)
                mbar_init(smem_addr(&ctl.sffull[s]), 1);
            for (int i = 0; i < kMaxSfSets; ++i) {
                mbar_init(smem_addr(&ctl.sffree[i]), static_cast<uint32_t>(acc_step));
                mbar_init(smem_addr(&ctl.sfset_ready[i]), 2 * 4);   // both CTAs' staging warps (even CTA's copy)
            }
        }
        ctl.abort = 0;
        fence_mbar_init();
    }
    // Both CTAs' barriers must exist before any copy, commit or arrive
    // crosses the pair.
    cluster_sync_all();
    if (warp == 1) {
        tmem_alloc_pair(smem_addr(&ctl.tmem_base), kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    grid_dep_wait();   // inputs may come from the previous launch in the stream
    if (threadIdx.x == 0)
        grid_dep_launch_dependents();
    const uint32_t tmem_base = ctl.tmem_base;
    if (grouped) {
        if (warp == 0)
            build_group_table(ctl, a, [&](int m) { return ceil_div(m, 2 * kTileM) * n_tiles; });
        __syncthreads();
        total = ctl.units_total;
    }
    // Whole-tile waves, and the K blocks of the remaining tiles [sk0, sk0 + T)
    // split into P equal ranges: over every pair (k_splits == 0, stream-K),
    // or k_splits ranges per remaining tile (k_splits >= 2: each tile of the
    // last partial wave is split k_splits ways along K).
    const int dp_tiles = stream_k && !grouped ? (total / ncl) * ncl : total;
    const long long sk0 = static_cast<long long>(dp_tiles) * num_kb;
    const long long T = static_cast<long long>(total - dp_tiles) * num_kb;
    long long P = T < static_cast<long long>(ncl) ? T : static_cast<long long>(ncl);
    if (a.k_splits >= 2) {
        const long long want = static_cast<long long>(a.k_splits) * (total - dp_tiles);
        P = want < P ? want : P;
    }

    // Only called when T > 0 (a stream-K segment exists).
    auto range_begin = [&](long long c) { return sk0 + c * T / P; };
    auto pair_of = [&](long long x) { return static_cast<int>(((x - sk0 + 1) * P - 1) / T); };
    // A pair's work: its range [pos0, end) of the split K blocks (empty if
    // none; at most two pieces, as a range never exceeds a tile's K blocks)
    // and whole tiles cid, cid + ncl, ... below dp_tiles.  Order: first the
    // range's piece that ends inside a tile (a tile's K-earlier part: a later
    // contributor will add it), then one whole tile, then the range's piece
    // that finishes a tile (its contributor then finds the earlier parts
    // published long ago and sums them while its MMA issuer runs the next
    // whole tile), then the remaining whole tiles.  A piece's partial slot
    // is kind 0 if it starts the range, else kind 1.
    struct Walker {
        long long pos0;          // range start
        long long pos, lim;      // later pieces of the range, [pos, lim)
        long long e_lo, e_hi;    // the piece run first, [e_lo, e_hi) (empty if none)
        int u;                   // next whole tile
        int state;
    };
    auto make_walker = [&]() {
        Walker w;
        w.u = cid;
        w.state = 0;
        w.pos0 = w.pos = w.lim = w.e_lo = w.e_hi = 0;
        if (T > 0 && cid < P) {
            const long long b = range_begin(cid), e = range_begin(static_cast<long long>(cid) + 1);
            w.pos0 = w.pos = b;
            w.lim = e;
            if (e % num_kb != 0) {   // the range ends inside a tile: run that piece first
                const long long ts = (e - 1) / num_kb * num_kb;
                w.e_lo = ts > b ? ts : b;
                w.e_hi = e;
                w.lim = w.e_lo;
            }
        }
        return w;
    };
    // Next segment: tile (rasterised in bands of raster_band 256-row tiles,
    // M fastest), this CTA's first row and the tile's first column.
    auto next_seg = [&](Walker &w, PairSeg &x) {
        int u = 0;
        bool found = false;
        auto piece = [&](long long lo, long long hi) {
            u = static_cast<int>(lo / num_kb);
            x.kb0 = static_cast<int>(lo - static_cast<long long>(u) * num_kb);
            x.kb1 = x.kb0 + static_cast<int>(hi - lo);
            x.kind = lo == w.pos0 ? 0 : 1;
            found = true;
        };
        auto whole = [&]() {
            if (w.u >= dp_tiles)
                return;
            u = w.u;
            x.kb0 = 0;
            x.kb1 = num_kb;
            x.kind = 0;
            w.u += ncl;
            found = true;
        };
        if (w.state == 0) {
            w.state = 1;
            if (w.e_hi > w.e_lo)
                piece(w.e_lo, w.e_hi);
        }
        if (!found && w.state == 1) {
            w.state = 2;
            whole();
        }
        if (!found && w.state == 2) {
            if (w.pos < w.lim) {
                const long long tile_end = (w.pos / num_kb + 1) * num_kb;
                const long long hi = w.lim < tile_end ? w.lim : tile_end;
                piece(w.pos, hi);
                w.pos = hi;
            } else {
                w.state = 3;
            }
        }
        if (!found && w.state == 3)
            whole();
        if (!found)
            return false;
        x.tile = u;
        int local = u, mt = m_tiles;
        x.g = 0;
        x.mv = a.rows_a;
        if (grouped) {
            x.g = find_group(ctl, a.groups, u);
            local = u - ctl.group_prefix[x.g];
            x.mv = ctl.group_m[x.g];
            mt = ceil_div(x.mv, 2 * kTileM);
        }
        const int band_units = a.raster_band * n_tiles;
        const int band = local / band_units;
        const int in_band = local - band * band_units;
        const int rows_left = mt - band * a.raster_band;
        const int gm = rows_left < a.raster_band ? rows_left : a.raster_band;
        // group-local first row of this CTA's 128 rows
        x.m0 = (band * a.raster_band + in_band % gm) * (2 * kTileM) + static_cast<int>(rank) * kTileM;
        x.n0 = (in_band / gm) * a.tile_n;
        return true;
    };

    bool aborted = false;
    if (warp == 0) {
        // ------------------------------- loader -------------------------------
        int stage = 0;
        uint32_t phase = 0;
        long long issued = 0;
        uint32_t sf_par = 0, sf_used = 0;   // per stage: parity of scale fills posted, any posted
        const bool drop = (a.flags & FP8G_DEBUG_DROP_FIRST_LOAD) && blockIdx.x == 0;
        Walker wk = make_walker();
        PairSeg x;
        while (!aborted && next_seg(wk, x)) {
            for (int kb = x.kb0; kb < x.kb1; ++kb) {
                if (!warp_wait(smem_addr(&ctl.empty[stage]), phase ^ 1u, ctl, a.timeout_ns,
                               kRoleLoader, stage)) {
                    aborted = true;
                    break;
                }
                if constexpr (kBS) {
                    if (sf_load_at(kb, x.kb0, a.sf_k) && !(drop && issued == 0)) {
                        sf_par ^= 1u << stage;
                        sf_used |= 1u << stage;
                    }
                }
                if (lane == 0 && !(drop && issued == 0)) {
                    uint8_t *sa = sm.stages + static_cast<size_t>(stage) * a.stage_bytes;
                    if (leader)
                        mbar_arrive_expect_tx(smem_addr(&ctl.full[stage]), tx_pair);
                    const uint32_t fb = mapa_shared(smem_addr(&ctl.full[stage]), 0);
                    tma_load_3d_pair(smem_addr(sa), &tm_a, fb, kb * kBlockK, a_row(a, ctl, x.g, x.m0),
                                     a_grp(a, x.g));
                    tma_load_3d_pair(smem_addr(sa + a_bytes), &tm_b, fb, kb * kBlockK,
                                     x.n0 + static_cast<int>(rank) * half_n, x.g);
                    if constexpr (kBS) {
                        if (sf_load_at(kb, x.kb0, a.sf_k)) {
                            const uint32_t sb = smem_addr(&ctl.sffull[stage]);
                            const int y = sf_first_group(kb, a.sf_k);
                            mbar_arrive_expect_tx(sb, sf_bytes);
                            tma_load_3d(smem_addr(sa + a.sf_off), &tm_sa, sb, x.m0, y, 0);
                            tma_load_3d(smem_addr(sa + a.sf_off + 4 * kTileM), &tm_sb, sb, x.n0, y, 0);
                        }
                    }
                }
                __syncwarp();
                ++issued;
                if (++stage == a.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!aborted) {
            // Wait until the pair MMA has released every stage this CTA filled.
            for (int i = 0; i < a.stages; ++i) {
                if (!warp_wait(smem_addr(&ctl.empty[stage]), phase ^ 1u, ctl, a.timeout_ns,
                               kRoleLoader, stage)) {
                    aborted = true;
                    break;
                }
                if (++stage == a.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        // The odd CTA's copies complete on the even CTA's full barriers, so
        // only the even CTA can observe them: the odd CTA reports how many
        // stage fills it issued (it issues none after this).
        if (!leader) {
            if (lane == 0) {
                st_shared_cluster_u32(mapa_shared(smem_addr(const_cast<int32_t *>(&ctl.peer_issued)), 0),
                                      static_cast<uint32_t>(issued));
                mbar_arrive_cluster(mapa_shared(smem_addr(&ctl.peer_done), 0));
            }
            __syncwarp();
        }
        if (aborted && leader) {
            // Stage s's barrier is armed by this CTA (one arrival expecting
            // both CTAs' bytes, its own half copied with it) and filled by the
            // odd CTA's half.  Either side issues round r + 1 only after the
            // MMA consumed round r, so the rounds armed and filled differ by at
            // most one: the pending phase lacks either the odd half (complete
            // it here) or the arrival (post it, expecting only the odd half).
            // Waiting (bounded) for that phase then observes every copy of
            // both CTAs landed.
            long long peer = issued;
            if (warp_wait_drain<true>(smem_addr(&ctl.peer_done), 0, 4 * a.timeout_ns))
                peer = static_cast<long long>(static_cast<uint32_t>(ctl.peer_issued));
            const uint32_t odd_bytes = tx_pair / 2;
            auto rounds = [&](long long n, int s) {
                return n / a.stages + (static_cast<long long>(s) < n % a.stages ? 1 : 0);
            };
            for (int s = 0; s < a.stages; ++s) {
                const long long armed = rounds(issued, s) - ((drop && s == 0 && issued > 0) ? 1 : 0);
                const long long filled = rounds(peer, s);
                const long long last = armed > filled ? armed : filled;
                if (last <= 0)
                    continue;
                const uint32_t fb = smem_addr(&ctl.full[s]);
                if (lane == 0) {
                    if (armed == filled + 1)
                        mbar_complete_tx(fb, odd_bytes);
                    else if (filled == armed + 1)
                        mbar_arrive_expect_tx(fb, odd_bytes);
                }
                __syncwarp();
                warp_wait_drain(fb, static_cast<uint32_t>((last - 1) & 1), a.timeout_ns);
            }
        }
        // Scale bytes complete on each CTA's own barriers.
        if constexpr (kBS)
            sf_loader_drain(ctl, a, sf_par, sf_used, a.stages);
    } else if (warp == 1 && !kBS) {
        // ----------------------------- MMA issuer -----------------------------
        if (leader) {
            const uint32_t idesc = make_idesc(a.a_fmt, a.b_fmt, 2 * kTileM, a.tile_n);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool issued_any = false;
            Walker wk = make_walker();
            PairSeg x;
            while (!aborted && next_seg(wk, x)) {
                if (!warp_wait(smem_addr(&ctl.tempty[acc]), acc_phase ^ 1u, ctl, a.timeout_ns, kRoleMma,
                               100 + acc)) {
                    aborted = true;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * acc_stride);
                for (int kb = x.kb0; kb < x.kb1; ++kb) {
                    if (!warp_wait(smem_addr(&ctl.full[stage]), phase, ctl, a.timeout_ns, kRoleMma,
                                   stage)) {
                        aborted = true;
                        break;
                    }
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t sa = smem_addr(sm.stages + static_cast<size_t>(stage) * a.stage_bytes);
                        const uint64_t adesc = smem_desc_k_sw128(sa);
                        const uint64_t bdesc = smem_desc_k_sw128(sa + a_bytes);
#pragma unroll
                        for (int k = 0; k < kBlockK / 32; ++k)
                            mma_f8f6f4_pair(d_tmem, adesc + 2u * k, bdesc + 2u * k, idesc,
                                            (kb != x.kb0 || k != 0) ? 1u : 0u);
                        mma_commit_pair_mc(smem_addr(&ctl.empty[stage]), 0x3);
                    }
                    __syncwarp();
                    issued_any = true;
                    if (++stage == a.stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (aborted)
                    break;
                if (lane == 0)
                    mma_commit_pair_mc(smem_addr(&ctl.tfull[acc]), 0x3);
                __syncwarp();
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // Both CTAs' epilogues must be done with every accumulator (their
            // arrivals on this CTA's tempty have all landed) before TMEM goes.
            for (int i = 0; i < 2 && !aborted; ++i) {
                if (!warp_wait(smem_addr(&ctl.tempty[acc]), acc_phase ^ 1u, ctl, a.timeout_ns, kRoleMma,
                               100 + acc))
                    aborted = true;
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (issued_any) {
                if (lane == 0)
                    mma_commit_pair(smem_addr(&ctl.drain));
                __syncwarp();
                warp_wait_drain(smem_addr(&ctl.drain), 0, a.timeout_ns);
            }
        }
    } else if (kBS && (warp == 1 || (warp == 6 && a.dual_mma))) {
        // ---------------------- MMA issuers, block-scaled ----------------------
        // Even CTA only: one or two issuing threads (warps 1 and 6).  With
        // two, issuer i takes the K blocks whose running index in this pair
        // is i mod 2, into its own accumulator; the epilogues add the two.
        // Scale sets come from both CTAs' staging warps; a set is retired in
        // both CTAs by a multicast commit.
        if (leader) {
            const int me = warp == 1 ? 0 : 1;
            const uint32_t idesc_bs = make_idesc_bs(a.a_fmt, a.b_fmt, 2 * kTileM, a.tile_n, 0);
            const uint32_t sets_tmem = tmem_base + static_cast<uint32_t>(a.sf_col0);
            uint32_t set_tmem = sets_tmem;
            int j = -1;   // scale loads passed
            int stage = 0;
            uint32_t phase = 0;
            uint32_t par = 0;   // running K-block index mod 2
            int acc = 0;
            uint32_t acc_phase = 0;
            bool issued_any = false;
            Walker wk = make_walker();
            PairSeg x;
            while (!aborted && next_seg(wk, x)) {
                if (!warp_wait(smem_addr(&ctl.tempty[acc]), acc_phase ^ 1u, ctl, a.timeout_ns, kRoleMma,
                               100 + acc)) {
                    aborted = true;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>((acc * acc_step + me) * acc_stride);
                bool first = true;
                for (int kb = x.kb0; kb < x.kb1; ++kb) {
                    if (sf_load_at(kb, x.kb0, a.sf_k) &&
                        !sf_next_set<true>(ctl, a, j, sets_tmem, set_cols, set_tmem)) {
                        aborted = true;
                        break;
                    }
                    if (acc_step == 1 || static_cast<int>(par) == me) {
                        if (!warp_wait(smem_addr(&ctl.full[stage]), phase, ctl, a.timeout_ns, kRoleMma, stage)) {
                            aborted = true;
                            break;
                        }
                        tc_fence_after();
                        if (lane == 0) {
                            const uint32_t sa = smem_addr(sm.stages + static_cast<size_t>(stage) * a.stage_bytes);
                            const uint64_t adesc = smem_desc_k_sw128(sa);
                            const uint64_t bdesc = smem_desc_k_sw128(sa + a_bytes);
#pragma unroll
                            for (int k = 0; k < kBlockK / 32; ++k) {
                                const uint32_t id =
                                    a.sf_k == 1 ? static_cast<uint32_t>(kb & 3) : static_cast<uint32_t>(k);
                                mma_f8f6f4_bs_pair(d_tmem, adesc + 2u * k, bdesc + 2u * k,
                                                   idesc_bs | (id << 4) | (id << 29), set_tmem, set_tmem + 4u,
                                                   (!first || k != 0) ? 1u : 0u);
                            }
                            mma_commit_pair_mc(smem_addr(&ctl.empty[stage]), 0x3);
                        }
                        __syncwarp();
                        first = false;
                        issued_any = true;
                    }
                    par ^= 1u;
                    if (++stage == a.stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (aborted)
                    break;
                if (lane == 0)
                    mma_commit_pair_mc(smem_addr(&ctl.tfull[acc]), 0x3);
                __syncwarp();
                if (++acc == n_bufs) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // Issuer 0: both CTAs' epilogues must be done with every
            // accumulator before TMEM goes.
            for (int i = 0; i < n_bufs && !aborted && me == 0; ++i) {
                if (!warp_wait(smem_addr(&ctl.tempty[acc]), acc_phase ^ 1u, ctl, a.timeout_ns, kRoleMma,
                               100 + acc))
                    aborted = true;
                if (++acc == n_bufs) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (issued_any) {
                uint64_t *db = me == 0 ? &ctl.drain : &ctl.drain2;
                if (lane == 0)
                    mma_commit_pair(smem_addr(db));
                __syncwarp();
                warp_wait_drain(smem_addr(db), 0, a.timeout_ns);
            }
        }
    } else if (kBS && warp >= 7) {
        // --------------------- block-scale staging into TMEM ---------------------
        // Warps 7-10 of each CTA: its own 128 rows' A-side scales and the
        // whole tile's B-side scales (each CTA's tensor core scales all N
        // columns), written into its own TMEM; arrivals go to the even CTA.
        if constexpr (kBS) {
            const uint32_t sets_q = tmem_base + static_cast<uint32_t>(a.sf_col0) +
                                    (static_cast<uint32_t>((warp & 3) * 32) << 16);
            int stage = 0;
            uint32_t sf_par = 0;   // per stage: parity of the next scale fill to wait for
            int j = -1;
            Walker wk = make_walker();
            PairSeg x;
            while (!aborted && next_seg(wk, x)) {
                for (int kb = x.kb0; kb < x.kb1; ++kb) {
                    if (sf_load_at(kb, x.kb0, a.sf_k)) {
                        ++j;
                        if (!warp_wait(smem_addr(&ctl.sffull[stage]), (sf_par >> stage) & 1u, ctl, a.timeout_ns,
                                       kRoleScales, stage) ||
                            !sf_stage_tmem<true>(ctl, a,
                                                 sm.stages + static_cast<size_t>(stage) * a.stage_bytes + a.sf_off,
                                                 a.tile_n, j, sets_q, set_cols)) {
                            aborted = true;
                            break;
                        }
                        sf_par ^= 1u << stage;
                    }
                    if (++stage == a.stages)
                        stage = 0;
                }
            }
        }
    } else if (warp >= 2 && warp <= 5) {
        // ------------------------------ epilogue ------------------------------
        const int q = warp & 3;
        const int row = q * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t par = 0;   // running K-block index mod 2 (which issuer took a segment's first K block)
        __nv_bfloat16 *dout = static_cast<__nv_bfloat16 *>(a.d);
        // Stream-K partial tiles: slot (CTA, kind) of [tile_n/4 column groups]
        // [128 rows][4 columns] FP32; a warp access covers 512 contiguous bytes.
        const int64_t part4 = kTileM * static_cast<int64_t>(a.tile_n) / 4;
        float4 *slots = reinterpret_cast<float4 *>(a.workspace);
        Walker wk = make_walker();
        PairSeg x;
        while (next_seg(wk, x)) {
            if (!warp_wait(smem_addr(&ctl.tfull[acc]), acc_phase, ctl, a.timeout_ns, kRoleEpilogue,
                           200 + acc)) {
                aborted = true;
                break;
            }
            tc_fence_after();
            const int lrow = x.m0 + row;   // row within the group (dense: within D)
            const bool row_ok = lrow < x.mv;
            const int64_t grow = (grouped ? static_cast<int64_t>(ctl.group_row0[x.g]) : int64_t(0)) + lrow;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(acc * acc_step * acc_stride);
            // With two issuers: the one that took the segment's first K block
            // always has data, the other one if the segment has two or more.
            const uint32_t t_first = t_row + par * static_cast<uint32_t>(acc_stride);
            const uint32_t t_second = t_row + (par ^ 1u) * static_cast<uint32_t>(acc_stride);
            const bool both = acc_step == 2 && x.kb1 - x.kb0 >= 2;
            if (acc_step == 2)
                par ^= static_cast<uint32_t>((x.kb1 - x.kb0) & 1);
            // 32 accumulator columns of this thread's row, summed over issuers.
            auto ld32 = [&](int c, uint32_t (&r)[32]) {
                tmem_ld_32x32b_x32(t_first + static_cast<uint32_t>(c), r);
                if constexpr (kBS) {
                    if (both) {
                        uint32_t r2[32];
                        tmem_ld_32x32b_x32(t_second + static_cast<uint32_t>(c), r2);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            r[i] = __float_as_uint(__uint_as_float(r[i]) + __uint_as_float(r2[i]));
                    }
                }
            };
            const float rf = (kEpi && row_ok) ? row_factor(a, x.g, grow) : 1.0f;
            const RowTargets tg = row_targets(grow * static_cast<int64_t>(a.n), row_ok);
            if (x.kb0 == 0 && x.kb1 == num_kb) {
                for (int c = 0; c < a.tile_n; c += 32) {
                    uint32_t r[32];
                    ld32(c, r);
                    store_rows32<kEpi>(a, dout, r, rf, x.g, grow, row_ok, x.n0 + c, tg);
                }
            } else {
                // Contributors of this tile: the pairs whose ranges meet it,
                // in K order.  Pairs after the first start their range inside
                // this tile (slot kind 0); only the first pair's range may
                // have begun in an earlier tile.
                const long long t0 = static_cast<long long>(x.tile) * num_kb;
                const int first = pair_of(t0);
                const int n_contrib = pair_of(t0 + num_kb - 1) - first + 1;
                const int kind_first = range_begin(first) >= t0 ? 0 : 1;
                // Per (tile, CTA rank, epilogue warp): {arrived, published}.
                // Every contributor arrives; all but the last then publish
                // their FP32 partial tile and count it as published.  The
                // last arriver publishes nothing: it waits (bounded) until the
                // others' partials are out -- they have all arrived, so none
                // of them waits on anything -- and sums them with its own,
                // still in TMEM, in K order.
                int32_t *cnt = a.counters + ((static_cast<int64_t>(x.tile) * 2 + rank) * 4 + q) * 2;
                int prev = 0;
                if (lane == 0)
                    prev = atomicAdd(cnt, 1);
                prev = __shfl_sync(0xffffffffu, prev, 0);
                if (prev != n_contrib - 1) {
                    float4 *mine = slots + (static_cast<int64_t>(blockIdx.x) * 2 + x.kind) * part4;
                    for (int c = 0; c < a.tile_n; c += 32) {
                        uint32_t r[32];
                        ld32(c, r);
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            mine[(c / 4 + v) * kTileM + row] =
                                make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                            __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
                    }
                    __threadfence();
                    __syncwarp();
                    if (lane == 0)
                        atomicAdd(cnt + 1, 1);
                } else {
                    int ok = 1;
                    if (lane == 0) {
                        ok = wait_count_at_least(cnt + 1, n_contrib - 1, a.timeout_ns) ? 1 : 0;
                        if (!ok) {
                            ctl.abort = 1;
                            record_status(FP8G_ERR_TIMEOUT, kRoleEpilogue, 500 + q);
                        }
                        cnt[0] = 0;   // ready for the next launch
                        cnt[1] = 0;
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    __threadfence();
                    const int me = cid - first;   // this pair's place in K order
                    // (plain instantiations only: the block-scaled ones, with
                    // 352 threads, have no registers to spare for it)
                    const bool two = !kBS && n_contrib == 2;
                    if (two && ok) {
                        // One other contributor: its next 32 columns are loaded
                        // while this 32 are summed (two chunks of loads in flight).
                        const int other = 1 - me;
                        const int kind = other == 0 ? kind_first : 0;
                        const float4 *src = slots + ((static_cast<int64_t>(2 * (first + other)) + rank) * 2 + kind) *
                                                        part4 + row;
                        float4 nxt[8];
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            nxt[v] = __ldcg(src + v * kTileM);
                        for (int c = 0; c < a.tile_n; c += 32) {
                            float4 cur[8];
#pragma unroll
                            for (int v = 0; v < 8; ++v)
                                cur[v] = nxt[v];
                            if (c + 32 < a.tile_n) {
#pragma unroll
                                for (int v = 0; v < 8; ++v)
                                    nxt[v] = __ldcg(src + ((c + 32) / 4 + v) * kTileM);
                            }
                            uint32_t own[32];
                            ld32(c, own);
                            uint32_t bits_v[32];
#pragma unroll
                            for (int v = 0; v < 8; ++v) {
                                const float o[4] = {cur[v].x, cur[v].y, cur[v].z, cur[v].w};
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    const float mine_f = __uint_as_float(own[4 * v + j]);
                                    bits_v[4 * v + j] = __float_as_uint(me == 0 ? mine_f + o[j] : o[j] + mine_f);
                                }
                            }
                            store_rows32<kEpi>(a, dout, bits_v, rf, x.g, grow, row_ok, x.n0 + c, tg);
                        }
                    }
                    for (int c = 0; c < a.tile_n && ok && !two; c += 32) {
                        uint32_t own[32];
                        ld32(c, own);
                        float acc_v[32];
                        for (int i = 0; i < n_contrib; ++i) {
                            float part[32];
                            if (i == me) {
#pragma unroll
                                for (int j = 0; j < 32; ++j)
                                    part[j] = __uint_as_float(own[j]);
                            } else {
                                const int kind = i == 0 ? kind_first : 0;
                                const float4 *src = slots +
                                                    ((static_cast<int64_t>(2 * (first + i)) + rank) * 2 + kind) *
                                                        part4 +
                                                    (c / 4) * kTileM + row;
#pragma unroll
                                for (int v = 0; v < 8; ++v) {
                                    const float4 f = __ldcg(src + v * kTileM);
                                    part[4 * v] = f.x;
                                    part[4 * v + 1] = f.y;
                                    part[4 * v + 2] = f.z;
                                    part[4 * v + 3] = f.w;
                                }
                            }
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                acc_v[j] = i == 0 ? part[j] : acc_v[j] + part[j];
                        }
                        uint32_t bits_v[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            bits_v[j] = __float_as_uint(acc_v[j]);
                        store_rows32<kEpi>(a, dout, bits_v, rf, x.g, grow, row_ok, x.n0 + c, tg);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive_cluster(mapa_shared(smem_addr(&ctl.tempty[acc]), 0));
            if (++acc == n_bufs) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    // Pair exit: neither CTA leaves while the other may still touch its
    // shared memory or barriers.  Every copy into either CTA has been seen
    // to land by then (the loaders' drains above), and the even CTA's MMA
    // issuer has waited for its tensor-core work.
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0)
        mbar_arrive_cluster(mapa_shared(smem_addr(&ctl.pair_exit), rank ^ 1u));
    if (warp == 0)
        warp_wait_drain<true>(smem_addr(&ctl.pair_exit), 0, 4 * a.timeout_ns);
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

// =====================================================================================
// k_gemm_swap: SwapAB.  Weights (B) on M, tokens (A) on a runtime N.
//
// Work is a list of output tiles (group, token chunk, 128 weight rows), each
// needing num_kb K blocks.  Stream-K: the tiles' K blocks are laid end to end
// and every CTA takes an equal contiguous range, so all SMs stream the same
// number of weight bytes.  A range covers whole tiles plus at most two
// partial ones (its first and last segment); a partial segment publishes an
// FP32 partial tile, and the contributor whose arrival completes the tile
// sums all contributions in K order and writes BF16.  Whole-tile mode (one
// tile per unit, no partials) is kept for comparison.
// =====================================================================================
struct SwapSeg {
    int g, tok0, n_tok, n_mma, w0, kb0, kb1, tile;
    int kind;   // 0: first segment of this CTA's range, 1: a later segment
};

struct SwapWalker {
    // stream-K: k-block positions [pos, end) of the linearised (tile, kb) space
    long long pos, end;
    // whole-tile mode: tile index u, stepping by the grid
    int u;
    bool first;
};

template <bool kBS, bool kEpi>
__global__ void __launch_bounds__(kBS ? kThreadsTmemScaled : kThreads, 1)
    k_gemm_swap(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_t,
                const __grid_constant__ CUtensorMap tm_sw, const __grid_constant__ CUtensorMap tm_st,
                const GemmArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    // The tensor maps are kernel parameters, never written by an earlier
    // launch: fetch their descriptors now, while programmatic dependent
    // launch may still hold this CTA before griddepcontrol.wait.
    if (threadIdx.x == 0) {
        tma_prefetch_map(&tm_w);
        tma_prefetch_map(&tm_t);
        if constexpr (kBS) {
            tma_prefetch_map(&tm_sw);
            tma_prefetch_map(&tm_st);
        }
    }
    const Smem sm = carve(smem_raw, a);
    SmemCtl &ctl = *sm.ctl;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_tiles = ceil_div(a.n, kTileM);   // 128 weight rows per tile
    const int cap = a.tile_n;                    // tokens per chunk
    const int num_kb = a.num_kb;
    const bool stream_k = a.k_splits != 1;       // 1 = whole tiles only
    const uint32_t w_bytes = kTileM * kBlockK;   // 16 KB weight box
    // Accumulators: two of 256 columns, or two of 128 (tile_n <= 128) so
    // that two CTAs -- this launch's and the next one's -- fit in TMEM.
    // With block scales: two accumulators of `cap` columns per MMA issuer
    // (issuer i's accumulator of buffer b at column (2b + i) * cap with two
    // issuers), then the TMEM scale sets.
    const uint32_t tmem_cols = (a.tmem_cols == 256 && !kBS) ? 256u : static_cast<uint32_t>(kTmemCols);
    const int acc_stride = kBS ? cap : static_cast<int>(tmem_cols / 2);
    const int acc_step = (kBS && a.dual_mma) ? 2 : 1;
    const int set_cols = sf_set_cols(cap);

    if (threadIdx.x == 0)
        init_barriers(ctl, a.stages, static_cast<uint32_t>(acc_step));
    if (warp == 0) {
        // A dense problem's table reads nothing from global memory; a
        // grouped one reads masked_m or the offsets, which the previous
        // launch in the stream may write.
        if (a.prefetch_kb == 0)
            grid_dep_wait();
        build_group_table(ctl, a, [&](int m) { return ceil_div(m, cap) * n_tiles; });
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&ctl.tmem_base), tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl.tmem_base;
    const int total_tiles = ctl.units_total;
    const long long T = static_cast<long long>(total_tiles) * num_kb;
    // Partition count: never more ranges than k-blocks, so every range that
    // meets a tile is non-empty and arrives on the tile's counter.  CTAs
    // beyond it get no stream-K work.
    const long long P = T < static_cast<long long>(gridDim.x) ? T : static_cast<long long>(gridDim.x);

    // CTA whose stream-K range contains k-block position x.
    auto cta_of = [&](long long x) { return static_cast<int>(((x + 1) * P - 1) / T); };
    auto range_begin = [&](long long b) { return b * T / P; };

    auto make_walker = [&]() {
        SwapWalker w;
        if (static_cast<long long>(blockIdx.x) < P) {
            w.pos = range_begin(blockIdx.x);
            w.end = range_begin(static_cast<long long>(blockIdx.x) + 1);
        } else {
            w.pos = w.end = 0;
        }
        w.u = blockIdx.x;
        w.first = true;
        return w;
    };
    // Next segment of this CTA's work; false when done.
    auto next_seg = [&](SwapWalker &w, SwapSeg &x) {
        int tile;
        if (stream_k) {
            if (w.pos >= w.end)
                return false;
            tile = static_cast<int>(w.pos / num_kb);
            x.kb0 = static_cast<int>(w.pos - static_cast<long long>(tile) * num_kb);
            const long long left = w.end - w.pos;
            x.kb1 = left < num_kb - x.kb0 ? x.kb0 + static_cast<int>(left) : num_kb;
            w.pos += x.kb1 - x.kb0;
        } else {
            if (w.u >= total_tiles)
                return false;
            tile = w.u;
            x.kb0 = 0;
            x.kb1 = num_kb;
            w.u += gridDim.x;
        }
        x.tile = tile;
        x.kind = w.first ? 0 : 1;
        w.first = false;
        x.g = find_group(ctl, a.groups, tile);
        const int local = tile - ctl.group_prefix[x.g];
        const int nt = local % n_tiles;
        const int chunk = local / n_tiles;
        x.tok0 = chunk * cap;
        const int left_tok = ctl.group_m[x.g] - x.tok0;
        x.n_tok = left_tok < cap ? left_tok : cap;
        x.n_mma = (x.n_tok + 15) & ~15;
        x.w0 = nt * kTileM;
        return true;
    };

    // Dense problems: fetch the first prefetch_kb K blocks of this CTA's
    // weights into L2 while the previous launch may still run; the loads
    // after griddepcontrol.wait then find them there.  (The token rows are
    // shared by every CTA and come from L2 after the first one's load.)
    if (a.prefetch_kb > 0 && warp == 2 && lane == 0) {
        SwapWalker wk = make_walker();
        SwapSeg x;
        int left = a.prefetch_kb;
        while (left > 0 && next_seg(wk, x))
            for (int kb = x.kb0; kb < x.kb1 && left > 0; ++kb, --left)
                tma_prefetch_l2_3d(&tm_w, kb * kBlockK, x.w0, x.g);
    }
    grid_dep_wait();   // inputs may come from the previous launch in the stream
    if (threadIdx.x == 0)
        grid_dep_launch_dependents();

    if (warp == 0) {
        // ------------------------------- loader -------------------------------
        int stage = 0;
        uint32_t phase = 0;
        long long issued = 0;
        bool aborted = false;
        const bool drop = (a.flags & FP8G_DEBUG_DROP_FIRST_LOAD) && blockIdx.x == 0;
        const uint64_t w_policy = policy_evict_first();   // weights are read once
        uint32_t sf_par = 0, sf_used = 0;   // per stage: parity of scale fills posted, any posted
        SwapWalker wk = make_walker();
        SwapSeg x;
        while (!aborted && next_seg(wk, x)) {
            // Token rows in TMA boxes of tok_box rows, enough boxes to cover
            // the valid tokens.  Rows past them up to the MMA's n_mma hold
            // whatever the stage held before; they only reach accumulator
            // columns that are never stored.
            const int n_load = ((x.n_tok + a.tok_box - 1) / a.tok_box) * a.tok_box;
            const uint32_t tx = w_bytes + static_cast<uint32_t>(n_load) * kBlockK;
            for (int kb = x.kb0; kb < x.kb1; ++kb) {
                if (!warp_wait(smem_addr(&ctl.empty[stage]), phase ^ 1u, ctl, a.timeout_ns,
                               kRoleLoader, stage)) {
                    aborted = true;
                    break;
                }
                const bool sf = kBS && sf_load_at(kb, x.kb0, a.sf_k) && !(drop && issued == 0);
                if (lane == 0 && !(drop && issued == 0)) {
                    uint8_t *sw = sm.stages + static_cast<size_t>(stage) * a.stage_bytes;
                    const uint32_t fb = smem_addr(&ctl.full[stage]);
                    mbar_arrive_expect_tx(fb, tx);
                    tma_load_3d_hint(smem_addr(sw), &tm_w, fb, kb * kBlockK, x.w0, x.g, w_policy);
                    for (int r = 0; r < n_load; r += a.tok_box)
                        tma_load_3d(smem_addr(sw + w_bytes + static_cast<uint32_t>(r) * kBlockK), &tm_t, fb,
                                    kb * kBlockK, a_row(a, ctl, x.g, x.tok0 + r), a_grp(a, x.g));
                    if (sf) {
                        const uint32_t sb = smem_addr(&ctl.sffull[stage]);
                        const int y = sf_first_group(kb, a.sf_k);
                        mbar_arrive_expect_tx(sb, 4u * static_cast<uint32_t>(kTileM + cap));
                        tma_load_3d_hint(smem_addr(sw + a.sf_off), &tm_sw, sb, x.w0, y, x.g, w_policy);
                        tma_load_3d(smem_addr(sw + a.sf_off + 4 * kTileM), &tm_st, sb, x.tok0, y, x.g);
                    }
                }
                if (sf) {
                    sf_par ^= 1u << stage;
                    sf_used |= 1u << stage;
                }
                __syncwarp();
                ++issued;
                if (++stage == a.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        loader_tail(ctl, a, stage, phase, issued, aborted, drop);
        if constexpr (kBS)
            sf_loader_drain(ctl, a, sf_par, sf_used, a.stages);
    } else if (warp == 1 && !kBS) {
        // ----------------------------- MMA issuer -----------------------------
        // MMA operand A = weight tile (format of B), operand B = token tile
        // (format of A).
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool issued_any = false;
        SwapWalker wk = make_walker();
        SwapSeg x;
        while (next_seg(wk, x)) {
            const uint32_t idesc = make_idesc(a.b_fmt, a.a_fmt, kTileM, static_cast<uint32_t>(x.n_mma));
            if (!warp_wait(smem_addr(&ctl.tempty[acc]), acc_phase ^ 1u, ctl, a.timeout_ns, kRoleMma,
                           100 + acc))
                break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * acc_stride);
            bool ok = true;
            for (int kb = x.kb0; kb < x.kb1; ++kb) {
                if (!warp_wait(smem_addr(&ctl.full[stage]), phase, ctl, a.timeout_ns, kRoleMma,
                               stage)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t sw = smem_addr(sm.stages + static_cast<size_t>(stage) * a.stage_bytes);
                    const uint64_t wdesc = smem_desc_k_sw128(sw);
                    const uint64_t tdesc = smem_desc_k_sw128(sw + w_bytes);
#pragma unroll
                    for (int k = 0; k < kBlockK / 32; ++k)
                        mma_f8f6f4(d_tmem, wdesc + 2u * k, tdesc + 2u * k, idesc,
                                   (kb != x.kb0 || k != 0) ? 1u : 0u);
                    mma_commit(smem_addr(&ctl.empty[stage]));
                }
                __syncwarp();
                issued_any = true;
                if (++stage == a.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok)
                break;
            if (lane == 0)
                mma_commit(smem_addr(&ctl.tfull[acc]));
            __syncwarp();
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        mma_drain(ctl, a, issued_any);
    } else if (kBS && (warp == 1 || (warp == 6 && a.dual_mma))) {
        // ---------------------- MMA issuers, block-scaled ----------------------
        // One block-scaled MMA costs an issuing thread far more time than a
        // plain one, so with room in TMEM two threads issue (warps 1 and 6):
        // issuer i takes the K blocks whose running index in this CTA is
        // i mod 2, into its own accumulator; the epilogue adds the two.  Both
        // walk every K block to follow the stage ring and the scale sets,
        // which the staging warps write into TMEM.  At each scale load an
        // issuer retires the previous set (a commit on sffree, counted once
        // per issuer) and waits for the next one.
        const int me = warp == 1 ? 0 : 1;
        int stage = 0;
        uint32_t phase = 0;
        uint32_t par = 0;   // running K-block index mod 2
        int acc = 0;
        uint32_t acc_phase = 0;
        bool issued_any = false;
        const uint32_t sets_tmem = tmem_base + static_cast<uint32_t>(a.sf_col0);
        int j = -1;   // scale loads passed
        uint32_t set_tmem = sets_tmem;
        bool ok = true;
        SwapWalker wk = make_walker();
        SwapSeg x;
        while (ok && next_seg(wk, x)) {
            const uint32_t idesc_bs = make_idesc_bs(a.b_fmt, a.a_fmt, kTileM, static_cast<uint32_t>(x.n_mma), 0);
            if (!warp_wait(smem_addr(&ctl.tempty[acc]), acc_phase ^ 1u, ctl, a.timeout_ns, kRoleMma,
                           100 + acc))
                break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>((acc * acc_step + me) * acc_stride);
            bool first = true;
            for (int kb = x.kb0; kb < x.kb1; ++kb) {
                if (sf_load_at(kb, x.kb0, a.sf_k) && !sf_next_set(ctl, a, j, sets_tmem, set_cols, set_tmem)) {
                    ok = false;
                    break;
                }
                if (acc_step == 1 || static_cast<int>(par) == me) {
                    if (!warp_wait(smem_addr(&ctl.full[stage]), phase, ctl, a.timeout_ns, kRoleMma, stage)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t sw = smem_addr(sm.stages + static_cast<size_t>(stage) * a.stage_bytes);
                        const uint64_t wdesc = smem_desc_k_sw128(sw);
                        const uint64_t tdesc = smem_desc_k_sw128(sw + w_bytes);
#pragma unroll
                        for (int k = 0; k < kBlockK / 32; ++k) {
                            const uint32_t id = a.sf_k == 1 ? static_cast<uint32_t>(kb & 3) : static_cast<uint32_t>(k);
                            mma_f8f6f4_bs(d_tmem, wdesc + 2u * k, tdesc + 2u * k, idesc_bs | (id << 4) | (id << 29),
                                          set_tmem, set_tmem + 4u, (!first || k != 0) ? 1u : 0u);
                        }
                        mma_commit(smem_addr(&ctl.empty[stage]));
                    }
                    __syncwarp();
                    first = false;
                    issued_any = true;
                }
                par ^= 1u;
                if (++stage == a.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok)
                break;
            // Both issuers arrive, whether or not this one had a K block of
            // the segment (the epilogue knows which accumulators hold data).
            if (lane == 0)
                mma_commit(smem_addr(&ctl.tfull[acc]));
            __syncwarp();
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        mma_drain(ctl, a, issued_any, me == 0 ? &ctl.drain : &ctl.drain2);
    } else if (kBS && warp >= 7) {
        // --------------------- block-scale staging into TMEM ---------------------
        // Warps 7-10, one per TMEM lane quadrant: for each scale load, wait
        // for its stage and write the TMEM scale set (sf_stage_tmem).
        if constexpr (kBS) {
            const uint32_t sets_q = tmem_base + static_cast<uint32_t>(a.sf_col0) +
                                    (static_cast<uint32_t>((warp & 3) * 32) << 16);
            int stage = 0;
            uint32_t sf_par = 0;   // per stage: parity of the next scale fill to wait for
            int j = -1;
            bool stop = false;
            SwapWalker wk = make_walker();
            SwapSeg x;
            while (!stop && next_seg(wk, x)) {
                for (int kb = x.kb0; kb < x.kb1; ++kb) {
                    if (sf_load_at(kb, x.kb0, a.sf_k)) {
                        ++j;
                        if (!warp_wait(smem_addr(&ctl.sffull[stage]), (sf_par >> stage) & 1u, ctl, a.timeout_ns,
                                       kRoleScales, stage) ||
                            !sf_stage_tmem(ctl, a, sm.stages + static_cast<size_t>(stage) * a.stage_bytes + a.sf_off,
                                           cap, j, sets_q, set_cols)) {
                            stop = true;
                            break;
                        }
                        sf_par ^= 1u << stage;
                    }
                    if (++stage == a.stages)
                        stage = 0;
                }
            }
        }
    } else if (warp >= 2 && warp <= 5) {
        // ------------------------------ epilogue ------------------------------
        // Thread = weight row n (TMEM lane), registers = tokens (TMEM columns).
        // For a fixed token the 32 lanes of a warp write 32 consecutive n.
        const int q = warp & 3;
        const int row = q * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        __nv_bfloat16 *dout = static_cast<__nv_bfloat16 *>(a.d);
        // Partial tiles: slot (cta, kind) of [cap/4 token groups][128 weight
        // rows][4 tokens] FP32.  A thread owns one weight row and moves 4 tokens
        // per 16-byte access; a warp touches 512 consecutive bytes.
        const int64_t part_stride4 = kTileM * static_cast<int64_t>(cap) / 4;
        float4 *slots = reinterpret_cast<float4 *>(a.workspace);
        uint32_t par = 0;   // running K-block index mod 2 (which issuer took a segment's first K block)
        SwapWalker wk = make_walker();
        SwapSeg x;
        while (next_seg(wk, x)) {
            if (!warp_wait(smem_addr(&ctl.tfull[acc]), acc_phase, ctl, a.timeout_ns, kRoleEpilogue,
                           200 + acc))
                break;
            tc_fence_after();
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(acc * acc_step * acc_stride);
            // With two issuers: the one that took the segment's first K block
            // always has data; the other one only if the segment has two or
            // more K blocks.
            const uint32_t t_first = t_row + par * static_cast<uint32_t>(acc_stride);
            const uint32_t t_second = t_row + (par ^ 1u) * static_cast<uint32_t>(acc_stride);
            const bool both = acc_step == 2 && x.kb1 - x.kb0 >= 2;
            if (acc_step == 2)
                par ^= static_cast<uint32_t>((x.kb1 - x.kb0) & 1);
            // 16 accumulator columns of this thread's row, summed over issuers.
            auto ld16 = [&](int c, uint32_t (&r)[16]) {
                tmem_ld_32x32b_x16(t_first + static_cast<uint32_t>(c), r);
                if constexpr (kBS) {
                    if (both) {
                        uint32_t r2[16];
                        tmem_ld_32x32b_x16(t_second + static_cast<uint32_t>(c), r2);
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            r[i] = __float_as_uint(__uint_as_float(r[i]) + __uint_as_float(r2[i]));
                    }
                }
            };
            const int64_t grow0 = static_cast<int64_t>(ctl.group_row0[x.g]) + x.tok0;   // output row of token 0
            const int col_base = x.w0 + q * 32;                                         // this warp's 32 columns
            const bool whole = x.kb0 == 0 && x.kb1 == num_kb;
            if (whole) {
                for (int c = 0; c < x.n_mma; c += 16) {
                    uint32_t r[16];
                    ld16(c, r);
                    swap_store16<kEpi>(a, dout, r, x.g, grow0 + c, x.n_tok - c, col_base);
                }
            } else {
                // Contributors of this tile: the CTAs whose ranges meet it,
                // in K order.
                const long long t0 = static_cast<long long>(x.tile) * num_kb;
                const int first = cta_of(t0);
                const int n_contrib = cta_of(t0 + num_kb - 1) - first + 1;
                // Every contributor after the first starts its range inside
                // this tile, so the tile is its first segment (slot kind 0);
                // the first contributor's range may have begun in an earlier
                // tile.  (No division inside the reduction loop.)
                const int kind_first = range_begin(first) >= t0 ? 0 : 1;
                // Per (tile, epilogue warp): {arrived, published}.  Every
                // contributor arrives first; all but the last then publish
                // their FP32 partial tile and count it as published.  The
                // last arriver publishes nothing: it waits (bounded) until
                // the others' partials are out and sums them with its own,
                // still in TMEM, in K order.
                int32_t *cnt = a.counters + (static_cast<int64_t>(x.tile) * 4 + q) * 2;
                int prev = 0;
                if (lane == 0)
                    prev = atomicAdd(cnt, 1);
                prev = __shfl_sync(0xffffffffu, prev, 0);
                if (prev != n_contrib - 1) {
                    float4 *mine = slots + (static_cast<int64_t>(blockIdx.x) * 2 + x.kind) * part_stride4;
                    for (int c = 0; c < x.n_mma; c += 16) {
                        uint32_t r[16];
                        ld16(c, r);
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            mine[(c / 4 + v) * kTileM + row] =
                                make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                            __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
                    }
                    __threadfence();
                    __syncwarp();
                    if (lane == 0)
                        atomicAdd(cnt + 1, 1);
                } else {
                    int ok = 1;
                    if (lane == 0) {
                        ok = wait_count_at_least(cnt + 1, n_contrib - 1, a.timeout_ns) ? 1 : 0;
                        if (!ok) {
                            ctl.abort = 1;
                            record_status(FP8G_ERR_TIMEOUT, kRoleEpilogue, 500 + q);
                        }
                        cnt[0] = 0;   // ready for the next launch
                        cnt[1] = 0;
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    __threadfence();
                    const int me = static_cast<int>(blockIdx.x) - first;   // this CTA's place in K order
                    for (int c = 0; c < x.n_mma && ok; c += 16) {
                        uint32_t own[16];
                        ld16(c, own);
                        float acc_v[16];
                        for (int p0 = 0; p0 < n_contrib; p0 += 4) {
                            // four contributors' 16 tokens per batch, every load
                            // unconditional (this CTA's own slot is read but unused)
                            float4 buf[4][4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int ci = (p0 + i < n_contrib) ? p0 + i : 0;
                                const int cta = first + ci;
                                const int kind = ci == 0 ? kind_first : 0;
                                const float4 *src = slots + (static_cast<int64_t>(cta) * 2 + kind) * part_stride4 +
                                                    (c / 4) * kTileM + row;
#pragma unroll
                                for (int w = 0; w < 4; ++w)
                                    buf[i][w] = __ldcg(src + w * kTileM);
                            }
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                if (p0 + i >= n_contrib)
                                    break;
                                float part[16];
                                if (p0 + i == me) {
#pragma unroll
                                    for (int j = 0; j < 16; ++j)
                                        part[j] = __uint_as_float(own[j]);
                                } else {
#pragma unroll
                                    for (int w = 0; w < 4; ++w) {
                                        part[4 * w] = buf[i][w].x;
                                        part[4 * w + 1] = buf[i][w].y;
                                        part[4 * w + 2] = buf[i][w].z;
                                        part[4 * w + 3] = buf[i][w].w;
                                    }
                                }
#pragma unroll
                                for (int j = 0; j < 16; ++j)
                                    acc_v[j] = (p0 + i == 0) ? part[j] : acc_v[j] + part[j];
                            }
                        }
                        uint32_t bits_v[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            bits_v[j] = __float_as_uint(acc_v[j]);
                        swap_store16<kEpi>(a, dout, bits_v, x.g, grow0 + c, x.n_tok - c, col_base);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(smem_addr(&ctl.tempty[acc]));
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, tmem_cols);
    }
}

// =====================================================================================
// Launchers
// =====================================================================================
constexpr int kSmemLimitDevices = 64;

// Launch with programmatic stream serialisation (unless FP8G_NO_PDL): the
// kernel may start while the previous launch in the stream finishes; it
// waits (griddepcontrol.wait) before touching global memory.
template <typename Kernel, typename... Maps>
static cudaError_t launch_pdl(Kernel kernel, int threads, int grid, size_t smem, cudaStream_t stream,
                              const GemmArgs &args, const Maps &...maps)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = (args.flags & FP8G_NO_PDL) ? 0 : 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, maps..., args);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

// The dynamic shared-memory limit of a kernel is a property of the kernel in
// the device's context: set it once per device (and whenever a larger size
// is wanted) instead of on every launch.
template <typename Kernel>
static cudaError_t set_smem_limit(Kernel kernel, size_t smem, std::atomic<int> *done)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const int want = static_cast<int>(smem);
    const bool cached = dev >= 0 && dev < kSmemLimitDevices;
    if (cached && done[dev].load(std::memory_order_acquire) >= want)
        return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, want);
    if (e == cudaSuccess && cached) {
        int cur = done[dev].load(std::memory_order_relaxed);
        while (cur < want && !done[dev].compare_exchange_weak(cur, want, std::memory_order_release))
            ;
    }
    return e;
}

template <bool kBS, bool kEpi>
static cudaError_t launch_mn_t(const CUtensorMap &tm_a, const CUtensorMap &tm_b, const CUtensorMap &tm_sa,
                               const CUtensorMap &tm_sb, const GemmArgs &args, int grid, size_t smem,
                               cudaStream_t stream)
{
    static std::atomic<int> done[kSmemLimitDevices];
    cudaError_t e = set_smem_limit(k_gemm_mn<kBS, kEpi>, smem, done);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(k_gemm_mn<kBS, kEpi>, kBS ? kThreadsTmemScaled : kThreads, grid, smem, stream, args, tm_a, tm_b,
                      tm_sa, tm_sb);
}

// Output scales or a fused epilogue select the kernels' full store path.
static bool wants_epi(const GemmArgs &args) { return args.epi || args.scale_a || args.scale_b; }

// Two MMA issuers need an even number of stages (>= 2): each stage then
// always feeds the same issuer, so no parity wait on it can skip a phase.
static bool dual_ok(const GemmArgs &args)
{
    return !args.dual_mma || (args.sf_k && args.stages >= 2 && (args.stages & 1) == 0);
}

cudaError_t launch_gemm_mn(const CUtensorMap &tm_a, const CUtensorMap &tm_b, const CUtensorMap &tm_sa,
                           const CUtensorMap &tm_sb, const GemmArgs &args, int grid, size_t smem,
                           cudaStream_t stream)
{
    if (smem < smem_bytes_of(args) || !dual_ok(args) ||
        (args.sf_k == 1 && (args.sf_ring < 1 || args.sf_ring > kSfRingSlots || args.sf_slot_bytes % 128 != 0 ||
                            args.sf_slot_bytes < 4 * (kTileM + args.tile_n))) ||
        (args.sf_k == 4 && args.sf_ring != 0))
        return cudaErrorInvalidValue;
    const bool epi = wants_epi(args);
    if (args.sf_k)
        return epi ? launch_mn_t<true, true>(tm_a, tm_b, tm_sa, tm_sb, args, grid, smem, stream)
                   : launch_mn_t<true, false>(tm_a, tm_b, tm_sa, tm_sb, args, grid, smem, stream);
    return epi ? launch_mn_t<false, true>(tm_a, tm_b, tm_sa, tm_sb, args, grid, smem, stream)
               : launch_mn_t<false, false>(tm_a, tm_b, tm_sa, tm_sb, args, grid, smem, stream);
}

template <bool kBS, bool kEpi>
static cudaError_t launch_mn2_t(const CUtensorMap &tm_a, const CUtensorMap &tm_b, const CUtensorMap &tm_sa,
                                const CUtensorMap &tm_sb, const GemmArgs &args, int grid, size_t smem,
                                cudaStream_t stream)
{
    static std::atomic<int> done[kSmemLimitDevices];
    cudaError_t e = set_smem_limit(k_gemm_mn2<kBS, kEpi>, smem, done);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(k_gemm_mn2<kBS, kEpi>, kBS ? kThreadsTmemScaled : kThreads, grid, smem, stream, args, tm_a, tm_b,
                      tm_sa, tm_sb);
}

cudaError_t launch_gemm_mn2(const CUtensorMap &tm_a, const CUtensorMap &tm_b, const CUtensorMap &tm_sa,
                            const CUtensorMap &tm_sb, const GemmArgs &args, int grid, size_t smem,
                            cudaStream_t stream)
{
    // Grouped problems: plain kernels, whole tiles.
    const bool grouped = args.groups != 1 || args.masked_m != nullptr || args.group_offsets != nullptr;
    if (smem < smem_bytes_of(args) || (grid & 1) ||
        (grouped && (args.sf_k || args.k_splits != 1)) || !dual_ok(args))
        return cudaErrorInvalidValue;
    const bool epi = wants_epi(args);
    if (args.sf_k)
        return epi ? launch_mn2_t<true, true>(tm_a, tm_b, tm_sa, tm_sb, args, grid, smem, stream)
                   : launch_mn2_t<true, false>(tm_a, tm_b, tm_sa, tm_sb, args, grid, smem, stream);
    return epi ? launch_mn2_t<false, true>(tm_a, tm_b, tm_sa, tm_sb, args, grid, smem, stream)
               : launch_mn2_t<false, false>(tm_a, tm_b, tm_sa, tm_sb, args, grid, smem, stream);
}

template <bool kBS, bool kEpi>
static cudaError_t launch_swap_t(const CUtensorMap &tm_w, const CUtensorMap &tm_t, const CUtensorMap &tm_sw,
                                 const CUtensorMap &tm_st, const GemmArgs &args, int grid, size_t smem,
                                 cudaStream_t stream)
{
    static std::atomic<int> done[kSmemLimitDevices];
    cudaError_t e = set_smem_limit(k_gemm_swap<kBS, kEpi>, smem, done);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(k_gemm_swap<kBS, kEpi>, kBS ? kThreadsTmemScaled : kThreads, grid, smem, stream, args, tm_w, tm_t,
                      tm_sw, tm_st);
}

cudaError_t launch_gemm_swap(const CUtensorMap &tm_w, const CUtensorMap &tm_t, const CUtensorMap &tm_sw,
                             const CUtensorMap &tm_st, const GemmArgs &args, int grid, size_t smem,
                             cudaStream_t stream)
{
    if (smem < smem_bytes_of(args) || !dual_ok(args))
        return cudaErrorInvalidValue;
    const bool epi = wants_epi(args);
    if (args.sf_k)
        return epi ? launch_swap_t<true, true>(tm_w, tm_t, tm_sw, tm_st, args, grid, smem, stream)
                   : launch_swap_t<true, false>(tm_w, tm_t, tm_sw, tm_st, args, grid, smem, stream);
    return epi ? launch_swap_t<false, true>(tm_w, tm_t, tm_sw, tm_st, args, grid, smem, stream)
               : launch_swap_t<false, false>(tm_w, tm_t, tm_sw, tm_st, args, grid, smem, stream);
}

cudaError_t read_and_clear_status(int32_t info[4])
{
    cudaError_t e = cudaMemcpyFromSymbol(info, g_status, 4 * sizeof(int32_t));
    if (e != cudaSuccess)
        return e;
    const int32_t zero[4] = {0, 0, 0, 0};
    return cudaMemcpyToSymbol(g_status, zero, 4 * sizeof(int32_t));
}

}  // namespace fp8g
