// Launch interface between the host API (api.cu) and the sm_103a kernels
// (kernels.cu).  Plain structs only; no torch types.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fp8g {

constexpr int kBlockK = 128;         // K bytes per pipeline stage (one 128-byte swizzle row)
constexpr int kTileM = 128;          // MMA M: rows of the operand on the M side
constexpr int kMaxStages = 16;
// Weight bytes per CTA that a dense launch fetches into L2 before
// griddepcontrol.wait: 128 KB, or 64 KB when two CTAs share an SM (the
// next launch's CTAs are then resident from this launch's start, and a
// larger early fetch competes with this launch's stream).  Measured on the
// small-M weight-streaming shapes against 32 KB to 1 MB.
constexpr int kEarlyPrefetchBytes = 128 * 1024;
inline int early_prefetch_kb(int weight_bytes_per_kb, bool shared_sm)
{
    const int kb = (shared_sm ? kEarlyPrefetchBytes / 2 : kEarlyPrefetchBytes) / weight_bytes_per_kb;
    return kb > 1 ? kb : 1;
}
constexpr int kMaxGroups = 1024;
constexpr int kThreads = 192;        // warp 0 loader, warp 1 MMA issuer, warps 2-5 epilogue
constexpr int kThreadsTmemScaled = 352;  // block-scaled instantiations: + warp 6, second MMA issuer,
                                         // and warps 7-10, scale sets into TMEM
constexpr int kMaxSfSets = 4;        // TMEM block-scale sets in flight
constexpr int kSfRingSlots = 3;      // single-SM block-scaled tiles: scale loads in flight
constexpr int kTmemCols = 512;       // two accumulators of up to 256 columns
constexpr int kAccStride = 256;
constexpr int kCtlFixedBytes = 768;  // barriers, TMEM slot, flags
constexpr int kSmemAlignPad = 1024;  // dynamic smem base rounded up to 1024 B

// Control block: fixed part plus three int32 tables per group (unit prefix,
// valid rows, first output row), rounded up to 128 bytes.
inline int ctl_bytes_for(int groups)
{
    const int b = kCtlFixedBytes + 4 * (3 * groups + 1);
    return (b + 127) & ~127;
}

// Roles recorded in the device status word.
enum Role : int { kRoleLoader = 0, kRoleMma = 1, kRoleEpilogue = 2, kRoleScheduler = 3, kRoleScales = 4 };

struct GemmArgs {
    // Problem.  Token operand A is [groups, rows_a, k]; weight operand B is
    // [groups, n, k]; output D is [groups, rows_a, n] BF16.
    int32_t rows_a;            // M (dense) or M_max (grouped)
    int32_t n;
    int32_t k;
    int32_t groups;
    int32_t num_kb;            // ceil(k / kBlockK)
    const int32_t *masked_m;   // device [groups] or nullptr (all rows valid)
    const int32_t *group_offsets;  // contiguous layout: device [groups + 1]; group g owns rows
                               // offsets[g] .. offsets[g+1]-1 of A [rows_a, k] and D [rows_a, n]
                               // (rows_a = M_total); nullptr: the [groups, rows_a] layouts
    void *d;
    // Tiling.
    int32_t tile_n;            // mn kernel: N tile (32..256, multiple of 32)
                               // swap kernel: token chunk (16..256, multiple of 16)
    int32_t stages;            // pipeline depth (1..kMaxStages)
    int32_t stage_bytes;       // bytes per stage (multiple of 1024)
    int32_t k_splits;          // swap kernel: 1 = whole tiles per unit; otherwise stream-K
                               // (equal k-block ranges per CTA, partial tiles reduced).
                               // SM-pair kernel: 1 = whole tiles; 0 = the tiles of the last
                               // partial wave stream-K over every pair; s >= 2 = each of those
                               // tiles split s ways along K (s ranges per tile)
    int32_t raster_band;       // mn kernel: M tiles per rasterisation band
    int32_t tmem_cols;         // swap kernel: 256 (two 128-column accumulators, two CTAs
                               // may share an SM) or 512 (default)
    uint32_t a_fmt, b_fmt;     // 0 = E4M3, 1 = E5M2 (of A and B as passed by the caller)
    uint32_t flags;            // FP8G_DEBUG_* bits
    uint64_t timeout_ns;       // limit of every barrier wait
    // Output scales (nullptr: none).  D = bf16(sa * sb * sum):
    //   sa = scale_a[g * rows_a + m] if sa_per_row, else scale_a[g];
    //   sb = scale_b[g * n + col]    if sb_per_col, else scale_b[g].
    const float *scale_a;
    const float *scale_b;
    int32_t sa_per_row;
    int32_t sb_per_col;
    // Block scales (UE8M0, one byte per row per K group).  sf_k = 0: none;
    // else K groups per 128-wide K block (1: groups of 128 elements, 4:
    // groups of 32).  Every load brings 4 groups per row (4 K blocks' worth
    // for sf_k = 1, one K block's for sf_k = 4) into the stage it rides with.
    int32_t sf_k;
    int32_t sf_off;            // byte offset of the scale area inside a stage
    int32_t sf_col0;           // first TMEM column of the block-scale sets
    int32_t sf_sets;           // TMEM block-scale sets (2..kMaxSfSets)
    int32_t sf_ring;           // single-SM tile kernel with 128-element groups (required there): the
                               // scale loads have a ring of sf_ring slots of sf_slot_bytes after the
                               // stages, each load issued one scale set ahead of the operands;
                               // 0 (every other case): scale bytes ride in the stage of their
                               // first K block
    int32_t sf_slot_bytes;     // bytes per ring slot: [4][128] side A then [4][tile_n] side B, 128-aligned
    int32_t dual_mma;          // block-scaled SwapAB / single-SM kernels: two MMA-issuing threads,
                               // each with its own accumulators, alternating K blocks
    int32_t tok_box;           // swap kernel: token rows per TMA box of a chunk (a multiple of 16
                               // dividing tile_n, or a dense problem's whole token count; the host
                               // encodes the token map with this box)
    int32_t prefetch_kb;       // dense problems (one group, no masked_m, no offsets): K blocks of
                               // this CTA's first work fetched into L2 before griddepcontrol.wait,
                               // so that they stream while the previous launch drains; 0: none
    int32_t a_box_rows;        // token-tile kernel: A rows per TMA box (the host encodes the A map with
                               // it); 0: 128.  Fewer only for dense problems of fewer rows
    int32_t spare_ctas;        // token-tile kernel, dense problems whose weights fit in half of L2:
                               // the SMs this launch leaves idle.  CTAs 0 .. spare_ctas-1 are the
                               // ones that start early, on those SMs, while the previous launch
                               // still runs: before griddepcontrol.wait they fetch the weight
                               // tiles of every CTA congruent to them modulo spare_ctas into L2
                               // (0: each CTA fetches its first prefetch_kb K blocks only)
    int32_t acc_bufs;          // block-scaled tile kernels: accumulator buffers per issuer (0 or 2:
                               // two; 1: one, when two issuers' four or a 256-wide tile's two
                               // accumulators and the scale sets do not fit in TMEM)
    // Fused epilogue (epi != 0): out = round(act(alpha * v + beta * c_in + bias)),
    // v the (scaled) product; c_in BF16 shaped like D or nullptr; bias FP32
    // [groups][n] or nullptr; act ReLU when relu != 0; round_mode 0 nearest
    // even, 1 toward zero, 2 toward +inf, 3 toward -inf.
    int32_t epi;
    int32_t relu;
    int32_t round_mode;
    float alpha;
    float beta;
    const void *c_in;
    const float *bias;
    float *workspace;          // swap kernel, stream-K: 2 FP32 partial tiles per CTA
                               // (128 x tile_n floats each)
    int32_t *counters;         // stream-K: {arrived, published} per (tile, epilogue warp) (SwapAB)
                               // or per (tile, CTA of the pair, epilogue warp) (SM pair); zero at rest
};

// Block-scaled stage layout.  After the two operand tiles (MMA side A: 128
// rows; side B: box_b rows) a stage holds the raw scale bytes as TMA writes
// them ([4][128] then [4][box_b]: four K groups per row).  A TMEM scale set
// has 4 columns for side A and 4 per 128 rows of side B.
inline int sf_stage_bytes(int box_b) { return 4 * (kTileM + box_b); }
__host__ __device__ inline int sf_set_cols(int box_b) { return 4 + 4 * ((box_b + 127) / 128); }

// Shared-memory footprint of a launch (stages + control block + alignment).
inline size_t smem_bytes_for(int stages, int stage_bytes, int groups)
{
    return static_cast<size_t>(stages) * stage_bytes + ctl_bytes_for(groups) + kSmemAlignPad;
}

// The same for a planned launch: stages, the scale ring if any, control block.
inline size_t smem_bytes_of(const GemmArgs &a)
{
    return smem_bytes_for(a.stages, a.stage_bytes, a.groups) + static_cast<size_t>(a.sf_ring) * a.sf_slot_bytes;
}

// `smem` must be at least smem_bytes_of(args); the host passes the whole per-block budget so that exactly one CTA (and one
// 512-column TMEM allocation) is resident per SM.
// tm_sa / tm_sb: block-scale maps of the MMA's A and B sides (read only when
// args.sf_k != 0; any valid map otherwise).
cudaError_t launch_gemm_mn(const CUtensorMap &tm_a, const CUtensorMap &tm_b, const CUtensorMap &tm_sa,
                           const CUtensorMap &tm_sb, const GemmArgs &args, int grid, size_t smem,
                           cudaStream_t stream);
// Dense only: clusters of two CTAs, 256 x tile_n tiles, B box of tile_n/2 rows.
// With block scales tm_sa covers A's scales (box 128 rows) and tm_sb B's
// (box tile_n rows: each CTA loads the whole tile's).
cudaError_t launch_gemm_mn2(const CUtensorMap &tm_a, const CUtensorMap &tm_b, const CUtensorMap &tm_sa,
                            const CUtensorMap &tm_sb, const GemmArgs &args, int grid, size_t smem,
                            cudaStream_t stream);
cudaError_t launch_gemm_swap(const CUtensorMap &tm_w, const CUtensorMap &tm_t, const CUtensorMap &tm_sw,
                             const CUtensorMap &tm_st, const GemmArgs &args, int grid, size_t smem,
                             cudaStream_t stream);

// Scratch a swap-kernel launch needs: partial tiles (2 per CTA) and counters.
inline size_t swap_partials_bytes(int grid, int tile_n)
{
    return static_cast<size_t>(grid) * 2 * kTileM * static_cast<size_t>(tile_n) * sizeof(float);
}
// Two counters (arrived, published) per (tile, epilogue warp).
inline size_t swap_counter_bytes(long long tiles) { return static_cast<size_t>(tiles) * 8 * sizeof(int32_t); }
// SM-pair kernel: two counters per (tile, CTA of the pair, epilogue warp).
inline size_t pair_counter_bytes(long long tiles) { return static_cast<size_t>(tiles) * 16 * sizeof(int32_t); }

// Status word of the current device: read it, then clear it.
cudaError_t read_and_clear_status(int32_t info[4]);

}  // namespace fp8g
