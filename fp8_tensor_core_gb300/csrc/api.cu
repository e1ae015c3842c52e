// Host side of the C ABI declared in include/fp8g.h: argument validation,
// variant selection (SwapAB or not, tile sizes, pipeline depth, stream-K),
// TMA tensor-map encoding and kernel launch.
//
// Sources: "DeepGEMM：基于 Hopper Tensor Core 的 FP8 矩阵乘法内核优化实践"
// (sheratonhq.com/news/187119) §1.3 (large shapes fill every SM; small
// shapes take a simpler path), §3.3 (TMA descriptors prepared by the host),
// §6.2-6.4 (every K step clipped to the real length; alignment of the
// descriptor fields matters); "一次“转置”，半张算力：DeepSeek SwapAB 漂流史"
// (hwcomputing.csdn.net) §3.1 (ENABLE_SWAPAB switch), §3.5 (swap only
// pays for small per-expert token counts; the switch-over depends on the
// shape and the SM count); "MLS 三个访存 Bug 深度剖析" Bug 1 (base
// addresses and offsets kept in 64 bits: tensor maps take full pointers).
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <thread>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "fp8g.h"
#include "kernels.cuh"

namespace fp8g {
namespace {

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;
constexpr int kMaxDevices = 64;
// SwapAB is weighed against token tiles (a cost model) when a problem has
// at most this many token rows per group (the weights then fill the 128-row
// MMA side and the tokens a narrow runtime N).
constexpr int64_t kSwapAutoMaxTokens = 128;        // dense and block-scaled problems
constexpr int64_t kSwapAutoMaxGroupTokens = 255;   // plain grouped problems
constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;
constexpr int64_t kSpareFetchMaxBytes = int64_t(64) << 20;   // weights fetched by early CTAs: <= half of L2

std::atomic<uint64_t> g_timeout_ns{kDefaultTimeoutNs};

struct DeviceInfo {
    bool ready = false;
    int sms = 0;
    int cc_major = 0, cc_minor = 0;
    int smem_optin = 0;
};

// Stream-K scratch of one (device, stream): FP32 partial tiles indexed by
// the CTA and arrival counters indexed by the output tile.  Two launches that
// shared one such area could run at the same time on unordered streams and
// overwrite each other's partials and counts, so every stream has its own;
// launches on one stream are ordered by the stream (a launch's loads and
// stores all follow griddepcontrol.wait, i.e. the previous launch's end).
// The per-thread default stream is one stream per host thread, so its
// entries are told apart by the thread as well.
struct Workspace {
    int dev = -1;
    cudaStream_t stream = nullptr;
    std::thread::id thread{};
    float *ws = nullptr;
    size_t ws_bytes = 0;
    int32_t *counters = nullptr;
    size_t counter_bytes = 0;
};

std::mutex g_mu;
constexpr int64_t kDefaultInitTiles = 65536;   // fp8g_init(0): counters for this many stream-K tiles
DeviceInfo g_dev[kMaxDevices];
std::vector<Workspace> g_ws;   // one entry per (device, stream[, thread]), under g_mu

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

std::atomic<int> g_have_device{0};   // set once a device has been seen (the count cannot drop later)

int current_device(int *dev, DeviceInfo *info)
{
    if (!g_have_device.load(std::memory_order_acquire)) {
        int count = 0;
        if (cudaGetDeviceCount(&count) != cudaSuccess || count <= 0) {
            cudaGetLastError();
            return FP8G_ERR_NO_DEVICE;
        }
        g_have_device.store(1, std::memory_order_release);
    }
    if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices)
        return FP8G_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo &d = g_dev[*dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, *dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, *dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, *dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, *dev) !=
                cudaSuccess)
            return FP8G_ERR_CUDA;
        d.ready = true;
    }
    *info = d;
    // The kernels are built for sm_103a only.
    if (info->cc_major != 10 || info->cc_minor != 3)
        return FP8G_ERR_UNSUPPORTED;
    return FP8G_OK;
}

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Tensor maps are encoded once per (base address, extents, box) and kept in
// a small direct-mapped cache: a map is a pure function of those fields, so
// a hit returns exactly what encoding would (a freed and reallocated buffer
// at the same address with the same extents gets the same, correct map).
// Encoding costs the host a driver call per operand; repeated calls with the
// same buffers -- the serving and graph-building pattern -- skip it.
struct MapKey {
    const void *base;
    uint64_t d0, d1, d2, ld;
    uint32_t box0, box1;
    uint32_t kind;   // 1: operand map (SWIZZLE_128B), 2: block-scale map
    bool operator==(const MapKey &o) const
    {
        return base == o.base && d0 == o.d0 && d1 == o.d1 && d2 == o.d2 && ld == o.ld && box0 == o.box0 &&
               box1 == o.box1 && kind == o.kind;
    }
};
struct MapSlot {
    MapKey key{};
    CUtensorMap map;
    bool used = false;
};
constexpr int kMapCacheSlots = 256;
std::mutex g_map_mu;
MapSlot g_maps[kMapCacheSlots];

size_t map_slot(const MapKey &k)
{
    uint64_t h = reinterpret_cast<uintptr_t>(k.base) * 0x9E3779B97F4A7C15ull;
    for (uint64_t v : {k.d0, k.d1, k.d2, k.ld, (static_cast<uint64_t>(k.box0) << 32) | k.box1,
                       static_cast<uint64_t>(k.kind)})
        h = (h ^ v) * 0x100000001B3ull;
    return static_cast<size_t>((h ^ (h >> 29)) % kMapCacheSlots);
}

bool cached_map(CUtensorMap *m, const MapKey &key, bool (*encode)(CUtensorMap *, const MapKey &))
{
    const size_t i = map_slot(key);
    {
        std::lock_guard<std::mutex> lk(g_map_mu);
        if (g_maps[i].used && g_maps[i].key == key) {
            *m = g_maps[i].map;
            return true;
        }
    }
    if (!encode(m, key))
        return false;
    std::lock_guard<std::mutex> lk(g_map_mu);
    g_maps[i].key = key;
    g_maps[i].map = *m;
    g_maps[i].used = true;
    return true;
}

// 3-D map over a [groups, rows, k] byte tensor, box {128 bytes of K, box_rows, 1},
// 128-byte swizzle, out-of-bounds elements read as zero.
bool encode_operand(CUtensorMap *m, const MapKey &key)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return false;
    const cuuint64_t dims[3] = {key.d0, key.d1, key.d2};
    const cuuint64_t strides[2] = {key.d0, key.d1 * key.d0};
    const cuuint32_t box[3] = {key.box0, key.box1, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    std::memset(m, 0, sizeof(*m));
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(key.base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_map(CUtensorMap *m, const void *base, int64_t k, int64_t rows, int64_t groups, uint32_t box_rows)
{
    const MapKey key{base, static_cast<uint64_t>(k), static_cast<uint64_t>(rows), static_cast<uint64_t>(groups), 0,
                     static_cast<uint32_t>(kBlockK), box_rows, 1u};
    return cached_map(m, key, encode_operand);
}

// 3-D map over block scales [groups, ks, ld] bytes (row r of K group j at
// byte r of that group's vector), box {box_rows, box_k, 1}, no swizzle,
// rows >= `rows` and groups >= ks read as zero.
bool encode_scales(CUtensorMap *m, const MapKey &key)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return false;
    const cuuint64_t dims[3] = {key.d0, key.d1, key.d2};
    const cuuint64_t strides[2] = {key.ld, key.d1 * key.ld};
    const cuuint32_t box[3] = {key.box0, key.box1, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    std::memset(m, 0, sizeof(*m));
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(key.base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_sf_map(CUtensorMap *m, const void *base, int64_t rows, int64_t ks, int64_t groups, int64_t ld,
                 uint32_t box_rows, uint32_t box_k)
{
    const MapKey key{base, static_cast<uint64_t>(rows), static_cast<uint64_t>(ks), static_cast<uint64_t>(groups),
                     static_cast<uint64_t>(ld), box_rows, box_k, 2u};
    return cached_map(m, key, encode_scales);
}

// Device pointers already found to be device (or managed) memory: the
// grouped calls check their masked_m / offsets pointer once per address
// instead of asking the driver on every call.
constexpr int kPtrCacheSlots = 64;
std::mutex g_ptr_mu;
const void *g_dev_ptrs[kPtrCacheSlots];

bool is_device_pointer(const void *p)
{
    const size_t i = (reinterpret_cast<uintptr_t>(p) >> 4) % kPtrCacheSlots;
    {
        std::lock_guard<std::mutex> lk(g_ptr_mu);
        if (g_dev_ptrs[i] == p)
            return true;
    }
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
        return false;
    std::lock_guard<std::mutex> lk(g_ptr_mu);
    g_dev_ptrs[i] = p;
    return true;
}

// Stages that fit the per-block shared-memory budget beside the control
// block and `other_bytes` more (FP8G_STAGES(n) caps it; the one-stage debug
// mode forces 1).
int pick_stages(const DeviceInfo &d, int stage_bytes, int groups, uint32_t flags, int other_bytes = 0)
{
    if (flags & FP8G_DEBUG_ONE_STAGE)
        return 1;
    const int budget = d.smem_optin - ctl_bytes_for(groups) - kSmemAlignPad - other_bytes;
    int s = std::max(1, std::min(kMaxStages, budget / stage_bytes));
    const int cap = static_cast<int>((flags >> 20) & 15u);
    if (cap > 0)
        s = std::min(s, cap);
    return s;
}

// The handle under which a stream's workspace is kept: the legacy default
// stream has two names (0 and cudaStreamLegacy).
cudaStream_t stream_key(cudaStream_t s) { return s == cudaStreamLegacy ? nullptr : s; }

// Entry of (dev, stream), created empty if absent.  Caller holds g_mu.
Workspace &workspace_of(int dev, cudaStream_t stream)
{
    stream = stream_key(stream);
    const std::thread::id th = stream == cudaStreamPerThread ? std::this_thread::get_id() : std::thread::id{};
    for (Workspace &w : g_ws)
        if (w.dev == dev && w.stream == stream && w.thread == th)
            return w;
    Workspace w;
    w.dev = dev;
    w.stream = stream;
    w.thread = th;
    g_ws.push_back(w);
    return g_ws.back();
}

// Frees an entry's buffers (cudaFree waits for the device's work); the
// device must be current.
bool free_workspace(Workspace &w)
{
    bool ok = true;
    if (w.ws && cudaFree(w.ws) != cudaSuccess)
        ok = false;
    if (w.counters && cudaFree(w.counters) != cudaSuccess)
        ok = false;
    w.ws = nullptr;
    w.counters = nullptr;
    w.ws_bytes = w.counter_bytes = 0;
    return ok;
}

// Stream-K workspace of (current device, stream), grown on demand (the
// first call needing a larger one allocates; later calls reuse it).
int ensure_workspace(int dev, cudaStream_t stream, size_t ws_bytes, size_t counter_bytes, float **ws,
                     int32_t **counters)
{
    std::lock_guard<std::mutex> lk(g_mu);
    Workspace &w = workspace_of(dev, stream);
    if (w.ws_bytes < ws_bytes) {
        if (w.ws)
            cudaFree(w.ws);
        w.ws = nullptr;
        w.ws_bytes = 0;
        if (cudaMalloc(&w.ws, ws_bytes) != cudaSuccess)
            return FP8G_ERR_CUDA;
        w.ws_bytes = ws_bytes;
    }
    if (w.counter_bytes < counter_bytes) {
        if (w.counters)
            cudaFree(w.counters);
        w.counters = nullptr;
        w.counter_bytes = 0;
        if (cudaMalloc(&w.counters, counter_bytes) != cudaSuccess)
            return FP8G_ERR_CUDA;
        if (cudaMemset(w.counters, 0, counter_bytes) != cudaSuccess)
            return FP8G_ERR_CUDA;
        w.counter_bytes = counter_bytes;
    }
    *ws = w.ws;
    *counters = w.counters;
    return FP8G_OK;
}

int check_common(const void *A, const void *B, void *D, int64_t N, int64_t K, int a_dtype,
                 int b_dtype)
{
    if (!A || !B || !D)
        return FP8G_ERR_INVALID_ARG;
    if (N <= 0 || K <= 0 || N > kMaxDim || K > kMaxDim)
        return FP8G_ERR_INVALID_ARG;
    if (K % 16 != 0 || N % 8 != 0)
        return FP8G_ERR_INVALID_ARG;
    if ((a_dtype != FP8G_E4M3 && a_dtype != FP8G_E5M2) ||
        (b_dtype != FP8G_E4M3 && b_dtype != FP8G_E5M2))
        return FP8G_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(B) || !aligned16(D))
        return FP8G_ERR_MISALIGNED;
    return FP8G_OK;
}

// N tile of the non-swapped kernel: the candidate with the fewest tile
// column-equivalents over whole waves of SMs.
int pick_tile_n(int64_t m_tiles_total, int64_t N, int sms, int max_tn = 256)
{
    static const int cands[] = {256, 224, 192, 160, 128};
    int best = 128;
    double best_cost = 1e300;
    for (int tn : cands) {
        if (tn > max_tn)
            continue;
        const int64_t units = m_tiles_total * cdiv(N, tn);
        const int64_t waves = cdiv(units, sms);
        const double cost = static_cast<double>(waves) * (tn + 32);
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best = tn;
        }
    }
    return best;
}

// Pair-kernel plan: N tile and work split, from a cost model in units of
// "one K block of a 256-wide tile".  Narrower tiles pay a fixed cost per MMA
// instruction over fewer columns (measured per unit of width: 192 wide
// ~18 % slower per K block; a 224-wide K block takes as long as a 256-wide
// one -- 4096^3 in four waves of either: 48.2 vs 47.8 us at 2.07 GHz, and
// 50.2 vs 49.5 us under the sustained power cap).  Whole tiles pay for the
// last partial wave of pairs.  When that wave holds at most half as many
// tiles as there are pairs and every pair has a whole tile to run as well,
// each of its tiles can instead be split s ways along K (s ranges of
// num_kb / s K blocks, at least kMinSplitKb each, on s x tail pairs): a
// pair runs the piece that starts a tile first, then a whole tile, then the
// piece that finishes a tile, whose contributor sums the earlier partial
// tiles (published long before) while its MMA issuer runs the next whole
// tile.  The publishing and summing cost the busiest pair about
// kSplitOverheadKb K blocks per extra contributor (fit on GB300 at 2.07 GHz,
// same box, split vs whole: 4096^3 45.1 vs 47.4 us, 4096 x 4096 x 3072 36.0
// vs 37.7 us, 6400 x 2560 x 2048 29.0 vs 28.2 us); with no whole tile to
// overlap the sum is exposed (1024 x 1024 x 8192: 29.7 vs 23.9 us), so the
// split needs a whole wave.  Stream-K over every pair (FP8G_STREAM_K) stays
// opt-in; FP8G_WHOLE_TILES keeps whole tiles.
constexpr int kMaxTailSplit = 4;
constexpr int kMinSplitKb = 8;
constexpr double kSplitOverheadKb = 9.0;

struct PairPlan {
    int tile_n;
    int k_split;   // GemmArgs::k_splits of the SM-pair kernel: 1 whole tiles, 0 stream-K, >= 2 tail split
};

PairPlan plan_pair(int64_t m_tiles2, int64_t N, int num_kb, int pairs, uint32_t flags, int max_tn, bool allow_split)
{
    static const int cands[] = {256, 224, 192, 160, 128};
    static const double cost_per_kb[] = {1.0, 1.15, 1.18, 1.30, 1.45};
    PairPlan best{max_tn, 1};
    double best_cost = 1e300;
    const int tn_override = static_cast<int>((flags >> 16) & 15u);
    // FP8G_SPLIT_TAIL: only split plans compete (when some width allows one).
    const bool force_split = (flags & FP8G_SPLIT_TAIL) && allow_split && !(flags & (FP8G_WHOLE_TILES | FP8G_STREAM_K));
    PairPlan best_split{0, 1};
    double best_split_cost = 1e300;
    for (int i = 0; i < 5; ++i) {
        const int tn = cands[i];
        if (tn > max_tn)
            continue;
        if (tn_override >= 1 && tn_override <= 8 && tn != std::min(32 * tn_override, max_tn))
            continue;
        const int64_t units = m_tiles2 * cdiv(N, tn);
        const double width = static_cast<double>(tn) / 256.0;
        const double dp = static_cast<double>(cdiv(units, pairs)) * num_kb * cost_per_kb[i] * width;
        if (dp < best_cost - 1e-9) {
            best_cost = dp;
            best = {tn, 1};
        }
        const int64_t tail = units % pairs;
        if (!allow_split || tail == 0 || (flags & FP8G_WHOLE_TILES))
            continue;
        if (flags & FP8G_STREAM_K) {
            // complete waves of whole tiles, then the last wave's tiles split evenly
            const double sk = (static_cast<double>(units / pairs) * num_kb +
                               static_cast<double>(tail) * num_kb / pairs + 3.0) *
                              cost_per_kb[i] * width;
            if (sk < best_cost - 1e-9) {
                best_cost = sk;
                best = {tn, 0};
            }
            continue;
        }
        const int s = static_cast<int>(std::min<int64_t>({kMaxTailSplit, pairs / tail, num_kb / kMinSplitKb}));
        if (s >= 2 && (units >= pairs || force_split)) {
            const double split = (static_cast<double>(units / pairs) * num_kb + static_cast<double>(num_kb) / s +
                                  kSplitOverheadKb * (s - 1)) *
                                 cost_per_kb[i] * width;
            if (split < best_cost - 1e-9) {
                best_cost = split;
                best = {tn, s};
            }
            if (split < best_split_cost - 1e-9) {
                best_split_cost = split;
                best_split = {tn, s};
            }
        }
    }
    if (force_split && best_split.tile_n)
        best = best_split;
    if (tn_override >= 1 && tn_override <= 8 && best.tile_n != std::min(32 * tn_override, max_tn))
        best = {std::min(32 * tn_override, max_tn), 1};
    return best;
}

// SwapAB or 128-row token tiles, for G groups of (up to) M tokens each.
// Both stream every weight byte once from HBM.  Token tiles: one CTA per
// weight tile, so few tiles leave SMs idle and one SM streams at most ~55
// GB/s (a group's further token tiles find the weights in L2), and every
// token tile runs 128-row MMAs however few rows are valid.  SwapAB with
// stream-K keeps every SM streaming; per K block of 128 it pays ~316 ns
// plus ~0.8 ns per token (rounded to 16) in MMA issue, plus a partial-tile
// reduction that grows with the tokens and with fewer K blocks per tile.
// Constants measured on GB300 at 2.07 GHz: groups of 32 / 96 / 160 tokens
// (16 groups, N x K of 4096 x 7168 and 7168 x 2048), the masked decode and
// the dense small-M shapes; the estimates pick the faster kernel on all of
// them (SwapAB at 16 x 160 tokens, N = 4096, K = 7168: 92.3 vs 102.7 us;
// token tiles at 32 and 96 tokens and at N = 7168, K = 2048).
bool swap_beats_token_tiles(int64_t G, int64_t M, int64_t N, int64_t K, int sms)
{
    const double bytes = static_cast<double>(G) * (static_cast<double>(N) * K + static_cast<double>(M) * K +
                                                   2.0 * M * N);
    const double hbm = 6.7e12, per_sm = 55e9, tensor = 2.5e15;
    const int64_t m_tiles = G * cdiv(M, kTileM);
    const int tn = pick_tile_n(m_tiles, N, sms);
    const int64_t weight_tiles = G * cdiv(N, tn);
    const double t_tiles = std::max({bytes / hbm,
                                     static_cast<double>(tn) * K * static_cast<double>(cdiv(weight_tiles, sms)) /
                                         per_sm,
                                     2.0 * static_cast<double>(m_tiles) * kTileM * N * K / tensor}) +
                           5e-6;
    const double tok = static_cast<double>(cdiv(M, 16) * 16);
    const double num_kb = static_cast<double>(cdiv(K, kBlockK));
    const double kb_per_sm = static_cast<double>(G) * cdiv(N, kTileM) * num_kb / sms;
    const double t_swap =
        std::max(bytes / hbm, kb_per_sm * (316e-9 + 0.8e-9 * tok)) + 8e-6 + 0.06e-6 * tok * 16.0 / num_kb;
    return t_swap < t_tiles;
}

// Token rows per TMA box in the SwapAB kernel (a multiple of 16 that
// divides the chunk).  Measured (same box, A/B): 16-row boxes are best for
// plain chunks of 32 tokens (masked decode 142.0 vs 144.5 us with one
// 32-row box), one box of the whole chunk for larger chunks (64 tokens,
// N=7168, K=16384: 32.9 -> 28.4 us) and for block-scaled chunks (masked
// decode 162.6 -> 141.3 us).  A dense problem whose tokens fit one chunk
// (dense_rows > 0) loads exactly its rows in one box: rows of a box past
// the tensor's end cost the copy engine time to fill.
int swap_token_box(int64_t cap, bool block_scaled, uint32_t flags, int64_t dense_rows)
{
    const int override_rows = static_cast<int>((flags >> 24) & 15u) * 16;   // FP8G_TOKEN_BOX(n)
    if (override_rows > 0 && cap % override_rows == 0)
        return override_rows;
    if (dense_rows > 0 && dense_rows <= cap)
        return static_cast<int>(dense_rows);
    if (block_scaled || cap > 32)
        return static_cast<int>(cap);
    return 16;
}

struct Problem {
    const void *A, *B;
    void *D;
    const int32_t *masked_m;
    const int32_t *group_offsets;   // contiguous layout (rows_a = M_total), else nullptr
    int64_t G, rows_a, N, K;
    int64_t token_hint;   // expected valid tokens per group (<= rows_a)
    int a_dtype, b_dtype;
    uint32_t flags;
    const float *scale_a = nullptr;   // see GemmArgs
    const float *scale_b = nullptr;
    bool sa_per_row = false, sb_per_col = false;
    // Block scales: [G][ks][ld] UE8M0 bytes; sf_k = 128 / group size (0: none).
    const uint8_t *sf_a = nullptr, *sf_b = nullptr;
    int64_t sf_a_ld = 0, sf_b_ld = 0;
    int sf_k = 0;
    // Fused epilogue (see GemmArgs).
    bool epi = false;
    float alpha = 1.0f, beta = 0.0f;
    const void *c_in = nullptr;
    const float *bias = nullptr;
    int relu = 0, round_mode = 0;
};

int check_epilogue(const fp8g_epilogue *e, Problem &p)
{
    if (!e)
        return FP8G_OK;
    if (e->activation != FP8G_ACT_NONE && e->activation != FP8G_ACT_RELU)
        return FP8G_ERR_INVALID_ARG;
    if (e->round_mode < FP8G_ROUND_RN || e->round_mode > FP8G_ROUND_RD)
        return FP8G_ERR_INVALID_ARG;
    if ((e->c && !aligned16(e->c)) || (e->bias && !aligned16(e->bias)))
        return FP8G_ERR_MISALIGNED;
    p.epi = true;
    p.alpha = e->alpha;
    p.beta = e->beta;
    p.c_in = e->c;
    p.bias = e->bias;
    p.relu = e->activation == FP8G_ACT_RELU ? 1 : 0;
    p.round_mode = e->round_mode;
    return FP8G_OK;
}

// Largest tile (token chunk, or N tile) whose two accumulators leave TMEM
// room for at least two stages' scale sets.
constexpr int kMaxBlockScaledTile = 224;   // widest block-scaled tile with two accumulator buffers
constexpr int kWideBlockScaledKb = 48;     // K blocks from which single-SM block-scaled tiles go 256 wide

int check_blockscales(const uint8_t *sf_a, int64_t sf_a_ld, const uint8_t *sf_b, int64_t sf_b_ld,
                      int group_k, int64_t rows, int64_t N, Problem &p)
{
    if (!sf_a || !sf_b)
        return FP8G_ERR_INVALID_ARG;
    if (group_k != 32 && group_k != 128)
        return FP8G_ERR_INVALID_ARG;
    if (sf_a_ld < rows || sf_b_ld < N || sf_a_ld > kMaxDim || sf_b_ld > kMaxDim)
        return FP8G_ERR_INVALID_ARG;
    if (sf_a_ld % 16 != 0 || sf_b_ld % 16 != 0 || !aligned16(sf_a) || !aligned16(sf_b))
        return FP8G_ERR_MISALIGNED;
    p.sf_a = sf_a;
    p.sf_b = sf_b;
    p.sf_a_ld = sf_a_ld;
    p.sf_b_ld = sf_b_ld;
    p.sf_k = kBlockK / group_k;
    return FP8G_OK;
}

// Stage layout of a block-scaled launch whose MMA B side has box_b rows:
// operand tiles, then the scale area (at args.sf_off), the whole rounded up to
// 1024 bytes.  TMEM: two accumulators of box_b columns, then as many scale
// sets (up to kMaxSfSets) as the remaining columns hold.
void plan_blockscaled(GemmArgs &args, const DeviceInfo &info, int box_b, int groups, uint32_t flags)
{
    args.sf_off = kTileM * kBlockK + box_b * kBlockK;
    args.stage_bytes = (args.sf_off + sf_stage_bytes(box_b) + 1023) & ~1023;
    args.sf_col0 = 2 * box_b;
    args.sf_sets = std::min(kMaxSfSets, (kTmemCols - 2 * box_b) / sf_set_cols(box_b));
    args.stages = pick_stages(info, args.stage_bytes, groups, flags);
}

// Scale arguments: both pointers given (16-byte aligned device memory), each
// with one entry per group or one per output row (A: `row_len` rows in all)
// / per column of every group (B).
int check_scales(const float *sa, int64_t sa_len, const float *sb, int64_t sb_len, int64_t G,
                 int64_t row_len, int64_t N, Problem &p)
{
    if (!sa || !sb)
        return FP8G_ERR_INVALID_ARG;
    if (!aligned16(sa) || !aligned16(sb))
        return FP8G_ERR_MISALIGNED;
    if (sa_len != G && sa_len != row_len)
        return FP8G_ERR_INVALID_ARG;
    if (sb_len != G && sb_len != G * N)
        return FP8G_ERR_INVALID_ARG;
    p.scale_a = sa;
    p.scale_b = sb;
    p.sa_per_row = sa_len == row_len && row_len != G;
    p.sb_per_col = sb_len == G * N && N != 1;
    return FP8G_OK;
}

void describe_as(fp8g_plan *out, int kernel, int tile_n, const GemmArgs &args, bool stream_k, bool shared_sm,
                 int token_box, int grid)
{
    out->kernel = kernel;
    out->tile_n = tile_n;
    out->stages = args.stages;
    out->stream_k = stream_k ? 1 : 0;
    out->mma_issuers = args.dual_mma ? 2 : 1;
    out->shared_sm = shared_sm ? 1 : 0;
    out->token_box = token_box;
    out->grid = grid;
    out->k_split = stream_k ? 0 : 1;
}

// Plans and enqueues the launch for `p`.  With `forced`, plans for that
// device instead of the current one; with `describe`, fills it and returns
// before anything is allocated, encoded or enqueued.
int launch(const Problem &p, cudaStream_t stream, const DeviceInfo *forced = nullptr, fp8g_plan *describe = nullptr)
{
    int dev = 0;
    DeviceInfo info;
    int st = FP8G_OK;
    if (forced)
        info = *forced;
    else if ((st = current_device(&dev, &info)) != FP8G_OK)
        return st;

    const uint32_t mode = p.flags & FP8G_SWAP_MASK;
    if (mode == 3u)
        return FP8G_ERR_INVALID_ARG;
    // Plain grouped problems of fewer than 256 tokens per group (the SM-pair
    // kernel's tile) weigh SwapAB against token tiles; dense and block-scaled
    // ones only up to 128 tokens (above that the SM-pair or token-tile
    // kernels take them).
    const bool grouped_problem = p.G > 1 || p.masked_m || p.group_offsets;
    bool swap = mode == FP8G_SWAP_ON ||
                (mode == FP8G_SWAP_AUTO &&
                 p.token_hint <= (grouped_problem && !p.sf_k ? kSwapAutoMaxGroupTokens : kSwapAutoMaxTokens));
    if (swap && mode == FP8G_SWAP_AUTO)
        swap = swap_beats_token_tiles(p.G, p.token_hint, p.N, p.K, info.sms);
    const int num_kb = static_cast<int>(cdiv(p.K, kBlockK));
    const bool dense = p.G == 1 && !p.masked_m && !p.group_offsets;

    GemmArgs args;
    std::memset(&args, 0, sizeof(args));
    args.rows_a = static_cast<int32_t>(p.rows_a);
    args.n = static_cast<int32_t>(p.N);
    args.k = static_cast<int32_t>(p.K);
    args.groups = static_cast<int32_t>(p.G);
    args.num_kb = num_kb;
    args.masked_m = p.masked_m;
    args.group_offsets = p.group_offsets;
    args.d = p.D;
    args.a_fmt = static_cast<uint32_t>(p.a_dtype);
    args.b_fmt = static_cast<uint32_t>(p.b_dtype);
    args.flags = p.flags;
    args.timeout_ns = g_timeout_ns.load();
    args.scale_a = p.scale_a;
    args.scale_b = p.scale_b;
    args.sa_per_row = p.sa_per_row ? 1 : 0;
    args.sb_per_col = p.sb_per_col ? 1 : 0;
    args.k_splits = 1;
    args.raster_band = 1;
    args.sf_k = p.sf_k;
    const int64_t ks = p.sf_k ? cdiv(p.K, kBlockK / p.sf_k) : 0;
    args.epi = p.epi ? 1 : 0;
    args.alpha = p.alpha;
    args.beta = p.beta;
    args.c_in = p.c_in;
    args.bias = p.bias;
    args.relu = p.relu;
    args.round_mode = p.round_mode;

    CUtensorMap tm0, tm1, tm2, tm3;
    if (swap) {
        const int64_t cap = std::min<int64_t>(p.sf_k ? kMaxBlockScaledTile : 256,
                                              cdiv(std::max<int64_t>(p.token_hint, 1), 16) * 16);
        const int64_t chunks = cdiv(p.rows_a, cap);
        const int64_t n_tiles = cdiv(p.N, kTileM);
        const int64_t tiles_upper = p.G * chunks * n_tiles;
        if (tiles_upper > kMaxDim || tiles_upper * num_kb > (int64_t(1) << 53))
            return FP8G_ERR_UNSUPPORTED;
        // Stream-K over all (tile, k-block) pairs unless whole tiles are asked for.
        const bool whole_tiles = (p.flags & FP8G_WHOLE_TILES) != 0;
        int grid = static_cast<int>(std::min<int64_t>(info.sms, whole_tiles ? tiles_upper
                                                                            : tiles_upper * num_kb));
        if (grid <= 0)
            return FP8G_OK;
        args.tile_n = static_cast<int32_t>(cap);
        args.tok_box = swap_token_box(cap, p.sf_k != 0, p.flags, dense ? p.rows_a : 0);
        args.stage_bytes = static_cast<int32_t>(kTileM * kBlockK + cap * kBlockK);
        // Co-residency: with at most 128 tokens per chunk the accumulators fit
        // 256 TMEM columns; capping shared memory at half the SM lets the next
        // launch's CTAs become resident (and finish their set-up) while this
        // one drains.
        // Shared SM by default for dense problems of up to 16 tokens: the
        // next launch's set-up then overlaps this one's drain (measured
        // 26.1 -> 24.8 us at N = 7168, K = 16384; no gain at 32 or more
        // tokens, a loss for the masked grouped decode).
        const bool share_auto = !(p.flags & FP8G_NO_SHARE_SM) && dense &&
                                cap <= 16;
        const bool share_sm = ((p.flags & FP8G_SHARE_SM) || share_auto) && cap <= 128 && !p.sf_k;
        size_t smem_request = static_cast<size_t>(info.smem_optin);
        if (share_sm) {
            const int half = info.smem_optin / 2 - 1024;   // leave room for two CTAs' reserved smem
            const int s_half = (half - ctl_bytes_for(static_cast<int>(p.G)) - kSmemAlignPad) / args.stage_bytes;
            args.stages = std::max(1, std::min(kMaxStages, s_half));
            const uint32_t cap_st = (p.flags >> 20) & 15u;
            if (cap_st > 0)
                args.stages = std::min<int>(args.stages, static_cast<int>(cap_st));
            if (p.flags & FP8G_DEBUG_ONE_STAGE)
                args.stages = 1;
            args.tmem_cols = 256;
            smem_request = smem_bytes_for(args.stages, args.stage_bytes, static_cast<int>(p.G));
        } else if (p.sf_k) {
            plan_blockscaled(args, info, static_cast<int>(cap), static_cast<int>(p.G), p.flags);
            args.tmem_cols = 512;
            // Two MMA issuers when four accumulators of the chunk and at
            // least two scale sets fit in TMEM.
            const int set_cols = sf_set_cols(static_cast<int>(cap));
            const int sets_dual = std::min<int>(kMaxSfSets, (kTmemCols - 4 * static_cast<int>(cap)) / set_cols);
            // (An even stage count keeps each stage with one issuer, whose
            // parity waits on it then never skip a phase.)
            if (sets_dual >= 2 && !(p.flags & FP8G_ONE_MMA_ISSUER) && args.stages >= 2) {
                args.dual_mma = 1;
                args.sf_col0 = static_cast<int32_t>(4 * cap);
                args.sf_sets = sets_dual;
                args.stages &= ~1;
            }
        } else {
            args.stages = pick_stages(info, args.stage_bytes, static_cast<int>(p.G), p.flags);
            args.tmem_cols = 512;
        }
        args.k_splits = whole_tiles ? 1 : 0;
        args.prefetch_kb = dense ? early_prefetch_kb(kTileM * kBlockK, share_sm) : 0;
        if (describe) {
            describe_as(describe, FP8G_KERNEL_SWAP_AB, static_cast<int>(cap), args, !whole_tiles, share_sm,
                        args.tok_box, grid);
            return FP8G_OK;
        }
        if (!whole_tiles) {
            st = ensure_workspace(dev, stream, swap_partials_bytes(grid, static_cast<int>(cap)),
                                  swap_counter_bytes(tiles_upper), &args.workspace, &args.counters);
            if (st != FP8G_OK)
                return st;
        }
        if (!make_map(&tm0, p.B, p.K, p.N, p.G, kTileM) ||
            !make_map(&tm1, p.A, p.K, p.rows_a, p.group_offsets ? 1 : p.G, static_cast<uint32_t>(args.tok_box)))
            return FP8G_ERR_CUDA;
        if (p.sf_k) {
            // MMA side A = weights (B's scales), side B = tokens (A's scales).
            if (!make_sf_map(&tm2, p.sf_b, p.N, ks, p.G, p.sf_b_ld, kTileM, 4) ||
                !make_sf_map(&tm3, p.sf_a, p.rows_a, ks, p.G, p.sf_a_ld, static_cast<uint32_t>(cap), 4))
                return FP8G_ERR_CUDA;
        } else {
            tm2 = tm0;
            tm3 = tm1;
        }
        return launch_gemm_swap(tm0, tm1, tm2, tm3, args, grid, smem_request, stream) == cudaSuccess
                   ? FP8G_OK
                   : FP8G_ERR_CUDA;
    }

    // Dense problems with more than one 128-row token tile: two SMs per
    // 256-row tile (cta_group::2), unless single-SM tiles are asked for.
    // Block scales: the pair kernel only pays for 128-element groups and long K
    // (measured on GB300: 2-6 % faster at K >= 7168, even at K = 4096, 7-13 %
    // slower at K = 2048 or with 32-element groups, whose per-K-block scale
    // copies weigh more in the pair's longer K block).
    // SM-pair tiles (256 token rows): dense problems with more than 128 rows;
    // grouped ones (plain, whole tiles) whose groups hold 256 or more tokens
    // on average (contiguous layout) or at most (masked layout's hint).
    const bool grouped = p.masked_m || p.group_offsets || p.G > 1;
    const int64_t group_tokens = p.group_offsets ? p.rows_a / p.G : p.token_hint;
    const bool pair_ok = grouped ? (!p.sf_k && (group_tokens >= 2 * kTileM || (p.flags & FP8G_PAIR_TILES)))
                                 : (p.rows_a > kTileM && (!p.sf_k || (p.flags & FP8G_PAIR_TILES)));
    if (pair_ok && !(p.flags & FP8G_SINGLE_SM_TILES)) {
        // 256-row tiles: exact for dense; for groups an upper bound (each
        // group boundary can add a partial tile) sizes the grid, and the
        // expected tokens per group the tile width.
        const int64_t m_tiles2 = grouped ? (p.group_offsets ? cdiv(p.rows_a, 2 * kTileM) + p.G
                                                            : p.G * cdiv(p.rows_a, 2 * kTileM))
                                         : cdiv(p.rows_a, 2 * kTileM);
        const int64_t m_tiles2_plan = grouped ? p.G * cdiv(std::max<int64_t>(group_tokens, 1), 2 * kTileM) : m_tiles2;
        const int pairs = info.sms / 2;
        const PairPlan plan = plan_pair(m_tiles2_plan, p.N, num_kb, pairs, p.flags, p.sf_k ? kMaxBlockScaledTile : 256,
                                        !grouped);
        const int tile_n = plan.tile_n;
        const int64_t units = m_tiles2 * cdiv(p.N, tile_n);
        if (units > kMaxDim || units * num_kb > (int64_t(1) << 53))
            return FP8G_ERR_UNSUPPORTED;
        args.tile_n = tile_n;
        args.k_splits = plan.k_split;
        const bool split_k = plan.k_split != 1;
        if (p.sf_k) {
            // Operand tiles (own 128 A rows, half of the B rows), then the scale
            // area for 128 A rows and the whole tile's tile_n B rows.
            args.sf_off = kTileM * kBlockK + (tile_n / 2) * kBlockK;
            args.stage_bytes = (args.sf_off + sf_stage_bytes(tile_n) + 1023) & ~1023;
            args.sf_col0 = 2 * tile_n;
            args.sf_sets = std::min(kMaxSfSets, (kTmemCols - 2 * tile_n) / sf_set_cols(tile_n));
        } else {
            args.stage_bytes = kTileM * kBlockK + (tile_n / 2) * kBlockK;
        }
        args.stages = pick_stages(info, args.stage_bytes, static_cast<int>(p.G), p.flags);
        if (p.sf_k && !(p.flags & FP8G_ONE_MMA_ISSUER) && args.stages >= 2) {
            // Two MMA issuers in the even CTA, as for single-SM tiles.
            const int set_cols = sf_set_cols(tile_n);
            const int sets2 = std::min(kMaxSfSets, (kTmemCols - 4 * tile_n) / set_cols);
            if (sets2 >= 2 || ((p.flags & FP8G_TWO_MMA_ISSUERS) && args.sf_sets >= 2)) {
                args.dual_mma = 1;
                args.acc_bufs = sets2 >= 2 ? 2 : 1;
                args.sf_col0 = args.acc_bufs * 2 * tile_n;
                if (sets2 >= 2)
                    args.sf_sets = sets2;
                args.stages &= ~1;
            }
        }
        // Bands of 256-row tiles whose token rows total ~32 MB stay in L2 while
        // the weight tiles stream past them (8192 x 18432 x 7168: DRAM reads
        // 641 MB with 48 MB bands, 400 MB with 32 MB, 489 MB with 24 MB;
        // 600 -> 589 us).
        const int64_t band = (32ll << 20) / (2 * kTileM * p.K);
        args.raster_band = static_cast<int32_t>(std::max<int64_t>(1, std::min<int64_t>(band, m_tiles2)));
        // Pairs with work: every pair for stream-K (or whole tiles beyond one
        // wave); with a tail split, the pairs of the whole waves or the split
        // tail's s ranges per tile, whichever is more.
        const int64_t busy = plan.k_split == 0 ? units * num_kb
                                               : (plan.k_split >= 2 ? std::max(units - units % pairs,
                                                                               units % pairs * plan.k_split)
                                                                    : units);
        const int grid = 2 * static_cast<int>(std::min<int64_t>(busy, pairs));
        if (describe) {
            describe_as(describe, FP8G_KERNEL_SM_PAIRS, tile_n, args, split_k, false, kTileM, grid);
            describe->k_split = plan.k_split;
            return FP8G_OK;
        }
        if (!make_map(&tm0, p.A, p.K, p.rows_a, p.group_offsets ? 1 : p.G, kTileM) ||
            !make_map(&tm1, p.B, p.K, p.N, p.G, static_cast<uint32_t>(tile_n / 2)))
            return FP8G_ERR_CUDA;
        if (p.sf_k) {
            if (!make_sf_map(&tm2, p.sf_a, p.rows_a, ks, 1, p.sf_a_ld, kTileM, 4) ||
                !make_sf_map(&tm3, p.sf_b, p.N, ks, 1, p.sf_b_ld, static_cast<uint32_t>(tile_n), 4))
                return FP8G_ERR_CUDA;
        } else {
            tm2 = tm0;
            tm3 = tm1;
        }
        if (split_k) {
            st = ensure_workspace(dev, stream, static_cast<size_t>(grid) * 2 * kTileM * tile_n * sizeof(float),
                                  pair_counter_bytes(units), &args.workspace, &args.counters);
            if (st != FP8G_OK)
                return st;
        }
        return launch_gemm_mn2(tm0, tm1, tm2, tm3, args, grid, static_cast<size_t>(info.smem_optin), stream) ==
                       cudaSuccess
                   ? FP8G_OK
                   : FP8G_ERR_CUDA;
    }

    const int64_t m_tiles = cdiv(p.rows_a, kTileM);
    // Block scales with long K: 256-wide tiles and one accumulator buffer.
    // A block-scaled MMA costs its issuing thread the same at N = 256 as at
    // 224, and the epilogue's hold on the issuer at every tile is small
    // against a long main loop.  (FP8G_TILE_N(8) asks for it at any K.)
    const int tn_override = static_cast<int>((p.flags >> 16) & 15u);
    const bool bs_wide = p.sf_k && (num_kb >= kWideBlockScaledKb || tn_override == 8);
    const int max_tn = p.sf_k && !bs_wide ? kMaxBlockScaledTile : 256;
    int tile_n = pick_tile_n(p.G * m_tiles, p.N, info.sms, max_tn);
    if (tn_override >= 1 && tn_override <= 8)
        tile_n = std::min(32 * tn_override, max_tn);
    const int64_t units_upper = p.G * m_tiles * cdiv(p.N, tile_n);
    if (units_upper > kMaxDim)
        return FP8G_ERR_UNSUPPORTED;
    args.tile_n = tile_n;
    if (p.sf_k) {
        plan_blockscaled(args, info, tile_n, static_cast<int>(p.G), p.flags);
        // 128-element groups: the scale loads use their own ring, issued a
        // scale set (four K blocks) ahead of the operands, so a stage holds
        // only the operand tiles -- at 224 columns that leaves room for a
        // fifth stage.  Measured on GB300 (same box, graph replay, 1x128 /
        // 128x128 scales), scales riding in the stage of a set's first K
        // block against the ring: 4096^3 67.9 -> 65.0 us, 8192x7168x18432
        // 872 -> 818-851 us, 8192x18432x7168 885 -> 858-868 us.  With
        // 32-element groups (a set per K block) the ring's slot wait at every
        // K block made 4096^3 slower (101.8 -> 109.5 us): their scales stay in
        // the stages.
        if (p.sf_k == 1) {
            args.sf_ring = kSfRingSlots;
            args.sf_slot_bytes = sf_stage_bytes(tile_n);
            args.sf_off = 0;
            args.stage_bytes = kTileM * kBlockK + tile_n * kBlockK;
            args.stages = pick_stages(info, args.stage_bytes, static_cast<int>(p.G), p.flags,
                                      args.sf_ring * args.sf_slot_bytes);
        }
        if (tile_n > kMaxBlockScaledTile) {   // one accumulator buffer, then the scale sets
            args.acc_bufs = 1;
            args.sf_col0 = tile_n;
            args.sf_sets = std::min(kMaxSfSets, (kTmemCols - tile_n) / sf_set_cols(tile_n));
        }
        // Two MMA issuers (alternate K blocks, one accumulator each): with
        // two accumulator buffers per issuer when four tiles and two scale
        // sets fit in TMEM; with one (the epilogue then holds the issuers
        // back at every tile) only for 32-element groups, where it measured
        // faster than one issuer -- with 128-element groups it was slower.
        // (An even stage count keeps each stage with one issuer.)
        if (!(p.flags & FP8G_ONE_MMA_ISSUER) && args.stages >= 2) {
            const int set_cols = sf_set_cols(tile_n);
            const int sets2 = std::min(kMaxSfSets, (kTmemCols - 4 * tile_n) / set_cols);
            const int sets1 = std::min(kMaxSfSets, (kTmemCols - 2 * tile_n) / set_cols);
            if (sets2 >= 2 || (sets1 >= 2 && (p.sf_k == 4 || (p.flags & FP8G_TWO_MMA_ISSUERS)))) {
                args.dual_mma = 1;
                args.acc_bufs = sets2 >= 2 ? 2 : 1;
                args.sf_col0 = args.acc_bufs * 2 * tile_n;
                args.sf_sets = sets2 >= 2 ? sets2 : sets1;
                args.stages &= ~1;
            }
        }
    } else {
        args.stage_bytes = kTileM * kBlockK + tile_n * kBlockK;
        args.stages = pick_stages(info, args.stage_bytes, static_cast<int>(p.G), p.flags);
    }
    // Bands of M tiles whose token rows total about 48 MB stay resident in L2
    // while the weight tiles stream past them.
    const int64_t band = (48ll << 20) / (kTileM * p.K);
    args.raster_band = static_cast<int32_t>(std::max<int64_t>(1, std::min<int64_t>(band, m_tiles)));
    args.a_box_rows = dense && p.rows_a < kTileM ? static_cast<int32_t>(p.rows_a) : 0;
    const int grid = static_cast<int>(std::min<int64_t>(units_upper, info.sms));
    args.prefetch_kb = dense ? early_prefetch_kb(static_cast<int>(tile_n) * kBlockK, false) : 0;
    // Dense launches that leave SMs idle: the CTAs that start there fetch
    // the whole launch's weights into L2 while the previous launch runs.
    // Measured on GB300 (same box, graph replay): N=24576, K=1536 token tiles
    // (128 CTAs) 9.35 -> 8.75 us at M=1, 10.03 -> 8.82 us at M=64; with
    // weights of 117 MB (N=7168, K=16384) it lost (39.9 -> 46.3 us), so only
    // weights up to half of L2 are fetched this way.
    if (dense && grid < info.sms && p.N * p.K <= kSpareFetchMaxBytes)
        args.spare_ctas = info.sms - grid;
    if (describe) {
        describe_as(describe, FP8G_KERNEL_TOKEN_TILES, tile_n, args, false, false,
                    args.a_box_rows ? args.a_box_rows : kTileM, grid);
        return FP8G_OK;
    }
    if (!make_map(&tm0, p.A, p.K, p.rows_a, p.group_offsets ? 1 : p.G,
                  args.a_box_rows ? static_cast<uint32_t>(args.a_box_rows) : kTileM) ||
        !make_map(&tm1, p.B, p.K, p.N, p.G, static_cast<uint32_t>(tile_n)))
        return FP8G_ERR_CUDA;
    if (p.sf_k) {
        if (!make_sf_map(&tm2, p.sf_a, p.rows_a, ks, p.G, p.sf_a_ld, kTileM, 4) ||
            !make_sf_map(&tm3, p.sf_b, p.N, ks, p.G, p.sf_b_ld, static_cast<uint32_t>(tile_n), 4))
            return FP8G_ERR_CUDA;
    } else {
        tm2 = tm0;
        tm3 = tm1;
    }
    if (grid <= 0)
        return FP8G_OK;
    return launch_gemm_mn(tm0, tm1, tm2, tm3, args, grid, static_cast<size_t>(info.smem_optin), stream) ==
                   cudaSuccess
               ? FP8G_OK
               : FP8G_ERR_CUDA;
}

}  // namespace
}  // namespace fp8g

using namespace fp8g;

namespace fp8g {
namespace {

int apply_scales(const fp8g_scales *sc, int64_t G, int64_t rows, int64_t N, Problem &p)
{
    if (!sc)
        return FP8G_OK;
    int st = FP8G_OK;
    if (sc->out_a || sc->out_b) {
        st = check_scales(sc->out_a, sc->out_a_len, sc->out_b, sc->out_b_len, G, p.group_offsets ? rows : G * rows,
                          N, p);
        if (st != FP8G_OK)
            return st;
    }
    if (sc->block_a || sc->block_b) {
        // The A-side scale map's row coordinate would need 16-aligned group offsets.
        if (p.group_offsets)
            return FP8G_ERR_UNSUPPORTED;
        st = check_blockscales(sc->block_a, sc->block_a_ld, sc->block_b, sc->block_b_ld, sc->block_k, rows, N, p);
    }
    return st;
}

int dense_ex(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K, int a_dtype, int b_dtype,
             const fp8g_scales *sc, const fp8g_epilogue *epi, uint32_t flags, cudaStream_t stream)
{
    int st = check_common(A, B, D, N, K, a_dtype, b_dtype);
    if (st != FP8G_OK)
        return st;
    if (M <= 0 || M > kMaxDim)
        return FP8G_ERR_INVALID_ARG;
    Problem p{A, B, D, nullptr, nullptr, 1, M, N, K, M, a_dtype, b_dtype, flags};
    if ((st = apply_scales(sc, 1, M, N, p)) != FP8G_OK || (st = check_epilogue(epi, p)) != FP8G_OK)
        return st;
    return launch(p, stream);
}

int grouped_ex(const void *A, const void *B, void *D, const int32_t *masked_m, int64_t G, int64_t M_max, int64_t N,
               int64_t K, int64_t max_m_hint, int a_dtype, int b_dtype, const fp8g_scales *sc,
               const fp8g_epilogue *epi, uint32_t flags, cudaStream_t stream)
{
    int st = check_common(A, B, D, N, K, a_dtype, b_dtype);
    if (st != FP8G_OK)
        return st;
    if (!masked_m)
        return FP8G_ERR_INVALID_ARG;
    if (G <= 0 || M_max <= 0 || M_max > kMaxDim || max_m_hint < 0 || max_m_hint > M_max)
        return FP8G_ERR_INVALID_ARG;
    if (G > kMaxGroups)
        return FP8G_ERR_UNSUPPORTED;
    if (G * M_max > kMaxDim || G * N > kMaxDim)
        return FP8G_ERR_UNSUPPORTED;
    if (!aligned16(masked_m))
        return FP8G_ERR_MISALIGNED;
    const int64_t hint = max_m_hint > 0 ? max_m_hint : M_max;
    Problem p{A, B, D, masked_m, nullptr, G, M_max, N, K, hint, a_dtype, b_dtype, flags};
    if ((st = apply_scales(sc, G, M_max, N, p)) != FP8G_OK || (st = check_epilogue(epi, p)) != FP8G_OK)
        return st;
    if (!is_device_pointer(masked_m))
        return FP8G_ERR_INVALID_ARG;
    return launch(p, stream);
}

int contiguous_ex(const void *A, const void *B, void *D, const int32_t *offsets, int64_t G, int64_t M_total,
                  int64_t N, int64_t K, int64_t max_m_hint, int a_dtype, int b_dtype, const fp8g_scales *sc,
                  const fp8g_epilogue *epi, uint32_t flags, cudaStream_t stream)
{
    int st = check_common(A, B, D, N, K, a_dtype, b_dtype);
    if (st != FP8G_OK)
        return st;
    if (!offsets || G <= 0 || M_total <= 0 || M_total > kMaxDim || max_m_hint < 0 || max_m_hint > M_total)
        return FP8G_ERR_INVALID_ARG;
    if (G > kMaxGroups)
        return FP8G_ERR_UNSUPPORTED;
    if (G * N > kMaxDim)
        return FP8G_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(offsets) & 3u) != 0)
        return FP8G_ERR_MISALIGNED;
    const int64_t hint = max_m_hint > 0 ? max_m_hint : M_total;
    Problem p{A, B, D, nullptr, offsets, G, M_total, N, K, hint, a_dtype, b_dtype, flags};
    if ((st = apply_scales(sc, G, M_total, N, p)) != FP8G_OK || (st = check_epilogue(epi, p)) != FP8G_OK)
        return st;
    if (!is_device_pointer(offsets))
        return FP8G_ERR_INVALID_ARG;
    return launch(p, stream);
}

}  // namespace
}  // namespace fp8g

extern "C" int fp8_gemm_grouped_contiguous(const void *A, const void *B, void *D, const int32_t *group_offsets,
                                           int64_t G, int64_t M_total, int64_t N, int64_t K, int64_t max_m_hint,
                                           int a_dtype, int b_dtype, uint32_t flags, cudaStream_t stream)
{
    return contiguous_ex(A, B, D, group_offsets, G, M_total, N, K, max_m_hint, a_dtype, b_dtype, nullptr, nullptr,
                         flags, stream);
}

extern "C" int fp8_gemm_grouped_contiguous_ex(const void *A, const void *B, void *D, const int32_t *group_offsets,
                                              int64_t G, int64_t M_total, int64_t N, int64_t K, int64_t max_m_hint,
                                              int a_dtype, int b_dtype, const fp8g_scales *scales,
                                              const fp8g_epilogue *epilogue, uint32_t flags, cudaStream_t stream)
{
    return contiguous_ex(A, B, D, group_offsets, G, M_total, N, K, max_m_hint, a_dtype, b_dtype, scales, epilogue,
                         flags, stream);
}

extern "C" int fp8_gemm_nt(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K,
                           int a_dtype, int b_dtype, uint32_t flags, cudaStream_t stream)
{
    return dense_ex(A, B, D, M, N, K, a_dtype, b_dtype, nullptr, nullptr, flags, stream);
}

extern "C" int fp8_gemm_grouped_masked(const void *A, const void *B, void *D, const int32_t *masked_m,
                                       int64_t G, int64_t M_max, int64_t N, int64_t K, int64_t max_m_hint,
                                       int a_dtype, int b_dtype, uint32_t flags, cudaStream_t stream)
{
    return grouped_ex(A, B, D, masked_m, G, M_max, N, K, max_m_hint, a_dtype, b_dtype, nullptr, nullptr, flags,
                      stream);
}

extern "C" int fp8_gemm_nt_ex(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K,
                              int a_dtype, int b_dtype, const fp8g_scales *scales, const fp8g_epilogue *epilogue,
                              uint32_t flags, cudaStream_t stream)
{
    return dense_ex(A, B, D, M, N, K, a_dtype, b_dtype, scales, epilogue, flags, stream);
}

extern "C" int fp8_gemm_grouped_masked_ex(const void *A, const void *B, void *D, const int32_t *masked_m,
                                          int64_t G, int64_t M_max, int64_t N, int64_t K, int64_t max_m_hint,
                                          int a_dtype, int b_dtype, const fp8g_scales *scales,
                                          const fp8g_epilogue *epilogue, uint32_t flags, cudaStream_t stream)
{
    return grouped_ex(A, B, D, masked_m, G, M_max, N, K, max_m_hint, a_dtype, b_dtype, scales, epilogue, flags,
                      stream);
}

extern "C" int fp8_gemm_nt_scaled(const void *A, const void *B, void *D, int64_t M, int64_t N,
                                  int64_t K, int a_dtype, int b_dtype, const float *scale_a,
                                  int64_t scale_a_len, const float *scale_b, int64_t scale_b_len,
                                  uint32_t flags, cudaStream_t stream)
{
    if (!scale_a || !scale_b)
        return FP8G_ERR_INVALID_ARG;
    const fp8g_scales sc{scale_a, scale_a_len, scale_b, scale_b_len, nullptr, 0, nullptr, 0, 0};
    return dense_ex(A, B, D, M, N, K, a_dtype, b_dtype, &sc, nullptr, flags, stream);
}

extern "C" int fp8_gemm_grouped_masked_scaled(const void *A, const void *B, void *D,
                                              const int32_t *masked_m, int64_t G, int64_t M_max,
                                              int64_t N, int64_t K, int64_t max_m_hint, int a_dtype,
                                              int b_dtype, const float *scale_a, int64_t scale_a_len,
                                              const float *scale_b, int64_t scale_b_len, uint32_t flags,
                                              cudaStream_t stream)
{
    if (!scale_a || !scale_b)
        return FP8G_ERR_INVALID_ARG;
    const fp8g_scales sc{scale_a, scale_a_len, scale_b, scale_b_len, nullptr, 0, nullptr, 0, 0};
    return grouped_ex(A, B, D, masked_m, G, M_max, N, K, max_m_hint, a_dtype, b_dtype, &sc, nullptr, flags,
                      stream);
}

extern "C" int fp8_gemm_nt_blockscaled(const void *A, const void *B, void *D, int64_t M, int64_t N,
                                       int64_t K, int a_dtype, int b_dtype, const uint8_t *sf_a,
                                       int64_t sf_a_ld, const uint8_t *sf_b, int64_t sf_b_ld,
                                       int sf_group_k, uint32_t flags, cudaStream_t stream)
{
    if (!sf_a || !sf_b)
        return FP8G_ERR_INVALID_ARG;
    const fp8g_scales sc{nullptr, 0, nullptr, 0, sf_a, sf_a_ld, sf_b, sf_b_ld, sf_group_k};
    return dense_ex(A, B, D, M, N, K, a_dtype, b_dtype, &sc, nullptr, flags, stream);
}

extern "C" int fp8_gemm_grouped_masked_blockscaled(const void *A, const void *B, void *D,
                                                   const int32_t *masked_m, int64_t G, int64_t M_max,
                                                   int64_t N, int64_t K, int64_t max_m_hint, int a_dtype,
                                                   int b_dtype, const uint8_t *sf_a, int64_t sf_a_ld,
                                                   const uint8_t *sf_b, int64_t sf_b_ld, int sf_group_k,
                                                   uint32_t flags, cudaStream_t stream)
{
    if (!sf_a || !sf_b)
        return FP8G_ERR_INVALID_ARG;
    const fp8g_scales sc{nullptr, 0, nullptr, 0, sf_a, sf_a_ld, sf_b, sf_b_ld, sf_group_k};
    return grouped_ex(A, B, D, masked_m, G, M_max, N, K, max_m_hint, a_dtype, b_dtype, &sc, nullptr, flags,
                      stream);
}

extern "C" int fp8g_get_device_status(int32_t *info, cudaStream_t stream)
{
    if (!info)
        return FP8G_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return FP8G_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess)
        return FP8G_ERR_CUDA;
    if (read_and_clear_status(info) != cudaSuccess)
        return FP8G_ERR_CUDA;
    if (info[0] == FP8G_ERR_TIMEOUT) {
        // An aborted stream-K launch can leave arrival counts behind, in the
        // workspace of whichever stream it ran on: once the device is idle,
        // clear the counters of every stream of this device.
        if (cudaDeviceSynchronize() != cudaSuccess)
            return FP8G_ERR_CUDA;
        std::lock_guard<std::mutex> lk(g_mu);
        for (Workspace &w : g_ws)
            if (w.dev == dev && w.counters && cudaMemset(w.counters, 0, w.counter_bytes) != cudaSuccess)
                return FP8G_ERR_CUDA;
        if (cudaDeviceSynchronize() != cudaSuccess)
            return FP8G_ERR_CUDA;
    }
    return FP8G_OK;
}

extern "C" int fp8g_init(int64_t max_tiles, cudaStream_t stream)
{
    int dev = 0;
    DeviceInfo info;
    int st = current_device(&dev, &info);
    if (st != FP8G_OK)
        return st;
    if (max_tiles < 0 || max_tiles > kMaxDim)
        return FP8G_ERR_INVALID_ARG;
    const int64_t tiles = max_tiles ? max_tiles : kDefaultInitTiles;
    // The largest partial-tile area any launch takes: two FP32 tiles of 128
    // x 256 per CTA, one CTA per SM (SwapAB chunks and SM-pair tiles are at
    // most 256 wide); counters as the SM-pair kernel counts them (one pair
    // per tile, CTA and epilogue warp; the SwapAB kernel needs half that).
    const size_t ws_bytes = static_cast<size_t>(info.sms) * 2 * kTileM * 256 * sizeof(float);
    float *ws = nullptr;
    int32_t *counters = nullptr;
    return ensure_workspace(dev, stream, ws_bytes, pair_counter_bytes(tiles), &ws, &counters);
}

extern "C" int fp8g_release_stream(cudaStream_t stream)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return FP8G_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    const cudaStream_t key = stream_key(stream);
    const std::thread::id th = key == cudaStreamPerThread ? std::this_thread::get_id() : std::thread::id{};
    for (size_t i = 0; i < g_ws.size(); ++i) {
        Workspace &w = g_ws[i];
        if (w.dev != dev || w.stream != key || w.thread != th)
            continue;
        if (cudaStreamSynchronize(stream) != cudaSuccess)
            return FP8G_ERR_CUDA;
        const bool ok = free_workspace(w);
        g_ws.erase(g_ws.begin() + static_cast<std::ptrdiff_t>(i));
        return ok ? FP8G_OK : FP8G_ERR_CUDA;
    }
    return FP8G_OK;
}

extern "C" int fp8g_shutdown(void)
{
    std::lock_guard<std::mutex> lk(g_mu);
    int prev = 0;
    const bool have_prev = cudaGetDevice(&prev) == cudaSuccess;
    int rc = FP8G_OK;
    for (Workspace &w : g_ws) {
        if (cudaSetDevice(w.dev) != cudaSuccess) {
            rc = FP8G_ERR_CUDA;
            continue;
        }
        if (!free_workspace(w))
            rc = FP8G_ERR_CUDA;
    }
    g_ws.clear();
    if (have_prev)
        cudaSetDevice(prev);
    else
        cudaGetLastError();
    return rc;
}

extern "C" int fp8g_describe_plan(int layout, int64_t G, int64_t rows, int64_t N, int64_t K, int64_t token_hint,
                                  int sf_group_k, uint32_t flags, int sms, int smem_optin, fp8g_plan *out)
{
    if (!out)
        return FP8G_ERR_INVALID_ARG;
    std::memset(out, 0, sizeof(*out));
    if (layout < 0 || layout > 2 || G <= 0 || rows <= 0 || N <= 0 || K <= 0 || rows > kMaxDim || N > kMaxDim ||
        K > kMaxDim || K % 16 != 0 || N % 8 != 0 || token_hint < 0 || token_hint > rows ||
        (layout == 0 && G != 1) || sms < 0 || smem_optin < 0 || (sms == 0) != (smem_optin == 0) ||
        (sf_group_k != 0 && sf_group_k != 32 && sf_group_k != 128))
        return FP8G_ERR_INVALID_ARG;
    if (G > kMaxGroups || G * N > kMaxDim || (layout == 1 && G * rows > kMaxDim) || (layout == 2 && sf_group_k))
        return FP8G_ERR_UNSUPPORTED;
    // Planning reads no operand: the layout pointers only mark the layout.
    static const int32_t kLayoutMark[1] = {0};
    const int64_t hint = layout == 0 ? rows : (token_hint > 0 ? token_hint : rows);
    Problem p{nullptr, nullptr, nullptr, layout == 1 ? kLayoutMark : nullptr, layout == 2 ? kLayoutMark : nullptr,
              G, rows, N, K, hint, FP8G_E4M3, FP8G_E4M3, flags};
    p.sf_k = sf_group_k ? static_cast<int>(kBlockK / sf_group_k) : 0;
    DeviceInfo info;
    if (sms > 0) {
        info.ready = true;
        info.sms = sms;
        info.smem_optin = smem_optin;
        info.cc_major = 10;
        info.cc_minor = 3;
    } else {
        int dev = 0;
        const int st = current_device(&dev, &info);
        if (st != FP8G_OK)
            return st;
    }
    return launch(p, nullptr, &info, out);
}

extern "C" uint64_t fp8g_set_wait_timeout_ns(uint64_t ns)
{
    return g_timeout_ns.exchange(ns ? ns : kDefaultTimeoutNs);
}

extern "C" const char *fp8g_status_string(int code)
{
    switch (code) {
    case FP8G_OK: return "FP8G_OK";
    case FP8G_ERR_INVALID_ARG: return "FP8G_ERR_INVALID_ARG";
    case FP8G_ERR_MISALIGNED: return "FP8G_ERR_MISALIGNED";
    case FP8G_ERR_UNSUPPORTED: return "FP8G_ERR_UNSUPPORTED";
    case FP8G_ERR_CUDA: return "FP8G_ERR_CUDA";
    case FP8G_ERR_TIMEOUT: return "FP8G_ERR_TIMEOUT";
    case FP8G_ERR_NO_DEVICE: return "FP8G_ERR_NO_DEVICE";
    case FP8G_ERR_MASKED_M_RANGE: return "FP8G_ERR_MASKED_M_RANGE";
    default: return "FP8G_UNKNOWN_STATUS";
    }
}

extern "C" int fp8g_version(void) { return 100; }
