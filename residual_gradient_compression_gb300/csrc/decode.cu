// AdaComp decode-and-accumulate for sm_103a: K learners' sparse ternary messages
// are summed into one dense fp32 gradient, learner by learner.
//
// The pages say only that data-parallel learners exchange their quantised
// gradients ("AdaComp (Adaptive Residual Gradient Compression)", abstract and
// summary paragraph); this library reads the combination as a plain sum in learner
// order, dense[j] = fl32(dense[j] + sign * s_k) for k = 0..K-1.
//
// Five launches:
//   tile_sums   per (learner, run of tiles): check that the message is long enough to
//               hold its header and counts, check the header's B and the tiles'
//               per-bin counts, and sum the counts of each tile;
//   tile_scan   per (message, chunk of tiles): exclusive prefix of the tile sums, i.e.
//               where each tile's codes start in that message, the message's total,
//               and the check that its length is exactly 8 + 2B + w * total;
//   check       per (learner, 128 bins, or one tile of long bins): within every bin
//               the code offsets rise strictly and stay below the bin's length;
//   accumulate  per tile of the layers that are streamed: the dense tile is staged
//               in shared memory, every learner's codes for the tile are applied in
//               learner order, and the tile is written back;
//   sparse_accumulate  per tile of the layers whose learners sent few codes: the
//               codes are added in place in global memory, learner by learner.
// A message that fails any check is rejected as a whole before anything is added
// (its flag in the workspace). One warp owns each bin range of a tile, no two threads
// touch one element within a learner, and no float atomics are used, so the result
// is deterministic.
#include "adacomp_internal.cuh"

namespace adacomp {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kDecThreads = 256;

// Layer of tile t from a shared-memory array of the layers' first tiles.
__device__ __forceinline__ int layer_of(const uint32_t* tb, int num_layers, uint32_t t)
{
    int lo = 0, hi = num_layers - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (tb[mid] <= t) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ unsigned long long* layer_codes(uint8_t* ws)
{
    return reinterpret_cast<unsigned long long*>(ws + kDecodeLayerCodes);
}

// One byte per layer, set when the layer is summed in place in global memory,
// without staging its dense tiles: when all learners together sent fewer than
// n / 16 of its elements, each code costs about one 32-byte sector read and write,
// against 8 bytes per element for streaming the dense array. (The fused SGD step
// always streams: every element's weights and momentum change.)
constexpr size_t kDecodeSparseFlags = 1040;  // after the bad-message bytes
__device__ __forceinline__ uint8_t* sparse_flags(uint8_t* ws) { return ws + kDecodeSparseFlags; }

__device__ __forceinline__ uint64_t* tile_offsets(uint8_t* ws, int k, uint32_t T)
{
    return reinterpret_cast<uint64_t*>(ws + kDecodeFixed + (size_t)k * decode_per_learner(T));
}

__device__ __forceinline__ uint32_t* tile_sums_of(uint8_t* ws, int k, uint32_t T)
{
    return reinterpret_cast<uint32_t*>(ws + kDecodeFixed + (size_t)k * decode_per_learner(T) + decode_sums_offset(T));
}

constexpr uint32_t kBadSum = 0xffffffffu;  // the sum of a tile whose counts are invalid

// Layer of validation task u (tasks of a learner are numbered across the layers).
__device__ __forceinline__ int layer_of_task(const uint32_t* vb, int num_layers, uint32_t u)
{
    int lo = 0, hi = num_layers - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (vb[mid] <= u) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// A run of whole tiles of one layer holding at most kValBins bins (or one tile when
// a tile holds more): the unit of work of the counting and validation kernels.
struct Run {
    int layer;
    uint32_t t0, ntiles;  // first tile (global index) and tiles
    uint32_t b0, nb;      // first bin (in the layer) and bins
};

__device__ __forceinline__ Run run_of(const KGroup& g, const uint32_t* vb, uint32_t u)
{
    Run R;
    R.layer = layer_of_task(vb, g.num_layers, u);
    const KLayer& ly = g.layer[R.layer];
    const uint32_t tpt = val_tiles_per_task(ly.bins_per_tile);
    const uint32_t i0 = (u - vb[R.layer]) * tpt;  // first tile within the layer
    R.t0 = ly.tile_begin + i0;
    R.ntiles = min(tpt, ly.num_tiles - i0);
    R.b0 = i0 * ly.bins_per_tile;
    R.nb = (uint32_t)min((uint64_t)R.ntiles * ly.bins_per_tile, (uint64_t)(ly.nbins - R.b0));
    return R;
}

// One warp per (learner k, run): the message must be at least 8 + 2B bytes long
// (else nothing of it is read), the header's B must equal the layer's B, and no
// count may exceed its bin's length; otherwise every tile sum of the run is
// kBadSum. Lanes take the run's bins (all loads issued at once, coalesced) and add
// them into per-tile sums in shared memory. The warp of a message's first run also
// clears the message's rejection byte, which the later kernels set.
__global__ void __launch_bounds__(kDecThreads) tile_sums_kernel(const __grid_constant__ KGroup g,
                                                                const __grid_constant__ DecodeParams p, uint8_t* ws)
{
    ptx::griddep_wait();  // whatever the stream ran before
    __shared__ uint32_t vb[kMaxGroup + 1];
    __shared__ uint32_t sums_s[kDecThreads / 32][kValBins];
    for (int e = threadIdx.x; e <= g.num_layers; e += kDecThreads) vb[e] = p.val_begin[e];
    if (blockIdx.x == 0 && threadIdx.x == 0) reinterpret_cast<uint32_t*>(ws)[2] = 0u;  // scan blocks done
    __syncthreads();
    const uint32_t T = g.total_tiles;
    const int K = p.K;
    const int lane = threadIdx.x & 31;
    const uint32_t per_learner = vb[g.num_layers];
    const uint64_t task = (uint64_t)blockIdx.x * (kDecThreads / 32) + (threadIdx.x >> 5);
    if (task >= (uint64_t)K * per_learner) return;
    const int k = (int)(task / per_learner);
    const Run R = run_of(g, vb, (uint32_t)(task - (uint64_t)k * per_learner));
    const int l = R.layer;
    const KLayer& ly = g.layer[l];
    if (R.t0 == ly.tile_begin && lane == 0) ws[16 + l * K + k] = 0;
    uint32_t* out = tile_sums_of(ws, k, T) + R.t0;
    const uint8_t* msg = p.msg[l * K + k];
    if (p.len[l * K + k] < 8ull + 2ull * ly.nbins) {  // too short for its header and counts: read nothing
        for (uint32_t i = lane; i < R.ntiles; i += 32) out[i] = kBadSum;
        return;
    }
    const uint32_t hdr_b = *reinterpret_cast<const uint32_t*>(msg + 4);
    const uint16_t* cnt = reinterpret_cast<const uint16_t*>(msg + 8) + R.b0;
    const uint32_t last_len = (uint32_t)(ly.n - (int64_t)(ly.nbins - 1) * ly.bin_len);
    bool ok = true;
    if (R.ntiles == 1) {  // one tile (possibly of more than kValBins bins): a warp sum
        uint32_t sum = 0;
        for (uint32_t b = lane; b < R.nb; b += 32) {
            const uint32_t c = cnt[b];
            ok = ok && c <= (R.b0 + b == ly.nbins - 1 ? last_len : (uint32_t)ly.bin_len);
            sum += c;
        }
        ok = __all_sync(kFull, ok) && hdr_b == ly.nbins;
        sum = __reduce_add_sync(kFull, sum);
        if (lane == 0) out[0] = ok ? sum : kBadSum;
        return;
    }
    uint32_t* sums = sums_s[threadIdx.x >> 5];
    for (uint32_t i = lane; i < R.ntiles; i += 32) sums[i] = 0u;
    __syncwarp();
    uint32_t c[kValBins / 32];
#pragma unroll
    for (int i = 0; i < (int)(kValBins / 32); ++i) {
        const uint32_t b = i * 32 + lane;
        c[i] = b < R.nb ? cnt[b] : 0u;
    }
#pragma unroll
    for (int i = 0; i < (int)(kValBins / 32); ++i) {
        const uint32_t b = i * 32 + lane;
        if (b < R.nb) {
            ok = ok && c[i] <= (R.b0 + b == ly.nbins - 1 ? last_len : (uint32_t)ly.bin_len);
            if (c[i]) atomicAdd(&sums[b / ly.bins_per_tile], c[i]);
        }
    }
    ok = __all_sync(kFull, ok) && hdr_b == ly.nbins;
    __syncwarp();
    for (uint32_t i = lane; i < R.ntiles; i += 32) out[i] = ok ? sums[i] : kBadSum;
}

// Grid (chunk, layer * K + learner): the tile sums of one message become the tiles'
// exclusive code offsets, a chunk of CH tiles per CTA. The CTA sums the message's
// tiles before its chunk (coalesced, kScanPer loads per thread in flight; the
// repeated reads are small and hit L2), then scans its own chunk in passes of
// kScanPer * 1024 tiles (thread tid loads tiles pass + i * 1024 + tid; the warps scan
// each row with shuffles and one warp scans the row-by-warp totals in row order). A
// chunk with a bad tile rejects the message; the CTA of the message's last chunk
// checks that its length is exactly 8 + 2B + w * (its code count) and records that
// count. The last CTA of the grid decides, per layer, whether the layer is summed in
// place (all learners' codes < n / 16).
constexpr int kScanThreads = 1024;
constexpr int kScanWarps = kScanThreads / 32;
constexpr int kScanPer = 4;

__global__ void __launch_bounds__(kScanThreads) tile_scan_kernel(const __grid_constant__ KGroup g,
                                                                 const __grid_constant__ DecodeParams p, uint8_t* ws,
                                                                 uint32_t CH)
{
    ptx::griddep_wait();  // the tile sums
    __shared__ unsigned long long wt[kScanPer][kScanWarps];
    __shared__ unsigned long long wx[kScanPer][kScanWarps];
    __shared__ unsigned long long red[kScanWarps];
    __shared__ unsigned long long carry_s;
    __shared__ uint32_t last_s;
    const int K = p.K;
    const int lk = blockIdx.y;
    const int l = lk / K, k = lk - (lk / K) * K;
    const KLayer& ly = g.layer[l];
    const uint32_t T = g.total_tiles;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (blockIdx.x == 0 && blockIdx.y == 0 && tid == 0) {
        reinterpret_cast<uint32_t*>(ws)[0] = (uint32_t)K;
        reinterpret_cast<uint32_t*>(ws)[1] = (uint32_t)g.num_layers;
    }
    const uint32_t nt = ly.num_tiles;
    const uint32_t c0 = blockIdx.x * CH;
    if (c0 < nt) {
        const uint32_t c1 = min(nt, c0 + CH);
        const uint32_t* sum = tile_sums_of(ws, k, T) + ly.tile_begin;
        uint64_t* off = tile_offsets(ws, k, T) + ly.tile_begin;
        // the codes of the message's tiles before the chunk
        unsigned long long before = 0;
        for (uint32_t i0 = 0; i0 < c0; i0 += kScanPer * kScanThreads) {
            uint32_t v[kScanPer];
#pragma unroll
            for (int u = 0; u < kScanPer; ++u) {
                const uint32_t i = i0 + u * kScanThreads + tid;
                v[u] = i < c0 ? sum[i] : 0u;
            }
#pragma unroll
            for (int u = 0; u < kScanPer; ++u) before += v[u];
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) before += __shfl_xor_sync(kFull, before, o);
        if (lane == 0) red[warp] = before;
        if (tid == 0) carry_s = 0ull;
        __syncthreads();
        if (warp == 0) {
            unsigned long long b = red[lane];
#pragma unroll
            for (int o = 16; o; o >>= 1) b += __shfl_xor_sync(kFull, b, o);
            if (lane == 0) carry_s = b;
        }
        __syncthreads();
        bool bad = false;
        for (uint32_t base = c0; base < c1; base += kScanPer * kScanThreads) {
            uint64_t v[kScanPer], inc[kScanPer];
            bool mine_bad = false;
#pragma unroll
            for (int i = 0; i < kScanPer; ++i) {
                const uint32_t j = base + i * kScanThreads + tid;
                const uint32_t x = j < c1 ? sum[j] : 0u;
                mine_bad = mine_bad || x == kBadSum;
                v[i] = x;
            }
            if (__syncthreads_or(mine_bad)) {  // a bad tile: the whole message is rejected
                bad = true;
                break;
            }
#pragma unroll
            for (int i = 0; i < kScanPer; ++i) {
                inc[i] = v[i];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned long long y = __shfl_up_sync(kFull, inc[i], o);
                    if (lane >= o) inc[i] += y;
                }
                if (lane == 31) wt[i][warp] = inc[i];
            }
            __syncthreads();
            if (warp == 0) {
                unsigned long long c = carry_s;
#pragma unroll
                for (int i = 0; i < kScanPer; ++i) {
                    const unsigned long long x = wt[i][lane];
                    unsigned long long sx = x;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const unsigned long long y = __shfl_up_sync(kFull, sx, o);
                        if (lane >= o) sx += y;
                    }
                    wx[i][lane] = c + (sx - x);
                    c += __shfl_sync(kFull, sx, 31);
                }
                if (lane == 0) carry_s = c;
            }
            __syncthreads();
#pragma unroll
            for (int i = 0; i < kScanPer; ++i) {
                const uint32_t j = base + i * kScanThreads + tid;
                if (j < c1) off[j] = wx[i][warp] + (inc[i] - v[i]);
            }
        }
        __syncthreads();
        if (tid == 0) {
            if (c1 == nt) {  // the message's last chunk: its code count and its length
                const unsigned long long total = carry_s;
                bad = bad || p.len[lk] != 8ull + 2ull * ly.nbins + (unsigned long long)ly.code_bytes * total;
                layer_codes(ws)[lk] = total;
            }
            if (bad) ws[16 + lk] = 1;
        }
    }
    if (tid == 0) {
        __threadfence();
        last_s = atomicAdd(reinterpret_cast<uint32_t*>(ws) + 2, 1u) == gridDim.x * gridDim.y - 1u ? 1u : 0u;
    }
    __syncthreads();
    if (last_s) {  // every message is scanned: decide which layers are summed in place
        __threadfence();
        for (int e = tid; e < g.num_layers; e += kScanThreads) {
            const volatile unsigned long long* c = layer_codes(ws) + (size_t)e * K;
            const volatile uint8_t* badb = ws + 16 + e * K;
            unsigned long long sum = 0;
            for (int j = 0; j < K; ++j) sum += badb[j] ? 0ull : c[j];
            sparse_flags(ws)[e] = sum * 16ull < (unsigned long long)g.layer[e].n ? 1 : 0;
        }
    }
}

// One warp per (learner k, task of at most kChkBins bins) of a message not already
// rejected: within every bin the code offsets must rise strictly (a message gives
// each element at most one code) and stay below the bin's length (L_T, or the
// layer's last, shorter bin); otherwise the message is rejected as a whole, before
// anything is added. Bins shorter than kChkLongBin: lane b takes the counts of bins
// b, b + 32, ... of the task (coalesced) and their exclusive prefix (warp scans); the
// task's codes are one contiguous run, which the lanes read 32 at a time (coalesced),
// each offset compared with the one before it (a shuffle) and with its bin's length;
// the descents found are matched against those at the bins' first codes. Longer
// bins: one task per tile, the lanes over each bin's codes.
__device__ __forceinline__ int layer_of_chk(const uint32_t* cb, int num_layers, uint32_t u)
{
    int lo = 0, hi = num_layers - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cb[mid] <= u) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// The lanes over a run of `run` codes of kW bytes from `codes` (a message whose start
// is 16-byte aligned, so every 16-byte block that holds one of its bytes may be read):
// 16 bytes per lane, i.e. 16 / kW codes, 32 lanes a round, kChkDepth rounds loaded
// at once. Counts the descents (a
// code whose offset is not above that of the code before it; the first code has none
// before it) and the largest offset of the lane's codes.
constexpr int kChkDepth = 4;

template <int kW>
__device__ __forceinline__ void chk_run(const uint8_t* codes, uint32_t run, uint32_t& descents, int32_t& omax,
                                        int lane)
{
    constexpr int E = 16 / kW;
    const uintptr_t a = reinterpret_cast<uintptr_t>(codes);
    const uint4* ch = reinterpret_cast<const uint4*>(a & ~uintptr_t(15));
    const int32_t skip = (int32_t)((a & 15u) / kW);  // codes of the first block before position 0
    const uint32_t nch = (uint32_t)(skip + (int64_t)run + E - 1) / E;
    int32_t carry = -1;  // the offset before the lane's first code, from the previous round
    // kChkDepth rounds' loads are issued before the first of them is used
    for (uint32_t g0 = 0; g0 < nch; g0 += 32 * kChkDepth) {
        uint4 v[kChkDepth];
#pragma unroll
        for (int d = 0; d < kChkDepth; ++d) {
            const uint32_t ci = g0 + 32 * d + (uint32_t)lane;
            v[d] = ci < nch ? ch[ci] : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int d = 0; d < kChkDepth; ++d) {
            const uint32_t ci = g0 + 32 * d + (uint32_t)lane;
            if (g0 + 32 * d >= nch) break;
            const int64_t q0 = (int64_t)ci * E - skip;  // position of the block's first code
            const uint32_t wv[4] = {v[d].x, v[d].y, v[d].z, v[d].w};
            int32_t o[E];
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const uint32_t code =
                    kW == 2 ? (wv[e >> 1] >> ((e & 1) * 16)) & 0xffffu : (wv[e >> 2] >> ((e & 3) * 8)) & 0xffu;
                o[e] = q0 + e < 0 ? -1 : (int32_t)(code >> 1);
            }
            int32_t prev = __shfl_up_sync(kFull, o[E - 1], 1);
            if (lane == 0) prev = carry;
            carry = __shfl_sync(kFull, o[E - 1], 31);
            if (q0 >= 0 && q0 + E <= (int64_t)run) {  // every code of the block is in the run
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    descents += o[e] <= prev ? 1u : 0u;
                    omax = max(omax, o[e]);
                    prev = o[e];
                }
            } else if (ci < nch) {  // the run's first or last block
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int64_t q = q0 + e;
                    if (q >= 0 && q < (int64_t)run) {
                        descents += o[e] <= prev ? 1u : 0u;
                        omax = max(omax, o[e]);
                    }
                    prev = o[e];
                }
            }
        }
    }
}

// Loads that the compiler keeps where they are written (ahead of a branch that could
// make them unneeded), so that they are in flight together.
__device__ __forceinline__ uint32_t ld_early_u8(const uint8_t* a)
{
    unsigned short v;
    asm volatile("ld.global.u8 %0, [%1];" : "=h"(v) : "l"(a));
    return v;
}
__device__ __forceinline__ uint32_t ld_early_u8_nc(const uint8_t* a)
{
    unsigned short v;
    asm volatile("ld.global.nc.u8 %0, [%1];" : "=h"(v) : "l"(a));
    return v;
}
__device__ __forceinline__ uint32_t ld_early_u16(const uint16_t* a)
{
    unsigned short v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(a));
    return v;
}
__device__ __forceinline__ uint64_t ld_early_u64(const uint64_t* a)
{
    uint64_t v;
    asm volatile("ld.global.nc.u64 %0, [%1];" : "=l"(v) : "l"(a));
    return v;
}

// kLongOnly: every layer's bins have kChkLongBin elements or more. Those walks are
// bound by load latency and run best with four CTAs per SM; the short-bin path runs
// best unconstrained (74 registers, no spills).
template <bool kLongOnly>
__global__ void __launch_bounds__(kDecThreads, kLongOnly ? 4 : 1) check_kernel(const __grid_constant__ KGroup g,
                                                            const __grid_constant__ DecodeParams p, uint8_t* ws)
{
    ptx::griddep_wait();  // the offsets and the rejections so far
    constexpr int R = (int)(kChkBins / 32);  // bins per lane
    __shared__ uint32_t cb[kMaxGroup + 1];
    for (int e = threadIdx.x; e <= g.num_layers; e += kDecThreads) cb[e] = p.chk_begin[e];
    __syncthreads();
    const int K = p.K;
    const int lane = threadIdx.x & 31;
    const uint32_t per_learner = cb[g.num_layers];
    const uint64_t task = (uint64_t)blockIdx.x * (kDecThreads / 32) + (threadIdx.x >> 5);
    if (task >= (uint64_t)K * per_learner) return;
    const int k = (int)(task / per_learner);
    const uint32_t u = (uint32_t)(task - (uint64_t)k * per_learner);
    const int l = layer_of_chk(cb, g.num_layers, u);
    const KLayer& ly = g.layer[l];
    // A message too short for its counts was rejected by the counting kernel and
    // nothing of it is read; otherwise its rejection byte (set by the counting or the
    // scan kernel), its counts and its tile offset are loaded together, and a
    // rejected message is left there.
    if (p.len[l * K + k] < 8ull + 2ull * ly.nbins) return;
    const uint32_t rejected = ld_early_u8(ws + 16 + l * K + k);
    const uint32_t i = u - cb[l];
    const uint32_t bpt = ly.bins_per_tile;
    if (kLongOnly || ly.bin_len >= kChkLongBin) {  // long bins: task i is tile i, the lanes over each bin's codes
        const uint32_t tb0 = i * bpt;
        const uint32_t nbt = min(bpt, ly.nbins - tb0);  // <= 4 bins of 1024 or more
        const uint8_t* msg = p.msg[l * K + k];
        const uint32_t c = (uint32_t)lane < nbt ? ld_early_u16(reinterpret_cast<const uint16_t*>(msg + 8) + tb0 + lane) : 0u;
        const uint64_t toff = ld_early_u64(tile_offsets(ws, k, g.total_tiles) + ly.tile_begin + i);
        if (rejected) return;
        uint32_t incl = c;
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            const uint32_t y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += y;
        }
        const uint8_t* codes = msg + 8 + 2ull * ly.nbins;
        const bool wide = ly.code_bytes == 2;
        bool ok = true;
        for (uint32_t b = 0; b < nbt; ++b) {
            const uint32_t cb_ = __shfl_sync(kFull, c, (int)b);
            const uint64_t first = toff + __shfl_sync(kFull, incl - c, (int)b);
            const uint32_t len = tb0 + b == ly.nbins - 1 ? (uint32_t)(ly.n - (int64_t)(ly.nbins - 1) * ly.bin_len)
                                                         : (uint32_t)ly.bin_len;
            int32_t carry = -1;  // the previous round's last offset
            for (uint32_t j0 = 0; j0 < cb_; j0 += 32) {
                const uint32_t j = j0 + lane;
                const int32_t o = j < cb_ ? (int32_t)((wide ? reinterpret_cast<const uint16_t*>(codes)[first + j]
                                                            : codes[first + j]) >> 1)
                                          : 0x7fffffff;
                int32_t prev = __shfl_up_sync(kFull, o, 1);
                if (lane == 0) prev = carry;
                ok = ok && (j >= cb_ || ((uint32_t)o < len && o > prev));
                carry = __shfl_sync(kFull, o, 31);
            }
        }
        if (!__all_sync(kFull, ok) && lane == 0) ws[16 + l * K + k] = 1;
        return;
    }
    // the task's bins [b0, b0 + nb) of the layer
    uint32_t b0, nb;
    uint32_t pre = 0;  // tile-spanning tasks: the codes of the tile's bins before the task's
    const bool whole = bpt <= kChkBins;  // the task is whole tiles
    if (whole) {
        const uint32_t tpt = kChkBins / bpt;
        b0 = i * tpt * bpt;
        nb = min(tpt * bpt, ly.nbins - b0);
    } else {
        const uint32_t per = (bpt + kChkBins - 1) / kChkBins;
        const uint32_t tile = i / per;
        const uint32_t tb0 = tile * bpt;
        b0 = tb0 + (i - tile * per) * kChkBins;
        const uint32_t tend = min(tb0 + bpt, ly.nbins);
        if (b0 >= tend) return;
        nb = min(kChkBins, tend - b0);
    }
    const uint8_t* msg = p.msg[l * K + k];
    const uint16_t* cnt = reinterpret_cast<const uint16_t*>(msg + 8);
    uint32_t c[R], ex[R];  // bin r * 32 + lane: its count and the task's codes before it
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const uint32_t j = r * 32 + lane;
        c[r] = j < nb ? ld_early_u16(cnt + b0 + j) : 0u;
    }
    const uint64_t toff = ld_early_u64(tile_offsets(ws, k, g.total_tiles) + ly.tile_begin + b0 / bpt);
    if (rejected) return;
    if (!whole) {
        const uint32_t tb0 = (b0 / bpt) * bpt;
        for (uint32_t b = tb0 + lane; b < b0; b += 32) pre += cnt[b];
        pre = __reduce_add_sync(kFull, pre);
    }
    uint32_t run = 0;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        uint32_t incl = c[r];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += y;
        }
        ex[r] = run + incl - c[r];
        run += __shfl_sync(kFull, incl, 31);
    }
    // The task's codes are contiguous: positions 0 .. run - 1 from its first code.
    const uint64_t first = toff + pre;
    const bool wide = ly.code_bytes == 2;
    const uint8_t* codes = msg + 8 + 2ull * ly.nbins + (uint64_t)ly.code_bytes * first;
    auto off_at = [&](uint32_t q) -> int32_t {
        return (int32_t)((wide ? reinterpret_cast<const uint16_t*>(codes)[q] : codes[q]) >> 1);
    };
    // A descent is a position q >= 1 whose offset is not above the one before it. The
    // offsets rise strictly within every bin exactly when every descent is the first
    // code of a bin, i.e. when the descents number as many as the first codes (of the
    // nonempty bins, past position 0) that are descents.
    // (the codes at the bins' first codes are loaded before the run's, so that both
    // are in flight at once)
    uint32_t at_cur[R], at_prev[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        at_cur[r] = at_prev[r] = 0u;
        if (c[r] != 0u && ex[r] != 0u) {
            if (wide) {
                at_cur[r] = ld_early_u16(reinterpret_cast<const uint16_t*>(codes) + ex[r]);
                at_prev[r] = ld_early_u16(reinterpret_cast<const uint16_t*>(codes) + ex[r] - 1u);
            } else {
                at_cur[r] = ld_early_u8_nc(codes + ex[r]);
                at_prev[r] = ld_early_u8_nc(codes + ex[r] - 1u);
            }
        }
    }
    uint32_t descents = 0;
    int32_t omax = -1;
    if (run) {
        if (wide) chk_run<2>(codes, run, descents, omax, lane);
        else chk_run<1>(codes, run, descents, omax, lane);
    }
    uint32_t at_starts = 0;
#pragma unroll
    for (int r = 0; r < R; ++r)
        if (c[r] != 0u && ex[r] != 0u) at_starts += (at_cur[r] >> 1) <= (at_prev[r] >> 1) ? 1u : 0u;
    // Every offset is below its bin's length: L_T, except in the layer's last bin, whose
    // codes end the task when the task holds that bin; once the offsets rise within it,
    // its last code is its largest.
    bool ok = __reduce_max_sync(kFull, (uint32_t)(omax + 1)) <= (uint32_t)ly.bin_len &&
              __reduce_add_sync(kFull, descents) == __reduce_add_sync(kFull, at_starts);
    if (ok && b0 + nb == ly.nbins && cnt[ly.nbins - 1] != 0u)
        ok = off_at(run - 1u) < (int32_t)(ly.n - (int64_t)(ly.nbins - 1) * ly.bin_len);
    if (!__all_sync(kFull, ok) && lane == 0) ws[16 + l * K + k] = 1;
}

// Persistent over tiles (CTA c takes tiles c, c + grid, ...). The dense tiles
// stream through a ring of kAccStages shared-memory stages: bulk copies (TMA) load a
// tile kAccStages - 1 tiles ahead, and the finished tile goes back with a bulk
// store, so loads, stores and the code scatter overlap.
// A stage holds the tile from the 16-byte boundary at or before its first element;
// the bulk store covers the tile's 16-byte-aligned interior and the threads store
// the (at most three) elements at each end, which neighbouring tiles share a
// 16-byte line with.
// Inside a tile, warp w owns a contiguous range of the tile's bins for every
// learner, so the learners' additions to one element all come from one warp in
// learner order; warps need no barrier between learners. Each warp finds where its
// codes start (the tile's offset in the message plus the counts of the tile's bins
// before its range), and each lane takes a contiguous run of those codes, finds the
// bin of its first code by binary search and walks forward.
constexpr int kAccStages = 2;

// One tile-sized fp32 array: a stage holds the dense tile (plain sum) or the
// gradient sum (a decode fused with an optimiser step, whose weights and state are
// read from and written to global memory directly).
__host__ __device__ inline uint32_t acc_array_bytes(uint32_t tile_cap) { return ((tile_cap + 8) * 4 + 127) & ~127u; }
__host__ __device__ inline uint32_t acc_stage_bytes(uint32_t tile_cap, int opt = kOptNone)
{
    return acc_array_bytes(tile_cap);
}
__host__ __device__ inline uint32_t acc_pre_bytes(uint32_t max_bins)
{
    return (uint32_t)(kDecThreads / 32) * ((max_bins + 8) / 8 + 2) * 4;
}
__host__ __device__ inline uint32_t acc_smem_bytes(uint32_t tile_cap, uint32_t max_bins, int opt = kOptNone)
{
    return kAccStages * acc_stage_bytes(tile_cap, opt) + ((acc_pre_bytes(max_bins) + 127) & ~127u) + 128;
}

struct AccTile {
    int layer;
    uint32_t first_bin;
    int bins;
    int64_t ts, te;  // element range [ts, te) of the layer
    int64_t a0;      // 16-byte boundary at or before ts: element a0 is at stage[0]
};

// Per-CTA copy of what the accumulate kernels look up per tile: each layer's
// first tile, whether it is summed in place, and which (layer, learner) messages
// passed every check.
struct LayerIndex {
    uint32_t tb[kMaxGroup];
    uint8_t sparse[kMaxGroup];
    uint8_t ok[kMaxDecodePairs];
};

__device__ __forceinline__ void load_index(LayerIndex& X, const KGroup& g, uint8_t* ws, int K, bool opt)
{
    for (int e = threadIdx.x; e < g.num_layers; e += blockDim.x) {
        X.tb[e] = g.layer[e].tile_begin;
        X.sparse[e] = !opt && sparse_flags(ws)[e] != 0 ? 1 : 0;
    }
    for (int e = threadIdx.x; e < g.num_layers * K; e += blockDim.x) X.ok[e] = ws[16 + e] == 0 ? 1 : 0;
}

__device__ __forceinline__ AccTile acc_tile(const KGroup& g, const LayerIndex& X, uint32_t t)
{
    AccTile A;
    A.layer = layer_of(X.tb, g.num_layers, t);
    const KLayer& ly = g.layer[A.layer];
    A.first_bin = (t - ly.tile_begin) * ly.bins_per_tile;
    A.bins = (int)min(ly.bins_per_tile, ly.nbins - A.first_bin);
    A.ts = (int64_t)A.first_bin * ly.bin_len;
    A.te = min(A.ts + (int64_t)A.bins * ly.bin_len, ly.n);
    A.a0 = A.ts & ~(int64_t)3;
    return A;
}

// Thread 0, fused optimiser steps: prefetch tile t's weights and optimiser state
// (the 16-byte-aligned interior of the tile) into L2 a tile ahead, so that the
// optimiser step's loads of them hit L2.
template <int kOpt>
__device__ __forceinline__ void opt_prefetch(const KGroup& g, const LayerIndex& X, const DecodeParams& p, uint32_t t)
{
    const AccTile A = acc_tile(g, X, t);
    const int64_t c0 = (A.ts + 3) & ~(int64_t)3, c1 = A.te & ~(int64_t)3;
    if (c1 <= c0) return;
    const uint32_t bytes = (uint32_t)(c1 - c0) * 4u;
    ptx::bulk_prefetch_l2(p.dense[A.layer] + c0, bytes);
    ptx::bulk_prefetch_l2(p.mom[A.layer] + c0, bytes);
    if (kOpt == kOptAdam) ptx::bulk_prefetch_l2(p.mom2[A.layer] + c0, bytes);
}

// Thread 0: start tile t's dense slice into a stage (plain sum only). The copy ends
// at the 16-byte boundary at or after the tile unless that lies past the array, in
// which case the last few elements are loaded with plain loads.
template <int kOpt>
__device__ void acc_issue(const KGroup& g, const LayerIndex& X, const DecodeParams& p, uint32_t t, float* st,
                          uint32_t arr_floats, uint64_t* bar)
{
    const AccTile A = acc_tile(g, X, t);
    const int64_t n = g.layer[A.layer].n;
    if (X.sparse[A.layer]) {  // summed in place by the sparse kernel: nothing to stage
        ptx::mbar_arrive(bar);
        return;
    }
    int64_t a1 = (A.te + 3) & ~(int64_t)3;
    if (a1 > n) a1 = A.te & ~(int64_t)3;
    const uint32_t bytes = a1 > A.a0 ? (uint32_t)(a1 - A.a0) * 4u : 0u;
    const float* src = p.dense[A.layer];
    for (int64_t j = max(a1, A.ts); j < A.te; ++j) st[j - A.a0] = src[j];
    if (a1 < A.te) ptx::fence_proxy_async_smem();
    ptx::mbar_arrive_expect_tx(bar, bytes);
    if (bytes) ptx::bulk_g2s(st, src + A.a0, bytes, bar);
}

__device__ __forceinline__ bool acc_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns)
{
    uint64_t start = 0;
    while (!ptx::mbar_try_wait_sleep(bar, parity, 20000u)) {
        const uint64_t now = ptx::globaltimer();
        if (start == 0) start = now;
        else if (now - start > timeout_ns) return false;
    }
    return true;
}

// Warp `warp` adds learner k's codes for bins [b0, b1) of tile A to the staged
// dense tile sd (element ts + x at sd[x]), in two parts so that the first part can
// run while the dense tile is still loading. acc_prefix: the codes of the tile's
// bins before b0 and the exclusive prefix of the warp's bins in `pre` (b1 - b0 + 1
// entries); returns the warp's code count and sets *before. acc_walk: each lane
// takes a contiguous run of the warp's codes, finds the bin of its first code by
// binary search and walks forward.
__device__ __forceinline__ uint32_t acc_prefix(const AccTile& A, const uint8_t* msg, int b0, int b1, uint32_t* pre,
                                               uint32_t* before_out, int lane)
{
    const uint16_t* cnt = reinterpret_cast<const uint16_t*>(msg + 8) + A.first_bin;
    uint32_t before = 0;
    for (int b = lane; b < b0; b += 32) before += cnt[b];
#pragma unroll
    for (int o = 16; o; o >>= 1) before += __shfl_xor_sync(kFull, before, o);
    uint32_t run = 0;
    for (int c0 = b0; c0 < b1; c0 += 32) {
        const int b = c0 + lane;
        const uint32_t c = b < b1 ? cnt[b] : 0u;
        uint32_t incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += y;
        }
        if (b < b1) pre[b - b0] = run + incl - c;
        run += __shfl_sync(kFull, incl, 31);
    }
    if (lane == 0) pre[b1 - b0] = run;
    __syncwarp();
    *before_out = before;
    return run;
}

// The first kPrefetch codes of each lane's run and the learner's scale, loaded
// before the dense tile has landed (they do not depend on it).
constexpr int kPrefetch = 4;
struct CodePrefetch {
    uint32_t c[kPrefetch];
    float s;
};

__device__ __forceinline__ void acc_fetch(const KLayer& ly, const uint8_t* msg, uint64_t off, uint32_t before,
                                          uint32_t total, int lane, CodePrefetch& P)
{
    P.s = *reinterpret_cast<const float*>(msg);
    const uint32_t per = (total + 31) / 32;
    const uint32_t i0 = min(total, lane * per), iend = min(total, i0 + per);
    const uint8_t* codes = msg + 8 + 2ull * ly.nbins + (unsigned long long)ly.code_bytes * (off + before);
#pragma unroll
    for (int j = 0; j < kPrefetch; ++j) {
        P.c[j] = 0u;
        if (i0 + j < iend)
            P.c[j] = ly.code_bytes == 1 ? codes[i0 + j] : reinterpret_cast<const uint16_t*>(codes)[i0 + j];
    }
}

// Each lane takes a contiguous run of the warp's codes (the first kPrefetch from
// P when use_prefetch), finds the bin of its first code by binary search in the warp's
// bin prefix and walks forward, adding sign * s to sd[bin * L_T + offset].
__device__ __forceinline__ void acc_walk_pf(const KLayer& ly, const AccTile& A, const uint8_t* msg, uint64_t off,
                                            uint32_t before, uint32_t total, int b0, int b1, float* sd,
                                            const uint32_t* pre, int lane, const CodePrefetch& P,
                                            bool use_prefetch)
{
    const float s = use_prefetch ? P.s : *reinterpret_cast<const float*>(msg);
    const uint32_t per = (total + 31) / 32;
    const uint32_t i0 = min(total, lane * per);
    const uint32_t iend = min(total, i0 + per);
    if (i0 < iend) {
        const uint8_t* codes = msg + 8 + 2ull * ly.nbins + (unsigned long long)ly.code_bytes * (off + before);
        const int64_t last_len = ly.n - (int64_t)(ly.nbins - 1) * ly.bin_len;
        int lo = 0, hi = b1 - b0 - 1;  // last bin whose prefix is <= i0
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (pre[mid] <= i0) lo = mid;
            else hi = mid - 1;
        }
        int b = lo;
        uint32_t next = pre[b + 1];
        auto apply = [&](uint32_t i, uint32_t code) {
            while (i >= next) next = pre[++b + 1];
            const uint32_t o = code >> 1;
            const int bin = b0 + b;
            const int64_t len = (A.first_bin + bin == ly.nbins - 1) ? last_len : ly.bin_len;
            if ((int64_t)o < len) {  // always true for a validated message; keeps every write in the tile
                float* x = sd + (int64_t)bin * ly.bin_len + o;
                *x = __fadd_rn(*x, (code & 1u) ? -s : s);
            }
        };
        uint32_t i = i0;
        if (use_prefetch) {
#pragma unroll
            for (int j = 0; j < kPrefetch; ++j)
                if (i0 + j < iend) apply(i0 + j, P.c[j]);
            i = min(iend, i0 + kPrefetch);
        }
        for (; i < iend; ++i)
            apply(i, ly.code_bytes == 1 ? codes[i] : reinterpret_cast<const uint16_t*>(codes)[i]);
    }
    __syncwarp();  // pre is rewritten for the next learner; this learner's additions are done
}

__device__ __forceinline__ void acc_walk(const KLayer& ly, const AccTile& A, const uint8_t* msg, uint64_t off,
                                         uint32_t before, uint32_t total, int b0, int b1, float* sd,
                                         const uint32_t* pre, int lane)
{
    CodePrefetch none;
    acc_walk_pf(ly, A, msg, off, before, total, b0, b1, sd, pre, lane, none, false);
}

// Warp `warp` owns one bin of tile A (tiles of at most 8 bins): every learner's
// codes for that bin, learners kb .. kb + 31 per round. acc_bin_prep: lane k fetches
// learner kb + k's code count in the bin, its first code and its scale (the tile
// offset and the counts of the tile's bins up to this one, every load issued at
// once; none depends on the dense tile, so this runs while that is loading).
// acc_bin_apply: the codes of kAccWindow learners at a time are loaded at once (lane
// i holding code i of each) and added in learner order.
constexpr int kAccWindow = 8;

struct BinPrep {
    const uint8_t* codes;  // the learner's first code for this bin
    uint32_t c;            // its codes in this bin
    float s;               // its scale
};

__device__ __forceinline__ BinPrep acc_bin_prep(const KLayer& ly, const AccTile& A, const DecodeParams& p,
                                                const LayerIndex& X, uint8_t* ws, uint32_t T, uint32_t t, int l,
                                                int bin, int kb, int lane)
{
    BinPrep P;
    P.codes = nullptr;
    P.c = 0;
    P.s = 0.0f;
    const int K = p.K;
    const int k = kb + lane;
    if (k < K && X.ok[l * K + k]) {
        const uint8_t* msg = p.msg[l * K + k];
        const uint16_t* cnt = reinterpret_cast<const uint16_t*>(msg + 8) + A.first_bin;
        uint32_t c[8];
#pragma unroll
        for (int b = 0; b < 8; ++b) c[b] = b <= bin ? cnt[b] : 0u;
        const uint64_t off = tile_offsets(ws, k, T)[t];
        P.s = *reinterpret_cast<const float*>(msg);
        uint32_t before = 0, mine = 0;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            before += b < bin ? c[b] : 0u;
            mine += b == bin ? c[b] : 0u;
        }
        P.c = mine;
        P.codes = msg + 8 + 2ull * ly.nbins + (unsigned long long)ly.code_bytes * (off + before);
    }
    return P;
}

// Per warp, one 16-byte entry per learner of the round: its first code's address,
// its code count in the bin and its scale, read back as warp-wide broadcasts.
struct alignas(16) LearnerBin {
    const uint8_t* codes;
    uint32_t c;
    float s;
};

template <bool kWide>
__device__ __forceinline__ void acc_bin_apply_t(const KLayer& ly, int K, int kb, const BinPrep& P, float* x0,
                                                uint32_t len, LearnerBin* lb, int lane)
{
    const int kn = min(32, K - kb);
    const uint32_t big = __ballot_sync(kFull, P.c > 32u);  // learners with more codes than lanes in the bin
    lb[lane] = LearnerBin{P.codes, P.c, P.s};
    __syncwarp();
    for (int k0 = 0; k0 < kn; k0 += kAccWindow) {
        uint32_t cw[kAccWindow];
        if (kn - k0 >= kAccWindow && ((big >> k0) & ((1u << kAccWindow) - 1u)) == 0u) {
            // a whole window of learners with at most 32 codes each in the bin (warp-uniform)
#pragma unroll
            for (int w = 0; w < kAccWindow; ++w) {
                const LearnerBin e = lb[k0 + w];
                cw[w] = 0xffffffffu;
                if ((uint32_t)lane < e.c)
                    cw[w] = kWide ? (uint32_t)reinterpret_cast<const uint16_t*>(e.codes)[lane] : (uint32_t)e.codes[lane];
            }
#pragma unroll
            for (int w = 0; w < kAccWindow; ++w) {
                const uint32_t sb = __float_as_uint(lb[k0 + w].s);
                const uint32_t o = cw[w] >> 1;
                // sign * s: adding the code's low bit at bit 31 flips the sign bit of s
                if (o < len) x0[o] = __fadd_rn(x0[o], __uint_as_float(sb + (cw[w] << 31)));
                __syncwarp();
            }
            continue;
        }
#pragma unroll
        for (int w = 0; w < kAccWindow; ++w) {
            const int kk = min(k0 + w, kn - 1);
            const uint32_t ck = __shfl_sync(kFull, P.c, kk);
            const uint8_t* cp = reinterpret_cast<const uint8_t*>(__shfl_sync(kFull, (unsigned long long)P.codes, kk));
            cw[w] = 0xffffffffu;
            if (k0 + w < kn && (uint32_t)lane < ck)
                cw[w] = kWide ? (uint32_t)reinterpret_cast<const uint16_t*>(cp)[lane] : (uint32_t)cp[lane];
        }
#pragma unroll
        for (int w = 0; w < kAccWindow; ++w) {
            if (k0 + w >= kn) break;
            const int kk = k0 + w;
            const float s = __shfl_sync(kFull, P.s, kk);
            const uint32_t o = cw[w] >> 1;  // 0x7fffffff for no code: never below a bin length
            // sign * s by flipping the sign bit of s
            if (o < len) x0[o] = __fadd_rn(x0[o], __int_as_float(__float_as_int(s) ^ (int)(cw[w] << 31)));
            if ((big >> kk) & 1u) {  // more codes than lanes in this bin: the rest, in rounds
                const uint32_t ck = __shfl_sync(kFull, P.c, kk);
                const uint8_t* cp =
                    reinterpret_cast<const uint8_t*>(__shfl_sync(kFull, (unsigned long long)P.codes, kk));
                for (uint32_t i = 32 + lane; i < ck; i += 32) {
                    const uint32_t code = kWide ? (uint32_t)reinterpret_cast<const uint16_t*>(cp)[i] : (uint32_t)cp[i];
                    const uint32_t o2 = code >> 1;
                    if (o2 < len) x0[o2] = __fadd_rn(x0[o2], __int_as_float(__float_as_int(s) ^ (int)(code << 31)));
                }
            }
            __syncwarp();  // learner kk's additions come before learner kk + 1's
        }
    }
}

__device__ __forceinline__ void acc_bin_apply(const KLayer& ly, const AccTile& A, int K, int bin, int kb,
                                              const BinPrep& P, float* sd, LearnerBin* lb, int lane)
{
    const uint32_t len = (A.first_bin + bin == ly.nbins - 1)
                             ? (uint32_t)(ly.n - (int64_t)(ly.nbins - 1) * ly.bin_len) : (uint32_t)ly.bin_len;
    float* x0 = sd + (int64_t)bin * ly.bin_len;
    if (ly.code_bytes == 2) acc_bin_apply_t<true>(ly, K, kb, P, x0, len, lb, lane);
    else acc_bin_apply_t<false>(ly, K, kb, P, x0, len, lb, lane);
}

// One optimiser step over tile A's elements, the gradient sum in gs (element ts + x at
// gs[x]): weights and state are read from and written to global memory directly, the
// 16-byte-aligned interior four elements at a time, the (at most three) elements at
// each end one at a time (neighbouring tiles share those 16-byte lines).
template <int kOpt>
__device__ __forceinline__ void opt_elem(const DecodeParams& p, float gsum, float& w, float& m, float& v)
{
    if constexpr (kOpt == kOptSGD) {
        const float mv = __fadd_rn(__fmul_rn(p.mu, m), __fmul_rn(p.scale, gsum));
        m = mv;
        w = __fsub_rn(w, __fmul_rn(p.lr, mv));
    } else {
        const float gx = __fmul_rn(p.scale, gsum);
        const float mm = __fadd_rn(__fmul_rn(p.beta1, m), __fmul_rn(__fsub_rn(1.0f, p.beta1), gx));
        const float vv = __fadd_rn(__fmul_rn(p.beta2, v), __fmul_rn(__fsub_rn(1.0f, p.beta2), __fmul_rn(gx, gx)));
        m = mm;
        v = vv;
        // both moments zero (an element no learner has sent yet) and eps > 0: m/bc1 is
        // mm itself (a signed zero), sqrt(v/bc2) + eps is eps, and so the ratio is mm
        // exactly; the divisions and the square root are skipped
        const float ratio = (mm == 0.0f && vv == 0.0f && p.eps > 0.0f)
                                ? mm
                                : __fdiv_rn(__fdiv_rn(mm, p.bc1), __fadd_rn(__fsqrt_rn(__fdiv_rn(vv, p.bc2)), p.eps));
        w = __fsub_rn(w, __fmul_rn(p.lr, ratio));
    }
}

template <int kOpt>
__device__ __forceinline__ void opt_tile(const DecodeParams& p, const AccTile& A, const float* gs, int tid)
{
    float* W = p.dense[A.layer];
    float* M = p.mom[A.layer];
    float* V = kOpt == kOptAdam ? p.mom2[A.layer] : nullptr;
    const int64_t c0 = (A.ts + 3) & ~(int64_t)3, c1 = A.te & ~(int64_t)3;
    if (c1 > c0) {
        for (int64_t q = c0 / 4 + tid; q < c1 / 4; q += kDecThreads) {
            float4 w4 = reinterpret_cast<const float4*>(W)[q];
            float4 m4 = reinterpret_cast<const float4*>(M)[q];
            float4 v4 = make_float4(0.f, 0.f, 0.f, 0.f);
            if (kOpt == kOptAdam) v4 = reinterpret_cast<const float4*>(V)[q];
            const float* g4 = gs + (4 * q - A.ts);
            opt_elem<kOpt>(p, g4[0], w4.x, m4.x, v4.x);
            opt_elem<kOpt>(p, g4[1], w4.y, m4.y, v4.y);
            opt_elem<kOpt>(p, g4[2], w4.z, m4.z, v4.z);
            opt_elem<kOpt>(p, g4[3], w4.w, m4.w, v4.w);
            reinterpret_cast<float4*>(W)[q] = w4;
            reinterpret_cast<float4*>(M)[q] = m4;
            if (kOpt == kOptAdam) reinterpret_cast<float4*>(V)[q] = v4;
        }
        if (tid < 8) {  // the ends
            const int64_t j = tid < 4 ? A.ts + tid : c1 + (tid - 4);
            if ((tid < 4 && j < c0) || (tid >= 4 && j < A.te)) {
                float w = W[j], m = M[j], v = kOpt == kOptAdam ? V[j] : 0.0f;
                opt_elem<kOpt>(p, gs[j - A.ts], w, m, v);
                W[j] = w;
                M[j] = m;
                if (kOpt == kOptAdam) V[j] = v;
            }
        }
    } else {
        for (int64_t j = A.ts + tid; j < A.te; j += kDecThreads) {
            float w = W[j], m = M[j], v = kOpt == kOptAdam ? V[j] : 0.0f;
            opt_elem<kOpt>(p, gs[j - A.ts], w, m, v);
            W[j] = w;
            M[j] = m;
            if (kOpt == kOptAdam) V[j] = v;
        }
    }
}

// kOpt != kOptNone: the learners' codes are summed into a zeroed gradient tile g in
// shared memory and one optimiser step is applied to the tile's elements (opt_tile):
//   kOptSGD   v = fl32(fl32(mu * v) + fl32(scale * g)), w = fl32(w - fl32(lr * v));
//   kOptAdam  g' = fl32(scale * g), m = fl32(fl32(b1 m) + fl32(fl32(1 - b1) g')),
//             v = fl32(fl32(b2 v) + fl32(fl32(1 - b2) fl32(g' g'))),
//             w = fl32(w - fl32(lr fl32(fl32(m / bc1) / fl32(sqrt(fl32(v / bc2)) + eps))))
//             (correctly rounded division and square root).
// Plain sum: the dense tile is staged (bulk copies in, bulk store out).
template <int kOpt>
__global__ void __launch_bounds__(kDecThreads, 5) accumulate_kernel(const __grid_constant__ KGroup g,
                                                                 const __grid_constant__ DecodeParams p, uint8_t* ws)
{
    ptx::griddep_wait();  // every check
    constexpr bool kFused = kOpt != kOptNone;
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t stage_bytes = acc_stage_bytes(g.tile_cap, kOpt);
    const uint32_t arr_floats = acc_array_bytes(g.tile_cap) / 4;
    float* stage0 = reinterpret_cast<float*>(smem);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int pre_len = (g.max_bins + 8) / 8 + 2;
    uint32_t* pre = reinterpret_cast<uint32_t*>(smem + kAccStages * stage_bytes) + warp * pre_len;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kAccStages * stage_bytes +
                                                ((acc_pre_bytes(g.max_bins) + 127) & ~127u));
    const uint32_t T = g.total_tiles;
    const uint32_t G0 = blockIdx.x, GS = gridDim.x;
    const int K = p.K;
    auto stage = [&](int i) { return stage0 + (size_t)(i % kAccStages) * (stage_bytes / 4); };
    __shared__ LayerIndex X;
    __shared__ LearnerBin lb_s[kDecThreads / 32][32];
    LearnerBin* lbw = lb_s[warp];
    load_index(X, g, ws, p.K, kFused);
    __syncthreads();
    // The CTA's tiles are G0, G0 + GS, ...; tiles of layers summed in place (by the
    // sparse kernel) are jumped over a layer at a time.
    auto next_tile = [&](uint32_t t) -> uint32_t {
        while (t < T) {
            const int l = layer_of(X.tb, g.num_layers, t);
            if (!X.sparse[l]) return t;
            const uint32_t te = l + 1 < g.num_layers ? X.tb[l + 1] : T;
            t += ((te - t + GS - 1) / GS) * GS;  // the CTA's first tile at or after te
        }
        return T;
    };
    // Plain sum: tile window t (processed now) and t1 (copied into the other stage at
    // the start of this iteration, as soon as the bulk store of the tile that stage held
    // has read it, so the copy has the whole iteration to land). (Three stages measured
    // no faster.)
    static_assert(kAccStages == 2, "the ring below holds one tile ahead");
    uint32_t t = next_tile(G0);
    uint32_t t1 = t < T ? next_tile(t + GS) : T;

    if (tid == 0) {
        for (int k = 0; k < kAccStages; ++k) ptx::mbar_init(&bar[k], 1);
        ptx::fence_mbar_init();
        if (!kFused && t < T) acc_issue<kOpt>(g, X, p, t, stage(0), arr_floats, &bar[0]);
        if (kFused && t < T) opt_prefetch<kOpt>(g, X, p, t);
    }
    __syncthreads();

    bool poisoned = false;
    int i = 0;
    for (; t < T; ++i) {
        float* st = stage(i);
        if (!kFused && tid == 0 && t1 < T) {
            ptx::bulk_wait_read0();  // the store of the tile stage i + 1 held has read it
            acc_issue<kOpt>(g, X, p, t1, stage(i + 1), arr_floats, &bar[(i + 1) % kAccStages]);
        }
        if (kFused && tid == 0 && t1 < T) opt_prefetch<kOpt>(g, X, p, t1);
        const AccTile A = acc_tile(g, X, t);
        const KLayer& ly = g.layer[A.layer];
        const int l = A.layer;
        const int bpw = (A.bins + kDecThreads / 32 - 1) / (kDecThreads / 32);
        const int b0 = min(A.bins, warp * bpw), b1 = min(A.bins, b0 + bpw);
        if constexpr (kFused) {  // the gradient sum starts at zero
            float4* z = reinterpret_cast<float4*>(st);
            for (int64_t q = tid; q < (A.te - A.a0 + 3) / 4; q += kDecThreads) z[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // the first learners' offsets and counts do not depend on the dense tile:
        // fetch them while its copy is in flight
        BinPrep bp;
        CodePrefetch cp0;
        uint64_t off0 = 0;
        uint32_t before0 = 0, total0 = 0;
        if (bpw == 1) {
            if (b0 < b1) bp = acc_bin_prep(ly, A, p, X, ws, T, t, l, b0, 0, lane);
        } else if (b0 < b1 && X.ok[l * K]) {
            off0 = tile_offsets(ws, 0, T)[t];
            total0 = acc_prefix(A, p.msg[l * K], b0, b1, pre, &before0, lane);
            acc_fetch(ly, p.msg[l * K], off0, before0, total0, lane, cp0);
        }
        if (kFused) {
            __syncthreads();  // the zeroed gradient tile
        } else if (!__syncthreads_and(acc_wait(&bar[i % kAccStages], (uint32_t)(i / kAccStages) & 1u,
                                               g.timeout_ns))) {
            poisoned = true;
            break;
        }
        float* sd = st + (A.ts - A.a0);  // element ts + x at sd[x]
        if (bpw == 1) {
            if (b0 < b1) {
                for (int kb = 0; kb < K; kb += 32) {
                    if (kb) bp = acc_bin_prep(ly, A, p, X, ws, T, t, l, b0, kb, lane);
                    acc_bin_apply(ly, A, K, b0, kb, bp, sd, lbw, lane);
                }
            }
        } else if (b0 < b1) {
            for (int k = 0; k < K; ++k) {
                if (!X.ok[l * K + k]) continue;  // a rejected message adds nothing
                const uint64_t off = k ? tile_offsets(ws, k, T)[t] : off0;
                const uint8_t* msg = p.msg[l * K + k];
                uint32_t before = before0, total = total0;
                if (k) total = acc_prefix(A, msg, b0, b1, pre, &before, lane);
                acc_walk_pf(ly, A, msg, off, before, total, b0, b1, sd, pre, lane, cp0, k == 0);
            }
        }
        __syncthreads();
        if constexpr (kFused) {
            opt_tile<kOpt>(p, A, sd, tid);
            __syncthreads();  // the gradient tile is zeroed again for the next tile
        } else {
            // write back: ends by the threads, the aligned interior by one bulk store
            const int64_t c0 = (A.ts + 3) & ~(int64_t)3, c1 = A.te & ~(int64_t)3;
            float* dst = p.dense[l];
            if (c1 > c0) {
                if (tid < 8) {
                    const int64_t j = tid < 4 ? A.ts + tid : c1 + (tid - 4);
                    if ((tid < 4 && j < c0) || (tid >= 4 && j < A.te)) dst[j] = st[j - A.a0];
                }
            } else {
                for (int64_t j = A.ts + tid; j < A.te; j += kDecThreads) dst[j] = st[j - A.a0];
            }
            ptx::fence_proxy_async_smem();  // the threads' shared writes, before the bulk store reads them
            __syncthreads();
            if (tid == 0) {
                if (c1 > c0) ptx::bulk_s2g(dst + c0, st + (c0 - A.a0), (uint32_t)(c1 - c0) * 4u);
                ptx::bulk_commit();
            }
        }
        t = t1;
        t1 = t1 < T ? next_tile(t1 + GS) : T;
    }
    if (tid == 0) ptx::bulk_wait0();
    if (poisoned) {
        // a load never completed: flag every message of this CTA's remaining tiles'
        // layers, then give the loads still in flight one more bounded wait before
        // the CTA's shared memory is released
        for (uint32_t u = t; u < T; u += GS) {
            const int l = layer_of(X.tb, g.num_layers, u);
            for (int k = tid; k < K; k += kDecThreads) ws[16 + l * K + k] = 1;
        }
        // the load of the tile whose wait ran out, and that of the next tile
        acc_wait(&bar[i % kAccStages], (uint32_t)(i / kAccStages) & 1u, g.timeout_ns);
        if (t1 < T) acc_wait(&bar[(i + 1) % kAccStages], (uint32_t)((i + 1) / kAccStages) & 1u, g.timeout_ns);
    }
}

// Layers summed in place (plain sum only), no staging: warp u of the grid takes
// tiles u, u + warps, ... of those layers (the other layers are jumped over a layer
// at a time). For each learner in order the warp finds where the tile's codes start
// and the prefix of its bins' counts, then each lane takes a contiguous run of the
// codes and adds sign * s_k to the dense elements in global memory; the warp's
// barrier after each learner keeps learner order for every element.
__global__ void __launch_bounds__(kDecThreads) sparse_accumulate_kernel(const __grid_constant__ KGroup g,
                                                                        const __grid_constant__ DecodeParams p,
                                                                        uint8_t* ws)
{
    ptx::griddep_wait();  // the layers that were streamed are done
    extern __shared__ uint32_t sp_dyn[];  // per warp: the bins' count prefix
    __shared__ LayerIndex X;
    for (int e = threadIdx.x; e < g.num_layers; e += kDecThreads) {
        X.tb[e] = g.layer[e].tile_begin;
        X.sparse[e] = sparse_flags(ws)[e];
    }
    for (int e = threadIdx.x; e < g.num_layers * p.K; e += kDecThreads) X.ok[e] = ws[16 + e] == 0 ? 1 : 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t T = g.total_tiles;
    const uint32_t NW = gridDim.x * (kDecThreads / 32);
    uint32_t* pre = sp_dyn + warp * (g.max_bins + 2);
    const int K = p.K;
    uint32_t t = blockIdx.x * (kDecThreads / 32) + warp;
    for (;;) {
        while (t < T) {  // the warp's next tile of a layer summed in place
            const int l = layer_of(X.tb, g.num_layers, t);
            if (X.sparse[l]) break;
            const uint32_t te = l + 1 < g.num_layers ? X.tb[l + 1] : T;
            t += ((te - t + NW - 1) / NW) * NW;
        }
        if (t >= T) break;
        const AccTile A = acc_tile(g, X, t);
        const int l = A.layer;
        const KLayer& ly = g.layer[l];
        float* sd = p.dense[l] + A.ts;
        for (int k = 0; k < K; ++k) {
            if (!X.ok[l * K + k]) continue;  // a rejected message adds nothing
            const uint64_t off = tile_offsets(ws, k, T)[t];
            const uint8_t* msg = p.msg[l * K + k];
            uint32_t before = 0;
            const uint32_t total = acc_prefix(A, msg, 0, A.bins, pre, &before, lane);
            acc_walk(ly, A, msg, off, before, total, 0, A.bins, sd, pre, lane);
        }
        t += NW;
    }
}

struct DecDeviceInfo {
    int sms = 0;
    uint32_t smem_set[3] = {0, 0, 0};  // per accumulate kernel (plain sum, fused SGD, fused Adam)
    uint32_t sparse_smem_set = 0;
};
DecDeviceInfo g_ddev[64];

}  // namespace

cudaError_t launch_decode(const KGroup& g, const DecodeParams& p, void* ws, cudaStream_t stream)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    DecDeviceInfo& di = g_ddev[dev];
    if (di.sms == 0) {
        e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    uint8_t* w = static_cast<uint8_t*>(ws);
    const uint64_t vtasks = (uint64_t)p.K * p.val_begin[g.num_layers];  // (learner, run) tasks
    const uint64_t wpb = kDecThreads / 32;
    e = launch_after(tile_sums_kernel, dim3((unsigned)((vtasks + wpb - 1) / wpb)), dim3(kDecThreads), 0, stream, g, p, w);
    if (e != cudaSuccess) return e;
    // scan chunks: at least 8192 tiles, at most 64 chunks per message
    uint32_t max_tiles = 0;
    for (int l = 0; l < g.num_layers; ++l) max_tiles = g.layer[l].num_tiles > max_tiles ? g.layer[l].num_tiles : max_tiles;
    uint32_t CH = kScanPer * kScanThreads * 2;
    while ((max_tiles + CH - 1) / CH > 64u) CH += kScanPer * kScanThreads;
    const dim3 sgrid((max_tiles + CH - 1) / CH, (unsigned)(g.num_layers * p.K));
    e = launch_after(tile_scan_kernel, sgrid, dim3(kScanThreads), 0, stream, g, p, w, CH);
    if (e != cudaSuccess) return e;
    const uint64_t ctasks = (uint64_t)p.K * p.chk_begin[g.num_layers];  // (learner, kChkBins bins) tasks
    bool long_only = true;
    for (int l = 0; l < g.num_layers; ++l) long_only = long_only && g.layer[l].bin_len >= kChkLongBin;
    e = launch_after(long_only ? check_kernel<true> : check_kernel<false>, dim3((unsigned)((ctasks + wpb - 1) / wpb)),
                     dim3(kDecThreads), 0, stream, g, p, w);
    if (e != cudaSuccess) return e;
    const int opt = p.opt;
    const uint32_t smem = acc_smem_bytes(g.tile_cap, g.max_bins, opt);
    void (*kern)(KGroup, DecodeParams, uint8_t*) = opt == kOptAdam  ? accumulate_kernel<kOptAdam>
                                                   : opt == kOptSGD ? accumulate_kernel<kOptSGD>
                                                                    : accumulate_kernel<kOptNone>;
    if (smem > di.smem_set[opt]) {
        // opted in whenever it grows: the kernel's static shared memory counts
        // towards the 48 KB available without the opt-in
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        di.smem_set[opt] = smem;
    }
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kDecThreads, smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    const long long cap = (long long)di.sms * occ;
    const uint32_t grid = (uint32_t)((long long)g.total_tiles < cap ? (long long)g.total_tiles : cap);
    e = launch_after(kern, dim3(grid), dim3(kDecThreads), smem, stream, g, p, w);
    if (e != cudaSuccess || opt != kOptNone) return e;
    // the layers summed in place (the kernel skips the others)
    const uint32_t sp_smem = (kDecThreads / 32) * ((uint32_t)g.max_bins + 2) * 4;
    if (sp_smem > di.sparse_smem_set) {
        e = cudaFuncSetAttribute(sparse_accumulate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sp_smem);
        if (e != cudaSuccess) return e;
        di.sparse_smem_set = sp_smem;
    }
    const uint32_t sp_need = (g.total_tiles + kDecThreads / 32 - 1) / (kDecThreads / 32);
    const uint32_t sp_cap = (uint32_t)di.sms * 8;  // persistent: eight CTAs of eight warps per SM
    const uint32_t sp_grid = sp_need < sp_cap ? sp_need : sp_cap;
    return launch_after(sparse_accumulate_kernel, dim3(sp_grid), dim3(kDecThreads), sp_smem, stream, g, p, w);
}

}  // namespace adacomp
