// Internal definitions shared by the AdaComp kernels and the C ABI host code:
// per-layer launch descriptors, workspace layout, tile geometry and inline-PTX
// helpers (mbarrier, bulk async copies, proxy fences) for sm_103a.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <utility>

namespace adacomp {

// ---------------------------------------------------------------- limits
constexpr int kMaxBinLen = 8192;       // bins are processed whole inside one CTA
constexpr int kMaxGroup = 128;         // layers per launch (by-value kernel parameter)
constexpr int kMaxBinsPerTile = 1024;  // per-tile bin arrays in shared memory
constexpr int kTileTarget = 4096;      // elements per tile (whole bins)
constexpr int kThreads = 256;          // compress CTA size
constexpr int kWarps = kThreads / 32;
constexpr int kRounds = 4;             // lane-vectors per chunk: chunk <= 32*VEC*kRounds elements
constexpr int kWarpSliceMax = 509;     // warp-sliced tiles: a warp slice plus its alignment slots fits 512 slots
constexpr int kWarpScratch = 36;       // per-warp g_max / count scratch entries (bins per slice <= 31)
constexpr int kMaxBuffers = 4;         // look-back path: code staging buffers (one look-back warp each);
                                       // 3 are used (tiles of up to 8192 elements)
constexpr int kHistLo = 64;            // per-warp exponent buckets cover biased exponents [64, 192);
constexpr int kHistN = 128;            // maxima outside go straight to the layer's accumulator
constexpr uint32_t kHistBytesPerBuffer = kHistN * 8;  // one set per look-back warp
constexpr uint32_t kWarpScratchBytes = kWarps * 2 * kWarpScratch * 4;

// ---------------------------------------------------------------- descriptors
// One layer of a launch. Tiles of all layers are numbered consecutively in layer
// order; tile t of layer l covers bins [ (t - tile_begin) * bins_per_tile, ... ).
struct KLayer {
    float* residue;          // fp32[n], in/out
    const void* dw;          // fp32[n] or bf16[n]
    uint8_t* msg;            // message buffer
    int64_t n;               // elements
    uint32_t nbins;          // B = ceil(n / bin_len)
    int32_t bin_len;         // L_T
    uint32_t tile_begin;     // first global tile index of the layer
    uint32_t num_tiles;
    uint32_t bins_per_tile;
    uint8_t dw_bf16;
    uint8_t code_bytes;      // 1 if L_T < 64 else 2
    uint8_t vec;             // 4, 2 or 1: largest of these dividing L_T
    uint8_t bpw;             // warp-sliced tiles: bins per warp slice, floor(509 / L_T); 0: block-wide tiles
    uint32_t inv_len;        // ceil(2^32 / L_T): x / L_T == umulhi(x, inv_len) for x < 2^16
};
static_assert(sizeof(KLayer) == 64, "KLayer layout");

struct KGroup {
    KLayer layer[kMaxGroup];
    int32_t num_layers;
    uint32_t total_tiles;
    uint32_t tile_cap;       // max tile elements over the group (shared memory sizing)
    uint16_t max_bins;       // max bins per tile over the group
    uint16_t d_size;         // 4 if any layer has fp32 dW, else 2
    uint64_t timeout_ns;
    uint32_t inject_skip_tile;  // fault injection for tests: this tile never publishes (~0u: none)
    uint32_t needs_gbuf;        // some layer has bins shorter than 16 (G staged in shared memory)
    uint32_t lazy;              // deferred fix-up for warp-sliced layers (pending masks in the workspace)
    uint32_t local_selection;   // selection rule: 0 AdaComp (abs(G + dW) >= g_max), 1 Local Selection (abs(G) >= g_max)
    uint32_t big;               // every layer has kBigMinLen <= L_T <= kBigMaxLen: the block-sliced path
};

// Block-sliced path: bins longer than a warp slice. A tile (whole bins, at most
// max(kTileTarget, L_T) elements) is cut into kBigSlices slices of 512 slots from the
// 16-byte boundary at or before its first element; the bins that fit (at most 8).
constexpr int kBigMinLen = 510;
constexpr int kBigMaxLen = 8189;  // a one-bin tile plus its alignment slots fits 16 slices
constexpr int kBigSlices = 16;
constexpr int kBigMaxBins = 8;
__host__ __device__ inline bool is_big_len(int32_t L) { return L >= kBigMinLen && L <= kBigMaxLen; }

// Dynamic shared memory of the compress kernel (bytes), laid out in this order:
// 2 stages x {residue slice, dW slice}, layer table, G buffer, nbuf code staging buffers, g_max, counts,
// exponent buckets per look-back warp, per-warp bin scratch, per-stage tile geometry, control block (mbarriers,
// counters, hand-off slots).
struct SmemPlan {
    uint32_t r_bytes, d_bytes, layer_bytes, g_bytes, stg_bytes, bin_stride, bin_bytes, total;
};
__host__ __device__ inline SmemPlan smem_plan(uint32_t tile_cap, uint32_t d_size, uint32_t max_bins,
                                              uint32_t num_layers, uint32_t needs_gbuf, uint32_t nbuf)
{
    SmemPlan p;
    // slack past the tile: the phase slots (< 4 fp32, < 8 bf16) plus segments that
    // run up to 15 slots beyond the last element
    p.r_bytes = ((tile_cap + 32) * 4 + 127) & ~127u;
    p.d_bytes = ((tile_cap + 48) * d_size + 127) & ~127u;
    p.stg_bytes = (tile_cap * 2 + 127) & ~127u;
    p.bin_stride = max_bins + 1;                                     // entries per buffer
    p.bin_bytes = (nbuf * p.bin_stride * 4 + 127) & ~127u;           // all buffers
    p.layer_bytes = num_layers * 64u;                        // copy of the layer table
    p.g_bytes = needs_gbuf ? p.r_bytes : 0u;
    p.total = 2 * (p.r_bytes + p.d_bytes) + p.layer_bytes + p.g_bytes + nbuf * p.stg_bytes + 2 * p.bin_bytes +
              nbuf * kHistBytesPerBuffer + kWarpScratchBytes + 2048 + 1152;
    return p;
}

// ---------------------------------------------------------------- compress workspace
// [Ctl 64 B][LayerWs x num_layers][desc u64 x T][tile_excl u64 x T][lazy only: pending u16 x 256 x T]
// Each layer's accumulators are zero between calls (the finalise kernel clears
// them); the look-back descriptors carry the call's epoch instead of being cleared.
struct Ctl {
    uint32_t epoch;      // epoch of the last completed call (0: none); a call uses epoch % 255 + 1
    uint32_t fin_done;   // finalise blocks done with this call (the last one advances epoch)
    uint32_t pending;    // sliced path: the sent masks hold corrections a deferred fix-up left to the next call
    uint32_t reserved[13];
};

struct Result {              // written by each call, kept for adacomp_query
    float s;
    uint32_t status;
    uint64_t nnz;
    uint64_t msg_bytes;
    uint64_t pad;
};

struct LayerWs {
    unsigned long long acc[256];  // exact sum of g_max: integer mantissas per fp32 exponent
    uint32_t done;                // tiles finished; the last one finalises the layer
    uint32_t err;                 // device-side error bits of this call
    uint32_t pad[2];
    Result result;
    uint32_t pad2[4];
};
static_assert(sizeof(LayerWs) % 64 == 0, "LayerWs alignment");

__host__ __device__ inline size_t ws_layer_offset(int l) { return sizeof(Ctl) + (size_t)l * sizeof(LayerWs); }
__host__ __device__ inline size_t ws_desc_offset(int num_layers) { return sizeof(Ctl) + (size_t)num_layers * sizeof(LayerWs); }
// Deferred (lazy) fix-up: one 16-bit mask per compute lane and tile, bit 4k + i
// for the lane's register slot (k, i) of a warp-sliced tile, set when that element
// was sent and its residue still holds G.
constexpr size_t kPendBytesPerTile = kWarps * 32 * 2;
__host__ __device__ inline size_t ws_pend_offset(int num_layers, uint64_t total_tiles)
{
    return ws_desc_offset(num_layers) + 16 * (size_t)total_tiles;
}
__host__ __device__ inline size_t compress_ws_bytes(int num_layers, uint64_t total_tiles, bool lazy = false)
{
    return ws_pend_offset(num_layers, total_tiles) + (lazy ? kPendBytesPerTile * (size_t)total_tiles : 0);
}

// Compress workspace of a launch group whose layers are all warp-sliced (the
// sliced path: 16 <= L_T <= 509, no look-back):
// [Ctl][LayerWs x num_layers][tile code offset u64 x T, padded to 16 B]
// [tile code total u32 x T, padded to 16 B][sent mask u16 x 256 x T][sign mask u16 x 256 x T].
// A mask word belongs to compute lane (warp w, lane) of a tile: bit i is slot i of
// the lane's 16 consecutive slots. The tile totals are zero between calls; the
// other arrays are written by each call before they are read. The mask arrays start
// on 16-byte boundaries (the emitting kernel loads them 16 bytes at a time).
// (The block-sliced path uses the same layout with kBigSlices slices per tile.)
constexpr size_t kMaskBytesPerTile = kWarps * 32 * 2;
__host__ __device__ inline size_t mask_bytes_per_tile(bool big) { return (size_t)(big ? kBigSlices : kWarps) * 32 * 2; }
__host__ __device__ inline size_t pad16(size_t b) { return (b + 15) & ~(size_t)15; }
__host__ __device__ inline size_t sl_excl_offset(int num_layers) { return ws_desc_offset(num_layers); }
__host__ __device__ inline size_t sl_tot_offset(int num_layers, uint64_t T) { return sl_excl_offset(num_layers) + pad16(8 * (size_t)T); }
__host__ __device__ inline size_t sl_sent_offset(int num_layers, uint64_t T) { return sl_tot_offset(num_layers, T) + pad16(4 * (size_t)T); }
__host__ __device__ inline size_t sl_sign_offset(int num_layers, uint64_t T, bool big = false)
{
    return sl_sent_offset(num_layers, T) + mask_bytes_per_tile(big) * (size_t)T;
}
__host__ __device__ inline size_t sliced_ws_bytes(int num_layers, uint64_t T, bool big = false)
{
    return sl_sign_offset(num_layers, T, big) + mask_bytes_per_tile(big) * (size_t)T;
}
// Bytes at the start of a workspace that must be zero before its first call.
__host__ __device__ inline size_t ws_zero_prefix(int num_layers, uint64_t T, bool sliced)
{
    return sliced ? sl_sent_offset(num_layers, T) : ws_desc_offset(num_layers) + 8 * (size_t)T;
}

// Look-back descriptor: flag in bits 62..63, the call's epoch in bits 54..61, value
// in bits 0..53. A descriptor written by an earlier call (another epoch) reads as
// not yet published, so descriptors need no clearing between calls.
constexpr uint64_t kFlagAgg = 1ull << 62;
constexpr uint64_t kFlagIncl = 2ull << 62;
constexpr uint64_t kFlagErr = 3ull << 62;
constexpr int kEpochShift = 54;
constexpr uint64_t kEpochMask = 0xffull << kEpochShift;
constexpr uint64_t kValueMask = (1ull << kEpochShift) - 1;
// The call's epoch (1..255) from the one stored in the workspace, in descriptor position.
__host__ __device__ inline uint64_t call_epoch(uint32_t last) { return (uint64_t)(last % 255u + 1u) << kEpochShift; }
// Flag of descriptor d in the call with epoch bits ep (0: not published in this call).
__host__ __device__ inline uint32_t desc_flag(uint64_t d, uint64_t ep)
{
    return (d & kEpochMask) == ep ? (uint32_t)(d >> 62) : 0u;
}

// ---------------------------------------------------------------- decode workspace
// [fixed 10240 B: u32 K, u32 num_layers, u32 pad[2], u8 bad[num_layers * K] (up to byte 1040);
//  at byte 2048: u64 codes[num_layers * K], the code count of each (layer, learner) message]
// [per learner k: tile_off u64 x T]
// bad[l*K+k] and tile_off are written by every decode call before they are read, so
// the decode workspace needs no initialisation. tile_off = kBadOffset marks a
// (layer, learner) message that is skipped.
constexpr size_t kDecodeFixed = 10240;
constexpr size_t kDecodeLayerCodes = 2048;  // offset of the (layer, learner) code counts
constexpr int kMaxDecodePairs = 1024;  // num_layers * K per launch
constexpr uint64_t kBadOffset = ~0ull;
// Per learner: the tiles' code offsets (u64) and, before the scan turns them into
// offsets, the tiles' code sums (u32, 0xffffffff for a tile whose counts are invalid).
__host__ __device__ inline size_t decode_sums_offset(uint64_t total_tiles) { return 8 * (size_t)total_tiles; }
__host__ __device__ inline size_t decode_per_learner(uint64_t total_tiles)
{
    return 8 * (size_t)total_tiles + ((4 * (size_t)total_tiles + 15) & ~(size_t)15);
}
// Code validation: one task per run of whole tiles of one layer holding at most
// kValBins bins (one tile when a tile holds more).
constexpr uint32_t kValBins = 128;
__host__ __device__ inline uint32_t val_tiles_per_task(uint32_t bins_per_tile)
{
    return bins_per_tile >= kValBins ? 1u : kValBins / bins_per_tile;
}

// Code checks: bins of kChkLongBin elements or more take one task per tile, the lanes
// over each bin's codes; shorter bins one task per kChkBins bins, the lanes over the
// task's contiguous run of codes: floor(kChkBins / bpt) whole tiles per task, or, for
// tiles of more than kChkBins bins, ceil(bpt / kChkBins) tasks per tile.
constexpr uint32_t kChkBins = 128;
constexpr int32_t kChkLongBin = 1024;
__host__ __device__ inline uint32_t chk_tasks(uint32_t num_tiles, uint32_t bins_per_tile, int32_t bin_len)
{
    if (bin_len >= kChkLongBin) return num_tiles;
    if (bins_per_tile <= kChkBins) {
        const uint32_t tpt = kChkBins / bins_per_tile;
        return (num_tiles + tpt - 1) / tpt;
    }
    return num_tiles * ((bins_per_tile + kChkBins - 1) / kChkBins);
}

constexpr uint32_t kErrTimeout = 1;

// Optimiser step fused with the decode (DecodeParams::opt).
constexpr int kOptNone = 0;  // plain sum into dense
constexpr int kOptSGD = 1;   // momentum SGD on weights (dense) and momentum (mom)
constexpr int kOptAdam = 2;  // Adam on weights (dense), first moment (mom) and second moment (mom2)

struct DecodeParams {
    const uint8_t* msg[kMaxDecodePairs];  // [layer * K + k]
    uint64_t len[kMaxDecodePairs];        // the messages' lengths in bytes, same order
    float* dense[kMaxGroup];              // the dense sum, or the weights when opt != kOptNone
    float* mom[kMaxGroup];                // momentum (SGD) or first moment (Adam)
    float* mom2[kMaxGroup];               // second moment (Adam)
    uint32_t val_begin[kMaxGroup + 1];    // counting tasks per learner: layer l's are [val_begin[l], val_begin[l + 1])
    uint32_t chk_begin[kMaxGroup + 1];    // code-check tasks per learner, the same way
    int32_t K;
    int32_t opt;                          // kOptNone, kOptSGD or kOptAdam
    float lr, mu, scale;                  // SGD: w -= lr * v, v = mu * v + scale * g (Adam uses lr and scale)
    float beta1, beta2, eps, bc1, bc2;    // Adam: decay rates, epsilon, the step's bias corrections
};

// ---------------------------------------------------------------- host-side launchers
// Launches a kernel that begins with ptx::griddep_wait() behind the previous kernel of
// the stream with programmatic dependent launch: its blocks may be scheduled while
// that kernel's last blocks run, and wait there until its writes are visible.
template <typename... KArgs, typename... Args>
cudaError_t launch_after(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                         Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

cudaError_t launch_compress(const KGroup& g, void* ws, cudaStream_t stream, cudaEvent_t ev_before = nullptr,
                            cudaEvent_t ev_mid = nullptr, cudaEvent_t ev_after = nullptr);
cudaError_t launch_decode(const KGroup& g, const DecodeParams& p, void* ws, cudaStream_t stream);
cudaError_t launch_materialize(const KGroup& g, void* ws, cudaStream_t stream);
// The sliced path (every layer of the group warp-sliced).
bool group_is_sliced(const KGroup& g);
cudaError_t launch_compress_sliced(const KGroup& g, void* ws, cudaStream_t stream, cudaEvent_t ev_before,
                                   cudaEvent_t ev_mid, cudaEvent_t ev_after);
cudaError_t launch_materialize_sliced(const KGroup& g, void* ws, cudaStream_t stream);
}  // namespace adacomp

struct adacomp_layer;
namespace adacomp {
int prepare_single_compress(const adacomp_layer* h, float* residue, const void* dW, void* msg,
                            size_t msg_capacity, KGroup* g, size_t* ws_needed);
size_t compress_ws_of(const adacomp_layer* h);

}  // namespace adacomp

// ---------------------------------------------------------------- device helpers
#ifdef __CUDACC__
namespace adacomp {
namespace ptx {

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes mbarrier initialisation visible to the async proxy (bulk copies).
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// Returns true once the phase with the given parity has completed.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Same, but the thread may be suspended (without issuing) for up to hint_ns while
// the phase is incomplete; it resumes as soon as the phase completes.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Global -> shared bulk copy (non-tensor TMA), completion counted on an mbarrier.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Shared -> global bulk copy, tracked by the issuing thread's bulk group.
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_addr(src)),
                 "r"(bytes)
                 : "memory");
}

// Brings [src, src + bytes) into L2 (a bulk prefetch: no shared memory, no
// completion to wait for). src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Waits until every committed bulk store has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Waits until every committed bulk store has completed.
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Orders this thread's generic-proxy shared-memory writes before later async-proxy reads.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint64_t ld_relaxed(const uint64_t* p)
{
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed(uint64_t* p, uint64_t v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Programmatic dependent launch: a kernel launched with the programmatic stream
// serialisation attribute may start before the kernel ahead of it in the stream has
// finished; griddep_wait blocks until that kernel has completed and its writes are
// visible, and griddep_launch lets the next such kernel start early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" :::); }

}  // namespace ptx
}  // namespace adacomp
#endif
