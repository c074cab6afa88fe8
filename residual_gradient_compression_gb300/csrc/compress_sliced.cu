// AdaComp compression for launch groups whose layers all have 16 <= L_T <= 509
// (every conv and FC/LSTM layer of the usual configurations): the warp-sliced path;
// and for groups whose layers all have 510 <= L_T <= 8189: the block-sliced path
// (block_kernel below), which shares the finalise, emitting and codes kernels.
//
// Method: "AdaComp (Adaptive Residual Gradient Compression)", Claims > Mechanism
// #r629-local-bin-soft-threshold-and-mean-gmax-quantization (Algorithm 2 restated):
// G = residue + dW, H = G + dW, g_max(i) = max |G| over bin i, s = mean g_max, send
// |H| >= g_max(i) as sign(G) * s, residue = G - G_q (sent) or G (kept). Code widths:
// Claims > Application #r629-conv-40x-and-fc-lstm-200x-compression-across-optimizers.
//
// Three launches, none of which waits on another CTA:
//   slice_kernel     streams residue and dW once. A tile is eight warp slices of
//                    floor(509 / L_T) whole bins; every warp runs its own pipeline of
//                    bulk copies (cp.async.bulk into per-warp shared-memory stages,
//                    completion on per-warp mbarriers). Per slice: G, residue := G,
//                    bin maxima (exact, into exponent buckets), the selection masks
//                    (which do not depend on s), the per-bin counts, written straight
//                    into the message, and the tile's code total. The codes' positions
//                    are not needed yet, so no CTA ever waits for another.
//   slice_finalize   one CTA per (layer, chunk of 1024 tiles): the exclusive prefix of
//                    the tile code totals; the layer's last chunk also forms s from
//                    the exact sum and writes the header.
//   slice_emit       persistent warps, a run of tiles each, last tiles first: the codes
//                    written at their final positions, with the sign of G read back
//                    from the residue, and the fix-up residue = fl32(G - sign(G) s) of
//                    every sent element. When the fix-up is deferred to the next call,
//                    slice_codes takes its place: the signs come from a second mask
//                    and the residue is not touched.
// Only the sent mask (1 bit per element; 2 with the deferred fix-up) passes between
// the first and the last launch.
#include "adacomp_internal.cuh"
#include "compress_common.cuh"

#include <cuda_bf16.h>

namespace adacomp {
namespace {

constexpr int kSlots = 512;              // slots of a warp slice: 16 per lane
constexpr int kBkLo = 96, kBkN = 64;     // per-warp exponent buckets: biased exponents [96, 160)
constexpr int kBkSlices = 8;             // slices between flushes: 8 x 31 maxima below 2^24 fit 32 bits
constexpr uint32_t kRBytes = kSlots * 4;  // residue stage
constexpr uint32_t kDBytes32 = kSlots * 4;
constexpr uint32_t kDBytes16 = 1152;      // bf16 dW stage: up to 520 elements from the 16-byte boundary before slot 0

struct SlicePlan {
    uint32_t d_bytes, stage_bytes, stages_bytes, layer_bytes, total;
};
__host__ __device__ inline SlicePlan slice_plan(uint32_t d_size, int stages, int num_layers)
{
    SlicePlan p;
    p.d_bytes = d_size == 4 ? kDBytes32 : kDBytes16;
    p.stage_bytes = kRBytes + p.d_bytes;
    p.stages_bytes = kWarps * stages * p.stage_bytes;
    p.layer_bytes = (uint32_t)num_layers * 64u;
    p.total = p.stages_bytes + p.layer_bytes + kWarpScratchBytes + kWarps * kBkN * 4 + kWarps * stages * 8;
    return p;
}

// One warp slice: bins [wb0, wb0 + nb) of tile t, elements [we0, we1) of the tile.
struct Slice {
    int layer;
    int64_t ts;          // first element of the tile (index in its layer)
    uint32_t first_bin;  // first bin of the tile
    int wb0, nb;         // first bin of the slice (tile-relative) and its bin count
    int we0, we1;        // slice elements, tile-relative
    int64_t a0;          // layer element held by slot 0 of lane 0: the 16-byte boundary at or before ts + we0
};

// Slice w of tile t of layer `layer` (whose descriptor is ly).
__device__ __forceinline__ Slice slice_in(const KLayer& ly, int layer, uint32_t t, int w)
{
    Slice S;
    S.layer = layer;
    S.first_bin = (t - ly.tile_begin) * ly.bins_per_tile;
    const int bins = (int)min(ly.bins_per_tile, ly.nbins - S.first_bin);
    S.ts = (int64_t)S.first_bin * ly.bin_len;
    const int tl = (int)min((int64_t)bins * ly.bin_len, ly.n - S.ts);
    S.wb0 = min(bins, w * (int)ly.bpw);
    const int wb1 = min(bins, S.wb0 + (int)ly.bpw);
    S.nb = wb1 - S.wb0;
    S.we0 = S.wb0 * ly.bin_len;
    S.we1 = min(wb1 * ly.bin_len, tl);
    S.a0 = (S.ts + S.we0) & ~(int64_t)3;
    return S;
}

// Layer of tile t >= the first tile of layer l (tiles of a warp only move forward).
__device__ __forceinline__ int advance_layer(const KLayer* lays, int num_layers, uint32_t t, int l)
{
    while (l + 1 < num_layers && lays[l + 1].tile_begin <= t) ++l;
    return l;
}

// Layer of tile t from a shared-memory array of the layers' first tiles.
__device__ __forceinline__ int layer_of_tile(const uint32_t* tb, int num_layers, uint32_t t)
{
    int lo = 0, hi = num_layers - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tb[mid] <= t) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Starts layer elements [e0, e1) into a stage (run by one lane), slot 0 of the
// stage holding layer element a0 (a0 <= e0, a multiple of 4, e1 - a0 <= 512): bulk
// copies of the 16-byte-aligned spans covering the range, from a0 to the boundary
// at or after e1; only at the end of the layer's arrays are the last few elements
// loaded with plain loads. Returns false when nothing was copied (an empty range:
// the phase completes at once).
__device__ bool issue_range(const KLayer& ly, int64_t e0, int64_t e1, int64_t a0, float* rb, void* db, uint64_t* bar)
{
    if (e1 <= e0) {
        ptx::mbar_arrive(bar);
        return false;
    }
    int64_t a1 = (e1 + 3) & ~(int64_t)3;
    if (a1 > ly.n) a1 = e1 & ~(int64_t)3;
    const uint32_t rbytes = (uint32_t)(a1 - a0) * 4u;
    int64_t b0 = a0, b1 = a1;
    uint32_t dbytes = rbytes;
    if (ly.dw_bf16) {
        b0 = e0 & ~(int64_t)7;
        b1 = (e1 + 7) & ~(int64_t)7;
        if (b1 > ly.n) b1 = e1 & ~(int64_t)7;
        dbytes = (uint32_t)(b1 - b0) * 2u;
    }
    if (a1 < e1 || b1 < e1) {
        for (int64_t j = max(a1, e0); j < e1; ++j) rb[j - a0] = ly.residue[j];
        if (ly.dw_bf16) {
            for (int64_t j = max(b1, e0); j < e1; ++j)
                static_cast<uint16_t*>(db)[j - b0] = static_cast<const uint16_t*>(ly.dw)[j];
        } else {
            for (int64_t j = max(b1, e0); j < e1; ++j) static_cast<float*>(db)[j - a0] = static_cast<const float*>(ly.dw)[j];
        }
        ptx::fence_proxy_async_smem();  // before later bulk copies refill these bytes
    }
    ptx::mbar_arrive_expect_tx(bar, rbytes + dbytes);
    if (rbytes) ptx::bulk_g2s(rb, ly.residue + a0, rbytes, bar);
    if (dbytes) ptx::bulk_g2s(db, static_cast<const uint8_t*>(ly.dw) + b0 * (ly.dw_bf16 ? 2 : 4), dbytes, bar);
    return true;
}

// A warp slice's data (at most 509 elements from a 16-byte boundary).
__device__ __forceinline__ bool issue_slice(const KLayer& ly, const Slice& S, float* rb, void* db, uint64_t* bar)
{
    return issue_range(ly, S.ts + S.we0, S.ts + S.we1, S.a0, rb, db, bar);
}

// Bounded wait on an mbarrier phase, the thread sleeping in the barrier between
// checks of the time limit.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, uint64_t timeout_ns)
{
    uint64_t start = 0;
    while (!ptx::mbar_try_wait_sleep(bar, parity, 20000u)) {
        const uint64_t now = ptx::globaltimer();
        if (start == 0) start = now;
        else if (now - start > timeout_ns) return false;
    }
    return true;
}

// Adds a warp's 32-bit exponent buckets to layer lw's exact accumulator and clears them.
__device__ __forceinline__ void flush_hist(uint32_t* hist, LayerWs* lw, int lane)
{
    __syncwarp();
#pragma unroll
    for (int e = lane; e < kBkN; e += 32) {
        const uint32_t v = hist[e];
        if (v) {
            atomicAdd(&lw->acc[kBkLo + e], (unsigned long long)v);
            hist[e] = 0u;
        }
    }
    __syncwarp();
}

// Geometry of one lane's 16 slots within its slice (shared by the streaming and
// the emitting kernels): slot i holds tile element lane_e + i.
struct LaneGeo {
    int lane_e;        // tile element of slot 0
    uint32_t valid;    // slots holding elements of the slice (slot order)
    int bin_lo;        // slice-relative bin of the first valid slot
    int split;         // first slot of bin_lo + 1
};
__device__ __forceinline__ LaneGeo lane_geo(const Slice& S, const KLayer& ly, int lane)
{
    LaneGeo q;
    q.lane_e = (int)(S.a0 - S.ts) + kSeg * lane;
    const bool active = S.we1 > S.we0 && q.lane_e + kSeg > S.we0 && q.lane_e < S.we1;
    const int vlo = max(0, S.we0 - q.lane_e), vhi = min(kSeg, S.we1 - q.lane_e);
    q.valid = (active && vhi > vlo) ? (((1u << (vhi - vlo)) - 1u) << vlo) : 0u;
    const int rel0 = max(q.lane_e, S.we0) - S.we0;  // < 512, so umulhi divides exactly
    q.bin_lo = q.valid ? (int)__umulhi((uint32_t)rel0, ly.inv_len) : 0;
    q.split = (q.bin_lo + 1) * ly.bin_len - (q.lane_e - S.we0);
    return q;
}

// ---------------------------------------------------------------- block-sliced tiles
// Tiles of bins longer than a warp slice (kBigMinLen <= L_T <= kBigMaxLen) keep their
// whole bins (floor(4096 / L_T), at least one) and are cut into kBigSlices slices of
// 512 slots, slice w starting at slot 512 w from the 16-byte boundary at or before the
// tile's first element. A 512-slot slice meets at most three bins of 510 or more.
// In the returned Slice, wb0 is the tile-relative bin of the slice's first element and
// nb the tile's bin count; an empty slice (past the tile's end) has we0 == we1.
__device__ __forceinline__ Slice big_slice(const KLayer& ly, int layer, uint32_t t, int w)
{
    Slice S;
    S.layer = layer;
    S.first_bin = (t - ly.tile_begin) * ly.bins_per_tile;
    S.nb = (int)min(ly.bins_per_tile, ly.nbins - S.first_bin);
    S.ts = (int64_t)S.first_bin * ly.bin_len;
    const int tl = (int)min((int64_t)S.nb * ly.bin_len, ly.n - S.ts);
    S.a0 = (S.ts & ~(int64_t)3) + (int64_t)kSlots * w;
    const int rel = (int)(S.a0 - S.ts);  // tile element of slot 0: -3 .. 0 for slice 0
    S.we0 = max(0, rel);
    S.we1 = max(S.we0, min(tl, rel + kSlots));
    S.wb0 = (int)__umulhi((uint32_t)S.we0, ly.inv_len);  // tile elements are below 2^13: exact
    return S;
}

// Slices of a block-sliced tile that hold elements.
__device__ __forceinline__ int big_slices_used(const KLayer& ly, uint32_t t)
{
    const uint32_t fb = (t - ly.tile_begin) * ly.bins_per_tile;
    const int nb = (int)min(ly.bins_per_tile, ly.nbins - fb);
    const int64_t ts = (int64_t)fb * ly.bin_len;
    const int tl = (int)min((int64_t)nb * ly.bin_len, ly.n - ts);
    return ((int)(ts & 3) + tl + kSlots - 1) / kSlots;
}

// A lane's 16 slots in a block-sliced slice; bin_lo is tile-relative here.
__device__ __forceinline__ LaneGeo big_lane_geo(const Slice& S, const KLayer& ly, int lane)
{
    LaneGeo q;
    q.lane_e = (int)(S.a0 - S.ts) + kSeg * lane;
    const int vlo = max(0, S.we0 - q.lane_e), vhi = min(kSeg, S.we1 - q.lane_e);
    q.valid = vhi > vlo ? (((1u << (vhi - vlo)) - 1u) << vlo) : 0u;
    q.bin_lo = q.valid ? (int)__umulhi((uint32_t)max(q.lane_e, S.we0), ly.inv_len) : 0;
    q.split = (q.bin_lo + 1) * ly.bin_len - q.lane_e;
    return q;
}

// Slot-order mask <-> register order: register chunk k holds slot chunk k ^ rot.
__device__ __forceinline__ uint32_t to_reg_order(uint32_t m, int rot)
{
    uint32_t r = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) r |= ((m >> (4 * (k ^ rot))) & 0xfu) << (4 * k);
    return r;
}
__device__ __forceinline__ uint32_t to_slot_order(uint32_t r, int rot)
{
    uint32_t m = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) m |= ((r >> (4 * k)) & 0xfu) << (4 * (k ^ rot));
    return m;
}

// One lane's 16 slots of a slice whose data is in a stage (rs: residue, ds: dW;
// slot 0 of lane 0 holds layer element S.a0), the four 16-byte chunks visited in the
// bank-conflict-free rotated order: G = fl32(residue + dW) (after the deferred
// correction fl32(G - copysign(s_prev, G)) of the slots set in pm), |probe| into ah
// (-1 where G == 0, so that such elements are never sent), the mask of G < 0 (kLazy
// only), residue := G for the valid slots (vr) with 128-bit stores, and the maxima
// of |G| over the valid slots of the lane's two bins (lor, hir). Registers are in
// register order: chunk k is slot chunk k ^ rot.
template <bool kLazy, bool kLS>
__device__ __forceinline__ void lane_slots(const KLayer& ly, const Slice& Sl, const float* rs0, const void* ds, int lane,
                                           int rot, uint32_t pm, float s_prev, uint32_t vr, uint32_t lor, uint32_t hir,
                                           float (&ah)[4][4], uint32_t& ngr, float& m_lo, float& m_hi)
{
    const float* rs = rs0 + kSeg * lane;
    const int doff = ly.dw_bf16 ? (int)(Sl.a0 - ((Sl.ts + Sl.we0) & ~(int64_t)7)) : 0;
    float* gres = ly.residue + Sl.a0 + kSeg * lane;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int q0 = 4 * (k ^ rot);
        float4 r = *reinterpret_cast<const float4*>(rs + q0);
        if (kLazy && (pm & (0xfu << (4 * k)))) {
            if (pm & (1u << (4 * k + 0))) r.x = __fsub_rn(r.x, copysignf(s_prev, r.x));
            if (pm & (1u << (4 * k + 1))) r.y = __fsub_rn(r.y, copysignf(s_prev, r.y));
            if (pm & (1u << (4 * k + 2))) r.z = __fsub_rn(r.z, copysignf(s_prev, r.z));
            if (pm & (1u << (4 * k + 3))) r.w = __fsub_rn(r.w, copysignf(s_prev, r.w));
        }
        float d[4], gv[4];
        if (ly.dw_bf16) {
            const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(ds) + doff + kSeg * lane + q0);
            d[0] = bf16_lo(u.x); d[1] = bf16_hi(u.x); d[2] = bf16_lo(u.y); d[3] = bf16_hi(u.y);
        } else {
            const float4 v = *reinterpret_cast<const float4*>(static_cast<const float*>(ds) + kSeg * lane + q0);
            d[0] = v.x; d[1] = v.y; d[2] = v.z; d[3] = v.w;
        }
        gv[0] = __fadd_rn(r.x, d[0]);
        gv[1] = __fadd_rn(r.y, d[1]);
        gv[2] = __fadd_rn(r.z, d[2]);
        gv[3] = __fadd_rn(r.w, d[3]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t bit = 1u << (4 * k + e);
            // an element with G == 0 is never sent: its probe is made negative
            ah[k][e] = gv[e] != 0.0f ? fabsf(probe(gv[e], d[e], kLS)) : -1.0f;
            if (kLazy) ngr |= gv[e] < 0.0f ? bit : 0u;
            const float a = fabsf(gv[e]);
            // slots outside the slice hold stale data: neither maximum takes them,
            // and they are dropped from the sent mask by the caller
            m_lo = fmaxf(m_lo, (lor & bit) ? a : 0.0f);
            m_hi = fmaxf(m_hi, (hir & bit) ? a : 0.0f);
        }
        // residue := G (sent elements are corrected once s is known)
        const uint32_t vq = (vr >> (4 * k)) & 0xfu;
        float* gp = gres + q0;
        if (vq == 0xfu) {
            *reinterpret_cast<float4*>(gp) = make_float4(gv[0], gv[1], gv[2], gv[3]);
        } else if (vq) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if ((vq >> e) & 1u) gp[e] = gv[e];
        }
    }
}

// ---------------------------------------------------------------- streaming kernel
// Warp w of CTA c handles slice w of tiles c, c + grid, c + 2 grid, ...; its S
// stages hold the data of its next S slices. Per slice, per lane (16 slots in
// registers, the four 16-byte chunks visited in the bank-conflict-free rotated
// order): G = fl32(residue + dW), |probe| (-1 where G == 0, so that such elements
// are never sent), the mask of G < 0 (deferred fix-up only), residue := G with
// 128-bit stores, and the maxima of the lane's (at most two) bins; slots outside the
// slice hold stale data and are masked out of the maxima and the sent mask. The
// stage is then refilled with the warp's slice S ahead. Bin maxima and counts go
// through the warp's scratch (shared atomics), the counts into the message and the
// maxima into the warp's 32-bit exponent buckets (flushed to the layer's exact
// accumulator every 8 slices and when the warp moves on to another layer). The
// sent mask (and, deferred fix-up only, the sign mask) go to the workspace and the
// slice's code count is added to its tile's total.
//
// kLazy: the corrections the previous call deferred (its sent mask, when the
// workspace says they are pending) are applied as the residue is loaded,
// fl32(G - copysign(s_prev, G)), the same rounding the fix-up would have made.
// kLS: the Local Selection rule (the probe is G itself).
//
// Every wait is bounded: a copy that does not land in time marks the layer with
// ADACOMP_ERR_TIMEOUT and the warp stops (later slices only mark their layers);
// before the CTA exits the warp waits, bounded again, for its copies in flight.
template <int S, bool kLazy, bool kLS>
__global__ void __launch_bounds__(kThreads, 3) slice_kernel(const __grid_constant__ KGroup g, uint8_t* __restrict__ ws)
{
    ptx::griddep_wait();  // the kernel ahead in the stream
    extern __shared__ __align__(128) uint8_t smem[];
    const SlicePlan P = slice_plan(g.d_size, S, g.num_layers);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint8_t* stages = smem + (size_t)warp * S * P.stage_bytes;
    KLayer* lays = reinterpret_cast<KLayer*>(smem + P.stages_bytes);
    uint32_t* wg = reinterpret_cast<uint32_t*>(smem + P.stages_bytes + P.layer_bytes) + warp * 2 * kWarpScratch;
    uint32_t* wc = wg + kWarpScratch;
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem + P.stages_bytes + P.layer_bytes + kWarpScratchBytes) + warp * kBkN;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + P.stages_bytes + P.layer_bytes + kWarpScratchBytes +
                                                kWarps * kBkN * 4) + warp * S;
    auto stage_r = [&](int s) { return reinterpret_cast<float*>(stages + s * P.stage_bytes); };
    auto stage_d = [&](int s) { return static_cast<void*>(stages + s * P.stage_bytes + kRBytes); };

    {
        const uint4* src = reinterpret_cast<const uint4*>(&g.layer[0]);
        uint4* dst = reinterpret_cast<uint4*>(lays);
        for (int e = tid; e < g.num_layers * (int)(sizeof(KLayer) / 16); e += kThreads) dst[e] = src[e];
    }
    wg[lane] = 0u;
    wc[lane] = 0u;
    if (lane < kWarpScratch - 32) { wg[32 + lane] = 0u; wc[32 + lane] = 0u; }
    hist[lane] = 0u;
    hist[32 + lane] = 0u;
    if (lane == 0) {
        for (int s = 0; s < S; ++s) ptx::mbar_init(&bar[s], 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();  // layer table; the only block-wide barrier

    const uint32_t T = g.total_tiles, c = blockIdx.x, GS = gridDim.x;
    uint32_t* tile_tot = reinterpret_cast<uint32_t*>(ws + sl_tot_offset(g.num_layers, T));
    uint16_t* sent = reinterpret_cast<uint16_t*>(ws + sl_sent_offset(g.num_layers, T));
    uint16_t* sign = reinterpret_cast<uint16_t*>(ws + sl_sign_offset(g.num_layers, T));
    const bool pending = kLazy && reinterpret_cast<const volatile Ctl*>(ws)->pending != 0u;
    const int rot = seg_rot(lane);

    // lane 0 starts the warp's first S slices
    int iss_lo = 0;
    uint32_t inflight = 0;  // stages with a copy in flight (lane 0's view)
    if (lane == 0) {
        for (int s = 0; s < S; ++s) {
            const uint32_t t = c + s * GS;
            if (t >= T) break;
            iss_lo = advance_layer(lays, g.num_layers, t, iss_lo);
            const Slice Sl = slice_in(lays[iss_lo], iss_lo, t, warp);
            if (t == g.inject_skip_tile) continue;  // test hook: this copy is never started
            if (issue_slice(lays[Sl.layer], Sl, stage_r(s), stage_d(s), &bar[s])) inflight |= 1u << s;
        }
    }
    __syncwarp();

    int lo = 0, hist_layer = -1, hist_slices = 0;
    bool poisoned = false;
    uint32_t i_poison = 0;
    for (uint32_t i = 0;; ++i) {
        const uint32_t t = c + i * GS;
        if (t >= T) break;
        const int s = (int)(i % S);
        lo = advance_layer(lays, g.num_layers, t, lo);
        const KLayer& ly = lays[lo];
        const Slice Sl = slice_in(ly, lo, t, warp);
        LayerWs* lw = reinterpret_cast<LayerWs*>(ws + ws_layer_offset(Sl.layer));
        const size_t mi = ((size_t)t * kWarps + warp) * 32 + lane;  // this lane's mask word
        // the previous call's deferred corrections (its sent mask and s), loaded while
        // the stage's copy is still landing
        uint32_t pm = 0;
        float s_prev = 0.0f;
        if (kLazy && pending) {
            pm = sent[mi];
            s_prev = lw->result.s;
        }
        if (!poisoned && !__all_sync(kFull, wait_bounded(&bar[s], (i / S) & 1u, g.timeout_ns))) {
            poisoned = true;  // warp-uniform
            i_poison = i;
        }
        if (poisoned) {  // the stage's data may be incomplete: report, do not compute
            if (lane == 0) atomicOr(&lw->err, kErrTimeout);
            continue;
        }
        if (lane == 0) inflight &= ~(1u << s);
        if (Sl.layer != hist_layer || hist_slices == kBkSlices) {
            if (hist_layer >= 0) flush_hist(hist, reinterpret_cast<LayerWs*>(ws + ws_layer_offset(hist_layer)), lane);
            hist_layer = Sl.layer;
            hist_slices = 0;
        }
        ++hist_slices;
        const bool one_bin = ly.bpw == 1;  // warp-uniform: the slice is one bin (m_hi and c_hi are 0)
        LaneGeo q;
        uint32_t vr, lor, hir;
        // register order: chunk k of the lane is held at registers 4k..4k+3 and is
        // slot chunk k ^ rot; every per-element test below uses a compile-time bit
        if (one_bin) {  // every valid slot belongs to the slice's only bin
            q.lane_e = (int)(Sl.a0 - Sl.ts) + kSeg * lane;
            const int vlo = max(0, Sl.we0 - q.lane_e), vhi = min(kSeg, Sl.we1 - q.lane_e);
            q.valid = vhi > vlo ? (((1u << (vhi - vlo)) - 1u) << vlo) : 0u;
            q.bin_lo = 0;
            q.split = kSeg;
            vr = to_reg_order(q.valid, rot);
            lor = vr;
            hir = 0u;
        } else {
            q = lane_geo(Sl, ly, lane);
            const uint32_t lomask = q.split >= kSeg ? 0xffffu : ((1u << max(q.split, 0)) - 1u);  // slots of bin_lo
            vr = to_reg_order(q.valid, rot);
            lor = to_reg_order(lomask, rot) & vr;  // valid slots of bin_lo
            hir = vr & ~lor;                        // valid slots of bin_lo + 1
        }
        float ah[4][4];             // |probe| per register slot
        uint32_t ngr = 0;  // G < 0 (register order; kept for the deferred fix-up's codes only)
        float m_lo = 0.0f, m_hi = 0.0f;
        if (q.valid)
            lane_slots<kLazy, kLS>(ly, Sl, stage_r(s), stage_d(s), lane, rot, pm, s_prev, vr, lor, hir, ah, ngr, m_lo,
                                   m_hi);
        // the stage is not read again: lane 0 refills it with the slice S ahead (one
        // warp's shared memory accesses are performed in order, so its reads of the
        // stage precede the copy)
        __syncwarp();
        if (lane == 0) {
            const uint32_t tn = t + S * GS;
            if (tn < T) {
                iss_lo = advance_layer(lays, g.num_layers, tn, iss_lo);
                const Slice Sn = slice_in(lays[iss_lo], iss_lo, tn, warp);
                if (tn != g.inject_skip_tile &&
                    issue_slice(lays[Sn.layer], Sn, stage_r(s), stage_d(s), &bar[s]))
                    inflight |= 1u << s;
            }
        }
        if (one_bin) {  // a warp reduction instead of 32 lanes' atomics on one word
            const uint32_t x = __reduce_max_sync(kFull, __float_as_uint(m_lo));
            if (lane == 0) wg[0] = x;
        } else {
            if (m_lo > 0.0f) atomicMax(&wg[q.bin_lo], __float_as_uint(m_lo));
            if (m_hi > 0.0f) atomicMax(&wg[q.bin_lo + 1], __float_as_uint(m_hi));
        }
        __syncwarp();
        uint32_t fr = 0;  // sent slots, register order
        if (q.valid) {
            const float gm_lo = __uint_as_float(wg[q.bin_lo]);
            const float gm_hi = hir ? __uint_as_float(wg[q.bin_lo + 1]) : 0.0f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t bit = 1u << (4 * k + e);
                    fr |= ah[k][e] >= ((lor & bit) ? gm_lo : gm_hi) ? bit : 0u;
                }
            }
            fr &= vr;
            if (!one_bin) {
                const uint32_t c_lo = __popc(fr & lor), c_hi = __popc(fr & ~lor);
                if (c_lo) atomicAdd(&wc[q.bin_lo], c_lo);
                if (c_hi) atomicAdd(&wc[q.bin_lo + 1], c_hi);
            }
        }
        if (one_bin) {
            const uint32_t n1 = __reduce_add_sync(kFull, (uint32_t)__popc(fr));
            if (lane == 0) wc[0] = n1;
        }
        __syncwarp();
        // the slice's bins: counts into the message, maxima into the buckets; the
        // scratch is left zero
        if (lane < Sl.nb) {
            const uint32_t u = wg[lane];  // the bin maximum, |G| as fp32 bits
            reinterpret_cast<uint16_t*>(ly.msg + 8)[Sl.first_bin + Sl.wb0 + lane] = (uint16_t)wc[lane];
            if (u) {
                const uint32_t E = u >> 23;
                const unsigned long long M = E ? ((u & 0x7fffffu) | 0x800000u) : (u & 0x7fffffu);
                if (E - kBkLo < (uint32_t)kBkN) atomicAdd(&hist[E - kBkLo], (uint32_t)M);
                else atomicAdd(&lw->acc[E], M);
            }
        }
        __syncwarp();
        wg[lane] = 0u;
        wc[lane] = 0u;
        sent[mi] = (uint16_t)fr;  // register order (the emitting kernel reorders)
        if (kLazy) sign[mi] = (uint16_t)(ngr & fr);  // without the fix-up, the emitting kernel has no G
        const uint32_t total = __reduce_add_sync(kFull, (uint32_t)__popc(fr));
        if (lane == 0 && total) atomicAdd(&tile_tot[t], total);
    }
    if (hist_layer >= 0) flush_hist(hist, reinterpret_cast<LayerWs*>(ws + ws_layer_offset(hist_layer)), lane);
    if (poisoned && lane == 0) {
        // copies that may still be in flight get one more bounded wait before the
        // CTA's shared memory is released
        for (uint32_t j = i_poison; j < i_poison + S; ++j) {
            const int s = (int)(j % S);
            if (c + j * GS < T && (inflight >> s) & 1u) wait_bounded(&bar[s], (j / S) & 1u, g.timeout_ns);
        }
    }
}

// ---------------------------------------------------------------- block-sliced streaming kernel
// One tile at a time per CTA (tiles c, c + grid, ...), warp w streaming slice w of
// each through its own S-stage pipeline of bulk copies, as in slice_kernel. The CTA
// has one warp per slice of the group's widest tile (W <= 16; slices past a tile's
// end are empty). A bin now spans several warps, so its maximum and count meet in
// shared memory. Per tile, in two passes over the warp's stage:
//   1. G = fl32(residue + dW), residue := G, and the lanes' bin maxima, folded per
//      bin (a 512-slot slice meets at most three bins) with warp reductions and one
//      shared atomicMax per bin; then one block barrier;
//   2. the selection against the bins' maxima, from the probes abs(H) that pass 1
//      wrote over the lane's residue slots of the stage (cheaper than keeping them in
//      registers across the barrier: fewer registers, more resident warps), the
//      masks, and the per-bin counts (warp reductions, one shared atomicAdd per bin);
//      then the stage is refilled.
// The counts of tile i are complete at the barrier of tile i + 1, where the finishing
// warp (the last) writes them into the message, adds the maxima to the CTA's exponent
// buckets (64-bit, one per fp32 exponent, flushed to the layer's exact accumulator
// when the CTA moves to another layer and at the end) and writes the tile's code
// total. Maxima and counts rotate through three buffers, so one barrier per tile
// suffices. The sent mask (and with the fix-up deferred, the sign mask) of every
// slice holding elements goes to the workspace, 16 slices per tile; the finalising
// and emitting kernels follow. Waits are bounded as in slice_kernel; a warp whose
// copy did not land marks the layer, computes nothing further, and keeps taking part
// in the barriers.
constexpr int kBigMaxRegs = 64;

struct BigPlan {
    uint32_t d_bytes, stage_bytes, stages_bytes, layer_bytes, total;
};
__host__ __device__ inline BigPlan big_plan(uint32_t d_size, int stages, int num_layers, int warps)
{
    BigPlan p;
    p.d_bytes = d_size == 4 ? kDBytes32 : kDBytes16;
    p.stage_bytes = kRBytes + p.d_bytes;
    p.stages_bytes = (uint32_t)warps * stages * p.stage_bytes;
    p.layer_bytes = (uint32_t)num_layers * 64u;
    // + maxima and counts [3][kBigMaxBins] u32 each, 256 u64 exponent buckets, barriers
    p.total = p.stages_bytes + p.layer_bytes + 6 * kBigMaxBins * 4 + 256 * 8 + (uint32_t)warps * stages * 8;
    return p;
}

// Chunk q0 .. q0 + 3 of a lane's slots from a stage (rs: the lane's residue slots,
// ds: the stage's dW, doff: the dW stage offset of slot 0 of lane 0): G = fl32(residue
// + dW) after the deferred correction of the slots set in pmk, and dW.
template <bool kLazy>
__device__ __forceinline__ void chunk_g(bool bf16, const float* rs, const void* ds, int doff, int lane, int q0,
                                        uint32_t pmk, float s_prev, float (&gv)[4], float (&d)[4])
{
    float4 r = *reinterpret_cast<const float4*>(rs + q0);
    if (kLazy && pmk) {
        if (pmk & 1u) r.x = __fsub_rn(r.x, copysignf(s_prev, r.x));
        if (pmk & 2u) r.y = __fsub_rn(r.y, copysignf(s_prev, r.y));
        if (pmk & 4u) r.z = __fsub_rn(r.z, copysignf(s_prev, r.z));
        if (pmk & 8u) r.w = __fsub_rn(r.w, copysignf(s_prev, r.w));
    }
    if (bf16) {
        const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(ds) + doff + kSeg * lane + q0);
        d[0] = bf16_lo(u.x); d[1] = bf16_hi(u.x); d[2] = bf16_lo(u.y); d[3] = bf16_hi(u.y);
    } else {
        const float4 v = *reinterpret_cast<const float4*>(static_cast<const float*>(ds) + kSeg * lane + q0);
        d[0] = v.x; d[1] = v.y; d[2] = v.z; d[3] = v.w;
    }
    gv[0] = __fadd_rn(r.x, d[0]);
    gv[1] = __fadd_rn(r.y, d[1]);
    gv[2] = __fadd_rn(r.z, d[2]);
    gv[3] = __fadd_rn(r.w, d[3]);
}

template <int S, bool kLazy, bool kLS>
__global__ void __maxnreg__(kBigMaxRegs) block_kernel(const __grid_constant__ KGroup g, uint8_t* __restrict__ ws)
{
    ptx::griddep_wait();  // the kernel ahead in the stream
    extern __shared__ __align__(128) uint8_t smem[];
    const int W = (int)(blockDim.x >> 5);
    const BigPlan P = big_plan(g.d_size, S, g.num_layers, W);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint8_t* stages = smem + (size_t)warp * S * P.stage_bytes;
    KLayer* lays = reinterpret_cast<KLayer*>(smem + P.stages_bytes);
    uint32_t* bmax = reinterpret_cast<uint32_t*>(smem + P.stages_bytes + P.layer_bytes);  // [3][kBigMaxBins]
    uint32_t* bcnt = bmax + 3 * kBigMaxBins;                                              // [3][kBigMaxBins]
    unsigned long long* hist = reinterpret_cast<unsigned long long*>(bcnt + 3 * kBigMaxBins);
    uint64_t* bar = reinterpret_cast<uint64_t*>(hist + 256) + warp * S;
    auto stage_r = [&](int s) { return reinterpret_cast<float*>(stages + s * P.stage_bytes); };
    auto stage_d = [&](int s) { return static_cast<void*>(stages + s * P.stage_bytes + kRBytes); };

    {
        const uint4* src = reinterpret_cast<const uint4*>(&g.layer[0]);
        uint4* dst = reinterpret_cast<uint4*>(lays);
        for (int e = tid; e < g.num_layers * (int)(sizeof(KLayer) / 16); e += blockDim.x) dst[e] = src[e];
    }
    for (int e = tid; e < 6 * kBigMaxBins; e += blockDim.x) bmax[e] = 0u;
    for (int e = tid; e < 256; e += blockDim.x) hist[e] = 0ull;
    if (lane == 0) {
        for (int s = 0; s < S; ++s) ptx::mbar_init(&bar[s], 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();

    const uint32_t T = g.total_tiles, c = blockIdx.x, GS = gridDim.x;
    uint32_t* tile_tot = reinterpret_cast<uint32_t*>(ws + sl_tot_offset(g.num_layers, T));
    uint16_t* sent = reinterpret_cast<uint16_t*>(ws + sl_sent_offset(g.num_layers, T));
    uint16_t* sign = reinterpret_cast<uint16_t*>(ws + sl_sign_offset(g.num_layers, T, true));
    const bool pending = kLazy && reinterpret_cast<const volatile Ctl*>(ws)->pending != 0u;
    const int rot = seg_rot(lane);

    int iss_lo = 0;
    uint32_t inflight = 0;
    if (lane == 0) {
        for (int s = 0; s < S; ++s) {
            const uint32_t t = c + s * GS;
            if (t >= T) break;
            iss_lo = advance_layer(lays, g.num_layers, t, iss_lo);
            const Slice Sl = big_slice(lays[iss_lo], iss_lo, t, warp);
            if (t == g.inject_skip_tile) continue;  // test hook: this copy is never started
            if (issue_slice(lays[iss_lo], Sl, stage_r(s), stage_d(s), &bar[s])) inflight |= 1u << s;
        }
    }
    __syncwarp();

    // the finishing warp: tile tp's counts into the message, its maxima into the
    // buckets (flushed first if the tile starts another layer), its code total; the
    // buffers of parity `par` are left zero
    int hist_layer = -1;
    auto flush = [&]() {
        if (hist_layer < 0) return;
        LayerWs* hw = reinterpret_cast<LayerWs*>(ws + ws_layer_offset(hist_layer));
        __syncwarp();
        for (int e = lane; e < 256; e += 32) {
            const unsigned long long v = hist[e];
            if (v) {
                atomicAdd(&hw->acc[e], v);
                hist[e] = 0ull;
            }
        }
        __syncwarp();
    };
    auto finish = [&](uint32_t tp, int lp, int par) {
        if (lp != hist_layer) {
            flush();
            hist_layer = lp;
        }
        const KLayer& ly = lays[lp];
        const uint32_t fb = (tp - ly.tile_begin) * ly.bins_per_tile;
        const int nb = (int)min(ly.bins_per_tile, ly.nbins - fb);
        uint32_t cnt = 0;
        if (lane < nb) {
            cnt = bcnt[par * kBigMaxBins + lane];
            const uint32_t u = bmax[par * kBigMaxBins + lane];
            reinterpret_cast<uint16_t*>(ly.msg + 8)[fb + lane] = (uint16_t)cnt;
            if (u) {
                const uint32_t E = u >> 23;
                atomicAdd(&hist[E], (unsigned long long)(E ? ((u & 0x7fffffu) | 0x800000u) : (u & 0x7fffffu)));
            }
        }
        if (lane < kBigMaxBins) {
            bmax[par * kBigMaxBins + lane] = 0u;
            bcnt[par * kBigMaxBins + lane] = 0u;
        }
        const uint32_t total = __reduce_add_sync(kFull, cnt);
        if (lane == 0) tile_tot[tp] = total;
    };

    int lo = 0, l_prev = -1;
    uint32_t t_prev = 0, i = 0;
    bool poisoned = false;
    uint32_t i_poison = 0;
    for (;; ++i) {
        const uint32_t t = c + i * GS;
        if (t >= T) break;  // uniform over the CTA
        const int s = (int)(i % S), par = (int)(i % 3);
        lo = advance_layer(lays, g.num_layers, t, lo);
        const KLayer& ly = lays[lo];
        const Slice Sl = big_slice(ly, lo, t, warp);
        LayerWs* lw = reinterpret_cast<LayerWs*>(ws + ws_layer_offset(lo));
        const size_t mi = ((size_t)t * kBigSlices + warp) * 32 + lane;
        uint32_t pm = 0;
        float s_prev = 0.0f;
        if (kLazy && pending && Sl.we1 > Sl.we0) {
            pm = sent[mi];
            s_prev = lw->result.s;
        }
        if (!poisoned && !__all_sync(kFull, wait_bounded(&bar[s], (i / S) & 1u, g.timeout_ns))) {
            poisoned = true;
            i_poison = i;
        }
        if (poisoned && lane == 0) atomicOr(&lw->err, kErrTimeout);
        if (!poisoned && lane == 0) inflight &= ~(1u << s);
        // a tile of one bin (L_T > 2048): every slot of the slice belongs to bin 0
        const bool one_bin = Sl.nb == 1;  // uniform over the CTA
        LaneGeo q;
        uint32_t vr, lor, hir;
        if (one_bin) {
            q.lane_e = (int)(Sl.a0 - Sl.ts) + kSeg * lane;
            const int vlo = max(0, Sl.we0 - q.lane_e), vhi = min(kSeg, Sl.we1 - q.lane_e);
            q.valid = vhi > vlo ? (((1u << (vhi - vlo)) - 1u) << vlo) : 0u;
            q.bin_lo = 0;
            q.split = kSeg;
            if (poisoned) q.valid = 0u;  // the stage's data may be incomplete: compute nothing
            vr = to_reg_order(q.valid, rot);
            lor = vr;
            hir = 0u;
        } else {
            q = big_lane_geo(Sl, ly, lane);
            if (poisoned) q.valid = 0u;
            const uint32_t lomask = q.split >= kSeg ? 0xffffu : ((1u << max(q.split, 0)) - 1u);
            vr = to_reg_order(q.valid, rot);
            lor = to_reg_order(lomask, rot) & vr;
            hir = vr & ~lor;
        }
        float* rs = stage_r(s) + kSeg * lane;
        const void* ds = stage_d(s);
        const int doff = ly.dw_bf16 ? (int)(Sl.a0 - ((Sl.ts + Sl.we0) & ~(int64_t)7)) : 0;
        // pass 1: G, residue := G, the lane's bin maxima; the probe abs(H) (-1 where
        // G == 0, so that such elements are never sent) replaces the lane's residue
        // slots in the stage, and the signs of G are kept for the deferred fix-up
        float m_lo = 0.0f, m_hi = 0.0f;
        uint32_t ngr = 0;
        if (q.valid) {
            float* gres = ly.residue + Sl.a0 + kSeg * lane;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int q0 = 4 * (k ^ rot);
                float gv[4], d[4], ah[4];
                chunk_g<kLazy>(ly.dw_bf16, rs, ds, doff, lane, q0, (pm >> (4 * k)) & 0xfu, s_prev, gv, d);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t bit = 1u << (4 * k + e);
                    const float a = fabsf(gv[e]);
                    m_lo = fmaxf(m_lo, (lor & bit) ? a : 0.0f);
                    m_hi = fmaxf(m_hi, (hir & bit) ? a : 0.0f);
                    ah[e] = gv[e] != 0.0f ? fabsf(probe(gv[e], d[e], kLS)) : -1.0f;
                    if (kLazy) ngr |= gv[e] < 0.0f ? bit : 0u;
                }
                *reinterpret_cast<float4*>(rs + q0) = make_float4(ah[0], ah[1], ah[2], ah[3]);
                const uint32_t vq = (vr >> (4 * k)) & 0xfu;
                float* gp = gres + q0;
                if (vq == 0xfu) {
                    *reinterpret_cast<float4*>(gp) = make_float4(gv[0], gv[1], gv[2], gv[3]);
                } else if (vq) {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if ((vq >> e) & 1u) gp[e] = gv[e];
                }
            }
        }
        // the warp's bins (Sl.wb0 + 0, 1, 2): maxima as fp32 bits (non-negative, so
        // they order as unsigned integers)
        const int rb = q.bin_lo - Sl.wb0;  // 0, 1 or 2 for lanes holding elements
        if (one_bin) {
            const uint32_t x0 = __reduce_max_sync(kFull, __float_as_uint(m_lo));
            if (lane == 0 && x0) atomicMax(&bmax[par * kBigMaxBins], x0);
        } else {
            const uint32_t ulo = __float_as_uint(m_lo), uhi = __float_as_uint(m_hi);
            const uint32_t x0 = __reduce_max_sync(kFull, rb == 0 ? ulo : 0u);
            const uint32_t x1 = __reduce_max_sync(kFull, max(rb == 1 ? ulo : 0u, rb == 0 ? uhi : 0u));
            const uint32_t x2 = __reduce_max_sync(kFull, max(rb == 2 ? ulo : 0u, rb == 1 ? uhi : 0u));
            if (lane < 3) {
                const uint32_t x = lane == 0 ? x0 : (lane == 1 ? x1 : x2);
                if (x) atomicMax(&bmax[par * kBigMaxBins + Sl.wb0 + lane], x);
            }
        }
        __syncthreads();  // the tile's maxima are complete, and the previous tile's counts
        if (warp == W - 1 && l_prev >= 0) finish(t_prev, l_prev, (int)((i + 2) % 3));
        // pass 2: the selection against the bins' maxima, from the probes in the stage
        uint32_t fr = 0;
        if (q.valid) {
            const float gm_lo = __uint_as_float(bmax[par * kBigMaxBins + q.bin_lo]);
            const float gm_hi = hir ? __uint_as_float(bmax[par * kBigMaxBins + q.bin_lo + 1]) : 0.0f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float4 a4 = *reinterpret_cast<const float4*>(rs + 4 * (k ^ rot));
                const float ah[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t bit = 1u << (4 * k + e);
                    fr |= ah[e] >= ((lor & bit) ? gm_lo : gm_hi) ? bit : 0u;
                }
            }
            fr &= vr;
        }
        // the probes written into the stage (generic proxy) come before the bulk copy
        // that refills it (async proxy)
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && !poisoned) {  // the stage is not read again: refill it with the tile S ahead
            const uint32_t tn = t + S * GS;
            if (tn < T) {
                iss_lo = advance_layer(lays, g.num_layers, tn, iss_lo);
                const Slice Sn = big_slice(lays[iss_lo], iss_lo, tn, warp);
                if (tn != g.inject_skip_tile && issue_slice(lays[iss_lo], Sn, stage_r(s), stage_d(s), &bar[s]))
                    inflight |= 1u << s;
            }
        }
        if (one_bin) {
            const uint32_t n0 = __reduce_add_sync(kFull, (uint32_t)__popc(fr));
            if (lane == 0 && n0) atomicAdd(&bcnt[par * kBigMaxBins], n0);
        } else {
            const uint32_t c_lo = __popc(fr & lor), c_hi = __popc(fr & hir);
            const uint32_t n0 = __reduce_add_sync(kFull, rb == 0 ? c_lo : 0u);
            const uint32_t n1 = __reduce_add_sync(kFull, (rb == 1 ? c_lo : 0u) + (rb == 0 ? c_hi : 0u));
            const uint32_t n2 = __reduce_add_sync(kFull, (rb == 2 ? c_lo : 0u) + (rb == 1 ? c_hi : 0u));
            if (lane < 3) {
                const uint32_t x = lane == 0 ? n0 : (lane == 1 ? n1 : n2);
                if (x) atomicAdd(&bcnt[par * kBigMaxBins + Sl.wb0 + lane], x);
            }
        }
        if (Sl.we1 > Sl.we0) {
            sent[mi] = (uint16_t)fr;  // register order (the emitting kernel reorders)
            if (kLazy) sign[mi] = (uint16_t)(ngr & fr);
        }
        t_prev = t;
        l_prev = lo;
    }
    __syncthreads();  // the last tile's counts
    if (warp == W - 1) {
        if (l_prev >= 0) finish(t_prev, l_prev, (int)((i + 2) % 3));
        flush();
    }
    if (poisoned && lane == 0) {
        for (uint32_t j = i_poison; j < i_poison + S; ++j) {
            const int s = (int)(j % S);
            if (c + j * GS < T && (inflight >> s) & 1u) wait_bounded(&bar[s], (j / S) & 1u, g.timeout_ns);
        }
    }
}

// ---------------------------------------------------------------- finalise and scan
// Grid: x = chunk of kFinThreads tiles, y = layer (CTAs past a layer's last chunk
// exit at once). The CTA of chunk c sums the totals of the layer's tiles before the
// chunk itself (coalesced, kFinUnroll loads per thread in flight; the repeated reads
// are small and hit L2), scans its own chunk with one block scan, and writes the
// chunk's exclusive tile code offsets. The CTA of the layer's last chunk also forms s
// from the layer's exact sum (fp64, rounded once to fp32), the header {s, B} and the
// result area. The tile totals are left for the emitting kernel, which clears them.
constexpr int kFinThreads = 1024;
constexpr int kFinWarps = kFinThreads / 32;
constexpr int kFinUnroll = 8;

__global__ void __launch_bounds__(kFinThreads) slice_finalize_kernel(const __grid_constant__ KGroup g,
                                                                     uint8_t* __restrict__ ws)
{
    ptx::griddep_wait();  // the kernel ahead in the stream
    __shared__ unsigned long long tmp[256];
    __shared__ unsigned long long words[kSumWords];
    __shared__ unsigned long long red[kFinWarps];
    __shared__ uint32_t wt[kFinWarps];
    const int l = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const KLayer& ly = g.layer[l];
    const uint32_t nt = ly.num_tiles;
    const uint32_t c0 = blockIdx.x * kFinThreads;  // the chunk's first tile (layer-relative)
    if (c0 >= nt) return;
    const bool last_chunk = c0 + kFinThreads >= nt;
    LayerWs* lw = reinterpret_cast<LayerWs*>(ws + ws_layer_offset(l));
    const uint32_t T = g.total_tiles;
    const uint32_t* tot = reinterpret_cast<const uint32_t*>(ws + sl_tot_offset(g.num_layers, T)) + ly.tile_begin;
    uint64_t* excl = reinterpret_cast<uint64_t*>(ws + sl_excl_offset(g.num_layers)) + ly.tile_begin;
    if (last_chunk) {
        if (tid < kSumWords) words[tid] = 0ull;
        if (tid < 256) tmp[tid] = lw->acc[tid];
    }
    // the codes of the tiles before the chunk
    unsigned long long before = 0;
    for (uint32_t i0 = 0; i0 < c0; i0 += kFinUnroll * kFinThreads) {
        uint32_t v[kFinUnroll];
#pragma unroll
        for (int u = 0; u < kFinUnroll; ++u) {
            const uint32_t i = i0 + u * kFinThreads + tid;
            v[u] = i < c0 ? tot[i] : 0u;
        }
#pragma unroll
        for (int u = 0; u < kFinUnroll; ++u) before += v[u];
    }
    // the chunk's own tiles: one per thread, scanned
    const uint32_t j = c0 + tid;
    const uint32_t mine = j < nt ? tot[j] : 0u;
    // a warp's share: at most 32 x (tiles before the chunk / 1024) x 8189 codes < 2^32 for
    // layers below 2^36 elements
    before = __reduce_add_sync(kFull, (uint32_t)before);
    uint32_t incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) wt[warp] = incl;
    if (lane == 0) red[warp] = before;
    __syncthreads();
    if (warp == 0) {
        unsigned long long b = red[lane];  // the warps' shares of the codes before the chunk
#pragma unroll
        for (int o = 16; o; o >>= 1) b += __shfl_xor_sync(kFull, b, o);
        const uint32_t x = wt[lane];
        uint32_t sx = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(kFull, sx, o);
            if (lane >= o) sx += y;
        }
        __syncwarp();
        red[lane] = b + (sx - x);  // exclusive offset of warp `lane`'s first tile
    }
    __syncthreads();
    const unsigned long long off = red[warp] + (incl - mine);
    if (j < nt) excl[j] = off;
    if (!last_chunk) return;
    // the last chunk's last tile ends the layer
    __shared__ unsigned long long nnz_s;
    if (j == nt - 1) nnz_s = off + mine;
    __syncthreads();
    const unsigned long long nnz = nnz_s;
    if (warp == 0) {
        const double Ssum = exact_sum_warp(tmp, words, lane);
        if (lane == 0) {
            const float s = __double2float_rn(__ddiv_rn(Ssum, (double)ly.nbins));
            const bool bad = *reinterpret_cast<volatile uint32_t*>(&lw->err) != 0u;
            *reinterpret_cast<float*>(ly.msg) = s;
            *reinterpret_cast<uint32_t*>(ly.msg + 4) = ly.nbins;
            lw->result.s = s;
            lw->result.status = bad ? 6u /* ADACOMP_ERR_TIMEOUT */ : 0u;
            lw->result.nnz = bad ? 0ull : nnz;
            lw->result.msg_bytes = 8ull + 2ull * ly.nbins + (bad ? 0ull : (unsigned long long)ly.code_bytes * nnz);
            lw->done = 0;
            lw->err = 0;
        }
    }
    if (tid < 256) lw->acc[tid] = 0ull;
    if (l == 0 && tid == 0) reinterpret_cast<volatile Ctl*>(ws)->pending = g.lazy ? 1u : 0u;
}

// ---------------------------------------------------------------- codes and fix-up
// Persistent warps take the tiles last first (the residue lines the streaming kernel
// wrote last are the likeliest to be still in L2); a warp loads its next tile's masks
// and code offset before it emits the current tile.
// Emit lane L covers slice L >> 2, compute lanes 8 (L & 3) .. 8 (L & 3) + 7: one
// 16-byte load of their sent masks. The masks are stored in the streaming kernel's
// register order and are brought back to slot order here. An exclusive warp scan of
// the lanes' popcounts places each lane's sent elements, in element order (which is
// code order), in a per-warp list in shared memory; the warp then walks the list
// with consecutive lanes on consecutive codes, kFixBatch elements per lane at a time:
// all residue loads issued first (with a 64-byte L2 fill size: a scattered 4-byte
// load otherwise fills a whole 128-byte line), then the code ((element - its bin's
// first element) << 1) | (G < 0) and the residue fl32(G - sign(G) s). A tile with more
// than kListCap sent elements is listed and walked in rounds. The tiles' code totals
// (read by the finalising kernel) are cleared here for the next call. (With the
// fix-up deferred, slice_codes_kernel below writes the codes instead.)
constexpr int kEmitThreads = 256;
constexpr int kEmitWarps = kEmitThreads / 32;
constexpr int kListCap = 1024;
constexpr int kFixBatch = 4;

__device__ __forceinline__ float ld_fill64(const float* p)
{
    float v;
    asm volatile("ld.global.L2::64B.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

// The inputs of one tile's emission, loaded a tile ahead: per group of eight slices
// (one for warp-sliced tiles, two for block-sliced ones) the sent masks of the lane's
// eight compute lanes (register order).
template <int H>
struct EmitIn {
    uint4 f[H];
    uint64_t pos;   // the tile's first code position in its message
    int used;       // block-sliced tiles: slices holding elements (the others' masks are never written)
};

template <bool kBig>
__device__ __forceinline__ EmitIn<kBig ? 2 : 1> emit_load(const KGroup& g, const uint32_t* tb, const uint8_t* ws,
                                                         uint32_t T, uint32_t t, int lane)
{
    constexpr int H = kBig ? 2 : 1;
    EmitIn<H> in;
    in.used = kBig ? big_slices_used(g.layer[layer_of_tile(tb, g.num_layers, t)], t) : kWarps;
    const int hs = in.used > kWarps ? 2 : 1;  // groups holding elements
    const uint4* sent = reinterpret_cast<const uint4*>(ws + sl_sent_offset(g.num_layers, T));
#pragma unroll
    for (int h = 0; h < H; ++h)
        in.f[h] = h < hs ? sent[((size_t)t * H + h) * 32 + lane] : make_uint4(0u, 0u, 0u, 0u);
    in.pos = reinterpret_cast<const uint64_t*>(ws + sl_excl_offset(g.num_layers))[t];
    return in;
}

template <bool kBig>
__global__ void __launch_bounds__(kEmitThreads, kBig ? 4 : 5) slice_emit_kernel(const __grid_constant__ KGroup g,
                                                                             uint8_t* __restrict__ ws)
{
    ptx::griddep_wait();  // the kernel ahead in the stream
    constexpr int H = kBig ? 2 : 1;
    __shared__ uint32_t tb[kMaxGroup];  // first tile of each layer
    __shared__ uint16_t lists[kEmitWarps][kListCap];
    for (int e = threadIdx.x; e < g.num_layers; e += kEmitThreads) tb[e] = g.layer[e].tile_begin;
    __syncthreads();
    const int lane = threadIdx.x & 31;
    uint16_t* lst = lists[threadIdx.x >> 5];
    const uint32_t T = g.total_tiles;
    const uint32_t NW = gridDim.x * kEmitWarps;
    uint32_t q = blockIdx.x * kEmitWarps + (threadIdx.x >> 5);
    if (q >= T) return;
    const int cl0 = 8 * (lane & 3);  // the lane's first compute lane
    EmitIn<H> cur = emit_load<kBig>(g, tb, ws, T, T - 1u - q, lane);
    int l_cached = -1;
    float s = 0.0f;
    uint32_t status = 0;
    uint32_t* tile_tot = reinterpret_cast<uint32_t*>(ws + sl_tot_offset(g.num_layers, T));
    for (; q < T; q += NW) {
        const uint32_t t = T - 1u - q;
        const EmitIn<H> in = cur;
        if (q + NW < T) cur = emit_load<kBig>(g, tb, ws, T, T - 1u - (q + NW), lane);
        if (lane == 0) tile_tot[t] = 0u;  // the tile totals start the next call at zero
        const int l = layer_of_tile(tb, g.num_layers, t);
        const KLayer& ly = g.layer[l];
        if (l != l_cached) {
            const LayerWs* lw = reinterpret_cast<const LayerWs*>(ws + ws_layer_offset(l));
            s = lw->result.s;
            status = lw->result.status;
            l_cached = l;
        }
        if (status != 0u) continue;  // a layer whose streaming pass did not complete
        uint64_t pos_h = in.pos;  // first code position of the group of slices
#pragma unroll 1
        for (int h = 0; h < H; ++h) {
            const int w = kWarps * h + (lane >> 2);  // the lane's slice
            // (selected, not indexed, to stay out of local memory; empty slices hold no codes)
            const bool live = !kBig || w < in.used;
            const uint4 fh = live ? (h ? in.f[H - 1] : in.f[0]) : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t fw[4] = {fh.x, fh.y, fh.z, fh.w};
            // the lane's eight masks in slot order, and its count
            uint32_t m[8];
            uint32_t c = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                m[i] = to_slot_order((fw[i >> 1] >> (16 * (i & 1))) & 0xffffu, seg_rot(cl0 + i));
                c += __popc(m[i]);
            }
            uint32_t incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(kFull, incl, o);
                if (lane >= o) incl += y;
            }
            const uint32_t n = __shfl_sync(kFull, incl, 31);
            if (n == 0u) continue;
            const Slice Sl = kBig ? big_slice(ly, l, t, w) : slice_in(ly, l, t, w);
            const int x0 = (int)(Sl.a0 - Sl.ts) + kSeg * cl0;  // tile element of slot 0 of compute lane cl0
            float* res = ly.residue + Sl.ts;
            uint8_t* codes = ly.msg + 8 + 2ull * ly.nbins;
            for (uint32_t r0 = 0; r0 < n; r0 += kListCap) {
                // list this round's elements: positions r0 .. r0 + kListCap - 1 of the group
                uint32_t li = incl - c;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    uint32_t mm = m[i];
                    while (mm) {
                        const int b = __ffs(mm) - 1;
                        mm &= mm - 1;
                        if (li - r0 < (uint32_t)kListCap) lst[li - r0] = (uint16_t)(x0 + kSeg * i + b);
                        ++li;
                    }
                }
                __syncwarp();
                const uint32_t nr = min(n - r0, (uint32_t)kListCap);
                const uint64_t pos0 = pos_h + r0;
                for (uint32_t j0 = 0; j0 < nr; j0 += 32 * kFixBatch) {
                    uint32_t e[kFixBatch];
                    float v[kFixBatch];
#pragma unroll
                    for (int k = 0; k < kFixBatch; ++k) {
                        const uint32_t j = j0 + k * 32 + lane;
                        e[k] = j < nr ? (uint32_t)lst[j] : 0xffffffffu;
                    }
#pragma unroll
                    for (int k = 0; k < kFixBatch; ++k)
                        if (e[k] != 0xffffffffu) v[k] = ld_fill64(res + e[k]);
#pragma unroll
                    for (int k = 0; k < kFixBatch; ++k) {
                        if (e[k] == 0xffffffffu) continue;
                        const uint32_t neg = v[k] < 0.0f ? 1u : 0u;
                        const uint32_t off = e[k] - __umulhi(e[k], ly.inv_len) * (uint32_t)ly.bin_len;  // e < 2^16: exact
                        const uint32_t code = (off << 1) | neg;
                        const uint64_t pos = pos0 + j0 + k * 32 + lane;
                        if (ly.code_bytes == 1) codes[pos] = (uint8_t)code;
                        else reinterpret_cast<uint16_t*>(codes)[pos] = (uint16_t)code;
                        res[e[k]] = neg ? __fadd_rn(v[k], s) : __fsub_rn(v[k], s);
                    }
                }
                __syncwarp();  // the list is rewritten by the next round, group or tile
            }
            pos_h += n;
        }
    }
}

// ---------------------------------------------------------------- codes only (deferred fix-up)
// With the fix-up deferred, emitting touches no residue: the codes follow from the
// sent and sign masks alone. One warp per tile, every tile at once (no persistence:
// there are no residue lines to find in L2). The tile's masks are read as 32-bit
// words, a word holding two adjacent compute lanes' 16 slots (so the words, in
// order, cover the tile's slots in order): in each round lane i takes word
// 32 r + i, brings its two halves to slot order, and writes the codes of its set
// slots ((element - its bin's first element) << 1 | sign) at consecutive positions
// from the tile's offset plus the codes of the words before it (a warp scan).
// A word of two compute lanes' masks (cl, cl + 1, cl even: both have the same
// chunk rotation) from register order to slot order: nibble k of each half moves to
// k ^ rot.
__device__ __forceinline__ uint32_t word_to_slot_order(uint32_t x, int rot)
{
    const uint32_t n = ((x << 4) & 0xf0f0f0f0u) | ((x >> 4) & 0x0f0f0f0fu);  // rot bit 0: swap nibble pairs
    x = (rot & 1) ? n : x;
    const uint32_t b = __byte_perm(x, 0u, 0x2301);                         // rot bit 1: swap bytes per half
    return (rot & 2) ? b : x;
}

template <bool kBig>
__global__ void __launch_bounds__(kEmitThreads) slice_codes_kernel(const __grid_constant__ KGroup g,
                                                                   uint8_t* __restrict__ ws)
{
    ptx::griddep_wait();  // the kernel ahead in the stream
    constexpr int W = kBig ? kBigSlices : kWarps;  // slices per tile
    constexpr int R = W / 2;                       // rounds: 16 words per slice, 32 per round
    __shared__ uint32_t tb[kMaxGroup];  // first tile of each layer
    __shared__ uint32_t st[kMaxGroup];  // each layer's status
    for (int e = threadIdx.x; e < g.num_layers; e += kEmitThreads) {
        tb[e] = g.layer[e].tile_begin;
        st[e] = reinterpret_cast<const LayerWs*>(ws + ws_layer_offset(e))->result.status;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const uint32_t T = g.total_tiles;
    const uint32_t t = blockIdx.x * kEmitWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    const uint32_t* sent = reinterpret_cast<const uint32_t*>(ws + sl_sent_offset(g.num_layers, T)) + (size_t)t * W * 16;
    const uint32_t* sign = reinterpret_cast<const uint32_t*>(ws + sl_sign_offset(g.num_layers, T, kBig)) + (size_t)t * W * 16;
    const int l = layer_of_tile(tb, g.num_layers, t);
    const KLayer& ly = g.layer[l];
    // the tile: its first bin and element, bins and elements
    const uint32_t fb = (t - ly.tile_begin) * ly.bins_per_tile;
    const int nb = (int)min(ly.bins_per_tile, ly.nbins - fb);
    const int64_t ts = (int64_t)fb * ly.bin_len;
    const int used = kBig ? (int)(((int)(ts & 3) + (int)min((int64_t)nb * ly.bin_len, ly.n - ts) + kSlots - 1) / kSlots) : W;
    uint32_t f[R], ng[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const bool live = (r * 32 + lane) / 16 < used;  // the masks of empty slices are never written
        f[r] = live ? sent[r * 32 + lane] : 0u;
        ng[r] = live ? sign[r * 32 + lane] : 0u;
    }
    const uint64_t pos0 = reinterpret_cast<const uint64_t*>(ws + sl_excl_offset(g.num_layers))[t];
    if (lane == 0) reinterpret_cast<uint32_t*>(ws + sl_tot_offset(g.num_layers, T))[t] = 0u;  // zero for the next call
    if (st[l] != 0u) return;  // a layer whose streaming pass did not complete
    const bool wide = ly.code_bytes == 2;
    uint8_t* codes = ly.msg + 8 + 2ull * ly.nbins;
    const int cl0 = 2 * (lane & 15);  // the word's first compute lane
    const int rot = seg_rot(cl0);
    const uint32_t L = (uint32_t)ly.bin_len, inv = ly.inv_len;
    const int ts3 = (int)(ts & 3);
    uint64_t base = pos0;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const uint32_t fs = word_to_slot_order(f[r], rot);
        const uint32_t c = __popc(fs);
        uint32_t incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += y;
        }
        const uint32_t n = __shfl_sync(kFull, incl, 31);
        if (c) {
            const uint32_t sg = word_to_slot_order(ng[r], rot);
            const int w = 2 * r + (lane >> 4);  // the word's slice
            // tile element of slot 0 of the slice: from the 16-byte boundary at or before
            // its first element (warp slices: bins w * bpw ..; block slices: 512 w slots)
            int rel;
            if (kBig) {
                rel = kSlots * w - ts3;
            } else {
                const int we0 = min(nb, w * (int)ly.bpw) * (int)L;
                rel = we0 - (int)((ts + we0) & 3);
            }
            const uint32_t x0 = (uint32_t)(rel + kSeg * cl0);  // tile element of the word's bit 0 (bit 0 set: >= 0)
            uint8_t* cp = codes + (base + (incl - c)) * (wide ? 2u : 1u);
            uint32_t mm = fs, j = 0;
            while (mm) {
                const int b = __ffs(mm) - 1;
                mm &= mm - 1;
                const uint32_t x = x0 + (uint32_t)b;  // tile element, < 2^16
                const uint32_t code = ((x - __umulhi(x, inv) * L) << 1) | ((sg >> b) & 1u);
                if (wide) reinterpret_cast<uint16_t*>(cp)[j] = (uint16_t)code;
                else cp[j] = (uint8_t)code;
                ++j;
            }
        }
        base += n;
    }
}

// ---------------------------------------------------------------- materialise (deferred fix-up)
// Applies the corrections a call with a deferred fix-up left pending: for every
// slot whose bit is set in its lane's sent mask, residue = fl32(G - sign(G) s) with
// the layer's s from that call. One warp per (tile, slice); the empty slices of
// block-sliced tiles (whose masks are not written) are skipped.
template <bool kBig>
__global__ void __launch_bounds__(kEmitThreads) slice_materialize_kernel(const __grid_constant__ KGroup g,
                                                                         uint8_t* __restrict__ ws)
{
    ptx::griddep_wait();  // the kernel ahead in the stream
    constexpr int W = kBig ? kBigSlices : kWarps;  // slices per tile
    __shared__ uint32_t tb[kMaxGroup];  // first tile of each layer
    for (int e = threadIdx.x; e < g.num_layers; e += kEmitThreads) tb[e] = g.layer[e].tile_begin;
    __syncthreads();
    if (reinterpret_cast<const volatile Ctl*>(ws)->pending == 0u) return;
    const int lane = threadIdx.x & 31;
    const uint32_t T = g.total_tiles;
    const uint16_t* sent = reinterpret_cast<const uint16_t*>(ws + sl_sent_offset(g.num_layers, T));
    const uint64_t units = (uint64_t)T * W;
    const uint64_t nw = (uint64_t)gridDim.x * (kEmitThreads / 32);
    for (uint64_t u = (uint64_t)blockIdx.x * (kEmitThreads / 32) + (threadIdx.x >> 5); u < units; u += nw) {
        const uint32_t t = (uint32_t)(u / W);
        const int w = (int)(u % W);
        const int l = layer_of_tile(tb, g.num_layers, t);
        const Slice Sl = kBig ? big_slice(g.layer[l], l, t, w) : slice_in(g.layer[l], l, t, w);
        if (kBig && Sl.we1 <= Sl.we0) continue;
        const uint32_t f = to_slot_order(sent[((size_t)t * W + w) * 32 + lane], seg_rot(lane));
        if (!f) continue;
        const float s = reinterpret_cast<const LayerWs*>(ws + ws_layer_offset(l))->result.s;
        float* res = g.layer[l].residue + Sl.a0 + kSeg * lane;
#pragma unroll
        for (int i = 0; i < kSeg; ++i)
            if ((f >> i) & 1u) res[i] = __fsub_rn(res[i], copysignf(s, res[i]));
    }
}

struct SlicedDevice {
    int sms = 0;
    uint32_t smem_set[8] = {0, 0, 0, 0, 0, 0, 0, 0};  // largest dynamic shared memory opted in so far, per variant
    int emit_occ[2] = {0, 0};                         // resident CTAs per SM of the emitting kernel (warp-, block-sliced)
};
SlicedDevice g_sl_dev[64];

constexpr int kStages = 2;  // per-warp stages; with 3 CTAs per SM (74 registers) measured faster than 3 stages with 2
constexpr int kBigStages = 2;


}  // namespace

bool group_is_sliced(const KGroup& g)
{
    for (int l = 0; l < g.num_layers; ++l)
        if (!g.layer[l].bpw) return false;
    return g.num_layers > 0;
}

cudaError_t launch_compress_sliced(const KGroup& g, void* ws, cudaStream_t stream, cudaEvent_t ev_before,
                                   cudaEvent_t ev_mid, cudaEvent_t ev_after)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    SlicedDevice& di = g_sl_dev[dev];
    if (di.sms == 0) {
        e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    void (*kern)(KGroup, uint8_t*);
    uint32_t smem = 0, threads = 0;
    const int ki = (g.lazy ? 1 : 0) + (g.local_selection ? 2 : 0) + (g.big ? 4 : 0);
    if (g.big) {
        // one warp per slice of the widest tile: bins_per_tile bins (or the layer), plus
        // up to 3 alignment slots unless every tile starts on a 16-byte boundary
        int W = 1;
        for (int l = 0; l < g.num_layers; ++l) {
            const KLayer& ly = g.layer[l];
            const long long tl = (long long)ly.bins_per_tile * ly.bin_len < ly.n ? (long long)ly.bins_per_tile * ly.bin_len : ly.n;
            const long long off = (ly.num_tiles > 1 && (ly.bin_len & 3)) ? 3 : 0;
            const int w = (int)((off + tl + kSlots - 1) / kSlots);
            W = w > W ? w : W;
        }
        if (W > kBigSlices) return cudaErrorInvalidValue;
        smem = big_plan(g.d_size, kBigStages, g.num_layers, W).total;
        threads = (uint32_t)W * 32u;
        if (g.local_selection) kern = g.lazy ? block_kernel<kBigStages, true, true> : block_kernel<kBigStages, false, true>;
        else kern = g.lazy ? block_kernel<kBigStages, true, false> : block_kernel<kBigStages, false, false>;
    } else {
        smem = slice_plan(g.d_size, kStages, g.num_layers).total;
        threads = kThreads;
        if (g.local_selection) kern = g.lazy ? slice_kernel<kStages, true, true> : slice_kernel<kStages, false, true>;
        else kern = g.lazy ? slice_kernel<kStages, true, false> : slice_kernel<kStages, false, false>;
    }
    if (smem > di.smem_set[ki]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        di.smem_set[ki] = smem;
    }
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, (int)threads, smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    const long long cap = (long long)di.sms * occ;
    const uint32_t grid = (uint32_t)((long long)g.total_tiles < cap ? (long long)g.total_tiles : cap);
    if (ev_before && (e = cudaEventRecord(ev_before, stream)) != cudaSuccess) return e;
    if ((e = launch_after(kern, dim3(grid), dim3(threads), smem, stream, g, static_cast<uint8_t*>(ws))) != cudaSuccess)
        return e;
    if (ev_mid && (e = cudaEventRecord(ev_mid, stream)) != cudaSuccess) return e;
    uint32_t max_tiles = 0;  // the largest layer sets the chunks per layer
    for (int l = 0; l < g.num_layers; ++l) max_tiles = g.layer[l].num_tiles > max_tiles ? g.layer[l].num_tiles : max_tiles;
    const dim3 fgrid((max_tiles + kFinThreads - 1) / kFinThreads, (unsigned)g.num_layers);
    if ((e = launch_after(slice_finalize_kernel, fgrid, dim3(kFinThreads), 0, stream, g, static_cast<uint8_t*>(ws))) !=
        cudaSuccess)
        return e;
    if (g.lazy) {  // codes only: one warp per tile
        const uint32_t cgrid = (g.total_tiles + kEmitWarps - 1) / kEmitWarps;
        e = launch_after(g.big ? slice_codes_kernel<true> : slice_codes_kernel<false>, dim3(cgrid), dim3(kEmitThreads), 0,
                         stream, g, static_cast<uint8_t*>(ws));
        if (e != cudaSuccess) return e;
        if (ev_after) e = cudaEventRecord(ev_after, stream);
        return e;
    }
    // persistent: as many CTAs as are resident at once, each warp a run of tiles
    void (*ekern)(KGroup, uint8_t*) = g.big ? slice_emit_kernel<true> : slice_emit_kernel<false>;
    int& eocc = di.emit_occ[g.big ? 1 : 0];
    if (eocc == 0) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&eocc, ekern, kEmitThreads, 0);
        if (e != cudaSuccess) return e;
        if (eocc < 1) return cudaErrorInvalidConfiguration;
    }
    const uint32_t eneed = (g.total_tiles + kEmitWarps - 1) / kEmitWarps;
    const uint32_t ecap = (uint32_t)di.sms * (uint32_t)eocc;
    const uint32_t egrid = eneed < ecap ? eneed : ecap;
    if ((e = launch_after(ekern, dim3(egrid), dim3(kEmitThreads), 0, stream, g, static_cast<uint8_t*>(ws))) != cudaSuccess)
        return e;
    if (ev_after) e = cudaEventRecord(ev_after, stream);
    return e;
}

cudaError_t launch_materialize_sliced(const KGroup& g, void* ws, cudaStream_t stream)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    SlicedDevice& di = g_sl_dev[dev];
    if (di.sms == 0) {
        e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    const uint64_t units = (uint64_t)g.total_tiles * (g.big ? kBigSlices : kWarps);
    const uint64_t blocks_needed = (units + kEmitThreads / 32 - 1) / (kEmitThreads / 32);
    const uint64_t cap = (uint64_t)di.sms * 8;
    const uint32_t grid = (uint32_t)(blocks_needed < cap ? blocks_needed : cap);
    e = launch_after(g.big ? slice_materialize_kernel<true> : slice_materialize_kernel<false>, dim3(grid),
                     dim3(kEmitThreads), 0, stream, g, static_cast<uint8_t*>(ws));
    if (e != cudaSuccess) return e;
    // the corrections are applied: the next call must not apply them again
    return cudaMemsetAsync(static_cast<uint8_t*>(ws) + offsetof(Ctl, pending), 0, sizeof(uint32_t), stream);
}

}  // namespace adacomp
