// AdaComp compression for launch groups whose layers all have 16 <= L_T <= 509
// (every conv and FC/LSTM layer of the usual configurations): the sliced path.
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
//   slice_finalize   one CTA per layer: s from the exact sum, the header, and the
//                    exclusive prefix of the tile code totals.
//   slice_emit       persistent warps, a run of tiles each, last tiles first: the codes
//                    written at their final positions, with the sign of G read back
//                    from the residue, and the fix-up residue = fl32(G - sign(G) s) of
//                    every sent element (when the fix-up is deferred to the next call,
//                    the signs come from a second mask and the residue is not touched).
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

// Starts slice S's data into a stage (run by one lane): bulk copies of the
// 16-byte-aligned spans covering the slice, from the boundary at or before its
// first element (slot 0 of lane 0) to the one at or after its last; only at the
// end of the layer's arrays are the last few elements loaded with plain loads.
// The spans never exceed 512 slots: the slice has at most 509 elements. Returns
// false when nothing was copied (an empty slice: the phase completes at once).
__device__ bool issue_slice(const KLayer& ly, const Slice& S, float* rb, void* db, uint64_t* bar)
{
    if (S.we1 <= S.we0) {
        ptx::mbar_arrive(bar);
        return false;
    }
    const int64_t e0 = S.ts + S.we0, e1 = S.ts + S.we1;
    const int64_t a0 = S.a0;
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
        const LaneGeo q = lane_geo(Sl, ly, lane);
        const uint32_t lomask = q.split >= kSeg ? 0xffffu : ((1u << max(q.split, 0)) - 1u);  // slots of bin_lo
        // register order: chunk k of the lane is held at registers 4k..4k+3 and is
        // slot chunk k ^ rot; every per-element test below uses a compile-time bit
        const uint32_t vr = to_reg_order(q.valid, rot);
        const uint32_t lor = to_reg_order(lomask, rot) & vr;  // valid slots of bin_lo
        const uint32_t hir = vr & ~lor;                        // valid slots of bin_lo + 1
        float ah[4][4];             // |probe| per register slot
        uint32_t ngr = 0;  // G < 0 (register order; kept for the deferred fix-up's codes only)
        float m_lo = 0.0f, m_hi = 0.0f;
        if (q.valid) {
            const float* rs = stage_r(s) + kSeg * lane;
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
                    const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(stage_d(s)) + doff +
                                                                    kSeg * lane + q0);
                    d[0] = bf16_lo(u.x); d[1] = bf16_hi(u.x); d[2] = bf16_lo(u.y); d[3] = bf16_hi(u.y);
                } else {
                    const float4 v = *reinterpret_cast<const float4*>(static_cast<const float*>(stage_d(s)) + kSeg * lane + q0);
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
                    // and they are dropped from the sent mask below
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
        if (m_lo > 0.0f) atomicMax(&wg[q.bin_lo], __float_as_uint(m_lo));
        if (m_hi > 0.0f) atomicMax(&wg[q.bin_lo + 1], __float_as_uint(m_hi));
        __syncwarp();
        uint32_t fr = 0;  // sent slots, register order
        if (q.valid) {
            const float gm_lo = __uint_as_float(wg[q.bin_lo]);
            const float gm_hi = lomask != 0xffffu ? __uint_as_float(wg[q.bin_lo + 1]) : 0.0f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t bit = 1u << (4 * k + e);
                    fr |= ah[k][e] >= ((lor & bit) ? gm_lo : gm_hi) ? bit : 0u;
                }
            }
            fr &= vr;
            const uint32_t c_lo = __popc(fr & lor), c_hi = __popc(fr & ~lor);
            if (c_lo) atomicAdd(&wc[q.bin_lo], c_lo);
            if (c_hi) atomicAdd(&wc[q.bin_lo + 1], c_hi);
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
    // a warp's share: at most 32 x (tiles before the chunk / 1024) x 4072 codes < 2^32 for
    // layers below 2^38 elements
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
// 16-byte load of their sent masks (and, with the fix-up deferred, one of their sign
// masks). The masks are stored in the streaming kernel's register order and are
// brought back to slot order here. An exclusive warp scan of the lanes' popcounts
// places each lane's sent elements, in element order (which is code order), in a
// per-warp list in shared memory; the warp then walks the list with consecutive lanes
// on consecutive codes:
//   kFix: kFixBatch elements per lane at a time, all residue loads issued first (with
//         a 64-byte L2 fill size: a scattered 4-byte load otherwise fills a whole
//         128-byte line), then the code ((element - its bin's first element) << 1) |
//         (G < 0) and the residue fl32(G - sign(G) s);
//   otherwise the list entries carry the sign bit, and only the codes are written.
// A tile with more than kListCap sent elements is listed and walked in rounds. The
// tiles' code totals (read by the finalising kernel) are cleared here for the next
// call.
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

// The inputs of one tile's emission, loaded a tile ahead.
struct EmitIn {
    uint4 f;        // sent masks of the lane's eight compute lanes (register order)
    uint4 ng;       // their sign masks (deferred fix-up only)
    uint64_t pos;   // the tile's first code position in its message
};

template <bool kFix>
__device__ __forceinline__ EmitIn emit_load(const uint8_t* ws, int num_layers, uint32_t T, uint32_t t, int lane)
{
    EmitIn in;
    const uint4* sent = reinterpret_cast<const uint4*>(ws + sl_sent_offset(num_layers, T));
    in.f = sent[(size_t)t * 32 + lane];
    if (!kFix) in.ng = reinterpret_cast<const uint4*>(ws + sl_sign_offset(num_layers, T))[(size_t)t * 32 + lane];
    else in.ng = make_uint4(0u, 0u, 0u, 0u);
    in.pos = reinterpret_cast<const uint64_t*>(ws + sl_excl_offset(num_layers))[t];
    return in;
}

template <bool kFix>
__global__ void __launch_bounds__(kEmitThreads, 5) slice_emit_kernel(const __grid_constant__ KGroup g,
                                                                  uint8_t* __restrict__ ws)
{
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
    const int w = lane >> 2;         // the lane's slice
    const int cl0 = 8 * (lane & 3);  // its first compute lane
    EmitIn cur = emit_load<kFix>(ws, g.num_layers, T, T - 1u - q, lane);
    int l_cached = -1;
    float s = 0.0f;
    uint32_t status = 0;
    uint32_t* tile_tot = reinterpret_cast<uint32_t*>(ws + sl_tot_offset(g.num_layers, T));
    for (; q < T; q += NW) {
        const uint32_t t = T - 1u - q;
        const EmitIn in = cur;
        if (q + NW < T) cur = emit_load<kFix>(ws, g.num_layers, T, T - 1u - (q + NW), lane);
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
        // the lane's eight masks in slot order, and its count
        uint32_t m[8], ngm[8];
        const uint32_t fw[4] = {in.f.x, in.f.y, in.f.z, in.f.w};
        const uint32_t nw4[4] = {in.ng.x, in.ng.y, in.ng.z, in.ng.w};
        uint32_t c = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int rot = seg_rot(cl0 + i);
            m[i] = to_slot_order((fw[i >> 1] >> (16 * (i & 1))) & 0xffffu, rot);
            ngm[i] = kFix ? 0u : to_slot_order((nw4[i >> 1] >> (16 * (i & 1))) & 0xffffu, rot);
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
        const Slice Sl = slice_in(ly, l, t, w);
        const int x0 = (int)(Sl.a0 - Sl.ts) + kSeg * cl0;  // tile element of slot 0 of compute lane cl0
        float* res = ly.residue + Sl.ts;
        uint8_t* codes = ly.msg + 8 + 2ull * ly.nbins;
        for (uint32_t r0 = 0; r0 < n; r0 += kListCap) {
            // list this round's elements: positions r0 .. r0 + kListCap - 1 of the tile
            uint32_t li = incl - c;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uint32_t mm = m[i];
                while (mm) {
                    const int b = __ffs(mm) - 1;
                    mm &= mm - 1;
                    if (li - r0 < (uint32_t)kListCap)
                        lst[li - r0] = (uint16_t)((x0 + kSeg * i + b) | (((ngm[i] >> b) & 1u) << 15));
                    ++li;
                }
            }
            __syncwarp();
            const uint32_t nr = min(n - r0, (uint32_t)kListCap);
            const uint64_t pos0 = in.pos + r0;
            if constexpr (kFix) {
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
            } else {
                for (uint32_t j = lane; j < nr; j += 32) {
                    const uint32_t en = lst[j];
                    const uint32_t x = en & 0x7fffu;
                    const uint32_t off = x - __umulhi(x, ly.inv_len) * (uint32_t)ly.bin_len;
                    const uint32_t code = (off << 1) | (en >> 15);
                    if (ly.code_bytes == 1) codes[pos0 + j] = (uint8_t)code;
                    else reinterpret_cast<uint16_t*>(codes)[pos0 + j] = (uint16_t)code;
                }
            }
            __syncwarp();  // the list is rewritten by the next round or tile
        }
    }
}

// ---------------------------------------------------------------- materialise (deferred fix-up)
// Applies the corrections a call with a deferred fix-up left pending: for every
// slot whose bit is set in its lane's sent mask, residue = fl32(G - sign(G) s) with
// the layer's s from that call. One warp per (tile, slice).
__global__ void __launch_bounds__(kEmitThreads) slice_materialize_kernel(const __grid_constant__ KGroup g,
                                                                         uint8_t* __restrict__ ws)
{
    __shared__ uint32_t tb[kMaxGroup];  // first tile of each layer
    for (int e = threadIdx.x; e < g.num_layers; e += kEmitThreads) tb[e] = g.layer[e].tile_begin;
    __syncthreads();
    if (reinterpret_cast<const volatile Ctl*>(ws)->pending == 0u) return;
    const int lane = threadIdx.x & 31;
    const uint32_t T = g.total_tiles;
    const uint16_t* sent = reinterpret_cast<const uint16_t*>(ws + sl_sent_offset(g.num_layers, T));
    const uint64_t units = (uint64_t)T * kWarps;
    const uint64_t nw = (uint64_t)gridDim.x * (kEmitThreads / 32);
    for (uint64_t u = (uint64_t)blockIdx.x * (kEmitThreads / 32) + (threadIdx.x >> 5); u < units; u += nw) {
        const uint32_t t = (uint32_t)(u / kWarps);
        const int w = (int)(u % kWarps);
        const uint32_t f = to_slot_order(sent[((size_t)t * kWarps + w) * 32 + lane], seg_rot(lane));
        if (!f) continue;
        const int l = layer_of_tile(tb, g.num_layers, t);
        const Slice Sl = slice_in(g.layer[l], l, t, w);
        const float s = reinterpret_cast<const LayerWs*>(ws + ws_layer_offset(l))->result.s;
        float* res = g.layer[l].residue + Sl.a0 + kSeg * lane;
#pragma unroll
        for (int i = 0; i < kSeg; ++i)
            if ((f >> i) & 1u) res[i] = __fsub_rn(res[i], copysignf(s, res[i]));
    }
}

struct SlicedDevice {
    int sms = 0;
    uint32_t smem_set[4] = {0, 0, 0, 0};  // largest dynamic shared memory opted in so far, per variant
    int emit_occ[2] = {0, 0};             // resident CTAs per SM of the emitting kernel (deferred, eager)
};
SlicedDevice g_sl_dev[64];

constexpr int kStages = 2;  // per-warp stages; with 3 CTAs per SM (74 registers) measured faster than 3 stages with 2

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
    const SlicePlan P = slice_plan(g.d_size, kStages, g.num_layers);
    void (*kern)(KGroup, uint8_t*);
    if (g.local_selection) kern = g.lazy ? slice_kernel<kStages, true, true> : slice_kernel<kStages, false, true>;
    else kern = g.lazy ? slice_kernel<kStages, true, false> : slice_kernel<kStages, false, false>;
    const int ki = (g.lazy ? 1 : 0) + (g.local_selection ? 2 : 0);
    if (P.total > di.smem_set[ki]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P.total);
        if (e != cudaSuccess) return e;
        di.smem_set[ki] = P.total;
    }
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, P.total);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    const long long cap = (long long)di.sms * occ;
    const uint32_t grid = (uint32_t)((long long)g.total_tiles < cap ? (long long)g.total_tiles : cap);
    if (ev_before && (e = cudaEventRecord(ev_before, stream)) != cudaSuccess) return e;
    kern<<<grid, kThreads, P.total, stream>>>(g, static_cast<uint8_t*>(ws));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (ev_mid && (e = cudaEventRecord(ev_mid, stream)) != cudaSuccess) return e;
    uint32_t max_tiles = 0;  // the largest layer sets the chunks per layer
    for (int l = 0; l < g.num_layers; ++l) max_tiles = g.layer[l].num_tiles > max_tiles ? g.layer[l].num_tiles : max_tiles;
    const dim3 fgrid((max_tiles + kFinThreads - 1) / kFinThreads, (unsigned)g.num_layers);
    slice_finalize_kernel<<<fgrid, kFinThreads, 0, stream>>>(g, static_cast<uint8_t*>(ws));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // persistent: as many CTAs as are resident at once, each warp a run of tiles
    void (*ekern)(KGroup, uint8_t*) = g.lazy ? slice_emit_kernel<false> : slice_emit_kernel<true>;
    int& eocc = di.emit_occ[g.lazy ? 0 : 1];
    if (eocc == 0) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&eocc, ekern, kEmitThreads, 0);
        if (e != cudaSuccess) return e;
        if (eocc < 1) return cudaErrorInvalidConfiguration;
    }
    const uint32_t eneed = (g.total_tiles + kEmitWarps - 1) / kEmitWarps;
    const uint32_t ecap = (uint32_t)di.sms * (uint32_t)eocc;
    const uint32_t egrid = eneed < ecap ? eneed : ecap;
    ekern<<<egrid, kEmitThreads, 0, stream>>>(g, static_cast<uint8_t*>(ws));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
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
    const uint64_t units = (uint64_t)g.total_tiles * kWarps;
    const uint64_t blocks_needed = (units + kEmitThreads / 32 - 1) / (kEmitThreads / 32);
    const uint64_t cap = (uint64_t)di.sms * 8;
    const uint32_t grid = (uint32_t)(blocks_needed < cap ? blocks_needed : cap);
    slice_materialize_kernel<<<grid, kEmitThreads, 0, stream>>>(g, static_cast<uint8_t*>(ws));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // the corrections are applied: the next call must not apply them again
    return cudaMemsetAsync(static_cast<uint8_t*>(ws) + offsetof(Ctl, pending), 0, sizeof(uint32_t), stream);
}

}  // namespace adacomp
