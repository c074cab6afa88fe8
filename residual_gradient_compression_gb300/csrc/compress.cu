// AdaComp compression for sm_103a, the look-back path: launch groups whose bin
// lengths are neither all 16..509 nor all 510..8189 (those take the warp-sliced and
// block-sliced paths of compress_sliced.cu). One fused streaming
// kernel per launch group (G, H, bin maxima, selection, per-bin counts, code
// compaction with a decoupled look-back across tiles, residue := G), a finalise
// kernel (s, header) and one sparse fix-up kernel that applies
// residue -= sign(G) * s once s, the mean of the bin maxima, is known.
//
// Method: "AdaComp (Adaptive Residual Gradient Compression)", Claims > Mechanism
// #r629-local-bin-soft-threshold-and-mean-gmax-quantization (Algorithm 2 restated):
// G = residue + dW, H = G + dW, g_max(i) = max |G| over bin i, s = mean g_max, send
// |H| >= g_max(i) as sign(G) * s, residue = G - G_q (sent) or G (kept). Code widths:
// Claims > Application #r629-conv-40x-and-fc-lstm-200x-compression-across-optimizers.
//
// Data flow per tile (a whole number of bins, up to 8192 elements):
//   bulk copy (cp.async.bulk) residue + dW -> shared memory, double-buffered;
//   compute warps: G and the bin maxima, then flags, per-bin counts and codes
//            (warp-sliced tiles of a mixed group: per warp, without block barriers);
//   a look-back warp per staging buffer publishes the tile's code count, resolves its
//            exclusive prefix from predecessor tiles (Merrill & Garland's single-pass
//            scan), writes the counts and copies the staged codes into the message,
//            and adds the bin maxima, exactly, to the layer's exponent buckets.
#include "adacomp_internal.cuh"
#include "compress_common.cuh"

#include <cuda_bf16.h>

namespace adacomp {
namespace {


// Loads VEC consecutive elements at tile index i (residue slice at sr[pr + i],
// dW slice at sd[pd + i]). Vector alignment holds because every chunk starts on a
// bin boundary, L_T is a multiple of VEC and pr, pd are multiples of VEC.
template <int VEC, bool BF16>
__device__ __forceinline__ void load_rd(const float* sr, const void* sd, int ir, int id, float (&r)[VEC],
                                        float (&d)[VEC])
{
    if constexpr (VEC == 4) {
        float4 v = *reinterpret_cast<const float4*>(sr + ir);
        r[0] = v.x; r[1] = v.y; r[2] = v.z; r[3] = v.w;
        if constexpr (BF16) {
            uint2 u = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(sd) + id);
            d[0] = bf16_lo(u.x); d[1] = bf16_hi(u.x); d[2] = bf16_lo(u.y); d[3] = bf16_hi(u.y);
        } else {
            float4 w = *reinterpret_cast<const float4*>(static_cast<const float*>(sd) + id);
            d[0] = w.x; d[1] = w.y; d[2] = w.z; d[3] = w.w;
        }
    } else if constexpr (VEC == 2) {
        float2 v = *reinterpret_cast<const float2*>(sr + ir);
        r[0] = v.x; r[1] = v.y;
        if constexpr (BF16) {
            uint32_t u = *reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(sd) + id);
            d[0] = bf16_lo(u); d[1] = bf16_hi(u);
        } else {
            float2 w = *reinterpret_cast<const float2*>(static_cast<const float*>(sd) + id);
            d[0] = w.x; d[1] = w.y;
        }
    } else {
        r[0] = sr[ir];
        if constexpr (BF16) d[0] = bf16_lo(static_cast<const uint16_t*>(sd)[id]);
        else d[0] = static_cast<const float*>(sd)[id];
    }
}

template <int VEC>
__device__ __forceinline__ void store_g(float* sr, int ir, const float (&g)[VEC])
{
    if constexpr (VEC == 4) *reinterpret_cast<float4*>(sr + ir) = make_float4(g[0], g[1], g[2], g[3]);
    else if constexpr (VEC == 2) *reinterpret_cast<float2*>(sr + ir) = make_float2(g[0], g[1]);
    else sr[ir] = g[0];
}

template <int VEC>
__device__ __forceinline__ void load_g(const float* sr, int ir, float (&g)[VEC])
{
    if constexpr (VEC == 4) {
        float4 v = *reinterpret_cast<const float4*>(sr + ir);
        g[0] = v.x; g[1] = v.y; g[2] = v.z; g[3] = v.w;
    } else if constexpr (VEC == 2) {
        float2 v = *reinterpret_cast<const float2*>(sr + ir);
        g[0] = v.x; g[1] = v.y;
    } else {
        g[0] = sr[ir];
    }
}

template <int VEC, bool BF16>
__device__ __forceinline__ void load_d(const void* sd, int id, float (&d)[VEC])
{
    if constexpr (BF16) {
        const uint16_t* p = static_cast<const uint16_t*>(sd) + id;
        if constexpr (VEC == 4) {
            uint2 u = *reinterpret_cast<const uint2*>(p);
            d[0] = bf16_lo(u.x); d[1] = bf16_hi(u.x); d[2] = bf16_lo(u.y); d[3] = bf16_hi(u.y);
        } else if constexpr (VEC == 2) {
            uint32_t u = *reinterpret_cast<const uint32_t*>(p);
            d[0] = bf16_lo(u); d[1] = bf16_hi(u);
        } else {
            d[0] = bf16_lo(*p);
        }
    } else {
        float r[VEC];
        load_g<VEC>(static_cast<const float*>(sd), id, r);
#pragma unroll
        for (int k = 0; k < VEC; ++k) d[k] = r[k];
    }
}

// One tile's geometry and shared-memory slices.
struct Tile {
    float* gres;    // global residue at the element held in shared slot 0 (tile start - pr)
    const float* sr;  // residue slice; element i at sr[pr + i]
    float* gs;        // G for bins shorter than 16 (a buffer the bulk copies never target)
    const void* sd; // dW slice; element i at sd[pd + i]
    int pr, pd;
    int tl;         // elements in the tile
    int L;          // bin length
    int bins;       // bins in the tile (last bin may be partial)
    int cpb;        // chunks per bin
    int ch;         // chunk length (elements, multiple of VEC)
    uint32_t inv_len;  // ceil(2^32 / L)
    bool ls;           // Local Selection: the probe is G itself, not G + dW
};


struct ChunkRange {
    int bin, e0, e1;
};

__device__ __forceinline__ ChunkRange chunk_at(const Tile& T, int c)
{
    ChunkRange r;
    r.bin = c / T.cpb;
    int sub = c - r.bin * T.cpb;
    int bs = r.bin * T.L;
    int be = min(bs + T.L, T.tl);
    r.e0 = bs + sub * T.ch;
    r.e1 = min(r.e0 + T.ch, be);
    return r;
}

// Phase A: G = residue + dW (fp32, rounded once) replaces the residue slice; the
// largest |G| of each chunk is folded into g_max[bin] (as fp32 bits: |G| >= 0, so
// the integer order is the float order).
template <int VEC, bool BF16>
__device__ __forceinline__ void phase_a(const Tile& T, int c_begin, int c_end, uint32_t* gmax_s, int lane)
{
    for (int c = c_begin; c < c_end; ++c) {
        ChunkRange cr = chunk_at(T, c);
        if (cr.e0 >= cr.e1) continue;
        uint32_t m = 0;
        for (int v0 = cr.e0; v0 < cr.e1; v0 += 32 * VEC) {
            int i = v0 + lane * VEC;
            if (i < cr.e1) {
                float r[VEC], d[VEC], g[VEC];
                load_rd<VEC, BF16>(T.sr, T.sd, T.pr + i, T.pd + i, r, d);
#pragma unroll
                for (int k = 0; k < VEC; ++k) g[k] = __fadd_rn(r[k], d[k]);
                store_g<VEC>(T.gs, T.pr + i, g);
#pragma unroll
                for (int k = 0; k < VEC; ++k)
                    if (VEC == 1 || i + k < cr.e1) m = max(m, __float_as_uint(fabsf(g[k])));
            }
        }
        m = __reduce_max_sync(kFull, m);
        if (lane == 0) {
            if (T.cpb == 1) gmax_s[cr.bin] = m;
            else atomicMax(&gmax_s[cr.bin], m);
        }
    }
}

// Phase C: flag = G != 0 && |fl32(G + dW)| >= g_max[bin]; codes are ranked inside
// the warp with ballots and staged at stg[stg_base + rank] in element order.
// Returns the warp's code count; per-bin counts go to cnt_s.
template <int VEC, bool BF16>
__device__ __forceinline__ uint32_t phase_c(const Tile& T, int c_begin, int c_end, const uint32_t* gmax_s,
                                            uint32_t* cnt_s, uint16_t* stg, int stg_base, int lane)
{
    constexpr int kBits = VEC == 4 ? 3 : VEC == 2 ? 2 : 1;
    const uint32_t lt = lanemask_lt();
    uint32_t run = 0;
    for (int c = c_begin; c < c_end; ++c) {
        ChunkRange cr = chunk_at(T, c);
        if (cr.e0 >= cr.e1) continue;
        const float gm = __uint_as_float(gmax_s[cr.bin]);
        const int bs = cr.bin * T.L;
        uint32_t cc = 0;
        for (int v0 = cr.e0; v0 < cr.e1; v0 += 32 * VEC) {
            int i = v0 + lane * VEC;
            uint32_t f = 0;
            uint32_t code[VEC];
            if (i < cr.e1) {
                float g[VEC], d[VEC];
                load_g<VEC>(T.gs, T.pr + i, g);
                load_d<VEC, BF16>(T.sd, T.pd + i, d);
#pragma unroll
                for (int k = 0; k < VEC; ++k) {
                    float h = probe(g[k], d[k], T.ls);
                    bool sel = (VEC == 1 || i + k < cr.e1) && g[k] != 0.0f && fabsf(h) >= gm;
                    f |= (sel ? 1u : 0u) << k;
                    code[k] = (uint32_t)((i + k - bs) << 1) | (g[k] < 0.0f ? 1u : 0u);
                }
            }
            const uint32_t cl = __popc(f);
            uint32_t pre = 0, tot = 0;
#pragma unroll
            for (int b = 0; b < kBits; ++b) {
                uint32_t bal = __ballot_sync(kFull, (cl >> b) & 1u);
                pre += (uint32_t)__popc(bal & lt) << b;
                tot += (uint32_t)__popc(bal) << b;
            }
            uint32_t pos = (uint32_t)stg_base + run + pre;
#pragma unroll
            for (int k = 0; k < VEC; ++k)
                if ((f >> k) & 1u) stg[pos++] = (uint16_t)code[k];
            run += tot;
            cc += tot;
        }
        if (lane == 0) {
            if (T.cpb == 1) cnt_s[cr.bin] = cc;
            else atomicAdd(&cnt_s[cr.bin], cc);
        }
    }
    return run;
}

// ---------------------------------------------------------------- segment path (L_T >= 16)
// Each thread owns 16-element segments of the tile, aligned in shared memory:
// segment s holds slots [16 s, 16 s + 16) of the residue slice, i.e. tile elements
// e0 + idx with e0 = 16 s - pr. Since L_T >= 16 a segment spans at most two bins;
// slots idx < split belong to bin_lo, the rest to bin_lo + 1. Per segment the bin
// maxima and counts take at most two shared-memory atomics.
//
// The four 16-byte chunks of a segment are visited in the order q = k ^ rot, with
// rot = ((t >> 1) ^ (t >> 3)) & 3, which makes both the fp32 128-bit accesses
// (8 lanes per wavefront) and the bf16 64-bit accesses (16 lanes per wavefront)
// free of bank conflicts.
//
// Slots that hold no element of the tile (the alignment slots before it, the slots
// past its end) get G = 0 in phase A, so they never raise a maximum and are never
// selected; only the (rare) edge segments pay for that masking.

struct SegGeo {
    int e0;          // tile element of slot 0 (negative for the phase slots of segment 0)
    uint32_t valid;  // bit idx set when slot idx holds an element of this tile
    int bin_lo;      // bin of the first valid slot
    int split;       // first slot of bin_lo + 1 (may exceed 15)
    int off_lo;      // e0 - first element of bin_lo
};

__device__ __forceinline__ SegGeo seg_geo(const Tile& T, int s)
{
    SegGeo G;
    G.e0 = s * kSeg - T.pr;
    const int lo = max(0, -G.e0), hi = min(kSeg, T.tl - G.e0);
    G.valid = hi > lo ? (((1u << (hi - lo)) - 1u) << lo) : 0u;
    const int bin = (int)__umulhi((uint32_t)max(G.e0, 0), T.inv_len);
    G.bin_lo = bin;
    G.off_lo = G.e0 - bin * T.L;
    G.split = T.L - G.off_lo;
    return G;
}


// dW of slots 4q..4q+3 of segment s.
template <bool BF16>
__device__ __forceinline__ void seg_load_d(const Tile& T, int s, int q, float (&d)[4])
{
    if constexpr (BF16) {
        const uint16_t* p = static_cast<const uint16_t*>(T.sd) + (T.pd - T.pr) + s * kSeg + 4 * q;
        const uint2 u = *reinterpret_cast<const uint2*>(p);
        d[0] = bf16_lo(u.x); d[1] = bf16_hi(u.x); d[2] = bf16_lo(u.y); d[3] = bf16_hi(u.y);
    } else {
        const float4 v = *reinterpret_cast<const float4*>(static_cast<const float*>(T.sd) + s * kSeg + 4 * q);
        d[0] = v.x; d[1] = v.y; d[2] = v.z; d[3] = v.w;
    }
}

// Phase A, segment path: G = residue + dW over the slots, written to the residue
// in global memory; bin maxima. (Phase C forms G again from the stage, which is not
// released before it.) *mine gets the geometry of segment `tid`.
template <bool BF16>
__device__ __forceinline__ void phase_a_seg(const Tile& T, uint32_t* gmax_s, int tid, SegGeo* mine)
{
    const int nseg = (T.pr + T.tl + kSeg - 1) / kSeg;
    const int rot = seg_rot(tid);
    for (int s = tid; s < nseg; s += kThreads) {
        const SegGeo G = seg_geo(T, s);
        if (s == tid) *mine = G;
        const bool edge = G.valid != 0xffffu;
        const float* rs = T.sr + s * kSeg;
        float m_lo = 0.0f, m_hi = 0.0f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int q = k ^ rot;
            const int q0 = 4 * q;
            const float4 r = *reinterpret_cast<const float4*>(rs + q0);
            float d[4];
            seg_load_d<BF16>(T, s, q, d);
            float g[4];
            g[0] = __fadd_rn(r.x, d[0]);
            g[1] = __fadd_rn(r.y, d[1]);
            g[2] = __fadd_rn(r.z, d[2]);
            g[3] = __fadd_rn(r.w, d[3]);
            const uint32_t vq = (G.valid >> q0) & 0xfu;
            if (edge) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (!((vq >> i) & 1u)) g[i] = 0.0f;
            }
            // residue := G in global memory (sent elements are corrected by the fix-up kernel)
            float* gp = T.gres + s * kSeg + q0;
            if (vq == 0xfu) {
                *reinterpret_cast<float4*>(gp) = make_float4(g[0], g[1], g[2], g[3]);
            } else if (vq) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if ((vq >> i) & 1u) gp[i] = g[i];
            }
            if (q0 + 4 <= G.split) {
                m_lo = fmaxf(m_lo, fmaxf(fmaxf(fabsf(g[0]), fabsf(g[1])), fmaxf(fabsf(g[2]), fabsf(g[3]))));
            } else if (q0 >= G.split) {
                m_hi = fmaxf(m_hi, fmaxf(fmaxf(fabsf(g[0]), fabsf(g[1])), fmaxf(fabsf(g[2]), fabsf(g[3]))));
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (q0 + i < G.split) m_lo = fmaxf(m_lo, fabsf(g[i]));
                    else m_hi = fmaxf(m_hi, fabsf(g[i]));
                }
            }
        }
        if (m_lo > 0.0f) atomicMax(&gmax_s[G.bin_lo], __float_as_uint(m_lo));
        if (m_hi > 0.0f) atomicMax(&gmax_s[G.bin_lo + 1], __float_as_uint(m_hi));
    }
}

// Flags of one segment's 16 slots (bit idx): G != 0 && |probe| >= g_max, with G
// formed again from the stage (the same fp32 addition as in phase A); *ng_out gets
// the slots with G < 0. Slots outside the tile are never flagged.
template <bool BF16>
__device__ __forceinline__ uint32_t seg_flags(const Tile& T, const SegGeo& G, int s, int rot, float gm_lo,
                                              float gm_hi, uint32_t* ng_out)
{
    const float* rs = T.sr + s * kSeg;
    uint32_t f = 0, ng = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int q = k ^ rot;
        const int q0 = 4 * q;
        const float4 r = *reinterpret_cast<const float4*>(rs + q0);
        float d[4];
        seg_load_d<BF16>(T, s, q, d);
        const float g[4] = {__fadd_rn(r.x, d[0]), __fadd_rn(r.y, d[1]), __fadd_rn(r.z, d[2]), __fadd_rn(r.w, d[3])};
        uint32_t nib = 0, neg = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float h = probe(g[i], d[i], T.ls);
            const float gm = q0 + i < G.split ? gm_lo : gm_hi;
            nib |= (g[i] != 0.0f && fabsf(h) >= gm) ? (1u << i) : 0u;
            neg |= g[i] < 0.0f ? (1u << i) : 0u;
        }
        f |= nib << q0;
        ng |= neg << q0;
    }
    *ng_out = ng;
    return f & G.valid;
}

// Phase C, segment path: flags and codes per slot and per-bin counts. Round r of the
// 256 threads covers segments [256 r, 256 r + 256); each warp ranks its own codes of
// a round with a warp scan and stages them at stg[wbase + rank], wbase being the
// tile element of the warp's first segment in that round (a warp never has more
// codes than elements, so the runs stay disjoint), and records the run in run_src /
// run_cnt at index 8 r + warp. No barrier among the compute warps. Returns the
// number of runs (8 per round).
template <bool BF16>
__device__ __forceinline__ int phase_c_seg(const Tile& T, const uint32_t* gmax_s, uint32_t* cnt_s, uint16_t* stg,
                                           uint32_t* run_src, uint32_t* run_cnt, int tid)
{
    const int nseg = (T.pr + T.tl + kSeg - 1) / kSeg;
    const int rot = seg_rot(tid);
    const int lane = tid & 31, warp = tid >> 5;
    int r = 0;
    for (int base = 0; base < nseg; base += kThreads, ++r) {
        const int s = base + tid;
        uint32_t f = 0, ng = 0;
        SegGeo G;
        G.valid = 0; G.bin_lo = 0; G.split = kSeg; G.off_lo = 0; G.e0 = 0;
        if (s < nseg) {
            G = seg_geo(T, s);
            const float gm_lo = __uint_as_float(gmax_s[G.bin_lo]);
            const float gm_hi = G.split < kSeg ? __uint_as_float(gmax_s[G.bin_lo + 1]) : 0.0f;
            f = seg_flags<BF16>(T, G, s, rot, gm_lo, gm_hi, &ng);
            const uint32_t lomask = G.split >= kSeg ? 0xffffu : ((1u << max(G.split, 0)) - 1u);
            const uint32_t c_lo = __popc(f & lomask), c_hi = __popc(f & ~lomask);
            if (c_lo) atomicAdd(&cnt_s[G.bin_lo], c_lo);
            if (c_hi) atomicAdd(&cnt_s[G.bin_lo + 1], c_hi);
        }
        const uint32_t c = __popc(f);
        uint32_t incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += y;
        }
        const int wbase = max(kSeg * (base + 32 * warp) - T.pr, 0);
        if (lane == 31) {
            run_src[8 * r + warp] = (uint32_t)wbase;
            run_cnt[8 * r + warp] = incl;
        }
        uint32_t pos = (uint32_t)wbase + incl - c;
        while (f) {
            const int idx = __ffs(f) - 1;
            f &= f - 1;
            const int off = G.off_lo + idx - (idx < G.split ? 0 : T.L);
            stg[pos++] = (uint16_t)(((uint32_t)off << 1) | ((ng >> idx) & 1u));
        }
    }
    return 8 * r;
}

// ---------------------------------------------------------------- look-back
// Warp-cooperative exclusive prefix of tile t's code count over the tiles of its
// layer (single-pass scan with decoupled look-back, Merrill & Garland 2016). The
// tile's AGGREGATE (or, for a layer's first tile, its INCLUSIVE value) has already
// been published by the compute warps. Each round reads 128 predecessor
// descriptors (4 per lane, nearest first) and stops at the nearest INCLUSIVE one;
// then INCLUSIVE(prefix + total) is published. Every wait is bounded by timeout_ns
// of global time; on expiry (or a predecessor's error) the tile is published as
// ERROR and the function returns false.
constexpr int kLbPerLane = 4;

__device__ bool lookback_resolve(uint64_t* desc, uint32_t t, uint32_t tile_begin, uint32_t total, uint64_t ep,
                                 uint64_t timeout_ns, int lane, bool publish, uint64_t* excl_out)
{
    if (t == tile_begin) {
        *excl_out = 0;
        return true;
    }
    uint64_t excl = 0;
    int64_t j = (int64_t)t - 1;
    uint64_t start = 0;
    uint32_t sleep_ns = 32;
    bool ok = true;
    for (;;) {
        uint64_t dv[kLbPerLane];
#pragma unroll
        for (int m = 0; m < kLbPerLane; ++m) {
            const int64_t idx = j - (m * 32 + lane);
            dv[m] = idx >= (int64_t)tile_begin ? ptx::ld_relaxed(&desc[idx]) : (kFlagIncl | ep);
        }
        int mstar = kLbPerLane;
        uint32_t lim = 31;
        bool pending = false, error = false;
        uint32_t needed[kLbPerLane];
#pragma unroll
        for (int m = 0; m < kLbPerLane; ++m) {
            const uint32_t f = desc_flag(dv[m], ep);
            const uint32_t incl = __ballot_sync(kFull, f >= 2u);
            const uint32_t pend = __ballot_sync(kFull, f == 0u);
            const uint32_t err = __ballot_sync(kFull, f == 3u);
            uint32_t need = 0u;
            if (mstar == kLbPerLane) {
                if (incl) {
                    mstar = m;
                    lim = (uint32_t)(__ffs(incl) - 1);
                    need = (2u << lim) - 1u;
                } else {
                    need = kFull;
                }
            }
            needed[m] = need;
            pending |= (pend & need) != 0u;
            error |= (err & need) != 0u;
        }
        if (!pending) {
            if (error) { ok = false; break; }
            unsigned long long v = 0;
#pragma unroll
            for (int m = 0; m < kLbPerLane; ++m)
                if ((needed[m] >> lane) & 1u) v += dv[m] & kValueMask;
#pragma unroll
            for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
            excl += v;
            if (mstar < kLbPerLane) break;
            j -= 32 * kLbPerLane;
            start = 0;
            sleep_ns = 32;
            continue;
        }
        uint64_t now = 0;
        if (lane == 0) now = ptx::globaltimer();
        now = __shfl_sync(kFull, now, 0);
        if (start == 0) start = now;
        else if (now - start > timeout_ns) { ok = false; break; }
        __nanosleep(sleep_ns);
        if (sleep_ns < 256) sleep_ns <<= 1;
    }
    if (lane == 0 && publish) ptx::st_relaxed(&desc[t], ok ? (kFlagIncl | ep | (excl + total)) : (kFlagErr | ep));
    *excl_out = excl;
    return ok;
}

// ---------------------------------------------------------------- layer finalisation
// Run by one warp per layer after the compress kernel: s from the exact sum,
// header, result area; the accumulator and counters are left zeroed for the next
// call. `tmp` (256 entries) and `words` (kSumWords entries) are shared scratch;
// `words` must be zero on entry.
__device__ void finalize_layer(const KLayer& ly, LayerWs* lw, const uint64_t* desc, uint64_t ep,
                               unsigned long long* tmp, unsigned long long* words, int lane)
{
    for (int e = lane; e < 256; e += 32)
        tmp[e] = ptx::ld_relaxed(reinterpret_cast<const uint64_t*>(&lw->acc[e]));
    __syncwarp();
    const double S = exact_sum_warp(tmp, words, lane);
    if (lane == 0) {
        const float s = __double2float_rn(__ddiv_rn(S, (double)ly.nbins));
        const uint32_t err = *reinterpret_cast<volatile uint32_t*>(&lw->err);
        const uint64_t last = ptx::ld_relaxed(&desc[ly.tile_begin + ly.num_tiles - 1]);
        const bool bad = err != 0u || desc_flag(last, ep) != 2u;
        const uint64_t nnz = bad ? 0ull : (last & kValueMask);
        *reinterpret_cast<float*>(ly.msg) = s;
        *reinterpret_cast<uint32_t*>(ly.msg + 4) = ly.nbins;
        lw->result.s = s;
        lw->result.status = bad ? 6u /* ADACOMP_ERR_TIMEOUT */ : 0u;
        lw->result.nnz = nnz;
        lw->result.msg_bytes = 8ull + 2ull * ly.nbins + (unsigned long long)ly.code_bytes * nnz;
        lw->done = 0;
        lw->err = 0;
    }
    for (int e = lane; e < 256; e += 32) lw->acc[e] = 0ull;
}

// ---------------------------------------------------------------- tile geometry
struct TileGeo {
    int layer;
    int64_t ts;          // first element of the tile within its layer
    int tl;              // elements in the tile
    uint32_t first_bin;
    int bins;
};


#define ADACOMP_DISPATCH(V, BF, CALL)                                   \
    switch ((V) * 2 + (BF)) {                                           \
    case 8: { constexpr int VEC = 4; constexpr bool BF16 = false; CALL; } break; \
    case 9: { constexpr int VEC = 4; constexpr bool BF16 = true; CALL; } break;  \
    case 4: { constexpr int VEC = 2; constexpr bool BF16 = false; CALL; } break; \
    case 5: { constexpr int VEC = 2; constexpr bool BF16 = true; CALL; } break;  \
    case 2: { constexpr int VEC = 1; constexpr bool BF16 = false; CALL; } break; \
    default: { constexpr int VEC = 1; constexpr bool BF16 = true; CALL; } break; \
    }

// ---------------------------------------------------------------- compress kernel
// Persistent, cooperative (all CTAs co-resident) and warp-specialised. CTA c takes
// tiles c, c + grid, c + 2*grid, ... in order, so its next tile is known while the
// current one is processed (its bulk copies are already in flight) and the order
// holds nothing back: every tile's predecessors are processed by co-resident CTAs
// that never wait on a later tile, so the look-back cannot deadlock.
//
// Eight compute warps stream each tile; two look-back warps (one per staging
// buffer, so every other tile) publish the tile's code count, resolve its prefix
// and copy its codes into the message while the compute warps go on. Hand-off uses
// mbarriers: FULL[b] (each compute warp arrives once per tile) and EMPTY[b] (the
// look-back warp arrives when buffer b is free again), so a compute warp never
// waits for the other compute warps on the warp-sliced path.
// A stage is refilled as soon as every compute warp has taken what it needs from
// it: each warp bumps the stage's reader count, and the warp that completes it
// issues the bulk copies of the CTA's tile after next into the stage.
//
// Warp-sliced tiles (16 <= L_T <= 509): a tile is eight slices of
// bpw = floor(509 / L_T) whole bins, warp w owning slice w, so bin maxima, counts
// and code ranks are all warp-local and the compute warps never wait for one
// another inside a tile. Other bin lengths use block-wide phases (see above).
// Bin maxima are added to exponent buckets by the look-back warps (one set per
// look-back warp), which flush them to the layer's accumulator when they move to
// another layer; s is formed by the finalise kernel.
// Threads of a compress CTA with nb staging buffers (one look-back warp each).
__host__ __device__ constexpr int cta_threads(int nb) { return kThreads + 32 * nb; }
constexpr int kBarCompute = 1;
constexpr uint32_t kEndTile = 0xffffffffu;

constexpr int kMaxRuns = 24;  // code runs of a tile: 8 warps x at most 3 rounds of 256 segments
struct Slot {
    uint32_t t, layer, first_bin, bins;
    uint32_t nrun, pad0, pad1, pad2;
    uint32_t src[kMaxRuns], cnt[kMaxRuns];  // code runs: staging offset and length, in message order
};

// Shared-memory control block of the compress kernel.
struct Ctrl {
    uint64_t stage_full[2];   // bulk copies of the tile in each stage have landed
    uint64_t buf_full[kMaxBuffers];   // compute warps -> look-back warp of buffer b (count kWarps)
    uint64_t buf_empty[kMaxBuffers];  // look-back warp of buffer b -> compute warps (count 1)
    uint32_t users[2];        // compute warps done reading each stage
    uint32_t issued[2];       // tiles issued into each stage
    int32_t issue_layer;      // layer of the last tile issued
    uint32_t poisoned;        // a wait ran out: later tiles publish errors only
    uint64_t ep;              // this call's epoch, in descriptor position
    uint32_t wsum[kWarps];    // block scan scratch
    Slot slot[kMaxBuffers];
};
static_assert(sizeof(Ctrl) <= 1152, "control block exceeds its shared-memory allowance");

template <int ID, int N>
__device__ __forceinline__ void bar_sync() { asm volatile("bar.sync %0, %1;" ::"n"(ID), "n"(N) : "memory"); }
__device__ __forceinline__ void compute_sync() { bar_sync<kBarCompute, kThreads>(); }

// Bounded wait on an mbarrier phase; skipped (reported as failed) once the CTA is
// poisoned, so that a lost copy or hand-off costs at most one timeout per CTA.
// Between checks of the time limit the thread sleeps in the barrier (woken when
// the phase completes) instead of spinning: spinning warps take issue slots from
// the compute warps.
constexpr uint32_t kWaitHintNs = 20000;
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, uint64_t timeout_ns, uint32_t* poisoned)
{
    if (*reinterpret_cast<volatile uint32_t*>(poisoned)) return false;
    uint64_t start = 0;
    while (!ptx::mbar_try_wait_sleep(bar, parity, kWaitHintNs)) {
        const uint64_t now = ptx::globaltimer();
        if (start == 0) start = now;
        else if (now - start > timeout_ns) {
            *reinterpret_cast<volatile uint32_t*>(poisoned) = 1u;
            return false;
        }
    }
    return true;
}

// Starts tile t's data into a stage: bulk copies of the 16-byte-aligned spans that
// cover its residue and dW slices (plain loads for the few elements past the last
// 16-byte boundary of a layer's array), and the tile's geometry for the threads
// that will process it.
__device__ void issue_tile(const KLayer* lays, uint32_t t, int layer, float* sr, void* sd, uint64_t* bar,
                           TileGeo* info)
{
    TileGeo G;
    G.layer = layer;
    const KLayer& ly = lays[layer];
    G.first_bin = (t - ly.tile_begin) * ly.bins_per_tile;
    G.bins = (int)min(ly.bins_per_tile, ly.nbins - G.first_bin);
    G.ts = (int64_t)G.first_bin * ly.bin_len;
    G.tl = (int)min((int64_t)G.bins * ly.bin_len, ly.n - G.ts);
    *info = G;
    const int64_t te = G.ts + G.tl;
    // The copies start at the 16-byte boundary at or before the tile and end at the
    // one at or after it (reading into the next tile, whose elements are ignored);
    // only at the end of the layer's array do they stop at the boundary before it.
    const int64_t a0 = G.ts & ~(int64_t)3;
    int64_t a1 = (te + 3) & ~(int64_t)3;
    if (a1 > ly.n) a1 = te & ~(int64_t)3;
    const uint32_t rb = a1 > a0 ? (uint32_t)(a1 - a0) * 4u : 0u;
    int64_t b0 = a0, b1 = a1;
    uint32_t db = rb;
    if (ly.dw_bf16) {
        b0 = G.ts & ~(int64_t)7;
        b1 = (te + 7) & ~(int64_t)7;
        if (b1 > ly.n) b1 = te & ~(int64_t)7;
        db = b1 > b0 ? (uint32_t)(b1 - b0) * 2u : 0u;
    }
    const int pr = (int)(G.ts - a0), pd = (int)(G.ts - b0);
    if (a1 < te || b1 < te) {
        for (int64_t j = max(a1, G.ts); j < te; ++j) sr[pr + (j - G.ts)] = ly.residue[j];
        if (ly.dw_bf16) {
            for (int64_t j = max(b1, G.ts); j < te; ++j)
                static_cast<uint16_t*>(sd)[pd + (j - G.ts)] = static_cast<const uint16_t*>(ly.dw)[j];
        } else {
            for (int64_t j = max(b1, G.ts); j < te; ++j)
                static_cast<float*>(sd)[pd + (j - G.ts)] = static_cast<const float*>(ly.dw)[j];
        }
        ptx::fence_proxy_async_smem();  // before later bulk copies refill these bytes
    }
    ptx::mbar_arrive_expect_tx(bar, rb + db);
    if (rb) ptx::bulk_g2s(sr, ly.residue + a0, rb, bar);
    if (db) ptx::bulk_g2s(sd, static_cast<const uint8_t*>(ly.dw) + b0 * (ly.dw_bf16 ? 2 : 4), db, bar);
}

// Look-back warp that owns staging buffer b of nb, i.e. every nb-th tile of the CTA.
// For each such tile, in order: it sums the code runs, publishes the tile's
// AGGREGATE (INCLUSIVE for a layer's first tile), writes the per-bin counts into
// the message, adds the bin maxima to its exponent buckets and clears the bin
// arrays; then it resolves the tile's prefix with the look-back and copies the
// staged codes into the message.
struct LookbackCtx {
    uint16_t* stg;
    uint32_t* gmax;
    uint32_t* cnt;
    uint32_t bin_len;  // entries of gmax / cnt to clear
    unsigned long long* hist;  // this warp's exponent buckets
};

__device__ void lookback_warp(const KGroup& g, const KLayer* lays, uint8_t* ws, Ctrl* ctl, const LookbackCtx& C,
                              int b, int nb, int lane)
{
    uint64_t* desc = reinterpret_cast<uint64_t*>(ws + ws_desc_offset(g.num_layers));
    uint64_t* texcl = desc + g.total_tiles;
    int hist_layer = -1;
    for (uint32_t j = 0;; ++j) {
        const bool got = wait_phase(&ctl->buf_full[b], j & 1u, g.timeout_ns, &ctl->poisoned);
        const Slot& sl = ctl->slot[b];
        const uint32_t t = sl.t;
        if (t == kEndTile) break;
        if (!got || *reinterpret_cast<volatile uint32_t*>(&ctl->poisoned)) {
            // The CTA is poisoned: the tile's data or hand-off may be incomplete, so
            // only an error is published, for this tile and every later one of the
            // CTA's (the compute warps keep handing them over, or stop).
            if (!got) {
                const uint32_t T = g.total_tiles;
                int l = 0;
                for (uint32_t u = (uint32_t)blockIdx.x + (nb * j + b) * gridDim.x; u < T; u += nb * gridDim.x) {
                    l = layer_from(lays, g.num_layers, u, l);
                    if (lane == 0) {
                        ptx::st_relaxed(&desc[u], kFlagErr | ctl->ep);
                        atomicOr(&reinterpret_cast<LayerWs*>(ws + ws_layer_offset(l))->err, kErrTimeout);
                    }
                }
                break;
            }
            const int l = layer_from(lays, g.num_layers, t, 0);
            if (lane == 0) {
                ptx::st_relaxed(&desc[t], kFlagErr | ctl->ep);
                atomicOr(&reinterpret_cast<LayerWs*>(ws + ws_layer_offset(l))->err, kErrTimeout);
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&ctl->buf_empty[b]);
            continue;
        }
        const int l = (int)sl.layer;
        const KLayer& ly = lays[l];
        const int bins = (int)sl.bins;
        // code runs: exclusive offsets and the tile's total
        const uint32_t nrun = sl.nrun;
        const uint32_t v = lane < (int)nrun ? sl.cnt[lane] : 0u;
        uint32_t incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += y;
        }
        const uint32_t total = __shfl_sync(kFull, incl, 31);
        const uint32_t my_dst = incl - v;
        const uint32_t my_src = lane < (int)nrun ? sl.src[lane] : 0u;
        if (lane == 0 && t != g.inject_skip_tile)
            ptx::st_relaxed(&desc[t], (t == ly.tile_begin ? kFlagIncl : kFlagAgg) | ctl->ep | total);
        uint16_t* cdst = reinterpret_cast<uint16_t*>(ly.msg + 8) + sl.first_bin;
        for (int bb = lane; bb < bins; bb += 32) cdst[bb] = (uint16_t)C.cnt[bb];
        // the tile's bin maxima into the exponent buckets (flushed when the layer changes)
        LayerWs* lw = reinterpret_cast<LayerWs*>(ws + ws_layer_offset(l));
        if (l != hist_layer) {
            if (hist_layer >= 0)
                flush_buckets(C.hist, reinterpret_cast<LayerWs*>(ws + ws_layer_offset(hist_layer)), lane);
            hist_layer = l;
        }
        for (int b0 = 0; b0 < bins; b0 += 32) bucket_group(b0 + lane < bins ? C.gmax[b0 + lane] : 0u, C.hist, lw->acc, lane);
        __syncwarp();
        for (uint32_t bb = lane; bb < C.bin_len; bb += 32) { C.gmax[bb] = 0u; C.cnt[bb] = 0u; }
        uint64_t excl = 0;
        const bool ok = lookback_resolve(desc, t, ly.tile_begin, total, ctl->ep, g.timeout_ns, lane,
                                         t != g.inject_skip_tile, &excl);
        if (ok) {
            if (lane == 0) texcl[t] = excl;
            uint8_t* codes = ly.msg + 8 + 2ull * ly.nbins;
            for (uint32_t r = 0; r < nrun; ++r) {
                const uint32_t n = __shfl_sync(kFull, v, r);
                const unsigned long long base = excl + __shfl_sync(kFull, my_dst, r);
                const uint16_t* sp = C.stg + __shfl_sync(kFull, my_src, r);
                if (ly.code_bytes == 1) {
                    for (uint32_t k = lane; k < n; k += 32) codes[base + k] = (uint8_t)sp[k];
                } else {
                    uint16_t* c16 = reinterpret_cast<uint16_t*>(codes);
                    for (uint32_t k = lane; k < n; k += 32) c16[base + k] = sp[k];
                }
            }
        } else if (lane == 0) {
            atomicOr(&reinterpret_cast<LayerWs*>(ws + ws_layer_offset(l))->err, kErrTimeout);
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&ctl->buf_empty[b]);
    }
    if (hist_layer >= 0) flush_buckets(C.hist, reinterpret_cast<LayerWs*>(ws + ws_layer_offset(hist_layer)), lane);
}

// Warp-sliced tile: warp `warp` owns bins [wb0, wb1) of the tile, at most 509
// elements, held as up to 512 slots of 16 per lane (slot 0 of the warp is the
// 16-byte boundary at or before its first element). Per lane: G = residue + dW,
// residue := G in global memory, and |H| = |fl32(G + dW)| with the masks of G != 0
// and G < 0 kept in registers; `release` then gives the stage back. Bin maxima and
// counts go through the warp's scratch (wg, wc: zero on entry and on return) into
// the tile's maximum and count arrays, and the codes, ranked with a warp scan, to
// stg[we0 + rank], we0 being the warp's first tile element. Returns the warp's
// code count; *src gets we0.
template <bool BF16, class Release>
__device__ __forceinline__ uint32_t warp_tile(const KLayer& ly, const TileGeo& G, int pr, int pd, const float* sr,
                                              const void* sd, uint32_t* wg, uint32_t* wc, uint32_t* cnt_tile,
                                              uint16_t* stg, uint32_t* gmax_tile, int warp, int lane,
                                              uint16_t* pend, float s_prev, bool ls, uint32_t* src,
                                              Release&& release)
{
    const int L = ly.bin_len;
    const int bpw = ly.bpw;
    const int wb0 = min(G.bins, warp * bpw), wb1 = min(G.bins, wb0 + bpw);
    const int we0 = wb0 * L, we1 = min(wb1 * L, G.tl);
    const int e_first = (((pr + we0) & ~3) - pr) + kSeg * lane;  // tile element of the lane's slot 0
    const bool active = we1 > we0 && e_first + kSeg > we0 && e_first < we1;
    const int vlo = max(0, we0 - e_first), vhi = min(kSeg, we1 - e_first);
    const uint32_t valid = (active && vhi > vlo) ? (((1u << (vhi - vlo)) - 1u) << vlo) : 0u;
    const int rel0 = max(e_first, we0) - we0;
    const int bin_lo = active ? (int)__umulhi((uint32_t)rel0, ly.inv_len) : 0;  // warp-relative bin
    const int split = (bin_lo + 1) * L - (e_first - we0);  // first slot of bin_lo + 1
    const uint32_t lomask = split >= kSeg ? 0xffffu : ((1u << max(split, 0)) - 1u);  // slots of bin_lo
    const int rot = seg_rot(lane);
    // Register order: chunk k of the lane (4 slots) is held at registers 4k..4k+3 and
    // is slot chunk k ^ rot, so bit 4k + i of a register-order mask is slot
    // 4 (k ^ rot) + i. Every per-element test below uses a compile-time bit.
    uint32_t vr = 0, lor = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int q0 = 4 * (k ^ rot);
        vr |= ((valid >> q0) & 0xfu) << (4 * k);
        lor |= ((lomask >> q0) & 0xfu) << (4 * k);
    }
    lor &= vr;
    float ah[4][4];            // |probe| per register slot
    uint32_t nzr = 0, ngr = 0;  // G != 0, G < 0 (register order)
    float m_lo = 0.0f, m_hi = 0.0f;
    // deferred fix-up of the previous call: the residue of the slots it sent still
    // holds G; the correction fl32(G - sign(G) s_prev) is applied as they are loaded
    const uint32_t pm = pend ? (uint32_t)*pend : 0u;
    if (active) {
        const float* rs = sr + pr + e_first;
        float* gres = ly.residue + G.ts + e_first;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int q0 = 4 * (k ^ rot);
            float4 r = *reinterpret_cast<const float4*>(rs + q0);
            if (pm & (0xfu << (4 * k))) {
                if (pm & (1u << (4 * k + 0))) r.x = __fsub_rn(r.x, copysignf(s_prev, r.x));
                if (pm & (1u << (4 * k + 1))) r.y = __fsub_rn(r.y, copysignf(s_prev, r.y));
                if (pm & (1u << (4 * k + 2))) r.z = __fsub_rn(r.z, copysignf(s_prev, r.z));
                if (pm & (1u << (4 * k + 3))) r.w = __fsub_rn(r.w, copysignf(s_prev, r.w));
            }
            float d[4], gv[4];
            if constexpr (BF16) {
                const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(sd) + pd + e_first + q0);
                d[0] = bf16_lo(u.x); d[1] = bf16_hi(u.x); d[2] = bf16_lo(u.y); d[3] = bf16_hi(u.y);
            } else {
                const float4 w = *reinterpret_cast<const float4*>(static_cast<const float*>(sd) + pd + e_first + q0);
                d[0] = w.x; d[1] = w.y; d[2] = w.z; d[3] = w.w;
            }
            gv[0] = __fadd_rn(r.x, d[0]);
            gv[1] = __fadd_rn(r.y, d[1]);
            gv[2] = __fadd_rn(r.z, d[2]);
            gv[3] = __fadd_rn(r.w, d[3]);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t bit = 1u << (4 * k + i);
                if (!(vr & bit)) gv[i] = 0.0f;  // a slot outside the warp's bins
                ah[k][i] = fabsf(probe(gv[i], d[i], ls));
                nzr |= gv[i] != 0.0f ? bit : 0u;
                ngr |= gv[i] < 0.0f ? bit : 0u;
                const float a = fabsf(gv[i]);
                const bool lo = (lor & bit) != 0u;
                m_lo = fmaxf(m_lo, lo ? a : 0.0f);
                m_hi = fmaxf(m_hi, lo ? 0.0f : a);
            }
            // residue := G (sent elements are corrected by the fix-up kernel, or by the
            // next call when the fix-up is deferred)
            const uint32_t vq = (vr >> (4 * k)) & 0xfu;
            float* gp = gres + q0;
            if (vq == 0xfu) {
                *reinterpret_cast<float4*>(gp) = make_float4(gv[0], gv[1], gv[2], gv[3]);
            } else if (vq) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if ((vq >> i) & 1u) gp[i] = gv[i];
            }
        }
    }
    __syncwarp();
    release();  // the stage is not read again by this warp
    if (m_lo > 0.0f) atomicMax(&wg[bin_lo], __float_as_uint(m_lo));
    if (m_hi > 0.0f) atomicMax(&wg[bin_lo + 1], __float_as_uint(m_hi));
    __syncwarp();
    uint32_t fr = 0;  // sent slots, register order
    if (active) {
        const float gm_lo = __uint_as_float(wg[bin_lo]);
        const float gm_hi = lomask != 0xffffu ? __uint_as_float(wg[bin_lo + 1]) : 0.0f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t bit = 1u << (4 * k + i);
                fr |= ah[k][i] >= ((lor & bit) ? gm_lo : gm_hi) ? bit : 0u;
            }
        }
        fr &= nzr;
        const uint32_t c_lo = __popc(fr & lor), c_hi = __popc(fr & ~lor);
        if (c_lo) atomicAdd(&wc[bin_lo], c_lo);
        if (c_hi) atomicAdd(&wc[bin_lo + 1], c_hi);
    }
    __syncwarp();
    {
        // per bin of the slice: count and maximum to the tile's arrays; scratch back to zero
        const int nb = wb1 - wb0;
        if (lane < nb) {
            cnt_tile[wb0 + lane] = wc[lane];
            gmax_tile[wb0 + lane] = wg[lane];
        }
        wg[lane] = 0u;
        wc[lane] = 0u;
    }
    // codes are emitted in slot order: bring the sent and sign masks back to it
    uint32_t f = 0, ng = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int q0 = 4 * (k ^ rot);
        f |= ((fr >> (4 * k)) & 0xfu) << q0;
        ng |= ((ngr >> (4 * k)) & 0xfu) << q0;
    }
    const uint32_t c = __popc(f);
    uint32_t incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
    }
    const uint32_t total = __shfl_sync(kFull, incl, 31);
    // code of slot idx: ((slot's offset in its bin) << 1) | sign, i.e. base + 2 idx | sign
    const uint32_t base_lo = (uint32_t)((e_first - we0) - bin_lo * L) << 1;
    const uint32_t base_hi = base_lo - 2u * (uint32_t)L;
    uint16_t* sp = stg + we0 + incl - c;
    while (f) {
        const int idx = __ffs(f) - 1;
        f &= f - 1;
        *sp++ = (uint16_t)((idx < split ? base_lo : base_hi) + 2u * idx + ((ng >> idx) & 1u));
    }
    if (pend) *pend = (uint16_t)fr;  // corrections this call leaves to the next one
    *src = (uint32_t)we0;
    return total;
}

// One-round segment tile held in registers (at most 256 segments, one per thread):
// phase A computes G, residue := G, the bin maxima and, per slot, |H| = |fl32(G + dW)|
// and the masks of G != 0 and G < 0 (all phase C needs); after a barrier the stage
// is no longer read and is released; phase C then runs from the registers (flags,
// per-bin counts, codes ranked per warp and staged at stg[wbase + rank]). Returns
// the warp's code count.
template <bool BF16, class Release>
__device__ __forceinline__ uint32_t tile_in_registers(const Tile& T, uint32_t* gmax_s, uint32_t* cnt_s,
                                                      uint16_t* stg, int tid, int* wbase_out, Release&& release)
{
    const int nseg = (T.pr + T.tl + kSeg - 1) / kSeg;
    const int lane = tid & 31, warp = tid >> 5;
    const int s = tid;
    const int rot = seg_rot(tid);
    const bool active = s < nseg;
    SegGeo G;
    G.valid = 0; G.bin_lo = 0; G.split = kSeg; G.off_lo = 0; G.e0 = 0;
    float ah[4][4];          // |H| per slot
    uint32_t nz = 0, ng = 0;  // G != 0, G < 0 per slot
    if (active) {
        G = seg_geo(T, s);
        const bool edge = G.valid != 0xffffu;
        const float* rs = T.sr + s * kSeg;
        float m_lo = 0.0f, m_hi = 0.0f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int q0 = 4 * (k ^ rot);
            const float4 r = *reinterpret_cast<const float4*>(rs + q0);
            float d[4], g[4];
            seg_load_d<BF16>(T, s, q0 >> 2, d);
            g[0] = __fadd_rn(r.x, d[0]);
            g[1] = __fadd_rn(r.y, d[1]);
            g[2] = __fadd_rn(r.z, d[2]);
            g[3] = __fadd_rn(r.w, d[3]);
            const uint32_t vq = (G.valid >> q0) & 0xfu;
            if (edge) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (!((vq >> i) & 1u)) g[i] = 0.0f;
            }
            uint32_t nzq = 0, ngq = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                ah[k][i] = fabsf(probe(g[i], d[i], T.ls));
                nzq |= g[i] != 0.0f ? (1u << i) : 0u;
                ngq |= g[i] < 0.0f ? (1u << i) : 0u;
            }
            nz |= nzq << q0;
            ng |= ngq << q0;
            // residue := G in global memory (sent elements are corrected by the fix-up kernel)
            float* gp = T.gres + s * kSeg + q0;
            if (vq == 0xfu) {
                *reinterpret_cast<float4*>(gp) = make_float4(g[0], g[1], g[2], g[3]);
            } else if (vq) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if ((vq >> i) & 1u) gp[i] = g[i];
            }
            const float cm = fmaxf(fmaxf(fabsf(g[0]), fabsf(g[1])), fmaxf(fabsf(g[2]), fabsf(g[3])));
            if (q0 + 4 <= G.split) {
                m_lo = fmaxf(m_lo, cm);
            } else if (q0 >= G.split) {
                m_hi = fmaxf(m_hi, cm);
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (q0 + i < G.split) m_lo = fmaxf(m_lo, fabsf(g[i]));
                    else m_hi = fmaxf(m_hi, fabsf(g[i]));
                }
            }
        }
        if (m_lo > 0.0f) atomicMax(&gmax_s[G.bin_lo], __float_as_uint(m_lo));
        if (m_hi > 0.0f) atomicMax(&gmax_s[G.bin_lo + 1], __float_as_uint(m_hi));
    }
    compute_sync();  // all bin maxima are in; the stage is not read again
    release();
    uint32_t f = 0;
    if (active) {
        const float gm_lo = __uint_as_float(gmax_s[G.bin_lo]);
        const float gm_hi = G.split < kSeg ? __uint_as_float(gmax_s[G.bin_lo + 1]) : 0.0f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int q0 = 4 * (k ^ rot);
            uint32_t nib = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                nib |= ah[k][i] >= (q0 + i < G.split ? gm_lo : gm_hi) ? (1u << i) : 0u;
            f |= nib << q0;
        }
        f &= nz;
        const uint32_t lomask = G.split >= kSeg ? 0xffffu : ((1u << max(G.split, 0)) - 1u);
        const uint32_t c_lo = __popc(f & lomask), c_hi = __popc(f & ~lomask);
        if (c_lo) atomicAdd(&cnt_s[G.bin_lo], c_lo);
        if (c_hi) atomicAdd(&cnt_s[G.bin_lo + 1], c_hi);
    }
    const uint32_t c = __popc(f);
    uint32_t incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
    }
    const uint32_t total = __shfl_sync(kFull, incl, 31);
    const int wbase = max(kSeg * 32 * warp - T.pr, 0);
    uint32_t pos = (uint32_t)wbase + incl - c;
    while (f) {
        const int idx = __ffs(f) - 1;
        f &= f - 1;
        const int off = G.off_lo + idx - (idx < G.split ? 0 : T.L);
        stg[pos++] = (uint16_t)(((uint32_t)off << 1) | ((ng >> idx) & 1u));
    }
    *wbase_out = wbase;
    return total;
}

// Block-wide tile (bin lengths outside the warp-sliced range): phases A and C
// with barriers among the compute warps, kept out of line so that the
// warp-sliced path's register allocation does not pay for it.
template <class Release>
__device__ __noinline__ void block_tile(const KLayer& ly, const TileGeo G, int pr, int pd, float* sr_s, void* sd_s,
                                        float* gbuf, uint32_t* gmax_c, uint32_t* cnt_c, uint16_t* stg, Slot& sl,
                                        uint32_t* wsum, bool ls, int tid, Release* release_p)
{
    Release& release = *release_p;
    const int lane = tid & 31, warp = tid >> 5;
    const int64_t te = G.ts + G.tl;
    Tile Tl;
    Tl.gres = ly.residue + (G.ts - pr);
    Tl.sr = sr_s; Tl.gs = gbuf; Tl.sd = sd_s; Tl.pr = pr; Tl.pd = pd; Tl.tl = G.tl; Tl.L = ly.bin_len;
    Tl.bins = G.bins;
    Tl.ch = min(ly.bin_len, 32 * (int)ly.vec * kRounds);
    Tl.cpb = (ly.bin_len + Tl.ch - 1) / Tl.ch;
    Tl.inv_len = ly.inv_len;
    Tl.ls = ls;
    const bool seg = ly.bin_len >= kSeg;
    const bool one_round = seg && pr + G.tl <= kThreads * kSeg;
    const int nchunks = G.bins * Tl.cpb;
    const int cpw = (nchunks + kWarps - 1) / kWarps;
    const int c_begin = min(nchunks, warp * cpw), c_end = min(nchunks, c_begin + cpw);
    compute_sync();  // every compute warp is past its waits for this tile
    if (one_round) {
        // phases A and C with G and dW in registers; the stage is released in between
        int wb = 0;
        uint32_t wt;
        if (ly.dw_bf16) wt = tile_in_registers<true>(Tl, gmax_c, cnt_c, stg, tid, &wb, release);
        else wt = tile_in_registers<false>(Tl, gmax_c, cnt_c, stg, tid, &wb, release);
        if (lane == 0) {
            sl.src[warp] = (uint32_t)wb;
            sl.cnt[warp] = wt;
            if (warp == 0) sl.nrun = kWarps;
        }
    } else {
        // phase A: G (to the G buffer and global memory) and bin maxima
        SegGeo mine;
        if (seg) {
            if (ly.dw_bf16) phase_a_seg<true>(Tl, gmax_c, tid, &mine);
            else phase_a_seg<false>(Tl, gmax_c, tid, &mine);
        } else {
            ADACOMP_DISPATCH(ly.vec, ly.dw_bf16, (phase_a<VEC, BF16>(Tl, c_begin, c_end, gmax_c, lane)))
        }
        compute_sync();
        if (!seg) {  // short bins: residue := G from the G buffer, then phase C per warp
            for (int64_t j = G.ts + tid; j < te; j += kThreads) ly.residue[j] = gbuf[pr + (j - G.ts)];
            const int wb = c_begin < c_end ? chunk_at(Tl, c_begin).e0 : 0;
            uint32_t wt = 0;
            ADACOMP_DISPATCH(ly.vec, ly.dw_bf16,
                             (wt = phase_c<VEC, BF16>(Tl, c_begin, c_end, gmax_c, cnt_c, stg, wb, lane)))
            if (lane == 0) {
                sl.src[warp] = (uint32_t)wb;
                sl.cnt[warp] = wt;
                if (warp == 0) sl.nrun = kWarps;
            }
        } else {  // several rounds: one code run per warp and round
            int nrun;
            if (ly.dw_bf16) nrun = phase_c_seg<true>(Tl, gmax_c, cnt_c, stg, sl.src, sl.cnt, tid);
            else nrun = phase_c_seg<false>(Tl, gmax_c, cnt_c, stg, sl.src, sl.cnt, tid);
            if (tid == 0) sl.nrun = (uint32_t)nrun;
        }
        compute_sync();  // phase C was the last reader of the stage
        release();
    }
}

// kPaths: 1 = every layer of the launch is warp-sliced, 2 = none is, 3 = mixed.
// The single-path instantiations keep the warp-sliced path's registers free of
// the block-wide path's needs.
// kLazy: warp-sliced layers apply the previous call's deferred corrections and
// record their own instead of leaving them to the fix-up kernel.
template <int kPaths, int kNB, bool kLazy>
__global__ void __launch_bounds__(cta_threads(kNB), 2) compress_kernel(const __grid_constant__ KGroup g,
                                                                  uint8_t* __restrict__ ws)
{
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int kCtaThreads = cta_threads(kNB);
    const SmemPlan P = smem_plan(g.tile_cap, g.d_size, g.max_bins, g.num_layers, g.needs_gbuf, kNB);
    // stage s: residue slice at smem + s * stage_bytes, dW slice r_bytes after it
    const uint32_t stage_bytes = P.r_bytes + P.d_bytes;
    auto stage_r = [&](int s) { return reinterpret_cast<float*>(smem + s * stage_bytes); };
    auto stage_d = [&](int s) { return static_cast<void*>(smem + s * stage_bytes + P.r_bytes); };
    uint8_t* p = smem + 2 * stage_bytes;
    KLayer* lays = reinterpret_cast<KLayer*>(p); p += P.layer_bytes;
    float* gbuf = reinterpret_cast<float*>(p); p += P.g_bytes;  // G, for tiles processed through shared memory
    uint16_t* stg0 = reinterpret_cast<uint16_t*>(p); p += kNB * P.stg_bytes;
    const uint32_t stg_stride = P.stg_bytes / 2;
    uint32_t* gmax_s = reinterpret_cast<uint32_t*>(p); p += P.bin_bytes;  // kNB buffers of bin_stride
    uint32_t* cnt_s = reinterpret_cast<uint32_t*>(p); p += P.bin_bytes;   // kNB buffers of bin_stride
    const uint32_t bin_stride = P.bin_stride;
    unsigned long long* hist0 = reinterpret_cast<unsigned long long*>(p); p += kNB * kHistBytesPerBuffer;  // [buffer][kHistN] buckets
    uint32_t* wscr0 = reinterpret_cast<uint32_t*>(p); p += kWarpScratchBytes;  // [warp][2][kWarpScratch]
    TileGeo* info = reinterpret_cast<TileGeo*>(p); p += 2048;  // [2]: geometry of the tile in each stage
    Ctrl* ctl = reinterpret_cast<Ctrl*>(p);

    const uint32_t T = g.total_tiles;
    const uint32_t G0 = blockIdx.x, GS = gridDim.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    for (int e = tid; e < kNB * kHistN; e += kCtaThreads) hist0[e] = 0ull;
    for (int e = tid; e < kWarpScratchBytes / 4; e += kCtaThreads) wscr0[e] = 0u;
    {
        const uint4* src = reinterpret_cast<const uint4*>(&g.layer[0]);
        uint4* dst = reinterpret_cast<uint4*>(lays);
        for (int e = tid; e < g.num_layers * (int)(sizeof(KLayer) / 16); e += kCtaThreads) dst[e] = src[e];
    }
    __syncthreads();
    for (uint32_t e = tid; e < kNB * bin_stride; e += kCtaThreads) { gmax_s[e] = 0u; cnt_s[e] = 0u; }
    if (tid == 0) {
        ctl->users[0] = ctl->users[1] = 0u;
        ctl->issued[0] = ctl->issued[1] = 0u;
        ctl->poisoned = 0u;
        ctl->ep = call_epoch(*reinterpret_cast<volatile const uint32_t*>(&reinterpret_cast<const Ctl*>(ws)->epoch));
        for (int k = 0; k < 2; ++k) ptx::mbar_init(&ctl->stage_full[k], 1);
        for (int k = 0; k < kNB; ++k) {
            ptx::mbar_init(&ctl->buf_full[k], kWarps);
            ptx::mbar_init(&ctl->buf_empty[k], 1);
        }
        ptx::fence_mbar_init();
        int il = 0;
        for (int k = 0; k < 2; ++k) {
            const uint32_t t = G0 + k * GS;
            if (t < T) {
                il = layer_from(lays, g.num_layers, t, il);
                issue_tile(lays, t, il, stage_r(k), stage_d(k), &ctl->stage_full[k], &info[k]);
                ctl->issued[k] = 1u;
            }
        }
        ctl->issue_layer = il;
    }
    __syncthreads();

    uint32_t it = 0;
    if (warp >= kWarps) {
        const int b = warp - kWarps;  // look-back warp of staging buffer b
        LookbackCtx C;
        C.stg = stg0 + b * stg_stride;
        C.gmax = gmax_s + b * bin_stride;
        C.cnt = cnt_s + b * bin_stride;
        C.bin_len = bin_stride;
        C.hist = hist0 + b * kHistN;
        lookback_warp(g, lays, ws, ctl, C, b, kNB, lane);
    } else {
        uint32_t* wg = wscr0 + warp * 2 * kWarpScratch;
        uint32_t* wc = wg + kWarpScratch;
        for (;; ++it) {
            const uint32_t t = G0 + it * GS;
            if (t >= T) break;
            const int s = it & 1;                         // stage
            const int bf = (int)(it % (uint32_t)kNB);  // staging buffer and bin arrays
            // Bounded waits. A copy or hand-off that never completes poisons the CTA:
            // no further copies are issued, and the look-back warps publish only
            // errors from then on; the compute warps still run every tile (from
            // whatever the buffers hold: every index stays inside its buffer) so
            // that the hand-off protocol ends normally.
            wait_phase(&ctl->stage_full[s], (it >> 1) & 1u, g.timeout_ns, &ctl->poisoned);
            // the look-back warp of buffer bf has finished tile it - kNB: the
            // staging buffer and bin arrays bf are free and cleared
            if (it >= (uint32_t)kNB) wait_phase(&ctl->buf_empty[bf], (it / kNB - 1u) & 1u, g.timeout_ns, &ctl->poisoned);
            __syncwarp();
            const TileGeo G = info[s];
            const KLayer& ly = lays[G.layer];
            uint32_t* gmax_c = gmax_s + bf * bin_stride;
            uint32_t* cnt_c = cnt_s + bf * bin_stride;
            const int pr = (int)(G.ts & 3), pd = ly.dw_bf16 ? (int)(G.ts & 7) : pr;
            uint16_t* stg = stg0 + bf * stg_stride;
            Slot& sl = ctl->slot[bf];
            const uint32_t t_next = t + 2 * GS;
            // every compute warp calls this once per tile when it no longer reads the
            // stage; the last one starts the CTA's tile after next into it. No fence is
            // needed (and one would wait for this warp's global stores): the warp's
            // reads of the stage have returned their values, and one warp's shared
            // memory accesses are performed in order, so they precede its count.
            auto release = [&]() {
                if (lane == 0) {
                    asm volatile("" ::: "memory");
                    const uint32_t prev = atomicAdd(&ctl->users[s], 1u);
                    if (prev == kWarps - 1) {
                        ctl->users[s] = 0u;
                        if (t_next < T && !*reinterpret_cast<volatile uint32_t*>(&ctl->poisoned)) {
                            const int il = layer_from(lays, g.num_layers, t_next, ctl->issue_layer);
                            ctl->issue_layer = il;
                            issue_tile(lays, t_next, il, stage_r(s), stage_d(s), &ctl->stage_full[s], &info[s]);
                            ctl->issued[s] += 1u;
                        }
                    }
                }
                __syncwarp();
            };

            bool sliced;
            if constexpr (kPaths == 1) sliced = true;
            else if constexpr (kPaths == 2) sliced = false;
            else sliced = ly.bpw != 0;
            if (sliced) {
                if constexpr (kPaths & 1) {
                // warp-sliced tile: no barrier among the compute warps
                uint32_t src = 0, cnt;
                uint16_t* pend = nullptr;
                float s_prev = 0.0f;
                if constexpr (kLazy) {
                    pend = reinterpret_cast<uint16_t*>(ws + ws_pend_offset(g.num_layers, T)) +
                           ((size_t)t * kWarps + warp) * 32 + lane;
                    s_prev = reinterpret_cast<const LayerWs*>(ws + ws_layer_offset(G.layer))->result.s;
                }
                const bool ls = g.local_selection != 0;
                if (ly.dw_bf16)
                    cnt = warp_tile<true>(ly, G, pr, pd, stage_r(s), stage_d(s), wg, wc, cnt_c, stg, gmax_c, warp, lane,
                                          pend, s_prev, ls, &src, release);
                else
                    cnt = warp_tile<false>(ly, G, pr, pd, stage_r(s), stage_d(s), wg, wc, cnt_c, stg, gmax_c, warp, lane,
                                           pend, s_prev, ls, &src, release);
                if (lane == 0) {
                    sl.src[warp] = src;
                    sl.cnt[warp] = cnt;
                    if (warp == 0) sl.nrun = kWarps;
                }
                }
            } else {
                if constexpr ((kPaths & 2) != 0)
                    block_tile(ly, G, pr, pd, stage_r(s), stage_d(s), gbuf, gmax_c, cnt_c, stg, sl, ctl->wsum,
                               g.local_selection != 0, tid, &release);
            }
            if (tid == 0) {
                sl.t = t;
                sl.layer = (uint32_t)G.layer;
                sl.first_bin = G.first_bin;
                sl.bins = (uint32_t)G.bins;
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&ctl->buf_full[bf]);
        }
        // hand each look-back warp the end marker once it has released its buffer:
        // buffer b carried the tiles it' < it with it' % kNB == b. Every warp
        // waits for that release before it arrives: an arrival is not tied to a
        // phase, so one made early would count towards the last tile's hand-off.
        for (int b = 0; b < kNB; ++b) {
            const uint32_t uses = it > (uint32_t)b ? (it - b + kNB - 1) / kNB : 0u;  // tiles on buffer b
            if (lane == 0) {
                if (uses >= 1) wait_phase(&ctl->buf_empty[b], (uses - 1) & 1u, g.timeout_ns, &ctl->poisoned);
                if (warp == 0) ctl->slot[b].t = kEndTile;
                ptx::mbar_arrive(&ctl->buf_full[b]);
            }
            __syncwarp();
        }
    }
    __syncthreads();

    if (tid == 0 && *reinterpret_cast<volatile uint32_t*>(&ctl->poisoned)) {
        // Give the copies that may still be in flight one more bounded wait before
        // the CTA's shared memory is released.
        for (int k = 0; k < 2; ++k) {
            if (ctl->issued[k] == 0u) continue;
            const uint32_t par = (ctl->issued[k] - 1u) & 1u;
            uint64_t start = 0;
            while (!ptx::mbar_try_wait(&ctl->stage_full[k], par)) {
                const uint64_t now = ptx::globaltimer();
                if (start == 0) start = now;
                else if (now - start > g.timeout_ns) break;
            }
        }
    }
}

// One warp per layer, after the compress kernel: s from the layer's exact sum,
// header, result area; the accumulators are left zeroed for the next call.
__global__ void __launch_bounds__(32) finalize_kernel(const __grid_constant__ KGroup g, uint8_t* __restrict__ ws)
{
    __shared__ unsigned long long tmp[256];
    __shared__ unsigned long long words[kSumWords];
    const int l = blockIdx.x;
    if (threadIdx.x < kSumWords) words[threadIdx.x] = 0ull;
    __syncwarp();
    const uint64_t* desc = reinterpret_cast<const uint64_t*>(ws + ws_desc_offset(g.num_layers));
    Ctl* ctl = reinterpret_cast<Ctl*>(ws);
    const uint32_t last_epoch = *reinterpret_cast<volatile const uint32_t*>(&ctl->epoch);
    finalize_layer(g.layer[l], reinterpret_cast<LayerWs*>(ws + ws_layer_offset(l)), desc, call_epoch(last_epoch), tmp,
                   words, threadIdx.x);
    // the last block to finish records this call's epoch (every block has read the
    // previous one by then)
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(&ctl->fin_done, 1u) == (uint32_t)g.num_layers - 1u) {
            ctl->fin_done = 0u;
            ctl->epoch = last_epoch % 255u + 1u;
        }
    }
}

// ---------------------------------------------------------------- fix-up kernel
// For every sent element: residue = fl32(G - s) if G > 0, fl32(G + s) if G < 0
// (the residue still holds G). One warp per tile, tiles in reverse order so the
// most recently written residue lines are the likeliest to still be in L2. The
// warp turns the tile's per-bin counts into an exclusive prefix (shared memory,
// one array per warp); each lane then takes a contiguous run of the tile's codes,
// finds the bin of its first code by binary search and walks forward, gathering
// kFixBatch residues before it writes them back.
constexpr int kFixThreads = 256;
constexpr int kFixWarps = kFixThreads / 32;
constexpr int kFixBatch = 4;

__host__ __device__ inline uint32_t fix_smem_bytes(uint32_t num_layers, uint32_t max_bins)
{
    return num_layers * (uint32_t)sizeof(KLayer) + kFixWarps * (max_bins + 2) * 4;
}

__global__ void __launch_bounds__(kFixThreads) fixup_kernel(const __grid_constant__ KGroup g, uint8_t* __restrict__ ws)
{
    extern __shared__ uint4 fix_dyn[];
    KLayer* lays = reinterpret_cast<KLayer*>(fix_dyn);  // shared copy of the layer table
    for (int e = threadIdx.x; e < g.num_layers * (int)(sizeof(KLayer) / 16); e += kFixThreads)
        fix_dyn[e] = reinterpret_cast<const uint4*>(&g.layer[0])[e];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t* pre = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(fix_dyn) + g.num_layers * sizeof(KLayer)) +
                    warp * (g.max_bins + 2);
    __syncthreads();
    const uint64_t* texcl = reinterpret_cast<const uint64_t*>(ws + ws_desc_offset(g.num_layers)) + g.total_tiles;
    const uint32_t T = g.total_tiles;
    const uint32_t nw = gridDim.x * kFixWarps;

    for (uint32_t q = blockIdx.x * kFixWarps + warp; q < T; q += nw) {
        const uint32_t t = T - 1u - q;
        const int l = layer_from(lays, g.num_layers, t, 0);
        const KLayer& ly = lays[l];
        const uint32_t first_bin = (t - ly.tile_begin) * ly.bins_per_tile;
        const int bins = (int)min(ly.bins_per_tile, ly.nbins - first_bin);
        const int64_t ts = (int64_t)first_bin * ly.bin_len;
        const int tl = (int)min((int64_t)bins * ly.bin_len, ly.n - ts);
        const LayerWs* lw = reinterpret_cast<const LayerWs*>(ws + ws_layer_offset(l));
        if (lw->result.status == 0u && !(g.lazy && ly.bpw)) {  // deferred layers are corrected by the next call
            const uint16_t* cnt = reinterpret_cast<const uint16_t*>(ly.msg + 8) + first_bin;
            uint32_t run = 0;
            for (int b0 = 0; b0 < bins; b0 += 32) {
                const int b = b0 + lane;
                const uint32_t c = b < bins ? cnt[b] : 0u;
                uint32_t incl = c;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t y = __shfl_up_sync(kFull, incl, o);
                    if (lane >= o) incl += y;
                }
                if (b < bins) pre[b] = run + incl - c;
                run += __shfl_sync(kFull, incl, 31);
            }
            if (lane == 0) pre[bins] = run;
            __syncwarp();
            const uint32_t total = run;
            const uint32_t per = (total + 31) / 32;
            uint32_t i = min(total, lane * per);
            const uint32_t iend = min(total, i + per);
            if (i < iend) {
                const float s = lw->result.s;
                const uint8_t* codes = ly.msg + 8 + 2ull * ly.nbins + (unsigned long long)ly.code_bytes * texcl[t];
                float* res = ly.residue + ts;
                int lo = 0, hi = bins - 1;  // last bin whose prefix is <= i
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (pre[mid] <= i) lo = mid;
                    else hi = mid - 1;
                }
                int b = lo;
                uint32_t next = pre[b + 1];
                while (i < iend) {
                    int64_t off[kFixBatch];
                    uint32_t neg = 0;
                    float v[kFixBatch];
#pragma unroll
                    for (int u = 0; u < kFixBatch; ++u) {
                        off[u] = -1;
                        if (i + u < iend) {
                            while (i + u >= next) next = pre[++b + 1];
                            const uint32_t code = ly.code_bytes == 1 ? codes[i + u]
                                                                     : reinterpret_cast<const uint16_t*>(codes)[i + u];
                            const int64_t o = (int64_t)b * ly.bin_len + (code >> 1);
                            if (o < tl) off[u] = o;  // always true for codes this call produced
                            neg |= (code & 1u) << u;
                        }
                    }
#pragma unroll
                    for (int u = 0; u < kFixBatch; ++u)
                        if (off[u] >= 0) v[u] = res[off[u]];
#pragma unroll
                    for (int u = 0; u < kFixBatch; ++u)
                        if (off[u] >= 0) res[off[u]] = ((neg >> u) & 1u) ? __fadd_rn(v[u], s) : __fsub_rn(v[u], s);
                    i += kFixBatch;
                }
            }
        }
        __syncwarp();  // pre is rewritten for the next tile
    }
}

// ---------------------------------------------------------------- materialise (deferred fix-up)
// Applies the corrections a compress call with a deferred fix-up left pending:
// residue = fl32(G - sign(G) s) for every slot whose bit is set in its lane's mask,
// with s the layer's scale from that call; the masks are cleared. One CTA of
// 8 x 32 threads per tile, thread (warp, lane) owning the same slots as in the
// compress kernel's warp-sliced tile.
__global__ void __launch_bounds__(kThreads) materialize_kernel(const __grid_constant__ KGroup g,
                                                               uint8_t* __restrict__ ws)
{
    const uint32_t T = g.total_tiles;
    uint16_t* pend0 = reinterpret_cast<uint16_t*>(ws + ws_pend_offset(g.num_layers, T));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (uint32_t t = blockIdx.x; t < T; t += gridDim.x) {
        const int l = layer_from(g.layer, g.num_layers, t, 0);
        const KLayer& ly = g.layer[l];
        if (!ly.bpw) continue;
        uint16_t* pend = pend0 + ((size_t)t * kWarps + warp) * 32 + lane;
        const uint32_t pm = *pend;
        if (!pm) continue;
        const uint32_t first_bin = (t - ly.tile_begin) * ly.bins_per_tile;
        const int bins = (int)min(ly.bins_per_tile, ly.nbins - first_bin);
        const int64_t ts = (int64_t)first_bin * ly.bin_len;
        const int pr = (int)(ts & 3);
        const int wb0 = min(bins, warp * (int)ly.bpw);
        const int e_first = (((pr + wb0 * ly.bin_len) & ~3) - pr) + kSeg * lane;
        const int rot = seg_rot(lane);
        const float s = reinterpret_cast<const LayerWs*>(ws + ws_layer_offset(l))->result.s;
        float* res = ly.residue + ts + e_first;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int q0 = 4 * (k ^ rot);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (pm & (1u << (4 * k + i))) res[q0 + i] = __fsub_rn(res[q0 + i], copysignf(s, res[q0 + i]));
        }
        *pend = 0;
    }
}

}  // namespace

// ---------------------------------------------------------------- host launcher
namespace {
struct DeviceInfo {
    int sms = 0;
    uint32_t smem_set[5] = {0, 0, 0, 0, 0};  // largest dynamic shared memory opted in so far, per compress kernel
    uint32_t fix_smem_set = 0;  // same, fix-up kernel
};
DeviceInfo g_dev[64];
}  // namespace

cudaError_t launch_compress(const KGroup& g, void* ws, cudaStream_t stream, cudaEvent_t ev_before,
                            cudaEvent_t ev_mid, cudaEvent_t ev_after)
{
    if (group_is_sliced(g) || g.big) return launch_compress_sliced(g, ws, stream, ev_before, ev_mid, ev_after);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    DeviceInfo& di = g_dev[dev];
    if (di.sms == 0) {
        e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    int paths = 0;
    for (int l = 0; l < g.num_layers; ++l) paths |= g.layer[l].bpw ? 1 : 2;
    // here some layer is not warp-sliced (paths 2 or 3); three staging buffers
    const int nb = 3;
    const SmemPlan P = smem_plan(g.tile_cap, g.d_size, g.max_bins, g.num_layers, g.needs_gbuf, nb);
    void (*kern)(KGroup, uint8_t*);
    if (paths == 2) kern = compress_kernel<2, 3, false>;  // no warp-sliced layer: nothing is deferred
    else kern = g.lazy ? compress_kernel<3, 3, true> : compress_kernel<3, 3, false>;
    const int kidx = paths == 2 ? 2 : (g.lazy ? 3 : 4);
    const int threads = cta_threads(nb);
    if (P.total > di.smem_set[kidx]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P.total);
        if (e != cudaSuccess) return e;
        di.smem_set[kidx] = P.total;
    }
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, P.total);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    const long long cap = (long long)di.sms * occ;
    const uint32_t grid = (uint32_t)((long long)g.total_tiles < cap ? (long long)g.total_tiles : cap);
    if (ev_before && (e = cudaEventRecord(ev_before, stream)) != cudaSuccess) return e;
    {
        // all CTAs must be resident together: the look-back waits on other CTAs' tiles
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(threads);
        cfg.dynamicSmemBytes = P.total;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kern, g, static_cast<uint8_t*>(ws));
        if (e != cudaSuccess) return e;
    }
    if (ev_mid && (e = cudaEventRecord(ev_mid, stream)) != cudaSuccess) return e;
    finalize_kernel<<<g.num_layers, 32, 0, stream>>>(g, static_cast<uint8_t*>(ws));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (g.lazy && paths == 1) {  // every layer's corrections are deferred to the next call
        if (ev_after) e = cudaEventRecord(ev_after, stream);
        return e;
    }
    const uint32_t fsmem = fix_smem_bytes(g.num_layers, g.max_bins);
    if (fsmem > 48 * 1024 && fsmem > di.fix_smem_set) {
        e = cudaFuncSetAttribute(fixup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fsmem);
        if (e != cudaSuccess) return e;
        di.fix_smem_set = fsmem;
    }
    int focc = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&focc, fixup_kernel, kFixThreads, fsmem);
    if (e != cudaSuccess) return e;
    if (focc < 1) return cudaErrorInvalidConfiguration;
    const long long fwarps = (long long)di.sms * focc * kFixWarps;
    const long long fneed = ((long long)g.total_tiles < fwarps ? (long long)g.total_tiles : fwarps);
    const uint32_t fgrid = (uint32_t)((fneed + kFixWarps - 1) / kFixWarps);
    fixup_kernel<<<fgrid, kFixThreads, fsmem, stream>>>(g, static_cast<uint8_t*>(ws));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (ev_after) e = cudaEventRecord(ev_after, stream);
    return e;
}

cudaError_t launch_materialize(const KGroup& g, void* ws, cudaStream_t stream)
{
    if (group_is_sliced(g) || g.big) return launch_materialize_sliced(g, ws, stream);
    if (!g.lazy) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    DeviceInfo& di = g_dev[dev];
    if (di.sms == 0) {
        e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    const long long cap = (long long)di.sms * 8;
    const uint32_t grid = (uint32_t)((long long)g.total_tiles < cap ? (long long)g.total_tiles : cap);
    materialize_kernel<<<grid, kThreads, 0, stream>>>(g, static_cast<uint8_t*>(ws));
    return cudaGetLastError();
}

}  // namespace adacomp

// ---------------------------------------------------------------- compress without a caller workspace
// For callers that cannot allocate device memory (see adacomp_compress_static_ws in
// include/adacomp.h). The workspace lives in this file-scope array, which every GPU
// that loads the library holds until the process exits.
#include <atomic>
#include <cstddef>

#include "adacomp.h"

namespace adacomp {
adacomp_status launch_result(cudaError_t e, cudaStream_t stream);  // abi.cu
}

namespace {
constexpr size_t kStaticScratchBytes = ADACOMP_STATIC_WS_BYTES;  // 1 MiB
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];
// Device address of g_static_scratch, looked up once per device (index = device id).
std::atomic<void*> g_static_scratch_addr[64];
}  // namespace

extern "C" adacomp_status adacomp_compress_static_ws(adacomp_layer_t h, float* residue, const void* dW,
                                                     void* msg, size_t msg_capacity, void* result_out,
                                                     cudaStream_t stream)
{
    using namespace adacomp;
    if (!h) return ADACOMP_ERR_INVALID_ARG;
    if (compress_ws_of(h) > kStaticScratchBytes) return ADACOMP_ERR_WORKSPACE;  // layer too large
    KGroup g;  // on the host stack: nothing is allocated
    size_t ws_needed = 0;
    const int chk = prepare_single_compress(h, residue, dW, msg, msg_capacity, &g, &ws_needed);
    if (chk != ADACOMP_OK) return (adacomp_status)chk;
    if (g.lazy) return ADACOMP_ERR_INVALID_ARG;  // deferred corrections need a workspace kept by the caller
    if (result_out && (reinterpret_cast<uintptr_t>(result_out) & 7u)) return ADACOMP_ERR_ALIGNMENT;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return ADACOMP_ERR_CUDA;
    void* scratch = g_static_scratch_addr[dev].load(std::memory_order_acquire);
    if (!scratch) {
        // First call on this device (which is current): host code only has a stand-in
        // for the array's name, so fetch its device address.
        if (cudaGetSymbolAddress(&scratch, g_static_scratch) != cudaSuccess || !scratch) return ADACOMP_ERR_CUDA;
        g_static_scratch_addr[dev].store(scratch, std::memory_order_release);
    }
    // The array keeps the previous call's contents: zero the control word, the
    // layer's accumulators and the look-back descriptors this call relies on.
    const size_t zero_bytes = ws_zero_prefix(1, g.total_tiles, group_is_sliced(g) || g.big != 0);
    if (cudaMemsetAsync(scratch, 0, zero_bytes, stream) != cudaSuccess) return ADACOMP_ERR_CUDA;
    if (launch_compress(g, scratch, stream) != cudaSuccess) return ADACOMP_ERR_CUDA;
    if (result_out) {
        const uint8_t* res = static_cast<const uint8_t*>(scratch) + ws_layer_offset(0) + offsetof(LayerWs, result);
        if (cudaMemcpyAsync(result_out, res, sizeof(Result), cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
            return ADACOMP_ERR_CUDA;
    }
    return launch_result(cudaSuccess, stream);
}
