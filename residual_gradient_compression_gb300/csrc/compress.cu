// AdaComp compression for sm_103a: one fused streaming kernel per launch group
// (G, H, bin maxima, selection, per-bin counts, code compaction with a decoupled
// look-back across tiles, residue := G) and one sparse fix-up kernel that applies
// residue -= sign(G) * s once s, the mean of the bin maxima, is known.
//
// Method: "AdaComp (Adaptive Residual Gradient Compression)", Claims > Mechanism
// #r629-local-bin-soft-threshold-and-mean-gmax-quantization (Algorithm 2 restated):
// G = residue + dW, H = G + dW, g_max(i) = max |G| over bin i, s = mean g_max, send
// |H| >= g_max(i) as sign(G) * s, residue = G - G_q (sent) or G (kept). Code widths:
// Claims > Application #r629-conv-40x-and-fc-lstm-200x-compression-across-optimizers.
//
// Data flow per tile (a whole number of bins, about 4K elements):
//   bulk copy (TMA, cp.async.bulk) residue + dW -> shared memory, double-buffered;
//   phase A: G = residue + dW written back over the residue slice, per-chunk
//            max |G| reduced with redux.sync into g_max[bin];
//   bulk copy G -> residue in global memory (the final value of every kept element);
//   phase C: H = G + dW, flag = G != 0 && |H| >= g_max[bin]; warp ballots give each
//            code's rank; codes are staged in shared memory in element order;
//   look-back: the tile's code count is published and its exclusive prefix is
//            gathered from predecessor tiles (Merrill & Garland's single-pass scan);
//   codes and counts are written into the message; the bin maxima are added,
//   exactly, to the layer's exponent-bucketed integer accumulator.
// The tile that completes a layer turns the exact sum into s and writes the header.
#include "adacomp_internal.cuh"

#include <cuda_bf16.h>

namespace adacomp {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ uint32_t lanemask_lt()
{
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

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
    float* gs;        // G, same slot layout as sr (a buffer the bulk copies never target)
    const void* sd; // dW slice; element i at sd[pd + i]
    int pr, pd;
    int tl;         // elements in the tile
    int L;          // bin length
    int bins;       // bins in the tile (last bin may be partial)
    int cpb;        // chunks per bin
    int ch;         // chunk length (elements, multiple of VEC)
    uint32_t inv_len;  // ceil(2^32 / L)
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
                    float h = __fadd_rn(g[k], d[k]);
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
constexpr int kSeg = 16;

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

__device__ __forceinline__ int seg_rot(int tid) { return ((tid >> 1) ^ (tid >> 3)) & 3; }

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

// Phase A, segment path: G = residue + dW over the slots, written to the G buffer
// (for phase C) and to the residue in global memory; bin maxima. *mine gets
// the geometry of segment `tid` (the thread's only segment when the tile fits one
// round).
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
        float* gsp = T.gs + s * kSeg;
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
            *reinterpret_cast<float4*>(gsp + q0) = make_float4(g[0], g[1], g[2], g[3]);
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

// Flags of one segment's 16 slots (bit idx): G != 0 && |fl32(G + dW)| >= g_max.
template <bool BF16>
__device__ __forceinline__ uint32_t seg_flags(const Tile& T, const SegGeo& G, int s, int rot, float gm_lo,
                                              float gm_hi)
{
    const float* rs = T.gs + s * kSeg;
    uint32_t f = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int q = k ^ rot;
        const int q0 = 4 * q;
        const float4 gv = *reinterpret_cast<const float4*>(rs + q0);
        const float g[4] = {gv.x, gv.y, gv.z, gv.w};
        float d[4];
        seg_load_d<BF16>(T, s, q, d);
        uint32_t nib = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float h = __fadd_rn(g[i], d[i]);
            const float gm = q0 + i < G.split ? gm_lo : gm_hi;
            nib |= (g[i] != 0.0f && fabsf(h) >= gm) ? (1u << i) : 0u;
        }
        f |= nib << q0;
    }
    return f;
}

// Phase C, segment path: flags and codes per slot, per-bin counts, and a block-wide
// exclusive scan of the per-segment counts (in element order) that places every
// code at stg[rank]. For tiles of several rounds. Runs on the 256 compute threads
// (named barrier 1). Returns the tile's code count (same value in every thread).
template <bool BF16>
__device__ __forceinline__ uint32_t phase_c_seg(const Tile& T, const uint32_t* gmax_s, uint32_t* cnt_s,
                                                uint16_t* stg, uint32_t* wsum, int tid)
{
    const int nseg = (T.pr + T.tl + kSeg - 1) / kSeg;
    const int rot = seg_rot(tid);
    const int lane = tid & 31, warp = tid >> 5;
    uint32_t carry = 0;
    for (int base = 0; base < nseg; base += kThreads) {
        const int s = base + tid;
        uint32_t f = 0;
        SegGeo G;
        G.valid = 0; G.bin_lo = 0; G.split = kSeg; G.off_lo = 0; G.e0 = 0;
        if (s < nseg) {
            G = seg_geo(T, s);
            const float gm_lo = __uint_as_float(gmax_s[G.bin_lo]);
            const float gm_hi = G.split < kSeg ? __uint_as_float(gmax_s[G.bin_lo + 1]) : 0.0f;
            f = seg_flags<BF16>(T, G, s, rot, gm_lo, gm_hi);
            const uint32_t lomask = G.split >= kSeg ? 0xffffu : ((1u << max(G.split, 0)) - 1u);
            const uint32_t c_lo = __popc(f & lomask), c_hi = __popc(f & ~lomask);
            if (c_lo) atomicAdd(&cnt_s[G.bin_lo], c_lo);
            if (c_hi) atomicAdd(&cnt_s[G.bin_lo + 1], c_hi);
        }
        // block-wide exclusive scan of the per-thread counts
        const uint32_t c = __popc(f);
        uint32_t incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) wsum[warp] = incl;
        asm volatile("bar.sync %0, %1;" ::"n"(1), "n"(kThreads) : "memory");
        uint32_t woff = 0, tot = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const uint32_t v = wsum[w];
            woff += w < warp ? v : 0u;
            tot += v;
        }
        uint32_t pos = carry + woff + incl - c;
        const float* rs = T.gs + s * kSeg;
        while (f) {
            const int idx = __ffs(f) - 1;
            f &= f - 1;
            const int off = G.off_lo + idx - (idx < G.split ? 0 : T.L);
            stg[pos++] = (uint16_t)(((uint32_t)off << 1) | (rs[idx] < 0.0f ? 1u : 0u));
        }
        carry += tot;
        asm volatile("bar.sync %0, %1;" ::"n"(1), "n"(kThreads) : "memory");  // wsum reuse
    }
    return carry;
}

// Phase C, segment path, for tiles of one round (at most 256 segments, one per
// thread, whose geometry phase A computed): flags per slot and per-bin counts; each
// warp then ranks its own codes (shuffle scan of the per-thread counts) and stages
// them at stg[wbase + rank], wbase being the first tile element of the warp's
// segments (a warp never has more codes than elements, so the warps' ranges stay
// disjoint). Only the sent slots are visited when the codes are written. Returns
// the warp's code count.
template <bool BF16>
__device__ __forceinline__ uint32_t phase_c_seg_warp(const Tile& T, const SegGeo& G, const uint32_t* gmax_s,
                                                     uint32_t* cnt_s, uint16_t* stg, int tid, int* wbase_out)
{
    const int nseg = (T.pr + T.tl + kSeg - 1) / kSeg;
    const int lane = tid & 31, warp = tid >> 5;
    const int s = tid;
    uint32_t f = 0;
    if (s < nseg) {
        const float gm_lo = __uint_as_float(gmax_s[G.bin_lo]);
        const float gm_hi = G.split < kSeg ? __uint_as_float(gmax_s[G.bin_lo + 1]) : 0.0f;
        f = seg_flags<BF16>(T, G, s, seg_rot(tid), gm_lo, gm_hi);
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
    const float* rs = T.gs + s * kSeg;
    while (f) {
        const int idx = __ffs(f) - 1;
        f &= f - 1;
        const int off = G.off_lo + idx - (idx < G.split ? 0 : T.L);
        stg[pos++] = (uint16_t)(((uint32_t)off << 1) | (rs[idx] < 0.0f ? 1u : 0u));
    }
    *wbase_out = wbase;
    return total;
}

// ---------------------------------------------------------------- exact scale sum
// The layer's bin maxima arrive as integer mantissas bucketed by fp32 exponent:
// bucket E holds sum(M) over maxima with biased exponent E, where a value equals
// M * 2^(max(E,1) - 150). The exact sum is rebuilt as a 384-bit integer in units of
// 2^-149 and rounded once to the nearest fp64 (ties to even), so s does not depend
// on the order in which tiles finished.
__device__ double exact_sum_from_buckets(const unsigned long long* acc)
{
    constexpr int W = 12;
    uint32_t w[W];
#pragma unroll
    for (int i = 0; i < W; ++i) w[i] = 0;
    if (acc[255] != 0ull) return __longlong_as_double(0x7ff0000000000000ll);  // non-finite input
    for (int e = 0; e < 255; ++e) {
        const unsigned long long v = acc[e];
        if (v == 0ull) continue;
        const int sh = e ? e - 1 : 0;
        const int q = sh >> 5, b = sh & 31;
        const unsigned long long lo = v << b;
        const unsigned long long hi = b ? (v >> (64 - b)) : 0ull;
        const uint32_t part[4] = {(uint32_t)lo, (uint32_t)(lo >> 32), (uint32_t)hi, (uint32_t)(hi >> 32)};
        unsigned long long carry = 0;
        for (int i = 0; q + i < W; ++i) {
            unsigned long long t = (unsigned long long)w[q + i] + (i < 4 ? part[i] : 0u) + carry;
            w[q + i] = (uint32_t)t;
            carry = t >> 32;
            if (i >= 3 && carry == 0) break;
        }
    }
    int top = -1;
    for (int i = W - 1; i >= 0; --i)
        if (w[i]) { top = i * 32 + 31 - __clz(w[i]); break; }
    if (top < 0) return 0.0;
    const int lo = top - 52;
    if (lo <= 0) {
        unsigned long long m = ((unsigned long long)w[1] << 32) | w[0];
        return ldexp((double)m, -149);
    }
    const int q = lo >> 5, off = lo & 31;
    const unsigned long long x = (unsigned long long)w[q] | ((unsigned long long)(q + 1 < W ? w[q + 1] : 0u) << 32);
    const unsigned long long x2 = q + 2 < W ? w[q + 2] : 0u;
    unsigned long long mant = off ? ((x >> off) | (x2 << (64 - off))) : x;
    mant &= (1ull << 53) - 1;
    const int rb = lo - 1;
    const uint32_t round = (w[rb >> 5] >> (rb & 31)) & 1u;
    uint32_t sticky = 0;
    if (rb > 0) {
        const int sq = (rb - 1) >> 5;
        for (int i = 0; i < sq; ++i) sticky |= w[i];
        const int nb = ((rb - 1) & 31) + 1;  // bits 0 .. rb-1 of word sq
        sticky |= w[sq] & (nb == 32 ? 0xffffffffu : ((1u << nb) - 1u));
    }
    if (round && (sticky || (mant & 1ull))) ++mant;
    return ldexp((double)mant, lo - 149);
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

__device__ bool lookback_resolve(uint64_t* desc, uint32_t t, uint32_t tile_begin, uint32_t total,
                                 uint64_t timeout_ns, int lane, bool publish, uint64_t* excl_out)
{
    if (t == tile_begin) {
        *excl_out = 0;
        return true;
    }
    uint64_t excl = 0;
    int64_t j = (int64_t)t - 1;
    uint64_t start = 0;
    uint32_t sleep_ns = 64;
    bool ok = true;
    for (;;) {
        uint64_t dv[kLbPerLane];
#pragma unroll
        for (int m = 0; m < kLbPerLane; ++m) {
            const int64_t idx = j - (m * 32 + lane);
            dv[m] = idx >= (int64_t)tile_begin ? ptx::ld_relaxed(&desc[idx]) : kFlagIncl;
        }
        int mstar = kLbPerLane;
        uint32_t lim = 31;
        bool pending = false, error = false;
        uint32_t needed[kLbPerLane];
#pragma unroll
        for (int m = 0; m < kLbPerLane; ++m) {
            const uint32_t f = (uint32_t)(dv[m] >> 62);
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
            sleep_ns = 64;
            continue;
        }
        uint64_t now = 0;
        if (lane == 0) now = ptx::globaltimer();
        now = __shfl_sync(kFull, now, 0);
        if (start == 0) start = now;
        else if (now - start > timeout_ns) { ok = false; break; }
        __nanosleep(sleep_ns);
        if (sleep_ns < 512) sleep_ns <<= 1;
    }
    if (lane == 0 && publish) ptx::st_relaxed(&desc[t], ok ? (kFlagIncl | (excl + total)) : kFlagErr);
    *excl_out = excl;
    return ok;
}

// ---------------------------------------------------------------- layer finalisation
// Run by one warp of the CTA whose tile completed the layer: s from the exact sum,
// header, result area; the accumulator and counters are left zeroed for the next
// call. `tmp` is a zeroed 256-entry shared buffer; it is zeroed again on return.
__device__ void finalize_layer(const KLayer& ly, LayerWs* lw, const uint64_t* desc, unsigned long long* tmp,
                               int lane)
{
    __threadfence();
    for (int e = lane; e < 256; e += 32)
        tmp[e] = ptx::ld_relaxed(reinterpret_cast<const uint64_t*>(&lw->acc[e]));
    __syncwarp();
    if (lane == 0) {
        const double S = exact_sum_from_buckets(tmp);
        const float s = __double2float_rn(__ddiv_rn(S, (double)ly.nbins));
        const uint32_t err = *reinterpret_cast<volatile uint32_t*>(&lw->err);
        const uint64_t last = ptx::ld_relaxed(&desc[ly.tile_begin + ly.num_tiles - 1]);
        const bool bad = err != 0u || (last >> 62) != 2u;
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
    __syncwarp();
    for (int e = lane; e < 256; e += 32) {
        lw->acc[e] = 0ull;
        tmp[e] = 0ull;
    }
    __syncwarp();
}

// ---------------------------------------------------------------- tile geometry
struct TileGeo {
    int layer;
    int64_t ts;          // first element of the tile within its layer
    int tl;              // elements in the tile
    uint32_t first_bin;
    int bins;
};


// Bounded wait on a stage's mbarrier phase; true when the data has landed.
__device__ __forceinline__ bool wait_stage(uint64_t* bar, uint32_t parity, uint64_t timeout_ns)
{
    uint64_t start = 0;
    while (!ptx::mbar_try_wait(bar, parity)) {
        const uint64_t now = ptx::globaltimer();
        if (start == 0) start = now;
        else if (now - start > timeout_ns) return false;
    }
    return true;
}

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
// Eight compute warps stream a tile through phases A and C (three barriers per
// tile), publish its code count and hand the staged codes to one of two look-back
// warps (one per staging buffer), which resolves the tile's prefix and copies the
// codes into the message while the compute warps go on. Hand-off uses named
// barriers FULL[b] (compute -> look-back warp b) and EMPTY[b] (back).
// Bin maxima accumulate per CTA in exponent buckets and are flushed to the layer's
// accumulator when the CTA moves to another layer; s is formed afterwards by the
// finalise kernel.
constexpr int kLookbackWarps = 2;  // one per staging buffer
constexpr int kCtaThreads = kThreads + 32 * kLookbackWarps;
constexpr int kBarCompute = 1;
constexpr int kBarFull = 2;   // + buffer
constexpr int kBarEmpty = 4;  // + buffer
constexpr uint32_t kEndTile = 0xffffffffu;

struct Slot {
    uint32_t t, total, layer, nrun;
    uint32_t first_bin, bins, pad0, pad1;
    uint32_t src[kWarps], dst[kWarps], cnt[kWarps];
};

template <int ID, int N>
__device__ __forceinline__ void bar_sync() { asm volatile("bar.sync %0, %1;" ::"n"(ID), "n"(N) : "memory"); }
template <int ID, int N>
__device__ __forceinline__ void bar_arrive() { asm volatile("bar.arrive %0, %1;" ::"n"(ID), "n"(N) : "memory"); }
// Named barriers of the buffer-indexed pairs (the compute warps and the look-back
// warp that owns buffer b), with the index known only at run time.
constexpr int kPair = kThreads + 32;
__device__ __forceinline__ void full_sync(int b) { if (b) bar_sync<kBarFull + 1, kPair>(); else bar_sync<kBarFull, kPair>(); }
__device__ __forceinline__ void full_arrive(int b) { if (b) bar_arrive<kBarFull + 1, kPair>(); else bar_arrive<kBarFull, kPair>(); }
__device__ __forceinline__ void empty_sync(int b) { if (b) bar_sync<kBarEmpty + 1, kPair>(); else bar_sync<kBarEmpty, kPair>(); }
__device__ __forceinline__ void empty_arrive(int b) { if (b) bar_arrive<kBarEmpty + 1, kPair>(); else bar_arrive<kBarEmpty, kPair>(); }
__device__ __forceinline__ void compute_sync() { bar_sync<kBarCompute, kThreads>(); }


// Barrier among the compute threads that also ANDs a predicate over them.
__device__ __forceinline__ bool compute_and(bool p)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred a, b;\n\t"
        "setp.ne.u32 a, %1, 0;\n\t"
        "bar.red.and.pred b, %2, %3, a;\n\t"
        "selp.u32 %0, 1, 0, b;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)p), "n"(kBarCompute), "n"(kThreads)
        : "memory");
    return r != 0;
}

// Layer of tile t, searching from layer `lo` (tiles of a CTA only move forward).
// `lays` is the CTA's shared-memory copy of the layer table: kernel parameters
// indexed at run time would be served by the small constant cache, and a miss
// costs an L2 round trip.
__device__ __forceinline__ int layer_from(const KLayer* lays, int num_layers, uint32_t t, int lo)
{
    int hi = num_layers - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (lays[mid].tile_begin <= t) lo = mid;
        else hi = mid - 1;
    }
    return lo;
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
    ptx::mbar_arrive_expect_tx(bar, rb + db);
    if (rb) ptx::bulk_g2s(sr, ly.residue + a0, rb, bar);
    if (db) ptx::bulk_g2s(sd, static_cast<const uint8_t*>(ly.dw) + b0 * (ly.dw_bf16 ? 2 : 4), db, bar);
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
}

// Exponent buckets of the bin maxima: warp `w` of `nw` handles the groups of 32
// bins b0 = 32 w, 32 (w + nw), ... A group of 32 maxima mostly has the largest
// exponent present or the one below it: both are summed with one warp reduction
// each (at most 32 x 2^24 < 2^32); any other exponent is summed in a loop. Lane 0
// adds each sum to the CTA's shared buckets with a 64-bit shared atomic.
__device__ __forceinline__ void bucket_bins(const uint32_t* gmax_s, int bins, unsigned long long* hist, int lane,
                                            int w, int nw)
{
    for (int b0 = 32 * w; b0 < bins; b0 += 32 * nw) {
        const int b = b0 + lane;
        const uint32_t u = b < bins ? gmax_s[b] : 0u;
        const uint32_t E = u >> 23;
        const uint32_t M = E ? ((u & 0x7fffffu) | 0x800000u) : (u & 0x7fffffu);
        if (__ballot_sync(kFull, u != 0u) == 0u) continue;
        const uint32_t Eh = __reduce_max_sync(kFull, u ? E : 0u);
        const uint32_t s_hi = __reduce_add_sync(kFull, (u && E == Eh) ? M : 0u);
        const uint32_t s_lo = __reduce_add_sync(kFull, (u && Eh > 0 && E == Eh - 1) ? M : 0u);
        if (lane == 0) {
            if (s_hi) atomicAdd(&hist[Eh], (unsigned long long)s_hi);
            if (s_lo) atomicAdd(&hist[Eh - 1], (unsigned long long)s_lo);
        }
        uint32_t left = __ballot_sync(kFull, u != 0u && E + 1 < Eh);
        while (left) {
            const uint32_t Ek = __shfl_sync(kFull, E, __ffs(left) - 1);
            const bool mine = ((left >> lane) & 1u) && E == Ek;
            const uint32_t sum = __reduce_add_sync(kFull, mine ? M : 0u);
            if (lane == 0) atomicAdd(&hist[Ek], (unsigned long long)sum);
            left &= ~__ballot_sync(kFull, mine);
        }
        __syncwarp();
    }
}

// Adds a warp's shared buckets to layer lw's accumulator and clears them.
__device__ __forceinline__ void flush_buckets(unsigned long long* hist, LayerWs* lw, int lane)
{
    __syncwarp();
    for (int e = lane; e < 256; e += 32) {
        const unsigned long long v = hist[e];
        if (v) {
            atomicAdd(&lw->acc[e], v);
            hist[e] = 0ull;
        }
    }
    __syncwarp();
}

// Look-back warp that owns staging buffer b, i.e. every other tile of the CTA.
// For each such tile, in order: it writes the per-bin counts into the message and
// clears the bin arrays; then it resolves the tile's prefix with the look-back (by
// now the predecessors have had time to publish) and copies the staged codes into
// the message.
struct LookbackCtx {
    uint16_t* stg;
    uint32_t* gmax;
    uint32_t* cnt;
    uint32_t bin_len;  // entries of gmax / cnt to clear
};

__device__ void lookback_warp(const KGroup& g, const KLayer* lays, uint8_t* ws, const Slot* slots, const LookbackCtx& C,
                              int b, int lane)
{
    uint64_t* desc = reinterpret_cast<uint64_t*>(ws + ws_desc_offset(g.num_layers));
    uint64_t* texcl = desc + g.total_tiles;
    for (;;) {
        full_sync(b);
        const Slot& sl = slots[b];
        const uint32_t t = sl.t;
        if (t == kEndTile) break;
        const int l = (int)sl.layer;
        const KLayer& ly = lays[l];
        const int bins = (int)sl.bins;
        uint16_t* cdst = reinterpret_cast<uint16_t*>(ly.msg + 8) + sl.first_bin;
        for (int bb = lane; bb < bins; bb += 32) cdst[bb] = (uint16_t)C.cnt[bb];
        __syncwarp();
        for (uint32_t bb = lane; bb < C.bin_len; bb += 32) { C.gmax[bb] = 0u; C.cnt[bb] = 0u; }
        uint64_t excl = 0;
        const bool ok = lookback_resolve(desc, t, ly.tile_begin, sl.total, g.timeout_ns, lane,
                                         t != g.inject_skip_tile, &excl);
        if (ok) {
            if (lane == 0) texcl[t] = excl;
            uint8_t* codes = ly.msg + 8 + 2ull * ly.nbins;
            for (uint32_t r = 0; r < sl.nrun; ++r) {
                const uint32_t n = sl.cnt[r];
                const uint16_t* sp = C.stg + sl.src[r];
                const unsigned long long base = excl + sl.dst[r];
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
        empty_arrive(b);
    }
}

// One-round segment tile held in registers (at most 256 segments, one per thread):
// phase A computes G, residue := G, the bin maxima and, per slot, |H| = |fl32(G + dW)|
// and the masks of G != 0 and G < 0 (all phase C needs); after a barrier the stage
// is no longer read and thread 0 refills it with the CTA's tile after next; phase C
// then runs from the registers (flags, per-bin counts, codes ranked per warp and
// staged at stg[wbase + rank]). Returns the warp's code count.
template <bool BF16, class Refill>
__device__ __forceinline__ uint32_t tile_in_registers(const Tile& T, uint32_t* gmax_s, uint32_t* cnt_s,
                                                      uint16_t* stg, int tid, int* wbase_out, Refill&& refill)
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
                ah[k][i] = fabsf(__fadd_rn(g[i], d[i]));
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
    if (tid == 0) refill();
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

__global__ void __launch_bounds__(kCtaThreads, 2) compress_kernel(const __grid_constant__ KGroup g,
                                                                  uint8_t* __restrict__ ws)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const SmemPlan P = smem_plan(g.tile_cap, g.d_size, g.max_bins, g.num_layers, g.needs_gbuf);
    uint8_t* p = smem;
    float* sr[2];
    void* sd[2];
    sr[0] = reinterpret_cast<float*>(p); p += P.r_bytes;
    sd[0] = p; p += P.d_bytes;
    sr[1] = reinterpret_cast<float*>(p); p += P.r_bytes;
    sd[1] = p; p += P.d_bytes;
    KLayer* lays = reinterpret_cast<KLayer*>(p); p += P.layer_bytes;
    float* gbuf = reinterpret_cast<float*>(p); p += P.g_bytes;  // G, for tiles not held in registers
    uint16_t* stg0 = reinterpret_cast<uint16_t*>(p); p += 2 * P.stg_bytes;
    const uint32_t stg_stride = P.stg_bytes / 2;
    uint32_t* gmax_s = reinterpret_cast<uint32_t*>(p); p += P.bin_bytes;  // 2 buffers of bin_stride
    uint32_t* cnt_s = reinterpret_cast<uint32_t*>(p); p += P.bin_bytes;   // 2 buffers of bin_stride
    const uint32_t bin_stride = P.bin_bytes / 8;
    unsigned long long* hist = reinterpret_cast<unsigned long long*>(p); p += 4096;  // [256] exponent buckets + spare
    TileGeo* info = reinterpret_cast<TileGeo*>(p); p += 2048;  // [2]: geometry of the tile in each stage
    uint64_t* bar = reinterpret_cast<uint64_t*>(p); p += 16;
    Slot* slots = reinterpret_cast<Slot*>(p); p += 2 * sizeof(Slot);
    uint32_t* wsum = reinterpret_cast<uint32_t*>(p);         // [8]
    uint32_t* wtot = wsum + 8;                               // [8]
    int32_t* wbase = reinterpret_cast<int32_t*>(wsum + 16);  // [8]

    uint64_t* desc = reinterpret_cast<uint64_t*>(ws + ws_desc_offset(g.num_layers));
    const uint32_t T = g.total_tiles;
    const uint32_t G0 = blockIdx.x, GS = gridDim.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    for (int e = tid; e < 512; e += kCtaThreads) hist[e] = 0ull;
    {
        const uint4* src = reinterpret_cast<const uint4*>(&g.layer[0]);
        uint4* dst = reinterpret_cast<uint4*>(lays);
        for (int e = tid; e < g.num_layers * (int)(sizeof(KLayer) / 16); e += kCtaThreads) dst[e] = src[e];
    }
    __syncthreads();
    for (uint32_t e = tid; e < 2 * bin_stride; e += kCtaThreads) { gmax_s[e] = 0u; cnt_s[e] = 0u; }
    int issue_layer = 0;  // layer of the last tile issued (thread 0 issues every tile)
    if (tid == 0) {
        ptx::mbar_init(&bar[0], 1);
        ptx::mbar_init(&bar[1], 1);
        ptx::fence_mbar_init();
        for (int k = 0; k < 2; ++k) {
            const uint32_t t = G0 + k * GS;
            if (t < T) {
                issue_layer = layer_from(lays, g.num_layers, t, issue_layer);
                issue_tile(lays, t, issue_layer, sr[k], sd[k], &bar[k], &info[k]);
            }
        }
    }
    __syncthreads();

    bool poisoned = false;
    uint32_t it = 0;
    if (warp >= kWarps) {
        const int b = warp - kWarps;  // look-back warp of staging buffer b
        LookbackCtx C;
        C.stg = stg0 + b * stg_stride;
        C.gmax = gmax_s + b * bin_stride;
        C.cnt = cnt_s + b * bin_stride;
        C.bin_len = bin_stride;
        lookback_warp(g, lays, ws, slots, C, b, lane);
    } else {
        int hist_layer = -1;
        for (;; ++it) {
            const uint32_t t = G0 + it * GS;
            if (t >= T) break;
            const int s = it & 1;  // stage, staging buffer and bin-array buffer
            const uint32_t parity = (it >> 1) & 1u;
            if (!compute_and(wait_stage(&bar[s], parity, g.timeout_ns))) {
                poisoned = true;
                break;
            }
            // the look-back warp of this parity has finished tile it-2: the staging
            // buffer and bin arrays of parity s are free and cleared
            if (it >= 2) empty_sync(s);
            const TileGeo G = info[s];
            const KLayer& ly = lays[G.layer];
            if (G.layer != hist_layer) {  // new layer: hand the buckets to the previous one
                if (warp == 1 && hist_layer >= 0)
                    flush_buckets(hist, reinterpret_cast<LayerWs*>(ws + ws_layer_offset(hist_layer)), lane);
                hist_layer = G.layer;
            }
            uint32_t* gmax_c = gmax_s + s * bin_stride;
            uint32_t* cnt_c = cnt_s + s * bin_stride;
            const int pr = (int)(G.ts & 3), pd = ly.dw_bf16 ? (int)(G.ts & 7) : pr;
            float* r_s = sr[s];
            void* d_s = sd[s];
            const int64_t te = G.ts + G.tl;

            Tile Tl;
            Tl.gres = ly.residue + (G.ts - pr);
            Tl.sr = r_s; Tl.gs = gbuf; Tl.sd = d_s; Tl.pr = pr; Tl.pd = pd; Tl.tl = G.tl; Tl.L = ly.bin_len; Tl.bins = G.bins;
            Tl.ch = min(ly.bin_len, 32 * (int)ly.vec * kRounds);
            Tl.cpb = (ly.bin_len + Tl.ch - 1) / Tl.ch;
            Tl.inv_len = ly.inv_len;
            const bool seg = ly.bin_len >= kSeg;
            const bool one_round = seg && pr + G.tl <= kThreads * kSeg;
            const int nchunks = G.bins * Tl.cpb;
            const int cpw = (nchunks + kWarps - 1) / kWarps;
            const int c_begin = min(nchunks, warp * cpw), c_end = min(nchunks, c_begin + cpw);

            uint16_t* stg = stg0 + s * stg_stride;
            Slot& sl = slots[s];
            const uint32_t t_next = t + 2 * GS;
            // thread 0: start the CTA's tile after next into stage s once it is free
            auto refill = [&]() {
                if (t_next < T) {
                    issue_layer = layer_from(lays, g.num_layers, t_next, issue_layer);
                    issue_tile(lays, t_next, issue_layer, sr[s], sd[s], &bar[s], &info[s]);
                }
            };
            if (one_round) {
                // phases A and C with G and dW in registers; the stage is refilled in between
                int wb = 0;
                uint32_t wt;
                if (ly.dw_bf16) wt = tile_in_registers<true>(Tl, gmax_c, cnt_c, stg, tid, &wb, refill);
                else wt = tile_in_registers<false>(Tl, gmax_c, cnt_c, stg, tid, &wb, refill);
                if (lane == 0) { wtot[warp] = wt; wbase[warp] = wb; }
                compute_sync();
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
                    if (lane == 0) { wtot[warp] = wt; wbase[warp] = wb; }
                    compute_sync();
                } else {  // several rounds: block-wide scan (ends with a barrier)
                    uint32_t total;
                    if (ly.dw_bf16) total = phase_c_seg<true>(Tl, gmax_c, cnt_c, stg, wsum, tid);
                    else total = phase_c_seg<false>(Tl, gmax_c, cnt_c, stg, wsum, tid);
                    if (tid == 0) {
                        sl.total = total;
                        sl.nrun = 1;
                        sl.src[0] = 0; sl.dst[0] = 0; sl.cnt[0] = total;
                    }
                }
                if (tid == 0) refill();  // phase C was the last reader of stage s
            }

            if (warp == 0) {
                if (one_round || !seg) {
                    const uint32_t v = lane < kWarps ? wtot[lane] : 0u;
                    uint32_t incl = v;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const uint32_t y = __shfl_up_sync(kFull, incl, o);
                        if (lane >= o) incl += y;
                    }
                    if (lane < kWarps) {
                        sl.src[lane] = (uint32_t)wbase[lane];
                        sl.dst[lane] = incl - v;
                        sl.cnt[lane] = v;
                    }
                    const uint32_t tot = __shfl_sync(kFull, incl, 31);
                    if (lane == 0) {
                        sl.total = tot;
                        sl.nrun = kWarps;
                    }
                }
                if (lane == 0) {
                    sl.t = t;
                    sl.layer = (uint32_t)G.layer;
                    sl.first_bin = G.first_bin;
                    sl.bins = (uint32_t)G.bins;
                    if (t != g.inject_skip_tile)
                        ptx::st_relaxed(&desc[t], (t == ly.tile_begin ? kFlagIncl : kFlagAgg) | sl.total);
                }
            } else {
                bucket_bins(gmax_c, G.bins, hist, lane, warp - 1, kWarps - 1);
            }
            full_arrive(s);
        }
        compute_sync();  // every warp's additions to the buckets are in
        if (warp == 1 && hist_layer >= 0)
            flush_buckets(hist, reinterpret_cast<LayerWs*>(ws + ws_layer_offset(hist_layer)), lane);
        // hand each look-back warp the end marker once it has released its buffer:
        // buffer b carried the tiles it' < it with it' % 2 == b
        for (int b = 0; b < 2; ++b) {
            if ((it + 1 - b) / 2 >= 1) empty_sync(b);
            if (tid == 0) slots[b].t = kEndTile;
            full_arrive(b);
        }
    }
    __syncthreads();

    if (poisoned && tid == 0) {
        // A bulk copy never completed: mark this CTA's remaining tiles as errors so
        // no other tile waits on them, then give the outstanding copies one more
        // bounded wait before the CTA's shared memory is released.
        int l = 0;
        for (uint32_t t = G0 + it * GS; t < T; t += GS) {
            l = layer_from(lays, g.num_layers, t, l);
            ptx::st_relaxed(&desc[t], kFlagErr);
            atomicOr(&reinterpret_cast<LayerWs*>(ws + ws_layer_offset(l))->err, kErrTimeout);
        }
    }
    if (poisoned && warp < kWarps) {
        wait_stage(&bar[it & 1], (it >> 1) & 1u, g.timeout_ns);
        if (G0 + (it + 1) * GS < T) wait_stage(&bar[(it + 1) & 1], ((it + 1) >> 1) & 1u, g.timeout_ns);
    }
}

// One warp per layer, after the compress kernel: s from the layer's exact sum,
// header, result area; the accumulators are left zeroed for the next call.
__global__ void __launch_bounds__(32) finalize_kernel(const __grid_constant__ KGroup g, uint8_t* __restrict__ ws)
{
    __shared__ unsigned long long tmp[256];
    const int l = blockIdx.x;
    for (int e = threadIdx.x; e < 256; e += 32) tmp[e] = 0ull;
    __syncwarp();
    const uint64_t* desc = reinterpret_cast<const uint64_t*>(ws + ws_desc_offset(g.num_layers));
    finalize_layer(g.layer[l], reinterpret_cast<LayerWs*>(ws + ws_layer_offset(l)), desc, tmp, threadIdx.x);
}

// ---------------------------------------------------------------- fix-up kernel
// For every sent element: residue = fl32(G - s) if G > 0, fl32(G + s) if G < 0
// (the residue still holds G). Tiles are visited in reverse order, so the most
// recently written residue lines are the likeliest to still be in L2. Also returns
// the look-back descriptors to zero for the next call.
constexpr int kFixThreads = 256;

__global__ void __launch_bounds__(kFixThreads) fixup_kernel(const __grid_constant__ KGroup g, uint8_t* __restrict__ ws)
{
    __shared__ uint32_t pre[kMaxBinsPerTile + 1];
    __shared__ uint32_t wsum[kFixThreads / 32];
    extern __shared__ uint4 fix_dyn[];
    KLayer* lays = reinterpret_cast<KLayer*>(fix_dyn);  // shared copy of the layer table
    for (int e = threadIdx.x; e < g.num_layers * (int)(sizeof(KLayer) / 16); e += kFixThreads)
        fix_dyn[e] = reinterpret_cast<const uint4*>(&g.layer[0])[e];
    __syncthreads();
    uint64_t* desc = reinterpret_cast<uint64_t*>(ws + ws_desc_offset(g.num_layers));
    const uint64_t* texcl = desc + g.total_tiles;
    const uint32_t T = g.total_tiles;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    for (uint32_t q = blockIdx.x; q < T; q += gridDim.x) {
        const uint32_t t = T - 1u - q;
        TileGeo G;
        G.layer = layer_from(lays, g.num_layers, t, 0);
        const KLayer& ly = lays[G.layer];
        G.first_bin = (t - ly.tile_begin) * ly.bins_per_tile;
        G.bins = (int)min(ly.bins_per_tile, ly.nbins - G.first_bin);
        G.ts = (int64_t)G.first_bin * ly.bin_len;
        G.tl = (int)min((int64_t)G.bins * ly.bin_len, ly.n - G.ts);
        const LayerWs* lw = reinterpret_cast<const LayerWs*>(ws + ws_layer_offset(G.layer));
        if (lw->result.status == 0u) {
            // exclusive prefix of this tile's per-bin counts (4 bins per thread)
            const uint16_t* cnt = reinterpret_cast<const uint16_t*>(ly.msg + 8) + G.first_bin;
            uint32_t c[4], loc = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int b = tid * 4 + k;
                c[k] = b < G.bins ? cnt[b] : 0u;
                loc += c[k];
            }
            uint32_t incl = loc;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                uint32_t y = __shfl_up_sync(kFull, incl, o);
                if (lane >= o) incl += y;
            }
            if (lane == 31) wsum[warp] = incl;
            __syncthreads();
            uint32_t woff = 0, total = 0;
            for (int w = 0; w < kFixThreads / 32; ++w) {
                if (w < warp) woff += wsum[w];
                total += wsum[w];
            }
            uint32_t run = woff + incl - loc;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int b = tid * 4 + k;
                if (b < G.bins) pre[b] = run;
                run += c[k];
            }
            __syncthreads();
            const float s = lw->result.s;
            const uint8_t* codes = ly.msg + 8 + 2ull * ly.nbins + (unsigned long long)ly.code_bytes * texcl[t];
            float* res = ly.residue + G.ts;
            for (uint32_t i = tid; i < total; i += kFixThreads) {
                int lo = 0, hi = G.bins - 1;  // last bin whose prefix is <= i
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (pre[mid] <= i) lo = mid;
                    else hi = mid - 1;
                }
                const uint32_t code = ly.code_bytes == 1 ? codes[i] : reinterpret_cast<const uint16_t*>(codes)[i];
                const int64_t off = (int64_t)lo * ly.bin_len + (code >> 1);
                if (off < G.tl) {  // always true for codes this call produced
                    float* r = res + off;
                    *r = (code & 1u) ? __fadd_rn(*r, s) : __fsub_rn(*r, s);
                }
            }
        }
        if (tid == 0) desc[t] = 0ull;
        __syncthreads();
    }
}

}  // namespace

// ---------------------------------------------------------------- host launcher
namespace {
struct DeviceInfo {
    int sms = 0;
    uint32_t smem_set = 0;  // largest dynamic shared memory opted in so far
};
DeviceInfo g_dev[64];
}  // namespace

cudaError_t launch_compress(const KGroup& g, void* ws, cudaStream_t stream, cudaEvent_t ev_before,
                            cudaEvent_t ev_mid, cudaEvent_t ev_after)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    DeviceInfo& di = g_dev[dev];
    if (di.sms == 0) {
        e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    const SmemPlan P = smem_plan(g.tile_cap, g.d_size, g.max_bins, g.num_layers, g.needs_gbuf);
    if (P.total > di.smem_set) {
        e = cudaFuncSetAttribute(compress_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P.total);
        if (e != cudaSuccess) return e;
        di.smem_set = P.total;
    }
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, compress_kernel, kCtaThreads, P.total);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    const long long cap = (long long)di.sms * occ;
    const uint32_t grid = (uint32_t)((long long)g.total_tiles < cap ? (long long)g.total_tiles : cap);
    if (ev_before && (e = cudaEventRecord(ev_before, stream)) != cudaSuccess) return e;
    {
        // all CTAs must be resident together: the look-back waits on other CTAs' tiles
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(kCtaThreads);
        cfg.dynamicSmemBytes = P.total;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, compress_kernel, g, static_cast<uint8_t*>(ws));
        if (e != cudaSuccess) return e;
    }
    if (ev_mid && (e = cudaEventRecord(ev_mid, stream)) != cudaSuccess) return e;
    finalize_kernel<<<g.num_layers, 32, 0, stream>>>(g, static_cast<uint8_t*>(ws));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const long long fcap = (long long)di.sms * 8;
    const uint32_t fgrid = (uint32_t)((long long)g.total_tiles < fcap ? (long long)g.total_tiles : fcap);
    fixup_kernel<<<fgrid, kFixThreads, g.num_layers * sizeof(KLayer), stream>>>(g, static_cast<uint8_t*>(ws));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (ev_after) e = cudaEventRecord(ev_after, stream);
    return e;
}

}  // namespace adacomp

// ---------------------------------------------------------------- compress without a caller workspace
// For callers that cannot allocate device memory (see adacomp_compress_static_ws in
// include/adacomp.h). The workspace lives in this file-scope array, which every GPU
// that loads the library holds until the process exits.
#include <atomic>
#include <cstddef>

#include "adacomp.h"

namespace {
constexpr size_t kStaticScratchBytes = size_t(1) << 20;  // 1 MiB
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
    const size_t zero_bytes = ws_desc_offset(1) + 8 * (size_t)g.total_tiles;
    if (cudaMemsetAsync(scratch, 0, zero_bytes, stream) != cudaSuccess) return ADACOMP_ERR_CUDA;
    if (launch_compress(g, scratch, stream) != cudaSuccess) return ADACOMP_ERR_CUDA;
    if (result_out) {
        const uint8_t* res = static_cast<const uint8_t*>(scratch) + ws_layer_offset(0) + offsetof(LayerWs, result);
        if (cudaMemcpyAsync(result_out, res, sizeof(Result), cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
            return ADACOMP_ERR_CUDA;
    }
    return ADACOMP_OK;
}
