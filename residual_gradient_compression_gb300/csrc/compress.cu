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
    float* sr;      // residue slice; element i at sr[pr + i]; phase A overwrites it with G
    const void* sd; // dW slice; element i at sd[pd + i]
    int pr, pd;
    int tl;         // elements in the tile
    int L;          // bin length
    int bins;       // bins in the tile (last bin may be partial)
    int cpb;        // chunks per bin
    int ch;         // chunk length (elements, multiple of VEC)
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
                store_g<VEC>(T.sr, T.pr + i, g);
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
                load_g<VEC>(T.sr, T.pr + i, g);
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
// layer. Publishes AGGREGATE(total), walks back 32 descriptors at a time until an
// INCLUSIVE one, then publishes INCLUSIVE(prefix + total). Every wait is bounded by
// timeout_ns of global time; on expiry (or a predecessor's error) the tile is
// published as ERROR and the function returns false.
__device__ bool lookback(uint64_t* desc, uint32_t t, uint32_t tile_begin, uint32_t total, uint64_t timeout_ns,
                         int lane, uint64_t* excl_out)
{
    if (t == tile_begin) {
        if (lane == 0) ptx::st_relaxed(&desc[t], kFlagIncl | total);
        *excl_out = 0;
        return true;
    }
    if (lane == 0) ptx::st_relaxed(&desc[t], kFlagAgg | total);
    uint64_t excl = 0;
    int64_t j = (int64_t)t - 1;
    uint64_t start = 0;
    uint32_t sleep_ns = 32;
    bool ok = true;
    for (;;) {
        const int64_t idx = j - lane;
        const uint64_t dv = idx >= (int64_t)tile_begin ? ptx::ld_relaxed(&desc[idx]) : kFlagIncl;
        const uint32_t flag = (uint32_t)(dv >> 62);
        const uint32_t incl = __ballot_sync(kFull, flag >= 2u);
        const uint32_t lim = incl ? (uint32_t)(__ffs(incl) - 1) : 31u;
        const uint32_t needed = (2u << lim) - 1u;
        const uint32_t pending = __ballot_sync(kFull, flag == 0u) & needed;
        if (pending == 0u) {
            if (__ballot_sync(kFull, flag == 3u) & needed) { ok = false; break; }
            unsigned long long v = ((uint32_t)lane <= lim) ? (dv & kValueMask) : 0ull;
#pragma unroll
            for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
            excl += v;
            if (incl) break;
            j -= 32;
            start = 0;
            continue;
        }
        uint64_t now = 0;
        if (lane == 0) now = ptx::globaltimer();
        now = __shfl_sync(kFull, now, 0);
        if (start == 0) start = now;
        else if (now - start > timeout_ns) { ok = false; break; }
        __nanosleep(sleep_ns);
        if (sleep_ns < 1024) sleep_ns <<= 1;
    }
    if (lane == 0) ptx::st_relaxed(&desc[t], ok ? (kFlagIncl | (excl + total)) : kFlagErr);
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

__device__ __forceinline__ int find_layer(const KGroup& g, uint32_t t)
{
    int lo = 0, hi = g.num_layers - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (g.layer[mid].tile_begin <= t) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// ---------------------------------------------------------------- tile geometry
struct TileGeo {
    int layer;
    int64_t ts;          // first element of the tile within its layer
    int tl;              // elements in the tile
    uint32_t first_bin;
    int bins;
};

__device__ __forceinline__ TileGeo tile_geo(const KGroup& g, uint32_t t)
{
    TileGeo G;
    G.layer = find_layer(g, t);
    const KLayer& ly = g.layer[G.layer];
    G.first_bin = (t - ly.tile_begin) * ly.bins_per_tile;
    G.bins = (int)min(ly.bins_per_tile, ly.nbins - G.first_bin);
    G.ts = (int64_t)G.first_bin * ly.bin_len;
    G.tl = (int)min((int64_t)G.bins * ly.bin_len, ly.n - G.ts);
    return G;
}

// Issues the bulk copies of tile t's residue and dW slices into one stage. Each copy
// covers the slice's 16-byte-aligned span that starts at or before the tile; the
// last few elements past the final 16-byte boundary are loaded with plain loads
// after the wait, so nothing outside the arrays is read.
__device__ void issue_load(const KGroup& g, uint32_t t, float* sr, void* sd, uint64_t* bar)
{
    const TileGeo G = tile_geo(g, t);
    const KLayer& ly = g.layer[G.layer];
    const int64_t a0 = G.ts & ~3ll, a1 = (G.ts + G.tl) & ~3ll;
    const uint32_t rb = a1 > a0 ? (uint32_t)(a1 - a0) * 4u : 0u;
    int64_t b0 = a0;
    uint32_t db = rb;
    if (ly.dw_bf16) {
        b0 = G.ts & ~7ll;
        const int64_t b1 = (G.ts + G.tl) & ~7ll;
        db = b1 > b0 ? (uint32_t)(b1 - b0) * 2u : 0u;
    }
    ptx::mbar_arrive_expect_tx(bar, rb + db);
    if (rb) ptx::bulk_g2s(sr, ly.residue + a0, rb, bar);
    if (db) ptx::bulk_g2s(sd, static_cast<const uint8_t*>(ly.dw) + b0 * (ly.dw_bf16 ? 2 : 4), db, bar);
}

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
// Persistent: each CTA takes tiles from a ticket counter in increasing order, so
// every tile's predecessors are already running or done and the look-back cannot
// deadlock. Two stages: the next tile's bulk copies are in flight while the
// current one is processed.
__global__ void __launch_bounds__(kThreads) compress_kernel(const __grid_constant__ KGroup g, uint8_t* __restrict__ ws)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const SmemPlan P = smem_plan(g.tile_cap, g.d_size, g.max_bins);
    uint8_t* p = smem;
    float* sr[2];
    void* sd[2];
    sr[0] = reinterpret_cast<float*>(p); p += P.r_bytes;
    sd[0] = p; p += P.d_bytes;
    sr[1] = reinterpret_cast<float*>(p); p += P.r_bytes;
    sd[1] = p; p += P.d_bytes;
    uint16_t* stg = reinterpret_cast<uint16_t*>(p); p += P.stg_bytes;
    uint32_t* gmax_s = reinterpret_cast<uint32_t*>(p); p += P.bin_bytes;
    uint32_t* cnt_s = reinterpret_cast<uint32_t*>(p); p += P.bin_bytes;
    unsigned long long* hist = reinterpret_cast<unsigned long long*>(p); p += 2048;
    uint64_t* bar = reinterpret_cast<uint64_t*>(p); p += 16;
    uint32_t* wtot = reinterpret_cast<uint32_t*>(p);         // [8] codes per warp
    uint32_t* wexcl = wtot + 8;                              // [8] warp prefix
    int32_t* wbase = reinterpret_cast<int32_t*>(wtot + 16);  // [8] staging base per warp
    uint32_t* tk = wtot + 24;                                // [2] held tickets
    uint32_t* flags = wtot + 26;                             // [0] layer+1 to finalise, [1] prefix ok
    unsigned long long* bexcl = reinterpret_cast<unsigned long long*>(wtot + 28);

    Ctl* ctl = reinterpret_cast<Ctl*>(ws);
    uint64_t* desc = reinterpret_cast<uint64_t*>(ws + ws_desc_offset(g.num_layers));
    uint64_t* texcl = desc + g.total_tiles;
    const uint32_t T = g.total_tiles;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    for (int e = tid; e < 256; e += kThreads) hist[e] = 0ull;
    if (tid == 0) {
        ptx::mbar_init(&bar[0], 1);
        ptx::mbar_init(&bar[1], 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        uint32_t t0 = atomicAdd(&ctl->ticket, 1u), t1 = T;
        if (t0 < T) {
            issue_load(g, t0, sr[0], sd[0], &bar[0]);
            t1 = atomicAdd(&ctl->ticket, 1u);
            if (t1 < T) issue_load(g, t1, sr[1], sd[1], &bar[1]);
            else t1 = T;
        } else {
            t0 = T;
        }
        tk[0] = t0;
        tk[1] = t1;
    }
    __syncthreads();

    uint32_t it = 0;
    bool poisoned = false;
    for (;;) {
        const uint32_t t = tk[0];
        if (t >= T) break;
        const int s = it & 1;
        const uint32_t parity = (it >> 1) & 1u;
        const TileGeo G = tile_geo(g, t);
        const KLayer& ly = g.layer[G.layer];
        LayerWs* lw = reinterpret_cast<LayerWs*>(ws + ws_layer_offset(G.layer));

        if (!__syncthreads_and(wait_stage(&bar[s], parity, g.timeout_ns))) { poisoned = true; break; }

        // tail elements past the last 16-byte boundary; clear per-bin arrays
        const int pr = (int)(G.ts & 3), pd = ly.dw_bf16 ? (int)(G.ts & 7) : pr;
        float* r_s = sr[s];
        void* d_s = sd[s];
        const int64_t te = G.ts + G.tl;
        for (int64_t j = max((int64_t)(te & ~(int64_t)3), G.ts) + tid; j < te; j += kThreads) r_s[pr + (j - G.ts)] = ly.residue[j];
        if (ly.dw_bf16) {
            for (int64_t j = max((int64_t)(te & ~(int64_t)7), G.ts) + tid; j < te; j += kThreads)
                static_cast<uint16_t*>(d_s)[pd + (j - G.ts)] = static_cast<const uint16_t*>(ly.dw)[j];
        } else {
            for (int64_t j = max((int64_t)(te & ~(int64_t)3), G.ts) + tid; j < te; j += kThreads)
                static_cast<float*>(d_s)[pd + (j - G.ts)] = static_cast<const float*>(ly.dw)[j];
        }
        for (int b = tid; b < G.bins; b += kThreads) { gmax_s[b] = 0u; cnt_s[b] = 0u; }
        __syncthreads();

        Tile Tl;
        Tl.sr = r_s; Tl.sd = d_s; Tl.pr = pr; Tl.pd = pd; Tl.tl = G.tl; Tl.L = ly.bin_len; Tl.bins = G.bins;
        Tl.ch = min(ly.bin_len, 32 * (int)ly.vec * kRounds);
        Tl.cpb = (ly.bin_len + Tl.ch - 1) / Tl.ch;
        const int nchunks = G.bins * Tl.cpb;
        const int cpw = (nchunks + kWarps - 1) / kWarps;
        const int c_begin = min(nchunks, warp * cpw), c_end = min(nchunks, c_begin + cpw);

        // phase A: G and bin maxima
        ADACOMP_DISPATCH(ly.vec, ly.dw_bf16, (phase_a<VEC, BF16>(Tl, c_begin, c_end, gmax_s, lane)))
        ptx::fence_proxy_async_smem();
        __syncthreads();

        // residue := G for the whole tile (sent elements are corrected by the fix-up kernel)
        {
            const int64_t c0 = (G.ts + 3) & ~3ll, c1 = te & ~3ll;
            if (c1 > c0) {
                if (tid == 0) {
                    ptx::bulk_s2g(ly.residue + c0, r_s + pr + (c0 - G.ts), (uint32_t)(c1 - c0) * 4u);
                    ptx::bulk_commit();
                }
                for (int64_t j = G.ts + tid; j < c0; j += kThreads) ly.residue[j] = r_s[pr + (j - G.ts)];
                for (int64_t j = c1 + tid; j < te; j += kThreads) ly.residue[j] = r_s[pr + (j - G.ts)];
            } else {
                for (int64_t j = G.ts + tid; j < te; j += kThreads) ly.residue[j] = r_s[pr + (j - G.ts)];
            }
        }

        // phase C: selection, per-bin counts, codes staged in element order
        const int stg_base = c_begin < c_end ? chunk_at(Tl, c_begin).e0 : 0;
        uint32_t wt = 0;
        ADACOMP_DISPATCH(ly.vec, ly.dw_bf16,
                         (wt = phase_c<VEC, BF16>(Tl, c_begin, c_end, gmax_s, cnt_s, stg, stg_base, lane)))
        if (lane == 0) { wtot[warp] = wt; wbase[warp] = stg_base; }
        __syncthreads();

        if (warp == 0) {
            // block scan over warps, then the look-back across tiles
            const uint32_t v = lane < kWarps ? wtot[lane] : 0u;
            uint32_t incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                uint32_t y = __shfl_up_sync(kFull, incl, o);
                if (lane >= o) incl += y;
            }
            if (lane < kWarps) wexcl[lane] = incl - v;
            const uint32_t total = __shfl_sync(kFull, incl, 31);
            uint64_t ex = 0;
            const bool okl = lookback(desc, t, ly.tile_begin, total, g.timeout_ns, lane, &ex);
            if (lane == 0) {
                *bexcl = ex;
                flags[1] = okl ? 1u : 0u;
                if (okl) texcl[t] = ex;
                else atomicOr(&lw->err, kErrTimeout);
            }
        } else if (warp == 1) {
            // exact sum of the tile's bin maxima, bucketed by exponent
            for (int b0 = 0; b0 < G.bins; b0 += 32) {
                const int b = b0 + lane;
                const uint32_t u = b < G.bins ? gmax_s[b] : 0u;
                const uint32_t E = u >> 23;
                const uint32_t M = E ? ((u & 0x7fffffu) | 0x800000u) : (u & 0x7fffffu);
                const uint32_t key = u ? E : 0x100u;
                const uint32_t peers = __match_any_sync(kFull, key);
                const uint32_t sum = __reduce_add_sync(peers, M);
                if (key != 0x100u && lane == __ffs(peers) - 1) hist[E] += sum;
                __syncwarp();
            }
            for (int e = lane; e < 256; e += 32) {
                const unsigned long long v = hist[e];
                if (v) {
                    atomicAdd(&lw->acc[e], v);
                    hist[e] = 0ull;
                }
            }
            __threadfence();
        } else {
            uint16_t* cdst = reinterpret_cast<uint16_t*>(ly.msg + 8) + G.first_bin;
            for (int b = tid - 64; b < G.bins; b += kThreads - 64) cdst[b] = (uint16_t)cnt_s[b];
        }
        __syncthreads();

        if (tid == 0) {
            __threadfence();
            const uint32_t old = atomicAdd(&lw->done, 1u);
            flags[0] = (old + 1u == ly.num_tiles) ? (uint32_t)G.layer + 1u : 0u;
        }
        if (flags[1]) {
            const uint32_t nw = wtot[warp];
            const unsigned long long base = *bexcl + wexcl[warp];
            const int sb = wbase[warp];
            uint8_t* codes = ly.msg + 8 + 2ull * ly.nbins;
            if (ly.code_bytes == 1) {
                for (uint32_t k = lane; k < nw; k += 32) codes[base + k] = (uint8_t)stg[sb + k];
            } else {
                uint16_t* c16 = reinterpret_cast<uint16_t*>(codes);
                for (uint32_t k = lane; k < nw; k += 32) c16[base + k] = stg[sb + k];
            }
        }
        if (tid == 0) {
            ptx::bulk_wait_read0();  // stage s is free once its G store has been read
            const uint32_t nxt = tk[1];
            uint32_t nn = T;
            if (nxt < T) {
                nn = atomicAdd(&ctl->ticket, 1u);
                if (nn < T) issue_load(g, nn, sr[s], sd[s], &bar[s]);
                else nn = T;
            }
            tk[0] = nxt;
            tk[1] = nn;
        }
        __syncthreads();
        if (flags[0]) {
            const int l = (int)flags[0] - 1;
            if (warp == 0)
                finalize_layer(g.layer[l], reinterpret_cast<LayerWs*>(ws + ws_layer_offset(l)), desc, hist, lane);
            __syncthreads();
        }
        ++it;
    }

    if (poisoned) {
        // A bulk copy never completed: retire the held tiles as errors so their
        // layers still finalise, then give the copies one more bounded wait before
        // the CTA's shared memory is released.
        for (int h = 0; h < 2; ++h) {
            const uint32_t t = tk[h];
            if (t < T) {
                const int l = find_layer(g, t);
                LayerWs* lw = reinterpret_cast<LayerWs*>(ws + ws_layer_offset(l));
                if (tid == 0) {
                    ptx::st_relaxed(&desc[t], kFlagErr);
                    atomicOr(&lw->err, kErrTimeout);
                    __threadfence();
                    const uint32_t old = atomicAdd(&lw->done, 1u);
                    flags[0] = (old + 1u == g.layer[l].num_tiles) ? 1u : 0u;
                }
                __syncthreads();
                if (flags[0] && warp == 0) finalize_layer(g.layer[l], lw, desc, hist, lane);
                __syncthreads();
            }
        }
        wait_stage(&bar[it & 1], (it >> 1) & 1u, g.timeout_ns);
        if (tk[1] < T) wait_stage(&bar[(it + 1) & 1], ((it + 1) >> 1) & 1u, g.timeout_ns);
        __syncthreads();
    }
    if (tid == 0) ptx::bulk_wait0();
}

// ---------------------------------------------------------------- fix-up kernel
// For every sent element: residue = fl32(G - s) if G > 0, fl32(G + s) if G < 0
// (the residue still holds G). Tiles are visited in reverse ticket order, so the
// most recently written residue lines are the likeliest to still be in L2. Also
// returns the look-back state to zero for the next call.
constexpr int kFixThreads = 256;

__global__ void __launch_bounds__(kFixThreads) fixup_kernel(const __grid_constant__ KGroup g, uint8_t* __restrict__ ws)
{
    __shared__ uint32_t pre[kMaxBinsPerTile + 1];
    __shared__ uint32_t wsum[kFixThreads / 32];
    Ctl* ctl = reinterpret_cast<Ctl*>(ws);
    uint64_t* desc = reinterpret_cast<uint64_t*>(ws + ws_desc_offset(g.num_layers));
    const uint64_t* texcl = desc + g.total_tiles;
    const uint32_t T = g.total_tiles;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (blockIdx.x == 0 && tid == 0) ctl->ticket = 0u;

    for (uint32_t q = blockIdx.x; q < T; q += gridDim.x) {
        const uint32_t t = T - 1u - q;
        const TileGeo G = tile_geo(g, t);
        const KLayer& ly = g.layer[G.layer];
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
    const SmemPlan P = smem_plan(g.tile_cap, g.d_size, g.max_bins);
    if (P.total > di.smem_set) {
        e = cudaFuncSetAttribute(compress_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P.total);
        if (e != cudaSuccess) return e;
        di.smem_set = P.total;
    }
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, compress_kernel, kThreads, P.total);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    const long long cap = (long long)di.sms * occ;
    const uint32_t grid = (uint32_t)((long long)g.total_tiles < cap ? (long long)g.total_tiles : cap);
    if (ev_before && (e = cudaEventRecord(ev_before, stream)) != cudaSuccess) return e;
    compress_kernel<<<grid, kThreads, P.total, stream>>>(g, static_cast<uint8_t*>(ws));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (ev_mid && (e = cudaEventRecord(ev_mid, stream)) != cudaSuccess) return e;
    const long long fcap = (long long)di.sms * 8;
    const uint32_t fgrid = (uint32_t)((long long)g.total_tiles < fcap ? (long long)g.total_tiles : fcap);
    fixup_kernel<<<fgrid, kFixThreads, 0, stream>>>(g, static_cast<uint8_t*>(ws));
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

#include "../../include/adacomp.h"

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
