// Device helpers shared by the compress kernels: bf16 widening, the selection
// probe, the segment chunk rotation, the exact sum of bin maxima from exponent
// buckets, the layer lookup of a tile, and the exponent bucketing of bin maxima.
#pragma once

#include "adacomp_internal.cuh"

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

// The value compared with g_max: H = fl32(G + dW) for AdaComp, G for Local
// Selection ("AdaComp (Adaptive Residual Gradient Compression)", Claims > Mechanism
// #r629-self-adjusting-sparsity-prevents-residual-explosion).
__device__ __forceinline__ float probe(float g, float d, bool ls) { return ls ? g : __fadd_rn(g, d); }

// Lanes own 16-slot segments; rotation of their four 16-byte chunks (see seg_geo).
constexpr int kSeg = 16;

__device__ __forceinline__ int seg_rot(int tid) { return ((tid >> 1) ^ (tid >> 3)) & 3; }

// ---------------------------------------------------------------- exact scale sum
// The layer's bin maxima arrive as integer mantissas bucketed by fp32 exponent:
// bucket E holds sum(M) over maxima with biased exponent E, where a value equals
// M * 2^(max(E,1) - 150). The exact sum is rebuilt as a 384-bit integer in units of
// 2^-149 and rounded once to the nearest fp64 (ties to even), so s does not depend
// on the order in which tiles finished.
//
// Warp-parallel: lane l shifts buckets 8l .. 8l+7 into place; their 32-bit pieces
// land in at most five consecutive words, which are added into `words` (twelve
// 64-bit partial sums in shared memory, zero on entry) with shared atomics. Lane 0
// then propagates the carries and rounds. Every lane returns the sum.
constexpr int kSumWords = 12;

__device__ double exact_sum_warp(const unsigned long long* acc, unsigned long long* words, int lane)
{
    if (acc[255] != 0ull) return __longlong_as_double(0x7ff0000000000000ll);  // non-finite input
    const int e_first = lane * 8;
    const int q0 = (e_first ? e_first - 1 : 0) >> 5;
    unsigned long long loc[5] = {0ull, 0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int e = e_first + j;
        const unsigned long long v = e < 255 ? acc[e] : 0ull;
        const int sh = e ? e - 1 : 0;
        const int dq = (sh >> 5) - q0;  // 0 or 1
        const int b = sh & 31;
        const unsigned long long lo = v << b;
        const unsigned long long hi = b ? (v >> (64 - b)) : 0ull;
        const unsigned long long p0 = lo & 0xffffffffull, p1 = lo >> 32, p2 = hi & 0xffffffffull, p3 = hi >> 32;
        if (dq == 0) { loc[0] += p0; loc[1] += p1; loc[2] += p2; loc[3] += p3; }
        else { loc[1] += p0; loc[2] += p1; loc[3] += p2; loc[4] += p3; }
    }
#pragma unroll
    for (int i = 0; i < 5; ++i)
        if (loc[i] && q0 + i < kSumWords) atomicAdd(&words[q0 + i], loc[i]);
    __syncwarp();
    double S = 0.0;
    if (lane == 0) {
        uint32_t w[kSumWords];
        unsigned long long carry = 0;
#pragma unroll
        for (int i = 0; i < kSumWords; ++i) {
            const unsigned long long t = words[i] + carry;
            w[i] = (uint32_t)t;
            carry = t >> 32;
        }
        int top = -1;
#pragma unroll
        for (int i = kSumWords - 1; i >= 0; --i)
            if (top < 0 && w[i]) top = i * 32 + 31 - __clz(w[i]);
        if (top >= 0) {
            const int lo = top - 52;  // weight of the last kept bit
            unsigned long long mant;
            int scale;
            if (lo <= 0) {
                mant = ((unsigned long long)w[1] << 32) | w[0];  // exact: fewer than 54 bits
                scale = -149;
            } else {
                const int q = lo >> 5, off = lo & 31;
                unsigned long long x = 0, x2 = 0;
#pragma unroll
                for (int i = 0; i < kSumWords; ++i) {
                    if (i == q) x |= w[i];
                    if (i == q + 1) x |= (unsigned long long)w[i] << 32;
                    if (i == q + 2) x2 = w[i];
                }
                mant = off ? ((x >> off) | (x2 << (64 - off))) : x;
                mant &= (1ull << 53) - 1;
                const int rb = lo - 1;  // round bit; the sticky bits lie below it
                uint32_t round = 0, sticky = 0;
#pragma unroll
                for (int i = 0; i < kSumWords; ++i) {
                    const int base = i * 32;
                    if (rb >= base && rb < base + 32) round = (w[i] >> (rb - base)) & 1u;
                    if (base + 32 <= rb) sticky |= w[i];
                    else if (base < rb) sticky |= w[i] & ((1u << (rb - base)) - 1u);
                }
                if (round && (sticky || (mant & 1ull))) ++mant;  // may carry to 2^53: still exact
                scale = lo - 149;
            }
            // mant * 2^scale, both exact in fp64 (scale lies well inside the normal range)
            S = __dmul_rn((double)mant, __longlong_as_double((long long)(scale + 1023) << 52));
        }
    }
    __syncwarp();
    return __shfl_sync(0xffffffffu, S, 0);
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


// Exponent buckets of 32 bin maxima (one per lane, 0 for none): the largest
// exponent present and the one below it are summed with one warp reduction each
// (at most 32 x 2^24 < 2^32); any other exponent is summed in a loop. Lane 0 adds
// each sum to the warp's shared buckets, or, for an exponent outside their window,
// to the layer's accumulator gacc.
// The shared buckets cover biased exponents [kLo, kLo + kN).
template <int kLo = kHistLo, int kN = kHistN>
__device__ __forceinline__ void bucket_add(unsigned long long* hist, unsigned long long* gacc, uint32_t E,
                                           uint32_t v)
{
    if (E - kLo < (uint32_t)kN) hist[E - kLo] += (unsigned long long)v;
    else atomicAdd(&gacc[E], (unsigned long long)v);
}

template <int kLo = kHistLo, int kN = kHistN>
__device__ __forceinline__ void bucket_group(uint32_t u, unsigned long long* hist, unsigned long long* gacc, int lane)
{
    if (__ballot_sync(kFull, u != 0u) == 0u) return;
    const uint32_t E = u >> 23;
    const uint32_t M = E ? ((u & 0x7fffffu) | 0x800000u) : (u & 0x7fffffu);
    const uint32_t Eh = __reduce_max_sync(kFull, u ? E : 0u);
    const uint32_t s_hi = __reduce_add_sync(kFull, (u && E == Eh) ? M : 0u);
    const uint32_t s_lo = __reduce_add_sync(kFull, (u && Eh > 0 && E == Eh - 1) ? M : 0u);
    if (lane == 0) {
        if (s_hi) bucket_add<kLo, kN>(hist, gacc, Eh, s_hi);
        if (s_lo) bucket_add<kLo, kN>(hist, gacc, Eh - 1, s_lo);
    }
    uint32_t left = __ballot_sync(kFull, u != 0u && E + 1 < Eh);
    while (left) {
        const uint32_t Ek = __shfl_sync(kFull, E, __ffs(left) - 1);
        const bool mine = ((left >> lane) & 1u) && E == Ek;
        const uint32_t sum = __reduce_add_sync(kFull, mine ? M : 0u);
        if (lane == 0) bucket_add<kLo, kN>(hist, gacc, Ek, sum);
        left &= ~__ballot_sync(kFull, mine);
    }
    __syncwarp();
}

// Adds a warp's buckets to layer lw's accumulator and clears them.
template <int kLo = kHistLo, int kN = kHistN>
__device__ __forceinline__ void flush_buckets(unsigned long long* hist, LayerWs* lw, int lane)
{
    __syncwarp();
    for (int e = lane; e < kN; e += 32) {
        const unsigned long long v = hist[e];
        if (v) {
            atomicAdd(&lw->acc[kLo + e], v);
            hist[e] = 0ull;
        }
    }
    __syncwarp();
}


}  // namespace
}  // namespace adacomp
