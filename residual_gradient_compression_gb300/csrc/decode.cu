// AdaComp decode-and-accumulate for sm_103a: K learners' sparse ternary messages
// are summed into one dense fp32 gradient, learner by learner.
//
// The pages say only that data-parallel learners exchange their quantised
// gradients ("AdaComp (Adaptive Residual Gradient Compression)", abstract and
// summary paragraph); this library reads the combination as a plain sum in learner
// order, dense[j] = fl32(dense[j] + sign * s_k) for k = 0..K-1.
//
// Three launches:
//   tile_sums   per (learner, tile): validate the header and the tile's per-bin
//               counts, and sum the counts;
//   tile_scan   per (layer, learner): exclusive prefix of the tile sums, i.e. where
//               each tile's codes start in that message;
//   accumulate  per tile: the dense tile is staged in shared memory, every learner's
//               codes for the tile are applied in learner order (a barrier between
//               learners), and the tile is written back. One CTA owns each tile, no
//               two threads touch one element within a learner, and no float atomics
//               are used, so the result is deterministic.
#include "adacomp_internal.cuh"

namespace adacomp {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kDecThreads = 256;

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

__device__ __forceinline__ uint64_t* tile_offsets(uint8_t* ws, int k, uint32_t T)
{
    return reinterpret_cast<uint64_t*>(ws + kDecodeFixed + (size_t)k * decode_per_learner(T));
}

// One warp per (learner k, tile t): header B must equal the layer's B, and no
// count may exceed its bin's length; otherwise the tile sum is kBadOffset.
__global__ void __launch_bounds__(kDecThreads) tile_sums_kernel(const __grid_constant__ KGroup g,
                                                                const __grid_constant__ DecodeParams p, uint8_t* ws)
{
    const uint32_t T = g.total_tiles;
    const int K = p.K;
    const int lane = threadIdx.x & 31;
    const uint64_t nwarps = (uint64_t)gridDim.x * (kDecThreads / 32);
    for (uint64_t task = (uint64_t)blockIdx.x * (kDecThreads / 32) + (threadIdx.x >> 5); task < (uint64_t)K * T;
         task += nwarps) {
        const int k = (int)(task / T);
        const uint32_t t = (uint32_t)(task - (uint64_t)k * T);
        const int l = find_layer(g, t);
        const KLayer& ly = g.layer[l];
        const uint8_t* msg = p.msg[l * K + k];
        const uint32_t first_bin = (t - ly.tile_begin) * ly.bins_per_tile;
        const int bins = (int)min(ly.bins_per_tile, ly.nbins - first_bin);
        bool ok = *reinterpret_cast<const uint32_t*>(msg + 4) == ly.nbins;
        uint32_t sum = 0;
        if (ok) {
            const uint16_t* cnt = reinterpret_cast<const uint16_t*>(msg + 8) + first_bin;
            const int64_t last_len = ly.n - (int64_t)(ly.nbins - 1) * ly.bin_len;
            for (int b = lane; b < bins; b += 32) {
                const uint32_t c = cnt[b];
                const int64_t len = (first_bin + b == ly.nbins - 1) ? last_len : ly.bin_len;
                ok = ok && (int64_t)c <= len;
                sum += c;
            }
        }
        ok = __all_sync(kFull, ok);
#pragma unroll
        for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
        if (lane == 0) tile_offsets(ws, k, T)[t] = ok ? (uint64_t)sum : kBadOffset;
    }
}

// One CTA per (layer, learner): tile sums -> exclusive offsets, in place. A layer
// message with any bad tile is marked bad as a whole.
__global__ void __launch_bounds__(1024) tile_scan_kernel(const __grid_constant__ KGroup g,
                                                         const __grid_constant__ DecodeParams p, uint8_t* ws)
{
    __shared__ uint32_t wsum[32];
    __shared__ uint32_t bad_s;
    const int K = p.K;
    const int l = blockIdx.x / K, k = blockIdx.x - (blockIdx.x / K) * K;
    const KLayer& ly = g.layer[l];
    uint64_t* off = tile_offsets(ws, k, g.total_tiles) + ly.tile_begin;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (blockIdx.x == 0 && tid == 0) {
        reinterpret_cast<uint32_t*>(ws)[0] = (uint32_t)K;
        reinterpret_cast<uint32_t*>(ws)[1] = (uint32_t)g.num_layers;
    }
    if (tid == 0) bad_s = 0u;
    __syncthreads();
    uint64_t carry = 0;
    for (uint32_t base = 0; base < ly.num_tiles; base += 1024) {
        const uint32_t i = base + tid;
        const uint64_t v = i < ly.num_tiles ? off[i] : 0ull;
        if (v == kBadOffset) bad_s = 1u;
        const uint32_t x = v == kBadOffset ? 0u : (uint32_t)v;
        uint32_t incl = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        uint64_t woff = 0, tot = 0;
        for (int w = 0; w < 32; ++w) {
            if (w < warp) woff += wsum[w];
            tot += wsum[w];
        }
        if (i < ly.num_tiles) off[i] = carry + woff + incl - x;
        carry += tot;
        __syncthreads();
    }
    const bool bad = bad_s != 0u;
    if (bad)
        for (uint32_t i = tid; i < ly.num_tiles; i += 1024) off[i] = kBadOffset;
    if (tid == 0) ws[16 + l * K + k] = bad ? 1 : 0;
}

// Grid-stride over tiles; dynamic shared memory = dense tile + count prefix.
__global__ void __launch_bounds__(kDecThreads) accumulate_kernel(const __grid_constant__ KGroup g,
                                                                 const __grid_constant__ DecodeParams p, uint8_t* ws)
{
    extern __shared__ __align__(16) uint8_t smem[];
    float* sd = reinterpret_cast<float*>(smem);
    uint32_t* pre = reinterpret_cast<uint32_t*>(smem + ((g.tile_cap + 8) * 4 + 15) / 16 * 16);
    __shared__ uint32_t wsum[kDecThreads / 32];
    const uint32_t T = g.total_tiles;
    const int K = p.K;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    for (uint32_t t = blockIdx.x; t < T; t += gridDim.x) {
        const int l = find_layer(g, t);
        const KLayer& ly = g.layer[l];
        const uint32_t first_bin = (t - ly.tile_begin) * ly.bins_per_tile;
        const int bins = (int)min(ly.bins_per_tile, ly.nbins - first_bin);
        const int64_t ts = (int64_t)first_bin * ly.bin_len;
        const int tl = (int)min((int64_t)bins * ly.bin_len, ly.n - ts);
        const int64_t te = ts + tl;
        const int ph = (int)(ts & 3);
        float* dense = p.dense[l];
        const int64_t last_len = ly.n - (int64_t)(ly.nbins - 1) * ly.bin_len;

        // stage the dense tile: 16-byte vectors over the aligned interior
        const int64_t c0 = (ts + 3) & ~(int64_t)3, c1 = te & ~(int64_t)3;
        if (c1 > c0) {
            const float4* src = reinterpret_cast<const float4*>(dense + c0);
            float4* dst = reinterpret_cast<float4*>(sd + ph + (c0 - ts));
            for (int64_t v = tid; v < (c1 - c0) / 4; v += kDecThreads) dst[v] = src[v];
            for (int64_t j = ts + tid; j < c0; j += kDecThreads) sd[ph + (j - ts)] = dense[j];
            for (int64_t j = c1 + tid; j < te; j += kDecThreads) sd[ph + (j - ts)] = dense[j];
        } else {
            for (int64_t j = ts + tid; j < te; j += kDecThreads) sd[ph + (j - ts)] = dense[j];
        }
        __syncthreads();

        for (int k = 0; k < K; ++k) {
            const uint64_t off = tile_offsets(ws, k, T)[t];
            if (off == kBadOffset) continue;
            const uint8_t* msg = p.msg[l * K + k];
            const float s = *reinterpret_cast<const float*>(msg);
            // exclusive prefix of the tile's counts (4 bins per thread)
            const uint16_t* cnt = reinterpret_cast<const uint16_t*>(msg + 8) + first_bin;
            uint32_t c[4], loc = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int b = tid * 4 + q;
                c[q] = b < bins ? cnt[b] : 0u;
                loc += c[q];
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
            for (int w = 0; w < kDecThreads / 32; ++w) {
                if (w < warp) woff += wsum[w];
                total += wsum[w];
            }
            uint32_t run = woff + incl - loc;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int b = tid * 4 + q;
                if (b < bins) pre[b] = run;
                run += c[q];
            }
            __syncthreads();
            const uint8_t* codes = msg + 8 + 2ull * ly.nbins + (unsigned long long)ly.code_bytes * off;
            for (uint32_t i = tid; i < total; i += kDecThreads) {
                int lo = 0, hi = bins - 1;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (pre[mid] <= i) lo = mid;
                    else hi = mid - 1;
                }
                const uint32_t code = ly.code_bytes == 1 ? codes[i] : reinterpret_cast<const uint16_t*>(codes)[i];
                const uint32_t o = code >> 1;
                const int64_t len = (first_bin + lo == ly.nbins - 1) ? last_len : ly.bin_len;
                if ((int64_t)o < len) {
                    float* x = sd + ph + (int64_t)lo * ly.bin_len + o;
                    *x = __fadd_rn(*x, (code & 1u) ? -s : s);
                } else {
                    ws[16 + l * K + k] = 1;  // offset outside its bin: ignored, message flagged
                }
            }
            __syncthreads();
        }

        if (c1 > c0) {
            float4* dst = reinterpret_cast<float4*>(dense + c0);
            const float4* src = reinterpret_cast<const float4*>(sd + ph + (c0 - ts));
            for (int64_t v = tid; v < (c1 - c0) / 4; v += kDecThreads) dst[v] = src[v];
            for (int64_t j = ts + tid; j < c0; j += kDecThreads) dense[j] = sd[ph + (j - ts)];
            for (int64_t j = c1 + tid; j < te; j += kDecThreads) dense[j] = sd[ph + (j - ts)];
        } else {
            for (int64_t j = ts + tid; j < te; j += kDecThreads) dense[j] = sd[ph + (j - ts)];
        }
        __syncthreads();
    }
}

struct DecDeviceInfo {
    int sms = 0;
    uint32_t smem_set = 0;
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
    const uint64_t tasks = (uint64_t)p.K * g.total_tiles;
    const uint64_t wpb = kDecThreads / 32;
    uint64_t sgrid = (tasks + wpb - 1) / wpb;
    if (sgrid > (uint64_t)di.sms * 16) sgrid = (uint64_t)di.sms * 16;
    tile_sums_kernel<<<(unsigned)sgrid, kDecThreads, 0, stream>>>(g, p, w);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    tile_scan_kernel<<<(unsigned)(g.num_layers * p.K), 1024, 0, stream>>>(g, p, w);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const uint32_t smem = (uint32_t)(((g.tile_cap + 8) * 4 + 15) / 16 * 16 + (g.max_bins + 1) * 4);
    if (smem > di.smem_set) {
        if (smem > 48 * 1024) {
            e = cudaFuncSetAttribute(accumulate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
        }
        di.smem_set = smem;
    }
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, accumulate_kernel, kDecThreads, smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    const long long cap = (long long)di.sms * occ;
    const uint32_t grid = (uint32_t)((long long)g.total_tiles < cap ? (long long)g.total_tiles : cap);
    accumulate_kernel<<<grid, kDecThreads, smem, stream>>>(g, p, w);
    return cudaGetLastError();
}

}  // namespace adacomp
