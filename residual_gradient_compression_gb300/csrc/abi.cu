// C ABI of libadacomp.so (declared in include/adacomp.h): handles, argument
// checks, workspace sizing and launches. The library allocates no device memory;
// every buffer and stream comes from the caller.
#include "adacomp_internal.cuh"

#include <cstddef>
#include <cstring>
#include <new>
#include <vector>

#include "adacomp.h"
#include <nvtx3/nvToolsExt.h>

struct adacomp_layer {
    std::vector<adacomp::KLayer> layers;  // device pointers are filled in per call
    uint32_t total_tiles = 0;
    uint32_t tile_cap = 0;
    uint16_t max_bins = 0;
    uint16_t d_size = 2;
    uint64_t timeout_ns = 2000000000ull;
    size_t compress_ws = 0;
    size_t decode_per_learner = 0;
    cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};  // optional timing events
    uint32_t inject_skip_tile = 0xffffffffu;           // test-only fault injection
    bool lazy = false;                                 // deferred fix-up (adacomp_set_lazy_fixup)
    uint32_t rule = ADACOMP_RULE_ADACOMP;              // selection rule (adacomp_set_selection_rule)
};

namespace adacomp {
// The status of a call's launches. Built with ADACOMP_DEBUG_CHECKS (a debug build),
// the call also waits for its stream, unless the stream is being captured, so that an
// error raised while its kernels run is returned by the call that launched them
// rather than by a later one.
adacomp_status launch_result(cudaError_t e, cudaStream_t stream)
{
    if (e != cudaSuccess) return ADACOMP_ERR_CUDA;
#ifdef ADACOMP_DEBUG_CHECKS
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return ADACOMP_ERR_CUDA;
    if (cap == cudaStreamCaptureStatusNone && cudaStreamSynchronize(stream) != cudaSuccess) return ADACOMP_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return ADACOMP_ERR_CUDA;
#else
    (void)stream;
#endif
    return ADACOMP_OK;
}
}  // namespace adacomp

namespace {
// A named range on the host timeline around an entry point's launches (a no-op
// unless a profiler that records NVTX ranges is attached), so that a trace shows
// which call issued which kernels.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};
}  // namespace

namespace {

using adacomp::KGroup;
using adacomp::KLayer;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

size_t max_msg_bytes(const KLayer& l) { return 8 + 2 * (size_t)l.nbins + (size_t)l.code_bytes * (size_t)l.n; }

// Every layer warp-sliced: the sliced path and its workspace layout.
bool handle_is_sliced(const adacomp_layer* h)
{
    for (const KLayer& k : h->layers)
        if (!k.bpw) return false;
    return !h->layers.empty();
}

// Every layer's bins longer than a warp slice (and at most kBigMaxLen): the
// block-sliced path, with the sliced path's workspace layout and 16 slices per tile.
bool handle_is_big(const adacomp_layer* h)
{
    for (const KLayer& k : h->layers)
        if (!adacomp::is_big_len(k.bin_len)) return false;
    return !h->layers.empty();
}

size_t compress_ws_for(const adacomp_layer* h)
{
    const int nl = (int)h->layers.size();
    if (handle_is_sliced(h)) return adacomp::sliced_ws_bytes(nl, h->total_tiles);
    if (handle_is_big(h)) return adacomp::sliced_ws_bytes(nl, h->total_tiles, true);
    return adacomp::compress_ws_bytes(nl, h->total_tiles, h->lazy);
}

adacomp_status make_group(adacomp_layer_t* out, int32_t num_layers, const int64_t* n, const int32_t* bin_len,
                          const int32_t* dtype, size_t* max_msg, size_t* cws, size_t* dws)
{
    if (!out) return ADACOMP_ERR_INVALID_ARG;
    *out = nullptr;
    if (num_layers < 1 || num_layers > ADACOMP_MAX_GROUP || !n || !bin_len || !dtype)
        return ADACOMP_ERR_INVALID_ARG;
    adacomp_layer* h = new (std::nothrow) adacomp_layer;
    if (!h) return ADACOMP_ERR_INVALID_ARG;
    uint64_t tiles = 0;
    for (int32_t i = 0; i < num_layers; ++i) {
        const int64_t N = n[i];
        const int32_t L = bin_len[i];
        if (N < 1 || L < 1 || L > adacomp::kMaxBinLen || (dtype[i] != ADACOMP_F32 && dtype[i] != ADACOMP_BF16)) {
            delete h;
            return ADACOMP_ERR_INVALID_ARG;
        }
        const int64_t B = (N + L - 1) / L;
        if (B >= (int64_t)1 << 32) { delete h; return ADACOMP_ERR_INVALID_ARG; }
        KLayer k;
        std::memset(&k, 0, sizeof k);
        k.n = N;
        k.nbins = (uint32_t)B;
        k.bin_len = L;
        // warp-sliced tiles: eight warp slices of floor(509 / L_T) whole bins each;
        // otherwise about kTileTarget elements of whole bins
        const int bpw = (L >= 16 && L <= adacomp::kWarpSliceMax) ? adacomp::kWarpSliceMax / L : 0;
        int64_t bpt = bpw ? (int64_t)adacomp::kWarps * bpw : adacomp::kTileTarget / L;
        if (bpt < 1) bpt = 1;
        if (bpt > adacomp::kMaxBinsPerTile) bpt = adacomp::kMaxBinsPerTile;
        if (bpt > B) bpt = B;
        k.bpw = (uint8_t)bpw;
        k.bins_per_tile = (uint32_t)bpt;
        k.num_tiles = (uint32_t)((B + bpt - 1) / bpt);
        k.tile_begin = (uint32_t)tiles;
        tiles += k.num_tiles;
        k.dw_bf16 = dtype[i] == ADACOMP_BF16 ? 1 : 0;
        k.code_bytes = L < 64 ? 1 : 2;
        k.vec = (L % 4 == 0) ? 4 : (L % 2 == 0) ? 2 : 1;
        k.inv_len = (uint32_t)(((1ull << 32) + (uint64_t)L - 1) / (uint64_t)L);
        if (!k.dw_bf16) h->d_size = 4;
        const uint64_t te = (uint64_t)bpt * (uint64_t)L;
        if (te > h->tile_cap) h->tile_cap = (uint32_t)te;
        if (bpt > h->max_bins) h->max_bins = (uint16_t)bpt;
        h->layers.push_back(k);
        if (max_msg) max_msg[i] = max_msg_bytes(k);
    }
    if (tiles >= (1ull << 31)) { delete h; return ADACOMP_ERR_INVALID_ARG; }
    h->total_tiles = (uint32_t)tiles;
    h->compress_ws = compress_ws_for(h);
    h->decode_per_learner = adacomp::decode_per_learner(tiles);
    if (cws) *cws = h->compress_ws;
    if (dws) *dws = h->decode_per_learner;
    *out = h;
    return ADACOMP_OK;
}

void fill_group(const adacomp_layer* h, KGroup* g)
{
    g->num_layers = (int32_t)h->layers.size();
    g->total_tiles = h->total_tiles;
    g->tile_cap = h->tile_cap;
    g->max_bins = h->max_bins;
    g->d_size = h->d_size;
    g->timeout_ns = h->timeout_ns;
    g->inject_skip_tile = h->inject_skip_tile;
    g->needs_gbuf = 0;
    g->lazy = h->lazy ? 1u : 0u;
    g->local_selection = h->rule == ADACOMP_RULE_LOCAL_SELECTION ? 1u : 0u;
    g->big = handle_is_big(h) ? 1u : 0u;
    for (const KLayer& k : h->layers)
        if (k.bin_len < 16) g->needs_gbuf = 1;  // the short-bin path stages G in shared memory
    for (size_t i = 0; i < h->layers.size(); ++i) g->layer[i] = h->layers[i];
}


adacomp_status launched(cudaError_t e, cudaStream_t stream) { return adacomp::launch_result(e, stream); }

}  // namespace

extern "C" {

adacomp_status adacomp_init_layer(adacomp_layer_t* out, int64_t n, int32_t bin_len, adacomp_dtype dw_dtype,
                                  size_t* max_msg_bytes, size_t* compress_ws_bytes,
                                  size_t* decode_ws_bytes_per_learner)
{
    const int32_t dt = (int32_t)dw_dtype;
    return make_group(out, 1, &n, &bin_len, &dt, max_msg_bytes, compress_ws_bytes, decode_ws_bytes_per_learner);
}

adacomp_status adacomp_init_group(adacomp_layer_t* out, int32_t num_layers, const int64_t* n,
                                  const int32_t* bin_len, const int32_t* dw_dtype, size_t* max_msg_bytes,
                                  size_t* compress_ws_bytes, size_t* decode_ws_bytes_per_learner)
{
    return make_group(out, num_layers, n, bin_len, dw_dtype, max_msg_bytes, compress_ws_bytes,
                      decode_ws_bytes_per_learner);
}

adacomp_status adacomp_compress_group(adacomp_layer_t h, float* const* residue, const void* const* dW,
                                      void* const* msg, const size_t* msg_capacity, void* ws, size_t ws_bytes,
                                      cudaStream_t stream)
{
    NvtxRange range("adacomp_compress");
    if (!h || !residue || !dW || !msg || !msg_capacity || !ws) return ADACOMP_ERR_INVALID_ARG;
    if (!aligned(ws, 16)) return ADACOMP_ERR_ALIGNMENT;
    if (ws_bytes < h->compress_ws) return ADACOMP_ERR_WORKSPACE;
    KGroup* g = new (std::nothrow) KGroup;
    if (!g) return ADACOMP_ERR_INVALID_ARG;
    std::memset(g, 0, sizeof *g);
    fill_group(h, g);
    for (size_t i = 0; i < h->layers.size(); ++i) {
        if (!residue[i] || !dW[i] || !msg[i]) { delete g; return ADACOMP_ERR_INVALID_ARG; }
        if (!aligned(residue[i], 16) || !aligned(dW[i], 16) || !aligned(msg[i], 16)) {
            delete g;
            return ADACOMP_ERR_ALIGNMENT;
        }
        if (msg_capacity[i] < max_msg_bytes(h->layers[i])) { delete g; return ADACOMP_ERR_CAPACITY; }
        g->layer[i].residue = residue[i];
        g->layer[i].dw = dW[i];
        g->layer[i].msg = static_cast<uint8_t*>(msg[i]);
    }
    const cudaError_t e = adacomp::launch_compress(*g, ws, stream, h->ev[0], h->ev[1], h->ev[2]);
    delete g;
    return launched(e, stream);
}

adacomp_status adacomp_compress(adacomp_layer_t h, float* residue, const void* dW, void* msg, size_t msg_capacity,
                                void* ws, size_t ws_bytes, cudaStream_t stream)
{
    if (!h) return ADACOMP_ERR_INVALID_ARG;
    if (h->layers.size() != 1) return ADACOMP_ERR_INVALID_ARG;
    return adacomp_compress_group(h, &residue, &dW, &msg, &msg_capacity, ws, ws_bytes, stream);
}

}  // extern "C"

namespace {
// The optimiser step fused with a decode call (none for the plain sum).
struct OptArgs {
    int opt = adacomp::kOptNone;
    float* const* mom = nullptr;   // momentum (SGD) or first moment (Adam), per layer
    float* const* mom2 = nullptr;  // second moment (Adam), per layer
    float lr = 0.0f, mu = 0.0f, scale = 1.0f;
    float beta1 = 0.0f, beta2 = 0.0f, eps = 0.0f, bc1 = 1.0f, bc2 = 1.0f;
};

// Shared by the plain decode and the decodes fused with an optimiser step.
adacomp_status decode_group(adacomp_layer_t h, const void* const* msgs, const uint64_t* msg_bytes, int32_t K,
                            float* const* dense, const OptArgs& o, void* ws, size_t ws_bytes, cudaStream_t stream)
{
    NvtxRange range(o.opt == adacomp::kOptAdam  ? "adacomp_decode_adam"
                    : o.opt == adacomp::kOptSGD ? "adacomp_decode_sgd"
                                                : "adacomp_decode_accumulate");
    if (!h || !msgs || !msg_bytes || !dense || !ws) return ADACOMP_ERR_INVALID_ARG;
    if ((o.opt != adacomp::kOptNone && !o.mom) || (o.opt == adacomp::kOptAdam && !o.mom2)) return ADACOMP_ERR_INVALID_ARG;
    const int64_t L = (int64_t)h->layers.size();
    if (K < 1 || K > ADACOMP_MAX_LEARNERS || (int64_t)K * L > adacomp::kMaxDecodePairs)
        return ADACOMP_ERR_INVALID_ARG;
    if (!aligned(ws, 16)) return ADACOMP_ERR_ALIGNMENT;
    if (ws_bytes < adacomp::kDecodeFixed + (size_t)K * h->decode_per_learner) return ADACOMP_ERR_WORKSPACE;
    KGroup* g = new (std::nothrow) KGroup;
    adacomp::DecodeParams* p = new (std::nothrow) adacomp::DecodeParams;
    if (!g || !p) { delete g; delete p; return ADACOMP_ERR_INVALID_ARG; }
    std::memset(g, 0, sizeof *g);
    std::memset(p, 0, sizeof *p);
    fill_group(h, g);
    p->K = K;
    p->opt = o.opt;
    p->lr = o.lr;
    p->mu = o.mu;
    p->scale = o.scale;
    p->beta1 = o.beta1;
    p->beta2 = o.beta2;
    p->eps = o.eps;
    p->bc1 = o.bc1;
    p->bc2 = o.bc2;
    uint32_t vt = 0, ct = 0;  // counting and code-check tasks per learner, layer by layer
    for (int64_t l = 0; l < L; ++l) {
        const KLayer& k = h->layers[(size_t)l];
        const uint32_t per = adacomp::val_tiles_per_task(k.bins_per_tile);
        p->val_begin[l] = vt;
        vt += (k.num_tiles + per - 1) / per;
        p->chk_begin[l] = ct;
        ct += adacomp::chk_tasks(k.num_tiles, k.bins_per_tile, k.bin_len);
    }
    p->val_begin[L] = vt;
    p->chk_begin[L] = ct;
    adacomp_status st = ADACOMP_OK;
    for (int64_t l = 0; l < L && st == ADACOMP_OK; ++l) {
        float* m1 = o.mom ? o.mom[l] : nullptr;
        float* m2 = o.mom2 ? o.mom2[l] : nullptr;
        if (!dense[l] || (o.mom && !m1) || (o.mom2 && !m2)) st = ADACOMP_ERR_INVALID_ARG;
        else if (!aligned(dense[l], 16) || (m1 && !aligned(m1, 16)) || (m2 && !aligned(m2, 16)))
            st = ADACOMP_ERR_ALIGNMENT;
        p->dense[l] = dense[l];
        p->mom[l] = m1;
        p->mom2[l] = m2;
        for (int32_t k = 0; k < K && st == ADACOMP_OK; ++k) {
            const void* m = msgs[l * K + k];
            if (!m) st = ADACOMP_ERR_INVALID_ARG;
            else if (!aligned(m, 16)) st = ADACOMP_ERR_ALIGNMENT;
            p->msg[l * K + k] = static_cast<const uint8_t*>(m);
            p->len[l * K + k] = msg_bytes[l * K + k];
        }
    }
    if (st == ADACOMP_OK) st = launched(adacomp::launch_decode(*g, *p, ws, stream), stream);
    delete g;
    delete p;
    return st;
}
}  // namespace

extern "C" {

adacomp_status adacomp_decode_accumulate_group(adacomp_layer_t h, const void* const* msgs, const uint64_t* msg_bytes,
                                               int32_t K, float* const* dense, void* ws, size_t ws_bytes,
                                               cudaStream_t stream)
{
    return decode_group(h, msgs, msg_bytes, K, dense, OptArgs(), ws, ws_bytes, stream);
}

adacomp_status adacomp_decode_sgd_group(adacomp_layer_t h, const void* const* msgs, const uint64_t* msg_bytes,
                                        int32_t K, float* const* weights, float* const* momentum, float lr, float mu,
                                        float grad_scale, void* ws, size_t ws_bytes, cudaStream_t stream)
{
    if (!momentum) return ADACOMP_ERR_INVALID_ARG;
    OptArgs o;
    o.opt = adacomp::kOptSGD;
    o.mom = momentum;
    o.lr = lr;
    o.mu = mu;
    o.scale = grad_scale;
    return decode_group(h, msgs, msg_bytes, K, weights, o, ws, ws_bytes, stream);
}

adacomp_status adacomp_decode_sgd(adacomp_layer_t h, const void* const* msgs, const uint64_t* msg_bytes, int32_t K,
                                  float* weights, float* momentum, float lr, float mu, float grad_scale, void* ws,
                                  size_t ws_bytes, cudaStream_t stream)
{
    if (!h) return ADACOMP_ERR_INVALID_ARG;
    if (h->layers.size() != 1) return ADACOMP_ERR_INVALID_ARG;
    return adacomp_decode_sgd_group(h, msgs, msg_bytes, K, &weights, &momentum, lr, mu, grad_scale, ws, ws_bytes,
                                    stream);
}

adacomp_status adacomp_decode_adam_group(adacomp_layer_t h, const void* const* msgs, const uint64_t* msg_bytes,
                                         int32_t K, float* const* weights, float* const* m, float* const* v, float lr,
                                         float beta1, float beta2, float eps, float bias_correction1,
                                         float bias_correction2, float grad_scale, void* ws, size_t ws_bytes,
                                         cudaStream_t stream)
{
    if (!m || !v) return ADACOMP_ERR_INVALID_ARG;
    if (!(bias_correction1 > 0.0f) || !(bias_correction2 > 0.0f)) return ADACOMP_ERR_INVALID_ARG;
    OptArgs o;
    o.opt = adacomp::kOptAdam;
    o.mom = m;
    o.mom2 = v;
    o.lr = lr;
    o.scale = grad_scale;
    o.beta1 = beta1;
    o.beta2 = beta2;
    o.eps = eps;
    o.bc1 = bias_correction1;
    o.bc2 = bias_correction2;
    return decode_group(h, msgs, msg_bytes, K, weights, o, ws, ws_bytes, stream);
}

adacomp_status adacomp_decode_adam(adacomp_layer_t h, const void* const* msgs, const uint64_t* msg_bytes, int32_t K,
                                   float* weights, float* m, float* v, float lr, float beta1, float beta2, float eps,
                                   float bias_correction1, float bias_correction2, float grad_scale, void* ws,
                                   size_t ws_bytes, cudaStream_t stream)
{
    if (!h) return ADACOMP_ERR_INVALID_ARG;
    if (h->layers.size() != 1) return ADACOMP_ERR_INVALID_ARG;
    return adacomp_decode_adam_group(h, msgs, msg_bytes, K, &weights, &m, &v, lr, beta1, beta2, eps,
                                     bias_correction1, bias_correction2, grad_scale, ws, ws_bytes, stream);
}

adacomp_status adacomp_decode_accumulate(adacomp_layer_t h, const void* const* msgs, const uint64_t* msg_bytes,
                                         int32_t K, float* dense, void* ws, size_t ws_bytes, cudaStream_t stream)
{
    if (!h) return ADACOMP_ERR_INVALID_ARG;
    if (h->layers.size() != 1) return ADACOMP_ERR_INVALID_ARG;
    return adacomp_decode_accumulate_group(h, msgs, msg_bytes, K, &dense, ws, ws_bytes, stream);
}

adacomp_status adacomp_query(adacomp_layer_t h, const void* ws, int32_t layer, cudaStream_t stream,
                             uint64_t* msg_bytes, float* s, int32_t* device_status)
{
    if (!h || !ws || layer < 0 || layer >= (int32_t)h->layers.size()) return ADACOMP_ERR_INVALID_ARG;
    adacomp::Result r;
    const uint8_t* src = static_cast<const uint8_t*>(ws) + adacomp::ws_layer_offset(layer) +
                         offsetof(adacomp::LayerWs, result);
    cudaError_t e = cudaMemcpyAsync(&r, src, sizeof r, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return ADACOMP_ERR_CUDA;
    if (msg_bytes) *msg_bytes = r.msg_bytes;
    if (s) *s = r.s;
    if (device_status) *device_status = (int32_t)r.status;
    return ADACOMP_OK;
}

adacomp_status adacomp_decode_status(adacomp_layer_t h, const void* ws, cudaStream_t stream,
                                     int32_t* device_status)
{
    if (!h || !ws) return ADACOMP_ERR_INVALID_ARG;
    uint8_t fixed[16 + adacomp::kMaxDecodePairs];  // K, layers, one bad-message byte per (layer, learner)
    cudaError_t e = cudaMemcpyAsync(fixed, ws, sizeof fixed, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return ADACOMP_ERR_CUDA;
    uint32_t K, L;
    std::memcpy(&K, fixed, 4);
    std::memcpy(&L, fixed + 4, 4);
    int32_t st = ADACOMP_OK;
    if ((uint64_t)K * L > (uint64_t)adacomp::kMaxDecodePairs) st = ADACOMP_ERR_BAD_MESSAGE;
    else
        for (uint32_t i = 0; i < K * L; ++i)
            if (fixed[16 + i]) st = ADACOMP_ERR_BAD_MESSAGE;
    if (device_status) *device_status = st;
    return ADACOMP_OK;
}

adacomp_status adacomp_set_timing_events(adacomp_layer_t h, cudaEvent_t before, cudaEvent_t mid,
                                         cudaEvent_t after)
{
    if (!h) return ADACOMP_ERR_INVALID_ARG;
    h->ev[0] = before;
    h->ev[1] = mid;
    h->ev[2] = after;
    return ADACOMP_OK;
}

adacomp_status adacomp_set_fault_injection(adacomp_layer_t h, uint32_t skip_tile)
{
    if (!h) return ADACOMP_ERR_INVALID_ARG;
    h->inject_skip_tile = skip_tile;
    return ADACOMP_OK;
}

adacomp_status adacomp_set_selection_rule(adacomp_layer_t h, int32_t rule)
{
    if (!h || (rule != ADACOMP_RULE_ADACOMP && rule != ADACOMP_RULE_LOCAL_SELECTION)) return ADACOMP_ERR_INVALID_ARG;
    h->rule = (uint32_t)rule;
    return ADACOMP_OK;
}

adacomp_status adacomp_set_lazy_fixup(adacomp_layer_t h, int32_t enable, size_t* compress_ws_bytes)
{
    if (!h) return ADACOMP_ERR_INVALID_ARG;
    h->lazy = enable != 0;
    h->compress_ws = compress_ws_for(h);
    if (compress_ws_bytes) *compress_ws_bytes = h->compress_ws;
    return ADACOMP_OK;
}

adacomp_status adacomp_materialize_group(adacomp_layer_t h, float* const* residue, void* ws, size_t ws_bytes,
                                         cudaStream_t stream)
{
    NvtxRange range("adacomp_materialize");
    if (!h || !residue || !ws) return ADACOMP_ERR_INVALID_ARG;
    if (!aligned(ws, 16)) return ADACOMP_ERR_ALIGNMENT;
    if (ws_bytes < h->compress_ws) return ADACOMP_ERR_WORKSPACE;
    if (!h->lazy) return ADACOMP_OK;  // nothing is ever deferred
    KGroup* g = new (std::nothrow) KGroup;
    if (!g) return ADACOMP_ERR_INVALID_ARG;
    std::memset(g, 0, sizeof *g);
    fill_group(h, g);
    for (size_t i = 0; i < h->layers.size(); ++i) {
        if (!residue[i]) { delete g; return ADACOMP_ERR_INVALID_ARG; }
        if (!aligned(residue[i], 16)) { delete g; return ADACOMP_ERR_ALIGNMENT; }
        g->layer[i].residue = residue[i];
    }
    const cudaError_t e = adacomp::launch_materialize(*g, ws, stream);
    delete g;
    return launched(e, stream);
}

adacomp_status adacomp_materialize(adacomp_layer_t h, float* residue, void* ws, size_t ws_bytes, cudaStream_t stream)
{
    if (!h) return ADACOMP_ERR_INVALID_ARG;
    if (h->layers.size() != 1) return ADACOMP_ERR_INVALID_ARG;
    return adacomp_materialize_group(h, &residue, ws, ws_bytes, stream);
}

adacomp_status adacomp_set_timeout_ns(adacomp_layer_t h, uint64_t timeout_ns)
{
    if (!h || timeout_ns == 0) return ADACOMP_ERR_INVALID_ARG;
    h->timeout_ns = timeout_ns;
    return ADACOMP_OK;
}

void adacomp_free(adacomp_layer_t h) { delete h; }

const char* adacomp_status_string(adacomp_status s)
{
    switch (s) {
    case ADACOMP_OK: return "ok";
    case ADACOMP_ERR_INVALID_ARG: return "invalid argument";
    case ADACOMP_ERR_ALIGNMENT: return "buffer not aligned";
    case ADACOMP_ERR_WORKSPACE: return "workspace too small";
    case ADACOMP_ERR_CAPACITY: return "message buffer too small";
    case ADACOMP_ERR_CUDA: return "CUDA error";
    case ADACOMP_ERR_TIMEOUT: return "device wait timed out";
    case ADACOMP_ERR_BAD_MESSAGE: return "malformed message";
    }
    return "unknown status";
}

}  // extern "C"

namespace adacomp {

// Argument checks and launch descriptor for one single-layer compress call, for
// entry points that supply their own workspace. Same checks as adacomp_compress
// apart from the workspace; *ws_needed receives the workspace size the call uses.
int prepare_single_compress(const adacomp_layer* h, float* residue, const void* dW, void* msg,
                            size_t msg_capacity, KGroup* g, size_t* ws_needed)
{
    if (!h || h->layers.size() != 1) return ADACOMP_ERR_INVALID_ARG;
    *ws_needed = h->compress_ws;
    if (!residue || !dW || !msg) return ADACOMP_ERR_INVALID_ARG;
    if (!aligned(residue, 16) || !aligned(dW, 16) || !aligned(msg, 16)) return ADACOMP_ERR_ALIGNMENT;
    if (msg_capacity < max_msg_bytes(h->layers[0])) return ADACOMP_ERR_CAPACITY;
    std::memset(g, 0, sizeof *g);
    fill_group(h, g);
    g->layer[0].residue = residue;
    g->layer[0].dw = dW;
    g->layer[0].msg = static_cast<uint8_t*>(msg);
    return ADACOMP_OK;
}

size_t compress_ws_of(const adacomp_layer* h) { return h ? h->compress_ws : 0; }

}  // namespace adacomp
