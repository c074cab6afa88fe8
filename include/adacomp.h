/*
 * adacomp.h — C ABI of the GB300 (sm_103a) AdaComp library, libadacomp.so.
 *
 * AdaComp ("AdaComp (Adaptive Residual Gradient Compression)", summary paragraph and
 * Claims > Mechanism #r629-local-bin-soft-threshold-and-mean-gmax-quantization) is a
 * per-layer residual gradient compressor for data-parallel training. For one layer
 * with residue r and gradient dW (N elements):
 *     G = r + dW,  H = G + dW,  bins of length L_T over G,
 *     g_max(i) = max |G| over bin i,  s = (1/B) sum_i g_max(i),
 *     send every element with |H| >= g_max(i) as sign(G) * s,
 *     r = G - sign(G) * s for sent elements, r = G for the rest.
 * Codes are 8 bits when L_T < 64 and 16 bits otherwise (Claims > Application
 * #r629-conv-40x-and-fc-lstm-200x-compression-across-optimizers; Curated
 * Limitations). The pages leave open the points below; this library reads them so:
 *   - a partial last bin is a bin; its g_max covers its own elements;
 *   - only G != 0 is sent (sign(0) has no code); the tie |H| == g_max is sent;
 *   - H = fl32(G + dW) after G is rounded; IEEE fp32 adds, no contraction;
 *   - s = fl32( fl64(exact sum of the g_max) / B ), independent of summation order;
 *   - decoding adds sign * s_k into a dense fp32 buffer learner by learner,
 *     k = 0..K-1, with no averaging.
 *
 * Message format (little-endian, no padding), produced by adacomp_compress:
 *     offset 0      float32  s
 *     offset 4      uint32   B = ceil(N / L_T)
 *     offset 8      uint16   count[B]          codes sent from each bin
 *     offset 8+2B   codes, bin by bin, ascending offset within a bin;
 *                   code = (offset_in_bin << 1) | (G < 0); uint8 if L_T < 64 else uint16
 * Its length is 8 + 2B + w * nnz bytes (w = code bytes, nnz = elements sent); it never
 * exceeds max_msg_bytes = 8 + 2B + w * N.
 *
 * Conventions shared by every call:
 *   - Pointers named "device" are CUDA device pointers (e.g. torch tensor data_ptr());
 *     the caller owns every buffer. The library never allocates device memory.
 *   - residue, dW, dense and msg must be 16-byte aligned (ADACOMP_ERR_ALIGNMENT).
 *   - Work is enqueued on `stream` and returns before it runs; results, the message
 *     length and the device-side status are read back with adacomp_query /
 *     adacomp_decode_status. Every call is deterministic: same inputs, same bits.
 *   - A debug build of the library (compiled with ADACOMP_DEBUG_CHECKS defined)
 *     makes every compress, decode and materialise call wait for `stream` after its
 *     launches, unless the stream is being captured, and return ADACOMP_ERR_CUDA
 *     when its kernels raised an error, so that the error is reported by the call
 *     that caused it.
 *   - Argument errors are reported synchronously before anything is enqueued.
 *     ADACOMP_ERR_CUDA reports a failed launch (cudaGetLastError).
 *   - Workspaces: a compress workspace must be zero-filled before its first use
 *     (e.g. torch.zeros); every completed compress call leaves the parts that must
 *     start at zero zeroed again (the rest is written before it is read), so it can
 *     be reused by later calls and by other handles that fit in it. Calls that share a workspace must not overlap on the
 *     GPU (use one stream, or order the streams). After any device-side error
 *     status, zero the workspace again before reusing it.
 *   - Device-side waits (for the bulk copies into shared memory, and, for handles
 *     whose bin lengths are not all 16..509 or all 510..8189, the look-back between
 *     tiles) are bounded by a timeout
 *     (default 2 s, adacomp_set_timeout_ns); on expiry the kernel records
 *     ADACOMP_ERR_TIMEOUT in the workspace and returns. Nothing traps.
 *   - L_T (bin_len) is limited to 1..8192 by this implementation (the format itself
 *     would allow offsets up to 32767).
 */
#ifndef ADACOMP_H
#define ADACOMP_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ADACOMP_OK = 0,
    ADACOMP_ERR_INVALID_ARG = 1,  /* n < 1, bin_len outside 1..8192, B >= 2^32, K outside 1..256 ... */
    ADACOMP_ERR_ALIGNMENT = 2,    /* a buffer is not 16-byte aligned */
    ADACOMP_ERR_WORKSPACE = 3,    /* ws is NULL or smaller than the size init returned */
    ADACOMP_ERR_CAPACITY = 4,     /* msg_capacity < max_msg_bytes */
    ADACOMP_ERR_CUDA = 5,         /* a CUDA runtime call or launch failed */
    ADACOMP_ERR_TIMEOUT = 6,      /* device: a bounded wait (a copy, or the look-back between tiles) ran out */
    ADACOMP_ERR_BAD_MESSAGE = 7   /* device: a message's length, B, counts or offsets do not fit this layer */
} adacomp_status;

typedef enum { ADACOMP_F32 = 0, ADACOMP_BF16 = 1 } adacomp_dtype;

/* Opaque host-side handle: layer sizes, bin length, dW dtype and tile geometry. It
 * holds no device memory and may be used from one host thread at a time. */
typedef struct adacomp_layer* adacomp_layer_t;

/*
 * Describes one layer of n elements compressed with bins of bin_len elements and a
 * dW of type dw_dtype ("AdaComp ...", Claims > Mechanism #r629-local-bin-...: one
 * compressor per layer, with its own residue).
 * Out (each may be NULL):
 *   max_msg_bytes                 bytes a message buffer needs (8 + 2B + w*n)
 *   compress_ws_bytes             bytes of compress workspace
 *   decode_ws_bytes_per_learner   decode workspace = ADACOMP_DECODE_WS_FIXED + K * this
 * Host only: makes no CUDA call. Errors: ADACOMP_ERR_INVALID_ARG.
 */
adacomp_status adacomp_init_layer(adacomp_layer_t* out, int64_t n, int32_t bin_len,
                                  adacomp_dtype dw_dtype, size_t* max_msg_bytes,
                                  size_t* compress_ws_bytes,
                                  size_t* decode_ws_bytes_per_learner);

/*
 * A group of num_layers layers (1..ADACOMP_MAX_GROUP) compressed by one launch
 * sequence: layer l has n[l] elements, bin length bin_len[l] and dW type
 * dw_dtype[l]. Each layer keeps its own bins, s and message, exactly as if it were
 * compressed alone; grouping only removes per-layer launches. max_msg_bytes is an
 * array of num_layers entries (or NULL). Host only.
 */
adacomp_status adacomp_init_group(adacomp_layer_t* out, int32_t num_layers, const int64_t* n,
                                  const int32_t* bin_len, const int32_t* dw_dtype,
                                  size_t* max_msg_bytes, size_t* compress_ws_bytes,
                                  size_t* decode_ws_bytes_per_learner);

#define ADACOMP_MAX_GROUP 128
#define ADACOMP_MAX_LEARNERS 256
#define ADACOMP_DECODE_WS_FIXED 10240

/*
 * One AdaComp step for one layer (Algorithm 2 as restated in Claims > Mechanism
 * #r629-local-bin-soft-threshold-and-mean-gmax-quantization).
 *   residue   device fp32[n], in/out: the carried residue, updated in place
 *             (zeros before the first step)
 *   dW        device fp32[n] or bf16[n] (the dtype given at init), read only
 *   msg       device buffer of msg_capacity >= max_msg_bytes bytes; receives the
 *             message (format above)
 *   ws        device compress workspace of ws_bytes >= compress_ws_bytes (see
 *             Workspaces above)
 * residue and dW must not overlap msg or ws. Errors: INVALID_ARG (NULL handle or
 * pointer), ALIGNMENT, CAPACITY, WORKSPACE, CUDA. Device-side status via
 * adacomp_query.
 */
adacomp_status adacomp_compress(adacomp_layer_t h, float* residue, const void* dW, void* msg,
                                size_t msg_capacity, void* ws, size_t ws_bytes,
                                cudaStream_t stream);

/*
 * adacomp_compress for callers that cannot allocate device memory: plugins and
 * hooks of communication or training frameworks that are handed only their
 * gradient and message buffers, and that run where allocating is not allowed (the
 * host application's allocator owns all device memory, or a fixed memory budget
 * leaves no room for a separate workspace). The paper has no counterpart; this is
 * an interface convenience of this library.
 *
 * Same arguments, checks and results as adacomp_compress, but the compress
 * workspace is an array of ADACOMP_STATIC_WS_BYTES (1 MiB) inside the library (a
 * file-scope __device__ array that every GPU loading the library keeps until the
 * process exits). It therefore takes single-layer handles whose compress_ws_bytes
 * (from adacomp_init_layer) is at most ADACOMP_STATIC_WS_BYTES; compare the two to
 * know whether a layer fits (roughly 3.9M elements for 16 <= L_T <= 509, whose
 * workspace holds two bits per element, about 2M at L_T = 510, rising with L_T to
 * the block-sliced limit of 8189, and far more for other bin lengths). Larger
 * layers get ADACOMP_ERR_WORKSPACE.
 * The call allocates nothing: it zeroes the part of the array it uses
 * (cudaMemsetAsync) and runs the same kernels on `stream`.
 *   result_out  optional device buffer of 32 bytes, 8-byte aligned, that receives
 *               {float s; uint32 status; uint64 nnz; uint64 msg_bytes; uint64 pad}
 *               (the values adacomp_query reports for adacomp_compress); NULL skips it.
 * The first call on each device looks up the array's device address with that
 * device current and keeps it for the life of the process; make that first call
 * before capturing any stream. The kept address belongs to the device's context:
 * after cudaDeviceReset of that device, do not call this entry point again in the
 * same process. All calls share the one array, so calls that overlap on a GPU
 * (different streams, or several host threads) race and corrupt each other's
 * results: serialise them.
 */
#define ADACOMP_STATIC_WS_BYTES ((size_t)1 << 20)
adacomp_status adacomp_compress_static_ws(adacomp_layer_t h, float* residue, const void* dW,
                                          void* msg, size_t msg_capacity, void* result_out,
                                          cudaStream_t stream);

/* adacomp_compress for every layer of a group: arrays of num_layers device pointers
 * (host arrays) and capacities; one workspace for the whole group. */
adacomp_status adacomp_compress_group(adacomp_layer_t h, float* const* residue,
                                      const void* const* dW, void* const* msg,
                                      const size_t* msg_capacity, void* ws, size_t ws_bytes,
                                      cudaStream_t stream);

/*
 * Sums K learners' messages into a dense gradient: for k = 0..K-1 in order, every
 * code of msgs[k] adds sign * s_k to dense[bin * L_T + offset] (one fp32 add each).
 * The pages only say that learners' quantised gradients are combined in
 * data-parallel training (abstract; summary paragraph); the plain sum is this
 * library's reading, and the caller zeroes dense for a fresh sum.
 *   msgs       host array of K device pointers, each a message of this layer
 *              starting on a 16-byte boundary
 *   msg_bytes  host array of K lengths in bytes, the length of each message as
 *              received (messages are variable-length: "AdaComp (Adaptive Residual
 *              Gradient Compression)", Claims > Limitation
 *              #r629-minibatch-size-activity-and-variable-message-length). Nothing
 *              past a message's length is used; the library may read the rest of the
 *              16-byte block its last byte lies in.
 *   dense      device fp32[n], in/out
 *   ws         device decode workspace, ws_bytes >= ADACOMP_DECODE_WS_FIXED
 *              + K * decode_ws_bytes_per_learner; needs no initialisation
 * One CTA owns each range of bins, so no two threads ever add to one element and
 * no float atomics are used. Every message is checked before anything is added, and
 * a message that fails a check is skipped entirely (it adds nothing; the others are
 * summed as usual) and ADACOMP_ERR_BAD_MESSAGE is recorded (adacomp_decode_status).
 * The checks: the length is at least 8 + 2B, the header's B is the layer's B, no
 * count exceeds its bin's length, the length is exactly 8 + 2B + w * (sum of the
 * counts), and within every bin the code offsets rise strictly and stay below the
 * bin's length (a message gives each element at most one code). Errors:
 * INVALID_ARG (K outside 1..256, NULL pointers), ALIGNMENT (dense or a message not
 * 16-byte aligned), WORKSPACE, CUDA.
 */
adacomp_status adacomp_decode_accumulate(adacomp_layer_t h, const void* const* msgs,
                                         const uint64_t* msg_bytes, int32_t K, float* dense,
                                         void* ws, size_t ws_bytes, cudaStream_t stream);

/* Decode for every layer of a group: msgs and msg_bytes are host arrays of
 * num_layers * K entries, layer-major (msgs[l * K + k]); dense a host array of
 * num_layers device pointers. K <= ADACOMP_MAX_LEARNERS and K * num_layers <= 1024. */
adacomp_status adacomp_decode_accumulate_group(adacomp_layer_t h, const void* const* msgs,
                                               const uint64_t* msg_bytes, int32_t K,
                                               float* const* dense, void* ws, size_t ws_bytes,
                                               cudaStream_t stream);

/*
 * Waits for `stream` and reads the result of the last compress call that used `ws`
 * for layer `layer` (0 for a single layer): the message length in bytes, s, and the
 * device status (ADACOMP_OK, ADACOMP_ERR_TIMEOUT). Any output may be NULL.
 */
adacomp_status adacomp_query(adacomp_layer_t h, const void* ws, int32_t layer,
                             cudaStream_t stream, uint64_t* msg_bytes, float* s,
                             int32_t* device_status);

/* Waits for `stream` and reads the device status of the last decode call that used
 * `ws` (ADACOMP_OK or ADACOMP_ERR_BAD_MESSAGE). */
adacomp_status adacomp_decode_status(adacomp_layer_t h, const void* ws, cudaStream_t stream,
                                     int32_t* device_status);

/*
 * Measurement hook (not part of the method): when set, every later compress call
 * on this handle records `before` on its stream before the streaming kernel, `mid`
 * between the streaming kernel and the kernels after it (scale, codes, fix-up), and
 * `after` once all are enqueued, so cudaEventElapsedTime gives the streaming
 * kernel's duration and that of the rest. The events are created and
 * owned by the caller; pass NULLs to stop recording.
 */
adacomp_status adacomp_set_timing_events(adacomp_layer_t h, cudaEvent_t before, cudaEvent_t mid,
                                         cudaEvent_t after);

/*
 * Fault injection for tests of the device-side timeout (not part of the method):
 * when skip_tile is a valid tile index of this handle's next compress calls, the
 * bulk copies of that tile are never started when every layer has 16 <= L_T <= 509
 * or every layer 510 <= L_T <= 8189 (its warps' waits run out), and otherwise the
 * tile never publishes its look-back
 * descriptor (the tiles after it in its layer wait for it); either way the layer
 * reports ADACOMP_ERR_TIMEOUT once the timeout has passed. Nothing faults or hangs. Pass 0xFFFFFFFF to switch it off (the default). After such a
 * call, zero the workspace before reusing it.
 */
adacomp_status adacomp_set_fault_injection(adacomp_layer_t h, uint32_t skip_tile);

/* Bound on each device-side wait, in nanoseconds (default 2e9). */
adacomp_status adacomp_set_timeout_ns(adacomp_layer_t h, uint64_t timeout_ns);

/* Decode fused with one momentum-SGD step (the optimisers the learners use:
 * "AdaComp (Adaptive Residual Gradient Compression)", Claims > Application
 * #r629-conv-40x-and-fc-lstm-200x-compression-across-optimizers; the update rule
 * itself is not on the pages and is read as the usual heavy-ball form without
 * dampening). For each element j of each layer, with g_j the learners' codes summed
 * from zero exactly as adacomp_decode_accumulate sums them (learner order, fp32):
 *     v_j = fl32( fl32(mu * v_j) + fl32(grad_scale * g_j) )
 *     w_j = fl32( w_j - fl32(lr * v_j) )
 * (no fused multiply-add). weights and momentum are fp32[n] per layer, in/out,
 * 16-byte aligned; grad_scale = 1/K averages instead of summing. The gradient is
 * never written to global memory: it lives only in the tile being updated. Same
 * messages, workspace and error reporting as adacomp_decode_accumulate (a rejected
 * message contributes nothing). */
adacomp_status adacomp_decode_sgd(adacomp_layer_t h, const void* const* msgs, const uint64_t* msg_bytes,
                                  int32_t K, float* weights, float* momentum, float lr, float mu,
                                  float grad_scale, void* ws, size_t ws_bytes, cudaStream_t stream);
adacomp_status adacomp_decode_sgd_group(adacomp_layer_t h, const void* const* msgs, const uint64_t* msg_bytes,
                                        int32_t K, float* const* weights, float* const* momentum, float lr,
                                        float mu, float grad_scale, void* ws, size_t ws_bytes,
                                        cudaStream_t stream);

/* Decode fused with one Adam step, the other optimiser the learners use
 * ("AdaComp (Adaptive Residual Gradient Compression)", Claims > Application
 * #r629-conv-40x-and-fc-lstm-200x-compression-across-optimizers; the update rule is
 * not on the pages and is read as Kingma and Ba's Adam with the bias corrections
 * written out). For each element j of each layer, with s_j the learners' codes summed
 * from zero exactly as adacomp_decode_accumulate sums them (learner order, fp32):
 *     g   = fl32(grad_scale * s_j)
 *     m_j = fl32( fl32(beta1 * m_j) + fl32(fl32(1 - beta1) * g) )
 *     v_j = fl32( fl32(beta2 * v_j) + fl32(fl32(1 - beta2) * fl32(g * g)) )
 *     w_j = fl32( w_j - fl32( lr * fl32( fl32(m_j / bias_correction1) /
 *                                        fl32( sqrt(fl32(v_j / bias_correction2)) + eps ) ) ) )
 * (IEEE fp32, correctly rounded division and square root, no fused multiply-add).
 * bias_correction1 = 1 - beta1^t and bias_correction2 = 1 - beta2^t for step t are
 * the caller's (both > 0; ADACOMP_ERR_INVALID_ARG otherwise). weights, m and v are
 * fp32[n] per layer, in/out, 16-byte aligned. The gradient lives only in the tile
 * being updated. Same messages, lengths, workspace and error reporting as
 * adacomp_decode_accumulate (a rejected message contributes nothing). */
adacomp_status adacomp_decode_adam(adacomp_layer_t h, const void* const* msgs, const uint64_t* msg_bytes,
                                   int32_t K, float* weights, float* m, float* v, float lr, float beta1,
                                   float beta2, float eps, float bias_correction1, float bias_correction2,
                                   float grad_scale, void* ws, size_t ws_bytes, cudaStream_t stream);
adacomp_status adacomp_decode_adam_group(adacomp_layer_t h, const void* const* msgs, const uint64_t* msg_bytes,
                                         int32_t K, float* const* weights, float* const* m, float* const* v,
                                         float lr, float beta1, float beta2, float eps, float bias_correction1,
                                         float bias_correction2, float grad_scale, void* ws, size_t ws_bytes,
                                         cudaStream_t stream);

/* Selection rule. ADACOMP_RULE_ADACOMP (the default) sends an element when
 * G != 0 and |fl32(G + dW)| >= g_max of its bin ("AdaComp (Adaptive Residual
 * Gradient Compression)", Claims > Mechanism
 * #r629-local-bin-soft-threshold-and-mean-gmax-quantization).
 * ADACOMP_RULE_LOCAL_SELECTION is the hard Local Selection rule that the same entry
 * contrasts with it (Claims > Mechanism
 * #r629-self-adjusting-sparsity-prevents-residual-explosion): no soft-threshold
 * probe, G != 0 and |G| >= g_max, i.e. only the bin maxima (all of them on a tie).
 * s, the codes, the message format, the residue update and decoding are the same
 * for both. Returns ADACOMP_ERR_INVALID_ARG for any other value. */
enum { ADACOMP_RULE_ADACOMP = 0, ADACOMP_RULE_LOCAL_SELECTION = 1 };
adacomp_status adacomp_set_selection_rule(adacomp_layer_t h, int32_t rule);

/* Deferred ("lazy") fix-up, the next step after the eager path
 * ("AdaComp (Adaptive Residual Gradient Compression)", Claims > Mechanism
 * #r629-local-bin-soft-threshold-and-mean-gmax-quantization: residue = G - G_q for
 * sent elements; the arithmetic is unchanged, only its time moves).
 *
 * With enable != 0, a compress call on this handle leaves the residue of the
 * elements it sent at G and records, in the compress workspace, one bit per such
 * element; the next compress call on the same workspace applies
 * residue = fl32(G - sign(G) * s_prev) to them as it loads them, before forming its
 * own G, and adacomp_materialize applies them on demand. Messages, s and every
 * later step are bit-identical to the eager path; the residue buffer holds the
 * eager residue only after adacomp_materialize. The fix-up is deferred for every
 * layer when all of the handle's layers have 16 <= L_T <= 509, or all have
 * 510 <= L_T <= 8189; in a handle that mixes the ranges or holds other bin lengths
 * it is deferred for the layers with 16 <= L_T <= 509 and the others are fixed up
 * eagerly as before.
 *
 * *compress_ws_bytes receives the workspace size in this mode (it grows by 512
 * bytes per tile unless all layers lie in one of the two ranges above, whose
 * workspaces hold the masks in both modes), and the workspace must be zero-filled before its first use. Consecutive
 * calls must use the same workspace; materialise before checkpointing the residue,
 * before switching the mode off, or after a call that reported an error (then also
 * zero the workspace). adacomp_compress_static_ws rejects such handles
 * (ADACOMP_ERR_INVALID_ARG): its workspace is not kept between calls. */
adacomp_status adacomp_set_lazy_fixup(adacomp_layer_t h, int32_t enable, size_t* compress_ws_bytes);

/* Applies every pending deferred correction to residue[] (layer order of the
 * handle) and clears it; asynchronous on `stream`. Does nothing when the handle
 * defers nothing. Same alignment and workspace rules as adacomp_compress. */
adacomp_status adacomp_materialize(adacomp_layer_t h, float* residue, void* ws, size_t ws_bytes,
                                   cudaStream_t stream);
adacomp_status adacomp_materialize_group(adacomp_layer_t h, float* const* residue, void* ws, size_t ws_bytes,
                                         cudaStream_t stream);

/* Releases the handle. adacomp_free(NULL) does nothing. */
void adacomp_free(adacomp_layer_t h);

/* Static text for a status code. */
const char* adacomp_status_string(adacomp_status s);

#ifdef __cplusplus
}
#endif

#endif /* ADACOMP_H */
