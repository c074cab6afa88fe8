/*
 * AdaComp CPU oracle — TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded restatement of AdaComp's per-layer compressor
 * and of the K-learner decoder, used to check the CUDA path. Only the test suite,
 * the package's smoke check and the benchmark's CPU-baseline leg may load it; the
 * product path never does. It shares no code, header, table or helper with the
 * CUDA library.
 *
 * Method source: "AdaComp (Adaptive Residual Gradient Compression)", the curated
 * entry's summary paragraph and its Claims > Mechanism
 * #r629-local-bin-soft-threshold-and-mean-gmax-quantization (Algorithm 2 restated):
 *   G = residue + dW;  H = G + dW;  bins of length L_T over G;
 *   g_max(i) = max |G| over bin i;  s = (1/B) sum_i g_max(i);
 *   send every element with |H| >= g_max(i) as sign(G) * s;
 *   residue = G - G_q for sent elements, residue = G for the rest.
 * Code widths: Claims > Application #r629-conv-40x-and-fc-lstm-200x-... and
 * Curated Limitations (8-bit codes when L_T < 64, 16-bit otherwise).
 *
 * Readings taken where the pages are silent (each is pinned by a test):
 *   - a partial last bin counts as a bin; its g_max is over its own elements;
 *   - an element is sent only when G != 0 (sign(0) has no code);
 *   - the tie |H| == g_max is sent;
 *   - H = fl32(G + dW), evaluated after G is rounded;
 *   - s = fl32( fl64(exact sum of g_max) / B ), i.e. the exact real sum rounded
 *     once to fp64, divided by B in fp64, rounded once to fp32;
 *   - message = s (f32 LE) | B (u32 LE) | count[B] (u16 LE) | codes in bin order
 *     and ascending offset, code = offset << 1 | (G < 0);
 *   - decode adds sign * s_k into a dense fp32 buffer for k = 0..K-1 in order.
 *
 * Build: gcc -O2 -ffp-contract=off -shared -fPIC (no fast-math, no FMA contraction).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_CAPACITY 2
#define ORACLE_ERR_BAD_MESSAGE 3

static float u32_as_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t f32_as_u32(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* bf16 -> fp32 widening is exact: the 16 bits become the top half of the fp32 word. */
static float bf16_bits_to_f32(uint16_t h) { return u32_as_f32((uint32_t)h << 16); }

static int64_t bin_count(int64_t n, int32_t L) { return (n + L - 1) / L; }
static int code_width(int32_t L) { return L < 64 ? 1 : 2; }

int64_t adacomp_oracle_max_msg_bytes(int64_t n, int32_t L)
{
    if (n < 1 || L < 1) return -1;
    return 8 + 2 * bin_count(n, L) + (int64_t)code_width(L) * n;
}

/*
 * Exact sum of non-negative finite fp32 values, rounded to the nearest fp64
 * (ties to even). Every fp32 is an integer multiple of 2^-149, so the sum is
 * accumulated as a plain multi-word integer in units of 2^-149 and rounded once.
 */
#define SUM_WORDS 12 /* 384 bits: 2^277 per term, room for 2^100 terms */

static void big_add_shifted(uint32_t *acc, uint64_t m, int shift)
{
    int word = shift / 32, bit = shift % 32;
    /* m < 2^24, so m << bit fits in 56 bits: spread it over three words */
    uint64_t v = m << bit;
    uint64_t carry = 0;
    for (int i = word; i < SUM_WORDS; ++i) {
        uint64_t part = (i == word) ? (v & 0xffffffffu) : (i == word + 1) ? (v >> 32) : 0;
        uint64_t t = (uint64_t)acc[i] + part + carry;
        acc[i] = (uint32_t)t;
        carry = t >> 32;
        if (i > word + 1 && carry == 0) break;
    }
}

static int big_get_bit(const uint32_t *acc, int i) { return (acc[i / 32] >> (i % 32)) & 1; }

double adacomp_oracle_exact_sum_f32(const float *x, int64_t n)
{
    uint32_t acc[SUM_WORDS];
    memset(acc, 0, sizeof acc);
    for (int64_t i = 0; i < n; ++i) {
        uint32_t u = f32_as_u32(x[i]) & 0x7fffffffu; /* callers pass values >= 0 */
        uint32_t e = u >> 23, f = u & 0x7fffffu;
        if (e == 255) return (double)INFINITY; /* not finite: unspecified, report inf */
        uint64_t m = e ? (f | 0x800000u) : f;
        int shift = e ? (int)e - 1 : 0; /* value = m * 2^(max(e,1) - 150) = m * 2^shift * 2^-149 */
        big_add_shifted(acc, m, shift);
    }
    int top = -1;
    for (int i = SUM_WORDS * 32 - 1; i >= 0; --i)
        if (big_get_bit(acc, i)) { top = i; break; }
    if (top < 0) return 0.0;
    uint64_t mant = 0;
    int lo = top - 52; /* lowest bit kept in the 53-bit significand */
    if (lo <= 0) {
        for (int i = top; i >= 0; --i) mant = (mant << 1) | (uint64_t)big_get_bit(acc, i);
        return ldexp((double)mant, -149);
    }
    for (int i = top; i >= lo; --i) mant = (mant << 1) | (uint64_t)big_get_bit(acc, i);
    int round = big_get_bit(acc, lo - 1);
    int sticky = 0;
    for (int i = lo - 2; i >= 0; --i)
        if (big_get_bit(acc, i)) { sticky = 1; break; }
    if (round && (sticky || (mant & 1))) mant += 1; /* mant may become 2^53: still exact */
    return ldexp((double)mant, lo - 149);
}

static float load_dw(const void *dw, int dw_bf16, int64_t j)
{
    if (dw_bf16) return bf16_bits_to_f32(((const uint16_t *)dw)[j]);
    return ((const float *)dw)[j];
}

static void put_u16(uint8_t *p, uint32_t v) { p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); }
static void put_u32(uint8_t *p, uint32_t v)
{
    p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); p[2] = (uint8_t)(v >> 16); p[3] = (uint8_t)(v >> 24);
}
static uint32_t get_u16(const uint8_t *p) { return (uint32_t)p[0] | ((uint32_t)p[1] << 8); }
static uint32_t get_u32(const uint8_t *p)
{
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

/*
 * One AdaComp step for one layer (Algorithm 2 as restated in the curated entry's
 * Mechanism claim). residue is updated in place. Optional outputs: s, g_max[B],
 * sel[n] (1 = sent). literal_zero_select = 1 applies |H| >= g_max without the
 * G != 0 conjunct (documentation only: it sends zeros as +s codes).
 * local_selection = 1 is the hard Local Selection rule the entry contrasts with
 * AdaComp (Claims > Mechanism #r629-self-adjusting-sparsity-prevents-residual-
 * explosion): no soft-threshold probe, so the comparison is |G| >= g_max and only
 * a bin's maxima are sent; everything else (s, codes, residue) is unchanged.
 */
int adacomp_oracle_compress(int64_t n, int32_t L, int dw_bf16, float *residue, const void *dw,
                            uint8_t *msg, uint64_t msg_cap, uint64_t *msg_len,
                            float *s_out, float *gmax_out, uint8_t *sel_out,
                            int literal_zero_select, int local_selection)
{
    if (n < 1 || L < 1 || L > 32768 || !residue || !dw || !msg) return ORACLE_ERR_ARG;
    int64_t B = bin_count(n, L);
    if (B >= ((int64_t)1 << 32)) return ORACLE_ERR_ARG;
    int w = code_width(L);
    if (msg_cap < (uint64_t)(8 + 2 * B)) return ORACLE_ERR_CAPACITY;

    float *G = (float *)malloc((size_t)n * sizeof(float));
    float *H = (float *)malloc((size_t)n * sizeof(float));
    float *gmax = (float *)malloc((size_t)B * sizeof(float));
    if (!G || !H || !gmax) { free(G); free(H); free(gmax); return ORACLE_ERR_ARG; }

    /* G = residue + dW, then H = G + dW: two separately rounded fp32 additions */
    for (int64_t j = 0; j < n; ++j) {
        float d = load_dw(dw, dw_bf16, j);
        G[j] = residue[j] + d;
        H[j] = G[j] + d;
        if (local_selection) H[j] = G[j]; /* Local Selection: compare G itself */
    }

    /* g_max(i): largest |G| in bin i; the last bin may be shorter than L */
    for (int64_t b = 0; b < B; ++b) {
        int64_t lo = b * L, hi = lo + L < n ? lo + L : n;
        float m = 0.0f;
        for (int64_t j = lo; j < hi; ++j)
            if (fabsf(G[j]) > m) m = fabsf(G[j]);
        gmax[b] = m;
    }

    /* s = mean of g_max over all B bins */
    double S = adacomp_oracle_exact_sum_f32(gmax, B);
    float s = (float)(S / (double)B);

    put_u32(msg, f32_as_u32(s));
    put_u32(msg + 4, (uint32_t)B);
    uint8_t *counts = msg + 8;
    uint64_t pos = 8 + 2 * (uint64_t)B; /* next code byte */

    for (int64_t b = 0; b < B; ++b) {
        int64_t lo = b * L, hi = lo + L < n ? lo + L : n;
        uint32_t cnt = 0;
        for (int64_t j = lo; j < hi; ++j) {
            int nonzero = G[j] != 0.0f;
            int sel = (literal_zero_select || nonzero) && fabsf(H[j]) >= gmax[b];
            if (sel_out) sel_out[j] = (uint8_t)sel;
            if (sel) {
                uint32_t code = ((uint32_t)(j - lo) << 1) | (G[j] < 0.0f ? 1u : 0u);
                if (pos + (uint64_t)w > msg_cap) {
                    free(G); free(H); free(gmax);
                    return ORACLE_ERR_CAPACITY;
                }
                if (w == 1) msg[pos] = (uint8_t)code;
                else put_u16(msg + pos, code);
                pos += (uint64_t)w;
                ++cnt;
                /* residue = G - sign(G) * s */
                if (G[j] > 0.0f) residue[j] = G[j] - s;
                else if (G[j] < 0.0f) residue[j] = G[j] + s;
                else residue[j] = G[j];
            } else {
                residue[j] = G[j];
            }
        }
        put_u16(counts + 2 * b, cnt);
    }

    if (msg_len) *msg_len = pos;
    if (s_out) *s_out = s;
    if (gmax_out) memcpy(gmax_out, gmax, (size_t)B * sizeof(float));
    free(G); free(H); free(gmax);
    return ORACLE_OK;
}

/*
 * Whether one message of length len (bytes) is a well-formed message of a layer of
 * n elements with bins of L. Messages are variable-length ("AdaComp (Adaptive
 * Residual Gradient Compression)", Claims > Limitation
 * #r629-minibatch-size-activity-and-variable-message-length), so the length that
 * came with the message is checked against what its counts say, and nothing past it
 * is read. The checks, in order: room for the header and the counts (8 + 2B bytes);
 * the header's B is the layer's; no count exceeds its bin's length; the length is
 * exactly 8 + 2B + w * (sum of the counts); within every bin the code offsets rise
 * strictly (the compressor lists a bin's sent elements once each, in ascending
 * offset) and stay below the bin's length.
 */
static int message_ok(int64_t n, int32_t L, const uint8_t *m, uint64_t len)
{
    int64_t B = bin_count(n, L);
    int w = code_width(L);
    if (!m || len < 8 + 2 * (uint64_t)B) return 0;
    if ((int64_t)get_u32(m + 4) != B) return 0;
    uint64_t total = 0;
    for (int64_t b = 0; b < B; ++b) {
        int64_t blen = (b + 1) * L < n ? L : n - b * L;
        uint32_t cnt = get_u16(m + 8 + 2 * b);
        if ((int64_t)cnt > blen) return 0;
        total += cnt;
    }
    if (len != 8 + 2 * (uint64_t)B + (uint64_t)w * total) return 0;
    uint64_t pos = 8 + 2 * (uint64_t)B;
    for (int64_t b = 0; b < B; ++b) {
        int64_t blen = (b + 1) * L < n ? L : n - b * L;
        uint32_t cnt = get_u16(m + 8 + 2 * b);
        int64_t prev = -1;
        for (uint32_t c = 0; c < cnt; ++c) {
            uint32_t code = (w == 1) ? m[pos] : get_u16(m + pos);
            pos += (uint64_t)w;
            int64_t off = (int64_t)(code >> 1);
            if (off >= blen || off <= prev) return 0;
            prev = off;
        }
    }
    return 1;
}

/*
 * Decode-and-accumulate: dense[j] += (sign ? -s_k : +s_k) for every code of
 * message k, k = 0..K-1 in order. Every message is checked first (message_ok); a
 * message that fails adds nothing, the others are summed as usual, and the call
 * returns ORACLE_ERR_BAD_MESSAGE (bad_out[k], when given, marks each rejected
 * message). lens[k] is message k's length in bytes.
 */
int adacomp_oracle_decode_accumulate(int64_t n, int32_t L, const uint8_t *const *msgs, const uint64_t *lens,
                                     int32_t K, float *dense, uint8_t *bad_out)
{
    if (n < 1 || L < 1 || L > 32768 || K < 1 || !msgs || !lens || !dense) return ORACLE_ERR_ARG;
    int64_t B = bin_count(n, L);
    int w = code_width(L);
    int any_bad = 0;
    for (int32_t k = 0; k < K; ++k) {
        int ok = message_ok(n, L, msgs[k], lens[k]);
        if (bad_out) bad_out[k] = (uint8_t)!ok;
        if (!ok) any_bad = 1;
    }
    for (int32_t k = 0; k < K; ++k) {
        if (!message_ok(n, L, msgs[k], lens[k])) continue;
        const uint8_t *m = msgs[k];
        float s = u32_as_f32(get_u32(m));
        uint64_t pos = 8 + 2 * (uint64_t)B;
        for (int64_t b = 0; b < B; ++b) {
            uint32_t cnt = get_u16(m + 8 + 2 * b);
            for (uint32_t c = 0; c < cnt; ++c) {
                uint32_t code = (w == 1) ? m[pos] : get_u16(m + pos);
                pos += (uint64_t)w;
                int64_t j = b * L + (int64_t)(code >> 1);
                dense[j] = dense[j] + ((code & 1u) ? -s : s);
            }
        }
    }
    return any_bad ? ORACLE_ERR_BAD_MESSAGE : ORACLE_OK;
}

/*
 * Decode K messages into the aggregated gradient g (a zero-filled fp32 buffer,
 * learners in order, exactly as adacomp_oracle_decode_accumulate, a rejected
 * message adding nothing) and apply one momentum-SGD step to weights w and
 * momentum v (the optimiser of the entry's Claims > Application
 * #r629-conv-40x-and-fc-lstm-200x-compression-across-optimizers; the rule is read as
 * the heavy-ball form without dampening):
 *     v = fl32(fl32(mu * v) + fl32(scale * g));   w = fl32(w - fl32(lr * v)).
 * Returns ORACLE_ERR_BAD_MESSAGE when a message was rejected (the step is still
 * applied with the others).
 */
int adacomp_oracle_decode_sgd(int64_t n, int32_t L, const uint8_t *const *msgs, const uint64_t *lens, int32_t K,
                              float *w, float *v, float lr, float mu, float scale)
{
    if (n < 1 || !w || !v) return ORACLE_ERR_ARG;
    float *g = (float *)calloc((size_t)n, sizeof(float));
    if (!g) return ORACLE_ERR_ARG;
    int rc = adacomp_oracle_decode_accumulate(n, L, msgs, lens, K, g, NULL);
    if (rc != ORACLE_OK && rc != ORACLE_ERR_BAD_MESSAGE) { free(g); return rc; }
    for (int64_t j = 0; j < n; ++j) {
        float momentum = mu * v[j];
        float step = scale * g[j];
        v[j] = momentum + step;
        float delta = lr * v[j];
        w[j] = w[j] - delta;
    }
    free(g);
    return rc;
}

/*
 * Decode K messages into the aggregated gradient (a zero-filled fp32 buffer,
 * learners in order, exactly as adacomp_oracle_decode_accumulate, a rejected message
 * adding nothing) and apply one Adam step to weights w, first moment m and second
 * moment v (Adam is the other optimiser of the entry's Claims > Application
 * #r629-conv-40x-and-fc-lstm-200x-compression-across-optimizers; the pages give no
 * rule, so it is read as Kingma and Ba's Adam with the bias corrections written
 * out, each operation an fp32 operation rounded once, no fused multiply-add):
 *     g  = fl32(scale * sum)
 *     m  = fl32( fl32(beta1 * m) + fl32(fl32(1 - beta1) * g) )
 *     v  = fl32( fl32(beta2 * v) + fl32(fl32(1 - beta2) * fl32(g * g)) )
 *     mh = fl32(m / bc1);   vh = fl32(v / bc2)
 *     w  = fl32( w - fl32( lr * fl32( mh / fl32(sqrt(vh) + eps) ) ) )
 * bc1 = 1 - beta1^t and bc2 = 1 - beta2^t (step t's bias corrections) are given by
 * the caller. Returns ORACLE_ERR_BAD_MESSAGE when a message was rejected (the step
 * is still applied with the others).
 */
int adacomp_oracle_decode_adam(int64_t n, int32_t L, const uint8_t *const *msgs, const uint64_t *lens, int32_t K,
                               float *w, float *m, float *v, float lr, float beta1, float beta2, float eps,
                               float bc1, float bc2, float scale)
{
    if (n < 1 || !w || !m || !v) return ORACLE_ERR_ARG;
    float *sum = (float *)calloc((size_t)n, sizeof(float));
    if (!sum) return ORACLE_ERR_ARG;
    int rc = adacomp_oracle_decode_accumulate(n, L, msgs, lens, K, sum, NULL);
    if (rc != ORACLE_OK && rc != ORACLE_ERR_BAD_MESSAGE) { free(sum); return rc; }
    float one_minus_b1 = 1.0f - beta1;
    float one_minus_b2 = 1.0f - beta2;
    for (int64_t j = 0; j < n; ++j) {
        float g = scale * sum[j];
        float m_keep = beta1 * m[j];
        float m_add = one_minus_b1 * g;
        m[j] = m_keep + m_add;
        float g2 = g * g;
        float v_keep = beta2 * v[j];
        float v_add = one_minus_b2 * g2;
        v[j] = v_keep + v_add;
        float m_hat = m[j] / bc1;
        float v_hat = v[j] / bc2;
        float denom = sqrtf(v_hat) + eps;
        float ratio = m_hat / denom;
        float delta = lr * ratio;
        w[j] = w[j] - delta;
    }
    free(sum);
    return rc;
}
