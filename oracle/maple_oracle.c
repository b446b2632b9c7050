/*
 * Plain, single-threaded CPU oracle for the ternary mixture-of-experts FFN step
 * described for DeepGrove's Maple-Preview.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file: only the test suite, the smoke check and the CPU-baseline leg of the
 * benchmark use it.  It shares no code, header, table or constant with the CUDA
 * library; every step is written out from the pages in fp64.
 *
 * Passages followed (page title, section):
 *  - "Maple-Preview: a 20B reasoning model where 97% of the weights are -1, 0, or +1"
 *    (ai.thesatyajit.com), section "The claim, verified from the bytes": every row
 *    holds exactly the three values -s, 0, +s with s per output row (BitNet b1.58
 *    shape), produced by absmean ternarization; the MoE router is full precision and
 *    picks 8 of 256 experts by logit margin.
 *  - same page, section "The 5.31 GB claim reconciles": five trits per byte,
 *    3^5 = 243 <= 256, plus per-row scales.
 *  - same page, section "The shipped code does no quantization": the expert body
 *    down(act(clamp(gate x, max=7)) * clamp(up x, -7, 7)).
 *  - "IA de 20B Rodando a 120 tok/s no iPhone" (codeinsider.com.br), section
 *    "Pesos ternarios: quando menos e absurdamente mais": weight 0 skips the
 *    activation, +1 adds it, -1 subtracts it; section "256 experts, 8 ativos":
 *    8 of 256 experts are active per token.
 *  - "DeepGrove ... Maple-Preview" (jj-blog), config bullets: hidden 2048,
 *    moe_intermediate_size 512, 256 experts, top-8, no shared expert.
 *
 * Readings where the pages are silent (each is listed with its reason in the
 * design notes):
 *  - rounding is round-half-to-even, so |w|/s == 0.5 gives 0;
 *  - an all-zero row has s = 0 and all trits 0 (no epsilon);
 *  - digit i of a byte is (q_{5b+i} + 1) and the byte is sum_i digit_i * 3^i, with
 *    the lowest column index as the least significant base-3 digit; K-tail trits
 *    are 0 (digit 1);
 *  - the router adds an optional per-expert bias, ranks logits with ties going to
 *    the lower expert index, and normalises the k selected with a softmax;
 *  - act_fn is SiLU; the clamp bound is a parameter (7 for Maple, +inf for plain
 *    SwiGLU);
 *  - the k expert outputs are combined as y = sum_j w_j * expert_j(x).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG (-1)
#define ORACLE_BAD_CODE (-6)

/* bf16 is the upper half of an IEEE binary32; widening to double is exact. */
static double bf16_bits_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int64_t oracle_packed_row_bytes(int64_t K) { return (K + 4) / 5; }

/*
 * Absmean ternarization of one bf16 row-major matrix [rows x K].
 * s_r = (1/K) * sum_j |w_rj|, accumulated in fp64 and rounded once to fp32;
 * q_rj = clamp(round(w_rj / s_r), -1, 1) with round-half-to-even.
 * ("The claim, verified from the bytes": -s, 0, +s per row, absmean shape.)
 */
int oracle_ternarize(const uint16_t* w, int64_t rows, int64_t K, int8_t* q, float* s) {
    if (!w || !q || !s || rows < 0 || K <= 0) return ORACLE_BAD_ARG;
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* wr = w + r * K;
        double acc = 0.0;
        for (int64_t j = 0; j < K; ++j) acc += fabs(bf16_bits_to_double(wr[j]));
        float sf = (float)(acc / (double)K);
        s[r] = sf;
        for (int64_t j = 0; j < K; ++j) {
            double v = bf16_bits_to_double(wr[j]);
            int8_t t = 0;
            if (sf != 0.0f) {
                double ratio = v / (double)sf;
                double rounded = nearbyint(ratio); /* default mode: ties to even */
                if (rounded > 1.0) rounded = 1.0;
                if (rounded < -1.0) rounded = -1.0;
                t = (int8_t)rounded;
            }
            q[r * K + j] = t;
        }
    }
    return ORACLE_OK;
}

/*
 * Trits and scales of a matrix whose rows are already ternary.  The released
 * checkpoint stores each expert weight as a bf16 value -s, 0 or +s of its row ("The
 * claim, verified from the bytes": exactly three values per row), so the row's scale
 * is its largest magnitude and each trit is the sign of its weight:
 * s_r = max_j |w_rj| and q_rj = sign(w_rj) (0 for +0 and -0).  A row with two different
 * nonzero magnitudes is not ternary: it is counted in *bad_rows and still gets the
 * sign trits and the max scale.
 */
int oracle_ternary_exact(const uint16_t* w, int64_t rows, int64_t K, int8_t* q, float* s, int64_t* bad_rows) {
    if (!w || !q || !s || !bad_rows || rows < 0 || K <= 0) return ORACLE_BAD_ARG;
    *bad_rows = 0;
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* wr = w + r * K;
        double m = 0.0;
        for (int64_t j = 0; j < K; ++j) {
            double a = fabs(bf16_bits_to_double(wr[j]));
            if (a > m) m = a;
        }
        int bad = 0;
        for (int64_t j = 0; j < K; ++j) {
            double v = bf16_bits_to_double(wr[j]);
            int8_t t = 0;
            if (v > 0.0) t = 1;
            if (v < 0.0) t = -1;
            if (t != 0 && fabs(v) != m) bad = 1;
            q[r * K + j] = t;
        }
        s[r] = (float)m; /* a bf16 magnitude: exact in fp32 */
        *bad_rows += bad;
    }
    return ORACLE_OK;
}

/*
 * Five trits per byte ("The 5.31 GB claim reconciles": 3^5 = 243 fits in 256).
 * byte = sum_{i=0..4} (q_{5b+i} + 1) * 3^i; missing tail trits count as 0.
 */
int oracle_pack(const int8_t* q, int64_t rows, int64_t K, uint8_t* packed) {
    if (!q || !packed || rows < 0 || K <= 0) return ORACLE_BAD_ARG;
    int64_t nb = oracle_packed_row_bytes(K);
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            int value = 0;
            int place = 1;
            for (int i = 0; i < 5; ++i) {
                int64_t j = 5 * b + i;
                int trit = (j < K) ? q[r * K + j] : 0;
                if (trit < -1 || trit > 1) return ORACLE_BAD_ARG;
                value += (trit + 1) * place;
                place *= 3;
            }
            packed[r * nb + b] = (uint8_t)value;
        }
    }
    return ORACLE_OK;
}

/*
 * Inverse of oracle_pack by repeated division by 3.  Codes 243..255 are not
 * produced by any trit pattern and are reported as ORACLE_BAD_CODE.
 */
int oracle_unpack(const uint8_t* packed, int64_t rows, int64_t K, int8_t* q) {
    if (!packed || !q || rows < 0 || K <= 0) return ORACLE_BAD_ARG;
    int64_t nb = oracle_packed_row_bytes(K);
    int status = ORACLE_OK;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            int code = packed[r * nb + b];
            if (code >= 243) {
                status = ORACLE_BAD_CODE;
                code = 121; /* decode as five zeros so that the output stays defined */
            }
            for (int i = 0; i < 5; ++i) {
                int digit = code % 3;
                code /= 3;
                int64_t j = 5 * b + i;
                if (j < K) q[r * K + j] = (int8_t)(digit - 1);
            }
        }
    }
    return status;
}

/* Ranking key for the router: larger logit first, then lower expert index. */
typedef struct {
    double logit;
    int32_t expert;
} ranked_logit;

static int rank_cmp(const void* a, const void* b) {
    const ranked_logit* x = (const ranked_logit*)a;
    const ranked_logit* y = (const ranked_logit*)b;
    if (x->logit > y->logit) return -1;
    if (x->logit < y->logit) return 1;
    return (x->expert < y->expert) ? -1 : (x->expert > y->expert);
}

/*
 * Full-precision router ("The claim, verified from the bytes": the router picks 8
 * of 256 experts from the logit margin and is kept in full precision).
 * logits[t][e] = sum_j x_tj * Wr_ej (+ bias_e), exact products in fp64;
 * idx[t][0..k) = the k largest logits in descending order (ties: lower index);
 * w[t][i] = softmax over the k selected logits.
 */
int oracle_route(const uint16_t* x, const uint16_t* Wr, const double* bias, int64_t T,
                 int64_t H, int64_t E, int64_t k, double* logits, int32_t* idx, double* w) {
    if (!x || !Wr || !logits || !idx || !w || T < 0 || H <= 0 || E <= 0 || k <= 0 || k > E)
        return ORACLE_BAD_ARG;
    ranked_logit* order = (ranked_logit*)malloc(sizeof(ranked_logit) * (size_t)E);
    if (!order) return ORACLE_BAD_ARG;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int64_t j = 0; j < H; ++j)
                acc += bf16_bits_to_double(x[t * H + j]) * bf16_bits_to_double(Wr[e * H + j]);
            if (bias) acc += bias[e];
            logits[t * E + e] = acc;
            order[e].logit = acc;
            order[e].expert = (int32_t)e;
        }
        qsort(order, (size_t)E, sizeof(ranked_logit), rank_cmp);
        double top = order[0].logit;
        double denom = 0.0;
        for (int64_t i = 0; i < k; ++i) denom += exp(order[i].logit - top);
        for (int64_t i = 0; i < k; ++i) {
            idx[t * k + i] = order[i].expert;
            w[t * k + i] = exp(order[i].logit - top) / denom;
        }
    }
    free(order);
    return ORACLE_OK;
}

/*
 * Token-to-expert grouping: counts[e] = number of (t, i) slots routed to e,
 * offsets = exclusive prefix sum of counts (E + 1 entries), perm lists the slot
 * numbers s = t * k + i of each expert in increasing slot order.
 */
int oracle_group(const int32_t* idx, int64_t T, int64_t k, int64_t E, int32_t* counts,
                 int32_t* offsets, int32_t* perm) {
    if (!idx || !counts || !offsets || !perm || T < 0 || k <= 0 || E <= 0) return ORACLE_BAD_ARG;
    int64_t slots = T * k;
    for (int64_t e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t s = 0; s < slots; ++s) {
        if (idx[s] < 0 || idx[s] >= E) return ORACLE_BAD_ARG;
        counts[idx[s]] += 1;
    }
    offsets[0] = 0;
    for (int64_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t* cursor = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
    if (!cursor) return ORACLE_BAD_ARG;
    for (int64_t e = 0; e < E; ++e) cursor[e] = offsets[e];
    for (int64_t s = 0; s < slots; ++s) perm[cursor[idx[s]]++] = (int32_t)s;
    free(cursor);
    return ORACLE_OK;
}

/* Dot product of one packed ternary row with a dense vector by the add / subtract /
 * skip rule ("Pesos ternarios": 0 skips, +1 adds, -1 subtracts). */
static double ternary_row_dot(const uint8_t* row, int64_t K, const double* v, int* bad) {
    double acc = 0.0;
    int64_t nb = oracle_packed_row_bytes(K);
    for (int64_t b = 0; b < nb; ++b) {
        int code = row[b];
        if (code >= 243) {
            *bad = 1;
            continue;
        }
        for (int i = 0; i < 5; ++i) {
            int digit = code % 3;
            code /= 3;
            int64_t j = 5 * b + i;
            if (j >= K) break;
            if (digit == 2)
                acc += v[j];
            else if (digit == 0)
                acc -= v[j];
        }
    }
    return acc;
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

/*
 * Expert FFN with weighted combine.  For each token t and each of its k slots i
 * with expert e = idx[t][i] and weight w[t][i]:
 *   g_r = s_gate[e][r] * <q_gate[e][r], x_t>,  u_r = s_up[e][r] * <q_up[e][r], x_t>
 *   h_r = silu(min(g_r, clamp)) * min(max(u_r, -clamp), clamp)
 *   y_t[c] += w[t][i] * s_down[e][c] * <q_down[e][c], h>
 * ("The shipped code does no quantization": the MapleMLP forward with its clamps.)
 * Layouts: gate, up [E][I][ceil(H/5)]; down [E][H][ceil(I/5)]; scales [E][I],
 * [E][I], [E][H]; x bf16 [T][H]; y fp64 [T][H].
 */
int oracle_moe_ffn(const uint8_t* gate, const uint8_t* up, const uint8_t* down,
                   const float* s_gate, const float* s_up, const float* s_down, int64_t E,
                   int64_t H, int64_t I, double clamp, const uint16_t* x, const int32_t* idx,
                   const double* w, int64_t T, int64_t k, double* y) {
    if (!gate || !up || !down || !s_gate || !s_up || !s_down || !x || !idx || !w || !y ||
        E <= 0 || H <= 0 || I <= 0 || T < 0 || k <= 0)
        return ORACLE_BAD_ARG;
    int64_t bh = oracle_packed_row_bytes(H);
    int64_t bi = oracle_packed_row_bytes(I);
    double* xv = (double*)malloc(sizeof(double) * (size_t)H);
    double* h = (double*)malloc(sizeof(double) * (size_t)I);
    if (!xv || !h) {
        free(xv);
        free(h);
        return ORACLE_BAD_ARG;
    }
    int bad = 0;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t j = 0; j < H; ++j) xv[j] = bf16_bits_to_double(x[t * H + j]);
        for (int64_t c = 0; c < H; ++c) y[t * H + c] = 0.0;
        for (int64_t i = 0; i < k; ++i) {
            int32_t e = idx[t * k + i];
            if (e < 0 || e >= E) {
                free(xv);
                free(h);
                return ORACLE_BAD_ARG;
            }
            for (int64_t r = 0; r < I; ++r) {
                double g = (double)s_gate[e * I + r] *
                           ternary_row_dot(gate + (e * I + r) * bh, H, xv, &bad);
                double u = (double)s_up[e * I + r] *
                           ternary_row_dot(up + (e * I + r) * bh, H, xv, &bad);
                double gc = (g < clamp) ? g : clamp;
                double uc = (u < -clamp) ? -clamp : ((u > clamp) ? clamp : u);
                h[r] = silu(gc) * uc;
            }
            for (int64_t c = 0; c < H; ++c) {
                double d = ternary_row_dot(down + (e * H + c) * bi, I, h, &bad);
                y[t * H + c] += w[t * k + i] * ((double)s_down[e * H + c] * d);
            }
        }
    }
    free(xv);
    free(h);
    return bad ? ORACLE_BAD_CODE : ORACLE_OK;
}
