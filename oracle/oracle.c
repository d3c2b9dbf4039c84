/*
 * oracle.c - plain, slow fp64 CPU oracle of the decode-time routed expert FFN.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and
 * the benchmark's CPU-baseline leg may call this library.  It shares no code
 * with the CUDA path: it parses the documented boundary blob format itself
 * and computes every result from its plain definition, in double precision,
 * with no blocking, fusion or reordering beyond the definition.
 *
 * What it computes (per token t, for one MoE layer):
 *   1. router GEMV   logit[e] = sum_h x[h] * W_r[e,h]
 *      ("the model's own router picks the experts": WISP post
 *      "WISP - 실행될 수 없는 것을 스트리밍하다", section "Insight" and
 *      "Lesson 2: the model's router is the best scheduler").
 *   2. scores: softmax over all E experts, or the logistic sigmoid.
 *   3. top-k by brute force: a full stable sort of all E by (score desc,
 *      id asc); k is a parameter of the model manifest (WARP post
 *      "WARP 소개", section on the cache-size paradox: num_experts_per_token).
 *   4. weights: softmax -> p_j / sum_sel p;  sigmoid -> s_j / sum_sel s.
 *   5. for each selected expert, its dense gate/up/down matrices are
 *      materialised from the low-bit record:
 *        RVQ (3.00 bits/weight residual vector quantisation, WASTE article
 *        "2.78조 파라미터 모델을 노트북에서", section on idle weights):
 *          W[r, 8q+i] = C0[c0][i] + C1[c1][i] + C2[c2][i]
 *        INT4 symmetric groups of 128 along the input dim:
 *          W[r, k] = q[r, k] * s[r, k/128]
 *      then g = Wg x, u = Wu x, h = g / (1 + exp(-g)) * u, y_e = Wd h.
 *   6. y = sum_j w_j y_{idx_j} (+ y_shared) is done by the Python wrapper.
 *
 * Parallelism: OpenMP over output rows only (each row is still the plain
 * loop); results do not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_RVQ = 1, OR_INT4 = 2 };
enum { OR_SOFTMAX = 0, OR_SIGMOID = 1 };

/* IEEE 754 binary16 -> double, written out from the format definition. */
static double half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int mant = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)mant, -24);                 /* subnormal: m * 2^-24 */
    else if (expo == 31)
        v = mant ? NAN : INFINITY;
    else
        v = ldexp(1.0 + mant / 1024.0, expo - 15);
    return sign ? -v : v;
}

/* bfloat16 -> double: the top 16 bits of an IEEE binary32. */
static double bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

int oracle_version(void) { return 1; }

int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Blob size of one matrix / one expert in the boundary format. */
long long oracle_matrix_bytes(int wfmt, int rows, int K)
{
    if (wfmt == OR_RVQ) {
        if (K % 8) return -1;
        return 3LL * 256 * 8 * 2 + (long long)rows * (K / 8) * 3;
    }
    if (wfmt == OR_INT4) {
        if (K % 128) return -1;
        return (long long)rows * K / 2 + (long long)rows * (K / 128) * 2;
    }
    return -1;
}

long long oracle_expert_bytes(int wfmt, int H, int F)
{
    long long a = oracle_matrix_bytes(wfmt, F, H);
    long long b = oracle_matrix_bytes(wfmt, H, F);
    if (a < 0 || b < 0) return -1;
    return 2 * a + b;
}

/* One row r of a matrix block, decoded into w[0..K) (fp64). */
static void decode_row(int wfmt, int rows, int K, const uint8_t* blk, int r, double* w)
{
    if (wfmt == OR_RVQ) {
        const uint8_t* cb = blk;                         /* fp16 [3][256][8] */
        const uint8_t* codes = blk + 3 * 256 * 8 * 2;    /* u8 [rows][K/8][3] */
        int G = K / 8;
        for (int q = 0; q < G; ++q) {
            for (int i = 0; i < 8; ++i) w[8 * q + i] = 0.0;
            for (int s = 0; s < 3; ++s) {
                int c = codes[((size_t)r * G + q) * 3 + s];
                for (int i = 0; i < 8; ++i) {
                    size_t off = (((size_t)s * 256 + c) * 8 + i) * 2;
                    uint16_t hb = (uint16_t)(cb[off] | (cb[off + 1] << 8));
                    w[8 * q + i] += half_to_double(hb);
                }
            }
        }
    } else {
        const uint8_t* nib = blk;                                 /* [rows][K/2] */
        const uint8_t* sc = blk + (size_t)rows * K / 2;           /* fp16 [rows][K/128] */
        int NG = K / 128;
        for (int k = 0; k < K; ++k) {
            uint8_t byte = nib[(size_t)r * (K / 2) + k / 2];
            int u = (k % 2 == 0) ? (byte & 0xf) : (byte >> 4);
            int q = (u >= 8) ? u - 16 : u;                /* two's complement nibble */
            size_t so = ((size_t)r * NG + k / 128) * 2;
            uint16_t hb = (uint16_t)(sc[so] | (sc[so + 1] << 8));
            w[k] = (double)q * half_to_double(hb);
        }
    }
}

/* Materialise a whole matrix block as dense fp64 W[rows][K]. */
int oracle_dense(int wfmt, int rows, int K, const uint8_t* blk, double* W)
{
    if (oracle_matrix_bytes(wfmt, rows, K) < 0) return 1;
    for (int r = 0; r < rows; ++r) decode_row(wfmt, rows, K, blk, r, W + (size_t)r * K);
    return 0;
}

/* y[n][rows] = W x[n][K], with W decoded row by row. */
int oracle_matvec(int wfmt, int rows, int K, const uint8_t* blk, int n,
                  const double* x, double* y)
{
    if (oracle_matrix_bytes(wfmt, rows, K) < 0) return 1;
#pragma omp parallel
    {
        double* w = (double*)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(static)
        for (int r = 0; r < rows; ++r) {
            decode_row(wfmt, rows, K, blk, r, w);
            for (int t = 0; t < n; ++t) {
                double acc = 0.0;
                const double* xt = x + (size_t)t * K;
                for (int k = 0; k < K; ++k) acc += w[k] * xt[k];
                y[(size_t)t * rows + r] = acc;
            }
        }
        free(w);
    }
    return 0;
}

/* SwiGLU expert: g = Wg x, u = Wu x, h = silu(g) * u, y = Wd h.
 * x [n][H] fp64, h [n][F] (may be NULL), y [n][H]. */
int oracle_expert(int wfmt, int H, int F, const uint8_t* blob, int n,
                  const double* x, double* h_out, double* y)
{
    long long mg = oracle_matrix_bytes(wfmt, F, H);
    long long md = oracle_matrix_bytes(wfmt, H, F);
    if (mg < 0 || md < 0 || n < 0) return 1;
    if (n == 0) return 0;
    double* g = (double*)malloc(sizeof(double) * (size_t)n * F);
    double* u = (double*)malloc(sizeof(double) * (size_t)n * F);
    double* h = (double*)malloc(sizeof(double) * (size_t)n * F);
    if (!g || !u || !h) { free(g); free(u); free(h); return 2; }
    oracle_matvec(wfmt, F, H, blob, n, x, g);
    oracle_matvec(wfmt, F, H, blob + mg, n, x, u);
    for (size_t i = 0; i < (size_t)n * F; ++i)
        h[i] = g[i] / (1.0 + exp(-g[i])) * u[i];
    oracle_matvec(wfmt, H, F, blob + 2 * mg, n, h, y);
    if (h_out) memcpy(h_out, h, sizeof(double) * (size_t)n * F);
    free(g); free(u); free(h);
    return 0;
}

/* Router + scores + brute-force top-k + weights for T tokens.
 * x_bf16 [T][H] (bf16 bits), Wr [E][H] fp32.  Outputs: logits, scores
 * [T][E]; idx [T][k] int, w [T][k] fp64 ordered by descending score;
 * gap[t] = score of rank k-1 minus score of rank k (INFINITY when k == E). */
int oracle_router(int T, int H, int E, int k, int kind,
                  const uint16_t* x_bf16, const float* Wr,
                  double* logits, double* scores, int* idx, double* w, double* gap)
{
    if (T < 0 || H <= 0 || E <= 0 || k <= 0 || k > E) return 1;
    if (kind != OR_SOFTMAX && kind != OR_SIGMOID) return 1;
    int* order = (int*)malloc(sizeof(int) * (size_t)E);
    if (!order) return 2;
    for (int t = 0; t < T; ++t) {
        double* lg = logits + (size_t)t * E;
        double* sc = scores + (size_t)t * E;
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int hh = 0; hh < H; ++hh)
                acc += bf16_to_double(x_bf16[(size_t)t * H + hh]) * (double)Wr[(size_t)e * H + hh];
            lg[e] = acc;
        }
        if (kind == OR_SOFTMAX) {
            double m = lg[0];
            for (int e = 1; e < E; ++e) if (lg[e] > m) m = lg[e];
            double z = 0.0;
            for (int e = 0; e < E; ++e) z += exp(lg[e] - m);
            for (int e = 0; e < E; ++e) sc[e] = exp(lg[e] - m) / z;
        } else {
            for (int e = 0; e < E; ++e) sc[e] = 1.0 / (1.0 + exp(-lg[e]));
        }
        /* stable insertion sort by (score desc, id asc): plain brute force */
        for (int e = 0; e < E; ++e) order[e] = e;
        for (int i = 1; i < E; ++i) {
            int v = order[i], j = i - 1;
            while (j >= 0 && sc[order[j]] < sc[v]) { order[j + 1] = order[j]; --j; }
            order[j + 1] = v;
        }
        double sum = 0.0;
        for (int j = 0; j < k; ++j) sum += sc[order[j]];
        for (int j = 0; j < k; ++j) {
            idx[(size_t)t * k + j] = order[j];
            w[(size_t)t * k + j] = sc[order[j]] / sum;
        }
        gap[t] = (k < E) ? sc[order[k - 1]] - sc[order[k]] : INFINITY;
    }
    free(order);
    return 0;
}
