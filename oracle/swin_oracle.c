/*
 * Plain float64 CPU oracle of the Swin shifted-window multi-head
 * self-attention block.  TEST INFRASTRUCTURE ONLY: the tests, the smoke
 * check and the benchmark's CPU-baseline leg load it; the GPU library never
 * does, and this file shares no code, header or table with the CUDA sources.
 *
 * What the block computes (pages: "Boosting Swin Transformer Speed:
 * Profiling, Mixed Precision, and Kernel Fusion Secrets", sections
 * Introduction and Training Optimization -- windowed attention, shifted
 * windows, window partition / shift / reverse index maps; "Swin Transformer
 * V2" (neura.market analysis), section How It Works -- relative position
 * bias, scaled cosine attention with tau clipped at 0.01, the meta-network G
 * over log-spaced coordinates):
 *
 *   S1  cyclic shift by -s:      xs[b,i,j] = x[b,(i+s) mod H,(j+s) mod W]
 *   S1  window partition:        window (b,wi,wj), token t = ti*M + tj
 *   S2  qkv = xw Wqkv^T + bqkv   (channel o = part*C + head*d + e, q,k,v)
 *   S3a V1 logit:  q.k / sqrt(d) + table[idx, head]
 *   S3b V2 logit:  cos(q,k) / max(tau_head, 0.01) + table[idx, head]
 *   S4  shift-region mask:       -inf between different regions (s > 0)
 *   S5  softmax over keys;  S6 o = p v;  S7 y = o Wproj^T + bproj
 *   S8  window reverse, then roll by +s back to the original frame
 *
 * The pages print no formula for the index maps, the mask, the relative
 * index or the V1/V2 logits (the V2 equation is lost from the page text).
 * Readings taken where they are silent:
 *   - roll by -s means the element at (i+s) mod n moves to i;
 *   - tokens are row-major inside a window, windows row-major per image;
 *   - relative index idx = (ri-rj+M-1)*(2M-1) + (ci-cj+M-1) with (r,c) the
 *     in-window coordinates of the query i and the key j (query minus key);
 *   - the shifted frame is cut into bands [0,H-M), [H-M,H-s), [H-s,H) per
 *     axis; region = (row band, column band); pairs from different regions
 *     are excluded outright (weight exactly zero);
 *   - V2: cos = q.k / (max(|q|,eps) max(|k|,eps)), eps = 1e-12, no 1/sqrt(d);
 *     logit_scale carries tau itself and 1/max(tau, 0.01) multiplies cos;
 *   - G: Linear(2->hidden, bias b1) -> ReLU -> Linear(hidden->heads, no
 *     bias) over (sign(dr) ln(1+|dr|), sign(dc) ln(1+|dc|)); its raw output
 *     is the table, row idx as above.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_V1 = 0, ORACLE_V2 = 1 };

/* ---- S1 / S8 index maps ------------------------------------------------ */

/* torch.roll semantics along one axis: y[i] = x[(i - r) mod n].  A cyclic
 * shift by -s is r = -s, so y[i] = x[(i + s) mod n]. */
static int roll_source(int i, int r, int n)
{
    int k = (i - r) % n;
    return k < 0 ? k + n : k;
}

/* y = roll(x, r) over the two spatial axes of a [B,H,W,C] tensor. */
void oracle_roll(const double *x, int B, int H, int W, int C, int r, double *y)
{
    for (int b = 0; b < B; ++b)
        for (int i = 0; i < H; ++i)
            for (int j = 0; j < W; ++j) {
                const double *src = x + (((size_t)b * H + roll_source(i, r, H)) * W
                                         + roll_source(j, r, W)) * C;
                double *dst = y + (((size_t)b * H + i) * W + j) * C;
                memcpy(dst, src, sizeof(double) * (size_t)C);
            }
}

/* xw[win][t][c] = xs[b, wi*M+ti, wj*M+tj, c], win = (b*(H/M)+wi)*(W/M)+wj,
 * t = ti*M + tj. */
void oracle_partition(const double *xs, int B, int H, int W, int C, int M, double *xw)
{
    const int nh = H / M, nw = W / M, N = M * M;
    for (int b = 0; b < B; ++b)
        for (int wi = 0; wi < nh; ++wi)
            for (int wj = 0; wj < nw; ++wj) {
                size_t win = ((size_t)b * nh + wi) * nw + wj;
                for (int t = 0; t < N; ++t) {
                    int i = wi * M + t / M, j = wj * M + t % M;
                    memcpy(xw + (win * N + t) * C, xs + (((size_t)b * H + i) * W + j) * C,
                           sizeof(double) * (size_t)C);
                }
            }
}

/* Inverse of oracle_partition. */
void oracle_reverse(const double *xw, int B, int H, int W, int C, int M, double *xs)
{
    const int nh = H / M, nw = W / M, N = M * M;
    for (int b = 0; b < B; ++b)
        for (int wi = 0; wi < nh; ++wi)
            for (int wj = 0; wj < nw; ++wj) {
                size_t win = ((size_t)b * nh + wi) * nw + wj;
                for (int t = 0; t < N; ++t) {
                    int i = wi * M + t / M, j = wj * M + t % M;
                    memcpy(xs + (((size_t)b * H + i) * W + j) * C, xw + (win * N + t) * C,
                           sizeof(double) * (size_t)C);
                }
            }
}

/* ---- S3 / S4 helpers --------------------------------------------------- */

/* Band of a shifted-frame coordinate p on an axis of length n:
 * 0 for [0,n-M), 1 for [n-M,n-s), 2 for [n-s,n). */
static int band(int p, int n, int M, int s)
{
    if (p < n - M) return 0;
    if (p < n - s) return 1;
    return 2;
}

static int rel_index(int ti, int tj, int M)
{
    int dr = ti / M - tj / M, dc = ti % M - tj % M;
    return (dr + M - 1) * (2 * M - 1) + (dc + M - 1);
}

typedef struct {
    int H, W, C, heads, M, s, mode;
    const double *Wqkv, *bqkv, *table, *tau, *Wproj, *bproj;
} block_params;

/* One window (b, wi, wj) of the shifted frame: gather its tokens from x
 * through partition o roll(-s), run S2..S7, scatter the result to out through
 * roll(+s) o reverse.  logits/probs (optional, heads*N*N each) receive the
 * per-head logits (-inf where masked) and softmax weights. */
static void window_block(const block_params *P, const double *x, double *out,
                         int b, int wi, int wj, double *logits, double *probs)
{
    const int M = P->M, N = M * M, C = P->C, h = P->heads, d = C / h;
    const int H = P->H, W = P->W, s = P->s;
    double *xw = malloc(sizeof(double) * (size_t)N * C);
    double *qkv = malloc(sizeof(double) * (size_t)N * 3 * C);
    double *o = malloc(sizeof(double) * (size_t)N * C);
    double *a = malloc(sizeof(double) * (size_t)N);
    int *region = malloc(sizeof(int) * (size_t)N);

    /* S1: token t of this window sits at shifted (i, j); roll(-s) reads the
     * original (i+s, j+s). */
    for (int t = 0; t < N; ++t) {
        int i = wi * M + t / M, j = wj * M + t % M;
        int oi = roll_source(i, -s, H), oj = roll_source(j, -s, W);
        memcpy(xw + (size_t)t * C, x + (((size_t)b * H + oi) * W + oj) * C, sizeof(double) * (size_t)C);
        region[t] = 3 * band(i, H, M, s) + band(j, W, M, s);
    }
    /* S2 */
    for (int t = 0; t < N; ++t)
        for (int oc = 0; oc < 3 * C; ++oc) {
            double acc = P->bqkv ? P->bqkv[oc] : 0.0;
            for (int c = 0; c < C; ++c) acc += xw[(size_t)t * C + c] * P->Wqkv[(size_t)oc * C + c];
            qkv[(size_t)t * 3 * C + oc] = acc;
        }
    /* S3..S6 per head */
    for (int hd = 0; hd < h; ++hd) {
        double inv_tau = 0.0;
        if (P->mode == ORACLE_V2) inv_tau = 1.0 / fmax(P->tau[hd], 0.01);
        for (int qi = 0; qi < N; ++qi) {
            const double *q = qkv + (size_t)qi * 3 * C + hd * d;
            double qn = 0.0;
            for (int e = 0; e < d; ++e) qn += q[e] * q[e];
            qn = fmax(sqrt(qn), 1e-12);
            for (int kj = 0; kj < N; ++kj) {
                const double *k = qkv + (size_t)kj * 3 * C + C + hd * d;
                double dot = 0.0, kn = 0.0;
                for (int e = 0; e < d; ++e) { dot += q[e] * k[e]; kn += k[e] * k[e]; }
                kn = fmax(sqrt(kn), 1e-12);
                double logit;
                if (P->mode == ORACLE_V2) logit = dot / (qn * kn) * inv_tau;
                else logit = dot / sqrt((double)d);
                logit += P->table[(size_t)rel_index(qi, kj, M) * h + hd];
                if (s > 0 && region[qi] != region[kj]) logit = -INFINITY;   /* S4 */
                a[kj] = logit;
            }
            /* S5: softmax; masked entries contribute exp(-inf) = 0 exactly. */
            double mx = -INFINITY, sum = 0.0;
            for (int kj = 0; kj < N; ++kj) mx = fmax(mx, a[kj]);
            if (logits) memcpy(logits + ((size_t)hd * N + qi) * N, a, sizeof(double) * (size_t)N);
            for (int kj = 0; kj < N; ++kj) { a[kj] = exp(a[kj] - mx); sum += a[kj]; }
            for (int kj = 0; kj < N; ++kj) a[kj] /= sum;
            if (probs) memcpy(probs + ((size_t)hd * N + qi) * N, a, sizeof(double) * (size_t)N);
            /* S6 */
            for (int e = 0; e < d; ++e) {
                double acc = 0.0;
                for (int kj = 0; kj < N; ++kj) acc += a[kj] * qkv[(size_t)kj * 3 * C + 2 * C + hd * d + e];
                o[(size_t)qi * C + hd * d + e] = acc;
            }
        }
    }
    /* S7 then S8: the token at shifted (i, j) returns to (i+s, j+s). */
    for (int t = 0; t < N; ++t) {
        int i = wi * M + t / M, j = wj * M + t % M;
        int oi = roll_source(i, -s, H), oj = roll_source(j, -s, W);
        double *y = out + (((size_t)b * H + oi) * W + oj) * C;
        for (int oc = 0; oc < C; ++oc) {
            double acc = P->bproj ? P->bproj[oc] : 0.0;
            for (int c = 0; c < C; ++c) acc += o[(size_t)t * C + c] * P->Wproj[(size_t)oc * C + c];
            y[oc] = acc;
        }
    }
    free(xw); free(qkv); free(o); free(a); free(region);
}

static int check_shape(int B, int H, int W, int C, int heads, int M, int s)
{
    if (B < 0 || H <= 0 || W <= 0 || C <= 0 || heads <= 0 || M <= 0) return -1;
    if (H % M || W % M || C % heads || s < 0 || s >= M) return -1;
    return 0;
}

/* Full block.  windows == NULL: every window; otherwise only the listed
 * window numbers (win = (b*(H/M)+wi)*(W/M)+wj) are computed, and only their
 * output tokens are written.  nthreads <= 0: OpenMP default. */
int oracle_forward(const double *x, int B, int H, int W, int C, int heads, int M, int s,
                   int mode, const double *Wqkv, const double *bqkv, const double *table,
                   const double *tau, const double *Wproj, const double *bproj, double *out,
                   const int64_t *windows, int64_t n_windows, int nthreads)
{
    if (check_shape(B, H, W, C, heads, M, s)) return -1;
    if (mode == ORACLE_V2 && !tau) return -1;
    block_params P = {H, W, C, heads, M, s, mode, Wqkv, bqkv, table, tau, Wproj, bproj};
    const int nh = H / M, nw = W / M;
    int64_t total = windows ? n_windows : (int64_t)B * nh * nw;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t k = 0; k < total; ++k) {
        int64_t win = windows ? windows[k] : k;
        int b = (int)(win / ((int64_t)nh * nw));
        int r = (int)(win % ((int64_t)nh * nw));
        window_block(&P, x, out, b, r / nw, r % nw, NULL, NULL);
    }
    (void)nthreads;
    return 0;
}

/* Per-head logits (-inf where masked) and softmax weights of one window,
 * each [heads, N, N]; the window's output tokens are also written to out. */
int oracle_window_attention(const double *x, int B, int H, int W, int C, int heads, int M,
                            int s, int mode, const double *Wqkv, const double *bqkv,
                            const double *table, const double *tau, const double *Wproj,
                            const double *bproj, int64_t win, double *logits, double *probs,
                            double *out)
{
    if (check_shape(B, H, W, C, heads, M, s)) return -1;
    block_params P = {H, W, C, heads, M, s, mode, Wqkv, bqkv, table, tau, Wproj, bproj};
    const int nh = H / M, nw = W / M;
    if (win < 0 || win >= (int64_t)B * nh * nw) return -1;
    int b = (int)(win / ((int64_t)nh * nw));
    int r = (int)(win % ((int64_t)nh * nw));
    window_block(&P, x, out, b, r / nw, r % nw, logits, probs);
    return 0;
}

/* Log-spaced continuous position bias: table[idx*heads + h] = G(coords)[h],
 * idx = (dr+M-1)*(2M-1) + (dc+M-1), dr, dc in [-(M-1), M-1];
 * G: hidden = ReLU(W1 u + b1) (W1 [hidden,2]), out = W2 hidden (W2 [heads,hidden]),
 * u = (sign(dr) ln(1+|dr|), sign(dc) ln(1+|dc|)). */
int oracle_cpb_table(int M, int heads, int hidden, const double *W1, const double *b1,
                     const double *W2, double *table)
{
    if (M <= 0 || heads <= 0 || hidden <= 0) return -1;
    const int L = 2 * M - 1;
    double *hid = malloc(sizeof(double) * (size_t)hidden);
    for (int dr = -(M - 1); dr <= M - 1; ++dr)
        for (int dc = -(M - 1); dc <= M - 1; ++dc) {
            double u0 = (dr > 0 ? 1.0 : dr < 0 ? -1.0 : 0.0) * log(1.0 + fabs((double)dr));
            double u1 = (dc > 0 ? 1.0 : dc < 0 ? -1.0 : 0.0) * log(1.0 + fabs((double)dc));
            for (int k = 0; k < hidden; ++k) {
                double v = W1[2 * k] * u0 + W1[2 * k + 1] * u1 + (b1 ? b1[k] : 0.0);
                hid[k] = v > 0.0 ? v : 0.0;
            }
            int idx = (dr + M - 1) * L + (dc + M - 1);
            for (int hd = 0; hd < heads; ++hd) {
                double acc = 0.0;
                for (int k = 0; k < hidden; ++k) acc += W2[(size_t)hd * hidden + k] * hid[k];
                table[(size_t)idx * heads + hd] = acc;
            }
        }
    free(hid);
    return 0;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
