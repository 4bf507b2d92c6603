/*
 * gdn_oracle.c -- plain, slow, fp64 CPU oracle of the gated DeltaNet token mixer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, calls or
 * includes this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header or constant table with the
 * CUDA path.
 *
 * Source of the method: the "Gated DeltaNet layer" paragraph of the
 * "Architecture cheat sheet (Qwen 3.6, ggml-org GGUF)" section of the xwen
 * CLAUDE.md page, plus "GGUF facts that differ from the HF checkpoint" on the
 * same page (multiply-ready norm weight, pre-baked ssm_a = -exp(A_log), tiled
 * V-head order, F32 conv/ssm_a/dt/norm tensors) and "RMSNorm eps 1e-6".
 *
 * Per (sequence, v-head) and per token, in the page's order:
 *   1. causal depthwise conv1d, kernel 4, no bias, over the full fused width,
 *      left context taken from the carried conv state (3 raw rows, oldest
 *      first).  Tap 3 multiplies the current token, tap 0 the oldest.
 *   2. SiLU over the whole fused stream.
 *   3. split q | k | v, head-major inside each block (channel = h*128 + i).
 *   4. L2 norm of q and k in clamp form x / max(||x||, eps).
 *   5. k/q heads tiled to H_v: v-head j reads q/k head j mod H_k.
 *   6. beta = sigmoid(b_raw), g = ssm_a * softplus(a_raw + dt_bias).
 *   7. delta rule on the state S (d_v x d_k, S[j][i], k-index contiguous):
 *        S <- exp(g) S;  s = S k;  d = (v - s) beta;  S[j][i] += d_j k_i;
 *        o = S q / sqrt(128)            (o from the updated state)
 *   8. gated RMSNorm over the head's 128 outputs:
 *        y_j = o_j / sqrt(mean(o^2) + eps) * norm_w[j] * silu(z_j)
 * After a sequence the conv state holds its last 3 raw input rows.
 *
 * Arithmetic is fp64 throughout; inputs arrive as float (every bf16 or fp32
 * value is exactly representable) and are widened exactly.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define D 128      /* head dimension, d_k = d_v (cheat sheet: head dims 128) */
#define KW 4       /* conv kernel width (cheat sheet: kernel 4)             */

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* log(1 + e^x), written as max(x,0) + log1p(e^-|x|) so it never overflows. */
static double softplus(double x) { return (x > 0 ? x : 0.0) + log1p(exp(-fabs(x))); }

static double silu(double x) { return x * sigmoid(x); }

/* Raw input of channel c at position p (p relative to the sequence start;
 * p < 0 reads the carried conv state, row 3+p). */
static double raw_at(const float* x, int64_t seq_start, int64_t C, const float* cst,
                     int64_t p, int64_t c) {
    if (p >= 0) return (double)x[(seq_start + p) * C + c];
    return (double)cst[(3 + p) * C + c];
}

/* Steps 1-2 for one channel at one position. */
static double conv_silu(const float* x, int64_t seq_start, int64_t C, const float* cst,
                        const float* conv_w, int64_t p, int64_t c) {
    double u = 0.0;
    for (int j = 0; j < KW; ++j)
        u += (double)conv_w[c * KW + j] * raw_at(x, seq_start, C, cst, p - 3 + j, c);
    return silu(u);
}

/*
 * Run the layer over n_seq packed sequences (cu_seqlens[n_seq+1], token rows
 * cu_seqlens[s] .. cu_seqlens[s+1]-1 of every [T][...] array).
 *
 *   x          [T][C]          C = 128*(2*Hk+Hv), fused q|k|v stream
 *   z          [T][Hv*128]     output gate
 *   a_raw      [T][Hv]         ssm_alpha output
 *   b_raw      [T][Hv]         ssm_beta output
 *   conv_w     [C][4]
 *   dt_bias    [Hv], ssm_a [Hv], norm_w [128]
 *   conv_state [n_seq][3][C]   in/out, raw rows oldest first
 *   S          [n_seq][Hv][128][128]  in/out (fp64)
 *   out        [T][Hv*128]     gated-normed output (fp64)
 *   prenorm    [T][Hv*128]     o before the gated norm, or NULL
 *   inter      [T][Hv][3*128+2] q_hat | k_hat | v | beta | g, or NULL
 * Returns 0, or -1 on bad arguments.
 */
int gdn_oracle_forward(int n_seq, const int64_t* cu_seqlens, int Hk, int Hv, double eps,
                       const float* x, const float* z, const float* a_raw, const float* b_raw,
                       const float* conv_w, const float* dt_bias, const float* ssm_a,
                       const float* norm_w, float* conv_state, double* S, double* out,
                       double* prenorm, double* inter, int n_threads) {
    if (n_seq < 0 || Hk <= 0 || Hv <= 0 || Hv % Hk != 0) return -1;
    const int64_t C = (int64_t)D * (2 * Hk + Hv);
    const int64_t HvD = (int64_t)Hv * D;
    const int64_t IW = 3 * D + 2;
    const double inv_sqrt_d = 1.0 / sqrt((double)D);
    const int64_t units = (int64_t)n_seq * Hv;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t u = 0; u < units; ++u) {
        const int s = (int)(u / Hv), h = (int)(u % Hv);
        const int kh = h % Hk;                       /* step 5: tiled head map */
        const int64_t t0 = cu_seqlens[s], len = cu_seqlens[s + 1] - cu_seqlens[s];
        const float* cst = conv_state + (int64_t)s * 3 * C;
        double* St = S + ((int64_t)s * Hv + h) * D * D;
        double q[D], k[D], v[D], o[D];
        const int64_t qc = (int64_t)kh * D, kc = (int64_t)Hk * D + kh * D,
                      vc = (int64_t)2 * Hk * D + (int64_t)h * D;

        for (int64_t p = 0; p < len; ++p) {
            const int64_t t = t0 + p;
            /* steps 1-3 */
            for (int i = 0; i < D; ++i) {
                q[i] = conv_silu(x, t0, C, cst, conv_w, p, qc + i);
                k[i] = conv_silu(x, t0, C, cst, conv_w, p, kc + i);
                v[i] = conv_silu(x, t0, C, cst, conv_w, p, vc + i);
            }
            /* step 4: clamp-form L2 norm */
            double nq = 0.0, nk = 0.0;
            for (int i = 0; i < D; ++i) { nq += q[i] * q[i]; nk += k[i] * k[i]; }
            nq = sqrt(nq); nk = sqrt(nk);
            const double dq = nq > eps ? nq : eps, dk = nk > eps ? nk : eps;
            for (int i = 0; i < D; ++i) { q[i] /= dq; k[i] /= dk; }
            /* step 6: gates */
            const double beta = sigmoid((double)b_raw[t * Hv + h]);
            const double g = (double)ssm_a[h] * softplus((double)a_raw[t * Hv + h] + (double)dt_bias[h]);
            const double eg = exp(g);
            if (inter) {
                double* it = inter + (t * Hv + h) * IW;
                for (int i = 0; i < D; ++i) { it[i] = q[i]; it[D + i] = k[i]; it[2 * D + i] = v[i]; }
                it[3 * D] = beta; it[3 * D + 1] = g;
            }
            /* step 7: delta rule, in the page's order */
            for (int j = 0; j < D; ++j)
                for (int i = 0; i < D; ++i) St[j * D + i] *= eg;
            for (int j = 0; j < D; ++j) {
                double sj = 0.0;
                for (int i = 0; i < D; ++i) sj += St[j * D + i] * k[i];
                const double dj = (v[j] - sj) * beta;
                for (int i = 0; i < D; ++i) St[j * D + i] += dj * k[i];
            }
            for (int j = 0; j < D; ++j) {
                double oj = 0.0;
                for (int i = 0; i < D; ++i) oj += St[j * D + i] * q[i];
                o[j] = oj * inv_sqrt_d;
            }
            /* step 8: gated RMSNorm */
            double ms = 0.0;
            for (int j = 0; j < D; ++j) ms += o[j] * o[j];
            ms /= (double)D;
            const double r = 1.0 / sqrt(ms + eps);
            for (int j = 0; j < D; ++j) {
                const int64_t oi = t * HvD + (int64_t)h * D + j;
                if (prenorm) prenorm[oi] = o[j];
                out[oi] = o[j] * r * (double)norm_w[j] * silu((double)z[oi]);
            }
        }
    }

    /* conv state: last 3 raw rows of (old state || this sequence's inputs) */
    for (int s = 0; s < n_seq; ++s) {
        const int64_t t0 = cu_seqlens[s], len = cu_seqlens[s + 1] - cu_seqlens[s];
        float* cst = conv_state + (int64_t)s * 3 * C;
        float* nw = (float*)malloc((size_t)(3 * C) * sizeof(float));
        if (!nw) return -1;
        for (int r = 0; r < 3; ++r) {
            const int64_t p = len - 3 + r;
            for (int64_t c = 0; c < C; ++c)
                nw[r * C + c] = p >= 0 ? x[(t0 + p) * C + c] : cst[(3 + p) * C + c];
        }
        memcpy(cst, nw, (size_t)(3 * C) * sizeof(float));
        free(nw);
    }
    return 0;
}

int gdn_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
