/* Runs the fp64 C oracle (oracle/gdn_oracle.c, linked in by the test) on small
 * cases that walk its edge paths -- an empty sequence, one-token and
 * chunk-crossing sequences, beta at 0 and 1 (b_raw = -inf, +inf), a strong
 * decay (ssm_a = -16, a_raw = 3), a zero conv tap set (q = 0) -- so that a build
 * with AddressSanitizer and UndefinedBehaviorSanitizer can catch an
 * out-of-bounds access or undefined arithmetic.  Exit status 0 and "ok" when
 * every call returns 0 and every output is finite. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

int gdn_oracle_forward(int n_seq, const int64_t* cu_seqlens, int Hk, int Hv, double eps, const float* x,
                       const float* z, const float* a_raw, const float* b_raw, const float* conv_w,
                       const float* dt_bias, const float* ssm_a, const float* norm_w, float* conv_state, double* S,
                       double* out, double* prenorm, double* inter, int n_threads);

static uint64_t rng = 0x9E3779B97F4A7C15ull;
static float frand(void) {   /* xorshift64*, uniform in [-1, 1) */
    rng ^= rng >> 12; rng ^= rng << 25; rng ^= rng >> 27;
    return (float)((double)((rng * 0x2545F4914F6CDD1Dull) >> 11) / 9007199254740992.0 * 2.0 - 1.0);
}

static int run(int Hk, int Hv, int n_seq, const int64_t* cu, int n_threads) {
    const int D = 128, C = D * (2 * Hk + Hv);
    const int64_t T = cu[n_seq];
    float* x = malloc(sizeof(float) * (size_t)(T * C + 1));
    float* z = malloc(sizeof(float) * (size_t)(T * Hv * D + 1));
    float* a = malloc(sizeof(float) * (size_t)(T * Hv + 1));
    float* b = malloc(sizeof(float) * (size_t)(T * Hv + 1));
    float* w = malloc(sizeof(float) * (size_t)C * 4);
    float* dt = malloc(sizeof(float) * (size_t)Hv);
    float* sa = malloc(sizeof(float) * (size_t)Hv);
    float* nw = malloc(sizeof(float) * D);
    float* cs = malloc(sizeof(float) * (size_t)n_seq * 3 * C);
    double* S = malloc(sizeof(double) * (size_t)n_seq * Hv * D * D);
    double* out = malloc(sizeof(double) * (size_t)(T * Hv * D + 1));
    double* pre = malloc(sizeof(double) * (size_t)(T * Hv * D + 1));
    double* inter = malloc(sizeof(double) * (size_t)(T * Hv * (3 * D + 2) + 1));
    if (!x || !z || !a || !b || !w || !dt || !sa || !nw || !cs || !S || !out || !pre || !inter) return 2;
    for (int64_t i = 0; i < T * C; ++i) x[i] = frand();
    for (int64_t i = 0; i < T * Hv * D; ++i) z[i] = frand();
    for (int64_t i = 0; i < T * Hv; ++i) { a[i] = frand(); b[i] = frand(); }
    for (int64_t i = 0; i < (int64_t)C * 4; ++i) w[i] = 0.25f * frand();
    for (int i = 0; i < Hv; ++i) { dt[i] = frand(); sa[i] = -1.0f - 7.5f * (frand() + 1.0f); }
    for (int i = 0; i < D; ++i) nw[i] = 1.0f + 0.1f * frand();
    for (int64_t i = 0; i < (int64_t)n_seq * 3 * C; ++i) cs[i] = frand();
    for (int64_t i = 0; i < (int64_t)n_seq * Hv * D * D; ++i) S[i] = 0.02 * frand();
    /* edge paths: beta = 1 and 0 on v-head 0, strong decay on v-head 1, q of q/k head 0 zero */
    for (int64_t t = 0; t < T; ++t) {
        b[t * Hv] = (t & 1) ? -INFINITY : INFINITY;
        if (Hv > 1) a[t * Hv + 1] = 3.0f;
    }
    if (Hv > 1) sa[1] = -16.0f;
    for (int i = 0; i < D * 4; ++i) w[i] = 0.0f;
    int rc = gdn_oracle_forward(n_seq, cu, Hk, Hv, 1e-6, x, z, a, b, w, dt, sa, nw, cs, S, out, pre, inter, n_threads);
    if (rc == 0)
        for (int64_t i = 0; i < T * Hv * D; ++i)
            if (!isfinite(out[i]) || !isfinite(pre[i])) { rc = 3; break; }
    if (rc == 0)
        for (int64_t i = 0; i < (int64_t)n_seq * Hv * D * D; ++i)
            if (!isfinite(S[i])) { rc = 4; break; }
    free(x); free(z); free(a); free(b); free(w); free(dt); free(sa); free(nw); free(cs); free(S); free(out);
    free(pre); free(inter);
    return rc;
}

int main(void) {
    const int64_t cu1[] = {0, 0, 1, 5, 70};    /* empty, one token, four tokens, 65 tokens */
    const int64_t cu2[] = {0, 3};
    int rc = run(1, 2, 4, cu1, 2);
    if (rc == 0) rc = run(2, 6, 1, cu2, 1);
    if (rc == 0) rc = run(2, 4, 4, cu1, 0);
    printf(rc == 0 ? "ok\n" : "failed %d\n", rc);
    return rc;
}
