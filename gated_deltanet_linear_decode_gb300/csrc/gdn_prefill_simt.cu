// gdn_prefill_simt.cu -- chunked (chunk = 64) prefill of the gated DeltaNet
// layer in fp32 on the CUDA cores.  It serves fp32 activations (whose
// tolerance needs fp32 products end to end) and is the plain-arithmetic
// counterpart of the tensor-core prefill.
//
// Method: xwen CLAUDE.md page, "Ground truth" (recurrent and chunk=64 forms of
// the delta rule) and "Architecture cheat sheet", "Gated DeltaNet layer".
// Chunked form used here, for a chunk of n <= 64 tokens entering with state
// S0 (S[j][i], j the v-row), Gam_t = g_1 + ... + g_t inside the chunk:
//   A[t][r] = beta_t e^{Gam_t - Gam_r} (k_t . k_r)          r < t
//   (I + A) U = diag(beta) V,  (I + A) W = diag(beta e^Gam) K  (forward substitution)
//   D = U - W S0^T
//   O = diag(e^Gam) Q S0^T + P D,  P[t][r] = e^{Gam_t - Gam_r} (q_t . k_r), r <= t
//   S_n = e^{Gam_n} S0 + D^T diag(e^{Gam_n - Gam}) K
// followed by o = O / sqrt(128) and the gated RMSNorm per token.
//
// One CTA of 256 threads per (sequence, v-head); the state and the chunk's
// Q, K, V/U/D and W/O live in shared memory (odd row strides keep the
// column walks free of bank conflicts).
#include "gdn_common.cuh"
#include <algorithm>

#include "gdn_internal.h"
#include "gdn_prefill_tc.cuh"

namespace gdn {

namespace {

constexpr int kThreads = 256;
constexpr int kLd = 129;            // row stride of the 128-wide tiles (floats)
constexpr int kLdA = 65;            // row stride of the 64x64 tiles
constexpr size_t kSimtSmemFloats =
    128 * kLd + 4 * 64 * kLd + 64 * kLdA + 2 * 64 + 2 * 64;   // S, Q, K, V, W, A/P, beta, g, Gam (fp64)
constexpr size_t kSimtSmemBytes = kSimtSmemFloats * sizeof(float);

__device__ __forceinline__ float conv4(float4 w, float x0, float x1, float x2, float cur) {
    return fmaf(w.w, cur, fmaf(w.z, x2, fmaf(w.y, x1, w.x * x0)));
}

// Each of the 256 threads owns rows m = tm + ii*GM and columns n = tn + jj*GN
// of an M x N product: C[m][n] = sum_k a(m, k) * b(k, n), handed to epi.
template <int M, int N, int TM, int TN, typename FA, typename FB, typename FE>
__device__ __forceinline__ void block_gemm(int K, FA a, FB b, FE epi) {
    constexpr int GM = M / TM, GN = N / TN;
    static_assert(GM * GN == kThreads, "tile grid must cover the block");
    const int tm = threadIdx.x / GN, tn = threadIdx.x % GN;
    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;
    for (int k = 0; k < K; ++k) {
        float av[TM], bv[TN];
#pragma unroll
        for (int i = 0; i < TM; ++i) av[i] = a(tm + i * GM, k);
#pragma unroll
        for (int j = 0; j < TN; ++j) bv[j] = b(k, tn + j * GN);
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) epi(tm + i * GM, tn + j * GN, acc[i][j]);
}

template <typename Tact, typename Tout>
__global__ void __launch_bounds__(kThreads, 1)
prefill_simt_kernel(const PrefillParams p) {
    const int s = blockIdx.x / p.Hv, h = blockIdx.x % p.Hv;
    const int kh = h % p.Hk;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = p.cu_seqlens[s];
    const int L = p.cu_seqlens[s + 1] - t0;
    const int C = p.C, HvD = p.Hv * kD;

    extern __shared__ float sm[];
    float* Ss = sm;                     // [128][kLd]   state S[j][i]
    float* Qs = Ss + 128 * kLd;         // [64][kLd]    q_hat
    float* Ks = Qs + 64 * kLd;          // [64][kLd]    k_hat, later K'
    float* Vs = Ks + 64 * kLd;          // [64][kLd]    beta v -> U -> D
    float* Ws = Vs + 64 * kLd;          // [64][kLd]    beta e^Gam k -> W -> O
    float* As = Ws + 64 * kLd;          // [64][kLdA]   A, later P
    float* beta_s = As + 64 * kLdA;     // [64]
    float* g_s = beta_s + 64;           // [64]
    // Gam in fp64: within a chunk |Gam| reaches hundreds, and the decay
    // weights need Gam_t - Gam_r to fp32 relative accuracy.
    double* gam_s = reinterpret_cast<double*>(g_s + 64);   // [64]

    // ---- initial state
    const bool sbf = (p.flags & kFlagStateBf16) != 0;
    const size_t plane0 = (static_cast<size_t>(s) * p.Hv + h) * kD * kD;
    float* Sg = static_cast<float*>(p.S) + plane0;                          // fp32 state
    __nv_bfloat16* Sgb = static_cast<__nv_bfloat16*>(p.S) + plane0;         // bf16 state
    for (int e = tid; e < kD * kD; e += kThreads) {
        const int j = e >> 7, i = e & 127;
        Ss[j * kLd + i] = p.zero_init ? 0.f : (sbf ? __bfloat162float(Sgb[e]) : Sg[e]);
    }

    const Tact* x = static_cast<const Tact*>(p.x);
    const Tact* cst = static_cast<const Tact*>(p.conv_state) + static_cast<size_t>(s) * 3 * C;
    const float a_dt = p.dt_bias[h], a_ssm = p.ssm_a[h];
    bool bad = false;

    for (int c0 = 0; c0 < L; c0 += kChunk) {
        const int n = min(kChunk, L - c0);
        __syncthreads();   // previous chunk fully consumed
        // ---- steps 1-6 for the chunk's tokens: warp w takes tokens w, w+8, ...
        for (int t = warp; t < kChunk; t += 8) {
            if (t < n) {
                const int pos = c0 + t;
                float q[4], k[4], v[4];
                float sq = 0.f, sk = 0.f;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = lane + 32 * u;
                    const int ch[3] = {kh * kD + i, p.Hk * kD + kh * kD + i, 2 * p.Hk * kD + h * kD + i};
                    float val[3];
#pragma unroll
                    for (int c = 0; c < 3; ++c) {
                        float win[4];
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const int row = pos - 3 + r;
                            win[r] = row >= 0 ? to_f(x[static_cast<size_t>(t0 + row) * C + ch[c]])
                                              : (p.zero_init ? 0.f : to_f(cst[(3 + row) * C + ch[c]]));
                        }
                        const float4 wv = *reinterpret_cast<const float4*>(p.conv_w + 4 * ch[c]);
                        val[c] = siluf_(conv4(wv, win[0], win[1], win[2], win[3]));
                    }
                    q[u] = val[0]; k[u] = val[1]; v[u] = val[2];
                    sq = fmaf(q[u], q[u], sq);
                    sk = fmaf(k[u], k[u], sk);
                }
                sq = warp_sum(sq);
                sk = warp_sum(sk);
                const float iq = 1.0f / fmaxf(sqrtf(sq), p.eps), ik = 1.0f / fmaxf(sqrtf(sk), p.eps);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = lane + 32 * u;
                    Qs[t * kLd + i] = q[u] * iq;
                    Ks[t * kLd + i] = k[u] * ik;
                    Vs[t * kLd + i] = v[u];
                }
                if (lane == 0) {
                    const size_t row = static_cast<size_t>(t0 + pos) * p.Hv + h;
                    beta_s[t] = sigmoidf_(ld_act(static_cast<const Tact*>(p.b_raw) + row));
                    g_s[t] = a_ssm * softplusf_(ld_act(static_cast<const Tact*>(p.a_raw) + row) + a_dt);
                }
            } else {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = lane + 32 * u;
                    Qs[t * kLd + i] = 0.f; Ks[t * kLd + i] = 0.f; Vs[t * kLd + i] = 0.f;
                }
                if (lane == 0) { beta_s[t] = 0.f; g_s[t] = 0.f; }
            }
        }
        __syncthreads();
        if (tid == 0) {
            double acc = 0.0;
            for (int t = 0; t < kChunk; ++t) { acc += static_cast<double>(g_s[t]); gam_s[t] = acc; }
        }
        __syncthreads();
        const double gl = gam_s[n - 1];
        // e^{Gam_t - Gam_r} and e^{Gam_t}, exponent formed in fp64
        auto dexp = [&](int t, int r) { return expf(static_cast<float>(gam_s[t] - gam_s[r])); };
        auto gexp = [&](int t) { return expf(static_cast<float>(gam_s[t])); };
        // ---- A = strict-lower beta_t e^{Gam_t - Gam_r} (k_t . k_r)
        block_gemm<64, 64, 4, 4>(
            kD, [&](int t, int i) { return Ks[t * kLd + i]; }, [&](int i, int r) { return Ks[r * kLd + i]; },
            [&](int t, int r, float acc) {
                As[t * kLdA + r] = r < t ? beta_s[t] * dexp(t, r) * acc : 0.f;
            });
        // ---- right-hand sides: beta V and beta e^Gam K
        for (int e = tid; e < 64 * kD; e += kThreads) {
            const int t = e >> 7, i = e & 127;
            Vs[t * kLd + i] *= beta_s[t];
            Ws[t * kLd + i] = beta_s[t] * gexp(t) * Ks[t * kLd + i];
        }
        __syncthreads();
        // ---- forward substitution (I + A) X = RHS, one column per thread
        {
            float* X = tid < kD ? Vs + tid : Ws + (tid - kD);
            for (int t = 1; t < n; ++t) {
                float acc = X[t * kLd];
                for (int r = 0; r < t; ++r) acc = fmaf(-As[t * kLdA + r], X[r * kLd], acc);
                X[t * kLd] = acc;
            }
        }
        __syncthreads();
        // ---- D = U - W S0^T   (in place over U)
        block_gemm<64, 128, 4, 8>(
            kD, [&](int t, int i) { return Ws[t * kLd + i]; }, [&](int i, int j) { return Ss[j * kLd + i]; },
            [&](int t, int j, float acc) { Vs[t * kLd + j] -= acc; });
        __syncthreads();
        // ---- P = causal e^{Gam_t - Gam_r} (q_t . k_r);  O = e^Gam Q S0^T (into W's buffer)
        block_gemm<64, 64, 4, 4>(
            kD, [&](int t, int i) { return Qs[t * kLd + i]; }, [&](int i, int r) { return Ks[r * kLd + i]; },
            [&](int t, int r, float acc) { As[t * kLdA + r] = r <= t ? dexp(t, r) * acc : 0.f; });
        block_gemm<64, 128, 4, 8>(
            kD, [&](int t, int i) { return Qs[t * kLd + i]; }, [&](int i, int j) { return Ss[j * kLd + i]; },
            [&](int t, int j, float acc) { Ws[t * kLd + j] = gexp(t) * acc; });
        __syncthreads();
        // ---- O += P D ;  K' = e^{Gam_n - Gam} K (in place)
        block_gemm<64, 128, 4, 8>(
            kChunk, [&](int t, int r) { return As[t * kLdA + r]; }, [&](int r, int j) { return Vs[r * kLd + j]; },
            [&](int t, int j, float acc) { Ws[t * kLd + j] += acc; });
        for (int e = tid; e < 64 * kD; e += kThreads) {
            const int t = e >> 7, i = e & 127;
            Ks[t * kLd + i] *= expf(static_cast<float>(gl - gam_s[t]));
        }
        __syncthreads();
        // ---- S = e^{Gam_n} S0 + D^T K'
        const float egl = expf(static_cast<float>(gl));
        block_gemm<128, 128, 8, 8>(
            kChunk, [&](int j, int t) { return Vs[t * kLd + j]; }, [&](int t, int i) { return Ks[t * kLd + i]; },
            [&](int j, int i, float acc) { Ss[j * kLd + i] = fmaf(egl, Ss[j * kLd + i], acc); });
        // ---- step 8: o = O / sqrt(128), gated RMSNorm, store
        for (int t = warp; t < n; t += 8) {
            const size_t row = static_cast<size_t>(t0 + c0 + t);
            float o[4], ss = 0.f;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                o[u] = Ws[t * kLd + lane + 32 * u] * kInvSqrtD;
                ss = fmaf(o[u], o[u], ss);
            }
            ss = warp_sum(ss);
            const float rs = 1.0f / sqrtf(ss * (1.0f / kD) + p.eps);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = lane + 32 * u;
                const size_t oi = row * HvD + h * kD + j;
                const float zz = ld_act(static_cast<const Tact*>(p.z) + oi);
                const float y = o[u] * rs * p.norm_w[j] * siluf_(zz);
                st_out(static_cast<Tout*>(p.out) + oi, y);
                if (p.prenorm) p.prenorm[oi] = o[u];
                if (p.flags & kFlagCheckFinite) bad |= nonfinite_bits(y);
            }
        }
    }
    __syncthreads();
    bool bad_s = false;
    for (int e = tid; e < kD * kD; e += kThreads) {
        const float v = Ss[(e >> 7) * kLd + (e & 127)];
        if (sbf)
            Sgb[e] = __float2bfloat16_rn(v);
        else
            Sg[e] = v;
        if (p.flags & kFlagCheckFinite) bad_s |= nonfinite_bits(v);
    }
    if (p.dev_status && (p.flags & kFlagCheckFinite)) {
        const int st = (__any_sync(0xffffffffu, bad_s) ? 1 : 0) | (__any_sync(0xffffffffu, bad) ? 2 : 0);
        if (lane == 0 && st) atomicOr(p.dev_status + s * p.Hv + h, st);
    }
}

}  // namespace

// Conv state after a prefill: the last 3 raw rows of (old state || sequence).
// Runs after the main kernel so every CTA has read the old rows first.
template <typename Tact>
__global__ void conv_state_finalize_kernel(const PrefillParams p) {
    // launched as a programmatic dependent of the prefill kernel, which reads the old rows
    grid_dependency_wait();
    grid_launch_dependents();
    const int s = blockIdx.y;
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= p.C) return;
    const int t0 = p.cu_seqlens[s], L = p.cu_seqlens[s + 1] - t0;
    Tact* cst = static_cast<Tact*>(p.conv_state) + static_cast<size_t>(s) * 3 * p.C;
    const Tact* x = static_cast<const Tact*>(p.x);
    Tact nv[3];
#pragma unroll
    for (int r = 0; r < 3; ++r) {
        const int pos = L - 3 + r;
        nv[r] = pos >= 0 ? x[static_cast<size_t>(t0 + pos) * p.C + c]
                         : (p.zero_init ? Tact(0.f) : cst[(3 + pos) * p.C + c]);
    }
#pragma unroll
    for (int r = 0; r < 3; ++r) cst[r * p.C + c] = nv[r];
}

template <typename Tact, typename Tout>
cudaError_t launch_prefill_simt_t(const PrefillParams& p, cudaStream_t stream) {
    auto k = prefill_simt_kernel<Tact, Tout>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSimtSmemBytes));
    if (e != cudaSuccess) return e;
    k<<<static_cast<unsigned>(p.n_seq) * p.Hv, kThreads, kSimtSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_prefill_simt(const PrefillParams& p, int act_dtype, int out_dtype, cudaStream_t stream) {
    if (act_dtype == 1)
        return out_dtype == 1 ? launch_prefill_simt_t<__nv_bfloat16, __nv_bfloat16>(p, stream)
                              : launch_prefill_simt_t<__nv_bfloat16, float>(p, stream);
    return out_dtype == 1 ? launch_prefill_simt_t<float, __nv_bfloat16>(p, stream)
                          : launch_prefill_simt_t<float, float>(p, stream);
}

cudaError_t launch_tensor_core_prefill(const PrefillParams& p, int out_dtype, cudaStream_t stream);
size_t tc_prefill_workspace_bytes(int Hk, int Hv, int n_seq, long long T);
void tc_prefill_bind_workspace(PrefillParams& p);

namespace {
bool use_tensor_cores(int act_dtype, uint32_t flags) { return act_dtype == 1 && !(flags & kFlagForceSimt); }
}  // namespace

size_t prefill_workspace_bytes(int Hk, int Hv, int n_seq, long long T, int act_dtype, uint32_t flags) {
    if (!use_tensor_cores(act_dtype, flags)) return 0;
    return tc_prefill_workspace_bytes(Hk, Hv, n_seq, T);
}

void prefill_bind_workspace(PrefillParams& p, int act_dtype) {
    if (use_tensor_cores(act_dtype, p.flags)) tc_prefill_bind_workspace(p);
}

// bf16 activations take the tensor-core path (chunk table, then one kernel
// whose preparation and chain roles run side by side); fp32 activations (whose 1e-5 tolerance needs fp32 products) take the CUDA-core
// kernel.  Either is followed by the conv-state update, which must run after
// every CTA has read the old rows.
cudaError_t launch_prefill(const PrefillParams& p, int act_dtype, int out_dtype, cudaStream_t stream) {
    cudaError_t e;
    if (use_tensor_cores(act_dtype, p.flags)) {
        e = launch_tensor_core_prefill(p, out_dtype, stream);
    } else {
        e = launch_prefill_simt(p, act_dtype, out_dtype, stream);
    }
    if (e != cudaSuccess) return e;
    // the test hook leaves every state of the tensor-core path as it was
    if ((p.flags & kFlagTestStall) && use_tensor_cores(act_dtype, p.flags)) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((p.C + 255) / 256, p.n_seq);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see grid_dependency_wait
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return act_dtype == 1 ? cudaLaunchKernelEx(&cfg, conv_state_finalize_kernel<__nv_bfloat16>, p)
                          : cudaLaunchKernelEx(&cfg, conv_state_finalize_kernel<float>, p);
}

}  // namespace gdn
