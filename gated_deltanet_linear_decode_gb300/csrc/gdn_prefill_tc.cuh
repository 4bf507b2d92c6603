// gdn_prefill_tc.cuh -- pieces shared by the two kernels of the tensor-core
// prefill: the chunk-preparation kernel (everything of a chunk that does not
// depend on the state) and the state pass (the chunk-to-chunk recurrence and
// the outputs), plus the layout of the records the first hands to the second.
//
// Method: xwen CLAUDE.md page, "Ground truth" (chunk = 64 form of the delta
// rule) and "Architecture cheat sheet", "Gated DeltaNet layer".  For a chunk
// of n <= 64 tokens entering with state S (S[j][i]), Gam_t = g_1 + ... + g_t:
//   A[t][r] = beta_t e^{Gam_t-Gam_r} (k_t . k_r), r < t;   T = (I + A)^{-1}
//   U = T diag(beta) V,   W = T diag(beta e^Gam) K,   D = U - W S^T
//   O = diag(e^Gam) Q S^T + P D,   P[t][r] = e^{Gam_t-Gam_r} (q_t . k_r), r <= t
//   S' = e^{Gam_n} S + D^T diag(e^{Gam_n-Gam}) K
// Only D, O and S' involve the state; A, T, U, W, P, the decay-scaled
// Q' = diag(e^Gam) Q and K' = diag(e^{Gam_n-Gam}) K and the decay vectors are
// computed for all chunks at once by the preparation kernel, so that
//   O = Q' S^T + P D,   S' = e^{Gam_n} S + D^T K'.
#pragma once

#include "gdn_common.cuh"
#include "gdn_tc.cuh"

namespace gdn {
namespace pf {

// ---------------------------------------------------------------- workspace records
// Per (chunk, v-head), fp16 tiles in the canonical no-swizzle layout (element
// (a, b) of a tile with A rows at cl_off(a, b, A)):
//   Q' = diag(e^Gam) Q hi, lo              64 (t) x 128 (i), 64 rows       2 x 16384 B
//   K' = diag(e^{Gam_last - Gam}) K hi, lo  64 (t) x 128 (i), 64 rows       2 x 16384 B
//   W^T hi                                  128 (i) x 64 (t), 128 rows         16384 B
//   P hi, lo                                64 (t) x 64 (r), 64 rows        2 x 8192 B
//   U                 fp32, float4 groups [t/4][j][t%4] (j = v-row)            32768 B
//   e^Gam_t [64] fp32, then e^{Gam_last - Gam_t} [64] fp32                       512 B
constexpr uint32_t kVRec = 131584;
constexpr uint32_t kRecQhi = 0, kRecQlo = 16384, kRecKhi = 32768, kRecKlo = 49152, kRecW = 65536, kRecPhi = 81920,
                   kRecPlo = 90112, kRecU = 98304, kRecEgam = 131072, kRecElast = 131328;

// Workspace = chunk table (int32 [n_seq+1], padded to 256 B), then the records
// of every (chunk, v-head).
__host__ __device__ inline size_t table_bytes(int n_seq) {
    return (static_cast<size_t>(n_seq + 1) * 4 + 255) / 256 * 256;
}

// ---------------------------------------------------------------- small math
__device__ __forceinline__ float conv4(float4 w, float x0, float x1, float x2, float cur) {
    return fmaf(w.w, cur, fmaf(w.z, x2, fmaf(w.y, x1, w.x * x0)));
}

// SiLU with the fast exponential and fast division (relative error of a few
// ulp, far inside the output tolerance; 0 for large negative x).
__device__ __forceinline__ float silu_fast(float x) { return x * __fdividef(1.0f, 1.0f + __expf(-x)); }

__device__ __forceinline__ void bf16x8_to_f32(uint4 u, float* f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void bf16x4_to_f32(uint2 u, float* f) {
    f[0] = __uint_as_float(u.x << 16); f[1] = __uint_as_float(u.x & 0xffff0000u);
    f[2] = __uint_as_float(u.y << 16); f[3] = __uint_as_float(u.y & 0xffff0000u);
}

__device__ __forceinline__ void st_out4(float* p, const float (&y)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(y[0], y[1], y[2], y[3]);
}
__device__ __forceinline__ void st_out4(__nv_bfloat16* p, const float (&y)[4]) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(y[0], y[1]), b = __floats2bfloat162_rn(y[2], y[3]);
    *reinterpret_cast<uint2*>(p) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
}

// (I + A)^{-1} for a strictly lower 64 x 64 A (fp32, row stride 65), by a
// block of kThreads >= 192 threads: the four 16 x 16 diagonal blocks by forward
// substitution (column c of block b per thread, each solved value folded into
// the rows below it at once), then the off-diagonal blocks level by level,
// T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj, four adjacent columns of one row per
// thread.  Xf is fp32 scratch [3][16][16].  Ends with a block barrier.
template <int kThreads>
__device__ void unit_lower_inverse(const float* Af, float* Tf, float* Xf) {
    const int tid = threadIdx.x;
    if (tid < 64) {
        const int b = tid >> 4, c = tid & 15, o = 16 * b;
        float x[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) x[t] = t == c ? 1.f : 0.f;
#pragma unroll
        for (int r = 0; r < 15; ++r)
#pragma unroll
            for (int t = r + 1; t < 16; ++t) x[t] = fmaf(-Af[(o + t) * 65 + o + r], x[r], x[t]);
#pragma unroll
        for (int t = 0; t < 16; ++t) Tf[(o + t) * 65 + o + c] = x[t];
    }
    for (int e = tid; e < 64 * 64; e += kThreads) {
        const int i = e >> 6, j = e & 63;
        if ((i >> 4) < (j >> 4)) Tf[i * 65 + j] = 0.f;
    }
    __syncthreads();
    for (int d = 1; d < 4; ++d) {
        const int nb = 4 - d;
        if (tid < nb * 64) {
            const int bi = d + (tid >> 6), bj = bi - d, rr = (tid >> 2) & 15, cc = (tid & 3) * 4;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int k = bj; k < bi; ++k)
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    const float a = Af[(16 * bi + rr) * 65 + 16 * k + m];
                    const float* tr = Tf + (16 * k + m) * 65 + 16 * bj + cc;
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[q] = fmaf(a, tr[q], acc[q]);
                }
#pragma unroll
            for (int q = 0; q < 4; ++q) Xf[(tid >> 6) * 256 + rr * 16 + cc + q] = acc[q];
        }
        __syncthreads();
        if (tid < nb * 64) {
            const int bi = d + (tid >> 6), bj = bi - d, rr = (tid >> 2) & 15, cc = (tid & 3) * 4;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                const float a = Tf[(16 * bi + rr) * 65 + 16 * bi + m];
                const float* xr = Xf + (tid >> 6) * 256 + m * 16 + cc;
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[q] = fmaf(a, xr[q], acc[q]);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) Tf[(16 * bi + rr) * 65 + 16 * bj + cc + q] = -acc[q];
        }
        __syncthreads();
    }
}

}  // namespace pf
}  // namespace gdn
