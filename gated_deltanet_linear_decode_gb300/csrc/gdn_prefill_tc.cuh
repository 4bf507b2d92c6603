// gdn_prefill_tc.cuh -- pieces shared by the two roles of the tensor-core
// prefill kernel: the preparation role (everything of a chunk that does not
// depend on the state) and the chain role (the chunk-to-chunk recurrence and
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

// ---------------------------------------------------------------- role synchronisation
// The preparation role runs on warps 0-7 of its CTA and meets at named barrier
// 1 (the CTA's other warps have left), never at the CTA-wide barrier 0.
// The preparation role's barrier: its 16 warps (named barrier 1, never the CTA-wide one).
__device__ __forceinline__ void prep_sync() { asm volatile("bar.sync 1, 512;" ::: "memory"); }

// Ready flags: a release store by the producer after its records are written,
// an acquire load by the consumer before it reads them.
__device__ __forceinline__ void st_release(int* p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_add(int* p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Order this thread's generic-proxy accesses to global memory (the flag just
// acquired) before its later async-proxy accesses (bulk copies of the records).
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}
// Drop one 128-byte line of a consumed record from L2 without writing it back.
__device__ __forceinline__ void discard_l2(const void* p) {
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}
// Global timer (ns) for the long, time-bounded waits on ready flags.
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
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

__device__ __forceinline__ void st_out8(float* p, const float* y) {
    reinterpret_cast<float4*>(p)[0] = make_float4(y[0], y[1], y[2], y[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(y[4], y[5], y[6], y[7]);
}
__device__ __forceinline__ void st_out8(__nv_bfloat16* p, const float* y) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 v = __floats2bfloat162_rn(y[2 * i], y[2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t*>(&v);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ void st_out4(float* p, const float (&y)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(y[0], y[1], y[2], y[3]);
}
__device__ __forceinline__ void st_out4(__nv_bfloat16* p, const float (&y)[4]) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(y[0], y[1]), b = __floats2bfloat162_rn(y[2], y[3]);
    *reinterpret_cast<uint2*>(p) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
}

// acc[x][0..3] += sum_{m<16} ax[m] b[m * bs + 0..3] for the rows a0, a1
// (a0, a1, b and bs * 4 bytes 16-byte aligned)
__device__ __forceinline__ void mac16x2x4(const float* a0, const float* a1, const float* b, int bs, float (&acc)[2][4]) {
#pragma unroll
    for (int m4 = 0; m4 < 4; ++m4) {
        const float4 u = *reinterpret_cast<const float4*>(a0 + 4 * m4);
        const float4 v = *reinterpret_cast<const float4*>(a1 + 4 * m4);
        const float au[4] = {u.x, u.y, u.z, u.w}, av[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int mm = 0; mm < 4; ++mm) {
            const float4 bv = *reinterpret_cast<const float4*>(b + (4 * m4 + mm) * bs);
            const float bb[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[0][e] = fmaf(au[mm], bb[e], acc[0][e]);
                acc[1][e] = fmaf(av[mm], bb[e], acc[1][e]);
            }
        }
    }
}

// (I + A)^{-1} for a strictly lower 64 x 64 A, by a block of 256 threads, in
// 16 x 16 blocks.  A and T are fp32 with row stride kTS (16-byte rows).
//   1. D_b = (I + A_bb)^{-1}, the diagonal blocks of T, by forward substitution:
//      column c of block b per thread, with the lower triangle of A_bb in its
//      registers, each solved value folded into the rows below it at once.
//   2. Ahat_ij = D_i A_ij for the six blocks below the diagonal.
//   3. T_ij = -sum_{k=j}^{i-1} Ahat_ik T_kj (from (I + A_ii) T_ij = -sum_{k<i}
//      A_ik T_kj), block diagonal by block diagonal; each step also forms the
//      sums over k that the next one can already take, so that every step has
//      work for most threads: step a gives T10, T21, T32 and Q20 = Ahat20 D0,
//      Q31 = Ahat31 D1, Q30 = Ahat30 D0; step b gives T20 = -(Q20 + Ahat21 T10),
//      T31 = -(Q31 + Ahat32 T21), R30 = Q30 + Ahat31 T10; step c gives
//      T30 = -(R30 + Ahat32 T20).
// In 2 and 3 a thread computes rows r and r + 8, columns 4c .. 4c + 3 of a
// block, from 16-byte shared-memory loads (no bank conflicts at row strides
// kTS and 20).  The strictly upper blocks of T are not written (callers treat
// them as zero).  Hf is fp32 scratch for nine 16 x 16 blocks of row stride 20
// (11520 bytes).  While threads 0-63 solve the diagonal blocks, threads
// 64 .. kThreads-1 run side(i) with i = tid - 64 (work of the caller's that
// needs no barrier of its own).  Ends with a barrier of the role's threads.
constexpr int kTS = 68;
template <int kThreads, typename Side>
__device__ void unit_lower_inverse(const float* Af, float* Tf, float* Hf, Side&& side) {
    static_assert(kThreads >= 256, "tilings below use threads 0-255");
    constexpr int kHS = 20;                  // row stride of a scratch block
    const int tid = threadIdx.x;
    if (tid < 64) {
        const int o = 16 * (tid >> 4), c = tid & 15;
        float a[16][16];   // a[t][m] = A_bb[t][m] for m < t (in 16-byte pieces; the rest unused)
#pragma unroll
        for (int t = 1; t < 16; ++t)
#pragma unroll
            for (int m4 = 0; 4 * m4 < t; ++m4) {
                const float4 v = *reinterpret_cast<const float4*>(Af + (o + t) * kTS + o + 4 * m4);
                a[t][4 * m4] = v.x; a[t][4 * m4 + 1] = v.y; a[t][4 * m4 + 2] = v.z; a[t][4 * m4 + 3] = v.w;
            }
        float x[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) x[t] = t == c ? 1.f : 0.f;
#pragma unroll
        for (int r = 0; r < 15; ++r)
#pragma unroll
            for (int t = r + 1; t < 16; ++t) x[t] = fmaf(-a[t][r], x[r], x[t]);
#pragma unroll
        for (int t = 0; t < 16; ++t) Tf[(o + t) * kTS + o + c] = x[t];
    } else {
        side(tid - 64);
    }
    prep_sync();
    // scratch blocks: Ahat (1,0) (2,0) (2,1) (3,0) (3,1) (3,2) at 0..5; Q20, Q31, Q30 / R30 at 6..8
    auto hb = [&](int k) { return Hf + k * 16 * kHS; };
    auto ah = [](int i, int j) { return i * (i - 1) / 2 + j; };
    const int q = tid & 31, r = q >> 2, c4 = 4 * (q & 3);   // rows r, r + 8 and columns c4 .. c4+3 of a block
    auto tblk = [&](int i, int j) { return Tf + (16 * i) * kTS + 16 * j; };
    auto mac = [&](const float* a, int as, const float* b, int bs, float (&acc)[2][4]) {
        mac16x2x4(a + r * as, a + (r + 8) * as, b + c4, bs, acc);
    };
    auto store = [&](float* dst, int stride, const float (&v)[2][4], float sg) {
#pragma unroll
        for (int x = 0; x < 2; ++x)
            *reinterpret_cast<float4*>(dst + (r + 8 * x) * stride + c4) =
                make_float4(sg * v[x][0], sg * v[x][1], sg * v[x][2], sg * v[x][3]);
    };
    auto load = [&](const float* src, float (&v)[2][4]) {
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            const float4 f = *reinterpret_cast<const float4*>(src + (r + 8 * x) * kHS + c4);
            v[x][0] = f.x; v[x][1] = f.y; v[x][2] = f.z; v[x][3] = f.w;
        }
    };
    // 2. Ahat_ij = D_i A_ij: items 0..191 (block = item / 32)
    if (tid < 6 * 32) {
        const int k = tid >> 5, i = k < 1 ? 1 : k < 3 ? 2 : 3, j = k - i * (i - 1) / 2;
        float acc[2][4] = {};
        mac(tblk(i, i), kTS, Af + (16 * i) * kTS + 16 * j, kTS, acc);
        store(hb(k), kHS, acc, 1.f);
    }
    prep_sync();
    // 3a. T10, T21, T32 and Q20, Q31, Q30
    if (tid < 6 * 32) {
        // Ahat block (i, j) times D_j: (1,0) (2,1) (3,2) give T blocks, (2,0) (3,1) (3,0) the Q sums
        const int k = tid >> 5, i = k < 3 ? k + 1 : (k == 3 ? 2 : 3), j = k < 3 ? k : (k == 4 ? 1 : 0);
        float acc[2][4] = {};
        mac(hb(ah(i, j)), kHS, tblk(j, j), kTS, acc);
        if (k < 3) store(tblk(i, j), kTS, acc, -1.f);
        else store(hb(3 + k), kHS, acc, 1.f);
    }
    prep_sync();
    // 3b. T20 = -(Q20 + Ahat21 T10), T31 = -(Q31 + Ahat32 T21), R30 = Q30 + Ahat31 T10
    if (tid < 3 * 32) {
        const int k = tid >> 5, i = k ? 3 : 2, kk = k == 1 ? 2 : 1, j = k == 1 ? 1 : 0;
        float acc[2][4];
        load(hb(6 + k), acc);
        mac(hb(ah(i, kk)), kHS, tblk(kk, j), kTS, acc);
        if (k < 2) store(tblk(i, j), kTS, acc, -1.f);
        else store(hb(8), kHS, acc, 1.f);
    }
    prep_sync();
    // 3c. T30 = -(R30 + Ahat32 T20)
    if (tid < 32) {
        float acc[2][4];
        load(hb(8), acc);
        mac(hb(ah(3, 2)), kHS, tblk(2, 0), kTS, acc);
        store(tblk(3, 0), kTS, acc, -1.f);
    }
    prep_sync();
}

}  // namespace pf
}  // namespace gdn
