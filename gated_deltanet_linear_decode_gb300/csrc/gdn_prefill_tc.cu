// gdn_prefill_tc.cu -- chunked (chunk = 64) prefill of the gated DeltaNet
// layer on the sm_103a tensor cores (tcgen05 MMAs, accumulators and the fp32
// state in tensor memory), for bf16 activations.
//
// Method: xwen CLAUDE.md page, "Ground truth" (recurrent and chunk=64 forms of
// the delta rule) and "Architecture cheat sheet", "Gated DeltaNet layer".
// For a chunk of n <= 64 tokens entering with state S (S[j][i]), with
// Gam_t = g_1 + ... + g_t inside the chunk:
//   A[t][r] = beta_t e^{Gam_t-Gam_r} (k_t . k_r), r < t;   T = (I + A)^{-1}
//   U = T diag(beta) V,   W = T diag(beta e^Gam) K,   D = U - W S^T
//   O = diag(e^Gam) Q S^T + P D,   P[t][r] = e^{Gam_t-Gam_r} (q_t . k_r), r <= t
//   S' = e^{Gam_n} S + D^T diag(e^{Gam_n-Gam}) K
// Every product whose M side is the state's v-row index j is taken transposed
// so the MMA runs at M = 128 (the full tensor-core height):
//   QK  [128 x 64]  = [Q ; K] K^T                 (QK^T and KK^T stacked)
//   U^T [128 x 64]  = V^T (T diag beta)^T
//   W^T [128 x 64]  = K^T (T diag(beta e^Gam))^T
//   D^T [128 x 64]  = U^T - S W^T
//   O1  [128 x 64]  = S Q^T ;  O2 = D^T P^T ;  O^T = O1 diag(e^Gam) + O2
//   S'  [128 x 128] = e^{Gam_n} S + (D^T diag(e^{Gam_n-Gam})) K
// Precision: the operands are fp32 values split into fp16 hi + lo and every
// product except S W^T takes three MMAs (hi.hi + hi.lo + lo.hi); a CPU study
// of the chunk form with rounded operands showed single-pass 16-bit (or tf32)
// products miss the 2e-3 output tolerance by 5x while this scheme lands two
// orders of magnitude inside it.  S W^T tolerates one pass.  T comes from a
// blocked forward substitution on the CUDA cores in fp32; Gam is accumulated
// in fp64 so the decay weights keep fp32 relative accuracy.
//
// One CTA of 8 warps per (sequence, v-head): warp w reads TMEM lane quarter
// w%4 (thread <-> state row j) and the column half w/4;
// the phases of a chunk run in order, each MMA group retired through one
// mbarrier (waits are bounded and report a timeout through dev_status bit 4).
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_tc.cuh"

namespace gdn {

namespace {

constexpr int kTcThreads = 256;   // 8 warps; warps w and w+4 share TMEM lane quarter w%4

// shared memory map (bytes)
constexpr uint32_t kQKs = 0;            // [Q;K] hi at +0, lo at +32768   (128 rows x 128, canonical)
constexpr uint32_t kR1 = 65536;         // V hi/lo + T.beta hi/lo + T.beta.e^Gam hi/lo | S hi/lo | O^T fp32
constexpr uint32_t kR3 = 131072;        // solve scratch | W hi | D^T hi/lo, D^T' hi/lo
constexpr uint32_t kPs = 196608;        // P hi at +0, lo at +8192        (64 x 64)
constexpr uint32_t kMisc = 212992;
constexpr uint32_t kTcSmemBytes = kMisc + 2048;

constexpr uint32_t kVs = kR1;           // V hi +0, lo +16384              (64 rows r x 128 j)
constexpr uint32_t kTb = kR1 + 32768;   // T diag(beta) hi +0, lo +8192    (64 x 64)
constexpr uint32_t kTbe = kR1 + 49152;  // T diag(beta e^Gam) hi, lo
constexpr uint32_t kSs = kR1;           // S hi +0, lo +32768              (128 j x 128 i)
constexpr uint32_t kOT = kR1;           // O^T as fp32 [64][kLdO]
constexpr int kLdO = 132;
constexpr uint32_t kAf = kR3;           // fp32 [64][65] A
constexpr uint32_t kTf = kR3 + 16640;   // fp32 [64][65] T
constexpr uint32_t kXf = kR3 + 33280;   // fp32 [3][16][16]
constexpr uint32_t kWh = kR3;           // W^T hi (128 i x 64 t)
constexpr uint32_t kA1 = kR3;           // D^T hi +0, lo +16384            (128 j x 64 t)
constexpr uint32_t kA2 = kR3 + 32768;   // D^T diag(e^{Gam_n-Gam}) hi, lo
constexpr uint32_t kDm = kR3 + 36864;   // fp32 [64][65] decay matrix e^{Gam_t-Gam_r} (r <= t)
constexpr uint32_t kXs = kR3;           // staged raw rows: [67][q 256 B | k 256 B | v 256 B]
constexpr uint32_t kXrow = 768;
constexpr uint32_t kZs = kR1 + 36864;   // staged z rows: [64][256 B], after O^T

// tensor-memory columns
constexpr uint32_t kColS = 0, kColQK = 128, kColDU = 192, kColW = 256, kColO1 = 320, kColO2 = 384;
constexpr uint32_t kTmemCols = 512;
constexpr int kWaitLimit = 1 << 22;

__device__ __forceinline__ float conv4(float4 w, float x0, float x1, float x2, float cur) {
    return fmaf(w.w, cur, fmaf(w.z, x2, fmaf(w.y, x1, w.x * x0)));
}

// SiLU with the fast exponential and fast division (relative error of a few
// ulp, far inside the output tolerance; 0 for large negative x).
__device__ __forceinline__ float silu_fast(float x) { return x * __fdividef(1.0f, 1.0f + __expf(-x)); }

__device__ __forceinline__ void st_out4(float* p, const float (&y)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(y[0], y[1], y[2], y[3]);
}
__device__ __forceinline__ void st_out4(__nv_bfloat16* p, const float (&y)[4]) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(y[0], y[1]), b = __floats2bfloat162_rn(y[2], y[3]);
    *reinterpret_cast<uint2*>(p) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
}

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

// (I + A)^{-1} for a strictly lower 64 x 64 A (fp32, row stride 65): the four
// 16 x 16 diagonal blocks by forward substitution (column c of block b per
// thread, each solved value folded into the rows below it at once), then the
// off-diagonal blocks level by level, T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj,
// four adjacent columns of one row per thread.
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
    for (int e = tid; e < 64 * 64; e += kTcThreads) {
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

template <typename Tout>
__global__ void __launch_bounds__(kTcThreads, 1)
prefill_tc_kernel(const PrefillParams p) {
    extern __shared__ __align__(1024) uint8_t sm[];
    const int s = blockIdx.x / p.Hv, h = blockIdx.x % p.Hv, kh = h % p.Hk;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = p.cu_seqlens[s];
    const int L = p.cu_seqlens[s + 1] - t0;
    const int C = p.C, HvD = p.Hv * kD;

    float* beta_s = reinterpret_cast<float*>(sm + kMisc);
    float* g_s = beta_s + 64;
    // Gam_t as an unevaluated sum ghi + glo of two floats (formed from an fp64
    // scan), so Gam_t - Gam_r keeps fp32 relative accuracy with fp32 arithmetic.
    float* ghi_s = reinterpret_cast<float*>(sm + kMisc + 512);
    float* glo_s = reinterpret_cast<float*>(sm + kMisc + 768);
    float* egam_s = reinterpret_cast<float*>(sm + kMisc + 1024);
    float* elast_s = reinterpret_cast<float*>(sm + kMisc + 1536);   // e^{Gam_last - Gam_t}
    uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(sm + kMisc + 1280);
    uint64_t* mbar = reinterpret_cast<uint64_t*>(sm + kMisc + 1288);
    int* err_s = reinterpret_cast<int*>(sm + kMisc + 1296);
    const uint32_t sb = tc::smem_u32(sm);

    if (warp == 0) tc::tmem_alloc(tmem_base_s, kTmemCols);
    if (tid == 0) {
        tc::mbar_init(mbar, 1);
        *err_s = 0;
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_base_s;
    const int quarter = warp & 3, chalf = warp >> 2;
    const int row = quarter * 32 + lane;                                          // TMEM lane = state row j
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);      // this warp's lane quarter
    auto dgam = [&](int t, int r) { return (ghi_s[t] - ghi_s[r]) + (glo_s[t] - glo_s[r]); };
    uint32_t phase = 0;
    bool abort = false;

    auto wait_mma = [&]() {
        const bool ok = tc::mbar_wait(mbar, phase, kWaitLimit);
        phase ^= 1u;
        if (!ok) atomicExch(err_s, 1);
        tc::fence_after_sync();
    };

    // ---- initial state into tensor memory (lane j = row j)
    float* Sg = p.S + (static_cast<size_t>(s) * p.Hv + h) * kD * kD;
    {
        float v[32];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            const int c = 2 * chalf + cc;
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                float4 f = p.zero_init ? make_float4(0.f, 0.f, 0.f, 0.f)
                                       : *reinterpret_cast<const float4*>(Sg + row * kD + 32 * c + i);
                v[i] = f.x; v[i + 1] = f.y; v[i + 2] = f.z; v[i + 3] = f.w;
            }
            tc::tmem_st32(tl + kColS + 32 * c, v);
        }
        tc::tmem_wait_st();
    }

    // ---- per-lane channel ownership for the prologue
    const bool is_q = lane < 16;
    const int qk_ch = (is_q ? kh * kD : p.Hk * kD + kh * kD) + 8 * (lane & 15);
    const int v_ch = 2 * p.Hk * kD + h * kD + 4 * lane;
    float4 wqk[8], wv[4];
#pragma unroll
    for (int i = 0; i < 8; ++i) wqk[i] = *reinterpret_cast<const float4*>(p.conv_w + 4 * (qk_ch + i));
#pragma unroll
    for (int i = 0; i < 4; ++i) wv[i] = *reinterpret_cast<const float4*>(p.conv_w + 4 * (v_ch + i));
    const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(p.x);
    const __nv_bfloat16* cst = static_cast<const __nv_bfloat16*>(p.conv_state) + static_cast<size_t>(s) * 3 * C;
    const float a_dt = p.dt_bias[h], a_ssm = p.ssm_a[h];
    bool bad = false;

    // Raw rows of positions cb-3 .. cb+n-1 (q/k channels of kh, v channels of h)
    // into shared memory with asynchronous copies; completed by the next drain.
    auto stage_rows = [&](int cb) {
        const int nrow = min(kChunk, L - cb) + 3;
        for (int e = tid; e < nrow * 48; e += kTcThreads) {
            const int rr = e / 48, piece = e % 48, sec = piece >> 4, off = (piece & 15) * 8;
            const int pos = cb - 3 + rr;
            const int ch = (sec == 0 ? kh * kD : sec == 1 ? p.Hk * kD + kh * kD : 2 * p.Hk * kD + h * kD) + off;
            uint8_t* dst = sm + kXs + rr * kXrow + sec * 256 + off * 2;
            if (pos >= 0)
                tc::cp_async16(dst, x + static_cast<size_t>(t0 + pos) * C + ch);
            else if (!p.zero_init)
                tc::cp_async16(dst, cst + (3 + pos) * C + ch);
            else
                *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
        }
    };
    // Raw gate inputs of token cb + tid (threads 0..63), 0 past the sequence.
    float nx_a = 0.f, nx_b = 0.f;
    auto load_gates = [&](int cb) {
        nx_a = 0.f;
        nx_b = 0.f;
        if (tid < min(kChunk, L - cb)) {
            const size_t gi = static_cast<size_t>(t0 + cb + tid) * p.Hv + h;
            nx_b = ld_act(static_cast<const __nv_bfloat16*>(p.b_raw) + gi);
            nx_a = ld_act(static_cast<const __nv_bfloat16*>(p.a_raw) + gi);
        }
    };
    if (L > 0) {
        stage_rows(0);
        load_gates(0);
    }

    for (int c0 = 0; c0 < L && !abort; c0 += kChunk) {
        const int n = min(kChunk, L - c0);
        // ===== phase a: gates of the chunk; its raw rows were staged during the
        // previous chunk's output phase (or before the loop) and land here.
        if (tid < kChunk) {
            beta_s[tid] = tid < n ? sigmoidf_(nx_b) : 0.f;
            g_s[tid] = tid < n ? a_ssm * softplusf_(nx_a + a_dt) : 0.f;
        }
        tc::cp_async_drain();
        __syncthreads();
        if (warp == 0) {
            // inclusive scan of g in fp64: lane l owns tokens 2l, 2l+1
            const double g0 = static_cast<double>(g_s[2 * lane]), g1 = static_cast<double>(g_s[2 * lane + 1]);
            double run = g0 + g1;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double up = __shfl_up_sync(0xffffffffu, run, o);
                if (lane >= o) run += up;
            }
            const double base = run - (g0 + g1);
            const double G0 = base + g0, G1 = run;
            const float h0 = static_cast<float>(G0), h1 = static_cast<float>(G1);
            ghi_s[2 * lane] = h0;
            glo_s[2 * lane] = static_cast<float>(G0 - static_cast<double>(h0));
            ghi_s[2 * lane + 1] = h1;
            glo_s[2 * lane + 1] = static_cast<float>(G1 - static_cast<double>(h1));
            egam_s[2 * lane] = __expf(h0);
            egam_s[2 * lane + 1] = __expf(h1);
        }
#pragma unroll 2
        for (int t = warp; t < kChunk; t += 8) {
            const uint32_t qrow = is_q ? t : 64 + t;
            if (t < n) {
                float win[4][8], winv[4][4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const uint8_t* row = sm + kXs + (t + r) * kXrow;
                    bf16x8_to_f32(*reinterpret_cast<const uint4*>(row + (is_q ? 0 : 256) + 16 * (lane & 15)), win[r]);
                    bf16x4_to_f32(*reinterpret_cast<const uint2*>(row + 512 + 8 * lane), winv[r]);
                }
                float val[8], ss = 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    val[i] = silu_fast(conv4(wqk[i], win[0][i], win[1][i], win[2][i], win[3][i]));
                    ss = fmaf(val[i], val[i], ss);
                }
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);   // within 16-lane halves
                const float inv = rsqrtf(fmaxf(ss, p.eps * p.eps));   // 1 / max(||x||, eps)
#pragma unroll
                for (int i = 0; i < 8; ++i) val[i] *= inv;
                uint4 hi, lo;
                tc::split8(val, hi, lo);
                const uint32_t o = tc::cl_off(qrow, 8 * (lane & 15), 128);
                *reinterpret_cast<uint4*>(sm + kQKs + o) = hi;
                *reinterpret_cast<uint4*>(sm + kQKs + 32768 + o) = lo;
                float vv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) vv[i] = silu_fast(conv4(wv[i], winv[0][i], winv[1][i], winv[2][i], winv[3][i]));
                uint2 vh, vl;
                tc::split4(vv, vh, vl);
                const uint32_t ov = tc::cl_off(t, 4 * lane, 64);
                *reinterpret_cast<uint2*>(sm + kVs + ov) = vh;
                *reinterpret_cast<uint2*>(sm + kVs + 16384 + ov) = vl;
            } else {
                const uint32_t o = tc::cl_off(qrow, 8 * (lane & 15), 128);
                *reinterpret_cast<uint4*>(sm + kQKs + o) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(sm + kQKs + 32768 + o) = make_uint4(0, 0, 0, 0);
                const uint32_t ov = tc::cl_off(t, 4 * lane, 64);
                *reinterpret_cast<uint2*>(sm + kVs + ov) = make_uint2(0, 0);
                *reinterpret_cast<uint2*>(sm + kVs + 16384 + ov) = make_uint2(0, 0);
            }
        }
        tc::fence_proxy_async();
        __syncthreads();
        const int nl = n - 1;   // last token of the chunk

        // ===== phase b: [Q;K] K^T  (3 passes, K = 128)
        if (tid == 0) {
            tc::fence_after_sync();
            constexpr uint32_t id = tc::idesc_f16(128, 64, 0, 0, 0);
            for (int ps = 0; ps < 3; ++ps) {
                const uint32_t a = sb + kQKs + (ps == 2 ? 32768u : 0u);
                const uint32_t b = sb + kQKs + (ps == 1 ? 32768u : 0u) + 1024u;
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_f16(tmem + kColQK, tc::sdesc(a + ks * 4096, 2048, 128), tc::sdesc(b + ks * 4096, 2048, 128),
                                id, (ps | ks) ? 1u : 0u);
            }
            tc::mma_commit(mbar);
        }
        // while the MMAs run: decay matrix e^{Gam_t - Gam_r} (r <= t, else 0) and
        // e^{Gam_last - Gam_t}; the staged raw rows under kDm are consumed
        {
            float* Dm = reinterpret_cast<float*>(sm + kDm);
            const int tt = tid >> 2, r0 = (tid & 3) * 16;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int r = r0 + i;
                Dm[tt * 65 + r] = r <= tt ? __expf(dgam(tt, r)) : 0.f;
            }
            if (tid < kChunk) elast_s[tid] = __expf(dgam(nl, tid));
        }
        __syncthreads();
        wait_mma();

        // ===== phase c: P and A from the stacked product; T = (I + A)^{-1}
        {
            float* Af = reinterpret_cast<float*>(sm + kAf);
            float* Tf = reinterpret_cast<float*>(sm + kTf);
            float* Xf = reinterpret_cast<float*>(sm + kXf);
            const float* Dm = reinterpret_cast<const float*>(sm + kDm);
            float v[32];
            const int t = row & 63;
            tc::tmem_ld32(tl + kColQK + 32 * chalf, v);
            if (row < 64) {           // rows of Q K^T -> P
#pragma unroll
                for (int g8 = 0; g8 < 4; ++g8) {
                    float pv[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int r = 32 * chalf + 8 * g8 + i;
                        pv[i] = Dm[t * 65 + r] * v[8 * g8 + i];
                    }
                    uint4 hi, lo;
                    tc::split8(pv, hi, lo);
                    const uint32_t o = tc::cl_off(t, 32 * chalf + 8 * g8, 64);
                    *reinterpret_cast<uint4*>(sm + kPs + o) = hi;
                    *reinterpret_cast<uint4*>(sm + kPs + 8192 + o) = lo;
                }
            } else {                  // rows of K K^T -> A
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int r = 32 * chalf + i;
                    Af[t * 65 + r] = r < t ? beta_s[t] * Dm[t * 65 + r] * v[i] : 0.f;
                }
            }
            tc::fence_before_sync();
            __syncthreads();
            unit_lower_inverse(Af, Tf, Xf);
            // T diag(beta) and T diag(beta e^Gam): thread -> row tid/4, 16 columns
            {
                const int tr = tid >> 2, r0 = (tid & 3) * 16;
#pragma unroll
                for (int g8 = 0; g8 < 2; ++g8) {
                    float a8[8], b8[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int r = r0 + 8 * g8 + i;
                        const float tv = Tf[tr * 65 + r];
                        a8[i] = tv * beta_s[r];
                        b8[i] = tv * beta_s[r] * egam_s[r];
                    }
                    uint4 hi, lo;
                    const uint32_t o = tc::cl_off(tr, r0 + 8 * g8, 64);
                    tc::split8(a8, hi, lo);
                    *reinterpret_cast<uint4*>(sm + kTb + o) = hi;
                    *reinterpret_cast<uint4*>(sm + kTb + 8192 + o) = lo;
                    tc::split8(b8, hi, lo);
                    *reinterpret_cast<uint4*>(sm + kTbe + o) = hi;
                    *reinterpret_cast<uint4*>(sm + kTbe + 8192 + o) = lo;
                }
            }
            tc::fence_proxy_async();
            __syncthreads();
        }

        // ===== phase d: U^T = V^T (T diag beta)^T ;  W^T = K^T (T diag(beta e^Gam))^T
        if (tid == 0) {
            tc::fence_after_sync();
            constexpr uint32_t id = tc::idesc_f16(128, 64, 1, 0, 0);
            for (int ps = 0; ps < 3; ++ps) {
                const uint32_t ah = ps == 2 ? 1u : 0u, bh = ps == 1 ? 1u : 0u;
                for (int ks = 0; ks < 4; ++ks) {
                    tc::mma_f16(tmem + kColDU, tc::sdesc(sb + kVs + ah * 16384 + ks * 256, 128, 1024),
                                tc::sdesc(sb + kTb + bh * 8192 + ks * 2048, 1024, 128), id, (ps | ks) ? 1u : 0u);
                    tc::mma_f16(tmem + kColW, tc::sdesc(sb + kQKs + ah * 32768 + 1024 + ks * 256, 128, 2048),
                                tc::sdesc(sb + kTbe + bh * 8192 + ks * 2048, 1024, 128), id, (ps | ks) ? 1u : 0u);
                }
            }
            tc::mma_commit(mbar);
        }
        wait_mma();

        // ===== phase e: W^T -> fp16 operand; S -> fp16 hi/lo operand and S <- e^{Gam_n} S
        {
            float v[32];
            tc::tmem_ld32(tl + kColW + 32 * chalf, v);
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
                uint4 hi, lo;
                tc::split8(v + 8 * g8, hi, lo);
                *reinterpret_cast<uint4*>(sm + kWh + tc::cl_off(row, 32 * chalf + 8 * g8, 128)) = hi;
            }
            const float egl = egam_s[nl];
            for (int cc = 0; cc < 2; ++cc) {
                const int c = 2 * chalf + cc;
                tc::tmem_ld32(tl + kColS + 32 * c, v);
#pragma unroll
                for (int g8 = 0; g8 < 4; ++g8) {
                    uint4 hi, lo;
                    tc::split8(v + 8 * g8, hi, lo);
                    const uint32_t o = tc::cl_off(row, 32 * c + 8 * g8, 128);
                    *reinterpret_cast<uint4*>(sm + kSs + o) = hi;
                    *reinterpret_cast<uint4*>(sm + kSs + 32768 + o) = lo;
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] *= egl;
                tc::tmem_st32(tl + kColS + 32 * c, v);
            }
            tc::tmem_wait_st();
            tc::fence_proxy_async();
            tc::fence_before_sync();
            __syncthreads();
        }

        // ===== phase f: D^T = U^T - S W^T (1 pass) ;  O1 = S Q^T (3 passes)
        if (tid == 0) {
            tc::fence_after_sync();
            constexpr uint32_t idw = tc::idesc_f16(128, 64, 0, 1, 1);
            for (int ks = 0; ks < 8; ++ks)
                tc::mma_f16(tmem + kColDU, tc::sdesc(sb + kSs + ks * 4096, 2048, 128),
                            tc::sdesc(sb + kWh + ks * 256, 128, 2048), idw, 1u);
            constexpr uint32_t idq = tc::idesc_f16(128, 64, 0, 0, 0);
            for (int ps = 0; ps < 3; ++ps) {
                const uint32_t ah = ps == 2 ? 32768u : 0u, bh = ps == 1 ? 32768u : 0u;
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_f16(tmem + kColO1, tc::sdesc(sb + kSs + ah + ks * 4096, 2048, 128),
                                tc::sdesc(sb + kQKs + bh + ks * 4096, 2048, 128), idq, (ps | ks) ? 1u : 0u);
            }
            tc::mma_commit(mbar);
        }
        wait_mma();

        // ===== phase g: D^T -> fp16 operands (plain and scaled by e^{Gam_n - Gam_t});
        // the chunk's z rows start loading behind the free S operand
        {
            for (int e = tid; e < n * 16; e += kTcThreads) {   // 16 x 16 B per row
                const int t = e >> 4, off = (e & 15) * 8;
                tc::cp_async16(sm + kZs + t * 256 + off * 2, static_cast<const __nv_bfloat16*>(p.z) +
                                                                  static_cast<size_t>(t0 + c0 + t) * HvD + h * kD + off);
            }
            float v[32];
            tc::tmem_ld32(tl + kColDU + 32 * chalf, v);
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
                float sc[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int t = 32 * chalf + 8 * g8 + i;
                    sc[i] = v[8 * g8 + i] * elast_s[t];
                }
                uint4 hi, lo;
                const uint32_t o = tc::cl_off(row, 32 * chalf + 8 * g8, 128);
                tc::split8(v + 8 * g8, hi, lo);
                *reinterpret_cast<uint4*>(sm + kA1 + o) = hi;
                *reinterpret_cast<uint4*>(sm + kA1 + 16384 + o) = lo;
                tc::split8(sc, hi, lo);
                *reinterpret_cast<uint4*>(sm + kA2 + o) = hi;
                *reinterpret_cast<uint4*>(sm + kA2 + 16384 + o) = lo;
            }
            tc::fence_proxy_async();
            tc::fence_before_sync();
            __syncthreads();
        }

        // ===== phase h: O2 = D^T P^T ;  S += (D^T diag(e^{Gam_n-Gam})) K   (3 passes each)
        if (tid == 0) {
            tc::fence_after_sync();
            constexpr uint32_t idp = tc::idesc_f16(128, 64, 0, 0, 0);
            constexpr uint32_t idk = tc::idesc_f16(128, 128, 0, 1, 0);
            for (int ps = 0; ps < 3; ++ps) {
                const uint32_t ah = ps == 2 ? 16384u : 0u;
                for (int ks = 0; ks < 4; ++ks) {
                    tc::mma_f16(tmem + kColO2, tc::sdesc(sb + kA1 + ah + ks * 4096, 2048, 128),
                                tc::sdesc(sb + kPs + (ps == 1 ? 8192u : 0u) + ks * 2048, 1024, 128), idp,
                                (ps | ks) ? 1u : 0u);
                    tc::mma_f16(tmem + kColS, tc::sdesc(sb + kA2 + ah + ks * 4096, 2048, 128),
                                tc::sdesc(sb + kQKs + (ps == 1 ? 32768u : 0u) + 1024 + ks * 256, 128, 2048), idk, 1u);
                }
            }
            tc::mma_commit(mbar);
        }
        wait_mma();

        // ===== phase i: o = (e^Gam O1 + O2)/sqrt(128) -> transpose -> gated RMSNorm -> out
        {
            float* OT = reinterpret_cast<float*>(sm + kOT);
            float v1[32], v2[32];
            tc::tmem_ld32(tl + kColO1 + 32 * chalf, v1);
            tc::tmem_ld32(tl + kColO2 + 32 * chalf, v2);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int t = 32 * chalf + i;
                OT[t * kLdO + row] = fmaf(egam_s[t], v1[i], v2[i]) * kInvSqrtD;
            }
            tc::cp_async_drain();
            tc::fence_before_sync();
            __syncthreads();
            if (*err_s) abort = true;
            if (!abort && c0 + kChunk < L) {   // next chunk's inputs load behind the output
                stage_rows(c0 + kChunk);
                load_gates(c0 + kChunk);
            }
            for (int t = warp; t < n; t += 8) {
                const float4 o4 = *reinterpret_cast<const float4*>(OT + t * kLdO + 4 * lane);
                float ss = o4.x * o4.x + o4.y * o4.y + o4.z * o4.z + o4.w * o4.w;
                ss = warp_sum(ss);
                const float rs = rsqrtf(ss * (1.0f / kD) + p.eps);
                const size_t oi = static_cast<size_t>(t0 + c0 + t) * HvD + h * kD + 4 * lane;
                float zf[4];
                bf16x4_to_f32(*reinterpret_cast<const uint2*>(sm + kZs + t * 256 + 8 * lane), zf);
                const float4 w4 = *reinterpret_cast<const float4*>(p.norm_w + 4 * lane);
                const float y[4] = {o4.x * rs * w4.x * silu_fast(zf[0]), o4.y * rs * w4.y * silu_fast(zf[1]),
                                    o4.z * rs * w4.z * silu_fast(zf[2]), o4.w * rs * w4.w * silu_fast(zf[3])};
                st_out4(static_cast<Tout*>(p.out) + oi, y);
                if (p.flags & kFlagCheckFinite)
                    bad |= nonfinite_bits(y[0]) | nonfinite_bits(y[1]) | nonfinite_bits(y[2]) | nonfinite_bits(y[3]);
                if (p.prenorm) *reinterpret_cast<float4*>(p.prenorm + oi) = o4;
            }
        }
    }

    // ---- final state out (lane j = row j)
    tc::cp_async_drain();
    __syncthreads();
    bool bad_s = false;
    {
        float v[32];
        for (int cc = 0; cc < 2; ++cc) {
            const int c = 2 * chalf + cc;
            tc::tmem_ld32(tl + kColS + 32 * c, v);
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                *reinterpret_cast<float4*>(Sg + row * kD + 32 * c + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                if (p.flags & kFlagCheckFinite)
                    bad_s |= nonfinite_bits(v[i]) | nonfinite_bits(v[i + 1]) | nonfinite_bits(v[i + 2]) |
                             nonfinite_bits(v[i + 3]);
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (p.dev_status) {
        int st = 0;
        if (p.flags & kFlagCheckFinite)
            st = (__any_sync(0xffffffffu, bad_s) ? 1 : 0) | (__any_sync(0xffffffffu, bad) ? 2 : 0);
        if (tid == 0 && *err_s) st |= 16;
        if (lane == 0 && st) atomicOr(p.dev_status + s * p.Hv + h, st);
    }
    if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

template <typename Tout>
cudaError_t launch_prefill_tc_t(const PrefillParams& p, cudaStream_t stream) {
    auto k = prefill_tc_kernel<Tout>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kTcSmemBytes));
    if (e != cudaSuccess) return e;
    k<<<static_cast<unsigned>(p.n_seq) * p.Hv, kTcThreads, kTcSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_prefill_tc(const PrefillParams& p, int out_dtype, cudaStream_t stream) {
    return out_dtype == 1 ? launch_prefill_tc_t<__nv_bfloat16>(p, stream) : launch_prefill_tc_t<float>(p, stream);
}

}  // namespace gdn
