// gdn_prefill_prep.cuh -- the preparation role of the tensor-core prefill
// kernel: the work of one chunk that does not depend on the state, for every
// chunk of every sequence (xwen CLAUDE.md page, "Ground truth": chunk = 64 form;
// "Architecture cheat sheet", "Gated DeltaNet layer": conv1d k=4 without bias,
// SiLU, clamp L2 norm, tiled heads, beta = sigmoid(b), g = ssm_a softplus(a + dt_bias)).
//
// One item = (chunk, q/k head kh) and a range of the group's v-heads (all of
// them, but one each for the call's first chunk), worked by 8 warps of a CTA
// (they meet at named barrier 1, never at the CTA-wide barrier).  While the chunk's raw rows and
// conv taps land it computes the gates of every v-head h with h mod H_k = kh
// (tiled heads): beta, g, Gam (fp64 scan), e^Gam, e^{Gam_last-Gam}.  It computes
// q_hat and k_hat of the chunk once -- and from them, while they are in
// registers, Q' = diag(e^Gam) Q and K' = diag(e^{Gam_last-Gam}) K of every one
// of those v-heads -> records -- and the raw products [Q; K] K^T once on the
// tensor cores, then for each of those v-heads:
//   decay matrix e^{Gam_t-Gam_r};
//   P = decay (.) Q K^T (r <= t) -> record, A = beta decay (.) K K^T (r < t);
//   T = (I + A)^{-1} on the CUDA cores (fp32);
//   U^T = V^T (T diag beta)^T, W^T = K^T (T diag(beta e^Gam))^T on the tensor
//   cores (fp16 hi/lo split, three MMAs per product) -> record.
// The records (layouts in gdn_prefill_tc.cuh) feed the chain role
// (gdn_prefill_chain.cuh), which finds each one through its ready flag.
#pragma once

#include "gdn_internal.h"
#include "gdn_prefill_tc.cuh"

namespace gdn {
namespace prep {

constexpr int kPrepThreads = 512;   // 16 warps

// shared memory map (bytes)
constexpr uint32_t kQKs = 0;           // [Q;K] hi +0, lo +32768   (128 rows x 128, canonical)
constexpr uint32_t kVs = 65536;        // V hi +0, lo +16384       (64 r x 128 j, canonical 64 rows)
constexpr uint32_t kTb = 98304;        // T diag(beta) hi +0, lo +8192 (first: q/k conv taps, float4 [256])
constexpr uint32_t kTbe = 114688;      // T diag(beta e^Gam) hi +0, lo +8192 (first: raw gates g [G][64])
constexpr uint32_t kAf = 131072;       // fp32 [64][pf::kTS] A
constexpr uint32_t kTf = 148480;       // fp32 [64][pf::kTS] T
constexpr uint32_t kDm = 167424;       // fp32 [64][65] decay matrix; then the solve's scratch (11520 bytes)
// Raw rows arrive by TMA in boxes of [67 positions][64 channels] (128-byte rows, the
// 16-byte chunks of row R permuted by R mod 8, boxes 1024-byte aligned): channel group
// cg (8 channels) of position row R is at box (cg / 8), row R, chunk (cg % 8) ^ (R % 8),
// so a warp reading one channel group of 32 consecutive rows hits every bank once per
// 8 rows.
constexpr int kXrows = 67;             // positions c0-3 .. c0+63
constexpr uint32_t kXBoxBytes = kXrows * 128;
constexpr uint32_t kXBoxStride = 9216;  // 1024-byte aligned boxes
constexpr uint32_t kXqk = 131072;      // raw q|k rows: boxes 0-1 q, 2-3 k (consumed before kAf.. are used)
constexpr uint32_t kXv = 184320;       // raw v rows of one v-head: boxes 0-1
constexpr uint32_t kMisc = 202112;     // TMEM base, mbarriers (MMA, q|k rows, v rows), error flag
constexpr uint32_t kGates = 202176;    // per v-head of the group: 6 x [64] fp32 (below)
__device__ __forceinline__ uint32_t xrow_off(int cg, int R) {
    return static_cast<uint32_t>((cg >> 3) * kXBoxStride + R * 128 + (((cg & 7) ^ (R & 7)) << 4));
}
constexpr uint32_t kGateBytes = 6 * 256;
// then the conv taps of the current v-head, float4 [128]
__host__ __device__ inline uint32_t taps_v_off(int G) { return kGates + static_cast<uint32_t>(G) * kGateBytes; }
__host__ __device__ inline uint32_t prep_smem(int G) { return taps_v_off(G) + 128 * 16; }
static_assert(kXqk % 1024 == 0 && kXv % 1024 == 0 && kXBoxStride >= kXBoxBytes, "TMA boxes of the raw rows");
static_assert(kXqk + 3 * kXBoxStride + kXBoxBytes <= kDm, "q/k staging overlaps the decay matrix");
static_assert(kDm + 64 * 65 * 4 <= kXv, "decay matrix overlaps the v staging");
static_assert(kXv + kXBoxStride + kXBoxBytes <= kMisc && kMisc + 40 <= kGates, "v staging overlaps the barriers");
static_assert(kAf + 64 * pf::kTS * 4 <= kTf && kTf + 64 * pf::kTS * 4 <= kDm, "A / T tiles overlap");

constexpr uint32_t kColQK = 0, kColU = 64, kColW = 128, kPrepTmemCols = 256;
constexpr int kWaitLimit = 1 << 22;
constexpr uint64_t kFlowTimeoutNs = 2000000000ull;

// Per-CTA state of the preparation role, kept across items: the tensor-memory
// base (kPrepTmemCols columns), the MMA-completion mbarrier and its phase, and
// a sticky error flag (a wait gave up).
struct Ctx {
    uint32_t tmem;
    uint64_t* mbar;
    uint32_t phase;
    int* err_s;
    bool no_flow;   // thread 0: the flow-control wait gave up once, so it is skipped from then on
    uint64_t* xbar;   // the q|k raw rows of the item landed (TMA)
    uint64_t* vbar;   // a v-head's raw rows landed (TMA)
    uint32_t xphase, vphase;
};

// Item (chunk gc, q/k head kh), v-heads g_lo .. g_hi-1 of the group (a whole item takes
// 0 .. G-1; the first chunk of a call is split into one item per v-head so that the chains
// can start sooner).
__device__ void item(const PrefillParams& p, int gc, int kh, int g_lo, int g_hi, uint8_t* sm, Ctx& cx) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int Hk = p.Hk, Hv = p.Hv, C = p.C;

    // Flow control: the records of (chunk gc, q/k head kh) are written once the H_v / H_k
    // chains of the group are done with chunk gc - ahead, so that the records in flight stay
    // in L2.  Thread 0 waits (bounded in time; it stops waiting for good once a chain has
    // given up), the others start staging, and the first barrier of the item holds every
    // record write until it is through.
    if (tid == 0 && gc >= p.ahead && !cx.no_flow) {
        const int* f = p.consumed + static_cast<size_t>(gc - p.ahead) * Hk + kh;
        const volatile int* abort_flag = p.abort_flag;
        const int need = Hv / Hk;
        if (pf::ld_acquire(f) < need) {
            const uint64_t tstart = pf::global_ns();
            uint32_t ns = 128;
            while (pf::ld_acquire(f) < need) {
                if (*abort_flag || pf::global_ns() - tstart > kFlowTimeoutNs) {
                    cx.no_flow = true;
                    break;
                }
                __nanosleep(ns);
                ns = min(ns * 2, 2048u);
            }
        }
    }

    // sequence of this chunk: the last s with chunk_base[s] <= gc (a non-empty one)
    const int* tab = p.chunk_base;
    int lo = 0, hi = p.n_seq;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (tab[mid] <= gc) lo = mid; else hi = mid;
    }
    const int s = lo;
    const int c0 = (gc - tab[s]) * kChunk;
    const int t0 = p.cu_seqlens[s];
    const int n = min(kChunk, p.cu_seqlens[s + 1] - t0 - c0);
    const int nl = n - 1;

    // Per v-head gate arrays (head g of the group at kGates + g * kGateBytes):
    // beta, e^g, Gam_t as an unevaluated sum ghi + glo of two floats (formed from
    // an fp64 scan, so Gam_t - Gam_r keeps fp32 relative accuracy), e^Gam_t and
    // e^{Gam_last - Gam_t}.
    auto gate = [&](int g, int k) { return reinterpret_cast<float*>(sm + kGates + g * kGateBytes) + 64 * k; };
    enum { kBeta = 0, kEg, kGhi, kGlo, kEgam, kElast };
    const int G = Hv / Hk;
    const float4* taps_qk = reinterpret_cast<const float4*>(sm + kTb);
    const float4* taps_v = reinterpret_cast<const float4*>(sm + taps_v_off(G));
    uint64_t* mbar = cx.mbar;
    int* err_s = cx.err_s;
    const uint32_t sb = tc::smem_u32(sm);
    const uint32_t tmem = cx.tmem;
    const int quarter = warp & 3, cq = warp >> 2;   // TMEM lane quarter; column quarter of a 64-wide tile
    const int row = quarter * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float* ghi_s = nullptr;
    const float* glo_s = nullptr;
    auto dgam = [&](int t, int r) { return (ghi_s[t] - ghi_s[r]) + (glo_s[t] - glo_s[r]); };
    auto wait_mma = [&]() {
        const bool ok = tc::mbar_wait(mbar, cx.phase, kWaitLimit);
        cx.phase ^= 1u;
        if (!ok) atomicExch(err_s, 1);
        tc::fence_after_sync();
    };

    // ---- stage the raw rows of positions c0-3 .. c0+63 by TMA (one thread; positions past the
    // tensor read as zeros, positions past the sequence are never used) and the conv taps.
    // In the first chunk of a sequence, rows 0-2 (positions -3 .. -1) are replaced, once
    // landed, by the carried conv state (zeros with zero_init).
    const __nv_bfloat16* cst = static_cast<const __nv_bfloat16*>(p.conv_state) + static_cast<size_t>(s) * 3 * C;
    const int y0 = t0 + c0 - 3;
    auto left_context = [&](uint32_t box0, int nbox, int ch0, int idx, int cnt) {
        // rows 0-2 of boxes box0 .. box0+nbox-1 (channels ch0 + 64 * box ..), 8 channels a thread
        for (int e = idx; e < nbox * 3 * 8; e += cnt) {
            const int bx = e / 24, R = (e / 8) % 3, c = e & 7;
            const uint4 v = p.zero_init ? make_uint4(0, 0, 0, 0)
                                        : *reinterpret_cast<const uint4*>(cst + R * C + ch0 + 64 * bx + 8 * c);
            *reinterpret_cast<uint4*>(sm + box0 + bx * kXBoxStride + R * 128 + ((c ^ R) << 4)) = v;
        }
    };
    auto stage_v_rows = [&](int h) {   // one thread
        tc::fence_proxy_async();   // the generic reads of the previous v rows come first
        tc::mbar_expect_tx(cx.vbar, 2 * kXBoxBytes);
        for (int bx = 0; bx < 2; ++bx)
            tc::tma_load_2d(sm + kXv + bx * kXBoxStride, &p.xmap, 2 * Hk * kD + h * kD + 64 * bx, y0, cx.vbar);
    };
    if (tid == 0) {
        tc::fence_proxy_async();
        tc::mbar_expect_tx(cx.xbar, 4 * kXBoxBytes);
        for (int bx = 0; bx < 4; ++bx)
            tc::tma_load_2d(sm + kXqk + bx * kXBoxStride, &p.xmap, (bx >> 1) * Hk * kD + kh * kD + 64 * (bx & 1), y0,
                            cx.xbar);
        stage_v_rows(kh + g_lo * Hk);
    }
    if (tid < 256)   // one q/k channel's taps per thread
        tc::cp_async16(sm + kTb + 16 * tid,
                       reinterpret_cast<const float4*>(p.conv_w) + ((tid >> 7) * Hk * kD + kh * kD + (tid & 127)));
    // v-head h's conv taps, by threads idx = 0 .. cnt-1
    auto stage_v_taps = [&](int h, int idx, int cnt) {
        for (int c = idx; c < kD; c += cnt)
            tc::cp_async16(sm + taps_v_off(G) + 16 * c, reinterpret_cast<const float4*>(p.conv_w) + (2 * Hk * kD + h * kD + c));
    };
    stage_v_taps(kh + g_lo * Hk, tid, kPrepThreads);
    // wait for v-head h's raw rows (all threads), then its left context in a first chunk
    auto land_v_rows = [&](int h) {
        if (!tc::mbar_wait(cx.vbar, cx.vphase, kWaitLimit)) atomicExch(err_s, 1);
        cx.vphase ^= 1u;
        if (c0 == 0) {
            left_context(kXv, 2, 2 * Hk * kD + h * kD, tid, kPrepThreads);
            pf::prep_sync();
        }
    };

    // ---- gates of every v-head of the group while the rows land: beta, g, e^g; then
    // warp g scans head g's g in fp64 into Gam, e^Gam and e^{Gam_last - Gam}
    {
        float* graw = reinterpret_cast<float*>(sm + kTbe);   // [G][64]
        static_assert(16 * 64 * 4 <= 16384, "raw gates of up to 16 v-heads");
        for (int e = tid; e < kChunk * G; e += kPrepThreads) {
            const int g = e >> 6, t = e & 63, h = kh + g * Hk;
            float bt = 0.f, gt = 0.f;
            if (t < n) {
                const size_t gi = static_cast<size_t>(t0 + c0 + t) * Hv + h;
                bt = sigmoidf_(ld_act(static_cast<const __nv_bfloat16*>(p.b_raw) + gi));
                gt = p.ssm_a[h] * softplusf_(ld_act(static_cast<const __nv_bfloat16*>(p.a_raw) + gi) + p.dt_bias[h]);
            }
            gate(g, kBeta)[t] = bt;
            graw[e] = gt;
            gate(g, kEg)[t] = __expf(gt);
        }
        pf::prep_sync();
        for (int g = warp; g < G; g += kPrepThreads / 32) {
            // inclusive scan in fp64: lane l owns tokens 2l, 2l+1
            const double g0 = static_cast<double>(graw[64 * g + 2 * lane]), g1 = static_cast<double>(graw[64 * g + 2 * lane + 1]);
            double run = g0 + g1;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double up = __shfl_up_sync(0xffffffffu, run, o);
                if (lane >= o) run += up;
            }
            const double G0 = run - g1, G1 = run;
            const double Gl = __shfl_sync(0xffffffffu, (nl & 1) ? G1 : G0, nl >> 1);   // Gam of the last token
            const float h0 = static_cast<float>(G0), h1 = static_cast<float>(G1);
            gate(g, kGhi)[2 * lane] = h0;
            gate(g, kGlo)[2 * lane] = static_cast<float>(G0 - static_cast<double>(h0));
            gate(g, kGhi)[2 * lane + 1] = h1;
            gate(g, kGlo)[2 * lane + 1] = static_cast<float>(G1 - static_cast<double>(h1));
            gate(g, kEgam)[2 * lane] = __expf(h0);
            gate(g, kEgam)[2 * lane + 1] = __expf(h1);
            gate(g, kElast)[2 * lane] = __expf(static_cast<float>(Gl - G0));
            gate(g, kElast)[2 * lane + 1] = __expf(static_cast<float>(Gl - G1));
        }
    }
    tc::cp_async_drain();
    if (!tc::mbar_wait(cx.xbar, cx.xphase, kWaitLimit)) atomicExch(err_s, 1);
    cx.xphase ^= 1u;
    if (c0 == 0) {
        left_context(kXqk, 2, kh * kD, tid, kPrepThreads);
        left_context(kXqk + 2 * kXBoxStride, 2, Hk * kD + kh * kD, tid, kPrepThreads);
    }
    pf::prep_sync();

    // ---- q_hat, k_hat: conv, SiLU, clamp L2 -> [Q;K] hi/lo in shared memory.
    // Warp w owns staged channel groups 2w, 2w+1 (q for w < 8, k for w >= 8;
    // their conv taps held in registers), lanes = tokens lane and 32 + lane; the
    // eight warps of a section meet in shared memory (the decay-matrix area,
    // unused until later) to form each token's norm.
    {
        const int sec = warp >> 3;
        float* ssq = reinterpret_cast<float*>(sm + kDm);   // [16 warps][64 tokens]
        float val[2][2][8];
        float ss[2] = {0.f, 0.f};
#pragma unroll
        for (int gq = 0; gq < 2; ++gq) {
            const int cg = 2 * warp + gq;   // 0..31
            float4 w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) w[i] = taps_qk[sec * kD + 8 * (cg & 15) + i];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int t = 32 * hf + lane;
                float win[4][8];
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    pf::bf16x8_to_f32(*reinterpret_cast<const uint4*>(sm + kXqk + xrow_off(cg, t + r)), win[r]);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float v = pf::silu_fast(pf::conv4(w[i], win[0][i], win[1][i], win[2][i], win[3][i]));
                    val[hf][gq][i] = t < n ? v : 0.f;
                    ss[hf] = fmaf(val[hf][gq][i], val[hf][gq][i], ss[hf]);
                }
            }
        }
        ssq[warp * 64 + lane] = ss[0];
        ssq[warp * 64 + 32 + lane] = ss[1];
        pf::prep_sync();
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int t = 32 * hf + lane;
            const float* q8 = ssq + 8 * sec * 64 + t;
            const float sum = ((q8[0] + q8[64]) + (q8[128] + q8[192])) + ((q8[256] + q8[320]) + (q8[384] + q8[448]));
            const float inv = rsqrtf(fmaxf(sum, p.eps * p.eps));   // 1 / max(||x||, eps)
#pragma unroll
            for (int gq = 0; gq < 2; ++gq) {
#pragma unroll
                for (int i = 0; i < 8; ++i) val[hf][gq][i] *= inv;
                uint4 vh, vl;
                tc::split8(val[hf][gq], vh, vl);
                const int ch = 8 * ((2 * warp + gq) & 15);
                const uint32_t so = tc::cl_off(64 * sec + t, ch, 128);
                *reinterpret_cast<uint4*>(sm + kQKs + so) = vh;
                *reinterpret_cast<uint4*>(sm + kQKs + 32768 + so) = vl;
                // Q' = diag(e^Gam) Q and K' = diag(e^{Gam_last - Gam}) K of every v-head of the
                // group -> fp16 hi/lo records (the gates are known by now)
                const uint32_t go = tc::cl_off(t, ch, 64);
#pragma unroll 1
                for (int g = g_lo; g < g_hi; ++g) {
                    const float e = gate(g, sec == 0 ? kEgam : kElast)[t];
                    float sv[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) sv[i] = e * val[hf][gq][i];
                    uint4 oh, ol;
                    tc::split8(sv, oh, ol);
                    uint8_t* dst = p.ws_v + (static_cast<size_t>(gc) * Hv + kh + g * Hk) * pf::kVRec +
                                   (sec == 0 ? pf::kRecQhi : pf::kRecKhi);
                    *reinterpret_cast<uint4*>(dst + go) = oh;
                    *reinterpret_cast<uint4*>(dst + 16384 + go) = ol;
                }
            }
        }
    }
    tc::fence_proxy_async();
    pf::prep_sync();
    // [Q;K] K^T (3 passes, K = 128): rows t < 64 give Q K^T, rows 64 + t give K K^T
    if (tid == 0) {
        tc::fence_after_sync();
        constexpr uint32_t id = tc::idesc_f16(128, 64, 0, 0, 0);
        for (int ps = 0; ps < 3; ++ps) {
            const uint32_t a = sb + kQKs + (ps == 2 ? 32768u : 0u);
            const uint32_t b = sb + kQKs + (ps == 1 ? 32768u : 0u) + 1024u;
            for (int ks = 0; ks < 8; ++ks)
                tc::mma_f16(tmem + kColQK, tc::sdesc(a + ks * 4096, 2048, 128), tc::sdesc(b + ks * 4096, 2048, 128), id,
                            (ps | ks) ? 1u : 0u);
        }
        tc::mma_commit(mbar);
    }

    const float* Af = reinterpret_cast<const float*>(sm + kAf);
    for (int g = g_lo; g < g_hi; ++g) {
        const int h = kh + g * Hk;
        uint8_t* vrec = p.ws_v + (static_cast<size_t>(gc) * Hv + h) * pf::kVRec;
        land_v_rows(h);
        const float* beta_s = gate(g, kBeta);
        const float* eg_s = gate(g, kEg);
        const float* egam_s = gate(g, kEgam);
        const float* elast_s = gate(g, kElast);
        ghi_s = gate(g, kGhi);
        glo_s = gate(g, kGlo);
        // v: conv, SiLU -> V hi/lo (64 r x 128 j); warp w: channel group w
        // (taps in registers), lanes = tokens lane and 32 + lane
        {
            const int cg = warp;
            float4 w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) w[i] = taps_v[8 * cg + i];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int t = 32 * hf + lane;
                uint4 vh = make_uint4(0, 0, 0, 0), vl = make_uint4(0, 0, 0, 0);
                if (t < n) {
                    float win[4][8], vv[8];
#pragma unroll
                    for (int r = 0; r < 4; ++r)
                        pf::bf16x8_to_f32(*reinterpret_cast<const uint4*>(sm + kXv + xrow_off(cg, t + r)), win[r]);
#pragma unroll
                    for (int i = 0; i < 8; ++i) vv[i] = pf::silu_fast(pf::conv4(w[i], win[0][i], win[1][i], win[2][i], win[3][i]));
                    tc::split8(vv, vh, vl);
                }
                const uint32_t ov = tc::cl_off(t, 8 * cg, 64);
                *reinterpret_cast<uint4*>(sm + kVs + ov) = vh;
                *reinterpret_cast<uint4*>(sm + kVs + 16384 + ov) = vl;
            }
        }
        pf::prep_sync();
        // decay matrix e^{Gam_t - Gam_r} (r <= t, else 0): one exponential at the right end
        // of the thread's 16 columns, then leftwards e^{Gam_t - Gam_{r-1}} = e^{Gam_t - Gam_r} e^{g_r};
        // e^Gam and e^{Gam_last - Gam_t} -> record
        {
            float* Dm = reinterpret_cast<float*>(sm + kDm);
            const int tt = tid & 63, r0 = (tid >> 6) * 8, rs = min(r0 + 7, tt);
            float val = rs >= r0 ? __expf(dgam(tt, rs)) : 0.f;
#pragma unroll
            for (int i = 7; i >= 0; --i) {
                const int r = r0 + i;
                Dm[tt * 65 + r] = r <= rs ? val : 0.f;
                if (r <= rs) val *= eg_s[r];
            }
            if (tid < kChunk) {
                reinterpret_cast<float*>(vrec + pf::kRecEgam)[tid] = egam_s[tid];
                reinterpret_cast<float*>(vrec + pf::kRecElast)[tid] = elast_s[tid];
            }
        }
        pf::prep_sync();
        if (g == g_lo) wait_mma();   // the [Q;K] K^T products
        else tc::fence_after_sync();
        // P (rows t < 64 of the product) -> record; A (rows 64 + t) -> shared fp32
        {
            const float* Dm = reinterpret_cast<const float*>(sm + kDm);
            float* Afw = reinterpret_cast<float*>(sm + kAf);
            float v[16];
            const int t = row & 63;
            tc::tmem_ld16(tl + kColQK + 16 * cq, v);
            if (row < 64) {
#pragma unroll
                for (int g8 = 0; g8 < 2; ++g8) {
                    float pv[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) pv[i] = Dm[t * 65 + 16 * cq + 8 * g8 + i] * v[8 * g8 + i];
                    uint4 ph, pl;
                    tc::split8(pv, ph, pl);
                    const uint32_t o = tc::cl_off(t, 16 * cq + 8 * g8, 64);
                    *reinterpret_cast<uint4*>(vrec + pf::kRecPhi + o) = ph;
                    *reinterpret_cast<uint4*>(vrec + pf::kRecPlo + o) = pl;
                }
            } else {
                const float bt = beta_s[t];
#pragma unroll
                for (int i = 0; i < 16; i += 4) {   // 16-byte stores: a row per lane, no bank conflicts
                    float a4[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int r = 16 * cq + i + k;
                        a4[k] = r < t ? bt * Dm[t * 65 + r] * v[i + k] : 0.f;
                    }
                    *reinterpret_cast<float4*>(Afw + t * pf::kTS + 16 * cq + i) = make_float4(a4[0], a4[1], a4[2], a4[3]);
                }
            }
        }
        tc::fence_before_sync();
        pf::prep_sync();
        // the next v-head's raw rows start loading while the diagonal blocks are solved
        pf::unit_lower_inverse<kPrepThreads>(Af, reinterpret_cast<float*>(sm + kTf), reinterpret_cast<float*>(sm + kDm),
                                             [&](int i) {
                                                 if (g + 1 < g_hi) {
                                                     if (i == 0) stage_v_rows(h + Hk);
                                                     stage_v_taps(h + Hk, i, kPrepThreads - 64);
                                                 }
                                             });
        // T diag(beta) and T diag(beta e^Gam): thread -> row tid%64, 16 columns
        {
            const float* Tf = reinterpret_cast<const float*>(sm + kTf);
            const int tr = tid & 63, r0 = (tid >> 6) * 8;
            {
                constexpr int g8 = 0;
                float a8[8], b8[8];
                const bool lower = (r0 >> 4) <= (tr >> 4);   // T is block lower triangular
                float t8[8] = {};
                if (lower) {   // 16-byte loads: a row per lane, no bank conflicts
                    const float4 u = *reinterpret_cast<const float4*>(Tf + tr * pf::kTS + r0 + 8 * g8);
                    const float4 w = *reinterpret_cast<const float4*>(Tf + tr * pf::kTS + r0 + 8 * g8 + 4);
                    t8[0] = u.x; t8[1] = u.y; t8[2] = u.z; t8[3] = u.w; t8[4] = w.x; t8[5] = w.y; t8[6] = w.z; t8[7] = w.w;
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int r = r0 + 8 * g8 + i;
                    const float tb = t8[i] * beta_s[r];
                    a8[i] = tb;
                    b8[i] = tb * egam_s[r];
                }
                uint4 hi8, lo8;
                const uint32_t o = tc::cl_off(tr, r0 + 8 * g8, 64);
                tc::split8(a8, hi8, lo8);
                *reinterpret_cast<uint4*>(sm + kTb + o) = hi8;
                *reinterpret_cast<uint4*>(sm + kTb + 8192 + o) = lo8;
                tc::split8(b8, hi8, lo8);
                *reinterpret_cast<uint4*>(sm + kTbe + o) = hi8;
                *reinterpret_cast<uint4*>(sm + kTbe + 8192 + o) = lo8;
            }
        }
        tc::fence_proxy_async();
        pf::prep_sync();
        // U^T = V^T (T diag beta)^T ;  W^T = K^T (T diag(beta e^Gam))^T   (3 passes each, K = 64)
        if (tid == 0) {
            tc::fence_after_sync();
            constexpr uint32_t id = tc::idesc_f16(128, 64, 1, 0, 0);
            for (int ps = 0; ps < 3; ++ps) {
                const uint32_t ah = ps == 2 ? 1u : 0u, bh = ps == 1 ? 1u : 0u;
                for (int ks = 0; ks < 4; ++ks) {
                    tc::mma_f16(tmem + kColU, tc::sdesc(sb + kVs + ah * 16384 + ks * 256, 128, 1024),
                                tc::sdesc(sb + kTb + bh * 8192 + ks * 2048, 1024, 128), id, (ps | ks) ? 1u : 0u);
                    tc::mma_f16(tmem + kColW, tc::sdesc(sb + kQKs + ah * 32768 + 1024 + ks * 256, 128, 2048),
                                tc::sdesc(sb + kTbe + bh * 8192 + ks * 2048, 1024, 128), id, (ps | ks) ? 1u : 0u);
                }
            }
            tc::mma_commit(mbar);
        }
        wait_mma();
        // W^T -> fp16 hi (rows i) and U^T -> fp32 (rows j) into the record
        {
            float v[16];
            tc::tmem_ld16(tl + kColW + 16 * cq, v);
#pragma unroll
            for (int g8 = 0; g8 < 2; ++g8) {
                uint4 wh, wl;
                tc::split8(v + 8 * g8, wh, wl);
                *reinterpret_cast<uint4*>(vrec + pf::kRecW + tc::cl_off(row, 16 * cq + 8 * g8, 128)) = wh;
            }
            tc::tmem_ld16(tl + kColU + 16 * cq, v);
            float4* U4 = reinterpret_cast<float4*>(vrec + pf::kRecU);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                U4[(4 * cq + q) * kD + row] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
        tc::cp_async_drain();
        tc::fence_before_sync();
        // publish v-head h: its records (this head's part and the Q', K' written before the
        // loop) are complete once every thread is through the barrier; one thread then
        // makes them visible at GPU scope (cumulative through the barrier) before the
        // head's ready flag, which the chain role acquires before reading them
        pf::prep_sync();
        if (tid == 0) {
            __threadfence();
            if (p.dev_status && *err_s) atomicOr(p.dev_status + s * Hv + h, 16);
            pf::st_release(p.ready + static_cast<size_t>(gc) * Hv + h, 1);
        }
    }
}

// Shared-memory bytes of the role for H_v / H_k = G.
__host__ __device__ inline uint32_t smem_bytes(int G) { return prep_smem(G); }

}  // namespace prep
}  // namespace gdn
