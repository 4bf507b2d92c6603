// gdn_prefill_state.cu -- second kernel of the tensor-core prefill: the
// chunk-to-chunk state recurrence and the layer output (xwen CLAUDE.md page,
// "Ground truth": chunk = 64 form; "Architecture cheat sheet", "Gated DeltaNet
// layer": o = S q / sqrt(128), gated RMSNorm y = o / sqrt(mean(o^2) + eps)
// * norm_w * silu(z)).  Every state-independent quantity of a chunk comes from
// the records of the preparation kernel.
//
// One CTA per (sequence, v-head); the fp32 state lives in tensor memory
// (lane j = v-row j).  Per chunk, with every product transposed so the MMA
// runs at M = 128:
//   Dacc = S W^T        (fp16 hi/lo of S x W^T hi, one MMA pass)
//   O1   = S Q^T        (three passes: hi.hi + hi.lo + lo.hi)
//   D^T  = U^T - Dacc,  D'^T = D^T diag(e^{Gam_last - Gam})
//   S    = e^{Gam_last} S + D'^T K   (three passes)
//   O2   = D^T P^T      (three passes)
//   o_t  = (e^{Gam_t} O1 + O2)[:, t] / sqrt(128)  -> gated RMSNorm -> out
// Warp roles:
//   warps 0-7   convert: S -> fp16 operand (and the decay of S), Dacc -> D, D'
//   warps 8-11  epilogue: O1, O2 -> o -> gated RMSNorm -> out (one chunk behind)
//   warp 12     control: one lane issues the bulk copies of the records and the MMAs
// and they meet only at mbarriers, so the epilogue of a chunk and the bulk
// copies of the next overlap the conversions and MMAs of the current one.
// Every wait has an iteration limit; a timeout sets dev_status bit 4.
#include "gdn_internal.h"
#include "gdn_prefill_tc.cuh"

namespace gdn {

namespace {

constexpr int kConvWarps = 8, kEpiWarps = 4;
constexpr int kCtrlWarp = kConvWarps + kEpiWarps;
constexpr int kStateThreads = (kConvWarps + kEpiWarps + 1) * 32;
constexpr int kConvThreads = kConvWarps * 32, kEpiThreads = kEpiWarps * 32;

// shared memory map (bytes)
constexpr uint32_t kSs = 0;           // S hi +0, lo +32768        (128 j x 128 i, canonical 128 rows)
constexpr uint32_t kDs = 65536;       // D hi +0, lo +16384; D' hi +32768, lo +49152  (128 j x 64 t)
constexpr uint32_t kQs = 131072;      // Q hi +0, lo +16384        (64 t x 128 i, canonical 64 rows)
constexpr uint32_t kKs = 163840;      // K hi +0, lo +16384
constexpr uint32_t kWs = 196608;      // W^T hi                   (128 i x 64 t, canonical 128 rows)
constexpr uint32_t kPs = 212992;      // P hi +0, lo +8192         (64 t x 64 r, canonical 64 rows)
constexpr uint32_t kRs = 229376;      // RMS partial sums [2][4][64] fp32
constexpr uint32_t kEs = 231424;      // e^Gam of even / odd chunks [2][64] fp32
constexpr uint32_t kBar = 231936;     // mbarriers, then the TMEM base and the error flag
constexpr uint32_t kStateSmem = kBar + 160;
static_assert(kStateSmem <= 232448, "shared memory of the state pass exceeds 227 KB");

// mbarrier slots
enum : int {
    kLdQ = 0, kLdK, kLdW, kLdP,        // record copies landed (transaction count)
    kMmaD, kMmaO1, kMmaS,              // MMA groups retired (tcgen05.commit)
    kMmaO2a, kMmaO2b,                  // O2 of even / odd chunks retired
    kSReady, kDReady,                  // converters wrote S / D operands (256 arrivals)
    kEpiA, kEpiB,                      // epilogue done with O buffers of even / odd chunks (128 arrivals)
    kRsReady,                          // epilogue wrote its per-token partial sums (128 arrivals)
    kLdEa, kLdEb,                      // e^Gam of an even / odd chunk landed
    kDrain,                            // error path: every MMA issued so far retired
    kNumBars
};

// tensor-memory columns
constexpr uint32_t kColS = 0, kColD = 128, kColO1 = 192, kColO2 = 320;   // O1 / O2: two buffers of 64
constexpr uint32_t kTmemCols = 512;
constexpr int kWaitLimit = 1 << 24;

template <typename Tout>
__global__ void __launch_bounds__(kStateThreads, 1) state_pass_kernel(const PrefillParams p) {
    extern __shared__ __align__(1024) uint8_t sm[];
    const int s = blockIdx.x / p.Hv, h = blockIdx.x % p.Hv, kh = h % p.Hk;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = p.cu_seqlens[s], L = p.cu_seqlens[s + 1] - t0;
    const int cbase = p.chunk_base[s], nch = p.chunk_base[s + 1] - cbase;
    const int Hv = p.Hv, Hk = p.Hk, HvD = Hv * kD;

    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBar);
    static_assert(8 * kNumBars + 8 <= 160, "mbarrier area");
    uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(sm + kBar + 8 * kNumBars);
    volatile int* err_s = reinterpret_cast<volatile int*>(sm + kBar + 8 * kNumBars + 4);
    const uint32_t sb = tc::smem_u32(sm);

    if (warp == 0) tc::tmem_alloc(tmem_base_s, kTmemCols);
    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i) {
            const uint32_t cnt = (i == kSReady || i == kDReady)                 ? kConvThreads
                                 : (i == kEpiA || i == kEpiB || i == kRsReady) ? kEpiThreads
                                                                               : 1;
            tc::mbar_init(bars + i, cnt);
        }
        *err_s = 0;
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_base_s;

    // Bounded wait that also gives up as soon as another role has timed out.
    // Converter and epilogue warps back off with short sleeps so that waiting
    // warps leave the issue slots to the working ones; the control lane polls.
    const bool sleepy = warp != kConvWarps + kEpiWarps;
    auto wait = [&](int bar, uint32_t parity) -> bool {
        uint32_t ns = 32;
        for (int it = 0; it < kWaitLimit; it += 8) {
            if (tc::mbar_wait(bars + bar, parity, 8)) return true;
            if (*err_s) return false;
            if (sleepy) {
                __nanosleep(ns);
                ns = min(ns * 2, 256u);
            }
        }
        *err_s = 1;
        return false;
    };

    float* Sg = p.S + (static_cast<size_t>(s) * Hv + h) * kD * kD;
    const uint8_t* vrec0 = p.ws_v + (static_cast<size_t>(cbase) * Hv + h) * pf::kVRec;
    const uint8_t* qkrec0 = p.ws_qk + (static_cast<size_t>(cbase) * Hk + kh) * pf::kQKRec;
    auto vrec = [&](int c) { return vrec0 + static_cast<size_t>(c) * Hv * pf::kVRec; };
    auto qkrec = [&](int c) { return qkrec0 + static_cast<size_t>(c) * Hk * pf::kQKRec; };

    // ---- initial state into tensor memory (converter warps; lane j = row j)
    const int quarter = warp & 3;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const int row = quarter * 32 + lane;
    if (warp < kConvWarps) {
        const int chalf = warp >> 2;
        float v[32];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            const int c = 2 * chalf + cc;
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                const float4 f = p.zero_init ? make_float4(0.f, 0.f, 0.f, 0.f)
                                             : *reinterpret_cast<const float4*>(Sg + row * kD + 32 * c + i);
                v[i] = f.x; v[i + 1] = f.y; v[i + 2] = f.z; v[i + 3] = f.w;
            }
            tc::tmem_st32(tl + kColS + 32 * c, v);
        }
        tc::tmem_wait_st();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    bool bad = false;
    if (warp == kCtrlWarp) {
        // ================= control: bulk copies of the records and the MMAs
        if (lane == 0 && nch > 0) {
            // chunks whose records were requested / seen landed, for the (Q, W) and
            // (K, P) barrier pairs (an error path drains the difference)
            int req_qw = 0, got_qw = 0, req_k = 0, req_p = 0, got_kp = 0;
            auto load = [&](int bar, void* dst, const uint8_t* src, uint32_t bytes) {
                tc::mbar_expect_tx(bars + bar, bytes);
                tc::bulk_g2s(dst, src, bytes, bars + bar);
            };
            auto load_q = [&](int c) { load(kLdQ, sm + kQs, qkrec(c) + pf::kRecQhi, 32768); };
            auto load_k = [&](int c) { load(kLdK, sm + kKs, qkrec(c) + pf::kRecKhi, 32768); req_k = c + 1; };
            auto load_w = [&](int c) { load(kLdW, sm + kWs, vrec(c) + pf::kRecW, 16384); req_qw = c + 1; };
            auto load_p = [&](int c) { load(kLdP, sm + kPs, vrec(c) + pf::kRecPhi, 16384); req_p = c + 1; };
            int req_e[2] = {0, 0}, got_e = 0;   // E copies are waited for by the epilogue
            auto load_e = [&](int c) {
                load(c & 1 ? kLdEb : kLdEa, sm + kEs + 256 * (c & 1), vrec(c) + pf::kRecEgam, 256);
                req_e[c & 1] = c + 1;
            };
            auto prefetch = [&](int c) {   // chunk c's records toward L2
                tc::bulk_prefetch_l2(qkrec(c), pf::kQKRec);
                tc::bulk_prefetch_l2(vrec(c), pf::kRecU);
            };
            load_q(0); load_w(0); load_k(0); load_p(0); load_e(0);
            if (nch > 1) { load_e(1); prefetch(1); }
            if (nch > 2) prefetch(2);
            (void)got_e;
            bool ok = true;
            int c = 0;
            for (; c < nch && ok; ++c) {
                const uint32_t pc = c & 1, b = c & 1, pb = (c >> 1) & 1;
                ok = wait(kSReady, pc) && wait(kLdW, pc) && wait(kLdQ, pc);
                if (!ok) break;
                got_qw = c + 1;
                tc::fence_after_sync();
                {   // Dacc = S W^T (1 pass, K = 128)
                    constexpr uint32_t id = tc::idesc_f16(128, 64, 0, 1, 0);
                    for (int ks = 0; ks < 8; ++ks)
                        tc::mma_f16(tmem + kColD, tc::sdesc(sb + kSs + ks * 4096, 2048, 128),
                                    tc::sdesc(sb + kWs + ks * 256, 128, 2048), id, ks ? 1u : 0u);
                    tc::mma_commit(bars + kMmaD);
                }
                if (c >= 2) {
                    if (!(ok = wait(b ? kEpiB : kEpiA, ((c - 2) >> 1) & 1))) break;
                    load_e(c);
                }
                if (c + 3 < nch) prefetch(c + 3);
                tc::fence_after_sync();
                {   // O1[b] = S Q^T (3 passes, K = 128)
                    constexpr uint32_t id = tc::idesc_f16(128, 64, 0, 0, 0);
                    for (int ps = 0; ps < 3; ++ps) {
                        const uint32_t ah = ps == 2 ? 32768u : 0u, bh = ps == 1 ? 16384u : 0u;
                        for (int ks = 0; ks < 8; ++ks)
                            tc::mma_f16(tmem + kColO1 + 64 * b, tc::sdesc(sb + kSs + ah + ks * 4096, 2048, 128),
                                        tc::sdesc(sb + kQs + bh + ks * 2048, 1024, 128), id, (ps | ks) ? 1u : 0u);
                    }
                    tc::mma_commit(bars + kMmaO1);
                }
                if (c + 1 < nch) {   // Q and W of the next chunk as soon as O1 (the last reader) retires
                    if (!(ok = wait(kMmaO1, pc))) break;
                    load_q(c + 1); load_w(c + 1);
                }
                ok = wait(kDReady, pc) && wait(kLdK, pc) && wait(kLdP, pc);
                if (!ok) break;
                got_kp = c + 1;
                tc::fence_after_sync();
                {   // S += D'^T K (3 passes, K = 64);  O2[b] = D^T P^T (3 passes, K = 64)
                    constexpr uint32_t idk = tc::idesc_f16(128, 128, 0, 1, 0);
                    for (int ps = 0; ps < 3; ++ps) {
                        const uint32_t ah = ps == 2 ? 16384u : 0u, bh = ps == 1 ? 16384u : 0u;
                        for (int ks = 0; ks < 4; ++ks)
                            tc::mma_f16(tmem + kColS, tc::sdesc(sb + kDs + 32768 + ah + ks * 4096, 2048, 128),
                                        tc::sdesc(sb + kKs + bh + ks * 256, 128, 1024), idk, 1u);
                    }
                    tc::mma_commit(bars + kMmaS);
                    constexpr uint32_t idp = tc::idesc_f16(128, 64, 0, 0, 0);
                    for (int ps = 0; ps < 3; ++ps) {
                        const uint32_t ah = ps == 2 ? 16384u : 0u, bh = ps == 1 ? 8192u : 0u;
                        for (int ks = 0; ks < 4; ++ks)
                            tc::mma_f16(tmem + kColO2 + 64 * b, tc::sdesc(sb + kDs + ah + ks * 4096, 2048, 128),
                                        tc::sdesc(sb + kPs + bh + ks * 2048, 1024, 128), idp, (ps | ks) ? 1u : 0u);
                    }
                    tc::mma_commit(bars + (b ? kMmaO2b : kMmaO2a));
                }
                if (c + 1 < nch) {   // K and P of the next chunk, each as soon as its buffer is free
                    if (!(ok = wait(kMmaS, pc))) break;
                    load_k(c + 1);
                    if (!(ok = wait(b ? kMmaO2b : kMmaO2a, pb))) break;
                    load_p(c + 1);
                }
            }
            if (!ok) {
                // error path: let every issued MMA retire and every issued copy land
                // before the CTA releases its tensor and shared memory
                tc::mma_commit(bars + kDrain);
                tc::mbar_wait(bars + kDrain, 0, kWaitLimit);
                if (req_qw > got_qw) {
                    tc::mbar_wait(bars + kLdQ, (req_qw - 1) & 1, kWaitLimit);
                    tc::mbar_wait(bars + kLdW, (req_qw - 1) & 1, kWaitLimit);
                }
                if (req_k > got_kp) tc::mbar_wait(bars + kLdK, (req_k - 1) & 1, kWaitLimit);
                // E copies: wait for the last one issued into each buffer (its parity)
                if (req_e[0]) tc::mbar_wait(bars + kLdEa, ((req_e[0] - 1) >> 1) & 1, kWaitLimit);
                if (req_e[1]) tc::mbar_wait(bars + kLdEb, ((req_e[1] - 1) >> 1) & 1, kWaitLimit);
                if (req_p > got_kp) tc::mbar_wait(bars + kLdP, (req_p - 1) & 1, kWaitLimit);
            }
        }
    } else if (warp < kConvWarps) {
        // ================= converters: thread = v-row j (lane quarter) x column half
        const int chalf = warp >> 2;
        bool ok = true;
        for (int c = 0; c < nch && ok; ++c) {
            const uint32_t pc = c & 1;
            const uint8_t* vr = vrec(c);
            // this chunk's U^T entries (used after the S conversion)
            float4 u4[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
                u4[q] = __ldg(reinterpret_cast<const float4*>(vr + pf::kRecU) + (8 * chalf + q) * kD + row);
            const float4* el4 = reinterpret_cast<const float4*>(vr + pf::kRecElast) + 8 * chalf;
            asm volatile("prefetch.global.L1 [%0];" ::"l"(el4));   // its 32 decay factors: one 128-byte line
            const float eg_last = __ldg(reinterpret_cast<const float*>(vr + pf::kRecEgam) + 63);
            if (c + 1 < nch) {   // the next chunk's U and decay vectors toward L2
                const uint8_t* vn = vrec(c + 1);
                tc::bulk_prefetch_l2(vn + pf::kRecU + tid * 128, 128);
                if (tid < 4) tc::bulk_prefetch_l2(vn + pf::kRecEgam + tid * 128, 128);
            }
            if (c > 0 && !(ok = wait(kMmaS, (c - 1) & 1))) break;
            tc::fence_after_sync();
            // S -> fp16 hi/lo operand; S <- e^{Gam_last} S   (this thread: row j, 64 columns)
            {
                float v[16];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int col = 64 * chalf + 16 * cc;
                    tc::tmem_ld16(tl + kColS + col, v);
#pragma unroll
                    for (int g8 = 0; g8 < 2; ++g8) {
                        uint4 hi, lo;
                        tc::split8(v + 8 * g8, hi, lo);
                        const uint32_t o = tc::cl_off(row, col + 8 * g8, 128);
                        *reinterpret_cast<uint4*>(sm + kSs + o) = hi;
                        *reinterpret_cast<uint4*>(sm + kSs + 32768 + o) = lo;
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] *= eg_last;
                    tc::tmem_st16(tl + kColS + col, v);
                }
                tc::tmem_wait_st();
            }
            tc::fence_proxy_async();
            tc::fence_before_sync();
            tc::mbar_arrive(bars + kSReady);
            if (!(ok = wait(kMmaD, pc))) break;
            if (c > 0 && !(ok = wait((c - 1) & 1 ? kMmaO2b : kMmaO2a, ((c - 1) >> 1) & 1))) break;
            tc::fence_after_sync();
            // D^T = U^T - Dacc ; D'^T = D^T diag(e^{Gam_last - Gam_t}) -> fp16 hi/lo operands
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float v[16];
                tc::tmem_ld16(tl + kColD + 32 * chalf + 16 * hh, v);
#pragma unroll
                for (int g8l = 0; g8l < 2; ++g8l) {
                    const int g8 = 2 * hh + g8l;
                    float d[8], dp[8];
                    const float4 ua = u4[2 * g8], ub = u4[2 * g8 + 1], ea = __ldg(el4 + 2 * g8), eb = __ldg(el4 + 2 * g8 + 1);
                    const float uu[8] = {ua.x, ua.y, ua.z, ua.w, ub.x, ub.y, ub.z, ub.w};
                    const float ee[8] = {ea.x, ea.y, ea.z, ea.w, eb.x, eb.y, eb.z, eb.w};
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        d[i] = uu[i] - v[8 * g8l + i];
                        dp[i] = d[i] * ee[i];
                    }
                    uint4 hi, lo;
                    const uint32_t o = tc::cl_off(row, 32 * chalf + 8 * g8, 128);
                    tc::split8(d, hi, lo);
                    *reinterpret_cast<uint4*>(sm + kDs + o) = hi;
                    *reinterpret_cast<uint4*>(sm + kDs + 16384 + o) = lo;
                    tc::split8(dp, hi, lo);
                    *reinterpret_cast<uint4*>(sm + kDs + 32768 + o) = hi;
                    *reinterpret_cast<uint4*>(sm + kDs + 49152 + o) = lo;
                }
            }
            tc::fence_proxy_async();
            tc::fence_before_sync();
            tc::mbar_arrive(bars + kDReady);
        }
        // final state out (after the last update)
        if (ok && nch > 0) ok = wait(kMmaS, (nch - 1) & 1);
        tc::fence_after_sync();
        if (ok) {
            float v[32];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int col = 2 * chalf + cc;
                tc::tmem_ld32(tl + kColS + 32 * col, v);
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    *reinterpret_cast<float4*>(Sg + row * kD + 32 * col + i) =
                        make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                    if (p.flags & kFlagCheckFinite)
                        bad |= nonfinite_bits(v[i]) | nonfinite_bits(v[i + 1]) | nonfinite_bits(v[i + 2]) |
                               nonfinite_bits(v[i + 3]);
                }
            }
        }
    } else {
        // ================= epilogue: thread = v-row j, the 64 tokens of a chunk in blocks of 16
        const int eq = warp - kConvWarps;   // lane quarter
        const int j = eq * 32 + lane;
        const uint32_t te = tmem + (static_cast<uint32_t>(eq * 32) << 16);
        float* Rs = reinterpret_cast<float*>(sm + kRs);
        const float wj = p.norm_w[j];
        const unsigned short* __restrict__ zj = static_cast<const unsigned short*>(p.z) + h * kD + j;
        Tout* __restrict__ outj = static_cast<Tout*>(p.out) + h * kD + j;
        float* __restrict__ prej = p.prenorm ? p.prenorm + h * kD + j : nullptr;
        const bool check = (p.flags & kFlagCheckFinite) != 0;
        // z of tokens [t, t + 16) of column j as raw bf16 bits (0 past the chunk)
        auto load_z = [&](uint32_t (&zr)[16], size_t row0, int nrem) {
#pragma unroll
            for (int i = 0; i < 16; ++i) zr[i] = i < nrem ? __ldg(zj + (row0 + i) * HvD) : 0u;
        };
        bool ok = true;
        for (int c = 0; c < nch && ok; ++c) {
            const uint32_t b = c & 1;
            const int c0 = c * kChunk, n = min(kChunk, L - c0);
            const size_t row0 = static_cast<size_t>(t0 + c0);
            if (c + 1 < nch) {   // next chunk's z rows toward L2: one 128-byte half row per thread
                const int t = tid - kConvThreads;   // 0..127
                if (t < 2 * min(kChunk, L - c0 - kChunk))
                    tc::bulk_prefetch_l2(static_cast<const __nv_bfloat16*>(p.z) + (row0 + kChunk + (t >> 1)) * HvD + h * kD +
                                             64 * (t & 1), 128);
            }
            uint32_t zc[16];
            load_z(zc, row0, n);
            if (!(ok = wait(b ? kMmaO2b : kMmaO2a, (c >> 1) & 1) && wait(b ? kLdEb : kLdEa, (c >> 1) & 1))) break;
            tc::fence_after_sync();
            const float* eg = reinterpret_cast<const float*>(sm + kEs + 256 * b);
            // pass 1: o = (e^Gam O1 + O2)/sqrt(128) back into the O1 buffer, norm_w silu(z) into
            // the O2 buffer, per-token partial sums of o^2 over this warp's 32 rows
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
                uint32_t zn[16];
                if (q < 3) load_z(zn, row0 + 16 * (q + 1), n - 16 * (q + 1));
                float v1[16], v2[16];
                const uint32_t c1 = kColO1 + 64 * b + 16 * q, c2 = kColO2 + 64 * b + 16 * q;
                tc::tmem_ld16(te + c1, v1);
                tc::tmem_ld16(te + c2, v2);
#pragma unroll
                for (int i = 0; i < 16; i += 4) {
                    const float4 e = *reinterpret_cast<const float4*>(eg + 16 * q + i);
                    const float ee[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        v1[i + k] = fmaf(ee[k], v1[i + k], v2[i + k]) * kInvSqrtD;
                        v2[i + k] = wj * pf::silu_fast(__uint_as_float(zc[i + k] << 16));
                    }
                }
                tc::tmem_st16(te + c1, v1);
                tc::tmem_st16(te + c2, v2);
#pragma unroll
                for (int i = 0; i < 16; ++i) v1[i] *= v1[i];
                const float ssum = reduce16_transposed(v1);
                if (lane < 16) Rs[(b * 4 + eq) * 64 + 16 * q + lane] = ssum;
#pragma unroll
                for (int i = 0; i < 16; ++i) zc[i] = zn[i];
            }
            tc::tmem_wait_st();
            tc::mbar_arrive(bars + kRsReady);
            if (!(ok = wait(kRsReady, c & 1))) break;
            // 1/sqrt(mean o^2 + eps) of tokens lane and 32 + lane
            const float* rb = Rs + b * 256;
            const float rs_a = rsqrtf(((rb[lane] + rb[64 + lane]) + (rb[128 + lane] + rb[192 + lane])) * (1.0f / kD) + p.eps);
            const float rs_b = rsqrtf(((rb[32 + lane] + rb[96 + lane]) + (rb[160 + lane] + rb[224 + lane])) * (1.0f / kD) + p.eps);
            // pass 2: y = o * rs * norm_w silu(z)
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
                float v1[16], v2[16];
                tc::tmem_ld16(te + kColO1 + 64 * b + 16 * q, v1);
                tc::tmem_ld16(te + kColO2 + 64 * b + 16 * q, v2);
                const float rsq = q < 2 ? rs_a : rs_b;
                Tout* oq = outj + (row0 + 16 * q) * HvD;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float rs = __shfl_sync(0xffffffffu, rsq, (16 * q + i) & 31);
                    const float y = v1[i] * rs * v2[i];
                    if (16 * q + i < n) {
                        st_out(oq + static_cast<size_t>(i) * HvD, y);
                        if (check) bad |= nonfinite_bits(y);
                        if (prej) prej[(row0 + 16 * q + i) * HvD] = v1[i];
                    }
                }
            }
            tc::fence_before_sync();
            tc::mbar_arrive(bars + (b ? kEpiB : kEpiA));
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (p.dev_status) {
        int st = 0;
        if (p.flags & kFlagCheckFinite) st = __any_sync(0xffffffffu, bad) ? (warp < kConvWarps ? 1 : 2) : 0;
        if (tid == 0 && *err_s) st |= 16;
        if (lane == 0 && st) atomicOr(p.dev_status + s * Hv + h, st);
    }
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

template <typename Tout>
cudaError_t launch_state_pass_t(const PrefillParams& p, cudaStream_t stream) {
    auto k = state_pass_kernel<Tout>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kStateSmem));
    if (e != cudaSuccess) return e;
    k<<<static_cast<unsigned>(p.n_seq) * p.Hv, kStateThreads, kStateSmem, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_state_pass(const PrefillParams& p, int out_dtype, cudaStream_t stream) {
    return out_dtype == 1 ? launch_state_pass_t<__nv_bfloat16>(p, stream) : launch_state_pass_t<float>(p, stream);
}

}  // namespace gdn
