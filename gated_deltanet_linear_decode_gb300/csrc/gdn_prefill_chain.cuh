// gdn_prefill_chain.cuh -- the chain role of the tensor-core prefill kernel:
// the chunk-to-chunk state recurrence and the layer output (xwen CLAUDE.md page,
// "Ground truth": chunk = 64 form; "Architecture cheat sheet", "Gated DeltaNet
// layer": o = S q / sqrt(128), gated RMSNorm y = o / sqrt(mean(o^2) + eps)
// * norm_w * silu(z)).  Every state-independent quantity of a chunk comes from
// the records of the preparation role, each read once its ready flag is set
// (and dropped from L2 once consumed).
//
// One CTA runs one (sequence, v-head) chain at a time; the fp32 state lives in tensor memory
// (lane j = v-row j), and so do its fp16 hi/lo parts and those of D, which the
// MMAs read as their A operand straight from tensor memory (only W^T, Q', K'
// and P come from shared memory, whose bandwidth bounds these MMAs).  Per chunk,
// with every product transposed so the MMA runs at M = 128:
//   Dacc = S W^T        (S hi x W^T hi, one MMA pass)
//   O    = S Q'^T       (Q' = diag(e^Gam) Q; three passes: hi.hi + hi.lo + lo.hi)
//   D^T  = U^T - Dacc
//   S    = e^{Gam_last} S + D^T K'   (K' = diag(e^{Gam_last - Gam}) K; three passes)
//   O   += D^T P^T      (three passes)
//   o_t  = O[:, t] / sqrt(128)  -> gated RMSNorm -> out
// Warp roles, meeting at mbarriers (the epilogue warps among themselves at a
// named barrier):
//   warps 0-7   convert: S -> fp16 hi/lo (and the decay of S), Dacc -> D hi/lo;
//               after each D conversion, the outputs of v-rows 64-127 of the
//               previous chunk from the staged O
//   warps 8-11  epilogue: O -> shared memory (row j per thread; double-buffered),
//               the per-token RMS factors, then token-major o -> gated RMSNorm ->
//               out for v-rows 0-63, a thread owning one token (z and out move in
//               16-byte pieces); up to two chunks behind (O is double-buffered in
//               tensor memory; z is staged by cp.async)
//   warp 12     control: one lane issues the MMAs
//   warp 13     copies: one lane waits for each record's ready flag and issues its
//               bulk copies as soon as the MMAs that read the buffer have retired,
//               then drops the consumed record from L2 and counts the chunk consumed
// Every wait has an iteration (or, for the ready flags, a time) limit; a
// timeout sets dev_status bit 4 and the abort flag that releases the
// preparation role's records-in-flight gate.
#pragma once

#include <type_traits>

#include "gdn_internal.h"
#include "gdn_prefill_tc.cuh"

namespace gdn {
namespace chain {

constexpr int kConvWarps = 8, kEpiWarps = 4;
constexpr int kCtrlWarp = kConvWarps + kEpiWarps;   // MMA issue
constexpr int kCopyWarp = kCtrlWarp + 1;            // bulk copies of the records
constexpr int kStateThreads = (kConvWarps + kEpiWarps + 2) * 32;
constexpr int kConvThreads = kConvWarps * 32, kEpiThreads = kEpiWarps * 32;
// The chain role's barrier: its 14 warps (named barrier 5; the CTA may hold idle warps too).
__device__ __forceinline__ void chain_sync() { asm volatile("bar.sync 5, %0;" ::"n"(kStateThreads) : "memory"); }

// shared memory map (bytes)
constexpr uint32_t kQs = 0;           // Q' hi +0, lo +16384       (64 t x 128 i, canonical 64 rows)
constexpr uint32_t kKs = 32768;       // K' hi +0, lo +16384       (64 t x 128 i, canonical 64 rows)
constexpr uint32_t kWs = 65536;       // W^T hi                   (128 i x 64 t, canonical 128 rows)
constexpr uint32_t kPs = 81920;       // P hi +0, lo +8192         (64 t x 64 r, canonical 64 rows)
constexpr int kOStride = 68;          // floats per v-row of the staged O (64 tokens + 4: no bank conflicts)
constexpr uint32_t kOstBytes = 128 * kOStride * 4;
constexpr uint32_t kOst = 98304;      // O of chunks c & 1 = 0, 1: fp32 [2][128 j][kOStride], staged for the outputs
constexpr uint32_t kRs = kOst + 2 * kOstBytes;   // per-token partial sums of O^2 [2][64] fp32
constexpr uint32_t kRS = kRs + 512;   // per-token norm factor of chunks c & 1 = 0, 1: [2][64] fp32
constexpr uint32_t kNw = kRS + 512;   // norm_w [128] fp32
constexpr uint32_t kBar = kNw + 512;  // mbarriers, then the TMEM base and the error flag
constexpr uint32_t kUs = (kBar + 176 + 127) / 128 * 128;   // the chunk's U, e^Gam, e^{Gam_last-Gam} (record tail)
constexpr uint32_t kUBytes = pf::kVRec - pf::kRecU;          // 33280
constexpr uint32_t kStateSmem = kUs + kUBytes;
static_assert(kStateSmem <= 232448, "shared memory of the chain role exceeds 227 KB");

// mbarrier slots
enum : int {
    kLdW = 0, kLdQ, kLdK, kLdP, kLdU,  // record copies landed (transaction count)
    kMmaD, kMmaO1, kMmaS,              // Dacc / first O group / state update retired (tcgen05.commit)
    kODone0, kODone1,                  // O of even / odd chunks complete
    kSReady, kDReady,                  // converters wrote the S / D operands (256 arrivals)
    kEpi0, kEpi1,                      // epilogue done with the O buffer of even / odd chunks (128 arrivals)
    kOutRdy0, kOutRdy1,                // staged O and norm factors of even / odd chunks ready (128 arrivals)
    kOutFree0, kOutFree1,              // converters done with the staged O of even / odd chunks (256 arrivals)
    kDrain,                            // error path: every MMA issued so far retired
    kNever,                            // test stall: nothing arrives
    kNumBars
};

// tensor-memory columns: S fp32, S hi / lo (fp16 pairs), Dacc fp32, D hi / lo
// (fp16 pairs, K = 64 t), O (two buffers of 64)
constexpr uint32_t kColS = 0, kColShi = 128, kColSlo = 192, kColD = 256, kColDhi = 320, kColDlo = 352, kColO = 384;
constexpr uint32_t kTmemCols = 512;
constexpr int kWaitLimit = 1 << 24;
constexpr uint64_t kReadyTimeoutNs = 2000000000ull;   // 2 s for a record to appear

// One chain: sequence s, v-head h, on the CTA's kStateThreads threads, with
// the CTA's tensor memory (kTmemCols columns at tmem).  Returns with every
// MMA retired, every copy landed and every thread past a CTA-wide barrier, so
// the next chain may reuse the barriers, shared and tensor memory.
template <typename Tout>
__device__ void run(const PrefillParams& p, int s, int h, uint8_t* sm, uint32_t tmem) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int Hv = p.Hv, HvD = Hv * kD;
    // this launch's chunks of sequence s: [cb, ce) of its own; the state comes in and goes out
    // through S (a launch that starts the sequence takes zeros instead under zero_init)
    const int cbase_s = p.chunk_base[s], nch_s = p.chunk_base[s + 1] - cbase_s;
    const int cb = max(0, p.chunk_lo - cbase_s), ce = min(nch_s, p.chunk_hi - cbase_s);
    // the state plane of (s, h): fp32, or bf16 under kFlagStateBf16 (read into fp32, rounded once when stored)
    const bool sbf = (p.flags & kFlagStateBf16) != 0;
    const int ss = sbf ? 2 : 4;
    uint8_t* Sg = static_cast<uint8_t*>(p.S) + (static_cast<size_t>(s) * Hv + h) * kD * kD * ss;
    if (cb >= ce) {
        // an empty sequence ends with its initial state: zeros under zero_init (written by the first launch)
        if (nch_s == 0 && p.zero_init && p.chunk_lo == 0)
            for (int e = tid; e < kD * kD * ss / 16; e += kStateThreads) reinterpret_cast<uint4*>(Sg)[e] = make_uint4(0, 0, 0, 0);
        return;
    }
    const bool zero_init = p.zero_init && cb == 0;
    const int cbase = cbase_s + cb, nch = ce - cb;
    const int t0 = p.cu_seqlens[s] + kChunk * cb;
    const int L = min(p.cu_seqlens[s + 1] - t0, kChunk * nch);

    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBar);
    static_assert(8 * kNumBars + 8 <= 176, "mbarrier area");
    volatile int* err_s = reinterpret_cast<volatile int*>(sm + kBar + 8 * kNumBars + 4);
    const uint32_t sb = tc::smem_u32(sm);
    const int kh = h % p.Hk;

    chain_sync();   // the previous chain of this CTA is done with every barrier
    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i) {
            uint32_t cnt = 1;
            if (i == kSReady || i == kDReady) cnt = kConvThreads;
            if (i == kEpi0 || i == kEpi1 || i == kOutRdy0 || i == kOutRdy1) cnt = kEpiThreads;
            if (i == kOutFree0 || i == kOutFree1) cnt = kConvThreads;
            asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(tc::smem_u32(bars + i)) : "memory");
            tc::mbar_init(bars + i, cnt);
        }
        *err_s = 0;
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tc::fence_before_sync();
    chain_sync();
    tc::fence_after_sync();

    // Bounded wait that also gives up as soon as another role has timed out.
    // Converter and epilogue warps back off with short sleeps (at most 64 ns) so
    // that waiting warps leave the issue slots to the working ones; the control
    // and copy lanes poll.
    const bool sleepy = warp != kCtrlWarp && warp != kCopyWarp;
    const uint32_t sleep_cap = 64u;
    auto wait = [&](int bar, uint32_t parity) -> bool {
        uint32_t ns = 32;
        for (int it = 0; it < kWaitLimit; it += 8) {
            if (tc::mbar_wait(bars + bar, parity, 8)) return true;
            if (*err_s) return false;
            if (sleepy) {
                __nanosleep(ns);
                ns = min(ns * 2, sleep_cap);
            }
        }
        *err_s = 1;
        return false;
    };

    const uint8_t* vrec0 = p.ws_v + (static_cast<size_t>(cbase) * Hv + h) * pf::kVRec;
    auto vrec = [&](int c) { return vrec0 + static_cast<size_t>(c) * Hv * pf::kVRec; };
    // Acquire the ready flag of chunk c's records (set by the preparation role once
    // they are written); bounded in time, and given up as soon as another role has.
    const int* ready = p.ready + static_cast<size_t>(cbase) * Hv + h;
    auto wait_ready = [&](int c) -> bool {
        const int* f = ready + static_cast<size_t>(c) * Hv;
        if (pf::ld_acquire(f)) return true;
        const uint64_t tstart = pf::global_ns();
        uint32_t ns = 64;
        for (;;) {
            if (pf::ld_acquire(f)) return true;
            if (*err_s) return false;
            if (pf::global_ns() - tstart > kReadyTimeoutNs) {
                *err_s = 1;
                return false;
            }
            __nanosleep(ns);
            ns = min(ns * 2, 2048u);
        }
    };

    // Gated RMSNorm outputs of chunk cc for token tt_ and v-rows v0 .. v0 + 8 NG - 1, from
    // the chunk's staged O and norm factor (buffers cc & 1).  zq holds the matching z (16
    // bytes per group of 8, from load_z).  The epilogue warps write v-rows 0-63 of every
    // chunk, the converter warps v-rows 64-127 (one chunk later, in their idle time).
    const float* nw_s = reinterpret_cast<const float*>(sm + kNw);
    const __nv_bfloat16* zbase = static_cast<const __nv_bfloat16*>(p.z) + h * kD;
    auto load_z = [&](int cc, int tt_, int v0, auto ngc, uint4* zq) {
        constexpr int NG = decltype(ngc)::value;
        const bool valid = cc < nch && cc * kChunk + tt_ < L;
        const uint4* src = reinterpret_cast<const uint4*>(zbase + static_cast<size_t>(t0 + cc * kChunk + tt_) * HvD + v0);
#pragma unroll
        for (int g = 0; g < NG; ++g) zq[g] = valid ? __ldg(src + g) : make_uint4(0, 0, 0, 0);
    };
    auto outputs = [&](int cc, int tt_, int v0, auto ngc, const uint4* zq, bool& bad_out) {
        constexpr int NG = decltype(ngc)::value;
        if (cc * kChunk + tt_ >= L) return;
        const size_t rowt = static_cast<size_t>(t0 + cc * kChunk + tt_);
        const float rs = reinterpret_cast<const float*>(sm + kRS)[(cc & 1) * 64 + tt_];
        const float* oc = reinterpret_cast<const float*>(sm + kOst + (cc & 1) * kOstBytes) + tt_;
        Tout* op = static_cast<Tout*>(p.out) + rowt * HvD + h * kD + v0;
        float* pp = p.prenorm ? p.prenorm + rowt * HvD + h * kD + v0 : nullptr;
        const bool check = (p.flags & kFlagCheckFinite) != 0;
#pragma unroll
        for (int g = 0; g < NG; ++g) {
            float zf[8], o[8], y[8];
            pf::bf16x8_to_f32(zq[g], zf);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                o[i] = oc[(v0 + 8 * g + i) * kOStride];
                y[i] = o[i] * rs * nw_s[v0 + 8 * g + i] * pf::silu_fast(zf[i]);
                if (check) bad_out |= nonfinite_bits(y[i]);
            }
            pf::st_out8(op + 8 * g, y);
            if (pp)
#pragma unroll
                for (int i = 0; i < 8; i += 4)
                    *reinterpret_cast<float4*>(pp + 8 * g + i) = make_float4(
                        o[i] * kInvSqrtD, o[i + 1] * kInvSqrtD, o[i + 2] * kInvSqrtD, o[i + 3] * kInvSqrtD);
        }
    };
    using G2 = std::integral_constant<int, 2>;
    using G4 = std::integral_constant<int, 4>;
    bool bad_out = false;   // a non-finite output (GDN_FLAG_CHECK_FINITE)

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
                const uint8_t* src = Sg + (row * kD + 32 * c + i) * ss;
                const float4 f = zero_init ? make_float4(0.f, 0.f, 0.f, 0.f)
                                           : (sbf ? StateIO<__nv_bfloat16>::ld(src) : StateIO<float>::ld(src));
                v[i] = f.x; v[i + 1] = f.y; v[i + 2] = f.z; v[i + 3] = f.w;
            }
            tc::tmem_st32(tl + kColS + 32 * c, v);
        }
        tc::tmem_wait_st();
    }
    // test hook: a wait that nothing ends, so every role takes its give-up path at once
    if (tid == 0 && (p.flags & kFlagTestStall) && !tc::mbar_wait(bars + kNever, 0, 1 << 12)) *err_s = 1;
    tc::fence_before_sync();
    chain_sync();
    tc::fence_after_sync();

    bool bad = false;
    if (warp == kCtrlWarp) {
        // ================= control: the MMAs
        if (lane == 0 && nch > 0) {
            bool ok = true;
            for (int c = 0; c < nch && ok; ++c) {
                const uint32_t pc = c & 1, b = c & 1;
                if (!(ok = wait(kSReady, pc) && wait(kLdW, pc))) break;
                tc::fence_after_sync();
                {   // Dacc = S W^T (1 pass, K = 128; A = S hi from tensor memory)
                    constexpr uint32_t id = tc::idesc_f16(128, 64, 0, 1, 0);
                    for (int ks = 0; ks < 8; ++ks)
                        tc::mma_f16_ts(tmem + kColD, tmem + kColShi + 8 * ks, tc::sdesc(sb + kWs + ks * 256, 128, 2048), id,
                                       ks ? 1u : 0u);
                    tc::mma_commit(bars + kMmaD);
                }
                if (!(ok = (c < 2 || wait(kEpi0 + b, ((c - 2) >> 1) & 1)) && wait(kLdQ, pc))) break;
                tc::fence_after_sync();
                {   // O[b] = S Q'^T (3 passes, K = 128)
                    constexpr uint32_t id = tc::idesc_f16(128, 64, 0, 0, 0);
                    for (int ps = 0; ps < 3; ++ps) {
                        const uint32_t ac = ps == 2 ? kColSlo : kColShi, bh = ps == 1 ? 16384u : 0u;
                        for (int ks = 0; ks < 8; ++ks)
                            tc::mma_f16_ts(tmem + kColO + 64 * b, tmem + ac + 8 * ks,
                                           tc::sdesc(sb + kQs + bh + ks * 2048, 1024, 128), id, (ps | ks) ? 1u : 0u);
                    }
                    tc::mma_commit(bars + kMmaO1);
                }
                if (!(ok = wait(kDReady, pc) && wait(kLdK, pc))) break;
                tc::fence_after_sync();
                {   // S += D^T K' (3 passes, K = 64);  O[b] += D^T P^T (3 passes, K = 64); A = D from tensor memory
                    constexpr uint32_t idk = tc::idesc_f16(128, 128, 0, 1, 0);
                    for (int ps = 0; ps < 3; ++ps) {
                        const uint32_t ac = ps == 2 ? kColDlo : kColDhi, bh = ps == 1 ? 16384u : 0u;
                        for (int ks = 0; ks < 4; ++ks)
                            tc::mma_f16_ts(tmem + kColS, tmem + ac + 8 * ks, tc::sdesc(sb + kKs + bh + ks * 256, 128, 1024),
                                           idk, 1u);
                    }
                    tc::mma_commit(bars + kMmaS);
                    if (!(ok = wait(kLdP, pc))) break;   // P is read only by the O update
                    constexpr uint32_t idp = tc::idesc_f16(128, 64, 0, 0, 0);
                    for (int ps = 0; ps < 3; ++ps) {
                        const uint32_t ac = ps == 2 ? kColDlo : kColDhi, bh = ps == 1 ? 8192u : 0u;
                        for (int ks = 0; ks < 4; ++ks)
                            tc::mma_f16_ts(tmem + kColO + 64 * b, tmem + ac + 8 * ks,
                                           tc::sdesc(sb + kPs + bh + ks * 2048, 1024, 128), idp, 1u);
                    }
                    tc::mma_commit(bars + kODone0 + b);
                }
            }
            if (!ok) {   // error path: let every issued MMA retire before the CTA releases its memory
                tc::mma_commit(bars + kDrain);
                tc::mbar_wait(bars + kDrain, 0, kWaitLimit);
            }
        }
    } else if (warp == kCopyWarp) {
        // ================= copies: the records of chunk c + 1 as soon as its ready flag is
        // set and chunk c's MMAs have freed the buffers; lane 0 issues, the whole warp drops
        // each consumed record from L2.  Lane 0 decides; the warp follows through shuffles.
        auto discard = [&](int c) {   // whole warp: record c is consumed
            const uint8_t* r = vrec(c);
            for (uint32_t o = 128u * lane; o < pf::kVRec; o += 128u * 32) pf::discard_l2(r + o);
        };
        int req_w = 0, req_q = 0, req_k = 0, req_p = 0, req_u = 0;   // chunks requested per barrier (an error path drains them)
        auto load = [&](int bar, uint32_t dst, int c, uint32_t off, uint32_t bytes, int& req) {
            tc::mbar_expect_tx(bars + bar, bytes);
            tc::bulk_g2s(sm + dst, vrec(c) + off, bytes, bars + bar);
            req = c + 1;
        };
        bool ok = true;
        if (lane == 0 && nch > 0) {
            if ((ok = wait_ready(0))) {
                pf::fence_proxy_async_global();
                load(kLdW, kWs, 0, pf::kRecW, 16384, req_w);
                load(kLdQ, kQs, 0, pf::kRecQhi, 32768, req_q);
                load(kLdK, kKs, 0, pf::kRecKhi, 32768, req_k);
                load(kLdP, kPs, 0, pf::kRecPhi, 16384, req_p);
                load(kLdU, kUs, 0, pf::kRecU, kUBytes, req_u);
            }
        }
        for (int c = 0; c + 1 < nch; ++c) {
            if (lane == 0 && ok) {
                const uint32_t pc = c & 1, b = c & 1, pb = (c >> 1) & 1;
                do {
                    if (!(ok = wait_ready(c + 1))) break;
                    pf::fence_proxy_async_global();
                    if (!(ok = wait(kMmaD, pc))) break;         // W^T read by Dacc; U read by the converters
                    load(kLdW, kWs, c + 1, pf::kRecW, 16384, req_w);
                    load(kLdU, kUs, c + 1, pf::kRecU, kUBytes, req_u);
                    if (!(ok = wait(kMmaO1, pc))) break;        // Q' read by the first O group
                    load(kLdQ, kQs, c + 1, pf::kRecQhi, 32768, req_q);
                    if (!(ok = wait(kMmaS, pc))) break;         // K' read by the state update (U by then too)
                    load(kLdK, kKs, c + 1, pf::kRecKhi, 32768, req_k);
                    if (!(ok = wait(kODone0 + b, pb))) break;   // P read by the O update
                    load(kLdP, kPs, c + 1, pf::kRecPhi, 16384, req_p);
                } while (false);
            }
            if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
            discard(c);
            if (lane == 0) pf::red_release_add(p.consumed + static_cast<size_t>(cbase + c) * p.Hk + kh, 1);   // done with chunk c
        }
        if (lane == 0 && ok && nch > 0) ok = wait(kODone0 + ((nch - 1) & 1), ((nch - 1) >> 1) & 1);
        if (__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) && nch > 0) {
            discard(nch - 1);
            if (lane == 0) pf::red_release_add(p.consumed + static_cast<size_t>(cbase + nch - 1) * p.Hk + kh, 1);
        }
        if (lane == 0 && !ok) {   // error path: let every issued copy land before the CTA moves on
            if (req_w) tc::mbar_wait(bars + kLdW, (req_w - 1) & 1, kWaitLimit);
            if (req_q) tc::mbar_wait(bars + kLdQ, (req_q - 1) & 1, kWaitLimit);
            if (req_k) tc::mbar_wait(bars + kLdK, (req_k - 1) & 1, kWaitLimit);
            if (req_p) tc::mbar_wait(bars + kLdP, (req_p - 1) & 1, kWaitLimit);
            if (req_u) tc::mbar_wait(bars + kLdU, (req_u - 1) & 1, kWaitLimit);
        }
    } else if (warp < kConvWarps) {
        // ================= converters: thread = v-row j (lane quarter) x column half; after
        // each D conversion, the outputs of the previous chunk's v-rows 64-127 (thread =
        // token tid % 64, v-rows 64 + 16 (tid / 64) ..)
        const int chalf = warp >> 2;
        const int ot = tid & 63, ov = 64 + 16 * (tid >> 6);
        uint4 zq[2];
        // outputs of chunk cc (its O and norm factors staged by the epilogue warps), then the
        // staged O buffer is handed back
        auto outputs_prev = [&](int cc) -> bool {
            if (!wait(kOutRdy0 + (cc & 1), (cc >> 1) & 1)) return false;
            outputs(cc, ot, ov, G2{}, zq, bad_out);
            tc::mbar_arrive(bars + kOutFree0 + (cc & 1));
            return true;
        };
        bool ok = true;
        for (int c = 0; c < nch && ok; ++c) {
            const uint32_t pc = c & 1;
            if (c > 0) load_z(c - 1, ot, ov, G2{}, zq);   // used after this chunk's D conversion
            // this chunk's U^T entries (used after the S conversion) and e^{Gam_last}, copied
            // into shared memory with the chunk's tiles (the buffer is refilled once every
            // converter has passed the S conversion, i.e. after Dacc is issued)
            if (!(ok = wait(kLdU, pc))) break;
            float4 u4[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) u4[q] = reinterpret_cast<const float4*>(sm + kUs)[(8 * chalf + q) * kD + row];
            const float eg_last = reinterpret_cast<const float*>(sm + kUs + (pf::kRecEgam - pf::kRecU))[63];
            if (c > 0 && !(ok = wait(kMmaS, (c - 1) & 1))) break;
            tc::fence_after_sync();
            // S -> fp16 hi/lo pairs in tensor memory; S <- e^{Gam_last} S   (this thread: row j, 64 columns)
            {
                float v[16];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int col = 64 * chalf + 16 * cc;
                    tc::tmem_ld16(tl + kColS + col, v);
                    uint32_t hi[8], lo[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) tc::split2(v[2 * k], v[2 * k + 1], hi[k], lo[k]);
                    tc::tmem_st8(tl + kColShi + col / 2, hi);
                    tc::tmem_st8(tl + kColSlo + col / 2, lo);
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] *= eg_last;
                    tc::tmem_st16(tl + kColS + col, v);
                }
                tc::tmem_wait_st();
            }
            tc::fence_before_sync();
            tc::mbar_arrive(bars + kSReady);
            if (!(ok = wait(kMmaD, pc))) break;
            if (c > 0 && !(ok = wait(kODone0 + ((c - 1) & 1), ((c - 1) >> 1) & 1))) break;   // D read by O(c-1)
            tc::fence_after_sync();
            // D^T = U^T - Dacc -> fp16 hi/lo pairs in tensor memory (this thread: row j, tokens 32 chalf ..)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float v[16];
                tc::tmem_ld16(tl + kColD + 32 * chalf + 16 * hh, v);
                uint32_t hi[8], lo[8];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 u = u4[4 * hh + q];
                    tc::split2(u.x - v[4 * q], u.y - v[4 * q + 1], hi[2 * q], lo[2 * q]);
                    tc::split2(u.z - v[4 * q + 2], u.w - v[4 * q + 3], hi[2 * q + 1], lo[2 * q + 1]);
                }
                tc::tmem_st8(tl + kColDhi + 16 * chalf + 8 * hh, hi);
                tc::tmem_st8(tl + kColDlo + 16 * chalf + 8 * hh, lo);
            }
            tc::tmem_wait_st();
            tc::fence_before_sync();
            tc::mbar_arrive(bars + kDReady);
            if (c > 0 && !(ok = outputs_prev(c - 1))) break;
        }
        if (ok && nch > 0) {   // the last chunk's outputs
            load_z(nch - 1, ot, ov, G2{}, zq);
            ok = outputs_prev(nch - 1);
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
                    uint8_t* dst = Sg + (row * kD + 32 * col + i) * ss;
                    const float4 f = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                    if (sbf)
                        StateIO<__nv_bfloat16>::st(reinterpret_cast<__nv_bfloat16*>(dst), f);
                    else
                        StateIO<float>::st(reinterpret_cast<float*>(dst), f);
                    if (p.flags & kFlagCheckFinite)
                        bad |= nonfinite_bits(v[i]) | nonfinite_bits(v[i + 1]) | nonfinite_bits(v[i + 2]) |
                               nonfinite_bits(v[i + 3]);
                }
            }
        }
    } else {   // warps kConvWarps .. kConvWarps + kEpiWarps - 1
        // ================= epilogue: per chunk, O row j -> staged O (shared memory, buffer
        // c & 1; the tensor-memory O buffer is then free), the per-token norm factors, and
        // the outputs of v-rows 0-63 (thread = token tt, v-rows 32 jh ..); the converters
        // write v-rows 64-127 from the same staged O
        const int eq = warp - kConvWarps;   // lane quarter
        const int j = eq * 32 + lane, e = tid - kConvThreads;
        const int tt = e & 63, jh = e >> 6;
        const uint32_t te = tmem + (static_cast<uint32_t>(eq * 32) << 16);
        float* Rs = reinterpret_cast<float*>(sm + kRs);
        float* RS = reinterpret_cast<float*>(sm + kRS);
        reinterpret_cast<float*>(sm + kNw)[e] = p.norm_w[e];
        // The 128 epilogue threads meet at named barrier 2 (no sleeping waits on the
        // output path).  The waits that can give up are followed by a vote at that
        // barrier, so every epilogue thread takes the same decision and none is left
        // waiting at a later barrier.
        auto epi_sync = [&]() { asm volatile("bar.sync 2, %0;" ::"n"(kEpiThreads) : "memory"); };
        auto epi_all = [&](bool good) -> bool {   // barrier + "every thread passed good"
            uint32_t any_bad;
            asm volatile(
                "{\n\t.reg .pred p, q;\n\tsetp.eq.u32 p, %1, 0;\n\tbar.red.or.pred q, 2, %2, p;\n\t"
                "selp.u32 %0, 1, 0, q;\n\t}"
                : "=r"(any_bad)
                : "r"(good ? 1u : 0u), "n"(kEpiThreads)
                : "memory");
            return any_bad == 0;
        };
        epi_sync();   // norm_w staged
        bool ok = true;
        uint4 zq[4];
        for (int c = 0; c < nch && ok; ++c) {
            const uint32_t b = c & 1;   // O buffers (tensor memory and staged)
            load_z(c, tt, 32 * jh, G4{}, zq);
            // O of chunk c complete, and the converters done with the staged O of chunk c - 2
            const bool got = wait(kODone0 + b, (c >> 1) & 1) && (c < 2 || wait(kOutFree0 + b, ((c - 2) >> 1) & 1));
            if (!(ok = epi_all(got))) break;
            tc::fence_after_sync();
            float* Ost = reinterpret_cast<float*>(sm + kOst + b * kOstBytes);
            {   // O row j (64 tokens) -> registers -> shared memory; the O buffer is then free
                float v[32];
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    tc::tmem_ld32(te + kColO + 64 * b + 32 * hf, v);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        *reinterpret_cast<float4*>(Ost + j * kOStride + 32 * hf + 4 * q) =
                            make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                }
            }
            tc::fence_before_sync();
            tc::mbar_arrive(bars + kEpi0 + b);
            epi_sync();   // O staged
            // token-major: partial sum of O^2 over v-rows 64 jh .. of token tt
            const float* oc = Ost + 64 * jh * kOStride + tt;
            float ss = 0.f;
#pragma unroll 16
            for (int r = 0; r < 64; ++r) ss = fmaf(oc[r * kOStride], oc[r * kOStride], ss);
            Rs[jh * 64 + tt] = ss;
            epi_sync();   // partial sums written
            // o = O / sqrt(128); y = o / sqrt(mean(o^2) + eps) * norm_w * silu(z): the factor
            // 1 / sqrt(mean(o^2) + eps) / sqrt(128) of token tt, for both output halves
            if (jh == 0) RS[b * 64 + tt] = rsqrtf((Rs[tt] + Rs[64 + tt]) * (kInvSqrtD * kInvSqrtD / kD) + p.eps) * kInvSqrtD;
            epi_sync();   // norm factors written; Rs may be reused by the next chunk
            tc::mbar_arrive(bars + kOutRdy0 + b);   // the converters may read the staged O and RS
            outputs(c, tt, 32 * jh, G4{}, zq, bad_out);
        }
    }

    tc::fence_before_sync();
    chain_sync();
    if (tid == 0 && *err_s) atomicExch(p.abort_flag, 1);   // no preparation CTA waits on this chain any more
    if (p.dev_status) {
        int st = 0;
        if (p.flags & kFlagCheckFinite)
            st = (__any_sync(0xffffffffu, bad) ? 1 : 0) | (__any_sync(0xffffffffu, bad_out) ? 2 : 0);
        if (tid == 0 && *err_s) st |= 16;
        if (lane == 0 && st) atomicOr(p.dev_status + s * Hv + h, st);
    }
    tc::fence_after_sync();
}

}  // namespace chain
}  // namespace gdn
