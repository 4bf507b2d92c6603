// gdn_recurrent_stream.cu -- persistent, TMA-streamed form of the recurrent
// gated DeltaNet step (decode step and speculative-verify walk) for large
// batches, where the fp32 state (64 KiB per (sequence, v-head)) is the whole
// cost and the kernel must keep HBM busy.
//
// Method: xwen CLAUDE.md page, "Architecture cheat sheet (Qwen 3.6, ggml-org
// GGUF)", "Gated DeltaNet layer" (recurrent step), and its "Drafting" section
// (per-position state planes for verify rollback).
//
// One CTA per SM loops over work items (sequence b, q/k head kh, v-head m of
// the group): items of one (b, kh) group are consecutive, and a group never
// leaves its CTA, so the in-place conv-state update has a single writer.  For
// every item a bulk asynchronous copy (cp.async.bulk, completion counted on an
// mbarrier) lands the head's 128 x 128 state tile and its inputs -- the raw
// rows of its q/k/v channels, z, conv taps -- in one of two shared-memory
// stages, two items ahead of the compute.  A producer warp issues the copies
// (issuing a bulk copy takes the issuing thread about as long as the copy
// engine needs for it, so it is kept off the compute warps).  On arrival the
// state goes to registers (warp w owns rows 16w..16w+15, lane = 4 consecutive
// columns) and the small inputs to a private area, and the stage is handed
// back to the producer at once.
//
// S.k and S.q of a warp's 16 rows (32 partial sums per lane) are reduced with
// one transposed butterfly (31 shuffles).  Decode and verify share this code,
// so verify checkpoints equal decode replays bit for bit.
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_tc.cuh"

namespace gdn {

namespace {

constexpr int kSThreads = 256;     // a compute group: 8 warps x 16 rows
constexpr int kLaunchThreads = kSThreads + 32;   // one compute group and the producer warp
constexpr int kWaitLimit = 1 << 22;   // polls of one stage wait before it gives up
constexpr int kStallLimit = 1 << 12;  // polls of the test stall (a barrier nothing arrives on)

// Bounded wait on phase `parity` of `mbar` that also gives up as soon as
// *abort is set (another warp gave up).
__device__ __forceinline__ bool stage_wait(uint64_t* mbar, uint32_t parity, volatile int* abort) {
    for (int it = 0; it < kWaitLimit; it += 16) {
        if (tc::mbar_wait(mbar, parity, 16)) return true;
        if (*abort) return false;
    }
    return false;
}

__device__ __forceinline__ float conv4(float4 w, float x0, float x1, float x2, float cur) {
    return fmaf(w.w, cur, fmaf(w.z, x2, fmaf(w.y, x1, w.x * x0)));
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint64_t* mbar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(tc::smem_u32(mbar))
                 : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(tc::smem_u32(mbar)), "r"(bytes)
                 : "memory");
}

// Byte layout of one stage (es = activation element size, ss = state element
// size): the state tile first, then the small inputs.
struct StageLayout {
    // conv taps (q|k|v), raw rows [K+3][q|k|v], z rows [K]; then, with ssm_alpha / ssm_beta
    // folded in (H > 0), the hidden rows [K][H], W_a[h] and W_b[h] (bf16)
    uint32_t cw, xr, zr, ab, bytes;
    __host__ __device__ StageLayout(int K, int es, int ss, int H) {
        cw = kD * kD * ss;
        xr = cw + 384 * 16;
        zr = xr + (K + 3) * 384 * es;
        ab = (zr + K * 128 * es + 15) & ~15u;
        bytes = H > 0 ? ab + (K + 2) * H * 2 : ab;
    }
};

// With a bf16 state the tile stays in its shared-memory stage while it is updated (read
// there for S.k, S.q and again for the update) instead of moving to registers: the kernel
// then fits 96 registers, and two CTAs per SM keep two tiles' latency chains in flight
// (2 x 9 warps leave 5 warps on some of the SM's four sub-partitions, whose 16,384
// registers allow 96 a thread).  The stage goes back to the producer once the item is done.
// An fp32 tile does not fit twice per SM that way, so the fp32 decode step (one token, no
// folded projections) runs two compute groups of 8 warps in one CTA instead, each holding
// one tile in a shared-memory stage, with three stages (the third one loading).
constexpr int kMaxRegsSmemState = 96;

// Stages of a CTA: two, or three for two compute groups where they fit (one loading while
// both groups update theirs).
__host__ __device__ constexpr int stage_count(int groups, bool third) { return groups > 1 && third ? 3 : 2; }

// Per-compute-group scratch after the stages (floats): q_hat|k_hat [K][256], v [K][128],
// o [128], norm partials [16], RMS partials [8], gates [K][2], folded a/b partials [K][8][2].
__host__ __device__ inline int group_scratch_floats(int K) { return (K * (256 + 128 + 2 + 16) + 152 + 3) & ~3; }

// Shared-memory bytes: the stages, the copy of the small inputs (when the tile goes to
// registers and its stage is handed back at once), norm_w, each group's scratch, barriers
// ("full" per stage and compute group, "empty" per stage, the test-stall barrier).
__host__ __device__ inline size_t stream_smem_bytes(const StageLayout& L, int K, int groups, int stages, bool copy_inputs) {
    const size_t cur = copy_inputs ? ((L.ab - L.cw + 15) & ~static_cast<size_t>(15)) : 0;
    return static_cast<size_t>(stages) * L.bytes + cur +
           4 * (128 + static_cast<size_t>(groups) * group_scratch_floats(K)) + ((groups + 1) * stages + 1) * 8 + 16;
}

template <typename Tact, typename Tout, typename Ts, bool kSmemState, int kGroups, int kStg>
__device__ __forceinline__ void recurrent_stream_body(const RecParams& p) {
    extern __shared__ __align__(128) uint8_t sm[];
    constexpr int es = sizeof(Tact), ss = sizeof(Ts);
    constexpr int kProducer = kGroups * kSThreads / 32;   // the producer warp
    static_assert(kSmemState || kGroups == 1, "two compute groups hold their tiles in shared memory");
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // compute group cg (warps 8cg .. 8cg+7) and the thread's place in it
    const int cg = kGroups > 1 ? (warp < kProducer ? tid / kSThreads : 0) : 0;
    const int ctid = tid - cg * kSThreads, cwarp = ctid >> 5;
    const int K = p.K, C = p.C, HvD = p.Hv * kD;
    const int r = p.Hv / p.Hk;
    const int n_groups = p.B * p.Hk;
    const int H = p.ab_hidden ? p.ab_H : 0;
    const StageLayout L(K, es, ss, H);
    // a private copy of the current item's small inputs (register form only), after the stages
    uint8_t* cur = sm + kStg * L.bytes;
    const uint32_t cur_bytes = L.ab - L.cw;
    float* nw_s = reinterpret_cast<float*>(cur + (kSmemState ? 0u : ((cur_bytes + 15) & ~15u)));   // [128]
    float* qk_s = nw_s + 128 + cg * group_scratch_floats(K);                      // [K][256] q_hat | k_hat
    float* v_s = qk_s + K * 256;                                                   // [K][128]
    float* o_s = v_s + K * 128;                                                    // [128]
    float* red = o_s + 128;                                                        // [2][8]
    float* part = red + 16;                                                        // [8]
    float* gates = part + 8;                                                       // [K][2]
    float* abp = gates + 2 * K;                               // [K][8 warps][2] folded a/b partial sums
    // full[s * kGroups + g]: stage s landed with an item of compute group g.  Each group waits
    // only on its own barriers, so it sees every phase of them in order (a group that skipped
    // the other group's fills of a shared stage could not tell one phase from the next but one).
    uint64_t* full = reinterpret_cast<uint64_t*>(nw_s + 128 + kGroups * group_scratch_floats(K));
    uint64_t* empty = full + kStg * kGroups;                                       // stage s handed back
    uint64_t* never = empty + kStg;                                                // test stall: no arrivals
    volatile int* abort_s = reinterpret_cast<volatile int*>(never + 1);            // a wait gave up
    // the compute group's barrier (named barrier 1 + cg, its 256 threads only)
    auto group_sync = [&]() { asm volatile("bar.sync %0, %1;" ::"r"(1 + cg), "n"(kSThreads) : "memory"); };
    auto group_sync_any = [&](int v) {   // the same, returning whether any thread of the group passed v != 0
        uint32_t res;
        asm volatile(
            "{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\tbar.red.or.pred q, %2, %3, p;\n\t"
            "selp.u32 %0, 1, 0, q;\n\t}"
            : "=r"(res)
            : "r"(v), "r"(1 + cg), "n"(kSThreads)
            : "memory");
        return res != 0;
    };

    if (tid == 0) {
        for (int st = 0; st < kStg; ++st) {
            for (int gg = 0; gg < kGroups; ++gg) tc::mbar_init(&full[st * kGroups + gg], 1);
            tc::mbar_init(&empty[st], 1);
        }
        tc::mbar_init(never, 1);
        *abort_s = 0;
    }
    // launched as a programmatic dependent: nothing global is touched before the previous
    // kernel in the stream is done (it may have written the state, the conv state or the inputs)
    grid_dependency_wait();
    if (tid < kD) nw_s[tid] = p.norm_w[tid];
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();
    grid_launch_dependents();

    // item i of this CTA -> (group, m); the items of a (sequence, q/k head) group are
    // consecutive, and compute group cg takes the CTA's groups cg, cg + kGroups, ...
    const int G = gridDim.x;
    const int my_groups = blockIdx.x < n_groups ? (n_groups - 1 - blockIdx.x) / G + 1 : 0;
    const int n_items = my_groups * r;
    auto item_group = [&](int i) { return blockIdx.x + (i / r) * G; };

    auto issue = [&](int i) {      // one thread: load item i into stage i % kStg
        const int g = item_group(i), m = i % r;
        const int b = g / p.Hk, kh = g % p.Hk, h = kh + m * p.Hk;
        uint64_t* mb = &full[(i % kStg) * kGroups + (i / r) % kGroups];
        const uint32_t base = tc::smem_u32(sm + (i % kStg) * L.bytes);
        const uint32_t seg = 128 * es;   // one head's channels of one row
        mbar_expect_tx(mb, L.bytes);
        const Ts* Sh = rec_state_in<Ts>(p, b) + static_cast<size_t>(h) * kD * kD;
        for (int q = 0; q < 4; ++q) bulk_g2s(base + q * 4096 * ss, Sh + q * 4096, 4096 * ss, mb);
        bulk_g2s(base + L.cw, p.conv_w + 4 * (kh * kD), 128 * 16, mb);
        bulk_g2s(base + L.cw + 128 * 16, p.conv_w + 4 * (p.Hk * kD + kh * kD), 128 * 16, mb);
        bulk_g2s(base + L.cw + 256 * 16, p.conv_w + 4 * (2 * p.Hk * kD + h * kD), 128 * 16, mb);
        const Tact* cin = static_cast<const Tact*>(p.conv_in) + static_cast<size_t>(b) * 3 * C;
        const Tact* xin = static_cast<const Tact*>(p.x) + static_cast<size_t>(b) * K * C;
        for (int rr = 0; rr < K + 3; ++rr) {
            const Tact* src = rr < 3 ? cin + rr * C : xin + static_cast<size_t>(rr - 3) * C;
            const uint32_t d = base + L.xr + rr * 3 * seg;
            bulk_g2s(d, src + kh * kD, seg, mb);
            bulk_g2s(d + seg, src + p.Hk * kD + kh * kD, seg, mb);
            bulk_g2s(d + 2 * seg, src + 2 * p.Hk * kD + h * kD, seg, mb);
        }
        const Tact* zin = static_cast<const Tact*>(p.z) + static_cast<size_t>(b) * K * HvD + h * kD;
        for (int t = 0; t < K; ++t) bulk_g2s(base + L.zr + t * seg, zin + static_cast<size_t>(t) * HvD, seg, mb);
        if (H > 0) {   // the folded projections' operands
            const uint32_t rb = static_cast<uint32_t>(H) * 2;
            const __nv_bfloat16* hid = static_cast<const __nv_bfloat16*>(p.ab_hidden) + static_cast<size_t>(b) * K * H;
            for (int t = 0; t < K; ++t) bulk_g2s(base + L.ab + t * rb, hid + static_cast<size_t>(t) * H, rb, mb);
            bulk_g2s(base + L.ab + K * rb, static_cast<const __nv_bfloat16*>(p.W_a) + static_cast<size_t>(h) * H, rb, mb);
            bulk_g2s(base + L.ab + (K + 1) * rb, static_cast<const __nv_bfloat16*>(p.W_b) + static_cast<size_t>(h) * H,
                     rb, mb);
        }
    };

    // Bit 4 of dev_status marks every (sequence, v-head) of item i0 and the compute group's
    // later items: a wait gave up, so their states and outputs were not (fully) written.
    auto report_from = [&](int i0) {
        if (!p.dev_status) return;
        int k = 0;
        for (int i = i0; i < n_items; ++i) {
            if ((i / r) % kGroups != cg) continue;
            if (k++ % kSThreads != ctid) continue;
            const int g = item_group(i);
            atomicOr(p.dev_status + (g / p.Hk) * p.Hv + g % p.Hk + (i % r) * p.Hk, 16);
        }
    };

    if (warp == kProducer) {
        // ================= producer: item i into stage i % kStg once item i - kStg has left it.
        // On a wait that gives up it issues nothing more, and it returns only once
        // every copy it issued has landed (none may land in a released CTA).
        if (lane == 0) {
            int issued = 0;
            bool ok = true;
            uint32_t fills = 0;      // parity of the fills of each full barrier so far (bit s * kGroups + g)
            uint32_t last_par = 0;   // parity of the fill of the last item issued into each stage (bit s)
            if (p.flags & kFlagTestStall) ok = tc::mbar_wait(never, 0, kStallLimit);   // never completes
            for (int i = 0; i < n_items && ok; ++i) {
                const int st = i % kStg, fb = st * kGroups + (i / r) % kGroups;
                if (i >= kStg && !(ok = stage_wait(&empty[st], ((i / kStg) - 1) & 1, abort_s))) break;
                issue(i);
                last_par = (last_par & ~(1u << st)) | (((fills >> fb) & 1u) << st);
                fills ^= 1u << fb;
                issued = i + 1;
            }
            if (!ok) {
                *abort_s = 1;
                for (int i = max(0, issued - kStg); i < issued; ++i) {
                    const int st = i % kStg;
                    tc::mbar_wait(&full[st * kGroups + (i / r) % kGroups], (last_par >> st) & 1u, kWaitLimit);
                }
            }
        }
        return;
    }

    float4 sreg[kSmemState ? 1 : 16];
    bool go_on = true;
    uint32_t phase = 0;   // parity of the next fill of full[s * kGroups + cg] this group waits for (bit s)
    for (int j = cg; j < my_groups && go_on; j += kGroups) {
      for (int m = 0; m < r; ++m) {
        const int i = j * r + m;
        const int g = item_group(i);
        const int b = g / p.Hk, kh = g % p.Hk, h = kh + m * p.Hk;
        const uint8_t* stg = sm + (i % kStg) * L.bytes;
        // gates for the item's tokens: plain loads, issued before the wait
        float a_raw = 0.f, b_raw = 0.f;
        if (ctid < K && !p.ab_hidden) {
            const size_t gi = (static_cast<size_t>(b) * K + ctid) * p.Hv + h;
            a_raw = ld_act(static_cast<const Tact*>(p.a_raw) + gi);
            b_raw = ld_act(static_cast<const Tact*>(p.b_raw) + gi);
        }
        const float a_dt = p.dt_bias[h], a_ssm = p.ssm_a[h];
        const int st = i % kStg;
        const bool landed = stage_wait(&full[st * kGroups + cg], (phase >> st) & 1u, abort_s);
        phase ^= 1u << st;
        // state rows -> registers (or left in the stage); small inputs -> private area (or read
        // in the stage, which the item then holds)
        uint8_t* const srow = const_cast<uint8_t*>(stg) + ((cwarp * 16) * kD + 4 * lane) * ss;   // my rows in the stage
        if constexpr (!kSmemState) {
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) sreg[rr] = StateIO<Ts>::ld(srow + rr * kD * ss);
            for (uint32_t e = ctid * 16; e < cur_bytes; e += kSThreads * 16)
                *reinterpret_cast<uint4*>(cur + e) = *reinterpret_cast<const uint4*>(stg + L.cw + e);
        }
        const uint8_t* in = kSmemState ? stg + L.cw : cur;
        if (ctid < K && !H) {
            gates[2 * ctid] = sigmoidf_(b_raw);
            gates[2 * ctid + 1] = a_ssm * softplusf_(a_raw + a_dt);
        }
        if (H > 0) {
            // ssm_alpha / ssm_beta folded in: each compute thread's share of the dot products of
            // the token's hidden row with W_a[h], W_b[h] (all in the stage), summed over warps below
            const __nv_bfloat16* sab = reinterpret_cast<const __nv_bfloat16*>(stg + L.ab);
            for (int t = 0; t < K; ++t) {
                const float2 pr = ab_dot_part<false>(sab + t * H, sab + K * H, sab + (K + 1) * H, H, ctid, kSThreads);
                const float sa = warp_sum(pr.x), sb = warp_sum(pr.y);
                if (lane == 0) {
                    abp[(t * 8 + cwarp) * 2] = sa;
                    abp[(t * 8 + cwarp) * 2 + 1] = sb;
                }
            }
        }
        // one decision for the group's warps, before anything is written: stop at the
        // first item whose stage did not land (what was read from it is discarded)
        if (group_sync_any(!landed)) {
            *abort_s = 1;
            report_from(i);
            go_on = false;
            break;
        }
        if (!kSmemState && ctid == 0) tc::mbar_arrive(&empty[i % kStg]);   // the stage may be refilled
        if (H > 0 && ctid < K) {
            // the folded a_raw, b_raw: the warps' partial sums (the next barrier orders them
            // before step 7)
            float sa = 0.f, sb = 0.f;
#pragma unroll
            for (int w8 = 0; w8 < 8; ++w8) {
                sa += abp[(ctid * 8 + w8) * 2];
                sb += abp[(ctid * 8 + w8) * 2 + 1];
            }
            gates[2 * ctid] = sigmoidf_(sb);
            gates[2 * ctid + 1] = a_ssm * softplusf_(sa + a_dt);
        }

        const float4* cw = reinterpret_cast<const float4*>(in);                       // [384] taps
        const Tact* xr = reinterpret_cast<const Tact*>(in + (L.xr - L.cw));            // [K+3][384]
        const Tact* zr = reinterpret_cast<const Tact*>(in + (L.zr - L.cw));            // [K][128]
        // ---- steps 1-4 for every token of the item: thread c < 256 owns q/k channel c, c < 128 v channel c.
        // q_hat and k_hat belong to the group: the group's first head computes them, the others reuse them.
        if (m > 0) {
            if (ctid < kD) {
                const float4 wv = cw[256 + ctid];
                for (int t = 0; t < K; ++t)
                    v_s[t * kD + ctid] =
                        siluf_(conv4(wv, to_f(xr[t * 384 + 256 + ctid]), to_f(xr[(t + 1) * 384 + 256 + ctid]),
                                     to_f(xr[(t + 2) * 384 + 256 + ctid]), to_f(xr[(t + 3) * 384 + 256 + ctid])));
            }
            group_sync();
        } else {
            const float4 w = cw[ctid];
            const float4 wv = ctid < kD ? cw[256 + ctid] : make_float4(0, 0, 0, 0);
            for (int t = 0; t < K; ++t) {
                const float val = siluf_(conv4(w, to_f(xr[t * 384 + ctid]), to_f(xr[(t + 1) * 384 + ctid]),
                                               to_f(xr[(t + 2) * 384 + ctid]), to_f(xr[(t + 3) * 384 + ctid])));
                const float sq = warp_sum(val * val);
                if (lane == 0) red[(cwarp >> 2) * 8 + (cwarp & 3)] = sq;
                if (ctid < kD)
                    v_s[t * kD + ctid] =
                        siluf_(conv4(wv, to_f(xr[t * 384 + 256 + ctid]), to_f(xr[(t + 1) * 384 + 256 + ctid]),
                                     to_f(xr[(t + 2) * 384 + 256 + ctid]), to_f(xr[(t + 3) * 384 + 256 + ctid])));
                group_sync();
                const float* rd = red + (cwarp >> 2) * 8;
                const float nrm = sqrtf((rd[0] + rd[1]) + (rd[2] + rd[3]));
                qk_s[t * 256 + ctid] = val / fmaxf(nrm, p.eps);
                group_sync();
            }
        }

        int* const status = (p.dev_status && (p.flags & kFlagCheckFinite)) ? p.dev_status + b * p.Hv + h : nullptr;
        for (int t = 0; t < K; ++t) {
            // ---- step 7 on my 16 rows
            const float4 qq = *reinterpret_cast<const float4*>(&qk_s[t * 256 + 4 * lane]);
            const float4 kk = *reinterpret_cast<const float4*>(&qk_s[t * 256 + 128 + 4 * lane]);
            const float kq = warp_sum(fmaf(kk.w, qq.w, fmaf(kk.z, qq.z, fmaf(kk.y, qq.y, kk.x * qq.x))));
            const float beta = gates[2 * t];
            const float eg = expf(gates[2 * t + 1]);
            Ts* Sout = rec_state_out<Ts>(p, b, t) + (static_cast<size_t>(h) * kD + cwarp * 16) * kD;
            // partial S.k and S.q of my 16 rows: slot 2rr = row rr . k, slot 2rr+1 = row rr . q
            float pv[32];
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) {
                const float4 sv = kSmemState ? StateIO<Ts>::ld(srow + rr * kD * ss) : sreg[rr];
                pv[2 * rr] = fmaf(sv.w, kk.w, fmaf(sv.z, kk.z, fmaf(sv.y, kk.y, sv.x * kk.x)));
                pv[2 * rr + 1] = fmaf(sv.w, qq.w, fmaf(sv.z, qq.z, fmaf(sv.y, qq.y, sv.x * qq.x)));
            }
            const float full_sum = reduce32_transposed(pv);   // lane 2rr: (S k)_rr, lane 2rr+1: (S q)_rr
            const int my_row = lane >> 1;
            // d = (v - e^g S.k) beta in the even lane; the odd lane forms o from it
            const float d_even = (v_s[t * kD + cwarp * 16 + my_row] - eg * full_sum) * beta;
            const float d_pair = __shfl_xor_sync(0xffffffffu, d_even, 1);
            const float o = fmaf(d_pair, kq, eg * full_sum) * kInvSqrtD;   // meaningful in odd lanes
            const float o_mine = (lane & 1) ? o : 0.f;
            const float ps = warp_sum(o_mine * o_mine);
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) {
                const float d = __shfl_sync(0xffffffffu, d_even, 2 * rr);
                const float4 sv = kSmemState ? StateIO<Ts>::ld(srow + rr * kD * ss) : sreg[rr];
                float4 nv;
                nv.x = fmaf(d, kk.x, eg * sv.x);
                nv.y = fmaf(d, kk.y, eg * sv.y);
                nv.z = fmaf(d, kk.z, eg * sv.z);
                nv.w = fmaf(d, kk.w, eg * sv.w);
                nv = StateIO<Ts>::round(nv);   // the next token continues from what a later call reads
                if constexpr (kSmemState) {
                    if (t + 1 < K) StateIO<Ts>::st_shared(srow + rr * kD * ss, nv);
                } else {
                    sreg[rr] = nv;
                }
                StateIO<Ts>::st(Sout + rr * kD + 4 * lane, nv);
                if (status && (nonfinite_bits(nv.x) | nonfinite_bits(nv.y) | nonfinite_bits(nv.z) | nonfinite_bits(nv.w)))
                    atomicOr(status, 1);
            }
            if (lane & 1) o_s[cwarp * 16 + my_row] = o;
            if (lane == 0) part[cwarp] = ps;
            group_sync();
            // ---- step 8: gated RMSNorm, thread c < 128 -> output j = c
            const size_t row = static_cast<size_t>(b) * K + t;
            if (ctid < kD) {
                float tot = 0.f;
#pragma unroll
                for (int w = 0; w < 8; ++w) tot += part[w];
                const float rs = 1.0f / sqrtf(tot * (1.0f / kD) + p.eps);
                const float ov = o_s[ctid];
                const float y = ov * rs * nw_s[ctid] * siluf_(to_f(zr[t * kD + ctid]));
                const size_t oi = row * HvD + h * kD + ctid;
                st_out(static_cast<Tout*>(p.out) + oi, y);
                if (p.prenorm) p.prenorm[oi] = ov;
                if (status && nonfinite_bits(y)) atomicOr(status, 2);
            }
            // ---- conv state after token t: rows t+1, t+2, t+3 of the raw window (bit-exact).
            // q/k channels are written by the group's last head only (every head of the
            // group has its inputs staged before that head runs).
            Tact* cout = static_cast<Tact*>(p.conv_out) + static_cast<size_t>(b) * p.conv_out_b +
                         static_cast<size_t>(t) * p.conv_out_p;
            if (ctid < kD) {
                const int cv = 2 * p.Hk * kD + h * kD + ctid;
#pragma unroll
                for (int q = 0; q < 3; ++q) cout[q * C + cv] = xr[(t + 1 + q) * 384 + 256 + ctid];
            }
            if (m == r - 1) {
                const int ch = ctid < kD ? kh * kD + ctid : p.Hk * kD + kh * kD + (ctid - kD);
#pragma unroll
                for (int q = 0; q < 3; ++q) cout[q * C + ch] = xr[(t + 1 + q) * 384 + ctid];
            }
            group_sync();
        }
        if constexpr (kSmemState) {
            // the item is done with its stage: hand it back (the generic writes of the state
            // above are ordered before the producer's next bulk copy into it)
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            group_sync();
            if (ctid == 0) tc::mbar_arrive(&empty[i % kStg]);
        }
      }
    }
}

template <typename Tact, typename Tout>
__global__ void __launch_bounds__(kLaunchThreads, 1) recurrent_stream_kernel(const RecParams p) {
    recurrent_stream_body<Tact, Tout, float, false, 1, 2>(p);
}
template <typename Tout>
__global__ void __maxnreg__(kMaxRegsSmemState) recurrent_stream_bf16s_kernel(const RecParams p) {
    recurrent_stream_body<__nv_bfloat16, Tout, __nv_bfloat16, true, 1, 2>(p);
}
// fp32 state, two compute groups of 8 warps and the producer warp (17 warps: 96 registers)
constexpr int kLaunchThreads2 = 2 * kSThreads + 32;
template <typename Tact, typename Tout, int kStg>
__global__ void __maxnreg__(kMaxRegsSmemState) recurrent_stream_2g_kernel(const RecParams p) {
    recurrent_stream_body<Tact, Tout, float, true, 2, kStg>(p);
}

}  // namespace

// Shared memory of the form launch_recurrent_stream falls back to (one compute group): what
// the caller checks against the device's limit before choosing the streaming kernel.
size_t recurrent_stream_smem(int K, int act_dtype, bool state_bf16, int ab_H) {
    const int es = act_dtype == 1 ? 2 : 4;
    const StageLayout L(K, es, state_bf16 ? 2 : 4, ab_H);
    return stream_smem_bytes(L, K, 1, 2, !state_bf16);
}

cudaError_t launch_recurrent_stream(const RecParams& p, int act_dtype, int out_dtype, int grid, cudaStream_t stream) {
    const bool sbf = (p.flags & kFlagStateBf16) != 0;
    const int es = act_dtype == 1 ? 2 : 4;
    const int H = p.ab_hidden ? p.ab_H : 0;
    const StageLayout L(p.K, es, sbf ? 2 : 4, H);
    int dev = 0, optin = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
    // an fp32 state without folded projections: two compute groups, with three stages where
    // they fit (the decode step), else two (the verify walk)
    const size_t smem3 = stream_smem_bytes(L, p.K, 2, 3, false), smem22 = stream_smem_bytes(L, p.K, 2, 2, false);
    const bool two_groups = !sbf && H == 0 && smem22 <= static_cast<size_t>(optin);
    const bool third = smem3 <= static_cast<size_t>(optin);
    const size_t smem = two_groups ? (third ? smem3 : smem22) : stream_smem_bytes(L, p.K, 1, 2, !sbf);
    auto go = [&](auto kernel, int threads) {
        cudaError_t r = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (r != cudaSuccess) return r;
        int per_sm = 1;
        if (sbf) {   // as many CTAs per SM as fit (the bf16-state kernel is built for two)
            r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem);
            if (r != cudaSuccess) return r;
            per_sm = per_sm < 1 ? 1 : (per_sm > 2 ? 2 : per_sm);
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(grid * per_sm));
        cfg.blockDim = dim3(static_cast<unsigned>(threads));
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see grid_dependency_wait
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kernel, p);
    };
    using bf = __nv_bfloat16;
    if (sbf)   // bf16 activations only (checked by the API)
        return out_dtype == 1 ? go(recurrent_stream_bf16s_kernel<bf>, kLaunchThreads)
                              : go(recurrent_stream_bf16s_kernel<float>, kLaunchThreads);
    if (two_groups && third) {
        if (act_dtype == 1)
            return out_dtype == 1 ? go(recurrent_stream_2g_kernel<bf, bf, 3>, kLaunchThreads2)
                                  : go(recurrent_stream_2g_kernel<bf, float, 3>, kLaunchThreads2);
        return out_dtype == 1 ? go(recurrent_stream_2g_kernel<float, bf, 3>, kLaunchThreads2)
                              : go(recurrent_stream_2g_kernel<float, float, 3>, kLaunchThreads2);
    }
    if (two_groups) {
        if (act_dtype == 1)
            return out_dtype == 1 ? go(recurrent_stream_2g_kernel<bf, bf, 2>, kLaunchThreads2)
                                  : go(recurrent_stream_2g_kernel<bf, float, 2>, kLaunchThreads2);
        return out_dtype == 1 ? go(recurrent_stream_2g_kernel<float, bf, 2>, kLaunchThreads2)
                              : go(recurrent_stream_2g_kernel<float, float, 2>, kLaunchThreads2);
    }
    if (act_dtype == 1)
        return out_dtype == 1 ? go(recurrent_stream_kernel<bf, bf>, kLaunchThreads)
                              : go(recurrent_stream_kernel<bf, float>, kLaunchThreads);
    return out_dtype == 1 ? go(recurrent_stream_kernel<float, bf>, kLaunchThreads)
                          : go(recurrent_stream_kernel<float, float>, kLaunchThreads);
}

}  // namespace gdn
