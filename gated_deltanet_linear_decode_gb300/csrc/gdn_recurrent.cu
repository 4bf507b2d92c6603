// gdn_recurrent.cu -- recurrent form of the gated DeltaNet layer on sm_103a:
// the decode step (one token per sequence, state updated in place) and the
// speculative-verify walk (K tokens per sequence, a state checkpoint after
// every position), plus the commit copy and the conv-state initialiser.
//
// Method: xwen CLAUDE.md page, "Architecture cheat sheet (Qwen 3.6, ggml-org
// GGUF)", "Gated DeltaNet layer": conv1d(k=4) -> SiLU -> split -> clamp L2 ->
// tiled heads -> gates -> S = S e^g; d = (v - S.k) beta; S += k (x) d;
// o = S.q / sqrt(128) -> gated RMSNorm.  Verify checkpoints: the page's
// "Drafting" section (per-position state planes for rollback).
//
// Work decomposition.  The state of one v-head is 128 rows x 128 fp32 (64
// KiB); every row j is independent given k_hat, q_hat, beta, g and v_j, and
// the only coupling between rows is the RMSNorm over the head's 128 outputs.
// All v-heads that share q/k head kh (h = kh + m*H_k) form a "group"; one
// thread-block CLUSTER handles one (sequence, group): CTA `rank` owns RPC rows
// of v-head m = rank / (128/RPC).  Each CTA
//   * issues its 128-bit state loads first (HBM-bound stream, one read and one
//     write per state byte),
//   * recomputes conv/SiLU/L2 for the 256 q/k channels of kh (L2-resident
//     after the first CTA) and conv/SiLU of its own RPC v channels,
//   * updates its rows in registers (lane = 4 consecutive columns, warp = 8
//     rows; S.k and S.q by warp shuffle),
//   * exchanges per-CTA partial sums of o^2 through distributed shared
//     memory to normalise each head, and writes y.
// The cluster barrier also orders the in-place conv-state update: the q/k
// channels of kh are read by every CTA of the cluster and rewritten only by
// rank 0 after the barrier; v channels are owned by exactly one CTA.
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {

namespace {

// conv over a 3-row window plus the current token: tap 3 * current + tap 2 *
// previous + tap 1 * two back + tap 0 * three back.  One fixed FMA order so
// every kernel that uses it rounds identically.
__device__ __forceinline__ float conv4(float4 w, float x0, float x1, float x2, float cur) {
    return fmaf(w.w, cur, fmaf(w.z, x2, fmaf(w.y, x1, w.x * x0)));
}

#ifndef GDN_REC_MIN_BLOCKS
#define GDN_REC_MIN_BLOCKS 8   // 8 CTAs of 128 threads per SM (64 registers)
#endif

template <typename Tact, typename Tout, typename Ts, int RPC>
__global__ void __launch_bounds__(RPC * 4, (GDN_REC_MIN_BLOCKS * 32 / RPC) > 0 ? (GDN_REC_MIN_BLOCKS * 32 / RPC) : 1)
recurrent_kernel(const RecParams p) {
    constexpr int NT = RPC * 4;      // threads
    constexpr int NW = NT / 32;      // warps, 8 rows each
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rank = static_cast<int>(cluster_ctarank());
    const int grp = blockIdx.x / p.CS;
    const int b = grp / p.Hk, kh = grp % p.Hk;
    const int m = rank / p.SPH;
    const int h = kh + m * p.Hk;
    const int j0 = (rank % p.SPH) * RPC;
    const int C = p.C;
    const int HvD = p.Hv * kD;

    __shared__ __align__(16) float q_s[kD];
    __shared__ __align__(16) float k_s[kD];
    __shared__ float v_s[RPC];
    __shared__ float o_s[RPC];
    __shared__ float red[2][NW];
    __shared__ float part[NW];
    __shared__ float gates[2];
    __shared__ float abp[NW][2];   // folded a/b: the warps' partial dot products
    __shared__ float rms_part[kMaxK];

    // launched as a programmatic dependent: nothing global is touched before the previous
    // kernel in the stream is done (it may have written the state, the conv state or the inputs)
    grid_dependency_wait();
    grid_launch_dependents();
    // ---- state rows: issue the 128-bit loads before anything else
    const Ts* Sin = rec_state_in<Ts>(p, b) + static_cast<size_t>(h) * kD * kD + static_cast<size_t>(j0) * kD;
    float4 s[8];
#pragma unroll
    for (int rr = 0; rr < 8; ++rr)
        s[rr] = StateIO<Ts>::ld_stream(Sin + static_cast<size_t>(warp * 8 + rr) * kD + 4 * lane);

    // ---- per-thread channel ownership: thread i < 128 owns q channel i and k
    // channel i of head kh; thread t < RPC owns v channel j0 + t of head h.
    const bool own_qk = tid < kD;
    const bool own_v = tid < RPC;
    const int cq = kh * kD + tid;
    const int ck = p.Hk * kD + kh * kD + tid;
    const int cv = 2 * p.Hk * kD + h * kD + j0 + tid;
    const Tact* xin = static_cast<const Tact*>(p.x);
    const Tact* cin = static_cast<const Tact*>(p.conv_in) + static_cast<size_t>(b) * 3 * C;
    Tact wq[3], wk[3], wv[3];
    float4 Wq = make_float4(0, 0, 0, 0), Wk = Wq, Wv = Wq;
    float nw = 0.f;
    if (own_qk) {
        Wq = *reinterpret_cast<const float4*>(p.conv_w + 4 * cq);
        Wk = *reinterpret_cast<const float4*>(p.conv_w + 4 * ck);
#pragma unroll
        for (int r = 0; r < 3; ++r) { wq[r] = cin[r * C + cq]; wk[r] = cin[r * C + ck]; }
    }
    if (own_v) {
        Wv = *reinterpret_cast<const float4*>(p.conv_w + 4 * cv);
#pragma unroll
        for (int r = 0; r < 3; ++r) wv[r] = cin[r * C + cv];
        nw = p.norm_w[j0 + tid];
    }
    const float a_dt = p.dt_bias[h];
    const float a_ssm = p.ssm_a[h];
    int* const status = (p.dev_status && (p.flags & kFlagCheckFinite)) ? p.dev_status + b * p.Hv + h : nullptr;

    for (int t = 0; t < p.K; ++t) {
        const size_t row = static_cast<size_t>(b) * p.K + t;      // token row
        const Tact* xr = xin + row * C;
        // ---- steps 1-3: conv, SiLU (q/k of kh; v of my rows)
        Tact xq{}, xk{}, xv{};
        float qv = 0.f, kv = 0.f, zsil = 0.f;
        if (own_qk) {
            xq = xr[cq];
            xk = xr[ck];
            qv = siluf_(conv4(Wq, to_f(wq[0]), to_f(wq[1]), to_f(wq[2]), to_f(xq)));
            kv = siluf_(conv4(Wk, to_f(wk[0]), to_f(wk[1]), to_f(wk[2]), to_f(xk)));
        }
        if (own_v) {
            xv = xr[cv];
            v_s[tid] = siluf_(conv4(Wv, to_f(wv[0]), to_f(wv[1]), to_f(wv[2]), to_f(xv)));
            zsil = siluf_(ld_act(static_cast<const Tact*>(p.z) + row * HvD + h * kD + j0 + tid));
        }
        if (!p.ab_hidden) {
            if (tid == 0) {
                // step 6: gates
                gates[0] = sigmoidf_(ld_act(static_cast<const Tact*>(p.b_raw) + row * p.Hv + h));
                gates[1] = a_ssm * softplusf_(ld_act(static_cast<const Tact*>(p.a_raw) + row * p.Hv + h) + a_dt);
            }
        } else {
            // ssm_alpha / ssm_beta folded in: a share of hidden[row] . W_a[h] and . W_b[h]
            const float2 pr = ab_dot_part<true>(static_cast<const __nv_bfloat16*>(p.ab_hidden) + row * p.ab_H,
                                          static_cast<const __nv_bfloat16*>(p.W_a) + static_cast<size_t>(h) * p.ab_H,
                                          static_cast<const __nv_bfloat16*>(p.W_b) + static_cast<size_t>(h) * p.ab_H,
                                          p.ab_H, tid, NT);
            const float sa = warp_sum(pr.x), sb = warp_sum(pr.y);
            if (lane == 0) {
                abp[warp][0] = sa;
                abp[warp][1] = sb;
            }
        }
        // ---- step 4: clamp-form L2 norms of q and k (threads 0..127 = warps 0..3)
        {
            const float sq = warp_sum(qv * qv), sk = warp_sum(kv * kv);
            if (lane == 0) { red[0][warp] = sq; red[1][warp] = sk; }
        }
        __syncthreads();
        if (p.ab_hidden && tid == 0) {
            // step 6 with the folded projections (read before the next barrier)
            float sa = 0.f, sb = 0.f;
#pragma unroll
            for (int w8 = 0; w8 < NW; ++w8) {
                sa += abp[w8][0];
                sb += abp[w8][1];
            }
            gates[0] = sigmoidf_(sb);
            gates[1] = a_ssm * softplusf_(sa + a_dt);
        }
        if (own_qk) {
            const float nq = sqrtf((red[0][0] + red[0][1]) + (red[0][2] + red[0][3]));
            const float nk = sqrtf((red[1][0] + red[1][1]) + (red[1][2] + red[1][3]));
            q_s[tid] = qv / fmaxf(nq, p.eps);
            k_s[tid] = kv / fmaxf(nk, p.eps);
        }
        __syncthreads();

        // ---- step 7: delta rule on my rows
        const float4 kk = *reinterpret_cast<const float4*>(&k_s[4 * lane]);
        const float4 qq = *reinterpret_cast<const float4*>(&q_s[4 * lane]);
        const float kq = warp_sum(fmaf(kk.w, qq.w, fmaf(kk.z, qq.z, fmaf(kk.y, qq.y, kk.x * qq.x))));
        const float beta = gates[0];
        const float eg = expf(gates[1]);
        float o[8];
#pragma unroll
        for (int rr = 0; rr < 8; ++rr) {
            const float4 sv = s[rr];
            const float pk = warp_sum(fmaf(sv.w, kk.w, fmaf(sv.z, kk.z, fmaf(sv.y, kk.y, sv.x * kk.x))));
            const float pq = warp_sum(fmaf(sv.w, qq.w, fmaf(sv.z, qq.z, fmaf(sv.y, qq.y, sv.x * qq.x))));
            const float vj = v_s[warp * 8 + rr];
            const float d = (vj - eg * pk) * beta;           // d = (v - (e^g S).k) beta
            float4 nv;
            nv.x = fmaf(d, kk.x, eg * sv.x);                 // S = e^g S + d k^T
            nv.y = fmaf(d, kk.y, eg * sv.y);
            nv.z = fmaf(d, kk.z, eg * sv.z);
            nv.w = fmaf(d, kk.w, eg * sv.w);
            s[rr] = StateIO<Ts>::round(nv);                  // what the stored state reads back as
            o[rr] = fmaf(d, kq, eg * pq) * kInvSqrtD;        // o = S_new.q / sqrt(128)
        }
        // state out: in place for a decode step, checkpoint t for a verify walk
        {
            Ts* Sout = rec_state_out<Ts>(p, b, t) + static_cast<size_t>(h) * kD * kD + static_cast<size_t>(j0) * kD;
#pragma unroll
            for (int rr = 0; rr < 8; ++rr) {
                StateIO<Ts>::st(Sout + static_cast<size_t>(warp * 8 + rr) * kD + 4 * lane, s[rr]);
                if (status && (nonfinite_bits(s[rr].x) | nonfinite_bits(s[rr].y) | nonfinite_bits(s[rr].z) |
                               nonfinite_bits(s[rr].w)))
                    atomicOr(status, 1);
            }
        }
        float ps = 0.f;
#pragma unroll
        for (int rr = 0; rr < 8; ++rr) {
            ps = fmaf(o[rr], o[rr], ps);
            if (lane == rr) o_s[warp * 8 + rr] = o[rr];
        }
        if (lane == 0) part[warp] = ps;
        __syncthreads();
        if (tid == 0) {
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) acc += part[w];
            rms_part[t] = acc;
        }
        // ---- step 8: gated RMSNorm across the CTAs holding this head
        cluster_sync_all();
        if (own_v) {
            float tot = 0.f;
            for (int r = 0; r < p.SPH; ++r) tot += ld_dsmem_f32(&rms_part[t], m * p.SPH + r);
            const float rs = 1.0f / sqrtf(tot * (1.0f / kD) + p.eps);
            const float ov = o_s[tid];
            const float y = ov * rs * nw * zsil;
            const size_t oi = row * HvD + h * kD + j0 + tid;
            st_out(static_cast<Tout*>(p.out) + oi, y);
            if (p.prenorm) p.prenorm[oi] = ov;
            if (status && nonfinite_bits(y)) atomicOr(status, 2);
        }
        // ---- conv state after token t: window (w1, w2, x_t); raw values, bit-exact
        Tact* cout = static_cast<Tact*>(p.conv_out) + static_cast<size_t>(b) * p.conv_out_b +
                     static_cast<size_t>(t) * p.conv_out_p;
        if (own_v) {
            cout[0 * C + cv] = wv[1]; cout[1 * C + cv] = wv[2]; cout[2 * C + cv] = xv;
            wv[0] = wv[1]; wv[1] = wv[2]; wv[2] = xv;
        }
        if (own_qk) {
            if (rank == 0) {   // every CTA of the cluster has read these channels
                cout[0 * C + cq] = wq[1]; cout[1 * C + cq] = wq[2]; cout[2 * C + cq] = xq;
                cout[0 * C + ck] = wk[1]; cout[1 * C + ck] = wk[2]; cout[2 * C + ck] = xk;
            }
            wq[0] = wq[1]; wq[1] = wq[2]; wq[2] = xq;
            wk[0] = wk[1]; wk[1] = wk[2]; wk[2] = xk;
        }
    }
    // no CTA leaves while another may still read its rms_part
    cluster_sync_all();
}

// Commit: copy checkpoint accept_len[b]-1 into the live state (bit-exact).
__global__ void commit_kernel(const CommitParams p) {
    // launched as a programmatic dependent of the verify walk, whose checkpoints it reads
    grid_dependency_wait();
    grid_launch_dependents();
    const int b = blockIdx.y;
    const int n = p.accept_len[b];
    if (n < 1 || n > p.K) return;
    if (p.ring_cur) {   // ring: the accepted checkpoint's slot becomes the live one; only the conv rows move
        const uint4* csrc = reinterpret_cast<const uint4*>(static_cast<const char*>(p.conv_ckpt) +
                                                           (static_cast<size_t>(b) * p.K + (n - 1)) * p.conv_bytes);
        uint4* cdst = reinterpret_cast<uint4*>(static_cast<char*>(p.conv_state) + static_cast<size_t>(b) * p.conv_bytes);
        for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < p.conv_bytes / 16;
             i += static_cast<size_t>(gridDim.x) * blockDim.x)
            cdst[i] = csrc[i];
        if (blockIdx.x == 0 && threadIdx.x == 0) p.ring_cur[b] = (p.ring_cur[b] + n) % p.ring_R;
        return;
    }
    const uint4* Ssrc = reinterpret_cast<const uint4*>(static_cast<const char*>(p.S_ckpt) +
                                                       (static_cast<size_t>(b) * p.K + (n - 1)) * p.S_bytes);
    uint4* Sdst = reinterpret_cast<uint4*>(static_cast<char*>(p.S) + static_cast<size_t>(b) * p.S_bytes);
    const size_t nS = p.S_bytes / 16;
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < nS;
         i += static_cast<size_t>(gridDim.x) * blockDim.x)
        Sdst[i] = Ssrc[i];
    const uint4* csrc = reinterpret_cast<const uint4*>(static_cast<const char*>(p.conv_ckpt) +
                                                       (static_cast<size_t>(b) * p.K + (n - 1)) * p.conv_bytes);
    uint4* cdst = reinterpret_cast<uint4*>(static_cast<char*>(p.conv_state) + static_cast<size_t>(b) * p.conv_bytes);
    const size_t nC = p.conv_bytes / 16;
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < nC;
         i += static_cast<size_t>(gridDim.x) * blockDim.x)
        cdst[i] = csrc[i];
}

// Conv-state initialiser: copy `prefix` or write zeros (16-byte words).
__global__ void conv_init_kernel(uint4* dst, const uint4* src, size_t n16) {
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n16;
         i += static_cast<size_t>(gridDim.x) * blockDim.x)
        dst[i] = src ? src[i] : make_uint4(0, 0, 0, 0);
}

// Status summary: the exact count of nonzero words, and the first `cap` of them
// (index, bits) in increasing index order.  One block of 1024 threads walks the
// words in tiles; a ballot per warp and a prefix over the warps give each
// faulted word its rank.
__global__ void __launch_bounds__(1024) state_faults_kernel(const int* st, int n, int cap, int* rep) {
    __shared__ int warp_cnt[32];
    __shared__ int base;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) base = 0;
    __syncthreads();
    for (int start = 0; start < n; start += 1024) {
        const int i = start + tid;
        const int v = i < n ? st[i] : 0;
        const unsigned m = __ballot_sync(0xffffffffu, v != 0);
        if (lane == 0) warp_cnt[warp] = __popc(m);
        __syncthreads();
        int pos = base + __popc(m & ((1u << lane) - 1u));
        for (int w = 0; w < warp; ++w) pos += warp_cnt[w];
        if (v != 0 && pos < cap) {
            rep[2 + 2 * pos] = i;
            rep[3 + 2 * pos] = v;
        }
        __syncthreads();
        if (tid == 0) {
            int t = 0;
            for (int w = 0; w < 32; ++w) t += warp_cnt[w];
            base += t;
        }
        __syncthreads();
    }
    if (tid == 0) {
        rep[0] = base;
        rep[1] = min(base, cap);
    }
}

// Reset of the faulted states: block (n, h) zeroes the live plane of (n, h) when
// its status word is nonzero, and its share of the conv rows of sequence n when
// any head of n is faulted.  The status words are read only; the host clears
// them after this kernel.
__global__ void state_reset_kernel(const ResetParams p) {
    const int n = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    const int* st = p.dev_status + static_cast<size_t>(n) * p.Hv;
    if (st[h] != 0) {
        const size_t slot = p.R > 0 ? static_cast<size_t>(n) * p.R + p.ring_cur[n] : static_cast<size_t>(n);
        uint4* plane = reinterpret_cast<uint4*>(static_cast<char*>(p.S) + (slot * p.Hv + h) * p.plane_bytes);
        for (size_t e = tid; e < p.plane_bytes / 16; e += blockDim.x) plane[e] = make_uint4(0, 0, 0, 0);
    }
    if (p.conv_state) {
        int any = 0;
        for (int j = tid; j < p.Hv; j += blockDim.x) any |= st[j];
        if (__syncthreads_or(any)) {
            uint4* c = reinterpret_cast<uint4*>(static_cast<char*>(p.conv_state) + static_cast<size_t>(n) * p.conv_bytes);
            for (size_t e = static_cast<size_t>(h) * blockDim.x + tid; e < p.conv_bytes / 16;
                 e += static_cast<size_t>(p.Hv) * blockDim.x)
                c[e] = make_uint4(0, 0, 0, 0);
        }
    }
}

template <typename Tact, typename Tout, typename Ts>
cudaError_t launch_rec_t(const RecParams& p, int rpc, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see grid_dependency_wait
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cfg.gridDim = dim3(static_cast<unsigned>(p.B) * p.Hk * p.CS);
    cfg.blockDim = dim3(rpc * 4);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    switch (rpc) {
        case 32: {
            auto k = recurrent_kernel<Tact, Tout, Ts, 32>;
            if (p.CS > 8) cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            return cudaLaunchKernelEx(&cfg, k, p);
        }
        case 64: {
            auto k = recurrent_kernel<Tact, Tout, Ts, 64>;
            if (p.CS > 8) cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            return cudaLaunchKernelEx(&cfg, k, p);
        }
        default: {
            auto k = recurrent_kernel<Tact, Tout, Ts, 128>;
            if (p.CS > 8) cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            return cudaLaunchKernelEx(&cfg, k, p);
        }
    }
}

}  // namespace

cudaError_t launch_recurrent(const RecParams& p, int act_dtype, int out_dtype, int rpc, cudaStream_t stream) {
    using bf = __nv_bfloat16;
    if (p.flags & kFlagStateBf16)   // bf16 activations only (checked by the API)
        return out_dtype == 1 ? launch_rec_t<bf, bf, bf>(p, rpc, stream) : launch_rec_t<bf, float, bf>(p, rpc, stream);
    if (act_dtype == 1)
        return out_dtype == 1 ? launch_rec_t<bf, bf, float>(p, rpc, stream) : launch_rec_t<bf, float, float>(p, rpc, stream);
    return out_dtype == 1 ? launch_rec_t<float, bf, float>(p, rpc, stream) : launch_rec_t<float, float, float>(p, rpc, stream);
}

cudaError_t launch_commit(const CommitParams& p, cudaStream_t stream) {
    const size_t per = (p.ring_cur ? p.conv_bytes : p.S_bytes) / 16;   // a ring moves the conv rows only
    unsigned bx = static_cast<unsigned>((per + 255) / 256);
    if (bx > 64) bx = 64;
    if (bx < 1) bx = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(bx, static_cast<unsigned>(p.B));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see grid_dependency_wait
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, commit_kernel, p);
}

cudaError_t launch_conv_init(void* dst, const void* src, size_t bytes, cudaStream_t stream) {
    const size_t n16 = bytes / 16;
    unsigned blocks = static_cast<unsigned>((n16 + 255) / 256);
    if (blocks > 1024) blocks = 1024;
    if (blocks < 1) blocks = 1;
    conv_init_kernel<<<blocks, 256, 0, stream>>>(static_cast<uint4*>(dst), static_cast<const uint4*>(src), n16);
    return cudaGetLastError();
}

cudaError_t launch_state_faults(const int* dev_status, int n, int cap, int* report, cudaStream_t stream) {
    state_faults_kernel<<<1, 1024, 0, stream>>>(dev_status, n, cap, report);
    return cudaGetLastError();
}

cudaError_t launch_state_reset(const ResetParams& p, cudaStream_t stream) {
    state_reset_kernel<<<dim3(p.N, p.Hv), 256, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return cudaMemsetAsync(const_cast<int*>(p.dev_status), 0, static_cast<size_t>(p.N) * p.Hv * sizeof(int), stream);
}

}  // namespace gdn
