// gdn_api.cu -- the C ABI of libgdn.so (include/gdn.h): argument validation,
// launch configuration and dispatch.  Host code only; every step of the
// layer runs in the kernels of gdn_recurrent.cu, gdn_recurrent_stream.cu and
// the gdn_prefill_*.cu files.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>

#include "gdn.h"
#include "gdn_internal.h"

namespace {

constexpr int kD = 128;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t act_size(int32_t dt) { return dt == GDN_BF16 ? 2 : 4; }

// Bytes of one recurrent-state element (the storage type the flags select).
size_t state_size(const gdn_dims* d) { return (d->flags & GDN_FLAG_STATE_BF16) ? 2 : 4; }

struct Range {
    const void* p;
    size_t bytes;
};

bool overlap(Range a, Range b) {
    if (!a.p || !b.p || a.bytes == 0 || b.bytes == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

// Every written range must be disjoint from every read-only range and from
// every other written range.
bool any_overlap(const Range* outs, int n_out, const Range* ins, int n_in) {
    for (int i = 0; i < n_out; ++i) {
        for (int j = 0; j < n_in; ++j)
            if (overlap(outs[i], ins[j])) return true;
        for (int j = i + 1; j < n_out; ++j)
            if (overlap(outs[i], outs[j])) return true;
    }
    return false;
}

gdn_status check_dims(const gdn_dims* d) {
    if (!d) return GDN_E_INVALID_ARG;
    if (d->H_k < 1 || d->H_v < 1 || d->H_k > 4096 || d->H_v > 4096) return GDN_E_INVALID_ARG;
    if (d->H_v % d->H_k != 0) return GDN_E_INVALID_ARG;
    if (!(d->eps > 0.0f) || !std::isfinite(d->eps)) return GDN_E_INVALID_ARG;
    if ((d->act_dtype != GDN_F32 && d->act_dtype != GDN_BF16) ||
        (d->out_dtype != GDN_F32 && d->out_dtype != GDN_BF16))
        return GDN_E_INVALID_ARG;
    if (d->flags & ~(GDN_FLAG_CHECK_FINITE | GDN_FLAG_PREFILL_FP32 | GDN_FLAG_STATE_BF16 | GDN_FLAG_TEST_STALL))
        return GDN_E_INVALID_ARG;
    if (d->H_v / d->H_k > 16) return GDN_E_UNSUPPORTED;
    if ((d->flags & GDN_FLAG_STATE_BF16) && d->act_dtype != GDN_BF16) return GDN_E_UNSUPPORTED;
    return GDN_OK;
}

gdn_status check_weights(const gdn_weights* w) {
    if (!w || !w->conv_w || !w->dt_bias || !w->ssm_a || !w->norm_w) return GDN_E_INVALID_ARG;
    if (!aligned16(w->conv_w) || !aligned16(w->dt_bias) || !aligned16(w->ssm_a) || !aligned16(w->norm_w))
        return GDN_E_ALIGNMENT;
    return GDN_OK;
}

gdn_status check_ptrs(std::initializer_list<const void*> required, std::initializer_list<const void*> optional) {
    for (const void* p : required)
        if (!p) return GDN_E_INVALID_ARG;
    for (const void* p : required)
        if (!aligned16(p)) return GDN_E_ALIGNMENT;
    for (const void* p : optional)
        if (p && !aligned16(p)) return GDN_E_ALIGNMENT;
    return GDN_OK;
}

// Rows of one v-head owned by one CTA of the recurrent kernel, chosen so a
// (sequence, q/k-head group) cluster has at most 8 CTAs where possible.
int rows_per_cta(int r) {
    if (r <= 2) return 32;
    if (r <= 4) return 64;
    return 128;
}

gdn_status cuda_status(cudaError_t e) { return e == cudaSuccess ? GDN_OK : GDN_E_CUDA; }

// Streaming (persistent, one CTA per SM) recurrent kernel when there are at
// least two (sequence, q/k-group) items per SM and its stages fit in shared
// memory; the cluster kernel otherwise.  The choice depends on B, H_k and K
// only (and, with ssm_alpha / ssm_beta folded in, the hidden size), never on the data.
bool use_stream_kernel(int B, int Hk, int K, int act_dtype, bool state_bf16, int ab_H, int* grid) {
    int dev = 0, sms = 0, smem = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return false;
    const long long items = static_cast<long long>(B) * Hk;
    if (items < 2LL * sms) return false;
    if (gdn::recurrent_stream_smem(K, act_dtype, state_bf16, ab_H) > static_cast<size_t>(smem)) return false;
    *grid = sms;
    return true;
}

}  // namespace

extern "C" {

const char* gdn_status_string(gdn_status s) {
    switch (s) {
        case GDN_OK: return "ok";
        case GDN_E_INVALID_ARG: return "invalid argument";
        case GDN_E_UNSUPPORTED: return "unsupported configuration";
        case GDN_E_ALIGNMENT: return "device pointer not 16-byte aligned";
        case GDN_E_CUDA: return "CUDA launch error";
        case GDN_E_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

int32_t gdn_version(void) { return 100; }

gdn_status gdn_conv_state_init(const gdn_dims* dims, int32_t n_seq, void* conv_state, const void* prefix,
                               gdn_stream_t stream) {
    gdn_status s = check_dims(dims);
    if (s != GDN_OK) return s;
    if (n_seq < 0) return GDN_E_INVALID_ARG;
    if (n_seq == 0) return GDN_OK;
    if ((s = check_ptrs({conv_state}, {prefix})) != GDN_OK) return s;
    const size_t C = static_cast<size_t>(kD) * (2 * dims->H_k + dims->H_v);
    const size_t bytes = static_cast<size_t>(n_seq) * 3 * C * act_size(dims->act_dtype);
    if (prefix && prefix != conv_state && overlap({prefix, bytes}, {conv_state, bytes})) return GDN_E_INVALID_ARG;
    if (prefix == conv_state) return GDN_OK;
    return cuda_status(gdn::launch_conv_init(conv_state, prefix, bytes, reinterpret_cast<cudaStream_t>(stream)));
}

// ring_cur != nullptr: S_in == S_out is a state ring [B][R][H_v][128][128] (see gdn_verify_k_ring).
// ssm_alpha / ssm_beta folded into the recurrent kernels (gdn_decode_step_ab)
struct AbFold {
    int32_t H;
    const void* hidden;
    const void* W_a;
    const void* W_b;
};

static gdn_status recurrent_common(const gdn_dims* dims, const gdn_weights* w, int32_t B, int32_t K,
                                   const void* x, const void* z, const void* a_raw, const void* b_raw,
                                   const void* conv_in, const void* S_in, void* conv_out, void* S_out,
                                   bool verify, void* out, float* prenorm_out, int32_t* dev_status,
                                   gdn_stream_t stream, const int32_t* ring_cur = nullptr, int32_t R = 0,
                                   const AbFold* ab = nullptr) {
    gdn_status s = check_dims(dims);
    if (s != GDN_OK) return s;
    if (B < 0 || K < 1 || K > GDN_MAX_VERIFY_K) return GDN_E_INVALID_ARG;
    if (ring_cur && (R < (verify ? K + 1 : 1) || R > GDN_MAX_VERIFY_K + 1)) return GDN_E_INVALID_ARG;
    if (ab && (ab->H < 8 || ab->H % 8 != 0)) return GDN_E_INVALID_ARG;
    if (ab && dims->act_dtype != GDN_BF16) return GDN_E_UNSUPPORTED;
    if (B == 0) return GDN_OK;
    if ((s = check_weights(w)) != GDN_OK) return s;
    if (ab) {
        // the folded projections take the place of a_raw / b_raw
        if ((s = check_ptrs({x, z, ab->hidden, ab->W_a, ab->W_b, conv_in, S_in, conv_out, S_out, out},
                            {prenorm_out, dev_status})) != GDN_OK)
            return s;
    } else if ((s = check_ptrs({x, z, a_raw, b_raw, conv_in, S_in, conv_out, S_out, out}, {prenorm_out, dev_status})) !=
               GDN_OK) {
        return s;
    }
    if (ring_cur && (s = check_ptrs({ring_cur}, {})) != GDN_OK) return s;
    const int Hk = dims->H_k, Hv = dims->H_v;
    const size_t C = static_cast<size_t>(kD) * (2 * Hk + Hv);
    const size_t ea = act_size(dims->act_dtype), eo = act_size(dims->out_dtype);
    const size_t T = static_cast<size_t>(B) * K;
    const size_t HvD = static_cast<size_t>(Hv) * kD;
    const size_t S_bytes = static_cast<size_t>(B) * Hv * kD * kD * state_size(dims);
    const size_t cv_bytes = static_cast<size_t>(B) * 3 * C * ea;
    // a ring is read and written in one buffer (like the in-place decode state)
    const size_t S_out_bytes = ring_cur ? S_bytes * R : (verify ? S_bytes * K : S_bytes);
    const size_t Hab = ab ? static_cast<size_t>(ab->H) : 0;
    const Range ins[] = {{x, T * C * ea}, {z, T * HvD * ea}, {ab ? nullptr : a_raw, T * Hv * ea},
                         {ab ? nullptr : b_raw, T * Hv * ea}, {w->conv_w, C * 16}, {w->dt_bias, Hv * 4u},
                         {w->ssm_a, Hv * 4u}, {w->norm_w, kD * 4u}, {verify ? conv_in : nullptr, cv_bytes},
                         {verify && !ring_cur ? S_in : nullptr, S_bytes}, {ring_cur, B * 4u},
                         {ab ? ab->hidden : nullptr, T * Hab * 2}, {ab ? ab->W_a : nullptr, Hv * Hab * 2},
                         {ab ? ab->W_b : nullptr, Hv * Hab * 2}};
    const Range outs[] = {{out, T * HvD * eo}, {prenorm_out, T * HvD * 4}, {dev_status, B * Hv * 4u},
                          {conv_out, verify ? cv_bytes * K : cv_bytes}, {S_out, S_out_bytes}};
    if (any_overlap(outs, 5, ins, 14)) return GDN_E_INVALID_ARG;

    gdn::RecParams p{};
    const int r = Hv / Hk;
    const int rpc = rows_per_cta(r);
    p.B = B; p.K = K; p.Hk = Hk; p.Hv = Hv; p.C = static_cast<int>(C);
    p.SPH = kD / rpc;
    p.CS = r * p.SPH;
    p.eps = dims->eps;
    p.flags = dims->flags;
    p.x = x; p.z = z; p.a_raw = a_raw; p.b_raw = b_raw;
    p.conv_w = w->conv_w; p.dt_bias = w->dt_bias; p.ssm_a = w->ssm_a; p.norm_w = w->norm_w;
    p.conv_in = conv_in; p.S_in = S_in; p.conv_out = conv_out; p.S_out = S_out;
    if (verify) {
        p.conv_out_b = static_cast<long long>(K) * 3 * C;  p.conv_out_p = static_cast<long long>(3 * C);
        p.S_out_b = static_cast<long long>(K) * Hv * kD * kD; p.S_out_p = static_cast<long long>(Hv) * kD * kD;
    } else {
        p.conv_out_b = static_cast<long long>(3 * C); p.conv_out_p = 0;
        p.S_out_b = static_cast<long long>(Hv) * kD * kD; p.S_out_p = 0;
    }
    p.out = out; p.prenorm = prenorm_out; p.dev_status = dev_status;
    p.ring_cur = ring_cur; p.ring_R = R; p.ring_shift = verify ? 1 : 0;
    if (ab) {
        p.a_raw = nullptr; p.b_raw = nullptr;
        p.ab_hidden = ab->hidden; p.W_a = ab->W_a; p.W_b = ab->W_b; p.ab_H = ab->H;
    }
    int grid = 0;
    if (use_stream_kernel(B, Hk, K, dims->act_dtype, (dims->flags & GDN_FLAG_STATE_BF16) != 0, ab ? ab->H : 0,
                          &grid))
        return cuda_status(gdn::launch_recurrent_stream(p, dims->act_dtype, dims->out_dtype, grid,
                                                        reinterpret_cast<cudaStream_t>(stream)));
    return cuda_status(gdn::launch_recurrent(p, dims->act_dtype, dims->out_dtype, rpc,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

gdn_status gdn_decode_step(const gdn_dims* dims, const gdn_weights* w, int32_t B, const void* x, const void* z,
                           const void* a_raw, const void* b_raw, void* conv_state, void* S, void* out,
                           float* prenorm_out, int32_t* dev_status, gdn_stream_t stream) {
    return recurrent_common(dims, w, B, 1, x, z, a_raw, b_raw, conv_state, S, conv_state, S, false, out,
                            prenorm_out, dev_status, stream);
}

gdn_status gdn_decode_step_ab(const gdn_dims* dims, const gdn_weights* w, int32_t B, int32_t H, const void* x,
                              const void* z, const void* hidden, const void* W_a, const void* W_b, void* conv_state,
                              void* S, void* out, float* prenorm_out, int32_t* dev_status, gdn_stream_t stream) {
    const AbFold ab{H, hidden, W_a, W_b};
    return recurrent_common(dims, w, B, 1, x, z, nullptr, nullptr, conv_state, S, conv_state, S, false, out,
                            prenorm_out, dev_status, stream, nullptr, 0, &ab);
}

gdn_status gdn_verify_k(const gdn_dims* dims, const gdn_weights* w, int32_t B, int32_t K, const void* x,
                        const void* z, const void* a_raw, const void* b_raw, const void* conv_state,
                        const void* S, void* conv_ckpt, void* S_ckpt, void* out, float* prenorm_out,
                        int32_t* dev_status, gdn_stream_t stream) {
    return recurrent_common(dims, w, B, K, x, z, a_raw, b_raw, conv_state, S, conv_ckpt, S_ckpt, true, out,
                            prenorm_out, dev_status, stream);
}

gdn_status gdn_commit(const gdn_dims* dims, int32_t B, int32_t K, const int32_t* accept_len, const void* conv_ckpt,
                      const void* S_ckpt, void* conv_state, void* S, gdn_stream_t stream) {
    gdn_status s = check_dims(dims);
    if (s != GDN_OK) return s;
    if (B < 0 || K < 1 || K > GDN_MAX_VERIFY_K) return GDN_E_INVALID_ARG;
    if (B == 0) return GDN_OK;
    if ((s = check_ptrs({accept_len, conv_ckpt, S_ckpt, conv_state, S}, {})) != GDN_OK) return s;
    const size_t C = static_cast<size_t>(kD) * (2 * dims->H_k + dims->H_v);
    gdn::CommitParams p{};
    p.B = B; p.K = K; p.accept_len = accept_len; p.conv_ckpt = conv_ckpt; p.S_ckpt = S_ckpt;
    p.conv_state = conv_state; p.S = S;
    p.S_bytes = static_cast<size_t>(dims->H_v) * kD * kD * state_size(dims);
    p.conv_bytes = 3 * C * act_size(dims->act_dtype);
    const Range ins[] = {{accept_len, B * 4u}, {conv_ckpt, p.conv_bytes * B * K}, {S_ckpt, p.S_bytes * B * K}};
    const Range outs[] = {{conv_state, p.conv_bytes * B}, {S, p.S_bytes * B}};
    if (any_overlap(outs, 2, ins, 3)) return GDN_E_INVALID_ARG;
    return cuda_status(gdn::launch_commit(p, reinterpret_cast<cudaStream_t>(stream)));
}

gdn_status gdn_decode_step_ring(const gdn_dims* dims, const gdn_weights* w, int32_t B, int32_t R, const void* x,
                                const void* z, const void* a_raw, const void* b_raw, void* conv_state, void* S_ring,
                                const int32_t* ring_cur, void* out, float* prenorm_out, int32_t* dev_status,
                                gdn_stream_t stream) {
    if (!ring_cur) return GDN_E_INVALID_ARG;
    return recurrent_common(dims, w, B, 1, x, z, a_raw, b_raw, conv_state, S_ring, conv_state, S_ring, false, out,
                            prenorm_out, dev_status, stream, ring_cur, R);
}

gdn_status gdn_verify_k_ring(const gdn_dims* dims, const gdn_weights* w, int32_t B, int32_t K, int32_t R,
                             const void* x, const void* z, const void* a_raw, const void* b_raw,
                             const void* conv_state, void* S_ring, const int32_t* ring_cur, void* conv_ckpt,
                             void* out, float* prenorm_out, int32_t* dev_status, gdn_stream_t stream) {
    if (!ring_cur) return GDN_E_INVALID_ARG;
    return recurrent_common(dims, w, B, K, x, z, a_raw, b_raw, conv_state, S_ring, conv_ckpt, S_ring, true, out,
                            prenorm_out, dev_status, stream, ring_cur, R);
}

gdn_status gdn_commit_ring(const gdn_dims* dims, int32_t B, int32_t K, int32_t R, const int32_t* accept_len,
                           const void* conv_ckpt, void* conv_state, int32_t* ring_cur, gdn_stream_t stream) {
    gdn_status s = check_dims(dims);
    if (s != GDN_OK) return s;
    if (B < 0 || K < 1 || K > GDN_MAX_VERIFY_K || R < K + 1 || R > GDN_MAX_VERIFY_K + 1) return GDN_E_INVALID_ARG;
    if (B == 0) return GDN_OK;
    if ((s = check_ptrs({accept_len, conv_ckpt, conv_state, ring_cur}, {})) != GDN_OK) return s;
    const size_t C = static_cast<size_t>(kD) * (2 * dims->H_k + dims->H_v);
    gdn::CommitParams p{};
    p.B = B; p.K = K; p.accept_len = accept_len; p.conv_ckpt = conv_ckpt; p.conv_state = conv_state;
    p.ring_cur = ring_cur; p.ring_R = R;
    p.S_bytes = static_cast<size_t>(dims->H_v) * kD * kD * state_size(dims);
    p.conv_bytes = 3 * C * act_size(dims->act_dtype);
    const Range ins[] = {{accept_len, B * 4u}, {conv_ckpt, p.conv_bytes * B * K}};
    const Range outs[] = {{conv_state, p.conv_bytes * B}, {ring_cur, B * 4u}};
    if (any_overlap(outs, 2, ins, 2)) return GDN_E_INVALID_ARG;
    return cuda_status(gdn::launch_commit(p, reinterpret_cast<cudaStream_t>(stream)));
}

gdn_status gdn_state_faults(const gdn_dims* dims, int32_t N, const int32_t* dev_status, int32_t cap,
                            int32_t* report, gdn_stream_t stream) {
    gdn_status s = check_dims(dims);
    if (s != GDN_OK) return s;
    if (N < 0 || cap < 0 || static_cast<int64_t>(N) * dims->H_v > INT32_MAX) return GDN_E_INVALID_ARG;
    if ((s = check_ptrs({dev_status, report}, {})) != GDN_OK) return s;
    const size_t n = static_cast<size_t>(N) * dims->H_v;
    const Range ins[] = {{dev_status, n * 4}};
    const Range outs[] = {{report, (2 + 2 * static_cast<size_t>(cap)) * 4}};
    if (any_overlap(outs, 1, ins, 1)) return GDN_E_INVALID_ARG;
    return cuda_status(gdn::launch_state_faults(dev_status, static_cast<int>(n), cap, report,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

gdn_status gdn_state_reset(const gdn_dims* dims, int32_t N, int32_t R, void* S, const int32_t* ring_cur,
                           void* conv_state, int32_t* dev_status, gdn_stream_t stream) {
    gdn_status s = check_dims(dims);
    if (s != GDN_OK) return s;
    if (N < 0 || R < 0 || R > GDN_MAX_VERIFY_K + 1 || (R > 0) != (ring_cur != nullptr)) return GDN_E_INVALID_ARG;
    if (N == 0) return GDN_OK;
    if ((s = check_ptrs({S, dev_status}, {ring_cur, conv_state})) != GDN_OK) return s;
    gdn::ResetParams p{};
    p.N = N; p.Hv = dims->H_v; p.R = R; p.S = S; p.ring_cur = ring_cur; p.conv_state = conv_state;
    p.plane_bytes = static_cast<size_t>(kD) * kD * state_size(dims);
    p.conv_bytes = 3 * static_cast<size_t>(kD) * (2 * dims->H_k + dims->H_v) * act_size(dims->act_dtype);
    p.dev_status = dev_status;
    const size_t S_bytes = static_cast<size_t>(N) * (R > 0 ? R : 1) * dims->H_v * p.plane_bytes;
    const Range ins[] = {{ring_cur, N * 4u}};
    const Range outs[] = {{S, S_bytes}, {conv_state, conv_state ? p.conv_bytes * N : 0},
                          {dev_status, static_cast<size_t>(N) * dims->H_v * 4}};
    if (any_overlap(outs, 3, ins, 1)) return GDN_E_INVALID_ARG;
    return cuda_status(gdn::launch_state_reset(p, reinterpret_cast<cudaStream_t>(stream)));
}

size_t gdn_prefill_workspace_bytes(const gdn_dims* dims, int32_t n_seq, int64_t T_total) {
    if (check_dims(dims) != GDN_OK || n_seq < 0 || T_total < 0) return 0;
    return gdn::prefill_workspace_bytes(dims->H_k, dims->H_v, n_seq, T_total, dims->act_dtype, dims->flags);
}

gdn_status gdn_prefill_chunked(const gdn_dims* dims, const gdn_weights* w, int32_t n_seq,
                               const int32_t* cu_seqlens_host, const int32_t* cu_seqlens_dev, const void* x,
                               const void* z, const void* a_raw, const void* b_raw, void* conv_state, void* S,
                               int32_t zero_init, void* out, float* prenorm_out, void* workspace,
                               size_t workspace_bytes, int32_t* dev_status, gdn_stream_t stream) {
    gdn_status s = check_dims(dims);
    if (s != GDN_OK) return s;
    if (n_seq < 0) return GDN_E_INVALID_ARG;
    if (n_seq == 0) return GDN_OK;
    if (!cu_seqlens_host || cu_seqlens_host[0] != 0) return GDN_E_INVALID_ARG;
    int max_len = 0;
    long long n_chunks = 0;
    for (int i = 0; i < n_seq; ++i) {
        const int32_t L = cu_seqlens_host[i + 1] - cu_seqlens_host[i];
        if (cu_seqlens_host[i + 1] < cu_seqlens_host[i]) return GDN_E_INVALID_ARG;
        if (L > max_len) max_len = L;
        n_chunks += (L + 63) / 64;   // chunks of 64 tokens
    }
    const int64_t T = cu_seqlens_host[n_seq];
    if ((s = check_weights(w)) != GDN_OK) return s;
    if ((s = check_ptrs({cu_seqlens_dev, conv_state, S}, {prenorm_out, dev_status, workspace})) != GDN_OK) return s;
    if (T > 0 && (s = check_ptrs({x, z, a_raw, b_raw, out}, {})) != GDN_OK) return s;
    const size_t need = gdn::prefill_workspace_bytes(dims->H_k, dims->H_v, n_seq, T, dims->act_dtype, dims->flags);
    if (need > 0 && (!workspace || workspace_bytes < need)) return GDN_E_WORKSPACE;
    const int Hk = dims->H_k, Hv = dims->H_v;
    const size_t C = static_cast<size_t>(kD) * (2 * Hk + Hv);
    const size_t ea = act_size(dims->act_dtype), eo = act_size(dims->out_dtype);
    const size_t HvD = static_cast<size_t>(Hv) * kD;
    const size_t Tz = static_cast<size_t>(T);
    const Range ins[] = {{x, Tz * C * ea}, {z, Tz * HvD * ea}, {a_raw, Tz * Hv * ea}, {b_raw, Tz * Hv * ea},
                         {w->conv_w, C * 16}, {w->dt_bias, Hv * 4u}, {w->ssm_a, Hv * 4u}, {w->norm_w, kD * 4u},
                         {cu_seqlens_dev, (n_seq + 1) * 4u}};
    const Range outs[] = {{out, Tz * HvD * eo}, {prenorm_out, Tz * HvD * 4}, {dev_status, n_seq * Hv * 4u},
                          {conv_state, n_seq * 3 * C * ea}, {S, static_cast<size_t>(n_seq) * Hv * kD * kD * state_size(dims)},
                          {workspace, need}};
    if (any_overlap(outs, 6, ins, 9)) return GDN_E_INVALID_ARG;

    gdn::PrefillParams p{};
    p.n_seq = n_seq; p.T = T; p.max_len = max_len; p.Hk = Hk; p.Hv = Hv; p.C = static_cast<int>(C);
    p.eps = dims->eps; p.flags = dims->flags; p.zero_init = zero_init != 0;
    p.cu_seqlens = cu_seqlens_dev;
    p.x = x; p.z = z; p.a_raw = a_raw; p.b_raw = b_raw;
    p.conv_w = w->conv_w; p.dt_bias = w->dt_bias; p.ssm_a = w->ssm_a; p.norm_w = w->norm_w;
    p.conv_state = conv_state; p.S = S; p.out = out; p.prenorm = prenorm_out; p.dev_status = dev_status;
    p.workspace = workspace;
    p.n_chunks = static_cast<int>(n_chunks);
    gdn::prefill_bind_workspace(p, dims->act_dtype);
    return cuda_status(gdn::launch_prefill(p, dims->act_dtype, dims->out_dtype, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
