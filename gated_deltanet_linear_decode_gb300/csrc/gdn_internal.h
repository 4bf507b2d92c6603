// gdn_internal.h -- launch parameter blocks shared by the host API and the
// kernels of libgdn.so (not installed; the public surface is include/gdn.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gdn {

constexpr uint32_t kFlagCheckFinite = 1u;
constexpr uint32_t kFlagForceSimt = 2u;   // GDN_FLAG_PREFILL_FP32
constexpr uint32_t kFlagStateBf16 = 4u;   // GDN_FLAG_STATE_BF16: states stored as bf16
constexpr uint32_t kFlagTestStall = 1u << 30;   // GDN_FLAG_TEST_STALL: exercise the give-up path of the waits

// Recurrent walk (decode step when K == 1 and the outputs alias the states;
// speculative verify when the outputs are the checkpoint planes).
struct RecParams {
    int B, K, Hk, Hv, C;
    int CS;    // CTAs per cluster = (H_v/H_k) * SPH
    int SPH;   // CTAs per v-head = 128 / rows-per-CTA
    float eps;
    uint32_t flags;
    const void* x;          // [B*K][C]
    const void* z;          // [B*K][Hv*128]
    const void* a_raw;      // [B*K][Hv]
    const void* b_raw;      // [B*K][Hv]
    const float* conv_w;    // [C][4]
    const float* dt_bias;   // [Hv]
    const float* ssm_a;     // [Hv]
    const float* norm_w;    // [128]
    const void* conv_in;    // [B][3][C]
    const void* S_in;       // [B][Hv][128][128], fp32 or bf16 (the kernel's state type)
    void* conv_out;         // element (b, t) at conv_out + b*conv_out_b + t*conv_out_p
    void* S_out;            // state (b, t) at S_out + b*S_out_b + t*S_out_p (elements)
    long long conv_out_b, conv_out_p;
    long long S_out_b, S_out_p;
    void* out;              // [B*K][Hv*128]
    float* prenorm;         // optional, [B*K][Hv*128]
    int* dev_status;        // optional, [B*Hv]
    // state ring (ring_cur != nullptr): S_in == S_out is [B][ring_R][Hv][128][128]; sequence b
    // reads slot ring_cur[b] and writes position t to slot (ring_cur[b] + ring_shift + t) % ring_R
    const int* ring_cur;
    int ring_R, ring_shift;
    // ssm_alpha / ssm_beta folded in (ab_hidden != nullptr): a_raw and b_raw of token row r
    // and v-head h are the fp32 dot products hidden[r] . W_a[h] and hidden[r] . W_b[h]
    // (bf16 operands, length ab_H); a_raw / b_raw above are then unused
    const void* ab_hidden;  // [B*K][ab_H] bf16
    const void* W_a;        // [Hv][ab_H] bf16
    const void* W_b;        // [Hv][ab_H] bf16
    int ab_H;
};

#ifdef __CUDACC__
// The state a sequence starts from, and where the state after its position t goes
// (Ts: the element type of the state, float or __nv_bfloat16).
template <typename Ts>
__device__ __forceinline__ const Ts* rec_state_in(const RecParams& p, int b) {
    const size_t plane = static_cast<size_t>(p.Hv) * 128 * 128;
    const Ts* S = static_cast<const Ts*>(p.S_in);
    return p.ring_cur ? S + (static_cast<size_t>(b) * p.ring_R + p.ring_cur[b]) * plane : S + static_cast<size_t>(b) * plane;
}
template <typename Ts>
__device__ __forceinline__ Ts* rec_state_out(const RecParams& p, int b, int t) {
    const size_t plane = static_cast<size_t>(p.Hv) * 128 * 128;
    Ts* S = static_cast<Ts*>(p.S_out);
    if (p.ring_cur)
        return S + (static_cast<size_t>(b) * p.ring_R + (p.ring_cur[b] + p.ring_shift + t) % p.ring_R) * plane;
    return S + static_cast<size_t>(b) * p.S_out_b + static_cast<size_t>(t) * p.S_out_p;
}
#endif

struct CommitParams {
    int B, K;
    int* ring_cur;          // ring commit: advance slot indices [B] (S, S_ckpt unused)
    int ring_R;
    const int* accept_len;  // [B]
    const void* conv_ckpt;  // [B][K][3][C]
    const void* S_ckpt;     // [B][K][Hv][128][128]
    void* conv_state;       // [B][3][C]
    void* S;                // [B][Hv][128][128]
    size_t S_bytes;         // Hv*128*128 * state element size
    size_t conv_bytes;      // 3*C*sizeof(act)
};

// Chunked prefill over packed sequences.
struct PrefillParams {
    CUtensorMap xmap;        // x [T][C] bf16, boxes of [67 positions][64 channels], 128-byte swizzle
    int n_seq;
    long long T;
    int max_len;
    int Hk, Hv, C;
    float eps;
    uint32_t flags;
    bool zero_init;
    const int* cu_seqlens;   // device [n_seq+1]
    const void* x;
    const void* z;
    const void* a_raw;
    const void* b_raw;
    const float* conv_w;
    const float* dt_bias;
    const float* ssm_a;
    const float* norm_w;
    void* conv_state;        // [n_seq][3][C] in/out
    void* S;                 // [n_seq][Hv][128][128] in/out, fp32 (bf16 under kFlagStateBf16)
    void* out;
    float* prenorm;
    int* dev_status;
    void* workspace;
    // tensor-core prefill: chunk table and records inside the workspace
    int n_chunks;            // total chunks over all sequences
    int chunk_lo, chunk_hi;  // global chunk range of this launch of the two kernels
    int* chunk_base;         // device [n_seq+1]
    uint8_t* ws_v;           // v-head records, [n_chunks][Hv]
    int* ready;              // [n_chunks][Hv] ready flags of the records, one per v-head (zeroed per call)
    int* consumed;           // [n_chunks][Hk] chains of the group done with the chunk's records (zeroed per call)
    int ahead;               // the preparation role writes chunk c once chunk c - ahead is consumed
    int* abort_flag;         // set by a chain that gave up: the preparation role stops waiting on chains
};

// Workspace bytes of gdn_prefill_chunked for the path that act_dtype / flags select.
size_t prefill_workspace_bytes(int Hk, int Hv, int n_seq, long long T, int act_dtype, uint32_t flags);
// Point the chunk table and record arrays of p into p.workspace.
void prefill_bind_workspace(PrefillParams& p, int act_dtype);
cudaError_t launch_prefill(const PrefillParams& p, int act_dtype, int out_dtype, cudaStream_t stream);

cudaError_t launch_recurrent(const RecParams& p, int act_dtype, int out_dtype, int rows_per_cta,
                             cudaStream_t stream);
size_t recurrent_stream_smem(int K, int act_dtype, bool state_bf16, int ab_H);
cudaError_t launch_recurrent_stream(const RecParams& p, int act_dtype, int out_dtype, int grid, cudaStream_t stream);
cudaError_t launch_commit(const CommitParams& p, cudaStream_t stream);
cudaError_t launch_conv_init(void* dst, const void* src, size_t bytes, cudaStream_t stream);
// Non-finite guard: summary of the status words, and the reset of the faulted states.
cudaError_t launch_state_faults(const int* dev_status, int n, int cap, int* report, cudaStream_t stream);
struct ResetParams {
    int N, Hv, R;            // R = 0: plain S [N][Hv][128][128]; else a ring [N][R][Hv][128][128]
    void* S;
    size_t plane_bytes;      // 128*128 * state element size
    const int* ring_cur;     // [N] live slot (rings only)
    void* conv_state;        // [N][conv_bytes] or null
    size_t conv_bytes;
    const int* dev_status;   // [N*Hv]
};
cudaError_t launch_state_reset(const ResetParams& p, cudaStream_t stream);

// A TMA tensor map of a 2-D bf16 tensor [outer][inner] (row pitch inner * 2 bytes, 16-byte
// aligned) with boxes of [box_outer <= 256][64] elements in the 128-byte swizzle layout;
// false if the driver refuses it (gdn_tma.cu).
bool make_tensor_map_bf16_sw128(CUtensorMap* m, const void* base, int inner, int outer, int box_outer);

// One GEMM of a projection call: out [T][rows] = in [T][K] . W [rows][K]^T (bf16).
struct ProjGemm {
    const void* W;
    void* out;
    int rows;
};
constexpr int kProjStreamMaxRows = 256;   // the weight-streaming kernel takes T <= this
// Up to 4 GEMMs sharing `in`, one launch (gdn_proj_stream.cu): a CTA per 128-row tile, or a
// cluster of 2 or 4 CTAs splitting its K when there are few tiles.  status: optional, bit 4.
cudaError_t launch_proj_stream(const ProjGemm* g, int n_gemm, const void* in, int T, int K, int* status,
                               bool test_stall, cudaStream_t stream);

}  // namespace gdn
