/*
 * gdn.h -- C ABI of the GB300 (sm_103a) gated DeltaNet token mixer library
 * (libgdn.so).
 *
 * The operation is the gated DeltaNet layer of the Qwen 3.6 hybrid models, as
 * defined on the xwen CLAUDE.md page, "Architecture cheat sheet (Qwen 3.6,
 * ggml-org GGUF)", paragraph "Gated DeltaNet layer", taken from the fused
 * attn_qkv stream onward:
 *
 *   1. causal depthwise conv1d, kernel 4, no bias, over the full fused width
 *      C = 128*(2*H_k + H_v); left context from a per-sequence conv state of
 *      the last 3 raw rows (oldest first); tap 3 multiplies the current token;
 *   2. SiLU over the whole fused stream;
 *   3. split q = channels [0, 128*H_k), k = [128*H_k, 256*H_k), v = the rest,
 *      head-major inside each block (channel = head*128 + i);
 *   4. L2 norm of q and k in clamp form x / max(||x||, eps);
 *   5. q/k heads tiled to H_v (v-head j reads q/k head j mod H_k -- the page's
 *      "GGUF facts" section: V-head order is tiled, not interleaved);
 *   6. beta = sigmoid(b_raw), g = ssm_a * softplus(a_raw + dt_bias), with
 *      ssm_a = -exp(A_log) pre-baked;
 *   7. delta rule on an fp32 state S per (sequence, v-head):
 *        S = S*exp(g);  d = (v - S.k)*beta;  S += k (x) d;  o = S.q/sqrt(128)
 *   8. gated RMSNorm over each head's 128 outputs:
 *        y = o / sqrt(mean(o^2) + eps) * norm_w * silu(z).
 *
 * Two forms compute it: a per-token recurrent step (gdn_decode_step and the
 * speculative-verify walk gdn_verify_k) and the chunked form with chunk = 64
 * (gdn_prefill_chunked; the page's "Ground truth" list names both forms).
 *
 * Conventions (all entry points):
 *   - Every pointer argument except the gdn_dims / gdn_weights structs and the
 *     cu_seqlens_host array is DEVICE memory, allocated and owned by the
 *     caller.  The library allocates no memory.  Between calls it keeps one
 *     auxiliary CUDA stream per device (created on first use by
 *     gdn_prefill_chunked, which overlaps its two kernels on it) and the fixed
 *     scratch array of gdn_prefill_chunked_static.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  A non-GDN_OK return from argument validation means
 *     nothing was enqueued.  GDN_E_CUDA reports a launch error.
 *   - Every device pointer must be 16-byte aligned (GDN_E_ALIGNMENT).
 *   - Errors are returned, never printed; the library never exits.
 *   - Layouts are dense row-major, innermost index last, in elements:
 *       x           [T][C]                act dtype
 *       z, out      [T][H_v*128]          act dtype / out dtype
 *       a_raw,b_raw [T][H_v]              act dtype
 *       conv_state  [N][3][C]             act dtype (raw rows, oldest first)
 *       S           [N][H_v][128][128]    fp32 (bf16 under GDN_FLAG_STATE_BF16),
 *                                         S[j][i]: j the v-row, i the k-index;
 *                                         "S.k" = sum_i S[j][i] k_i
 *     Every state argument (S, S_ckpt, S_ring) has the element type the
 *     flags select; the arithmetic is fp32 either way.
 *       conv_w      [C][4] fp32; dt_bias, ssm_a [H_v] fp32; norm_w [128] fp32
 *   - prenorm_out (optional, may be NULL) receives o before the gated norm,
 *     fp32 with out's layout.
 *   - dev_status (optional, may be NULL) is int32 [N*H_v].  When
 *     GDN_FLAG_CHECK_FINITE is set, the kernels OR bit 0 into
 *     dev_status[n*H_v + h] if the updated state of (n, h) holds a non-finite
 *     value and bit 1 if its output does.  Bit 4, whatever the flags, means
 *     that a bounded wait inside a kernel gave up and the state and outputs of
 *     (n, h) were not (fully) written (see GDN_FLAG_TEST_STALL).  The caller
 *     zeroes it and reads it after synchronising (the production failure mode
 *     the home-server page records: non-finite GDN state that persists in
 *     cached state).
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (the CUDA runtime's stream handle). */
typedef struct CUstream_st* gdn_stream_t;

typedef enum {
    GDN_OK = 0,
    GDN_E_INVALID_ARG = 1,   /* null pointer, bad size, bad enum, aliasing */
    GDN_E_UNSUPPORTED = 2,   /* valid but not supported (e.g. H_v/H_k > 16) */
    GDN_E_ALIGNMENT = 3,     /* a device pointer is not 16-byte aligned */
    GDN_E_CUDA = 4,          /* a CUDA launch or query failed */
    GDN_E_WORKSPACE = 5      /* workspace missing or too small */
} gdn_status;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

#define GDN_HEAD_DIM 128
#define GDN_CONV_KERNEL 4
#define GDN_CHUNK 64
#define GDN_MAX_VERIFY_K 16
#define GDN_FLAG_CHECK_FINITE 1u
/* gdn_prefill_chunked with bf16 activations: use the fp32 CUDA-core chunk
 * kernel instead of the tensor-core kernel (fp32 products end to end; slower).
 * fp32 activations always take that kernel. */
#define GDN_FLAG_PREFILL_FP32 2u
/* Recurrent state stored as bf16 instead of fp32 (the SGLang deployment on
 * the home-server page pins bf16 mamba-state pools).  Every call reads the
 * state into fp32, computes in fp32 exactly as with an fp32 state, and rounds
 * to nearest-even only when it stores a state: after a decode step, at each
 * verify checkpoint (the walk goes on from the rounded value, so checkpoints
 * still equal decode replays bit for bit) and once at the end of a prefill.
 * Halves the state bytes of the recurrent calls.  Requires act_dtype = GDN_BF16 (else
 * GDN_E_UNSUPPORTED). */
#define GDN_FLAG_STATE_BF16 4u
/* Test hook for the failure path of the kernels' bounded waits (no use in
 * production).  Every wait inside a kernel has an iteration limit; when one
 * gives up, the kernel stops issuing work, lets the asynchronous copies and
 * MMAs it already issued complete, writes nothing more, ORs bit 4 into
 * dev_status for every (sequence, v-head) it did not finish, and returns, so
 * the CUDA context stays usable.  With this flag the kernels that carry the
 * hook -- the streaming recurrent kernel that gdn_decode_step / gdn_verify_k
 * use when B*H_k is at least twice the SM count, the chain role (the
 * chunk-to-chunk state recurrence) of the bf16 tensor-core
 * gdn_prefill_chunked, and the weight-streaming kernel of gdn_in_proj /
 * gdn_out_proj (include/gdn_proj.h, T <= 256; its status word is the one
 * given to those calls) -- first wait on a barrier that nothing arrives
 * on, so that wait gives up after a few microseconds and the path above runs
 * with none of the call's work done: every (sequence, v-head) they own
 * reports bit 4 and S, conv_state and out keep their previous contents. */
#define GDN_FLAG_TEST_STALL (1u << 30)

typedef struct {
    int32_t H_k;        /* q/k heads (16 in both model sizes on the page)       */
    int32_t H_v;        /* v heads, H_v % H_k == 0, H_v/H_k <= 16 (32 or 48)   */
    float eps;          /* L2 clamp and RMSNorm eps (the page: 1e-6)            */
    int32_t act_dtype;  /* gdn_dtype of x, z, a_raw, b_raw, conv_state         */
    int32_t out_dtype;  /* gdn_dtype of out                                     */
    uint32_t flags;     /* GDN_FLAG_*                                           */
} gdn_dims;

typedef struct {
    const float* conv_w;   /* [C][4]   conv1d taps (F32 in the GGUF)           */
    const float* dt_bias;  /* [H_v]    ssm_dt.bias                             */
    const float* ssm_a;    /* [H_v]    ssm_a = -exp(A_log), pre-baked          */
    const float* norm_w;   /* [128]    ssm_norm.weight, multiply-ready          */
} gdn_weights;

/* Text of a status code (static storage; never NULL). */
const char* gdn_status_string(gdn_status status);

/* Library version, major*10000 + minor*100 + patch. */
int32_t gdn_version(void);

/*
 * gdn_conv_state_init -- set conv_state [n_seq][3][C] to `prefix` (same
 * layout; copied bit-exactly), or to zeros when prefix is NULL.  A fresh
 * sequence has no left context, so its conv state is zero; a caller with
 * fewer than 3 earlier rows left-pads them with zeros in `prefix`.
 * (The page's definition: conv state = last 3 columns of the fused stream.)
 */
gdn_status gdn_conv_state_init(const gdn_dims* dims, int32_t n_seq, void* conv_state,
                               const void* prefix, gdn_stream_t stream);

/*
 * gdn_decode_step -- one recurrent step (steps 1-8) for B independent
 * sequences, one token each.
 *   x [B][C], z [B][H_v*128], a_raw/b_raw [B][H_v]         (read)
 *   conv_state [B][3][C], S [B][H_v][128][128]             (read, updated in place)
 *   out [B][H_v*128], prenorm_out [B][H_v*128] or NULL     (written)
 * B == 0 is a no-op.  Inputs must not overlap outputs (other than the two
 * in/out states).
 */
gdn_status gdn_decode_step(const gdn_dims* dims, const gdn_weights* w, int32_t B,
                           const void* x, const void* z, const void* a_raw, const void* b_raw,
                           void* conv_state, void* S, void* out, float* prenorm_out,
                           int32_t* dev_status, gdn_stream_t stream);

/*
 * gdn_decode_step_ab -- gdn_decode_step with the ssm_alpha and ssm_beta
 * projections folded in (xwen CLAUDE.md page, "Architecture cheat sheet",
 * "Gated DeltaNet layer": a_raw = ssm_alpha(hidden), b_raw = ssm_beta(hidden)).
 * Instead of a_raw / b_raw the kernel reads the layer input and the two
 * weights and forms, for sequence b and v-head h,
 *   a_raw = sum_k hidden[b][k] W_a[h][k],   b_raw = sum_k hidden[b][k] W_b[h][k]
 * in fp32 from the bf16 operands, and uses them unrounded (gdn_in_proj rounds
 * its a_raw / b_raw outputs to bf16; here they never leave the chip).
 *   hidden [B][H] bf16; W_a, W_b [H_v][H] bf16 (the [out][in] layout of
 *   gdn_in_proj); H >= 8, H % 8 == 0 (else GDN_E_INVALID_ARG)
 * Requires act_dtype = GDN_BF16 (GDN_E_UNSUPPORTED otherwise).  Everything
 * else, including errors and dev_status, as gdn_decode_step.
 */
gdn_status gdn_decode_step_ab(const gdn_dims* dims, const gdn_weights* w, int32_t B, int32_t H,
                              const void* x, const void* z, const void* hidden, const void* W_a,
                              const void* W_b, void* conv_state, void* S, void* out,
                              float* prenorm_out, int32_t* dev_status, gdn_stream_t stream);

/*
 * gdn_verify_k -- speculative verify: B sequences, K tokens each (1 <=
 * GDN_MAX_VERIFY_K), token p of sequence b at row b*K + p.  Walks the
 * recurrence through the K tokens and keeps a state checkpoint after every
 * position (the page's "Drafting" section: verify-walk rollback from
 * per-position state planes; the NEXTN.md page's "GDN rollback").
 *   conv_state [B][3][C], S [B][H_v][128][128]             (read only)
 *   conv_ckpt [B][K][3][C], S_ckpt [B][K][H_v][128][128]   (written)
 *   out, prenorm_out [B*K][H_v*128]                        (written)
 * Checkpoint p is the state after consuming position p; it is bit-identical
 * to the state that p+1 calls of gdn_decode_step would leave.
 */
gdn_status gdn_verify_k(const gdn_dims* dims, const gdn_weights* w, int32_t B, int32_t K,
                        const void* x, const void* z, const void* a_raw, const void* b_raw,
                        const void* conv_state, const void* S, void* conv_ckpt, void* S_ckpt,
                        void* out, float* prenorm_out, int32_t* dev_status, gdn_stream_t stream);

/*
 * gdn_commit -- after a verify, make checkpoint accept_len[b]-1 the live state
 * of sequence b (bit-exact copy into conv_state[b] and S[b]).
 *   accept_len [B] int32 on the device, each in 1..K; a value outside that
 *   range leaves the sequence's state untouched.
 */
gdn_status gdn_commit(const gdn_dims* dims, int32_t B, int32_t K, const int32_t* accept_len,
                      const void* conv_ckpt, const void* S_ckpt, void* conv_state, void* S,
                      gdn_stream_t stream);

/*
 * State ring for speculative decoding, with a commit that copies no state.
 * The pages keep a state plane per drafted position so that a verify walk can
 * roll back (the page's "Drafting" section; the NEXTN.md page's "GDN
 * rollback"); gdn_verify_k + gdn_commit copy the accepted plane back into S.
 * With a ring the accepted plane becomes the live state where it lies.
 *   S_ring   [B][R][H_v][128][128] fp32 (bf16 under GDN_FLAG_STATE_BF16): R
 *            state slots per sequence
 *   ring_cur [B] int32 on the device: the live slot of each sequence, in 0..R-1
 * A caller starts from slot 0 holding the state (e.g. after a prefill into it)
 * and ring_cur all zero.
 *
 * gdn_verify_k_ring -- gdn_verify_k on the live slots: reads slot ring_cur[b],
 * writes checkpoint p to slot (ring_cur[b] + 1 + p) % R (K + 1 <= R <=
 * GDN_MAX_VERIFY_K + 1, so the live slot is never overwritten).  conv_state is
 * read and conv_ckpt [B][K][3][C] written as in gdn_verify_k; checkpoints,
 * outputs and conv checkpoints are bit-identical to gdn_verify_k's.
 */
gdn_status gdn_verify_k_ring(const gdn_dims* dims, const gdn_weights* w, int32_t B, int32_t K, int32_t R,
                             const void* x, const void* z, const void* a_raw, const void* b_raw,
                             const void* conv_state, void* S_ring, const int32_t* ring_cur, void* conv_ckpt,
                             void* out, float* prenorm_out, int32_t* dev_status, gdn_stream_t stream);

/*
 * gdn_commit_ring -- after gdn_verify_k_ring, accept accept_len[b] positions
 * (device int32 [B], each in 1..K): copies conv checkpoint accept_len[b]-1 into
 * conv_state[b] and sets ring_cur[b] = (ring_cur[b] + accept_len[b]) % R, the
 * slot of that state checkpoint.  A value outside 1..K leaves the sequence
 * untouched.  K and R as in the verify.
 */
gdn_status gdn_commit_ring(const gdn_dims* dims, int32_t B, int32_t K, int32_t R, const int32_t* accept_len,
                           const void* conv_ckpt, void* conv_state, int32_t* ring_cur, gdn_stream_t stream);

/*
 * gdn_decode_step_ring -- gdn_decode_step on the live slot of each sequence of
 * a ring (1 <= R <= GDN_MAX_VERIFY_K + 1), updated in place; bit-identical to
 * gdn_decode_step on that state.
 */
gdn_status gdn_decode_step_ring(const gdn_dims* dims, const gdn_weights* w, int32_t B, int32_t R, const void* x,
                                const void* z, const void* a_raw, const void* b_raw, void* conv_state, void* S_ring,
                                const int32_t* ring_cur, void* out, float* prenorm_out, int32_t* dev_status,
                                gdn_stream_t stream);

/*
 * Non-finite state guard (the home-server page's GDN state faults: a
 * non-finite recurrent state for one slot and two heads that stayed in the
 * cached state and was re-seeded on every later turn, while a report cap for
 * the life of the process had already silenced the fault reports).  The
 * detection is the dev_status word per (sequence, v-head) described above,
 * which every kernel ORs into under GDN_FLAG_CHECK_FINITE and which nothing
 * caps; these two calls read and act on those words.
 *
 * gdn_state_faults -- summarise dev_status [N*H_v] into report, int32
 * [2 + 2*cap] on the device: report[0] = the number of nonzero words (always
 * exact), report[1] = min(report[0], cap), then for i < report[1]:
 * report[2+2i] = n*H_v + h and report[3+2i] = its status bits, in increasing
 * index order.  The cap bounds only the listing.  dev_status is not changed.
 * GDN_E_INVALID_ARG for N < 0, cap < 0, N*H_v > INT32_MAX or overlapping
 * buffers.
 */
gdn_status gdn_state_faults(const gdn_dims* dims, int32_t N, const int32_t* dev_status, int32_t cap,
                            int32_t* report, gdn_stream_t stream);

/*
 * gdn_state_reset -- zero the recurrent state of every (n, h) whose
 * dev_status word is nonzero: the plane S[n][h], or with a state ring
 * (R >= 1 and ring_cur given) the live plane S_ring[n][ring_cur[n]][h]; when
 * conv_state is not NULL, also the conv rows of every sequence with at least
 * one such head.  Every dev_status word is then 0.  States of the other heads
 * and sequences are not touched.  R = 0 with ring_cur NULL for a plain
 * S [N][H_v][128][128]; anything else is GDN_E_INVALID_ARG.
 */
gdn_status gdn_state_reset(const gdn_dims* dims, int32_t N, int32_t R, void* S, const int32_t* ring_cur,
                           void* conv_state, int32_t* dev_status, gdn_stream_t stream);

/*
 * gdn_prefill_workspace_bytes -- device scratch that gdn_prefill_chunked needs
 * for n_seq sequences totalling T_total tokens (0 if none).
 */
size_t gdn_prefill_workspace_bytes(const gdn_dims* dims, int32_t n_seq, int64_t T_total);

/*
 * gdn_prefill_chunked -- the layer over n_seq packed sequences in chunked
 * form (chunk = 64; a sequence's last chunk may be partial).  Mathematically
 * equal to running gdn_decode_step token by token.
 *   cu_seqlens_host [n_seq+1]   HOST int32, non-decreasing, [0] = 0
 *   cu_seqlens_dev  [n_seq+1]   the same values on the device
 *   x [T][C], z [T][H_v*128], a_raw/b_raw [T][H_v]          (read)
 *   conv_state [n_seq][3][C], S [n_seq][H_v][128][128]      (updated in place;
 *                                   read only when zero_init == 0)
 *   zero_init != 0: the initial conv state and S are taken as zero (fresh
 *                   sequences) and are not read
 *   out, prenorm_out [T][H_v*128]                           (written)
 *   workspace of at least gdn_prefill_workspace_bytes() bytes (may be NULL
 *   when that is 0).
 */
gdn_status gdn_prefill_chunked(const gdn_dims* dims, const gdn_weights* w, int32_t n_seq,
                               const int32_t* cu_seqlens_host, const int32_t* cu_seqlens_dev,
                               const void* x, const void* z, const void* a_raw, const void* b_raw,
                               void* conv_state, void* S, int32_t zero_init, void* out,
                               float* prenorm_out, void* workspace, size_t workspace_bytes,
                               int32_t* dev_status, gdn_stream_t stream);

/*
 * Size in bytes of the fixed device scratch area behind
 * gdn_prefill_chunked_static (128 MiB).
 */
#define GDN_PREFILL_STATIC_SCRATCH_BYTES (128u * 1024u * 1024u)

/*
 * gdn_prefill_chunked_static -- gdn_prefill_chunked for callers that cannot
 * allocate device memory when they call it: a runtime whose allocator owns the
 * whole device pool, a plugin that is handed only its input and output
 * buffers, or code in a region where allocating is not allowed.  The pages
 * describe no such entry point; it is a convenience of this library.
 *
 * Arguments, layouts and results are those of gdn_prefill_chunked, without
 * the workspace.  The scratch comes instead from one area of
 * GDN_PREFILL_STATIC_SCRATCH_BYTES that the library declares statically in
 * device memory, so every GPU on which the library is used holds that area
 * until the process exits.  The call allocates and frees nothing.
 *
 * Limit: a problem whose gdn_prefill_workspace_bytes() exceeds
 * GDN_PREFILL_STATIC_SCRATCH_BYTES is rejected with GDN_E_WORKSPACE before
 * anything is enqueued (with bf16 activations and 48 v-heads, one sequence of
 * up to 1,280 tokens fits).  Calls that need no workspace (fp32 activations,
 * or GDN_FLAG_PREFILL_FP32) do not touch the area.
 *
 * Set-up: every call that needs the area looks up its device address on the
 * current device (cudaGetSymbolAddress, a host-side query; nothing is cached,
 * so the address stays right if the device's context is destroyed and created
 * again).  The first such call on a device can initialise the CUDA context
 * and load the library's device code; make that first call before any stream
 * capture.  A failed look-up returns GDN_E_CUDA.
 *
 * Sharing: every call uses the same area, which keeps the previous call's
 * contents; nothing in it has to start at zero, because each call writes
 * every byte it reads before reading it.  Calls whose work overlaps on the
 * GPU (two streams, or two host threads without ordering between their
 * streams) race on the area and corrupt each other's results: order them.
 */
gdn_status gdn_prefill_chunked_static(const gdn_dims* dims, const gdn_weights* w, int32_t n_seq,
                                      const int32_t* cu_seqlens_host, const int32_t* cu_seqlens_dev,
                                      const void* x, const void* z, const void* a_raw, const void* b_raw,
                                      void* conv_state, void* S, int32_t zero_init, void* out,
                                      float* prenorm_out, int32_t* dev_status, gdn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
