/*
 * gdn_proj.h -- the dense projections either side of the gated DeltaNet token
 * mixer of libgdn.so (include/gdn.h), for a caller that holds the layer's
 * hidden state instead of the mixer's inputs.
 *
 * Source: xwen CLAUDE.md page, "Architecture cheat sheet (Qwen 3.6, ggml-org
 * GGUF)", "Gated DeltaNet layer": the layer input goes through attn_qkv (the
 * fused q|k|v stream), attn_gate (z), ssm_alpha (a_raw) and ssm_beta (b_raw);
 * the gated RMSNorm output goes through ssm_out.  Hidden sizes on that page:
 * 5120 (27B, 16/48 heads) and 2048 (35B-A3B, 16/32 heads).
 *
 * Both calls are bf16 GEMMs with fp32 accumulation on the tensor cores
 * (out = in . W^T, W in the [out][in] layout of a linear layer's weight),
 * each output element rounded once to bf16 from its fp32 sum.  For T <= 256
 * (decode and speculative-verify batches: the weights are read once and used
 * by few rows, so the time is the weight stream) they run in the library's
 * own weight-streaming kernel: 128-row tiles of W and the input streamed by
 * TMA into shared memory, tcgen05 MMAs into tensor memory, K split over a
 * cluster of 2 or 4 CTAs whose partial sums meet in distributed shared
 * memory when there are fewer tiles than SMs; gdn_in_proj's four GEMMs share
 * one launch.  The kernel is launched as a programmatic dependent of the
 * previous kernel in the stream: it starts streaming the weights while that
 * kernel finishes, and reads the input and writes the outputs only after it
 * (so the weights must not be written by the kernel just before the call in
 * the stream; a copy or any earlier kernel is ordered as usual).  For T > 256 they run
 * through cuBLASLt (tensor-bound; one cuBLASLt handle per device is created
 * on first use and kept for the life of the process).  The order in which
 * the fp32 sums are formed differs between the two paths.
 *
 * Conventions as in gdn.h: caller-owned, 16-byte aligned device buffers,
 * asynchronous on `stream`, errors returned, outputs must not overlap inputs.
 * Requires act_dtype = out_dtype = GDN_BF16 (GDN_E_UNSUPPORTED otherwise).
 * The workspace is optional scratch for cuBLASLt at T > 256 (NULL / 0
 * allowed; a few MiB lets it pick faster kernels; the streaming kernel needs
 * none); the library allocates no device memory.
 * dev_status (optional, may be NULL) is one int32: the weight-streaming kernel
 * ORs bit 4 into it when one of its bounded waits gave up (its outputs are
 * then not written); the caller zeroes it and reads it after synchronising.
 */
#ifndef GDN_PROJ_H
#define GDN_PROJ_H

#include "gdn.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    const void* W_qkv;  /* [C][H]       attn_qkv,  C = 128*(2*H_k + H_v)  bf16 */
    const void* W_z;    /* [H_v*128][H] attn_gate                          bf16 */
    const void* W_a;    /* [H_v][H]     ssm_alpha                          bf16 */
    const void* W_b;    /* [H_v][H]     ssm_beta                           bf16 */
} gdn_in_proj_weights;

/*
 * gdn_in_proj -- the mixer's inputs from T rows of the hidden state:
 *   hidden [T][H]  ->  x [T][C], z [T][H_v*128], a_raw [T][H_v], b_raw [T][H_v]
 * (four GEMMs; each output element rounded once from its fp32 sum).
 * T == 0 is a no-op.  GDN_E_INVALID_ARG for T < 0, H < 8 or H % 8 != 0, null
 * pointers or overlaps; GDN_E_ALIGNMENT for a device pointer off 16 bytes
 * (dev_status: 4); GDN_E_CUDA if a launch fails, or cuBLASLt fails or finds
 * no kernel.
 */
gdn_status gdn_in_proj(const gdn_dims* dims, int32_t T, int32_t H, const void* hidden,
                       const gdn_in_proj_weights* w, void* x, void* z, void* a_raw, void* b_raw,
                       void* workspace, size_t workspace_bytes, int32_t* dev_status,
                       gdn_stream_t stream);

/*
 * gdn_out_proj -- ssm_out: y [T][H_v*128] (the mixer's out)  ->  out [T][H],
 * W_out [H][H_v*128] bf16.  Errors as gdn_in_proj.
 */
gdn_status gdn_out_proj(const gdn_dims* dims, int32_t T, int32_t H, const void* y, const void* W_out,
                        void* out, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                        gdn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_PROJ_H */
