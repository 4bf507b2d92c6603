// gdn_proj.cu -- the projections either side of the token mixer (include/gdn_proj.h):
// attn_qkv, attn_gate, ssm_alpha, ssm_beta before it and ssm_out after it (xwen CLAUDE.md
// page, "Architecture cheat sheet", "Gated DeltaNet layer").  They are dense GEMMs.  At
// decode-size batches (T <= 256) they are bound by the weight stream and run in the
// library's own weight-streaming kernel (gdn_proj_stream.cu: TMA + tcgen05, the four
// input GEMMs in one launch, K split over a cluster when there are few tiles); larger T
// is tensor-bound and runs through cuBLASLt (bf16 operands, fp32 accumulation).  This file is host code only: validation, dispatch, one
// cached cuBLASLt handle per device, and a cache of the chosen algorithm per shape.
#include <cublasLt.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <map>
#include <mutex>
#include <tuple>

#include "gdn.h"
#include "gdn_internal.h"
#include "gdn_proj.h"

namespace {

constexpr int kD = 128;
constexpr int kMaxDevices = 64;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Largest power of two (<= 256) dividing the address: the alignment cuBLASLt may assume.
uint32_t alignment_of(const void* p) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    uint32_t al = 256;
    while (al > 16 && (a & (al - 1)) != 0) al >>= 1;
    return al;
}

bool overlap(const void* a, size_t an, const void* b, size_t bn) {
    if (!a || !b || an == 0 || bn == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bn && b0 < a0 + an;
}

gdn_status check_proj_dims(const gdn_dims* d, int32_t T, int32_t H) {
    if (!d || d->H_k < 1 || d->H_v < 1 || d->H_k > 4096 || d->H_v > 4096 || d->H_v % d->H_k != 0)
        return GDN_E_INVALID_ARG;
    if (d->act_dtype != GDN_BF16 || d->out_dtype != GDN_BF16) return GDN_E_UNSUPPORTED;
    if (T < 0 || H < 8 || H % 8 != 0) return GDN_E_INVALID_ARG;
    return GDN_OK;
}

std::mutex g_mu;
cublasLtHandle_t g_handle[kMaxDevices] = {};
using AlgoKey = std::tuple<int, int, int, int, size_t, uint32_t, uint32_t, uint32_t>;
std::map<AlgoKey, cublasLtMatmulAlgo_t> g_algo;

// C[T][N] = A[T][K] . W[N][K]^T, all row-major bf16, fp32 accumulation.  In cuBLASLt's
// column-major terms: C^T (N x T) = op_T(W^T as K x N) . A^T (K x T).
gdn_status gemm_bf16(const void* A, const void* W, void* C, int T, int N, int K, void* ws, size_t wsb,
                     cudaStream_t stream) {
    if (T == 0) return GDN_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_E_CUDA;
    cublasLtHandle_t h;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_handle[dev] && cublasLtCreate(&g_handle[dev]) != CUBLAS_STATUS_SUCCESS) {
            g_handle[dev] = nullptr;
            return GDN_E_CUDA;
        }
        h = g_handle[dev];
    }
    cublasLtMatmulDesc_t op = nullptr;
    cublasLtMatrixLayout_t la = nullptr, lb = nullptr, lc = nullptr;
    cublasLtMatmulPreference_t pref = nullptr;
    gdn_status st = GDN_E_CUDA;
    const cublasOperation_t ta = CUBLAS_OP_T, tb = CUBLAS_OP_N;
    const uint32_t alW = alignment_of(W), alA = alignment_of(A), alC = alignment_of(C);
    do {
        if (cublasLtMatmulDescCreate(&op, CUBLAS_COMPUTE_32F, CUDA_R_32F) != CUBLAS_STATUS_SUCCESS) break;
        if (cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSA, &ta, sizeof ta) != CUBLAS_STATUS_SUCCESS ||
            cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSB, &tb, sizeof tb) != CUBLAS_STATUS_SUCCESS)
            break;
        if (cublasLtMatrixLayoutCreate(&la, CUDA_R_16BF, K, N, K) != CUBLAS_STATUS_SUCCESS ||
            cublasLtMatrixLayoutCreate(&lb, CUDA_R_16BF, K, T, K) != CUBLAS_STATUS_SUCCESS ||
            cublasLtMatrixLayoutCreate(&lc, CUDA_R_16BF, N, T, N) != CUBLAS_STATUS_SUCCESS)
            break;
        const AlgoKey key{dev, T, N, K, wsb, alW, alA, alC};
        cublasLtMatmulAlgo_t algo;
        bool have = false;
        {
            std::lock_guard<std::mutex> lk(g_mu);
            auto it = g_algo.find(key);
            if (it != g_algo.end()) { algo = it->second; have = true; }
        }
        if (!have) {
            if (cublasLtMatmulPreferenceCreate(&pref) != CUBLAS_STATUS_SUCCESS) break;
            const uint64_t wsb64 = wsb;
            cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &wsb64, sizeof wsb64);
            cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_A_BYTES, &alW, sizeof alW);
            cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_B_BYTES, &alA, sizeof alA);
            cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_C_BYTES, &alC, sizeof alC);
            cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_D_BYTES, &alC, sizeof alC);
            cublasLtMatmulHeuristicResult_t res = {};
            int n = 0;
            if (cublasLtMatmulAlgoGetHeuristic(h, op, la, lb, lc, lc, pref, 1, &res, &n) != CUBLAS_STATUS_SUCCESS ||
                n < 1)
                break;
            algo = res.algo;
            std::lock_guard<std::mutex> lk(g_mu);
            g_algo[key] = algo;
        }
        const float alpha = 1.0f, beta = 0.0f;
        if (cublasLtMatmul(h, op, &alpha, W, la, A, lb, &beta, C, lc, C, lc, &algo, ws, wsb, stream) !=
            CUBLAS_STATUS_SUCCESS)
            break;
        st = GDN_OK;
    } while (false);
    if (pref) cublasLtMatmulPreferenceDestroy(pref);
    if (lc) cublasLtMatrixLayoutDestroy(lc);
    if (lb) cublasLtMatrixLayoutDestroy(lb);
    if (la) cublasLtMatrixLayoutDestroy(la);
    if (op) cublasLtMatmulDescDestroy(op);
    return st;
}

}  // namespace

extern "C" {

gdn_status gdn_in_proj(const gdn_dims* dims, int32_t T, int32_t H, const void* hidden, const gdn_in_proj_weights* w,
                       void* x, void* z, void* a_raw, void* b_raw, void* workspace, size_t workspace_bytes,
                       int32_t* dev_status, gdn_stream_t stream) {
    gdn_status s = check_proj_dims(dims, T, H);
    if (s != GDN_OK) return s;
    if (T == 0) return GDN_OK;
    if (!w || !hidden || !w->W_qkv || !w->W_z || !w->W_a || !w->W_b || !x || !z || !a_raw || !b_raw ||
        (workspace_bytes > 0 && !workspace))
        return GDN_E_INVALID_ARG;
    const void* ptrs[] = {hidden, w->W_qkv, w->W_z, w->W_a, w->W_b, x, z, a_raw, b_raw};
    for (const void* p : ptrs)
        if (!aligned16(p)) return GDN_E_ALIGNMENT;
    if ((workspace && !aligned16(workspace)) || (dev_status && (reinterpret_cast<uintptr_t>(dev_status) & 3u)))
        return GDN_E_ALIGNMENT;
    const size_t Tz = static_cast<size_t>(T), Hz = static_cast<size_t>(H);
    const int C = kD * (2 * dims->H_k + dims->H_v), HvD = kD * dims->H_v, Hv = dims->H_v;
    const void* ins[] = {hidden, w->W_qkv, w->W_z, w->W_a, w->W_b};
    const size_t in_b[] = {Tz * Hz * 2, C * Hz * 2, HvD * Hz * 2, Hv * Hz * 2, Hv * Hz * 2};
    void* outs[] = {x, z, a_raw, b_raw, workspace};
    const size_t out_b[] = {Tz * C * 2, Tz * HvD * 2, Tz * Hv * 2, Tz * Hv * 2, workspace_bytes};
    for (int i = 0; i < 5; ++i) {
        for (int j = 0; j < 5; ++j)
            if (overlap(outs[i], out_b[i], ins[j], in_b[j])) return GDN_E_INVALID_ARG;
        for (int j = i + 1; j < 5; ++j)
            if (overlap(outs[i], out_b[i], outs[j], out_b[j])) return GDN_E_INVALID_ARG;
    }
    if (overlap(dev_status, 4, hidden, Tz * Hz * 2)) return GDN_E_INVALID_ARG;
    for (int i = 0; i < 5; ++i)
        if (overlap(dev_status, 4, outs[i], out_b[i])) return GDN_E_INVALID_ARG;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (T <= gdn::kProjStreamMaxRows) {
        const gdn::ProjGemm g[4] = {{w->W_qkv, x, C}, {w->W_z, z, HvD}, {w->W_a, a_raw, Hv}, {w->W_b, b_raw, Hv}};
        return gdn::launch_proj_stream(g, 4, hidden, T, H, dev_status, (dims->flags & GDN_FLAG_TEST_STALL) != 0, st) ==
                       cudaSuccess
                   ? GDN_OK
                   : GDN_E_CUDA;
    }
    if ((s = gemm_bf16(hidden, w->W_qkv, x, T, C, H, workspace, workspace_bytes, st)) != GDN_OK) return s;
    if ((s = gemm_bf16(hidden, w->W_z, z, T, HvD, H, workspace, workspace_bytes, st)) != GDN_OK) return s;
    if ((s = gemm_bf16(hidden, w->W_a, a_raw, T, Hv, H, workspace, workspace_bytes, st)) != GDN_OK) return s;
    return gemm_bf16(hidden, w->W_b, b_raw, T, Hv, H, workspace, workspace_bytes, st);
}

gdn_status gdn_out_proj(const gdn_dims* dims, int32_t T, int32_t H, const void* y, const void* W_out, void* out,
                        void* workspace, size_t workspace_bytes, int32_t* dev_status, gdn_stream_t stream) {
    gdn_status s = check_proj_dims(dims, T, H);
    if (s != GDN_OK) return s;
    if (T == 0) return GDN_OK;
    if (!y || !W_out || !out || (workspace_bytes > 0 && !workspace)) return GDN_E_INVALID_ARG;
    if (!aligned16(y) || !aligned16(W_out) || !aligned16(out) || (workspace && !aligned16(workspace)) ||
        (dev_status && (reinterpret_cast<uintptr_t>(dev_status) & 3u)))
        return GDN_E_ALIGNMENT;
    const size_t Tz = static_cast<size_t>(T), Hz = static_cast<size_t>(H);
    const int HvD = kD * dims->H_v;
    if (overlap(out, Tz * Hz * 2, y, Tz * HvD * 2) || overlap(out, Tz * Hz * 2, W_out, Hz * HvD * 2) ||
        overlap(workspace, workspace_bytes, y, Tz * HvD * 2) || overlap(workspace, workspace_bytes, W_out, Hz * HvD * 2) ||
        overlap(workspace, workspace_bytes, out, Tz * Hz * 2) || overlap(dev_status, 4, out, Tz * Hz * 2) ||
        overlap(dev_status, 4, y, Tz * HvD * 2))
        return GDN_E_INVALID_ARG;
    if (T <= gdn::kProjStreamMaxRows) {
        const gdn::ProjGemm g[1] = {{W_out, out, H}};
        return gdn::launch_proj_stream(g, 1, y, T, HvD, dev_status, (dims->flags & GDN_FLAG_TEST_STALL) != 0,
                                       reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
                   ? GDN_OK
                   : GDN_E_CUDA;
    }
    return gemm_bf16(y, W_out, out, T, H, HvD, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
