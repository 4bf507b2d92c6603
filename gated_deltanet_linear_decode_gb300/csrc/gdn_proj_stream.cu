// gdn_proj_stream.cu -- the projections either side of the token mixer at decode-size
// batches (T <= 256 rows of input): out[t][n] = sum_k in[t][k] W[n][k], bf16 operands,
// fp32 accumulation, bf16 out (xwen CLAUDE.md page, "Architecture cheat sheet", "Gated
// DeltaNet layer": attn_qkv, attn_gate, ssm_alpha, ssm_beta before the mixer, ssm_out
// after it).
//
// At these sizes the GEMM is bound by streaming the weights from HBM (each weight is
// used by only T <= 256 rows), and one SM takes in only about 1/150 of the HBM bandwidth,
// so the weight stream must be spread over the SMs.  A tile is 128 weight rows (the MMA's
// M; the batch rows are its N).  With about as many tiles as SMs each CTA streams one
// tile's whole K; with fewer, the S CTAs of a cluster (S = 2 or 4) split a tile's K and
// add their partial sums through distributed shared memory.
//   * One thread streams the [128 x 64] boxes of W and [N x 64] boxes of the input by TMA
//     (2-D tensor maps, 128-byte swizzle, zero fill past the edges) into a ring of stages;
//     one thread issues the tcgen05 MMAs (A = the W box, B = the input box, both K-major,
//     the accumulator [128 rows x N] in tensor memory) and releases each stage by
//     tcgen05.commit; four warps read the accumulator out.
//   * All the GEMMs of one call that share the input (attn_qkv, attn_gate, ssm_alpha,
//     ssm_beta) run as one launch over a common list of tiles.
//   * Launched as a programmatic dependent of the previous kernel in the stream: the first
//     stages' weight boxes are requested before griddepcontrol.wait (the weights are not
//     written by the kernels before it), the input boxes and every store after it.
// Every wait is bounded; a wait that gives up stops the CTA's copies and MMAs, lets what
// it issued complete, writes no output and sets bit 4 of the optional status word.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_tc.cuh"

namespace gdn {

namespace {

constexpr int kRowsPerTile = 128;   // weight rows per tile (the MMA's M)
constexpr int kBK = 64;             // K elements per k-block: one 128-byte swizzle row
constexpr int kWBoxBytes = kRowsPerTile * kBK * 2;
constexpr int kThreads = 192;       // warps 0-3 read out, warp 4 copies, warp 5 issues MMAs
constexpr int kWaitLimit = 1 << 22;
constexpr int kStallLimit = 1 << 12;   // polls of the test stall
constexpr int kMaxSegs = 4;

struct ProjSeg {
    void* out;    // [T][rows] bf16
    int rows;
    int tile0;    // first tile of this GEMM in the launch's tile list
};

struct alignas(64) ProjParams {
    CUtensorMap wmap[kMaxSegs];   // W of each GEMM: [rows][K] bf16, box 64 x 128
    CUtensorMap xmap;             // input [T][K] bf16, box 64 x npad
    ProjSeg seg[kMaxSegs];
    int n_seg, T, npad, n_kb, splits, stages, stage_bytes, tmem_cols;
    int* status;                  // optional: bit 4 when a wait gave up
    int test_stall;               // GDN_FLAG_TEST_STALL: the MMA thread first waits on a barrier nothing arrives on
};

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Shared-memory address of `local` in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_rank(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
// No memory clobber: consecutive loads issue back to back (the cluster barrier orders them).
__device__ __forceinline__ float4 ld_cluster_v4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr));
    return v;
}
__device__ __forceinline__ int ld_cluster_s32(uint32_t addr) {
    int v;
    asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__global__ void __launch_bounds__(kThreads, 1) proj_stream_kernel(const __grid_constant__ ProjParams p) {
    extern __shared__ __align__(1024) uint8_t sm_raw[];
    // the 128-byte swizzle pattern repeats every 1024 bytes: base the stages there
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = p.splits, stages = p.stages;
    const int tile = blockIdx.x / S;
    const int split = S > 1 ? static_cast<int>(cluster_rank()) : 0;
    int s = 0;
    while (s + 1 < p.n_seg && p.seg[s + 1].tile0 <= tile) ++s;
    const int r0 = (tile - p.seg[s].tile0) * kRowsPerTile;
    const int rows = p.seg[s].rows;
    const int kb0 = split * p.n_kb / S, kb1 = (split + 1) * p.n_kb / S, nk = kb1 - kb0;   // nk >= 1 (host)

    uint64_t* full = reinterpret_cast<uint64_t*>(sm + stages * p.stage_bytes);
    uint64_t* empty = full + stages;
    uint64_t* done = empty + stages;   // every MMA of this CTA has completed
    uint64_t* never = done + 1;        // test stall: nothing arrives
    uint32_t* tslot = reinterpret_cast<uint32_t*>(never + 1);
    int* bad = reinterpret_cast<int*>(tslot + 1);

    // producer (warp 4, lane 0): k-block kb0 + i into stage i mod stages
    const bool producer = warp == 4 && lane == 0;
    const void* wmap = &p.wmap[s];
    int issued = 0;
    auto issue_w = [&](int i) {
        const int st = i % stages;
        tc::mbar_expect_tx(full + st, static_cast<uint32_t>(p.stage_bytes));
        tc::tma_load_2d(sm + st * p.stage_bytes, wmap, (kb0 + i) * kBK, r0, full + st);
    };
    auto issue_x = [&](int i) {
        const int st = i % stages;
        tc::tma_load_2d(sm + st * p.stage_bytes + kWBoxBytes, &p.xmap, (kb0 + i) * kBK, 0, full + st);
    };
    if (producer) {
        for (int i = 0; i < stages; ++i) {
            tc::mbar_init(full + i, 1);
            tc::mbar_init(empty + i, 1);
        }
        tc::mbar_init(done, 1);
        tc::mbar_init(never, 1);
        *bad = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        // the first stages' weight boxes go out before anything else (they do not depend on
        // the previous kernel); the input boxes once that kernel's writes are visible
        for (; issued < nk && issued < stages; ++issued) issue_w(issued);
        grid_dependency_wait();
        for (int i = 0; i < issued; ++i) issue_x(i);
    }
    if (warp == 5) tc::tmem_alloc(tslot, static_cast<uint32_t>(p.tmem_cols));
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    grid_launch_dependents();
    const uint32_t tmem = *tslot;

    if (producer) {
        // refill each stage as soon as the MMAs have read it; stop once another role gave up
        for (int i = issued; i < nk; ++i) {
            bool got = false;
            for (int k = 0; k < kWaitLimit / 256 && !got; ++k) {
                if (*reinterpret_cast<volatile int*>(bad)) break;
                got = tc::mbar_wait(empty + i % stages, ((i / stages) & 1) ^ 1, 256);
            }
            if (!got) {
                atomicExch(bad, 1);
                break;
            }
            issue_w(i);
            issue_x(i);
            issued = i + 1;
        }
        if (*reinterpret_cast<volatile int*>(bad)) {
            // let the copies still in flight land before the CTA can leave
            for (int i = issued - stages > 0 ? issued - stages : 0; i < issued; ++i)
                tc::mbar_wait(full + i % stages, (i / stages) & 1, kWaitLimit);
        }
    } else if (warp == 5 && lane == 0) {
        const uint32_t idesc = tc::idesc_bf16(kRowsPerTile, p.npad);
        bool fail = p.test_stall && !tc::mbar_wait(never, 0, kStallLimit);
        for (int i = 0; i < nk && !fail; ++i) {
            const int st = i % stages;
            if (!tc::mbar_wait(full + st, (i / stages) & 1, kWaitLimit)) {
                fail = true;
                break;
            }
            tc::fence_after_sync();
            const uint32_t a = tc::smem_u32(sm + st * p.stage_bytes), b = a + kWBoxBytes;
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
                tc::mma_f16(tmem, tc::sdesc_sw128(a + 32 * kk), tc::sdesc_sw128(b + 32 * kk), idesc, (i | kk) != 0);
            tc::mma_commit(empty + st);   // the stage is free once these MMAs have read it
        }
        if (fail) {
            atomicExch(bad, 1);   // before the read-out can see the MMAs complete
            __threadfence_block();
        }
        tc::mma_commit(done);     // every MMA issued above has completed
    }

    // read-out: warp w holds weight rows 32w .. 32w+31 of the tile (tensor-memory lanes)
    if (warp < 4) {
        if (!tc::mbar_wait(done, 0, kWaitLimit)) atomicExch(bad, 1);
        tc::fence_after_sync();
        grid_dependency_wait();   // no store before the previous kernel is done with its reads
    }
    __syncthreads();   // the copy and MMA roles are through; `bad` is final for this CTA
    const bool ok = *reinterpret_cast<volatile int*>(bad) == 0;
    const int nl = 32 * warp + lane;   // this thread's row of the tile (warps 0-3)
    const int n = r0 + nl;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.seg[s].out);
    const uint32_t trow = tmem + (static_cast<uint32_t>(32 * warp) << 16);

    if (S == 1) {
        if (warp < 4) {
            if (ok) {
                for (int c0 = 0; c0 < p.npad; c0 += 16) {
                    float v[16];
                    tc::tmem_ld16(trow + c0, v);
                    if (n < rows) {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (c0 + j < p.T) out[static_cast<size_t>(c0 + j) * rows + n] = __float2bfloat16_rn(v[j]);
                    }
                }
            } else if (tid == 0 && p.status) {
                atomicOr(p.status, 16);
            }
        }
    } else {
        // partial sums -> this CTA's shared memory (the stages are idle now), [row][npad + 4]:
        // 16-byte rows whose float4 stores from 8 consecutive rows hit distinct banks
        const int ld = p.npad + 4;
        float* red = reinterpret_cast<float*>(sm);
        if (warp < 4 && ok) {
            for (int c0 = 0; c0 < p.npad; c0 += 16) {
                float v[16];
                tc::tmem_ld16(trow + c0, v);
#pragma unroll
                for (int j = 0; j < 16; j += 4)
                    *reinterpret_cast<float4*>(red + nl * ld + c0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
            }
        }
        cluster_sync();   // every partial of the tile is in place
        // CTA `split` adds rows [split * 128/S, (split+1) * 128/S) over the cluster
        bool all_ok = true;
        for (int q = 0; q < S; ++q) all_ok = all_ok && ld_cluster_s32(map_rank(tc::smem_u32(bad), q)) == 0;
        if (tid < 128) {
            const int share = kRowsPerTile / S;
            const uint32_t red_base = tc::smem_u32(red);
            if (all_ok) {
                // thread: one row, four consecutive t; the S partials of a float4 load together
                const int nq = (p.T + 3) / 4;
                for (int idx = tid; idx < share * nq; idx += 128) {
                    const int rl = split * share + idx % share, t0 = 4 * (idx / share);
                    const uint32_t off = red_base + static_cast<uint32_t>((rl * ld + t0) * 4);
                    float4 v[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (q < S) v[q] = ld_cluster_v4(map_rank(off, q));
                    float4 acc = v[0];
#pragma unroll
                    for (int q = 1; q < 4; ++q)
                        if (q < S) acc = make_float4(acc.x + v[q].x, acc.y + v[q].y, acc.z + v[q].z, acc.w + v[q].w);
                    if (r0 + rl < rows) {
                        const float a4[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (t0 + j < p.T) out[static_cast<size_t>(t0 + j) * rows + r0 + rl] = __float2bfloat16_rn(a4[j]);
                    }
                }
            } else if (tid == 0 && p.status) {
                atomicOr(p.status, 16);
            }
        }
        cluster_sync();   // no CTA leaves while another still reads its partials
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 5) tc::tmem_dealloc(tmem, static_cast<uint32_t>(p.tmem_cols));
}

int sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return sms;
}

}  // namespace

cudaError_t launch_proj_stream(const ProjGemm* g, int n_gemm, const void* in, int T, int K, int* status,
                               bool test_stall, cudaStream_t stream) {
    if (n_gemm < 1 || n_gemm > kMaxSegs || T < 1 || T > kProjStreamMaxRows || K < 8 || K % 8 != 0)
        return cudaErrorInvalidValue;
    const int sms = sm_count();
    if (sms < 1) return cudaErrorInvalidDevice;
    ProjParams p;
    memset(&p, 0, sizeof p);
    p.npad = (T + 15) / 16 * 16;
    p.T = T;
    p.n_kb = (K + kBK - 1) / kBK;
    p.n_seg = n_gemm;
    p.status = status;
    p.test_stall = test_stall ? 1 : 0;
    int tiles = 0;
    for (int i = 0; i < n_gemm; ++i) {
        if (g[i].rows < 1) return cudaErrorInvalidValue;
        p.seg[i].out = g[i].out;
        p.seg[i].rows = g[i].rows;
        p.seg[i].tile0 = tiles;
        tiles += (g[i].rows + kRowsPerTile - 1) / kRowsPerTile;
        if (!make_tensor_map_bf16_sw128(&p.wmap[i], g[i].W, K, g[i].rows, kRowsPerTile)) return cudaErrorInvalidValue;
    }
    if (!make_tensor_map_bf16_sw128(&p.xmap, in, K, T, p.npad)) return cudaErrorInvalidValue;
    // K split over a cluster of S = 2 or 4 CTAs while the tiles x S CTAs still fit one per SM
    // and each split keeps at least two k-blocks (clusters of 8 did not all fit at once)
    int S = 1;
    while (S < 4 && tiles * S * 2 <= sms && p.n_kb >= 4 * S) S *= 2;
    p.splits = S;
    // one CTA per SM, its shared memory a deep ring of stages (the partial sums of a split
    // reuse it: 128 x (npad + 4) floats fit in the stages for every npad <= 256)
    p.stage_bytes = kWBoxBytes + p.npad * kBK * 2;
    p.stages = 200 * 1024 / p.stage_bytes;
    if (p.stages > 16) p.stages = 16;
    if (p.stages < 2) p.stages = 2;
    int cols = 32;
    while (cols < p.npad) cols *= 2;
    p.tmem_cols = cols;
    const size_t smem = 1024 + static_cast<size_t>(p.stages) * p.stage_bytes + (2 * p.stages + 2) * 8 + 16;
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(proj_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(smem))) != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(tiles * S));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(S);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, proj_stream_kernel, p);
}

}  // namespace gdn
