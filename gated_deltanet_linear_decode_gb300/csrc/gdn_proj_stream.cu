// gdn_proj_stream.cu -- the projections either side of the token mixer at decode-size
// batches (T <= 256 rows of input): out[t][n] = sum_k in[t][k] W[n][k], bf16 operands,
// fp32 accumulation, bf16 out (xwen CLAUDE.md page, "Architecture cheat sheet", "Gated
// DeltaNet layer": attn_qkv, attn_gate, ssm_alpha, ssm_beta before the mixer, ssm_out
// after it).
//
// At these sizes the GEMM is bound by streaming the weights from HBM (each weight is
// used by only T <= 256 rows), and one SM ingests only about 1/152 of the HBM bandwidth,
// so every SM must stream an equal share.  The work is a list of k-blocks: 128 weight rows
// (a tile: the MMA's M; the batch rows are its N) x 64 of K, tile-major over all the
// GEMMs of the call.  CTA c of G takes the k-blocks [c*total/G, (c+1)*total/G): one or
// more runs ("segments") of consecutive k-blocks of a tile.
//   * One thread streams each k-block's [128 x 64] box of W and [N x 64] box of the input
//     by TMA (2-D tensor maps, 128-byte swizzle, zero fill past the edges) into a ring of
//     stages; one thread issues the tcgen05 MMAs (A = the W box, B = the input box, both
//     K-major) into one of two accumulators [128 rows x N] in tensor memory (one per
//     segment, alternating) and releases each stage by tcgen05.commit; four warps read
//     the accumulator out.
//   * A segment that is a whole tile writes its outputs.  Otherwise its fp32 partial sums
//     go to the workspace and it adds its k-block count to the tile's counter; the CTA
//     that completes the count adds the tile's partials and writes the outputs (then
//     clears the counter).  Without a workspace, or with about as many tiles as SMs (the
//     split would cost more than the idle SMs), each CTA takes one whole tile (G = tiles).
// Every wait is bounded; a wait that gives up stops the CTA's copies and MMAs, lets what
// it issued complete, writes no output and sets bit 4 of the optional status word.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "gdn_internal.h"
#include "gdn_tc.cuh"

namespace gdn {

namespace {

constexpr int kRowsPerTile = 128;   // weight rows per tile (the MMA's M)
constexpr int kBK = 64;             // K elements per k-block: one 128-byte swizzle row
constexpr int kWBoxBytes = kRowsPerTile * kBK * 2;
constexpr int kThreads = 192;       // warps 0-3 read out, warp 4 copies, warp 5 issues MMAs
constexpr int kWaitLimit = 1 << 22;
constexpr int kMaxSegs = 4;
constexpr int kMaxParts = 4;        // target runs per tile when a tile's K is split

struct ProjSeg {
    void* out;    // [T][rows] bf16
    int rows;
    int tile0;    // first tile of this GEMM in the launch's tile list
};

struct alignas(64) ProjParams {
    CUtensorMap wmap[kMaxSegs];   // W of each GEMM: [rows][K] bf16, box 64 x 128
    CUtensorMap xmap;             // input [T][K] bf16, box 64 x npad
    ProjSeg seg[kMaxSegs];
    int n_seg, T, npad, n_kb, tiles, stages, stage_bytes, tmem_cols;
    long long total;              // tiles * n_kb
    float* partial;               // [tiles][max_parts][npad][128] fp32 (workspace), or null
    int* counter;                 // [tiles] (workspace, zero at launch), or null
    int max_parts;
    int* status;                  // optional: bit 4 when a wait gave up
    int test_stall;               // GDN_FLAG_TEST_STALL: the MMA thread first waits on a barrier nothing arrives on
};

constexpr int kStallLimit = 1 << 12;   // polls of the test stall

__device__ __forceinline__ long long first_block(long long c, long long total, int G) { return c * total / G; }
// The CTA whose range holds k-block x: the largest c with first_block(c) <= x.
__device__ __forceinline__ int owner(long long x, long long total, int G) {
    return static_cast<int>(((x + 1) * G + total - 1) / total - 1);
}

__global__ void __launch_bounds__(kThreads, 1) proj_stream_kernel(const __grid_constant__ ProjParams p) {
    extern __shared__ __align__(1024) uint8_t sm_raw[];
    // the 128-byte swizzle pattern repeats every 1024 bytes: base the stages there
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int stages = p.stages, G = gridDim.x, n_kb = p.n_kb;
    const long long b0 = first_block(blockIdx.x, p.total, G), b1 = first_block(blockIdx.x + 1, p.total, G);
    const int nk = static_cast<int>(b1 - b0);   // >= 1: the host keeps G <= total

    uint64_t* full = reinterpret_cast<uint64_t*>(sm + stages * p.stage_bytes);
    uint64_t* empty = full + stages;
    uint64_t* done = empty + stages;    // [2]: accumulator b of a segment is complete
    uint64_t* freed = done + 2;         // [2]: the read-out is done with accumulator b
    uint64_t* drain = freed + 2;        // every MMA of this CTA has completed
    uint64_t* never = drain + 1;        // test stall: nothing arrives
    uint32_t* tslot = reinterpret_cast<uint32_t*>(never + 1);
    int* bad = reinterpret_cast<int*>(tslot + 1);
    int* last_s = bad + 1;

    // producer (warp 4, lane 0): the i-th k-block of this CTA into stage i mod stages
    const bool producer = warp == 4 && lane == 0;
    int issued = 0;
    auto issue = [&](int i) {
        const long long x = b0 + i;
        const int tile = static_cast<int>(x / n_kb), kb = static_cast<int>(x % n_kb);
        int g = 0;
        while (g + 1 < p.n_seg && p.seg[g + 1].tile0 <= tile) ++g;
        const int st = i % stages;
        uint8_t* buf = sm + st * p.stage_bytes;
        tc::mbar_expect_tx(full + st, static_cast<uint32_t>(p.stage_bytes));
        tc::tma_load_2d(buf, &p.wmap[g], kb * kBK, (tile - p.seg[g].tile0) * kRowsPerTile, full + st);
        tc::tma_load_2d(buf + kWBoxBytes, &p.xmap, kb * kBK, 0, full + st);
    };
    if (producer) {
        for (int i = 0; i < stages; ++i) {
            tc::mbar_init(full + i, 1);
            tc::mbar_init(empty + i, 1);
        }
        tc::mbar_init(done, 1);
        tc::mbar_init(done + 1, 1);
        tc::mbar_init(freed, 128);
        tc::mbar_init(freed + 1, 128);
        tc::mbar_init(drain, 1);
        tc::mbar_init(never, 1);
        *bad = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        // the first stages' copies go out before the CTA-wide set-up below
        for (; issued < nk && issued < stages; ++issued) issue(issued);
    }
    if (warp == 5) tc::tmem_alloc(tslot, static_cast<uint32_t>(p.tmem_cols));
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tslot;

    if (producer) {
        // refill each stage as soon as the MMAs have read it
        for (int i = issued; i < nk; ++i) {
            // wait for the stage in short polls, stopping as soon as another role gave up
            bool got = false;
            for (int k = 0; k < kWaitLimit / 256 && !got; ++k) {
                if (*reinterpret_cast<volatile int*>(bad)) break;
                got = tc::mbar_wait(empty + i % stages, ((i / stages) & 1) ^ 1, 256);
            }
            if (!got) {
                atomicExch(bad, 1);
                break;
            }
            issue(i);
            issued = i + 1;
        }
        if (*reinterpret_cast<volatile int*>(bad)) {
            // let the copies still in flight land before the CTA can leave
            for (int i = issued - stages > 0 ? issued - stages : 0; i < issued; ++i)
                tc::mbar_wait(full + i % stages, (i / stages) & 1, kWaitLimit);
        }
    } else if (warp == 5 && lane == 0) {
        // MMA issue: segment j accumulates into columns (j & 1) * npad
        const uint32_t idesc = tc::idesc_bf16(kRowsPerTile, p.npad);
        int i = 0, j = 0;
        bool fail = false;
        if (p.test_stall && !tc::mbar_wait(never, 0, kStallLimit)) {
            atomicExch(bad, 1);   // before the read-out can see segment 0 complete
            __threadfence_block();
            tc::mma_commit(done);
            fail = true;
        }
        while (i < nk && !fail) {
            const long long x = b0 + i;
            const int kb = static_cast<int>(x % n_kb);
            const int len = static_cast<int>(n_kb - kb < nk - i ? n_kb - kb : nk - i);
            const int buf = j & 1;
            // the read-out of segment j - 2 is done with this accumulator
            if (j >= 2 && !tc::mbar_wait(freed + buf, ((j >> 1) - 1) & 1, kWaitLimit)) {
                atomicExch(bad, 1);   // before the read-out can see segment j complete
                __threadfence_block();
                tc::mma_commit(done + buf);
                fail = true;
                break;
            }
            tc::fence_after_sync();
            const uint32_t acc = tmem + static_cast<uint32_t>(buf * p.npad);
            for (int q = 0; q < len; ++q, ++i) {
                const int st = i % stages;
                if (!tc::mbar_wait(full + st, (i / stages) & 1, kWaitLimit)) {
                    fail = true;
                    break;
                }
                tc::fence_after_sync();
                const uint32_t a = tc::smem_u32(sm + st * p.stage_bytes), b = a + kWBoxBytes;
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk)
                    tc::mma_f16(acc, tc::sdesc_sw128(a + 32 * kk), tc::sdesc_sw128(b + 32 * kk), idesc, (q | kk) != 0);
                tc::mma_commit(empty + st);   // the stage is free once these MMAs have read it
            }
            if (fail) {
                atomicExch(bad, 1);   // before the read-out can see segment j complete
                __threadfence_block();
            }
            tc::mma_commit(done + buf);       // segment j complete (or drained, flagged bad)
            ++j;
        }
        // nothing leaves (and tensor memory is not released) with an MMA in flight
        tc::mma_commit(drain);
        if (!tc::mbar_wait(drain, 0, kWaitLimit)) atomicExch(bad, 1);
    } else if (warp < 4) {
        // read-out: warp w holds weight rows 32w .. 32w+31 of the tile (tensor-memory lanes)
        const int nl = 32 * warp + lane;
        int i = 0, j = 0;
        while (i < nk) {
            const long long x = b0 + i;
            const int tile = static_cast<int>(x / n_kb), kb = static_cast<int>(x % n_kb);
            const int len = static_cast<int>(n_kb - kb < nk - i ? n_kb - kb : nk - i);
            const int buf = j & 1;
            const bool got = tc::mbar_wait(done + buf, (j >> 1) & 1, kWaitLimit);
            tc::fence_after_sync();
            // every read-out thread passed the wait and no role gave up
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (!got) atomicExch(bad, 1);
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (*reinterpret_cast<volatile int*>(bad)) {
                if (tid == 0 && p.status) atomicOr(p.status, 16);
                break;
            }
            int g = 0;
            while (g + 1 < p.n_seg && p.seg[g + 1].tile0 <= tile) ++g;
            const int rows = p.seg[g].rows;
            const int n = (tile - p.seg[g].tile0) * kRowsPerTile + nl;
            __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.seg[g].out);
            const uint32_t trow = tmem + (static_cast<uint32_t>(32 * warp) << 16) + static_cast<uint32_t>(buf * p.npad);
            const bool whole = kb == 0 && len == n_kb;
            if (whole) {
                for (int c0 = 0; c0 < p.npad; c0 += 16) {
                    float v[16];
                    tc::tmem_ld16(trow + c0, v);
                    if (n < rows) {
#pragma unroll
                        for (int q = 0; q < 16; ++q)
                            if (c0 + q < p.T) out[static_cast<size_t>(c0 + q) * rows + n] = __float2bfloat16_rn(v[q]);
                    }
                }
            } else {
                // part `part` of the tile's segments: partial [t][row] (rows contiguous)
                const long long tb = static_cast<long long>(tile) * n_kb;
                const int c_first = owner(tb, p.total, G);
                const int part = static_cast<int>(blockIdx.x) - c_first;
                const int n_parts = owner(tb + n_kb - 1, p.total, G) - c_first + 1;
                float* mine = p.partial + (static_cast<size_t>(tile) * p.max_parts + part) * p.npad * kRowsPerTile;
                for (int c0 = 0; c0 < p.npad; c0 += 16) {
                    float v[16];
                    tc::tmem_ld16(trow + c0, v);
#pragma unroll
                    for (int q = 0; q < 16; ++q) mine[static_cast<size_t>(c0 + q) * kRowsPerTile + nl] = v[q];
                }
                // the read-out's partial stores, then (one thread, cumulative through the
                // barrier) a release to the GPU and the count; the last part acquires
                asm volatile("bar.sync 1, 128;" ::: "memory");
                if (tid == 0) {
                    __threadfence();
                    *last_s = atomicAdd(p.counter + tile, len) + len == n_kb;
                    __threadfence();
                }
                asm volatile("bar.sync 1, 128;" ::: "memory");
                if (*reinterpret_cast<volatile int*>(last_s)) {
                    // the tile's last part: add the parts (warp w: tokens w, w+4, ..; lane: 4 rows)
                    const float4* base = reinterpret_cast<const float4*>(
                        p.partial + static_cast<size_t>(tile) * p.max_parts * p.npad * kRowsPerTile);
                    const int n0 = (tile - p.seg[g].tile0) * kRowsPerTile + 4 * lane;
                    // 16 tokens at a time, their loads of one part issued together
                    for (int k0 = warp; k0 < p.T; k0 += 64) {
                        float4 acc[16];
#pragma unroll
                        for (int k = 0; k < 16; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                        for (int q = 0; q < n_parts; ++q) {
                            const float4* part_q = base + static_cast<size_t>(q) * p.npad * (kRowsPerTile / 4) + lane;
#pragma unroll
                            for (int k = 0; k < 16; ++k) {
                                const int t = k0 + 4 * k;
                                if (t < p.T) {
                                    const float4 v = __ldcg(part_q + static_cast<size_t>(t) * (kRowsPerTile / 4));
                                    acc[k].x += v.x;
                                    acc[k].y += v.y;
                                    acc[k].z += v.z;
                                    acc[k].w += v.w;
                                }
                            }
                        }
#pragma unroll
                        for (int k = 0; k < 16; ++k) {
                            const int t = k0 + 4 * k;
                            if (t >= p.T) break;
                            const float a4[4] = {acc[k].x, acc[k].y, acc[k].z, acc[k].w};
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                if (n0 + e < rows) out[static_cast<size_t>(t) * rows + n0 + e] = __float2bfloat16_rn(a4[e]);
                        }
                    }
                    if (tid == 0) p.counter[tile] = 0;   // ready for the next call
                }
            }
            tc::fence_before_sync();
            tc::mbar_arrive(freed + buf);
            i += len;
            ++j;
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 5) tc::tmem_dealloc(tmem, static_cast<uint32_t>(p.tmem_cols));
}

// 2-D bf16 tensor [outer][inner] (row pitch inner * 2 bytes), box [box_outer][64], 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int inner, int outer, int box_outer) {
    return make_tensor_map_bf16_sw128(m, base, inner, outer, box_outer);
}

}  // namespace

namespace {

// The launch's k-block partition: G CTAs over tiles * n_kb k-blocks.
struct ProjPlan {
    int tiles, n_kb, npad, G, max_parts;
    long long total;
    size_t counter_bytes, ws_bytes;
};

ProjPlan plan_of(const int* rows, int n_gemm, int T, int K, int sms, bool split) {
    ProjPlan q;
    q.tiles = 0;
    for (int i = 0; i < n_gemm; ++i) q.tiles += (rows[i] + kRowsPerTile - 1) / kRowsPerTile;
    q.n_kb = (K + kBK - 1) / kBK;
    q.npad = (T + 15) / 16 * 16;
    q.total = static_cast<long long>(q.tiles) * q.n_kb;
    // every SM streams an equal share (at least two k-blocks a CTA, a tile in at most about
    // kMaxParts runs, since one CTA adds a tile's parts), or whole tiles
    if (split && q.tiles * 5 < sms * 3) {   // fewer tiles than about 0.6 x SMs: spread K as well
        long long G = sms;
        if (G > q.total / 2) G = q.total / 2;
        if (G > static_cast<long long>(q.tiles) * kMaxParts) G = static_cast<long long>(q.tiles) * kMaxParts;
        q.G = static_cast<int>(G);
    } else {
        q.G = q.tiles;
    }
    if (q.G < 1) q.G = 1;
    q.max_parts = 1;
    for (int t = 0; t < q.tiles; ++t) {
        const long long x0 = static_cast<long long>(t) * q.n_kb, x1 = x0 + q.n_kb - 1;
        const long long c0 = ((x0 + 1) * q.G + q.total - 1) / q.total - 1, c1 = ((x1 + 1) * q.G + q.total - 1) / q.total - 1;
        if (c1 - c0 + 1 > q.max_parts) q.max_parts = static_cast<int>(c1 - c0 + 1);
    }
    q.counter_bytes = (static_cast<size_t>(q.tiles) * 4 + 255) / 256 * 256;
    q.ws_bytes = q.counter_bytes + static_cast<size_t>(q.tiles) * q.max_parts * q.npad * kRowsPerTile * 4;
    return q;
}

int sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return sms;
}

}  // namespace

size_t proj_stream_workspace_bytes(const int* rows, int n_gemm, int T, int K) {
    const int sms = sm_count();
    if (sms < 1 || T < 1 || T > kProjStreamMaxRows || K < 8) return 0;
    return plan_of(rows, n_gemm, T, K, sms, true).ws_bytes;
}

cudaError_t launch_proj_stream(const ProjGemm* g, int n_gemm, const void* in, int T, int K, void* workspace,
                               size_t workspace_bytes, int* status, bool test_stall, cudaStream_t stream) {
    if (n_gemm < 1 || n_gemm > kMaxSegs || T < 1 || T > kProjStreamMaxRows || K < 8 || K % 8 != 0)
        return cudaErrorInvalidValue;
    const int sms = sm_count();
    if (sms < 1) return cudaErrorInvalidDevice;
    int rows[kMaxSegs];
    for (int i = 0; i < n_gemm; ++i) {
        if (g[i].rows < 1) return cudaErrorInvalidValue;
        rows[i] = g[i].rows;
    }
    ProjPlan q = plan_of(rows, n_gemm, T, K, sms, true);
    const bool split = workspace && workspace_bytes >= q.ws_bytes;
    if (!split) q = plan_of(rows, n_gemm, T, K, sms, false);

    ProjParams p;
    memset(&p, 0, sizeof p);
    p.npad = q.npad;
    p.T = T;
    p.n_kb = q.n_kb;
    p.n_seg = n_gemm;
    p.tiles = q.tiles;
    p.total = q.total;
    p.max_parts = q.max_parts;
    p.status = status;
    p.test_stall = test_stall ? 1 : 0;
    int tiles = 0;
    for (int i = 0; i < n_gemm; ++i) {
        p.seg[i].out = g[i].out;
        p.seg[i].rows = g[i].rows;
        p.seg[i].tile0 = tiles;
        tiles += (g[i].rows + kRowsPerTile - 1) / kRowsPerTile;
        if (!make_map(&p.wmap[i], g[i].W, K, g[i].rows, kRowsPerTile)) return cudaErrorInvalidValue;
    }
    if (!make_map(&p.xmap, in, K, T, p.npad)) return cudaErrorInvalidValue;
    cudaError_t e;
    if (split && q.G != q.tiles) {   // some tile is split between CTAs
        p.counter = static_cast<int*>(workspace);
        p.partial = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + q.counter_bytes);
        if ((e = cudaMemsetAsync(p.counter, 0, static_cast<size_t>(q.tiles) * 4, stream)) != cudaSuccess) return e;
    }
    // one CTA per SM, its shared memory a deep ring of stages
    p.stage_bytes = kWBoxBytes + p.npad * kBK * 2;
    p.stages = 200 * 1024 / p.stage_bytes;
    if (p.stages > 16) p.stages = 16;
    if (p.stages < 2) p.stages = 2;
    int cols = 32;
    while (cols < 2 * p.npad) cols *= 2;   // two accumulators of npad columns
    p.tmem_cols = cols;
    const size_t smem = 1024 + static_cast<size_t>(p.stages) * p.stage_bytes + (2 * p.stages + 6) * 8 + 16;
    if ((e = cudaFuncSetAttribute(proj_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(smem))) != cudaSuccess)
        return e;
    proj_stream_kernel<<<q.G, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
