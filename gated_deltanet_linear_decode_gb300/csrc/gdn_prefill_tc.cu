// gdn_prefill_tc.cu -- the tensor-core chunked prefill (bf16 activations) as
// one persistent kernel with two roles that run side by side:
//   * preparation CTAs (gdn_prefill_prep.cuh) take (chunk, q/k head) items in
//     chunk order from a global counter (the first chunk as one item per
//     v-head) and write, for every v-head of the q/k head's group, the chunk's
//     state-independent record (W^T, U, Q', K', P, decay vectors), setting each
//     v-head's ready flag as soon as its record is complete;
//   * chain CTAs (gdn_prefill_chain.cuh) each walk the chunks of one
//     (sequence, v-head) at a time, the state on chip, reading every record as
//     soon as its flag is set -- while it is still in L2 -- and dropping it from
//     L2 once consumed, so that records need not reach HBM.
// Method: xwen CLAUDE.md page, "Ground truth" (chunk = 64 form of the delta
// rule), "Architecture cheat sheet", "Gated DeltaNet layer".
//
// Chain CTAs wait on preparation CTAs (never the reverse), so the kernel is
// launched cooperatively: every CTA is resident at once (one per SM at most,
// by its shared memory), and every wait is bounded.
#include "gdn_internal.h"
#include "gdn_prefill_chain.cuh"
#include "gdn_prefill_prep.cuh"

namespace gdn {

namespace {

// Exclusive prefix of the per-sequence chunk counts: chunk_base[s] is the
// global index of sequence s's first chunk, chunk_base[n_seq] the total.  Also
// clears the ready flags [n_flags], the consumed counters [n_consumed] and
// the item counter and abort flag of this call.
__global__ void chunk_table_kernel(const int* cu_seqlens, int n_seq, int* chunk_base, int* ready, int n_flags,
                                   int* consumed, int n_consumed, int* counter) {
    // launched as a programmatic dependent: the previous kernel (a prefill of the same
    // workspace, for one) is done before anything is cleared
    grid_dependency_wait();
    grid_launch_dependents();
    __shared__ int carry_s;
    __shared__ int warp_s[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    for (int i = tid; i < n_flags; i += blockDim.x) ready[i] = 0;
    for (int i = tid; i < n_consumed; i += blockDim.x) consumed[i] = 0;
    if (tid == 0) {
        carry_s = 0;
        counter[0] = 0;   // item counter
        counter[1] = 0;   // abort flag
    }
    __syncthreads();
    for (int base = 0; base < n_seq; base += blockDim.x) {
        const int i = base + tid;
        const int cnt = i < n_seq ? (cu_seqlens[i + 1] - cu_seqlens[i] + kChunk - 1) / kChunk : 0;
        int v = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int up = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += up;
        }
        if (lane == 31) warp_s[warp] = v;
        __syncthreads();
        if (warp == 0) {
            int w = lane < nw ? warp_s[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int up = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += up;
            }
            if (lane < nw) warp_s[lane] = w;   // inclusive over warps
        }
        __syncthreads();
        const int carry = carry_s;
        const int incl = v + (warp > 0 ? warp_s[warp - 1] : 0) + carry;
        if (i < n_seq) chunk_base[i] = incl - cnt;
        __syncthreads();
        if (tid == blockDim.x - 1) carry_s = incl;
        __syncthreads();
    }
    if (tid == 0) chunk_base[n_seq] = carry_s;
}

// 512 threads: the preparation role's 16 warps; the chain role uses the first 14.
constexpr int kThreads = 512;
static_assert(kThreads >= prep::kPrepThreads && kThreads >= chain::kStateThreads, "the roles' warps");

// The preparation role bases its map on the next 1024-byte boundary (the 128-byte swizzle
// of its TMA boxes repeats every 1024 bytes), hence the extra 1024 bytes.
__host__ __device__ inline uint32_t fused_smem(int G) {
    return prep::smem_bytes(G) + 1024 > chain::kStateSmem ? prep::smem_bytes(G) + 1024 : chain::kStateSmem;
}

// CTAs [0, n_chain) run chains j = blockIdx.x, blockIdx.x + n_chain, ... of the
// n_seq * H_v (sequence-major); the others take preparation items.
template <typename Tout>
__global__ void __launch_bounds__(kThreads, 1) prefill_fused_kernel(const __grid_constant__ PrefillParams p, int n_chain,
                                                                    int* counter) {
    extern __shared__ __align__(1024) uint8_t sm[];
    __shared__ int item_s;
    const int tid = threadIdx.x, warp = tid >> 5;
    // launched as a programmatic dependent of the chunk-table kernel: nothing global (nor the
    // tensor memory) is touched before it is done
    grid_dependency_wait();
    grid_launch_dependents();
    if (static_cast<int>(blockIdx.x) < n_chain) {
        if (warp >= chain::kStateThreads / 32) return;   // the chain role runs on warps 0-13
        uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + chain::kBar + 8 * chain::kNumBars);
        if (warp == 0) tc::tmem_alloc(tslot, chain::kTmemCols);
        tc::fence_before_sync();
        chain::chain_sync();
        tc::fence_after_sync();
        const uint32_t tmem = *tslot;
        const int n_chains = p.n_seq * p.Hv;
        for (int j = blockIdx.x; j < n_chains; j += n_chain) chain::run<Tout>(p, j / p.Hv, j % p.Hv, sm, tmem);
        tc::fence_before_sync();
        chain::chain_sync();
        tc::fence_after_sync();
        if (warp == 0) tc::tmem_dealloc(tmem, chain::kTmemCols);
        return;
    }
    if (warp >= prep::kPrepThreads / 32) return;   // the preparation role runs on warps 0-7
    uint8_t* smp = sm + ((1024u - (tc::smem_u32(sm) & 1023u)) & 1023u);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smp + prep::kMisc);
    uint64_t* mbar = reinterpret_cast<uint64_t*>(smp + prep::kMisc + 8);
    int* err_s = reinterpret_cast<int*>(smp + prep::kMisc + 16);
    uint64_t* xbar = reinterpret_cast<uint64_t*>(smp + prep::kMisc + 24);
    uint64_t* vbar = reinterpret_cast<uint64_t*>(smp + prep::kMisc + 32);
    if (warp == 0) tc::tmem_alloc(tslot, prep::kPrepTmemCols);
    if (tid == 0) {
        tc::mbar_init(mbar, 1);
        tc::mbar_init(xbar, 1);
        tc::mbar_init(vbar, 1);
        *err_s = 0;
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.xmap)) : "memory");
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tc::fence_before_sync();
    pf::prep_sync();
    tc::fence_after_sync();
    prep::Ctx cx{*tslot, mbar, 0u, err_s, false, xbar, vbar, 0u, 0u};
    // items in chunk order, so every chain finds its next chunk among the earliest: first the
    // call's chunk 0 as one item per v-head (its chains start after one head's work), then
    // (chunk, q/k head) items of all the v-heads of the group
    const int G = p.Hv / p.Hk;
    const int n_first = p.Hv;
    const int n_items = n_first + (p.n_chunks - 1) * p.Hk;
    for (;;) {
        if (tid == 0) item_s = atomicAdd(counter, 1);
        pf::prep_sync();
        const int it = item_s;   // read by all before thread 0 can write the next one (the item syncs first)
        if (it >= n_items) break;
        if (it < n_first)
            prep::item(p, 0, it % p.Hk, it / p.Hk, it / p.Hk + 1, smp, cx);
        else
            prep::item(p, 1 + (it - n_first) / p.Hk, (it - n_first) % p.Hk, 0, G, smp, cx);
    }
    tc::fence_before_sync();
    pf::prep_sync();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(cx.tmem, prep::kPrepTmemCols);
}

// Workspace layout: chunk table, ready flags, consumed counters, item counter, records.
size_t flags_bytes(size_t n_chunks_bound, int Hk) { return (n_chunks_bound * Hk * 4 + 255) / 256 * 256; }

}  // namespace

// A sequence of L tokens has ceil(L/64) <= L/64 + 1 chunks, so T/64 + n_seq
// chunks bound every packing of T tokens.
size_t tc_prefill_workspace_bytes(int Hk, int Hv, int n_seq, long long T) {
    const size_t nc = static_cast<size_t>((T + kChunk - 1) / kChunk) + static_cast<size_t>(n_seq);
    return pf::table_bytes(n_seq) + flags_bytes(nc, Hv) + flags_bytes(nc, Hk) + 256 +
           nc * static_cast<size_t>(Hv) * pf::kVRec;
}

void tc_prefill_bind_workspace(PrefillParams& p) {
    const size_t nc = static_cast<size_t>((p.T + kChunk - 1) / kChunk) + static_cast<size_t>(p.n_seq);
    uint8_t* base = static_cast<uint8_t*>(p.workspace);
    p.chunk_base = reinterpret_cast<int*>(base);
    base += pf::table_bytes(p.n_seq);
    p.ready = reinterpret_cast<int*>(base);
    base += flags_bytes(nc, p.Hv);
    p.consumed = reinterpret_cast<int*>(base);
    base += flags_bytes(nc, p.Hk);
    p.ws_v = base + 256;   // the item counter and the abort flag sit in the 256 bytes before the records
    p.abort_flag = reinterpret_cast<int*>(p.ws_v - 256) + 1;
}

cudaError_t launch_tensor_core_prefill(const PrefillParams& p0, int out_dtype, cudaStream_t stream) {
    PrefillParams p = p0;
    p.chunk_lo = 0;
    p.chunk_hi = p.n_chunks;
    int* counter = reinterpret_cast<int*>(p.ws_v - 256);
    // the raw rows of a chunk (positions c0-3 .. c0+63) come in by TMA, 64 channels a box
    if (!make_tensor_map_bf16_sw128(&p.xmap, p.x, p.C, static_cast<int>(p.T), prep::kXrows)) return cudaErrorInvalidValue;
    int dev = 0, sms = 0, l2 = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev)) != cudaSuccess) return e;
    const int n_chains = p.n_seq * p.Hv;
    const int n_items = p.Hv + (p.n_chunks - 1) * p.Hk;
    // One chain per CTA while the chains take at most half the SMs; beyond that, one
    // v-head per chain CTA (every CTA then walks every sequence once), or a third of
    // the SMs.  The preparation role takes the rest, and at least one SM.
    int n_chain = n_chains <= sms / 2 ? n_chains : (p.Hv <= sms / 2 ? p.Hv : sms / 3);
    n_chain = n_chain < 1 ? 1 : n_chain;
    int n_prep = sms - n_chain;
    if (n_prep > n_items) n_prep = n_items;
    if (n_prep < 1) n_prep = 1;
    const int grid = n_chain + n_prep;
    const uint32_t smem = fused_smem(p.Hv / p.Hk);

    // Records of at most `ahead` chunks in flight, about 9/16 of L2, so that they stay in L2
    // between the preparation CTA that writes them and the chain that reads them (the rest
    // of L2 holds the activations and outputs streaming past).  Measured at T = 8192 on
    // 48 v-heads: DRAM traffic 1.07 GB unthrottled, 0.44 GB at 9/16, time within 3 %.
    // The gate needs every v-head of a sequence walked at once (each chain CTA then
    // meets the chunks in global order); with fewer chain CTAs than v-heads a chain may
    // start only after another has finished its sequence, so there is no gate.
    if (n_chain >= p.Hv) {
        p.ahead = static_cast<int>(static_cast<size_t>(l2) / 16 * 9 / (static_cast<size_t>(p.Hv) * pf::kVRec));
        if (p.ahead < 4) p.ahead = 4;
    } else {
        p.ahead = p.n_chunks;   // gc < n_chunks: never gated
    }
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1);
        cfg.blockDim = dim3(256);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see grid_dependency_wait
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if ((e = cudaLaunchKernelEx(&cfg, chunk_table_kernel, static_cast<const int*>(p.cu_seqlens), p.n_seq,
                                    p.chunk_base, p.ready, p.n_chunks * p.Hv, p.consumed, p.n_chunks * p.Hk,
                                    counter)) != cudaSuccess)
            return e;
    }

    auto go = [&](auto kernel) -> cudaError_t {
        cudaError_t r = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (r != cudaSuccess) return r;
        // cooperative (every CTA resident at once: chains wait on preparation CTAs) and a
        // programmatic dependent of the chunk-table kernel
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(grid));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        r = cudaLaunchKernelEx(&cfg, kernel, p, n_chain, counter);
        if (r == cudaErrorInvalidValue || r == cudaErrorNotSupported) {   // the pair refused: a plain cooperative launch
            (void)cudaGetLastError();
            cfg.numAttrs = 1;
            r = cudaLaunchKernelEx(&cfg, kernel, p, n_chain, counter);
        }
        return r;
    };
    return out_dtype == 1 ? go(prefill_fused_kernel<__nv_bfloat16>) : go(prefill_fused_kernel<float>);
}

}  // namespace gdn
