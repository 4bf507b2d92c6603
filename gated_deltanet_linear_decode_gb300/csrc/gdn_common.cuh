// gdn_common.cuh -- device helpers shared by the gated DeltaNet kernels
// (sm_103a).  Element loads/stores for the two activation dtypes, the gate
// functions of the layer, and thin inline-PTX wrappers for thread-block
// cluster barriers and distributed shared memory.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

constexpr int kD = 128;         // head dimension (d_k = d_v = 128)
constexpr int kConvW = 4;       // conv kernel width
constexpr int kChunk = 64;      // prefill chunk length
constexpr int kMaxK = 16;       // longest speculative verify walk
// 1/sqrt(128), rounded to fp32
constexpr float kInvSqrtD = 0.08838834764831845f;

// ---------------------------------------------------------------- dtype I/O
__device__ __forceinline__ float ld_act(const float* p) { return *p; }
__device__ __forceinline__ float ld_act(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ void st_out(float* p, float v) { *p = v; }
__device__ __forceinline__ void st_out(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// ---------------------------------------------------------------- gates (the layer's step 6 and the SiLU)
__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }
// log(1 + e^x) as max(x, 0) + log1p(e^-|x|): never overflows
__device__ __forceinline__ float softplusf_(float x) {
    return fmaxf(x, 0.0f) + log1pf(expf(-fabsf(x)));
}
__device__ __forceinline__ float siluf_(float x) { return x / (1.0f + expf(-x)); }

// Non-finite test on the bit pattern (exponent all ones): integer-only, so no
// floating-point assumption of the compiler can fold it away.
__device__ __forceinline__ bool nonfinite_bits(float v) {
    return (__float_as_uint(v) & 0x7f800000u) == 0x7f800000u;
}

// ---------------------------------------------------------------- warp reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Transposed butterfly reduction: each lane holds 32 partial sums v[0..31];
// afterwards v[0] of lane l is the sum over all 32 lanes of partial l
// (31 shuffles for 32 sums instead of 5 per sum).
__device__ __forceinline__ float reduce32_transposed(float (&v)[32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
            const float send = up ? v[i] : v[i + o];
            const float keep = up ? v[i + o] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return v[0];
}

// The same for 16 partial sums per lane: afterwards every lane l holds the
// sum over all 32 lanes of partial l % 16 (16 shuffles).
__device__ __forceinline__ float reduce16_transposed(float (&v)[16]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
            const float send = up ? v[i] : v[i + o];
            const float keep = up ? v[i + o] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 16);
}

// ---------------------------------------------------------------- clusters (PTX ISA: barrier.cluster, mapa, ld.shared::cluster)
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Read a float from the shared memory of CTA `rank` of this cluster, at the
// same offset as `local` has in this CTA.
__device__ __forceinline__ float ld_dsmem_f32(const float* local, uint32_t rank) {
    uint32_t la = static_cast<uint32_t>(__cvta_generic_to_shared(local));
    uint32_t ra;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(la), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
    return v;
}

// ---------------------------------------------------------------- streaming 128-bit global access
__device__ __forceinline__ float4 ld_f4_stream(const float* p) {
    float4 v;
    asm volatile("ld.global.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ void st_f4(float* p, float4 v) {
    asm volatile("st.global.v4.f32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w) : "memory");
}

}  // namespace gdn
