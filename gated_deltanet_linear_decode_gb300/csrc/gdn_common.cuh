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

// ---------------------------------------------------------------- folded a/b projections
// This thread's share of hidden . W_a and hidden . W_b (bf16 rows of H elements, H a
// multiple of 8, 16-byte aligned): the 8-element chunks i, i + step, ...  One fixed order
// of FMAs.  Returns (a part, b part).  kGlobal: the rows are in global memory (read
// through the read-only path), else in shared memory.
template <bool kGlobal>
__device__ __forceinline__ float2 ab_dot_part(const __nv_bfloat16* hid, const __nv_bfloat16* wa,
                                             const __nv_bfloat16* wb, int H, int i, int step) {
    auto ld = [](const __nv_bfloat16* row, int c) {
        const uint4* p = reinterpret_cast<const uint4*>(row) + c;
        if constexpr (kGlobal) return __ldg(p);
        else return *p;
    };
    float sa = 0.f, sb = 0.f;
    for (int c = i; c < (H >> 3); c += step) {
        const uint4 hv = ld(hid, c);
        const uint4 av = ld(wa, c);
        const uint4 bv = ld(wb, c);
        const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&hv);
        const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&av);
        const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&bv);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 hf = __bfloat1622float2(h2[e]), af = __bfloat1622float2(a2[e]), bf = __bfloat1622float2(b2[e]);
            sa = fmaf(hf.y, af.y, fmaf(hf.x, af.x, sa));
            sb = fmaf(hf.y, bf.y, fmaf(hf.x, bf.x, sb));
        }
    }
    return make_float2(sa, sb);
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

// ---------------------------------------------------------------- recurrent state storage
// Four consecutive state elements <-> a float4, for the two storage types
// (ld: a plain load through a generic pointer, global or shared memory).
// bf16 -> fp32 is exact (the bf16 bits are the upper half of the fp32
// pattern); fp32 -> bf16 rounds to nearest even.  round() gives the value a
// store followed by a load would give, so a walk that keeps the state in
// registers continues from exactly what a later call would read back.
// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialisation may start before the previous kernel in its stream has finished:
// grid_dependency_wait() returns once that kernel has completed and its writes are
// visible (at once when there is none), and grid_launch_dependents() lets the next
// such kernel start.  Kernels here wait before their first global access and let the
// next one start only after that, so at most two grids are resident at a time.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename Ts>
struct StateIO;

template <>
struct StateIO<float> {
    __device__ static __forceinline__ float4 ld_stream(const float* p) { return ld_f4_stream(p); }
    __device__ static __forceinline__ float4 ld(const void* p) { return *static_cast<const float4*>(p); }
    __device__ static __forceinline__ float4 round(float4 v) { return v; }
    __device__ static __forceinline__ void st(float* p, float4 v) { st_f4(p, v); }
    __device__ static __forceinline__ void st_shared(void* p, float4 v) { *static_cast<float4*>(p) = v; }
};

template <>
struct StateIO<__nv_bfloat16> {
    __device__ static __forceinline__ uint32_t pack(float lo, float hi) {
        const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&v);
    }
    __device__ static __forceinline__ float4 unpack(uint32_t a, uint32_t b) {
        return make_float4(__uint_as_float(a << 16), __uint_as_float(a & 0xffff0000u), __uint_as_float(b << 16),
                           __uint_as_float(b & 0xffff0000u));
    }
    __device__ static __forceinline__ float4 ld_stream(const __nv_bfloat16* p) {
        uint32_t a, b;
        asm volatile("ld.global.L1::no_allocate.v2.b32 {%0,%1}, [%2];" : "=r"(a), "=r"(b) : "l"(p));
        return unpack(a, b);
    }
    __device__ static __forceinline__ float4 ld(const void* p) {
        const uint2 v = *static_cast<const uint2*>(p);
        return unpack(v.x, v.y);
    }
    __device__ static __forceinline__ float4 round(float4 v) { return unpack(pack(v.x, v.y), pack(v.z, v.w)); }
    __device__ static __forceinline__ void st(__nv_bfloat16* p, float4 v) {
        asm volatile("st.global.v2.b32 [%0], {%1,%2};" ::"l"(p), "r"(pack(v.x, v.y)), "r"(pack(v.z, v.w)) : "memory");
    }
    __device__ static __forceinline__ void st_shared(void* p, float4 v) {
        *static_cast<uint2*>(p) = make_uint2(pack(v.x, v.y), pack(v.z, v.w));
    }
};

}  // namespace gdn
