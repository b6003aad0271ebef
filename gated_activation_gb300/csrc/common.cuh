// Internal helpers shared by the library's translation units (device side
// bf16 packing, streaming loads, warp reductions; host side argument checks
// and device facts).  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "gated_act.h"

namespace gact {

// ---------------------------------------------------------------- device side

// 8 bf16 values = one 16-byte vector, kept packed as four bf16x2 words.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Round two floats to bf16 (nearest even) and pack them, lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// 16-byte load of data that is read once: read-only path, no L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const void *p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ld_stream_u32(const uint32_t *p) {
    uint32_t r;
    asm("ld.global.nc.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ uint16_t ld_stream_u16(const uint16_t *p) {
    uint16_t r;
    asm("ld.global.nc.u16 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ void st_vec(void *p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// st_vec for an output that nothing else in the kernel reads or writes through
// another pointer: without the memory clobber the compiler may move other
// loads (a table read, a shared-memory read) across the store, so the reads
// of consecutive vectors overlap.  Volatile asm statements keep their order.
__device__ __forceinline__ void st_vec_out(void *p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
}

// Programmatic dependent launch.  Every kernel of the library waits for the
// preceding grid in its stream to finish (and its memory to be visible)
// before it touches global memory, and then lets the next PDL-launched grid
// in the stream begin launching, so that grid's launch latency and set-up
// overlap this one's tail.  Both are no-ops for a launch without the
// programmatic-serialization attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Paired fp32 arithmetic (PTX add/sub/mul/fma .f32x2 on sm_100 and later):
// one instruction for two lanes, each rounded as its scalar form would be.
__device__ __forceinline__ unsigned long long u64_of(float2 v) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(v.x), "f"(v.y));
    return r;
}
__device__ __forceinline__ float2 f2_of(unsigned long long r) {
    float2 v;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
    return v;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(u64_of(a)), "l"(u64_of(b)));
    return f2_of(d);
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
    unsigned long long d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(u64_of(a)), "l"(u64_of(b)));
    return f2_of(d);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(u64_of(a)), "l"(u64_of(b)));
    return f2_of(d);
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(u64_of(a)), "l"(u64_of(b)), "l"(u64_of(c)));
    return f2_of(d);
}

// Butterfly sum: every lane ends with the same bits (fp add is commutative
// and each step pairs the same two operands in both partner lanes).
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// ---------------------------------------------------------------- host side

// Per-device facts, queried once per device and cached.
int device_sm_count();

// Programmatic dependent launch is on unless the environment variable
// GATED_ACT_PDL is "0" when the library makes its first launch.
bool pdl_enabled();

// Launch `kernel` on `stream` with programmatic stream serialization (when
// enabled) and, for cluster > 1, a 1-D cluster of that many CTAs.
template <typename... Exp, typename... Act>
cudaError_t launch_kernel(void (*kernel)(Exp...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, int cluster, Act &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = static_cast<unsigned>(cluster);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (pdl_enabled()) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Act &&>(args)...);
}

// Record a CUDA error for gated_act_last_cuda_error() and map it to a status.
int cuda_status(cudaError_t e);

// The address kernels use for `p`: device (and managed) memory as is;
// page-locked host memory through its device mapping.  Sets *host when the
// bytes live in host memory.  Returns GATED_ACT_OK, or GATED_ACT_ERR_HOST for
// an address the runtime does not know (pageable memory, no allocation).
int resolve_ptr(const void *p, const void **dev, bool *host);

inline bool aligned(const void *p, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

// True when [a, a + na) and [b, b + nb) (byte ranges) intersect.
inline bool ranges_overlap(const void *a, uint64_t na, const void *b, uint64_t nb) {
    uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    if (na == 0 || nb == 0)
        return false;
    return x < y + nb && y < x + na;
}

}  // namespace gact
