// silu_and_mul for sm_103a: out = silu(gate) * up over [M, 2d] bf16 rows.
//
// Megatron-LM PR "Size MoE activation kernel grid to the row count",
// sections "What changed and why" and "Correctness": a pure elementwise op
// whose cost is launch geometry.  Here the grid is sized to the work (every
// thread owns kVecPerThread 16-byte output vectors, all loads issued before
// any math) rather than capped.  Per element the math is fp32 and independent
// of the geometry, so any grid gives the same bits.
#include <algorithm>

#include "common.cuh"

namespace gact {
namespace {

constexpr int kSiluThreads = 256;
constexpr int kVecPerThread = 2;

// silu(g) * u in fp32 as g * sigmoid(g), with the sigmoid taken from
// t = e^-|g| (never overflows): 1 / (1 + t) for g >= 0, t / (1 + t) below.
// The naive 1 / (1 + e^-g) overflows for g < -88.7 and returns -0 where the
// true product is still a normal bf16 number.
// e^x = 2^(x log2 e) on the hardware base-2 exponential (PTX ISA ex2.approx.f32,
// the non-flushing form: subnormal results survive, which keeps silu(g) for
// g in (-104, -87] a normal bf16 number instead of -0).
__device__ __forceinline__ float exp_neg_abs(float g) {
    const float x = -fabsf(g) * 1.4426950408889634f;
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 1 + t lies in (1, 2], where the hardware reciprocal (PTX ISA rcp.approx.f32)
// is within one fp32 ulp; the bf16 result tolerates far more.
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float silu_mul(float g, float u) {
    const float t = exp_neg_abs(g);
    const float r = rcp_approx(1.0f + t);
    return g * (g >= 0.f ? r : t * r) * u;
}

__device__ __forceinline__ uint32_t silu2(uint32_t g, uint32_t u) {
    return pack_bf16x2(silu_mul(bf16_lo(g), bf16_lo(u)), silu_mul(bf16_hi(g), bf16_hi(u)));
}

// Thread t of the grid owns 16-byte output vectors t, t + S, t + 2S, ...
// (S = all threads of the grid; consecutive threads take consecutive vectors,
// so every warp access is one contiguous run).  The first vector's (row,
// column) costs one division; each later one steps by (step_r, step_c) =
// (S / nv, S mod nv) with a carry, so the loop has no division.
__global__ void __launch_bounds__(kSiluThreads)
silu_vec(uint16_t *__restrict__ out, const uint16_t *__restrict__ in, int64_t M, int64_t nv,
         int64_t step_r, int64_t step_c, int64_t d) {
    pdl_wait();
    pdl_trigger();
    const int64_t first = static_cast<int64_t>(blockIdx.x) * kSiluThreads + threadIdx.x;
    int64_t r = first / nv, c = first - r * nv;
    int64_t rr[kVecPerThread], cc[kVecPerThread];
    uint4 g[kVecPerThread], u[kVecPerThread];
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) {
        rr[i] = r;
        cc[i] = c;
        if (r < M) {
            const uint16_t *gp = in + r * 2 * d + 8 * c;
            g[i] = ld_stream(gp);
            u[i] = ld_stream(gp + d);
        }
        r += step_r;
        c += step_c;
        if (c >= nv) {
            c -= nv;
            ++r;
        }
    }
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) {
        if (rr[i] < M) {
            const uint4 o = make_uint4(silu2(g[i].x, u[i].x), silu2(g[i].y, u[i].y),
                                       silu2(g[i].z, u[i].z), silu2(g[i].w, u[i].w));
            st_vec(out + rr[i] * d + 8 * cc[i], o);
        }
    }
}

// Any layout: one element per thread iteration, 2-byte accesses.
__global__ void __launch_bounds__(kSiluThreads)
silu_scalar(uint16_t *__restrict__ out, const uint16_t *__restrict__ in, int64_t M, int64_t d) {
    const int64_t total = M * d;
    const int64_t step = static_cast<int64_t>(gridDim.x) * kSiluThreads;
    pdl_wait();
    pdl_trigger();
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * kSiluThreads + threadIdx.x; e < total;
         e += step) {
        const int64_t r = e / d, c = e - r * d;
        const uint16_t *gp = in + r * 2 * d + c;
        const float g = __uint_as_float(static_cast<uint32_t>(ld_stream_u16(gp)) << 16);
        const float u = __uint_as_float(static_cast<uint32_t>(ld_stream_u16(gp + d)) << 16);
        out[e] = __bfloat16_as_ushort(__float2bfloat16_rn(silu_mul(g, u)));
    }
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace
}  // namespace gact

extern "C" int silu_and_mul(void *out, const void *in, int64_t M, int64_t d,
                            cudaStream_t stream) {
    using namespace gact;
    if (M < 0 || d <= 0)
        return GATED_ACT_ERR_SIZE;
    if (d > (int64_t(1) << 30) || M > (int64_t(1) << 40))
        return GATED_ACT_ERR_TOO_LARGE;
    if (M == 0)
        return GATED_ACT_OK;
    if (!out || !in)
        return GATED_ACT_ERR_NULL;
    if (!aligned(out, 2) || !aligned(in, 2))
        return GATED_ACT_ERR_ALIGN;
    const uint64_t out_bytes = 2ull * static_cast<uint64_t>(M * d);
    if (ranges_overlap(out, out_bytes, in, 2 * out_bytes))
        return GATED_ACT_ERR_OVERLAP;

    uint16_t *o = static_cast<uint16_t *>(out);
    const uint16_t *x = static_cast<const uint16_t *>(in);
    const bool vec_ok = aligned(in, 16) && aligned(out, 16) && d % 8 == 0;
    if (vec_ok) {
        const int64_t nv = d / 8, total = M * nv;
        const int64_t grid = ceil_div(ceil_div(total, kVecPerThread), kSiluThreads);
        if (grid > 0x7FFFFFFF)
            return GATED_ACT_ERR_TOO_LARGE;
        const int64_t S = grid * kSiluThreads;
        const cudaError_t e =
            launch_kernel(silu_vec, dim3(static_cast<unsigned>(grid)), dim3(kSiluThreads), 0,
                          stream, 1, o, x, M, nv, S / nv, S % nv, d);
        if (e != cudaSuccess)
            return cuda_status(e);
    } else {
        const int64_t grid = std::min<int64_t>(ceil_div(M * d, kSiluThreads), int64_t(1) << 20);
        const cudaError_t e = launch_kernel(silu_scalar, dim3(static_cast<unsigned>(grid)),
                                            dim3(kSiluThreads), 0, stream, 1, o, x, M, d);
        if (e != cudaSuccess)
            return cuda_status(e);
    }
    return cuda_status(cudaGetLastError());
}
