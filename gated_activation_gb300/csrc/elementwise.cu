// Row-wise elementwise activations for sm_103a, one kernel template:
//
//   silu_and_mul          out = silu(g) * u           Megatron-LM PR "Size MoE
//                         activation kernel grid to the row count", "What
//                         changed and why";
//   silu_and_mul_bounded  the same over the first n_rows rows only, n_rows
//                         read on the device (same section: the grid is fixed
//                         by the capture-time bound M, CTAs past the live rows
//                         exit early);
//   squared_relu          out = max(x, 0)^2, not gated (same page, "Scope and
//                         risks": the sibling activation kernel);
//   gelu_and_mul          out = gelu_tanh(g) * u, the dense form of the
//                         sparse-GELU page's activation.
//
// The cost of these ops is launch geometry (the MoE-activation page's
// finding): the grid is sized to the work, never capped.  A CTA owns
// contiguous blocks of VPT * 256 16-byte output vectors; thread t takes
// vectors t, t + 256, ... of a block, so every warp access is one contiguous
// run, all loads are issued before any math, and blocks past the live rows
// are skipped.  VPT = 1 for small launches (more CTAs, so more SMs start
// loading at once: measured on GB300, silu_and_mul at M = 256..4096, d = 768
// 3-13% faster), 2 from 2^20 output vectors on (1-3% faster there).
// Launches below 2^31 - 512 vectors index them in 32 bits (ew_vec32), larger
// ones in 64 bits (ew_vec).  The bounded kernel's one wave of CTAs walks
// blocks of 256 (VPT = 1): 8-25% faster than blocks of 512 at 256..16384
// live rows of 16384; it keeps 64-bit indices (the 32-bit form measured 1-14%
// slower).  Per element the math is fp32 and independent of the geometry, so
// any grid (and the scalar path) gives the same bits.
#include <algorithm>

#include "common.cuh"

namespace gact {
namespace {

constexpr int kThreads = 256;
constexpr int kVecPerThread = 2;            // large unbounded launches
constexpr int kBoundedVpt = 1;              // the bounded kernel's blocks
constexpr int64_t kSmallLaunchVectors = int64_t(1) << 20;   // VPT = 1 below

// e^{-|a|} as the square of h = e^{-|a|/2} = 2^{-|a| log2(e) / 2} (PTX ISA
// ex2.approx.ftz.f32, one special-function instruction).  h is a normal
// number for |a| < 174 (2^-126 at |a| = 174.7), where the flushing form of
// the exponential is exact to its approximation; the product h * h (an
// ordinary multiply, which keeps subnormals) carries e^{-|a|} down to the
// subnormal results that a product silu(a) * u of ordinary size can still
// need.  Beyond |a| = 174, e^{-|a|} < 2^-251 and every result that uses it
// rounds to zero in bf16 as it does in fp32.
__device__ __forceinline__ float exp_neg_abs(float a) {
    const float x = fabsf(a) * (-0.5f * 1.4426950408889634f);
    float h;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(h) : "f"(x));
    return h * h;
}

// 1 + t lies in [1, 2], where the flushing form of the hardware reciprocal
// (PTX ISA rcp.approx.ftz.f32, one special-function instruction) is within
// one fp32 ulp: no subnormal input or result can occur.
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// sigmoid(a) from t = e^{-|a|} (never overflows): 1 / (1 + t) for a >= 0,
// t / (1 + t) below.  The naive 1 / (1 + e^{-a}) overflows for a < -88.7.
__device__ __forceinline__ float sigmoid(float a) {
    const float t = exp_neg_abs(a);
    const float r = rcp_approx(1.0f + t);
    return a >= 0.f ? r : t * r;
}

struct SiluMul {
    static constexpr bool kGated = true;
    __device__ static float apply(float g, float u) { return g * sigmoid(g) * u; }
};

// gelu_tanh(g) = 0.5 g (1 + tanh(y)) = g * sigmoid(2y), y = sqrt(2/pi)(g + 0.044715 g^3);
// the sigmoid form has no cancellation for g << 0.
struct GeluMul {
    static constexpr bool kGated = true;
    __device__ static float apply(float g, float u) {
        constexpr float k2 = 2.0f * 0.7978845608028654f;
        constexpr float k2c = 2.0f * 0.7978845608028654f * 0.044715f;
        const float a = g * fmaf(k2c, g * g, k2);
        return g * sigmoid(a) * u;
    }
};

struct SquaredRelu {
    static constexpr bool kGated = false;
    __device__ static float apply(float x, float) {
        float r;
        asm("max.NaN.f32 %0, %1, 0f00000000;" : "=f"(r) : "f"(x));
        return r * r;
    }
};

template <class Op>
__device__ __forceinline__ uint32_t apply2(uint32_t g, uint32_t u) {
    return pack_bf16x2(Op::apply(bf16_lo(g), bf16_lo(u)), Op::apply(bf16_hi(g), bf16_hi(u)));
}

// Live rows: all M, or min(max(*n_rows, 0), M) read after the grid dependency.
template <bool BOUNDED>
__device__ __forceinline__ int64_t live_rows(int64_t M, const int32_t *n_rows) {
    if (!BOUNDED)
        return M;
    const int64_t n = static_cast<int64_t>(*n_rows);
    return n < 0 ? 0 : (n > M ? M : n);
}

// One block of VPT * 256 16-byte vectors starting at vector `first`.  Input
// row r starts at in + r * in_rs (gate; up at + d for a gated op), output row
// r at out + r * d.  (step_r, step_c) = (256 / nv, 256 mod nv) steps a
// thread's (row, column) by 256 vectors with a carry.
template <class Op, int VPT>
__device__ __forceinline__ void ew_block(uint16_t *__restrict__ out,
                                         const uint16_t *__restrict__ in, int64_t first,
                                         int64_t live, int64_t nv, int64_t in_rs, int64_t d,
                                         int64_t step_r, int64_t step_c) {
    int64_t r = (first + threadIdx.x) / nv;
    int64_t c = (first + threadIdx.x) - r * nv;
    int64_t rr[VPT], cc[VPT];
    uint4 g[VPT], u[VPT];
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        rr[i] = r;
        cc[i] = c;
        if (r < live) {
            const uint16_t *gp = in + r * in_rs + 8 * c;
            g[i] = ld_stream(gp);
            u[i] = Op::kGated ? ld_stream(gp + d) : make_uint4(0u, 0u, 0u, 0u);
        }
        r += step_r;
        c += step_c;
        if (c >= nv) {
            c -= nv;
            ++r;
        }
    }
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        if (rr[i] < live) {
            const uint4 o = make_uint4(apply2<Op>(g[i].x, u[i].x), apply2<Op>(g[i].y, u[i].y),
                                       apply2<Op>(g[i].z, u[i].z), apply2<Op>(g[i].w, u[i].w));
            st_vec(out + rr[i] * d + 8 * cc[i], o);
        }
    }
}

// ew_block with 32-bit vector indices: the launcher takes it when every
// vector index of the launch (M * nv plus one block) fits in 31 bits.  One
// 32-bit division per thread instead of a 64-bit one, and 32 registers at two
// vectors per thread (40 with 64-bit indices), so 8 CTAs fit an SM.
// Measured on GB300: silu_and_mul 1.4-4% faster at M = 256..65536, d = 768;
// dense gelu_and_mul 7% faster from 1024 x 8192 on.
template <class Op, int VPT>
__device__ __forceinline__ void ew_block32(uint16_t *__restrict__ out,
                                           const uint16_t *__restrict__ in, uint32_t first,
                                           uint32_t live, uint32_t nv, int64_t in_rs, int64_t d,
                                           uint32_t step_r, uint32_t step_c) {
    uint32_t r = (first + threadIdx.x) / nv;
    uint32_t c = (first + threadIdx.x) - r * nv;
    uint32_t rr[VPT], cc[VPT];
    uint4 g[VPT], u[VPT];
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        rr[i] = r;
        cc[i] = c;
        if (r < live) {
            const uint16_t *gp = in + static_cast<int64_t>(r) * in_rs + 8 * c;
            g[i] = ld_stream(gp);
            u[i] = Op::kGated ? ld_stream(gp + d) : make_uint4(0u, 0u, 0u, 0u);
        }
        r += step_r;
        c += step_c;
        if (c >= nv) {
            c -= nv;
            ++r;
        }
    }
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        if (rr[i] < live) {
            const uint4 o = make_uint4(apply2<Op>(g[i].x, u[i].x), apply2<Op>(g[i].y, u[i].y),
                                       apply2<Op>(g[i].z, u[i].z), apply2<Op>(g[i].w, u[i].w));
            st_vec(out + static_cast<int64_t>(rr[i]) * d + 8 * cc[i], o);
        }
    }
}

template <class Op, int VPT>
__global__ void __launch_bounds__(kThreads, 2048 / kThreads)
ew_vec32(uint16_t *__restrict__ out, const uint16_t *__restrict__ in, uint32_t M, uint32_t nv,
         int64_t in_rs, int64_t d, uint32_t step_r, uint32_t step_c) {
    pdl_wait();
    pdl_trigger();
    ew_block32<Op, VPT>(out, in, blockIdx.x * static_cast<uint32_t>(VPT * kThreads), M, nv, in_rs,
                        d, step_r, step_c);
}

// 16-byte path with 64-bit indices, one block per CTA (the grid covers all M
// rows): launches of 2^31 vectors or more.
template <class Op, int VPT>
__global__ void __launch_bounds__(kThreads)
ew_vec(uint16_t *__restrict__ out, const uint16_t *__restrict__ in, int64_t M, int64_t nv,
       int64_t in_rs, int64_t d, int64_t step_r, int64_t step_c) {
    pdl_wait();
    pdl_trigger();
    ew_block<Op, VPT>(out, in, static_cast<int64_t>(blockIdx.x) * VPT * kThreads, M, nv, in_rs,
                      d, step_r, step_c);
}

// 16-byte path over the live rows only: one wave of CTAs walks the blocks
// b, b + gridDim.x, ... that hold live rows, so no CTA is launched only to
// find its rows dead.  The grid depends on M alone.
template <class Op>
__global__ void __launch_bounds__(kThreads)
ew_vec_bounded(uint16_t *__restrict__ out, const uint16_t *__restrict__ in, int64_t M,
               int64_t nv, int64_t in_rs, int64_t d, int64_t step_r, int64_t step_c,
               const int32_t *n_rows) {
    pdl_wait();
    pdl_trigger();
    constexpr int64_t kVecPerCta = int64_t(kThreads) * kBoundedVpt;
    const int64_t live = live_rows<true>(M, n_rows);
    for (int64_t first = static_cast<int64_t>(blockIdx.x) * kVecPerCta; first < live * nv;
         first += static_cast<int64_t>(gridDim.x) * kVecPerCta)
        ew_block<Op, kBoundedVpt>(out, in, first, live, nv, in_rs, d, step_r, step_c);
}

// Any layout: one element per thread iteration, 2-byte accesses.
template <class Op, bool BOUNDED>
__global__ void __launch_bounds__(kThreads)
ew_scalar(uint16_t *__restrict__ out, const uint16_t *__restrict__ in, int64_t M, int64_t in_rs,
          int64_t d, const int32_t *n_rows) {
    pdl_wait();
    pdl_trigger();
    const int64_t total = live_rows<BOUNDED>(M, n_rows) * d;
    const int64_t step = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; e < total;
         e += step) {
        const int64_t r = e / d, c = e - r * d;
        const uint16_t *gp = in + r * in_rs + c;
        const float g = __uint_as_float(static_cast<uint32_t>(ld_stream_u16(gp)) << 16);
        const float u = Op::kGated
                            ? __uint_as_float(static_cast<uint32_t>(ld_stream_u16(gp + d)) << 16)
                            : 0.f;
        out[e] = __bfloat16_as_ushort(__float2bfloat16_rn(Op::apply(g, u)));
    }
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Shared validation and launch.  in_rs: input row stride in elements (2d for
// the contiguous gated ops, d for squared_relu, any >= width for gelu_and_mul).
template <class Op, bool BOUNDED>
int run(void *out, const void *in, int64_t M, int64_t d, int64_t in_rs, const int32_t *n_rows,
        cudaStream_t stream) {
    const int64_t width = Op::kGated ? 2 * d : d;
    if (M < 0 || d <= 0)
        return GATED_ACT_ERR_SIZE;
    if (in_rs < width)
        return GATED_ACT_ERR_STRIDE;
    if (d > (int64_t(1) << 30) || M > (int64_t(1) << 40) || in_rs > (int64_t(1) << 40))
        return GATED_ACT_ERR_TOO_LARGE;
    if (M == 0)
        return GATED_ACT_OK;
    if (!out || !in || (BOUNDED && !n_rows))
        return GATED_ACT_ERR_NULL;
    if (!aligned(out, 2) || !aligned(in, 2) || (BOUNDED && !aligned(n_rows, 4)))
        return GATED_ACT_ERR_ALIGN;
    const uint64_t out_bytes = 2ull * static_cast<uint64_t>(M * d);
    const uint64_t in_bytes = 2ull * static_cast<uint64_t>((M - 1) * in_rs + width);
    if (ranges_overlap(out, out_bytes, in, in_bytes))
        return GATED_ACT_ERR_OVERLAP;

    const void *dout, *din, *dn = n_rows;
    bool host = false;
    int rc;
    if ((rc = resolve_ptr(out, &dout, &host)) != GATED_ACT_OK ||
        (rc = resolve_ptr(in, &din, &host)) != GATED_ACT_OK ||
        (BOUNDED && (rc = resolve_ptr(n_rows, &dn, &host)) != GATED_ACT_OK))
        return rc;
    n_rows = static_cast<const int32_t *>(dn);
    uint16_t *o = static_cast<uint16_t *>(const_cast<void *>(dout));
    const uint16_t *x = static_cast<const uint16_t *>(din);
    const bool vec_ok = aligned(x, 16) && aligned(o, 16) && d % 8 == 0 && in_rs % 8 == 0;
    cudaError_t e;
    if (vec_ok) {
        const int64_t nv = d / 8;
        const int vpt = BOUNDED ? kBoundedVpt : M * nv >= kSmallLaunchVectors ? kVecPerThread : 1;
        int64_t grid = ceil_div(M * nv, int64_t(kThreads) * vpt);
        if (BOUNDED)   // one wave: 2048 threads per SM
            grid = std::min<int64_t>(grid, int64_t(device_sm_count()) * (2048 / kThreads));
        if (grid > 0x7FFFFFFF)
            return GATED_ACT_ERR_TOO_LARGE;
        const dim3 gd(static_cast<unsigned>(grid)), bd(kThreads);
        const int64_t sr = int64_t(kThreads) / nv, sc = int64_t(kThreads) % nv;
        if (BOUNDED)
            e = launch_kernel(ew_vec_bounded<Op>, gd, bd, 0, stream, 1, o, x, M, nv, in_rs, d, sr,
                              sc, n_rows);
        else if (M * nv + int64_t(kThreads) * vpt < (int64_t(1) << 31)) {
            const uint32_t M32 = static_cast<uint32_t>(M), nv32 = static_cast<uint32_t>(nv);
            const uint32_t sr32 = static_cast<uint32_t>(sr), sc32 = static_cast<uint32_t>(sc);
            if (vpt == 1)
                e = launch_kernel(ew_vec32<Op, 1>, gd, bd, 0, stream, 1, o, x, M32, nv32, in_rs, d,
                                  sr32, sc32);
            else
                e = launch_kernel(ew_vec32<Op, kVecPerThread>, gd, bd, 0, stream, 1, o, x, M32,
                                  nv32, in_rs, d, sr32, sc32);
        } else if (vpt == 1)
            e = launch_kernel(ew_vec<Op, 1>, gd, bd, 0, stream, 1, o, x, M, nv, in_rs, d, sr, sc);
        else
            e = launch_kernel(ew_vec<Op, kVecPerThread>, gd, bd, 0, stream, 1, o, x, M, nv, in_rs,
                              d, sr, sc);
    } else {
        const int64_t grid = std::min<int64_t>(ceil_div(M * d, kThreads), int64_t(1) << 20);
        e = launch_kernel(ew_scalar<Op, BOUNDED>, dim3(static_cast<unsigned>(grid)),
                          dim3(kThreads), 0, stream, 1, o, x, M, in_rs, d, n_rows);
    }
    if (e != cudaSuccess)
        return cuda_status(e);
    return cuda_status(cudaGetLastError());
}

}  // namespace
}  // namespace gact

extern "C" int silu_and_mul(void *out, const void *in, int64_t M, int64_t d,
                            cudaStream_t stream) {
    return gact::run<gact::SiluMul, false>(out, in, M, d, 2 * d, nullptr, stream);
}

extern "C" int silu_and_mul_bounded(void *out, const void *in, int64_t M, int64_t d,
                                    const int32_t *n_rows, cudaStream_t stream) {
    return gact::run<gact::SiluMul, true>(out, in, M, d, 2 * d, n_rows, stream);
}

extern "C" int gelu_and_mul(void *out, const void *in, int64_t T, int64_t d, int64_t row_stride,
                            cudaStream_t stream) {
    return gact::run<gact::GeluMul, false>(out, in, T, d, row_stride, nullptr, stream);
}

extern "C" int squared_relu(void *out, const void *in, int64_t M, int64_t d,
                            cudaStream_t stream) {
    return gact::run<gact::SquaredRelu, false>(out, in, M, d, d, nullptr, stream);
}
