// gelu_and_mul_sparse for sm_103a: Gemma3n's sparse GELU gate, fused into one
// pass over HBM.
//
// Definition (vLLM PR "[Performance] Add Triton kernel for Gemma3n sparse
// GELU", section "Purpose": per-row mean and variance, Gaussian thresholding,
// tanh GELU, gated multiplication), per row with gate g = [0, d), up u = [d, 2d):
//   mean = sum g / d,  std = sqrt(sum (g - mean)^2 / d),  cutoff = mean + std z,
//   out  = gelu_tanh(max(g - cutoff, 0)) * u,  fp32 math, one bf16 rounding.
//
// Every geometry reads each input element from HBM exactly once and keeps the
// row on chip (registers) between the statistics and the epilogue:
//   * warp rows   -- one warp per row, shuffles only (d <= 2048);
//   * CTA row     -- one CTA per row, or a cluster of C CTAs per row, each CTA
//                    holding a column slice; CTA partials (count, sum, M2)
//                    are exchanged through distributed shared memory and
//                    merged with the pairwise update of Chan, Golub and LeVeque
//                    (1979), so one cluster barrier serves mean and variance;
//   * scalar      -- any alignment or width: 2-byte loads, gate re-read from
//                    L1/L2 for each pass.
#include <algorithm>

#include "common.cuh"

namespace gact {
namespace {

constexpr float kSqrt2OverPi = 0.7978845608028654f;        // sqrt(2/pi)
constexpr float kCubicCoef = 0.7978845608028654f * 0.044715f;

constexpr int kWarpRowsThreads = 128;      // 4 rows per CTA in the warp-rows geometry
constexpr int kMaxCluster = 8;             // portable cluster size
constexpr int kMaxSliceVec = 4096;         // 16-byte gate vectors one CTA can hold (1024 x 4)
constexpr int kSplitSliceVec = 2048;       // split rows wider than this across a cluster
constexpr int kMinSliceVec = 256;          // do not split rows below this per CTA
constexpr int kScalarThreads = 256;

// tanh via the hardware approximation (PTX ISA tanh.approx.f32, maximum
// relative error about 2^-11).  In gelu_tanh the argument is never negative,
// so 1 + tanh lies in [1, 2] and its relative error stays below 2^-12.
__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// gelu_tanh(max(g - cutoff, 0)) * u.  The comparison form of relu keeps a NaN
// (fmaxf would turn it into 0).
__device__ __forceinline__ float sparse_gelu_mul(float g, float u, float cutoff) {
    float s = g - cutoff;
    s = (s < 0.f) ? 0.f : s;
    const float y = s * fmaf(kCubicCoef, s * s, kSqrt2OverPi);
    const float h = 0.5f * s;
    return fmaf(h, tanh_approx(y), h) * u;
}

__device__ __forceinline__ uint32_t epi2(uint32_t g, uint32_t u, float c) {
    return pack_bf16x2(sparse_gelu_mul(bf16_lo(g), bf16_lo(u), c),
                       sparse_gelu_mul(bf16_hi(g), bf16_hi(u), c));
}

__device__ __forceinline__ uint4 epilogue8(uint4 g, uint4 u, float c) {
    return make_uint4(epi2(g.x, u.x, c), epi2(g.y, u.y, c), epi2(g.z, u.z, c),
                      epi2(g.w, u.w, c));
}

__device__ __forceinline__ float sum8(uint4 g) {
    return ((bf16_lo(g.x) + bf16_hi(g.x)) + (bf16_lo(g.y) + bf16_hi(g.y))) +
           ((bf16_lo(g.z) + bf16_hi(g.z)) + (bf16_lo(g.w) + bf16_hi(g.w)));
}

__device__ __forceinline__ float sq(float x) { return x * x; }

// sum over the 8 values of (x - m)^2
__device__ __forceinline__ float ssd8(uint4 g, float m) {
    float a = sq(bf16_lo(g.x) - m), b = sq(bf16_hi(g.x) - m);
    a = fmaf(bf16_lo(g.y) - m, bf16_lo(g.y) - m, a);
    b = fmaf(bf16_hi(g.y) - m, bf16_hi(g.y) - m, b);
    a = fmaf(bf16_lo(g.z) - m, bf16_lo(g.z) - m, a);
    b = fmaf(bf16_hi(g.z) - m, bf16_hi(g.z) - m, b);
    a = fmaf(bf16_lo(g.w) - m, bf16_lo(g.w) - m, a);
    b = fmaf(bf16_hi(g.w) - m, bf16_hi(g.w) - m, b);
    return a + b;
}

// CTA-wide sum; every thread returns the same bits.
template <int NW>
__device__ __forceinline__ float block_sum(float v, float *red, int lane, int warp) {
    v = warp_sum(v);
    if (NW == 1)
        return v;
    if (lane == 0)
        red[warp] = v;
    __syncthreads();
    return warp_sum(lane < NW ? red[lane] : 0.f);
}

// ------------------------------------------------------------ cluster helpers
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Load a float from the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ float ld_peer(const float *local, uint32_t rank) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
    return v;
}

// ------------------------------------------------------------ warp rows
// One warp per row; lane l holds gate/up vectors l, l+32, ..., l+32(V-1).
template <int V>
__global__ void __launch_bounds__(kWarpRowsThreads, 4)
gelu_warp_rows(uint16_t *__restrict__ out, const uint16_t *__restrict__ in, int64_t T,
               int d, int64_t rs, float z) {
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * (kWarpRowsThreads / 32) +
                        (threadIdx.x >> 5);
    if (row >= T)
        return;
    const int nvec = d >> 3;
    const uint16_t *gp = in + row * rs;
    const uint16_t *up = gp + d;

    uint4 g[V], u[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
        const int v = lane + 32 * i;
        if (v < nvec) {
            g[i] = ld_stream(gp + 8 * v);
            u[i] = ld_stream(up + 8 * v);
        } else {
            g[i] = make_uint4(0u, 0u, 0u, 0u);   // +0 leaves the sum unchanged
            u[i] = g[i];
        }
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i)
        s += sum8(g[i]);
    s = warp_sum(s);
    const float mean = __fdiv_rn(s, static_cast<float>(d));
    float q = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i)
        if (lane + 32 * i < nvec)
            q += ssd8(g[i], mean);
    q = warp_sum(q);
    const float sd = __fsqrt_rn(__fdiv_rn(q, static_cast<float>(d)));
    const float cutoff = fmaf(sd, z, mean);

    uint16_t *op = out + row * static_cast<int64_t>(d);
#pragma unroll
    for (int i = 0; i < V; ++i) {
        const int v = lane + 32 * i;
        if (v < nvec)
            st_vec(op + 8 * v, epilogue8(g[i], u[i], cutoff));
    }
}

// ------------------------------------------------------------ CTA / cluster rows
// A cluster of C CTAs (C = 1: a lone CTA) owns one row at a time; CTA k of
// the cluster holds gate/up vectors [k sv, min((k+1) sv, d/8)), thread t the
// vectors k sv + t + NT i.  Rows advance by the number of clusters in the grid.
// CL = false: C must be 1 (no cluster code is compiled in).
template <int NT, int V, bool CL>
__global__ void __launch_bounds__(NT, (1024 / NT) > 0 ? (1024 / NT) : 1)
gelu_cta_rows(uint16_t *__restrict__ out, const uint16_t *__restrict__ in, int64_t T, int d,
              int64_t rs, float z, int C, int sv) {
    constexpr int NW = NT / 32;
    __shared__ float red[2][NW];
    __shared__ float xch[3];   // this CTA's (element count, sum, M2) for its peers

    if (!CL)
        C = 1;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rank = CL ? static_cast<int>(cluster_ctarank()) : 0;
    const int nvec = d >> 3;
    const int v0 = rank * sv;
    const int v1 = min(nvec, v0 + sv);
    const int nk = max(v1 - v0, 0) * 8;
    const int64_t nclusters = gridDim.x / C;

    for (int64_t row = blockIdx.x / C; row < T; row += nclusters) {
        const uint16_t *gp = in + row * rs;
        const uint16_t *up = gp + d;
        uint4 g[V], u[V];
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const int v = v0 + tid + NT * i;
            if (v < v1) {
                g[i] = ld_stream(gp + 8 * v);
                u[i] = ld_stream(up + 8 * v);
            } else {
                g[i] = make_uint4(0u, 0u, 0u, 0u);
                u[i] = g[i];
            }
        }
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < V; ++i)
            s += sum8(g[i]);
        s = block_sum<NW>(s, red[0], lane, warp);

        float mean, var;
        if (!CL) {
            mean = __fdiv_rn(s, static_cast<float>(d));
            float q = 0.f;
#pragma unroll
            for (int i = 0; i < V; ++i)
                if (v0 + tid + NT * i < v1)
                    q += ssd8(g[i], mean);
            q = block_sum<NW>(q, red[1], lane, warp);
            var = __fdiv_rn(q, static_cast<float>(d));
        } else {
            // local two-pass statistics of this CTA's slice ...
            const float mk = nk > 0 ? __fdiv_rn(s, static_cast<float>(nk)) : 0.f;
            float q = 0.f;
#pragma unroll
            for (int i = 0; i < V; ++i)
                if (v0 + tid + NT * i < v1)
                    q += ssd8(g[i], mk);
            q = block_sum<NW>(q, red[1], lane, warp);
            if (tid == 0) {
                xch[0] = static_cast<float>(nk);
                xch[1] = s;
                xch[2] = q;
            }
            cluster_arrive_release();
            cluster_wait_acquire();
            // ... merged over the cluster in rank order (lane k reads CTA k):
            // M2 = sum_k M2_k + sum_k n_k (mean_k - mean)^2.
            float n_k = 0.f, s_k = 0.f, q_k = 0.f;
            if (lane < C) {
                n_k = ld_peer(&xch[0], lane);
                s_k = ld_peer(&xch[1], lane);
                q_k = ld_peer(&xch[2], lane);
            }
            mean = __fdiv_rn(warp_sum(s_k), static_cast<float>(d));
            float between = 0.f;
            if (n_k > 0.f) {
                const float dm = __fdiv_rn(s_k, n_k) - mean;
                between = n_k * (dm * dm);
            }
            var = __fdiv_rn(warp_sum(q_k + between), static_cast<float>(d));
            cluster_arrive_release();   // this CTA is done reading its peers
        }
        const float sd = __fsqrt_rn(var);
        const float cutoff = fmaf(sd, z, mean);

        uint16_t *op = out + row * static_cast<int64_t>(d);
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const int v = v0 + tid + NT * i;
            if (v < v1)
                st_vec(op + 8 * v, epilogue8(g[i], u[i], cutoff));
        }
        if (CL)
            cluster_wait_acquire();   // peers are done with xch before it changes
    }
}

// ------------------------------------------------------------ scalar rows
// Any layout: one CTA per row, 2-byte loads; each pass re-reads the gate
// (from L1/L2 after the first pass).
__device__ __forceinline__ float ld_bf16(const uint16_t *p) {
    return __uint_as_float(static_cast<uint32_t>(ld_stream_u16(p)) << 16);
}

__global__ void __launch_bounds__(kScalarThreads)
gelu_scalar_rows(uint16_t *__restrict__ out, const uint16_t *__restrict__ in, int64_t T,
                 int64_t d, int64_t rs, float z) {
    constexpr int NW = kScalarThreads / 32;
    __shared__ float red[2][NW];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int64_t row = blockIdx.x; row < T; row += gridDim.x) {
        const uint16_t *gp = in + row * rs;
        const uint16_t *up = gp + d;
        float s = 0.f;
        for (int64_t j = tid; j < d; j += kScalarThreads)
            s += ld_bf16(gp + j);
        s = block_sum<NW>(s, red[0], lane, warp);
        const float mean = __fdiv_rn(s, static_cast<float>(d));
        float q = 0.f;
        for (int64_t j = tid; j < d; j += kScalarThreads) {
            const float e = ld_bf16(gp + j) - mean;
            q = fmaf(e, e, q);
        }
        q = block_sum<NW>(q, red[1], lane, warp);
        const float sd = __fsqrt_rn(__fdiv_rn(q, static_cast<float>(d)));
        const float cutoff = fmaf(sd, z, mean);
        uint16_t *op = out + row * d;
        for (int64_t j = tid; j < d; j += kScalarThreads) {
            const float y = sparse_gelu_mul(ld_bf16(gp + j), ld_bf16(up + j), cutoff);
            op[j] = __bfloat16_as_ushort(__float2bfloat16_rn(y));
        }
    }
}

// ------------------------------------------------------------ host side
using WarpFn = void (*)(uint16_t *, const uint16_t *, int64_t, int, int64_t, float);
using CtaFn = void (*)(uint16_t *, const uint16_t *, int64_t, int, int64_t, float, int, int);

WarpFn warp_fn(int v) {
    switch (v) {
    case 1: return gelu_warp_rows<1>;
    case 2: return gelu_warp_rows<2>;
    case 4: return gelu_warp_rows<4>;
    case 8: return gelu_warp_rows<8>;
    default: return nullptr;
    }
}

template <bool CL>
CtaFn cta_fn_t(int nt, int v) {
    if (v == 2) {
        switch (nt) {
        case 64: return gelu_cta_rows<64, 2, CL>;
        case 128: return gelu_cta_rows<128, 2, CL>;
        default: return nullptr;
        }
    }
    if (v == 4) {
        switch (nt) {
        case 64: return gelu_cta_rows<64, 4, CL>;
        case 128: return gelu_cta_rows<128, 4, CL>;
        case 256: return gelu_cta_rows<256, 4, CL>;
        case 512: return gelu_cta_rows<512, 4, CL>;
        case 1024: return gelu_cta_rows<1024, 4, CL>;
        default: return nullptr;
        }
    }
    return nullptr;
}

CtaFn cta_fn(int nt, int v, int cluster) {
    return cluster > 1 ? cta_fn_t<true>(nt, v) : cta_fn_t<false>(nt, v);
}

int pow2_ceil(int64_t x) {
    int p = 1;
    while (p < x)
        p <<= 1;
    return p;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct Plan {
    gated_act_plan pub;
    int sv;   // vectors per CTA slice (CTA rows)
};

// Threads and vectors per thread for a CTA slice of sv vectors.
void cta_shape(int64_t sv, int *nt, int *v) {
    if (sv <= kMinSliceVec) {
        *v = 2;
        *nt = std::max(64, pow2_ceil(ceil_div(sv, 2)));
    } else {
        *v = 4;
        *nt = std::max(64, pow2_ceil(ceil_div(sv, 4)));
    }
}

// check_ptrs = false (plan queries): pointers are only inspected for alignment.
int validate(const void *out, const void *in, int64_t T, int64_t d, int64_t rs,
             bool check_ptrs) {
    if (T < 0 || d <= 0)
        return GATED_ACT_ERR_SIZE;
    if (rs < 2 * d)
        return GATED_ACT_ERR_STRIDE;
    if (d > (int64_t(1) << 30) || rs > (int64_t(1) << 40) || T > (int64_t(1) << 40))
        return GATED_ACT_ERR_TOO_LARGE;
    if (T == 0 || !check_ptrs)
        return GATED_ACT_OK;
    if (!out || !in)
        return GATED_ACT_ERR_NULL;
    if (!aligned(out, 2) || !aligned(in, 2))
        return GATED_ACT_ERR_ALIGN;
    const uint64_t in_bytes = 2ull * static_cast<uint64_t>((T - 1) * rs + 2 * d);
    const uint64_t out_bytes = 2ull * static_cast<uint64_t>(T * d);
    if (ranges_overlap(out, out_bytes, in, in_bytes))
        return GATED_ACT_ERR_OVERLAP;
    return GATED_ACT_OK;
}

int make_plan(const void *out, const void *in, int64_t T, int64_t d, int64_t rs,
              int variant, int cluster, int sm_count, bool check_ptrs, Plan *p) {
    const int rc = validate(out, in, T, d, rs, check_ptrs);
    if (rc != GATED_ACT_OK)
        return rc;
    if (variant < GATED_ACT_VARIANT_AUTO || variant > GATED_ACT_VARIANT_SCALAR)
        return GATED_ACT_ERR_VARIANT;
    gated_act_plan &q = p->pub;
    q = gated_act_plan{};
    p->sv = 0;
    const bool vec_ok = aligned(in, 16) && aligned(out, 16) && d % 8 == 0 && rs % 8 == 0;
    const int64_t nvec = d / 8;
    const int sms = sm_count > 0 ? sm_count : (T > 0 ? device_sm_count() : 1);

    if (variant == GATED_ACT_VARIANT_AUTO) {
        if (!vec_ok || nvec > int64_t(kMaxSliceVec) * kMaxCluster)
            variant = GATED_ACT_VARIANT_SCALAR;
        else if (nvec <= 256)
            variant = GATED_ACT_VARIANT_WARP_ROWS;
        else
            variant = GATED_ACT_VARIANT_CTA_ROW;
        if (variant == GATED_ACT_VARIANT_CTA_ROW)
            cluster = 0;
    }

    if (variant == GATED_ACT_VARIANT_WARP_ROWS) {
        if (!vec_ok || nvec > 256)
            return GATED_ACT_ERR_VARIANT;
        q.variant = variant;
        q.cluster = 1;
        q.threads = kWarpRowsThreads;
        q.vec_per_thread = pow2_ceil(ceil_div(nvec, 32));
        q.rows_per_cta = kWarpRowsThreads / 32;
        q.grid = ceil_div(T, q.rows_per_cta);
        if (q.grid > 0x7FFFFFFF)
            return GATED_ACT_ERR_TOO_LARGE;
        return GATED_ACT_OK;
    }

    if (variant == GATED_ACT_VARIANT_CTA_ROW) {
        if (!vec_ok)
            return GATED_ACT_ERR_VARIANT;
        int C = cluster;
        if (C == 0) {
            C = 1;
            while (ceil_div(nvec, C) > kSplitSliceVec && C < kMaxCluster)
                C *= 2;
            while (T * C < sms && C < kMaxCluster && ceil_div(nvec, 2 * C) >= kMinSliceVec)
                C *= 2;
        }
        if (C < 1 || C > kMaxCluster || (C & (C - 1)) != 0)
            return GATED_ACT_ERR_VARIANT;
        const int64_t sv = ceil_div(nvec, C);
        if (sv > kMaxSliceVec)
            return GATED_ACT_ERR_VARIANT;
        int nt, v;
        cta_shape(sv, &nt, &v);
        q.variant = variant;
        q.cluster = C;
        q.threads = nt;
        q.vec_per_thread = v;
        q.rows_per_cta = 1;
        const int64_t max_clusters = 0x7FFFFFFF / C;
        q.grid = std::min<int64_t>(T, max_clusters) * C;
        p->sv = static_cast<int>(sv);
        return GATED_ACT_OK;
    }

    // scalar
    q.variant = GATED_ACT_VARIANT_SCALAR;
    q.cluster = 1;
    q.threads = kScalarThreads;
    q.vec_per_thread = 0;
    q.rows_per_cta = 1;
    q.grid = std::min<int64_t>(T, 0x7FFFFFFF);
    return GATED_ACT_OK;
}

int launch(const Plan &p, void *out, const void *in, int64_t T, int64_t d, int64_t rs,
           double z, cudaStream_t stream) {
    uint16_t *o = static_cast<uint16_t *>(out);
    const uint16_t *x = static_cast<const uint16_t *>(in);
    const float zf = static_cast<float>(z);
    const gated_act_plan &q = p.pub;
    const dim3 grid(static_cast<unsigned>(q.grid)), block(q.threads);
    switch (q.variant) {
    case GATED_ACT_VARIANT_WARP_ROWS:
        warp_fn(q.vec_per_thread)<<<grid, block, 0, stream>>>(o, x, T, static_cast<int>(d), rs, zf);
        break;
    case GATED_ACT_VARIANT_CTA_ROW: {
        CtaFn fn = cta_fn(q.threads, q.vec_per_thread, q.cluster);
        if (!fn)
            return GATED_ACT_ERR_VARIANT;
        if (q.cluster == 1) {
            fn<<<grid, block, 0, stream>>>(o, x, T, static_cast<int>(d), rs, zf, 1, p.sv);
        } else {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = grid;
            cfg.blockDim = block;
            cfg.dynamicSmemBytes = 0;
            cfg.stream = stream;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = q.cluster;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            const cudaError_t e = cudaLaunchKernelEx(&cfg, fn, o, x, T, static_cast<int>(d), rs,
                                                     zf, static_cast<int>(q.cluster), p.sv);
            if (e != cudaSuccess)
                return cuda_status(e);
        }
        break;
    }
    default:
        gelu_scalar_rows<<<grid, block, 0, stream>>>(o, x, T, d, rs, zf);
        break;
    }
    return cuda_status(cudaGetLastError());
}

}  // namespace
}  // namespace gact

extern "C" int gelu_and_mul_sparse_plan(const void *out, const void *in, int64_t T, int64_t d,
                                        int64_t row_stride, int variant, int cluster,
                                        int sm_count, gated_act_plan *plan) {
    if (!plan)
        return GATED_ACT_ERR_NULL;
    gact::Plan p;
    const int rc = gact::make_plan(out, in, T, d, row_stride, variant, cluster, sm_count, false, &p);
    if (rc != GATED_ACT_OK)
        return rc;
    *plan = p.pub;
    return GATED_ACT_OK;
}

extern "C" int gelu_and_mul_sparse_ex(void *out, const void *in, int64_t T, int64_t d,
                                      int64_t row_stride, double z, int variant, int cluster,
                                      cudaStream_t stream) {
    gact::Plan p;
    const int rc = gact::make_plan(out, in, T, d, row_stride, variant, cluster, 0, true, &p);
    if (rc != GATED_ACT_OK || T == 0)
        return rc;
    return gact::launch(p, out, in, T, d, row_stride, z, stream);
}

extern "C" int gelu_and_mul_sparse(void *out, const void *in, int64_t T, int64_t d,
                                   int64_t row_stride, double z, cudaStream_t stream) {
    return gelu_and_mul_sparse_ex(out, in, T, d, row_stride, z, GATED_ACT_VARIANT_AUTO, 0,
                                  stream);
}
