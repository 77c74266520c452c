// Update + row renormalisation of the fast weights, and their bf16 shadow.
//
//   W~_j = W_j + scale * D_j            (GD: D = dL/dW, scale = -1;
//                                        Muon: D = NS5(dL/dW), scale = -lr;
//                                        momentum: M = beta M + dL/dW kept,
//                                        D = M, scale = -1)
//   W'_j = W~_j * ||W_j|| / ||W~_j||     for every row j of W1, W2, W3
//
// (LaCT review page, "Local attention and nonlinear memory work together":
// the updated fast weights are L2-normalised; each row keeps the norm it had
// before the update.) A row whose updated norm is 0 cannot be rescaled: it
// is stored as updated (the zero row, factor 1); a non-finite norm sets the
// sticky status bit ST_NONFINITE.
//
// One warp per row; rows are contiguous in memory (W1, W3: dh rows of d;
// W2: d rows of dh). HBM-bound: reads W and D, writes W' and its bf16 copy.
#include "lact_internal.cuh"

namespace lact {

namespace {

template <typename R>
struct UpdArgs {
    R* W[3];
    const R* D[3];
    bf16* S[3];        // bf16 shadows (nullptr: none)
    R* Mo[3];          // momentum velocities (nullptr: none), updated in place
    R beta;
    int rows[3];       // rows per head of each matrix
    int len[3];        // row length of each matrix
    int BH;
    R scale;
    int* status;
};

template <typename R>
__device__ __forceinline__ R warp_sum(R x) {
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ void load_vec(const float* p, float* v, int n) {
    if (n == 4) {
        float4 x = *reinterpret_cast<const float4*>(p);
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    } else {
        for (int k = 0; k < n; ++k) v[k] = p[k];
    }
}
__device__ __forceinline__ void load_vec(const double* p, double* v, int n) {
    for (int k = 0; k < n; ++k) v[k] = p[k];
}
__device__ __forceinline__ void store_vec(float* p, const float* v, int n) {
    if (n == 4) *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    else for (int k = 0; k < n; ++k) p[k] = v[k];
}
__device__ __forceinline__ void store_vec(double* p, const double* v, int n) {
    for (int k = 0; k < n; ++k) p[k] = v[k];
}

// MAXV: pieces of 32*VEC elements of the longest row, fixed at compile time so
// the row stays in registers (sized to the shape: fewer registers, more warps
// resident, for the common row lengths up to 512).
template <typename R, int VEC, int MAXV>
__global__ void __launch_bounds__(256) k_update_renorm(UpdArgs<R> a) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t r0 = (int64_t)a.BH * a.rows[0], r1 = (int64_t)a.BH * a.rows[1];
    const int64_t r2 = (int64_t)a.BH * a.rows[2];
    if (warp >= r0 + r1 + r2) return;
    int m;
    int64_t row;
    if (warp < r0) { m = 0; row = warp; }
    else if (warp < r0 + r1) { m = 1; row = warp - r0; }
    else { m = 2; row = warp - r0 - r1; }
    const int len = a.len[m];
    R* w = a.W[m] + row * len;
    const R* dv = a.D[m] + row * len;
    R* mo = a.Mo[m] ? a.Mo[m] + row * len : nullptr;
    // Pass 1: both norms, the row kept in registers.
    R wt[MAXV][VEC];
    R n0 = 0, n1 = 0;
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
        const int c = (i * 32 + lane) * VEC;
        if (c < len) {
            R wv[VEC], gv[VEC];
            load_vec(w + c, wv, VEC);
            load_vec(dv + c, gv, VEC);
            if (mo) {
                R mv[VEC];
                load_vec(mo + c, mv, VEC);
#pragma unroll
                for (int k = 0; k < VEC; ++k) gv[k] = fma_r(a.beta, mv[k], gv[k]);
                store_vec(mo + c, gv, VEC);
            }
#pragma unroll
            for (int k = 0; k < VEC; ++k) {
                const R t = fma_r(a.scale, gv[k], wv[k]);
                wt[i][k] = t;
                n0 = fma_r(wv[k], wv[k], n0);
                n1 = fma_r(t, t, n1);
            }
        }
    }
    n0 = sqrt_r(warp_sum(n0));
    n1 = sqrt_r(warp_sum(n1));
    if (!isfinite(n0) || !isfinite(n1)) {
        if (lane == 0) atomicOr(a.status, ST_NONFINITE);
    }
    const R f = n1 > R(0) ? n0 / n1 : R(1);
    bf16* sh = a.S[m] ? a.S[m] + row * len : nullptr;
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
        const int c = (i * 32 + lane) * VEC;
        if (c < len) {
            R o[VEC];
#pragma unroll
            for (int k = 0; k < VEC; ++k) o[k] = wt[i][k] * f;
            store_vec(w + c, o, VEC);
            if (sh) {
                if (VEC == 4) {
                    __nv_bfloat162 p0 = __floats2bfloat162_rn((float)o[0], (float)o[1]);
                    __nv_bfloat162 p1 = __floats2bfloat162_rn((float)o[2], (float)o[3]);
                    uint2 u;
                    u.x = *reinterpret_cast<uint32_t*>(&p0);
                    u.y = *reinterpret_cast<uint32_t*>(&p1);
                    *reinterpret_cast<uint2*>(sh + c) = u;
                } else {
#pragma unroll
                    for (int k = 0; k < VEC; ++k) sh[c + k] = __float2bfloat16_rn((float)o[k]);
                }
            }
        }
    }
}

__global__ void k_shadow(const float* __restrict__ W, bf16* __restrict__ S, size_t n) {
    pdl_wait();
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        S[i] = __float2bfloat16_rn(W[i]);
}

template <typename A, typename B>
__global__ void k_convert(const A* __restrict__ src, B* __restrict__ dst, size_t n) {
    pdl_wait();
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        dst[i] = (B)src[i];
}

template <typename R>
cudaError_t update_t(const lact_state* st, const void* const g[3], double scale, void* const mom[3], double beta,
                     cudaStream_t s) {
    UpdArgs<R> a;
    const int d = st->cfg.d, dh = st->cfg.dh;
    for (int m = 0; m < 3; ++m) {
        a.W[m] = static_cast<R*>(st->W[m]);
        a.D[m] = static_cast<const R*>(g[m]);
        a.S[m] = st->cfg.io_dtype == LACT_BF16 ? st->Wsh[m] : nullptr;
        a.Mo[m] = mom ? static_cast<R*>(mom[m]) : nullptr;
        a.rows[m] = m >= st->nmat ? 0 : (m == 1 ? d : dh);   // the linear memory has W1 only
        a.len[m] = m == 1 ? dh : d;
    }
    a.BH = st->BH;
    a.scale = (R)scale;
    a.beta = (R)beta;
    a.status = st->status;
    const int64_t rows = (int64_t)st->BH * (a.rows[0] + a.rows[1] + a.rows[2]);
    const int blocks = (int)((rows * 32 + 255) / 256);
    // every row length here is a multiple of 32; float4 when a multiple of 128
    const int maxlen = d > dh ? d : dh;
    if (sizeof(R) == 4 && d % 128 == 0 && dh % 128 == 0) {
        if (maxlen <= 512) launch_pdl(k_update_renorm<R, 4, 4>, blocks, 256, 0, s, a);
        else launch_pdl(k_update_renorm<R, 4, 8>, blocks, 256, 0, s, a);
    } else {
        launch_pdl(k_update_renorm<R, 1, 32>, blocks, 256, 0, s, a);
    }
    g_launches++;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_update(const lact_state* st, const void* const g[3], double scale, void* const mom[3],
                          double beta, cudaStream_t s) {
    return st->f64 ? update_t<double>(st, g, scale, mom, beta, s) : update_t<float>(st, g, scale, mom, beta, s);
}

cudaError_t launch_shadow(const lact_state* st, cudaStream_t s) {
    if (st->cfg.io_dtype != LACT_BF16) return cudaSuccess;
    const size_t n = (size_t)st->BH * st->cfg.d * st->cfg.dh;
    for (int m = 0; m < st->nmat; ++m) {
        launch_pdl(k_shadow, st->num_sms * 4, 256, 0, s, static_cast<const float*>(st->W[m]), st->Wsh[m], n);
        g_launches++;
    }
    return cudaGetLastError();
}

cudaError_t launch_convert(const void* src, bool src_f64, void* dst, bool dst_f64, size_t n, int num_sms,
                           cudaStream_t s) {
    const int blocks = num_sms * 4;
    if (src_f64 && dst_f64)
        launch_pdl(k_convert<double, double>, blocks, 256, 0, s, static_cast<const double*>(src), static_cast<double*>(dst), n);
    else if (src_f64)
        launch_pdl(k_convert<double, float>, blocks, 256, 0, s, static_cast<const double*>(src), static_cast<float*>(dst), n);
    else if (dst_f64)
        launch_pdl(k_convert<float, double>, blocks, 256, 0, s, static_cast<const float*>(src), static_cast<double*>(dst), n);
    else
        launch_pdl(k_convert<float, float>, blocks, 256, 0, s, static_cast<const float*>(src), static_cast<float*>(dst), n);
    g_launches++;
    return cudaGetLastError();
}

}  // namespace lact
