// SIMT (CUDA-core) kernels of the LaCT chunk step:
//   readout   o_i = W2 (silu(W1 q_i) * (W3 q_i))
//   gradient  dL/dW of L = -sum_i eta_i <f_W(k_i), v_i>, split over tokens
//   reduction of the split-K partial sums in a fixed order
// R is the internal real type: fp64 for fp32-io states (whose Muon step must
// agree with an fp64 reading to 1e-4, see lact_api.cu), fp32 for bf16-io
// states on shapes the tensor-core kernels do not cover.
// Sources: LaCT review page, "Local attention and nonlinear memory work
// together" (SwiGLU memory, negative inner-product loss, per-token rates).
#include "lact_internal.cuh"

namespace lact {

namespace {

constexpr int NT = 256;   // threads per CTA

template <typename R> struct Tile;                       // tokens / hidden units per tile
template <> struct Tile<float> { static constexpr int TT = 32, HC = 32; };
template <> struct Tile<double> { static constexpr int TT = 16, HC = 16; };

template <typename R> __device__ __forceinline__ R sigmoid_r(R x) { return R(1) / (R(1) + exp_r(-x)); }

// o = f_W(q) for TT tokens of one (b, h) per CTA. Hidden units are visited
// HC at a time: u = silu(W1_r q) * (W3_r q) in shared memory, then o += W2_r u.
template <typename T, typename R, int D>
__global__ void __launch_bounds__(NT) k_apply_simt(TokView q, T* __restrict__ o,
                                                   const R* __restrict__ W1,
                                                   const R* __restrict__ W2,
                                                   const R* __restrict__ W3, int dh) {
    pdl_wait();
    constexpr int TT = Tile<R>::TT, HC = Tile<R>::HC;
    constexpr int DP = D + 1, HP = HC + 1;
    constexpr int G = NT / D;          // token groups in the W2 phase
    constexpr int TPG = TT / G;        // tokens per group
    static_assert(TPG >= 1, "tile too small for this head dim");
    extern __shared__ __align__(16) unsigned char smraw[];
    R* Qs = reinterpret_cast<R*>(smraw);   // [TT][DP]
    R* W1s = Qs + TT * DP;                 // [HC][DP]
    R* W3s = W1s + HC * DP;                // [HC][DP]
    R* W2s = W3s + HC * DP;                // [D][HP]
    R* Us = W2s + D * HP;                  // [TT][HP]

    const int bh = blockIdx.y, tid = threadIdx.x;
    const int64_t tt0 = (int64_t)blockIdx.x * TT;
    const int ntok = (int)min((int64_t)TT, q.n - tt0);
    const int64_t row0 = (int64_t)bh * q.n_total + q.t0 + tt0;
    const T* qp = static_cast<const T*>(q.p);
    for (int i = tid; i < TT * D; i += NT) {
        int r = i / D, c = i % D;
        Qs[r * DP + c] = r < ntok ? ld_io<R>(qp, (row0 + r) * D + c) : R(0);
    }
    const R* W1b = W1 + (size_t)bh * dh * D;
    const R* W3b = W3 + (size_t)bh * dh * D;
    const R* W2b = W2 + (size_t)bh * D * dh;
    const int j = tid % D, g = tid / D;
    R acc[TPG];
#pragma unroll
    for (int k = 0; k < TPG; ++k) acc[k] = R(0);

    for (int h0 = 0; h0 < dh; h0 += HC) {
        __syncthreads();
        for (int i = tid; i < HC * D; i += NT) {
            int r = i / D, c = i % D;
            W1s[r * DP + c] = W1b[(size_t)(h0 + r) * D + c];
            W3s[r * DP + c] = W3b[(size_t)(h0 + r) * D + c];
        }
        for (int i = tid; i < D * HC; i += NT) {
            int r = i / HC, c = i % HC;
            W2s[r * HP + c] = W2b[(size_t)r * dh + h0 + c];
        }
        __syncthreads();
        const int hid = tid % HC;
        for (int tk = tid / HC; tk < TT; tk += NT / HC) {
            R a1 = 0, a3 = 0;
#pragma unroll 8
            for (int c = 0; c < D; ++c) {
                R x = Qs[tk * DP + c];
                a1 = fma_r(x, W1s[hid * DP + c], a1);
                a3 = fma_r(x, W3s[hid * DP + c], a3);
            }
            Us[tk * HP + hid] = a1 * sigmoid_r(a1) * a3;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < TPG; ++k) {
            const int tk = g + k * G;
            R s = acc[k];
#pragma unroll 8
            for (int hc = 0; hc < HC; ++hc) s = fma_r(W2s[j * HP + hc], Us[tk * HP + hc], s);
            acc[k] = s;
        }
    }
    // o has q's layout: the same token slice of a [BH, n_total, D] tensor
#pragma unroll
    for (int k = 0; k < TPG; ++k) {
        const int tk = g + k * G;
        if (tk < ntok) st_io(o, (row0 + tk) * D + j, acc[k]);
    }
}

// Partial chunk gradient of one (split, hidden block of HC, head) per CTA.
// Per TT-token tile: h1 = W1_r k, h3 = W3_r k, a = W2_r^T v (shared memory),
// g = -eta v, u = silu(h1) h3, du = -eta a,
// dh1 = du h3 silu'(h1), dh3 = du silu(h1); then the three outer-product sums
// dW1_r += dh1 k^T, dW3_r += dh3 k^T, dW2_r += g u^T stay in registers.
template <typename T, typename R, int D>
__global__ void __launch_bounds__(NT) k_grad_simt(TokView k, TokView v, const float* __restrict__ eta,
                                                  const R* __restrict__ W1,
                                                  const R* __restrict__ W2,
                                                  const R* __restrict__ W3, int dh,
                                                  int tiles_per_split, R* __restrict__ partial,
                                                  int BH) {
    pdl_wait();
    constexpr int TT = Tile<R>::TT, HC = Tile<R>::HC;
    constexpr int DP = D + 1, HP = HC + 1;
    constexpr int G = NT / D;          // hidden groups in the accumulation phase
    constexpr int HPG = HC / G;        // hidden units per group
    static_assert(HPG >= 1, "tile too small for this head dim");
    extern __shared__ __align__(16) unsigned char smraw[];
    R* Ks = reinterpret_cast<R*>(smraw);   // [TT][DP]
    R* Vs = Ks + TT * DP;                  // [TT][DP]
    R* W1s = Vs + TT * DP;                 // [HC][DP]
    R* W3s = W1s + HC * DP;                // [HC][DP]
    R* W2s = W3s + HC * DP;                // [D][HP]   W2[:, r]
    R* P1 = W2s + D * HP;                  // [TT][HP]  dh1
    R* P3 = P1 + TT * HP;                  // [TT][HP]  dh3
    R* PU = P3 + TT * HP;                  // [TT][HP]  -eta u
    R* Es = PU + TT * HP;                  // [TT]

    const int split = blockIdx.x, h0 = blockIdx.y * HC, bh = blockIdx.z, tid = threadIdx.x;
    const R* W1b = W1 + (size_t)bh * dh * D;
    const R* W3b = W3 + (size_t)bh * dh * D;
    const R* W2b = W2 + (size_t)bh * D * dh;
    for (int i = tid; i < HC * D; i += NT) {
        int r = i / D, c = i % D;
        W1s[r * DP + c] = W1b[(size_t)(h0 + r) * D + c];
        W3s[r * DP + c] = W3b[(size_t)(h0 + r) * D + c];
    }
    for (int i = tid; i < D * HC; i += NT) {
        int r = i / HC, c = i % HC;
        W2s[r * HP + c] = W2b[(size_t)r * dh + h0 + c];
    }
    const int c = tid % D, g = tid / D;
    R a1[HPG], a2[HPG], a3[HPG];
#pragma unroll
    for (int i = 0; i < HPG; ++i) a1[i] = a2[i] = a3[i] = R(0);

    const T* kp = static_cast<const T*>(k.p);
    const T* vp = static_cast<const T*>(v.p);
    const int64_t ntiles = (k.n + TT - 1) / TT;
    const int64_t tb = (int64_t)split * tiles_per_split;
    const int64_t te = min(ntiles, tb + tiles_per_split);
    const int64_t krow = (int64_t)bh * k.n_total + k.t0;
    const int64_t vrow = (int64_t)bh * v.n_total + v.t0;
    for (int64_t t = tb; t < te; ++t) {
        const int64_t tt0 = t * TT;
        const int ntok = (int)min((int64_t)TT, k.n - tt0);
        __syncthreads();
        for (int i = tid; i < TT * D; i += NT) {
            int r = i / D, cc = i % D;
            bool ok = r < ntok;
            Ks[r * DP + cc] = ok ? ld_io<R>(kp, (krow + tt0 + r) * D + cc) : R(0);
            Vs[r * DP + cc] = ok ? ld_io<R>(vp, (vrow + tt0 + r) * D + cc) : R(0);
        }
        if (tid < TT) Es[tid] = tid < ntok ? (R)eta[krow + tt0 + tid] : R(0);
        __syncthreads();
        const int hid = tid % HC;
        for (int tk = tid / HC; tk < TT; tk += NT / HC) {
            R h1 = 0, h3 = 0, a = 0;
#pragma unroll 8
            for (int cc = 0; cc < D; ++cc) {
                R x = Ks[tk * DP + cc];
                h1 = fma_r(x, W1s[hid * DP + cc], h1);
                h3 = fma_r(x, W3s[hid * DP + cc], h3);
                a = fma_r(Vs[tk * DP + cc], W2s[cc * HP + hid], a);
            }
            const R e = Es[tk];
            const R s = sigmoid_r(h1);
            const R si = h1 * s;
            const R du = -e * a;
            P1[tk * HP + hid] = du * h3 * s * (R(1) + h1 * (R(1) - s));
            P3[tk * HP + hid] = du * si;
            PU[tk * HP + hid] = -e * (si * h3);
        }
        __syncthreads();
        for (int tk = 0; tk < TT; ++tk) {
            const R kc = Ks[tk * DP + c], vc = Vs[tk * DP + c];
#pragma unroll
            for (int i = 0; i < HPG; ++i) {
                const int hh = g * HPG + i;
                a1[i] = fma_r(P1[tk * HP + hh], kc, a1[i]);
                a3[i] = fma_r(P3[tk * HP + hh], kc, a3[i]);
                a2[i] = fma_r(PU[tk * HP + hh], vc, a2[i]);
            }
        }
    }
    const size_t mat = (size_t)BH * dh * D;
    R* p1 = partial + ((size_t)split * 3 + 0) * mat + (size_t)bh * dh * D;
    R* p2 = partial + ((size_t)split * 3 + 1) * mat + (size_t)bh * dh * D;
    R* p3 = partial + ((size_t)split * 3 + 2) * mat + (size_t)bh * dh * D;
#pragma unroll
    for (int i = 0; i < HPG; ++i) {
        const int hh = h0 + g * HPG + i;
        p1[(size_t)hh * D + c] = a1[i];
        p3[(size_t)hh * D + c] = a3[i];
        p2[(size_t)c * dh + hh] = a2[i];
    }
}

// out[m] (+)= sum over slots s = 0, 1, ... of partial[s][m], in that order.
template <typename R>
__global__ void k_reduce(const R* __restrict__ partial, int slots, size_t mat, int nmat, bool accumulate,
                         R* __restrict__ o0, R* __restrict__ o1, R* __restrict__ o2) {
    pdl_wait();
    const size_t n = (size_t)nmat * mat;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int m = (int)(i / mat);
        const size_t j = i - (size_t)m * mat;
        R* out = m == 0 ? o0 : (m == 1 ? o1 : o2);
        R acc = accumulate ? out[j] : R(0);
        for (int s = 0; s < slots; ++s) acc += partial[(size_t)s * n + i];
        out[j] = acc;
    }
}

template <typename R, int D>
size_t apply_smem() {
    constexpr int TT = Tile<R>::TT, HC = Tile<R>::HC;
    return sizeof(R) * (TT * (D + 1) + 2 * HC * (D + 1) + D * (HC + 1) + TT * (HC + 1));
}
template <typename R, int D>
size_t grad_smem() {
    constexpr int TT = Tile<R>::TT, HC = Tile<R>::HC;
    return sizeof(R) * (2 * TT * (D + 1) + 2 * HC * (D + 1) + D * (HC + 1) + 3 * TT * (HC + 1) + TT);
}

template <typename T, typename R, int D>
cudaError_t apply_t(const lact_state* st, TokView q, void* o, cudaStream_t s) {
    auto kern = k_apply_simt<T, R, D>;
    size_t sm = apply_smem<R, D>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((q.n + Tile<R>::TT - 1) / Tile<R>::TT), st->BH);
    launch_pdl(kern, grid, NT, sm, s, q, static_cast<T*>(o), static_cast<const R*>(st->W[0]),
                              static_cast<const R*>(st->W[1]), static_cast<const R*>(st->W[2]), st->cfg.dh);
    g_launches++;
    return cudaGetLastError();
}

template <typename T, typename R, int D>
cudaError_t grad_t(const lact_state* st, TokView k, TokView v, const float* eta, int* slots, cudaStream_t s) {
    constexpr int TT = Tile<R>::TT, HC = Tile<R>::HC;
    auto kern = k_grad_simt<T, R, D>;
    size_t sm = grad_smem<R, D>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    const int dh = st->cfg.dh;
    const int64_t ntiles = (k.n + TT - 1) / TT;
    const int units = st->BH * (dh / HC);
    // enough CTAs for ~4 waves, each split at least 8 tiles, at most kMaxSlots splits
    int64_t want = (4LL * st->num_sms + units - 1) / units;
    int64_t splits = want < (ntiles + 7) / 8 ? want : (ntiles + 7) / 8;
    if (splits < 1) splits = 1;
    if (splits > kMaxSlots) splits = kMaxSlots;
    int tps = (int)((ntiles + splits - 1) / splits);
    splits = (ntiles + tps - 1) / tps;
    if (splits < 1) splits = 1;
    dim3 grid((unsigned)splits, dh / HC, st->BH);
    launch_pdl(kern, grid, NT, sm, s, k, v, eta, static_cast<const R*>(st->W[0]), static_cast<const R*>(st->W[1]),
                              static_cast<const R*>(st->W[2]), dh, tps, static_cast<R*>(st->partial), st->BH);
    g_launches++;
    *slots = (int)splits;
    return cudaGetLastError();
}

template <int D>
cudaError_t apply_d(const lact_state* st, TokView q, void* o, cudaStream_t s) {
    if (st->f64) return apply_t<float, double, D>(st, q, o, s);
    return apply_t<bf16, float, D>(st, q, o, s);
}
template <int D>
cudaError_t grad_d(const lact_state* st, TokView k, TokView v, const float* eta, int* slots, cudaStream_t s) {
    if (st->f64) return grad_t<float, double, D>(st, k, v, eta, slots, s);
    return grad_t<bf16, float, D>(st, k, v, eta, slots, s);
}

}  // namespace

cudaError_t launch_apply_simt(const lact_state* st, TokView q, void* o, cudaStream_t s) {
    switch (st->cfg.d) {
        case 32: return apply_d<32>(st, q, o, s);
        case 64: return apply_d<64>(st, q, o, s);
        case 128: return apply_d<128>(st, q, o, s);
        case 256: return apply_d<256>(st, q, o, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_grad_simt(const lact_state* st, TokView k, TokView v, const float* eta, int* slots,
                             cudaStream_t s) {
    switch (st->cfg.d) {
        case 32: return grad_d<32>(st, k, v, eta, slots, s);
        case 64: return grad_d<64>(st, k, v, eta, slots, s);
        case 128: return grad_d<128>(st, k, v, eta, slots, s);
        case 256: return grad_d<256>(st, k, v, eta, slots, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_reduce(const lact_state* st, int slots, bool accumulate, void* const out[3], cudaStream_t s) {
    const size_t mat = (size_t)st->BH * st->cfg.dh * st->cfg.d;
    const size_t want = (st->nmat * mat + 255) / 256, cap = (size_t)st->num_sms * 8;
    const int blocks = (int)(want < cap ? want : cap);
    if (st->f64)
        launch_pdl(k_reduce<double>, blocks, 256, 0, s, static_cast<const double*>(st->partial), slots, mat, st->nmat,
                                                accumulate,
                                                static_cast<double*>(out[0]), static_cast<double*>(out[1]),
                                                static_cast<double*>(out[2]));
    else
        launch_pdl(k_reduce<float>, blocks, 256, 0, s, static_cast<const float*>(st->partial), slots, mat, st->nmat, accumulate,
                                               static_cast<float*>(out[0]), static_cast<float*>(out[1]),
                                               static_cast<float*>(out[2]));
    g_launches++;
    return cudaGetLastError();
}

}  // namespace lact

// ------------------------------------------------------------------------
// Raw-pointer launchers of the bf16-io gradient and reduction kernels above,
// for callers that hold no lact_state (the weights come straight from the
// caller, the partial sums go to a buffer the caller names).
namespace lact {

namespace {
template <int D>
cudaError_t grad_raw_d(int dh, int BH, const float* W1, const float* W2, const float* W3, TokView k, TokView v,
                       const float* eta, float* partial, int max_slots, int num_sms, int* slots, cudaStream_t s) {
    constexpr int TT = Tile<float>::TT, HC = Tile<float>::HC;
    auto kern = k_grad_simt<bf16, float, D>;
    const size_t sm = grad_smem<float, D>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    const int64_t ntiles = (k.n + TT - 1) / TT;
    const int units = BH * (dh / HC);
    int64_t want = (4LL * num_sms + units - 1) / units;
    int64_t splits = want < (ntiles + 7) / 8 ? want : (ntiles + 7) / 8;
    if (splits > max_slots) splits = max_slots;
    if (splits < 1) splits = 1;
    const int tps = (int)((ntiles + splits - 1) / splits);
    splits = (ntiles + tps - 1) / tps;
    if (splits < 1) splits = 1;
    dim3 grid((unsigned)splits, dh / HC, BH);
    launch_pdl(kern, grid, NT, sm, s, k, v, eta, W1, W2, W3, dh, tps, partial, BH);
    g_launches++;
    *slots = (int)splits;
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_grad_simt_bf16_raw(int d, int dh, int BH, const float* W1, const float* W2, const float* W3,
                                      TokView k, TokView v, const float* eta, float* partial, int max_slots,
                                      int num_sms, int* slots, cudaStream_t s) {
    switch (d) {
        case 32: return grad_raw_d<32>(dh, BH, W1, W2, W3, k, v, eta, partial, max_slots, num_sms, slots, s);
        case 64: return grad_raw_d<64>(dh, BH, W1, W2, W3, k, v, eta, partial, max_slots, num_sms, slots, s);
        case 128: return grad_raw_d<128>(dh, BH, W1, W2, W3, k, v, eta, partial, max_slots, num_sms, slots, s);
        case 256: return grad_raw_d<256>(dh, BH, W1, W2, W3, k, v, eta, partial, max_slots, num_sms, slots, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_reduce_f32_raw(const float* partial, int slots, size_t mat, float* o0, float* o1, float* o2,
                                  int num_sms, cudaStream_t s) {
    const size_t want = (3 * mat + 255) / 256, cap = (size_t)num_sms * 8;
    const int blocks = (int)(want < cap ? want : cap);
    launch_pdl(k_reduce<float>, blocks, 256, 0, s, partial, slots, mat, 3, false, o0, o1, o2);
    g_launches++;
    return cudaGetLastError();
}

}  // namespace lact
