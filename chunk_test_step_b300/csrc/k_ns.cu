// Muon step: quintic Newton-Schulz orthogonalisation of each gradient matrix
// (LaCT review page, "Local attention and nonlinear memory work together":
// Muon transforms matrix gradients with Newton-Schulz iterations).
//
// For every matrix G of the 3*B*H gradients, on the orientation with rows <=
// cols (m x n): X = G / (||G||_F + 1e-7), then ns_steps times
//     A = X X^T;  B = b A + c A A;  X = a X + B X
// with GEMM operands rounded to bf16 (X for X X^T, A for A A, B and X for
// B X); every sum and every stored matrix is in the state's internal real
// type (fp32, or fp64 for fp32-io states).
//
// This file is the generic CUDA-core form: one batched SIMT GEMM launch per
// product, over all matrices at once.
#include "lact_internal.cuh"

namespace lact {

namespace {

// Matrix mi of the batch: which gradient (0: W1, 1: W2, 2: W3) and head.
struct NsShape { int m, n, d, dh, BH; };

__device__ __forceinline__ void src_dims(int which, int d, int dh, int& rows, int& cols) {
    if (which == 1) { rows = d; cols = dh; } else { rows = dh; cols = d; }
}

// X[mi] = G / (||G||_F + eps), transposed when G has more rows than columns.
template <typename R>
__global__ void k_ns_prep(const R* __restrict__ g0, const R* __restrict__ g1,
                          const R* __restrict__ g2, R* __restrict__ X, NsShape sh, R eps) {
    pdl_wait();
    const int mi = blockIdx.x;
    const int which = mi / sh.BH, bh = mi % sh.BH;
    const R* G = (which == 0 ? g0 : which == 1 ? g1 : g2) + (size_t)bh * sh.d * sh.dh;
    int rows, cols;
    src_dims(which, sh.d, sh.dh, rows, cols);
    const int total = rows * cols;
    R ss = 0;
    for (int i = threadIdx.x; i < total; i += blockDim.x) ss = fma_r(G[i], G[i], ss);
    __shared__ R red[32];
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x < 32) {
        R t = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : R(0);
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (threadIdx.x == 0) red[0] = t;
    }
    __syncthreads();
    const R nrm = sqrt_r(red[0]) + eps;
    R* Xm = X + (size_t)mi * sh.m * sh.n;
    const bool tr = rows > cols;
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
        // i indexes X (m x n) row-major
        const int r = i / sh.n, c = i % sh.n;
        const R gv = tr ? G[(size_t)c * cols + r] : G[(size_t)r * cols + c];
        Xm[i] = gv / nrm;
    }
}

// G[mi] <- X[mi] back in the gradient's own orientation.
template <typename R>
__global__ void k_ns_unpack(const R* __restrict__ X, R* __restrict__ g0, R* __restrict__ g1,
                            R* __restrict__ g2, NsShape sh) {
    pdl_wait();
    const int mi = blockIdx.x;
    const int which = mi / sh.BH, bh = mi % sh.BH;
    R* G = (which == 0 ? g0 : which == 1 ? g1 : g2) + (size_t)bh * sh.d * sh.dh;
    int rows, cols;
    src_dims(which, sh.d, sh.dh, rows, cols);
    const bool tr = rows > cols;
    const R* Xm = X + (size_t)mi * sh.m * sh.n;
    for (int i = threadIdx.x; i < rows * cols; i += blockDim.x) {
        const int r = i / cols, c = i % cols;
        G[i] = tr ? Xm[(size_t)c * sh.n + r] : Xm[(size_t)r * sh.n + c];
    }
}

// Batched C = alpha * rnd(A) rnd(op(B)) + beta * Cin, all row-major fp32.
// A: [M, K]; B: [K, N] (transB = 0) or [N, K] (transB = 1); rnd = bf16 rounding.
// (16 TPT) x (16 TPT) output tile per CTA, 256 threads, TPT x TPT outputs per
// thread; every output sums over k in order, so the tile size does not change
// the result. TPT = 1 gives small matrices (the fp32-io layers' 64 x 64
// products) enough CTAs to spread over the GPU.
constexpr int BK = 16;

template <typename R, int TPT>
__global__ void __launch_bounds__(256) k_bgemm(const R* __restrict__ A, const R* __restrict__ B,
                                               const R* __restrict__ Cin, R* __restrict__ C,
                                               int M, int N, int K, size_t sA, size_t sB, size_t sC,
                                               int transB, R alpha, R beta) {
    pdl_wait();
    constexpr int BM = 16 * TPT, BN = 16 * TPT;
    __shared__ R As[BK][BM + 4];
    __shared__ R Bs[BK][BN + 4];
    const int bz = blockIdx.z;
    A += bz * sA; B += bz * sB; C += bz * sC;
    if (Cin) Cin += bz * sC;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    R acc[TPT][TPT];
#pragma unroll
    for (int i = 0; i < TPT; ++i)
#pragma unroll
        for (int j = 0; j < TPT; ++j) acc[i][j] = R(0);
    for (int k0 = 0; k0 < K; k0 += BK) {
        for (int i = tid; i < BM * BK; i += 256) {
            const int r = i / BK, kk = i % BK;
            const int gm = m0 + r, gk = k0 + kk;
            As[kk][r] = (gm < M && gk < K) ? round_bf16(A[(size_t)gm * K + gk]) : R(0);
        }
        for (int i = tid; i < BN * BK; i += 256) {
            int nn, kk;
            if (transB) { nn = i / BK; kk = i % BK; } else { kk = i / BN; nn = i % BN; }
            const int gn = n0 + nn, gk = k0 + kk;
            R x = 0;
            if (gn < N && gk < K) x = transB ? B[(size_t)gn * K + gk] : B[(size_t)gk * N + gn];
            Bs[kk][nn] = round_bf16(x);
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            R a[TPT], b[TPT];
#pragma unroll
            for (int i = 0; i < TPT; ++i) { a[i] = As[kk][ty + 16 * i]; b[i] = Bs[kk][tx + 16 * i]; }
#pragma unroll
            for (int i = 0; i < TPT; ++i)
#pragma unroll
                for (int j = 0; j < TPT; ++j) acc[i][j] = fma_r(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < TPT; ++i)
#pragma unroll
        for (int j = 0; j < TPT; ++j) {
            const int gm = m0 + ty + 16 * i, gn = n0 + tx + 16 * j;
            if (gm < M && gn < N) {
                const size_t o = (size_t)gm * N + gn;
                R r = alpha * acc[i][j];
                if (Cin) r = fma_r(beta, Cin[o], r);
                C[o] = r;
            }
        }
}

template <typename R>
cudaError_t bgemm(const R* A, const R* B, const R* Cin, R* C, int M, int N, int K,
                  size_t sA, size_t sB, size_t sC, int transB, R alpha, R beta, int batch,
                  cudaStream_t s) {
    // 64 x 64 tiles when they alone give a few waves of CTAs, else 16 x 16
    const int64_t big = (int64_t)((N + 63) / 64) * ((M + 63) / 64) * batch;
    if (big >= 4 * 148) {
        dim3 grid((N + 63) / 64, (M + 63) / 64, batch);
        launch_pdl(k_bgemm<R, 4>, grid, 256, 0, s, A, B, Cin, C, M, N, K, sA, sB, sC, transB, alpha, beta);
    } else {
        dim3 grid((N + 15) / 16, (M + 15) / 16, batch);
        launch_pdl(k_bgemm<R, 1>, grid, 256, 0, s, A, B, Cin, C, M, N, K, sA, sB, sC, transB, alpha, beta);
    }
    g_launches++;
    return cudaGetLastError();
}

template <typename R>
cudaError_t ns_t(const lact_state* st, void* const gv[3], cudaStream_t s) {
    const lact_config& c = st->cfg;
    NsShape sh;
    sh.d = c.d; sh.dh = c.dh; sh.BH = st->BH;
    sh.m = c.d < c.dh ? c.d : c.dh;
    sh.n = c.d < c.dh ? c.dh : c.d;
    const int batch = st->nmat * st->BH;
    R* g[3] = {static_cast<R*>(gv[0]), static_cast<R*>(gv[1]), static_cast<R*>(gv[2])};
    R* X = static_cast<R*>(st->ns[0]);
    R* X2 = static_cast<R*>(st->ns[1]);
    R* Am = static_cast<R*>(st->ns[2]);
    R* Bm = static_cast<R*>(st->ns[3]);
    const size_t sX = (size_t)sh.m * sh.n, sA = (size_t)sh.m * sh.m;
    launch_pdl(k_ns_prep<R>, batch, 256, 0, s, g[0], g[1], g[2], X, sh, R(1e-7));
    g_launches++;
    cudaError_t e = cudaGetLastError();
    for (int it = 0; it < c.ns_steps && e == cudaSuccess; ++it) {
        // A = rnd(X) rnd(X)^T
        e = bgemm<R>(X, X, nullptr, Am, sh.m, sh.m, sh.n, sX, sX, sA, 1, R(1), R(0), batch, s);
        if (e != cudaSuccess) break;
        // B = c * rnd(A) rnd(A) + b * A
        e = bgemm<R>(Am, Am, Am, Bm, sh.m, sh.m, sh.m, sA, sA, sA, 0, R(c.ns_c), R(c.ns_b), batch, s);
        if (e != cudaSuccess) break;
        // X' = rnd(B) rnd(X) + a * X
        e = bgemm<R>(Bm, X, X, X2, sh.m, sh.n, sh.m, sA, sX, sX, 0, R(1), R(c.ns_a), batch, s);
        R* t = X; X = X2; X2 = t;
    }
    if (e != cudaSuccess) return e;
    launch_pdl(k_ns_unpack<R>, batch, 256, 0, s, X, g[0], g[1], g[2], sh);
    g_launches++;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_newton_schulz(const lact_state* st, void* const g[3], cudaStream_t s) {
    return st->f64 ? ns_t<double>(st, g, s) : ns_t<float>(st, g, s);
}

}  // namespace lact
