// Muon's Newton-Schulz orthogonalisation on the sm_103a tensor cores
// (LaCT review page, "Local attention and nonlinear memory work together":
// Muon transforms each matrix gradient with Newton-Schulz iterations).
//
// One CTA per gradient matrix G (3 per head), for matrices whose short side is
// 128 and long side n <= 512 (a multiple of 64). On the orientation with
// rows <= cols (X is 128 x n):
//   X = G / (||G||_F + 1e-7)
//   repeat ns_steps times:
//     A  = Xb Xb^T             Xb = bf16(X): K-major operand, both sides   (TMEM)
//     AA = Ab Ab               Ab = bf16(A): K-major A, MN-major B        (TMEM)
//     B  = b A + c AA          fp32, from the unrounded A
//     BX = Bb Xb               Bb = bf16(B) K-major; Xb read MN-major     (TMEM)
//     X  = a X + BX            fp32
// The bf16 copy Xb stays in shared memory for the whole iteration (it is the
// operand of two GEMMs in two orientations); the fp32 X lives in an
// L2-resident scratch row per thread. The result overwrites G in G's own
// orientation.
//
// 256 threads: thread = row of X (TMEM lane) and half of its columns; thread
// 0 also issues the MMAs. Every wait is bounded and its outcome made
// block-uniform before any barrier that depends on it.
#include "lact_internal.cuh"
#include "tc_ptx.cuh"

namespace lact {

namespace {

using namespace tc;

constexpr int M = 128;
constexpr int NMAX = 512;
constexpr int NTHREADS = 256;
constexpr uint32_t ATOM = M * 128;                 // [128 rows][64 bf16] = 16 KB
constexpr uint32_t OFF_X = 0;                      // n/64 atoms of Xb
constexpr uint32_t OFF_A = (NMAX / 64) * ATOM;     // 2 atoms of Ab
constexpr uint32_t OFF_B = OFF_A + 2 * ATOM;       // 2 atoms of Bb
constexpr uint32_t SMEM_BYTES = OFF_B + 2 * ATOM + 1024;
constexpr uint32_t COL_A = 0, COL_AA = 128, COL_BX = 0;
constexpr uint64_t WAIT_NS = 2000000000ull;

struct NsArgs {
    float* g[3];      // gradients in place: W1 [BH,dh,d], W2 [BH,d,dh], W3 [BH,dh,d]
    float* xs;        // fp32 X scratch [3*BH][M][n]
    int BH, d, dh, n, steps;
    float a, b, c;
    int* status;
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&p);
}

// Offset of element (row, col) in a K-major operand made of 64-column atoms.
__device__ __forceinline__ uint32_t atom_off(uint32_t row, uint32_t col) {
    return (col >> 6) * ATOM + sw128_offset(row, col & 63u);
}

__device__ __forceinline__ uint4 pack8(const float* x) {
    return make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]), pack_bf16(x[6], x[7]));
}

__global__ void __launch_bounds__(NTHREADS, 1) k_ns_tc(const NsArgs a) {
    extern __shared__ __align__(16) unsigned char smraw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t mbar;
    __shared__ uint32_t tmem_slot;
    __shared__ float red[NTHREADS / 32];
    __shared__ int failed;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int mi = blockIdx.x, which = mi / a.BH, bh = mi % a.BH;
    const int rows = which == 1 ? a.d : a.dh, cols = which == 1 ? a.dh : a.d;
    const bool tr = rows > cols;
    const int n = a.n;
    float* G = a.g[which] + (size_t)bh * a.d * a.dh;
    float* X = a.xs + (size_t)mi * M * n;
    const uint32_t base = smem_u32(sm);
    const uint32_t bar = smem_u32(&mbar);

    if (tid == 0) {
        failed = (*reinterpret_cast<volatile int*>(a.status) & ST_TIMEOUT) ? 1 : 0;
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (failed) return;
    if (warp == 1) {
        __syncwarp();
        tmem_alloc(smem_u32(&tmem_slot), 512);
        tmem_relinquish();
    }
    // ---- X = G / (||G||_F + eps), as fp32 rows and as the bf16 operand
    float ss = 0.f;
    for (int i = tid; i < rows * cols; i += NTHREADS) ss = fmaf(G[i], G[i], ss);
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) red[warp] = ss;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    float tot = 0.f;
    for (int w = 0; w < NTHREADS / 32; ++w) tot += red[w];
    const float nrm = sqrtf(tot) + 1e-7f;
    const int q = warp & 3, half = warp >> 2;
    const int row = 32 * q + lane;             // row of X owned by this thread
    const int nh = n / 2;                      // its columns: [half * nh, half * nh + nh)
    // Element (row, j) of X is G[row][j], or G[j][row] when G is stored tall:
    // either way a warp's 32 rows read 32 consecutive or row-contiguous words.
    for (int c0 = half * nh; c0 < half * nh + nh; c0 += 8) {
        float x[8];
#pragma unroll
        for (int t = 0; t < 8; ++t)
            x[t] = (tr ? G[(size_t)(c0 + t) * cols + row] : G[(size_t)row * cols + c0 + t]) / nrm;
        float* xr = X + (size_t)row * n + c0;
        *reinterpret_cast<float4*>(xr) = make_float4(x[0], x[1], x[2], x[3]);
        *reinterpret_cast<float4*>(xr + 4) = make_float4(x[4], x[5], x[6], x[7]);
        *reinterpret_cast<uint4*>(sm + OFF_X + atom_off(row, c0)) = pack8(x);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
    uint32_t phase = 0;
    bool ok = true;

    // Wait for the MMAs just committed; the outcome is made block-uniform so
    // that every thread takes the same path through the barriers below.
    auto mma_done = [&]() -> bool {
        const bool r = __syncthreads_and(mbar_wait(bar, phase & 1, WAIT_NS) ? 1 : 0) != 0;
        __syncwarp();
        ++phase;
        tc_fence_after();
        return r;
    };
    auto sync_smem = [&]() {
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    };

    const uint32_t i_xx = idesc_bf16_f32(M, M, 0, 0);
    const uint32_t i_aa = idesc_bf16_f32(M, M, 0, 1);
    const uint64_t dX = sdesc_sw128(base + OFF_X, 16, 1024);      // Xb K-major
    const uint64_t dXmn = sdesc_sw128(base + OFF_X, ATOM, 1024);  // Xb MN-major
    const uint64_t dA = sdesc_sw128(base + OFF_A, 16, 1024);      // Ab K-major
    const uint64_t dAmn = sdesc_sw128(base + OFF_A, ATOM, 1024);  // Ab MN-major
    const uint64_t dB = sdesc_sw128(base + OFF_B, 16, 1024);      // Bb K-major
    for (int it = 0; it < a.steps && ok; ++it) {
        // A = Xb Xb^T
        if (tid == 0) {
            for (int j = 0; j < n / 16; ++j) {
                const uint64_t ko = (uint64_t)((j >> 2) * ATOM + (j & 3) * 32) >> 4;
                mma_bf16(tmem + COL_A, dX + ko, dX + ko, i_xx, j > 0 ? 1u : 0u);
            }
            mma_commit(bar);
        }
        if (!mma_done()) { ok = false; break; }
        // Ab = bf16(A)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t v[32];
            const int c0 = half * 64 + h * 32;
            tmem_ld32(lane_base + COL_A + c0, v);
            tmem_wait_ld();
            tmem_pin(v);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float x[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) x[t] = __uint_as_float(v[8 * c + t]);
                *reinterpret_cast<uint4*>(sm + OFF_A + atom_off(row, c0 + 8 * c)) = pack8(x);
            }
        }
        sync_smem();
        // AA = Ab Ab
        if (tid == 0) {
#pragma unroll
            for (int j = 0; j < M / 16; ++j) {
                const uint64_t ko = (uint64_t)((j >> 2) * ATOM + (j & 3) * 32) >> 4;
                mma_bf16(tmem + COL_AA, dA + ko, dAmn + j * 128, i_aa, j > 0 ? 1u : 0u);
            }
            mma_commit(bar);
        }
        if (!mma_done()) { ok = false; break; }
        // Bb = bf16(b A + c AA)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t va[32], vaa[32];
            const int c0 = half * 64 + h * 32;
            tmem_ld32(lane_base + COL_A + c0, va);
            tmem_ld32(lane_base + COL_AA + c0, vaa);
            tmem_wait_ld();
            tmem_pin(va);
            tmem_pin(vaa);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float bv[8];
#pragma unroll
                for (int t = 0; t < 8; ++t)
                    bv[t] = fmaf(a.c, __uint_as_float(vaa[8 * c + t]), a.b * __uint_as_float(va[8 * c + t]));
                *reinterpret_cast<uint4*>(sm + OFF_B + atom_off(row, c0 + 8 * c)) = pack8(bv);
            }
        }
        sync_smem();
        // BX = Bb Xb (N in pieces of at most 256)
        if (tid == 0) {
            for (int nb = 0; nb < n; nb += 256) {
                const int nn = n - nb < 256 ? n - nb : 256;
                const uint32_t idx = idesc_bf16_f32(M, nn, 0, 1);
                const uint64_t xo = (uint64_t)((nb / 64) * ATOM) >> 4;
#pragma unroll
                for (int j = 0; j < M / 16; ++j) {
                    const uint64_t ko = (uint64_t)((j >> 2) * ATOM + (j & 3) * 32) >> 4;
                    mma_bf16(tmem + COL_BX + nb, dB + ko, dXmn + xo + j * 128, idx, j > 0 ? 1u : 0u);
                }
            }
            mma_commit(bar);
        }
        if (!mma_done()) { ok = false; break; }
        // X = a X + BX; Xb = bf16(X). The fp32 row chunk is fetched before the
        // TMEM load so its L2 latency overlaps it.
        for (int c0 = half * nh; c0 < half * nh + nh; c0 += 32) {
            float* xr = X + (size_t)row * n + c0;
            float4 x4[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) x4[t] = *reinterpret_cast<const float4*>(xr + 4 * t);
            uint32_t v[32];
            tmem_ld32(lane_base + COL_BX + c0, v);
            tmem_wait_ld();
            tmem_pin(v);
            float xn[32];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                xn[4 * t + 0] = fmaf(a.a, x4[t].x, __uint_as_float(v[4 * t + 0]));
                xn[4 * t + 1] = fmaf(a.a, x4[t].y, __uint_as_float(v[4 * t + 1]));
                xn[4 * t + 2] = fmaf(a.a, x4[t].z, __uint_as_float(v[4 * t + 2]));
                xn[4 * t + 3] = fmaf(a.a, x4[t].w, __uint_as_float(v[4 * t + 3]));
                *reinterpret_cast<float4*>(xr + 4 * t) =
                    make_float4(xn[4 * t], xn[4 * t + 1], xn[4 * t + 2], xn[4 * t + 3]);
            }
#pragma unroll
            for (int c = 0; c < 4; ++c)
                *reinterpret_cast<uint4*>(sm + OFF_X + atom_off(row, c0 + 8 * c)) = pack8(xn + 8 * c);
        }
        sync_smem();
    }
    if (!ok) {
        if (lane == 0) atomicOr(a.status, ST_TIMEOUT);
    } else {
        // result back into G's own orientation (this thread's row, as read)
        for (int c0 = half * nh; c0 < half * nh + nh; c0 += 4) {
            const float4 x4 = *reinterpret_cast<const float4*>(X + (size_t)row * n + c0);
            if (tr) {
                G[(size_t)(c0 + 0) * cols + row] = x4.x;
                G[(size_t)(c0 + 1) * cols + row] = x4.y;
                G[(size_t)(c0 + 2) * cols + row] = x4.z;
                G[(size_t)(c0 + 3) * cols + row] = x4.w;
            } else {
                *reinterpret_cast<float4*>(G + (size_t)row * cols + c0) = x4;
            }
        }
    }
    // every MMA has completed once this commit lands (bounded drain), then
    // TMEM is freed
    if (tid == 0) {
        mma_commit(bar);
        mbar_wait(bar, phase & 1, WAIT_NS);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

bool ns_tc_supported(const lact_state* st) {
    const int m = st->cfg.d < st->cfg.dh ? st->cfg.d : st->cfg.dh;
    const int n = st->cfg.d < st->cfg.dh ? st->cfg.dh : st->cfg.d;
    return st->cfg.io_dtype == LACT_BF16 && m == M && n <= NMAX && n % 64 == 0;
}

cudaError_t launch_ns_tc(const lact_state* st, void* const g[3], cudaStream_t s) {
    NsArgs a;
    for (int m = 0; m < 3; ++m) a.g[m] = static_cast<float*>(g[m]);
    a.xs = static_cast<float*>(st->ns[0]);
    a.BH = st->BH;
    a.d = st->cfg.d;
    a.dh = st->cfg.dh;
    a.n = st->cfg.d < st->cfg.dh ? st->cfg.dh : st->cfg.d;
    a.steps = st->cfg.ns_steps;
    a.a = (float)st->cfg.ns_a;
    a.b = (float)st->cfg.ns_b;
    a.c = (float)st->cfg.ns_c;
    a.status = st->status;
    cudaError_t e = cudaFuncSetAttribute(k_ns_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    k_ns_tc<<<3 * st->BH, NTHREADS, SMEM_BYTES, s>>>(a);
    g_launches++;
    g_tc_launches++;
    return cudaGetLastError();
}

}  // namespace lact
