// The linear fast-weight memory: one d x d matrix W per (batch, head),
// read as o = W q (LaCT review page, "Local attention and nonlinear memory
// work together" and Fig. 8: the larger linear state that the smaller SwiGLU
// state is compared against). Its loss L = -sum_i eta_i <W k_i, v_i> has the
// chunk gradient dL/dW = -sum_i eta_i v_i k_i^T.
//
// Kernels here:
//   k_lin_apply_simt, k_lin_grad_simt - CUDA cores, any io dtype, the
//       internal real type (fp64 for fp32 io): the accuracy path;
//   k_lin_apply_tc - the readout on the tensor cores for bf16 io at d = 128:
//       per 128-query tile, O = Q W^T as one tcgen05 GEMM (Q and the bf16
//       shadow of W K-major, fp32 accumulator in TMEM).
// The gradient on the tensor cores is k_wgrad_tc with its A operand (V)
// scaled by -eta in shared memory (k_tc_wgrad.cu).
#include "lact_internal.cuh"
#include "tc_ptx.cuh"

namespace lact {

namespace {

constexpr int NT = 256;
constexpr int LT = 32;          // tokens per tile of the CUDA-core readout
constexpr int LG = 16;          // tokens per tile of the CUDA-core gradient

// o[t][i] = sum_j W[i][j] q[t][j]: one CTA per (32-token tile, head); the
// tile's queries are staged in shared memory as reals.
template <typename T, typename R>
__global__ void __launch_bounds__(NT) k_lin_apply_simt(TokView q, T* __restrict__ o, const R* __restrict__ W,
                                                       int d) {
    pdl_wait();
    extern __shared__ __align__(16) unsigned char smraw[];
    R* qs = reinterpret_cast<R*>(smraw);           // [LT][d]
    const int bh = blockIdx.y;
    const int64_t t0 = (int64_t)blockIdx.x * LT;
    const T* qp = static_cast<const T*>(q.p) + ((int64_t)bh * q.n_total + q.t0) * d;
    for (int i = threadIdx.x; i < LT * d; i += NT) {
        const int t = i / d, j = i % d;
        qs[i] = (t0 + t < q.n) ? ld_io<R>(qp, (t0 + t) * d + j) : R(0);
    }
    __syncthreads();
    const R* Wh = W + (size_t)bh * d * d;
    T* op = o + ((int64_t)bh * q.n_total + q.t0) * d;
    for (int i = threadIdx.x; i < LT * d; i += NT) {
        const int t = i / d, r = i % d;
        if (t0 + t >= q.n) continue;
        R acc = 0;
        for (int j = 0; j < d; ++j) acc = fma_r(Wh[(size_t)r * d + j], qs[t * d + j], acc);
        st_io(op, (t0 + t) * d + r, acc);
    }
}

// Partial dL/dW over a token range: partial[split][bh][i][j] =
// -sum_t eta_t v[t][i] k[t][j]. One CTA per (split, head); every thread owns
// d*d/256 entries and walks the range in 16-token tiles staged in shared
// memory (v already scaled by -eta).
template <typename T, typename R, int D>
__global__ void __launch_bounds__(NT) k_lin_grad_simt(TokView k, TokView v, const float* __restrict__ eta,
                                                      int tps, R* __restrict__ partial, int BH) {
    pdl_wait();
    __shared__ R ks[LG][D + 1];
    __shared__ R vs[LG][D + 1];
    constexpr int PER = D * D / NT;
    const int split = blockIdx.x, bh = blockIdx.y;
    const int64_t a0 = (int64_t)split * tps * LG;
    const int64_t a1 = min(k.n, a0 + (int64_t)tps * LG);
    const T* kp = static_cast<const T*>(k.p) + ((int64_t)bh * k.n_total + k.t0) * D;
    const T* vp = static_cast<const T*>(v.p) + ((int64_t)bh * v.n_total + v.t0) * D;
    const float* ep = eta + (int64_t)bh * k.n_total + k.t0;
    R acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0;
    for (int64_t b0 = a0; b0 < a1; b0 += LG) {
        __syncthreads();
        for (int i = threadIdx.x; i < LG * D; i += NT) {
            const int t = i / D, j = i % D;
            const bool live = b0 + t < a1;
            ks[t][j] = live ? ld_io<R>(kp, (b0 + t) * D + j) : R(0);
            vs[t][j] = live ? -(R)ep[b0 + t] * ld_io<R>(vp, (b0 + t) * D + j) : R(0);
        }
        __syncthreads();
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            const int idx = threadIdx.x + e * NT, r = idx / D, c = idx % D;
            R s = acc[e];
            for (int t = 0; t < LG; ++t) s = fma_r(vs[t][r], ks[t][c], s);
            acc[e] = s;
        }
    }
    R* out = partial + ((size_t)split * BH + bh) * D * D;
#pragma unroll
    for (int e = 0; e < PER; ++e) out[threadIdx.x + e * NT] = acc[e];
}

// ------------------------------------------------ tensor-core readout, d = 128
using namespace tc;
constexpr int TD = 128;
constexpr uint32_t TBOX = 128 * 128;                    // [128 rows][64 bf16] = 16 KB
constexpr uint32_t TSMEM = 4 * TBOX + 1024;             // Q (2 atoms), W (2 atoms)
constexpr uint64_t TWAIT_NS = 2000000000ull;

struct LinApplyArgs {
    bf16* o;
    int64_t n_total, t0, n;
    int* status;
};

__global__ void __launch_bounds__(128, 1)
k_lin_apply_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_w, const LinApplyArgs a) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(16) unsigned char smraw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ uint32_t tmem_slot;
    __shared__ int ok_sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = blockIdx.x, bh = blockIdx.y;
    const uint32_t base = smem_u32(sm);
    const uint32_t b_ld = smem_u32(&bars[0]), b_mma = smem_u32(&bars[1]);
    if (tid == 0) {
        ok_sh = (*reinterpret_cast<volatile int*>(a.status) & ST_TIMEOUT) ? 0 : 1;
        mbar_init(b_ld, 1);
        mbar_init(b_mma, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (!ok_sh) return;
    if (warp == 0) {
        __syncwarp();
        tmem_alloc(smem_u32(&tmem_slot), 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    if (tid == 0) {
        const int tok = (int)(a.t0 + (int64_t)tile * 128);
        mbar_expect_tx(b_ld, 4 * TBOX);
        for (int at = 0; at < 2; ++at) {
            tma_load_3d(base + at * TBOX, &tm_q, b_ld, at * 64, tok, bh);
            tma_load_2d(base + (2 + at) * TBOX, &tm_w, b_ld, at * 64, bh * TD);
        }
        bool ok = mbar_wait(b_ld, 0, TWAIT_NS);
        if (ok) {
            tc_fence_after();
            const uint32_t idesc = idesc_bf16_f32(128, TD, 0, 0);
            const uint64_t dQ = sdesc_sw128(base, 16, 1024), dW = sdesc_sw128(base + 2 * TBOX, 16, 1024);
#pragma unroll
            for (int j = 0; j < TD / 16; ++j) {
                const uint64_t ko = (uint64_t)((j >> 2) * TBOX + (j & 3) * 32) >> 4;
                mma_bf16(tmem, dQ + ko, dW + ko, idesc, j > 0 ? 1u : 0u);
            }
        } else {
            atomicOr(a.status, ST_TIMEOUT);
            ok_sh = 0;
        }
        mma_commit(b_mma);   // also the drain of any MMA issued above
    }
    __syncwarp();
    // every warp: its 32 TMEM lanes = 32 queries, 128 output columns
    const bool done = mbar_wait_warp(b_mma, 0, TWAIT_NS);
    __syncthreads();
    if (done && ok_sh) {
        tc_fence_after();
        const int row = 32 * warp + lane;
        const int64_t tok = (int64_t)tile * 128 + row;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * warp) << 16);
#pragma unroll
        for (int h = 0; h < TD / 32; ++h) {
            uint32_t v[32], pk[16];
            tmem_ld32(lane_base + h * 32, v);
            tmem_wait_ld();
            tmem_pin(v);
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                __nv_bfloat162 p = __floats2bfloat162_rn(__uint_as_float(v[j]), __uint_as_float(v[j + 1]));
                pk[j / 2] = *reinterpret_cast<uint32_t*>(&p);
            }
            // four lanes store one row's 64 bytes together after a transpose
            // within each quad of lanes (whole 32-byte sectors per warp store)
            uint4 ch[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) ch[c] = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            quad_transpose(ch, lane);
            const int64_t quad_tok = tok - (lane & 3);
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4)
                if (quad_tok + k4 < a.n)
                    *reinterpret_cast<uint4*>(a.o + ((int64_t)bh * a.n_total + a.t0 + quad_tok + k4) * TD + h * 32 +
                                              8 * (lane & 3)) = ch[k4];
        }
    } else if (tid == 0 && !done) {
        atomicOr(a.status, ST_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 128);
    }
}

template <typename T, typename R>
cudaError_t lin_apply_t(const lact_state* st, TokView q, void* o, cudaStream_t s) {
    const int d = st->cfg.d;
    const size_t sm = sizeof(R) * LT * d;
    cudaError_t e = cudaFuncSetAttribute(k_lin_apply_simt<T, R>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((q.n + LT - 1) / LT), st->BH);
    launch_pdl(k_lin_apply_simt<T, R>, grid, NT, sm, s, q, static_cast<T*>(o), static_cast<const R*>(st->W[0]), d);
    g_launches++;
    return cudaGetLastError();
}

template <typename T, typename R, int D>
cudaError_t lin_grad_t(const lact_state* st, TokView k, TokView v, const float* eta, int* slots, cudaStream_t s) {
    const int64_t ntiles = (k.n + LG - 1) / LG;
    // about two waves of CTAs, each at least 4 tiles, at most kMaxSlots splits
    int64_t splits = (2LL * st->num_sms + st->BH - 1) / st->BH;
    if (splits > (ntiles + 3) / 4) splits = (ntiles + 3) / 4;
    if (splits > kMaxSlots) splits = kMaxSlots;
    if (splits < 1) splits = 1;
    const int tps = (int)((ntiles + splits - 1) / splits);
    splits = (ntiles + tps - 1) / tps;
    if (splits < 1) splits = 1;
    dim3 grid((unsigned)splits, st->BH);
    launch_pdl(k_lin_grad_simt<T, R, D>, grid, NT, 0, s, k, v, eta, tps, static_cast<R*>(st->partial), st->BH);
    g_launches++;
    *slots = (int)splits;
    return cudaGetLastError();
}

template <int D>
cudaError_t lin_grad_d(const lact_state* st, TokView k, TokView v, const float* eta, int* slots, cudaStream_t s) {
    if (st->f64) return lin_grad_t<float, double, D>(st, k, v, eta, slots, s);
    return lin_grad_t<bf16, float, D>(st, k, v, eta, slots, s);
}

}  // namespace

bool lin_tc_supported(const lact_state* st) {
    return st->cfg.io_dtype == LACT_BF16 && st->cfg.d == TD && tmap_available();
}

cudaError_t launch_lin_apply(const lact_state* st, TokView q, void* o, cudaStream_t s) {
    if (!lin_tc_supported(st)) {
        if (st->f64) return lin_apply_t<float, double>(st, q, o, s);
        return lin_apply_t<bf16, float>(st, q, o, s);
    }
    CUtensorMap mq, mw;
    const int BH = st->BH;
    const uint64_t q_dims[3] = {(uint64_t)TD, (uint64_t)q.n_total, (uint64_t)BH};
    const uint64_t q_str[2] = {(uint64_t)TD * 2, (uint64_t)q.n_total * TD * 2};
    const uint32_t q_box[3] = {64, 128, 1};
    const uint64_t w_dims[2] = {(uint64_t)TD, (uint64_t)BH * TD};
    const uint64_t w_str[1] = {(uint64_t)TD * 2};
    const uint32_t w_box[2] = {64, 128};
    if (!make_tmap_bf16(&mq, q.p, 3, q_dims, q_str, q_box) || !make_tmap_bf16(&mw, st->Wsh[0], 2, w_dims, w_str, w_box))
        return cudaErrorInvalidValue;
    LinApplyArgs la;
    la.o = static_cast<bf16*>(o);
    la.n_total = q.n_total;
    la.t0 = q.t0;
    la.n = q.n;
    la.status = st->status;
    cudaError_t e = cudaFuncSetAttribute(k_lin_apply_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TSMEM);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((q.n + 127) / 128), BH);
    launch_pdl(k_lin_apply_tc, grid, 128, TSMEM, s, mq, mw, la);
    g_launches++;
    g_tc_launches++;
    return cudaGetLastError();
}

cudaError_t launch_lin_grad_simt(const lact_state* st, TokView k, TokView v, const float* eta, int* slots,
                                 cudaStream_t s) {
    switch (st->cfg.d) {
        case 32: return lin_grad_d<32>(st, k, v, eta, slots, s);
        case 64: return lin_grad_d<64>(st, k, v, eta, slots, s);
        case 128: return lin_grad_d<128>(st, k, v, eta, slots, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace lact
