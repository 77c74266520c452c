// Readout of the SwiGLU fast-weight memory on the sm_103a tensor cores
// (tcgen05 + TMA + TMEM), bf16 io, head dim D = 128 or 256:
//     o_i = W2 (silu(W1 q_i) * (W3 q_i))
// (LaCT review page, "Fast weights are temporary context memory": queries
// read the adapted weights; "Local attention and nonlinear memory work
// together": the three-matrix SwiGLU memory).
//
// One CTA per (head, 128-query tile). The hidden units are visited in blocks
// r of 64:
//   [H1 | H3] (TMEM, double-buffered) = Q . [W1_r ; W3_r]^T   (A, B K-major)
//   U_r = silu(H1) * H3 -> bf16, swizzled K-major operand       (epilogue)
//   O (TMEM, D cols) += U_r . W2[:, r]^T                        (A, B K-major)
// so the MMA of block r+1 overlaps the epilogue of block r. At D = 128 the W
// blocks are double-buffered through TMA; at D = 256 a W block is 96 KB and
// single-buffered, and the blocks run one after another. At the end O leaves
// TMEM as bf16.
//
// Warp roles (320 threads): warp 0 TMA, warp 1 TMEM owner + MMA issuer,
// warps 2..9 epilogue (thread = query, 32 of the 64 hidden units). Every
// wait is bounded; a wait that gives up sets ST_TIMEOUT and the CTA unwinds.
#include "lact_internal.cuh"
#include "tc_ptx.cuh"

namespace lact {

namespace {

using namespace tc;

constexpr int HB = 64;
constexpr int TT = 128;
constexpr int NTHREADS = 320;
constexpr uint32_t BOX = TT * 128;                  // [128 rows][64 bf16], 16 KB

// Shared-memory layout for head dim D with `WS` W-block stages.
template <int D, int WS>
struct ApplyLayout {
    static constexpr uint32_t OFF_Q = 0;                                  // D/64 k-atoms of the query tile
    static constexpr uint32_t OFF_W = (D / 64) * BOX;                     // stage s: Wcat (D/64 atoms), W2 (D rows)
    static constexpr uint32_t WC_BYTES = (D / 64) * BOX;
    static constexpr uint32_t W2_BYTES = D * 128;
    static constexpr uint32_t W_STAGE = WC_BYTES + W2_BYTES;
    static constexpr uint32_t OFF_U = OFF_W + WS * W_STAGE;               // 2 buffers of [128 tok][64 hid]
    static constexpr uint32_t SMEM_BYTES = OFF_U + 2 * BOX + 1024;
};

constexpr uint32_t COL_H13 = 0;     // buffer b at b * 128: H1 (64) | H3 (64)
constexpr uint32_t COL_O = 256;     // D columns
constexpr uint32_t TMEM_COLS = 512;
constexpr uint64_t WAIT_NS = 2000000000ull;

enum { B_Q = 0, B_WF = 1, B_WE = 3, B_HF = 5, B_HE = 7, B_UF = 9, B_UE = 11, B_O = 13, B_DRAIN = 14, NBARS = 15 };

struct ApplyArgs {
    bf16* o;             // [BH, n_total, D], same layout as q
    int64_t n_total;
    int64_t t0;
    int64_t n;
    int BH;
    int dh;
    int* status;
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&p);
}

template <int D, int WS>
__global__ void __launch_bounds__(NTHREADS, 1)
k_apply_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_w1,
           const __grid_constant__ CUtensorMap tm_w3, const __grid_constant__ CUtensorMap tm_w2, const ApplyArgs a) {
    extern __shared__ __align__(16) unsigned char smraw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t bars[NBARS];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ int skip_cta;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = blockIdx.x, bh = blockIdx.y;
    const int R = a.dh / HB;
    const uint32_t base = smem_u32(sm);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };
    typedef ApplyLayout<D, WS> Lo;
    constexpr uint32_t OFF_Q = Lo::OFF_Q, OFF_W = Lo::OFF_W, OFF_U = Lo::OFF_U, W_STAGE = Lo::W_STAGE;

    if (tid == 0) {
        skip_cta = (*reinterpret_cast<volatile int*>(a.status) & ST_TIMEOUT) ? 1 : 0;
        abort_flag = 0;
        mbar_init(bar(B_Q), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(B_WF + s), 1);
            mbar_init(bar(B_WE + s), 1);
            mbar_init(bar(B_HF + s), 1);
            mbar_init(bar(B_HE + s), 8);
            mbar_init(bar(B_UF + s), 8);
            mbar_init(bar(B_UE + s), 1);
        }
        mbar_init(bar(B_O), 1);
        mbar_init(bar(B_DRAIN), 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (skip_cta) return;
    if (warp == 1) {
        __syncwarp();
        tmem_alloc(smem_u32(&tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    volatile int* abort_v = &abort_flag;
    auto give_up = [&]() {
        atomicOr(a.status, ST_TIMEOUT);
        *abort_v = 1;
    };

    if (warp == 0) {
        if (lane == 0) {
            const int tok = (int)(a.t0 + (int64_t)tile * TT);
            mbar_expect_tx(bar(B_Q), (D / 64) * BOX);
            for (int at = 0; at < D / 64; ++at) tma_load_3d(base + OFF_Q + at * BOX, &tm_q, bar(B_Q), at * 64, tok, bh);
            int issued = 0;
            for (int r = 0; r < R && !*abort_v; ++r) {
                const int s = r % WS;
                if (r >= WS && !mbar_wait(bar(B_WE + s), ((r / WS) - 1) & 1, WAIT_NS)) { give_up(); break; }
                const uint32_t st = base + OFF_W + s * W_STAGE;
                const int wrow = bh * a.dh + r * HB;
                mbar_expect_tx(bar(B_WF + s), W_STAGE);
                for (int at = 0; at < D / 64; ++at) {
                    tma_load_2d(st + at * BOX, &tm_w1, bar(B_WF + s), at * 64, wrow);
                    tma_load_2d(st + at * BOX + BOX / 2, &tm_w3, bar(B_WF + s), at * 64, wrow);
                }
                tma_load_2d(st + Lo::WC_BYTES, &tm_w2, bar(B_WF + s), r * HB, bh * D);
                issued = r + 1;
            }
            mbar_wait(bar(B_Q), 0, WAIT_NS);
            for (int r = (issued > WS ? issued - WS : 0); r < issued; ++r)
                mbar_wait(bar(B_WF + (r % WS)), (r / WS) & 1, WAIT_NS);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t i_h = idesc_bf16_f32(128, 128, 0, 0);
            const uint32_t i_o = idesc_bf16_f32(128, D, 0, 0);
            // descriptor bases; offsets (address / 16) are added as constants
            const uint64_t dQ = sdesc_sw128(base + OFF_Q, 16, 1024);
            const uint64_t dWc = sdesc_sw128(base + OFF_W, 16, 1024);
            const uint64_t dW2 = sdesc_sw128(base + OFF_W + Lo::WC_BYTES, 16, 1024);
            const uint64_t dU = sdesc_sw128(base + OFF_U, 16, 1024);
            bool ok = mbar_wait(bar(B_Q), 0, WAIT_NS);
            if (!ok) give_up();
            auto out_mma = [&](int r) -> bool {
                const int u = r & 1;
                if (!mbar_wait(bar(B_UF + u), (r >> 1) & 1, WAIT_NS)) return false;
                tc_fence_after();
                const uint64_t wo = (uint64_t)((r % WS) * W_STAGE) >> 4, uo = (uint64_t)(u * BOX) >> 4;
                const uint32_t first = r > 0 ? 1u : 0u;
#pragma unroll
                for (int j = 0; j < HB / 16; ++j)
                    mma_bf16(tmem + COL_O, dU + uo + j * 2, dW2 + wo + j * 2, i_o, j > 0 ? 1u : first);
                mma_commit(bar(B_WE + r % WS));
                mma_commit(bar(B_UE + u));
                return true;
            };
            for (int r = 0; r < R && ok && !*abort_v; ++r) {
                const int s = r % WS, hb = r & 1;
                if (!mbar_wait(bar(B_WF + s), (r / WS) & 1, WAIT_NS)) { give_up(); ok = false; break; }
                if (r >= 2 && !mbar_wait(bar(B_HE + hb), ((r >> 1) - 1) & 1, WAIT_NS)) { give_up(); ok = false; break; }
                tc_fence_after();
                const uint64_t wo = (uint64_t)(s * W_STAGE) >> 4;
                const uint32_t th = tmem + COL_H13 + hb * 128;
#pragma unroll
                for (int j = 0; j < D / 16; ++j) {
                    const uint64_t ko = (uint64_t)((j >> 2) * BOX + (j & 3) * 32) >> 4;
                    mma_bf16(th, dQ + ko, dWc + wo + ko, i_h, j > 0 ? 1u : 0u);
                }
                mma_commit(bar(B_HF + hb));
                // With one W stage the next block's weights load only after
                // this block's output GEMM; with two, that GEMM trails by one.
                const int ro = WS == 1 ? r : r - 1;
                if (ro >= 0 && !out_mma(ro)) { give_up(); ok = false; break; }
            }
            if (WS > 1 && ok && !*abort_v && R > 0 && !out_mma(R - 1)) give_up();
            mma_commit(bar(B_O));
            mma_commit(bar(B_DRAIN));
            mbar_wait(bar(B_DRAIN), 0, WAIT_NS);
        }
    } else {
        const int q = warp & 3;
        const int hf = (warp - 2) >> 2;
        const int row = 32 * q + lane;                       // query within the tile
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        bool ok = true;
        for (int r = 0; r < R; ++r) {
            const int s = r & 1;   // H and U buffer of this block
            if (*abort_v || !mbar_wait_warp(bar(B_HF + s), (r >> 1) & 1, WAIT_NS)) { give_up(); ok = false; break; }
            tc_fence_after();
            uint32_t h1[32], h3[32];
            tmem_ld32(lane_base + COL_H13 + s * 128 + hf * 32, h1);
            tmem_ld32(lane_base + COL_H13 + s * 128 + 64 + hf * 32, h3);
            tmem_wait_ld();
            tmem_pin(h1);
            tmem_pin(h3);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_HE + s));
            uint32_t pu[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                float uu[2];
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const float x1 = __uint_as_float(h1[j + t]);
                    uu[t] = __fdividef(x1, 1.0f + __expf(-x1)) * __uint_as_float(h3[j + t]);
                }
                pu[j / 2] = pack_bf16(uu[0], uu[1]);
            }
            if (r >= 2 && !mbar_wait_warp(bar(B_UE + s), ((r >> 1) - 1) & 1, WAIT_NS)) { give_up(); ok = false; break; }
            unsigned char* ub = sm + OFF_U + s * BOX;
#pragma unroll
            for (int c = 0; c < 4; ++c)
                *reinterpret_cast<uint4*>(ub + sw128_offset(row, hf * 32 + c * 8)) =
                    make_uint4(pu[4 * c], pu[4 * c + 1], pu[4 * c + 2], pu[4 * c + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_UF + s));
        }
        if (ok && !*abort_v && mbar_wait_warp(bar(B_O), 0, WAIT_NS)) {
            tc_fence_after();
            const int64_t tok = (int64_t)tile * TT + row;
            // this thread's half of the output row: D/2 columns, D/64 loads of 32
#pragma unroll
            for (int h = 0; h < D / 64; ++h) {
                uint32_t v[32], packed[16];
                tmem_ld32(lane_base + COL_O + hf * (D / 2) + h * 32, v);
                tmem_wait_ld();
                tmem_pin(v);
#pragma unroll
                for (int j = 0; j < 32; j += 2) packed[j / 2] = pack_bf16(__uint_as_float(v[j]), __uint_as_float(v[j + 1]));
                if (tok < a.n) {
                    uint4* dst = reinterpret_cast<uint4*>(a.o + ((int64_t)bh * a.n_total + a.t0 + tok) * D + hf * (D / 2) +
                                                          h * 32);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        dst[c] = make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
                }
            }
        } else if (ok) {
            give_up();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace

bool apply_tc_supported(const lact_state* st) {
    return st->cfg.io_dtype == LACT_BF16 && (st->cfg.d == 128 || st->cfg.d == 256) && st->cfg.dh % HB == 0 &&
           tmap_available();
}

template <int D, int WS>
static cudaError_t launch_apply_d(const lact_state* st, TokView q, void* o, cudaStream_t s) {
    const int dh = st->cfg.dh, BH = st->BH;
    CUtensorMap mq, m1, m3, m2;
    const uint64_t q_dims[3] = {(uint64_t)D, (uint64_t)q.n_total, (uint64_t)BH};
    const uint64_t q_str[2] = {(uint64_t)D * 2, (uint64_t)q.n_total * D * 2};
    const uint32_t q_box[3] = {64, TT, 1};
    const uint64_t w13_dims[2] = {(uint64_t)D, (uint64_t)BH * dh};
    const uint64_t w13_str[1] = {(uint64_t)D * 2};
    const uint32_t w13_box[2] = {64, HB};
    const uint64_t w2_dims[2] = {(uint64_t)dh, (uint64_t)BH * D};
    const uint64_t w2_str[1] = {(uint64_t)dh * 2};
    const uint32_t w2_box[2] = {64, D};
    if (!make_tmap_bf16(&mq, q.p, 3, q_dims, q_str, q_box) ||
        !make_tmap_bf16(&m1, st->Wsh[0], 2, w13_dims, w13_str, w13_box) ||
        !make_tmap_bf16(&m3, st->Wsh[2], 2, w13_dims, w13_str, w13_box) ||
        !make_tmap_bf16(&m2, st->Wsh[1], 2, w2_dims, w2_str, w2_box))
        return cudaErrorInvalidValue;
    ApplyArgs aa;
    aa.o = static_cast<bf16*>(o);
    aa.n_total = q.n_total;
    aa.t0 = q.t0;
    aa.n = q.n;
    aa.BH = BH;
    aa.dh = dh;
    aa.status = st->status;
    constexpr uint32_t smem = ApplyLayout<D, WS>::SMEM_BYTES;
    cudaError_t e = cudaFuncSetAttribute(k_apply_tc<D, WS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((q.n + TT - 1) / TT), BH);
    k_apply_tc<D, WS><<<grid, NTHREADS, smem, s>>>(mq, m1, m3, m2, aa);
    g_launches++;
    g_tc_launches++;
    return cudaGetLastError();
}

cudaError_t launch_apply_tc(const lact_state* st, TokView q, void* o, cudaStream_t s) {
    if (st->cfg.d == 128) return launch_apply_d<128, 2>(st, q, o, s);
    return launch_apply_d<256, 1>(st, q, o, s);
}

}  // namespace lact
