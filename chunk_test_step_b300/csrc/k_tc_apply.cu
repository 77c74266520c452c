// Readout of the SwiGLU fast-weight memory on the sm_103a tensor cores
// (tcgen05 + TMA + TMEM), bf16 io, head dim D = 128 or 256:
//     o_i = W2 (silu(W1 q_i) * (W3 q_i))
// (LaCT review page, "Fast weights are temporary context memory": queries
// read the adapted weights; "Local attention and nonlinear memory work
// together": the three-matrix SwiGLU memory).
//
// One CTA per (head, 128-query tile); the launcher uses this kernel at head
// dim 256 and k_apply2_tc (k_tc_apply2.cu: two query tiles per CTA sharing
// every weight block) at 128. The hidden units are visited in blocks r of 64:
//   [H1 | H3] (TMEM, double-buffered) = Q . [W1_r ; W3_r]^T   (A, B K-major)
//   U_r = silu(H1) * H3 -> bf16, swizzled K-major operand       (epilogue)
//   O (TMEM, D cols) += U_r . W2[:, r]^T                        (A, B K-major)
// so the MMA of block r+1 overlaps the epilogue of block r. The weights
// stream through two TMA rings: [W1_r ; W3_r] in 64-wide head-dim pieces
// (128 rows, 16 KB; 4 slots) and W2[:, r] (D rows x 64, 2 slots), so the
// next block's weights load while the current block computes. At the end O
// leaves TMEM as bf16.
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
constexpr int CSLOTS = 4;                           // [W1_r ; W3_r] piece ring
constexpr uint32_t BOX = TT * 128;                  // [128 rows][64 bf16], 16 KB

// Shared-memory layout for head dim D.
template <int D>
struct ApplyLayout {
    static constexpr int NQ = D / 64;                                     // head-dim pieces
    static constexpr uint32_t OFF_Q = 0;                                  // NQ k-atoms of the query tile
    static constexpr uint32_t OFF_C = NQ * BOX;                           // CSLOTS pieces of [W1_r ; W3_r]
    static constexpr uint32_t W2_BYTES = D * 128;                         // [D rows][64 hidden]
    static constexpr uint32_t OFF_W2 = OFF_C + CSLOTS * BOX;              // 2 slots
    static constexpr uint32_t OFF_U = OFF_W2 + 2 * W2_BYTES;              // 2 buffers of [128 tok][64 hid]
    static constexpr uint32_t SMEM_BYTES = OFF_U + 2 * BOX + 1024;
};

constexpr uint32_t COL_H13 = 0;     // buffer b at b * 128: H1 (64) | H3 (64)
constexpr uint32_t COL_O = 256;     // D columns
constexpr uint32_t TMEM_COLS = 512;
constexpr uint64_t WAIT_NS = 2000000000ull;

enum {
    B_Q = 0, B_CF = 1, B_CE = 1 + CSLOTS, B_2F = 1 + 2 * CSLOTS, B_2E = B_2F + 2, B_HF = B_2E + 2, B_HE = B_HF + 2,
    B_UF = B_HE + 2, B_UE = B_UF + 2, B_O = B_UE + 2, B_DRAIN, NBARS
};

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

__device__ __forceinline__ float tanh_approx(float x) {
    float r;
    asm("tanh.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
k_apply_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_w1,
           const __grid_constant__ CUtensorMap tm_w3, const __grid_constant__ CUtensorMap tm_w2, const ApplyArgs a) {
    pdl_wait();
    pdl_trigger();
    typedef ApplyLayout<D> Lo;
    constexpr int NQ = Lo::NQ;
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

    if (tid == 0) {
        skip_cta = (*reinterpret_cast<volatile int*>(a.status) & ST_TIMEOUT) ? 1 : 0;
        abort_flag = 0;
        mbar_init(bar(B_Q), 1);
        for (int s = 0; s < CSLOTS; ++s) {
            mbar_init(bar(B_CF + s), 1);
            mbar_init(bar(B_CE + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(B_2F + s), 1);
            mbar_init(bar(B_2E + s), 1);
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
            mbar_expect_tx(bar(B_Q), NQ * BOX);
            for (int qd = 0; qd < NQ; ++qd) tma_load_3d(base + Lo::OFF_Q + qd * BOX, &tm_q, bar(B_Q), qd * 64, tok, bh);
            int issued_c = 0, issued_2 = 0;
            bool ok = true;
            for (int r = 0; r < R && ok && !*abort_v; ++r) {
                const int wrow = bh * a.dh + r * HB;
                for (int qd = 0; qd < NQ; ++qd) {
                    const int i = r * NQ + qd, s = i % CSLOTS;
                    if (i >= CSLOTS && !mbar_wait(bar(B_CE + s), ((i / CSLOTS) - 1) & 1, WAIT_NS)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    const uint32_t st = base + Lo::OFF_C + s * BOX;
                    mbar_expect_tx(bar(B_CF + s), BOX);
                    tma_load_2d(st, &tm_w1, bar(B_CF + s), qd * 64, wrow);
                    tma_load_2d(st + BOX / 2, &tm_w3, bar(B_CF + s), qd * 64, wrow);
                    issued_c = i + 1;
                }
                if (!ok) break;
                const int s2 = r & 1;
                if (r >= 2 && !mbar_wait(bar(B_2E + s2), ((r >> 1) - 1) & 1, WAIT_NS)) { give_up(); break; }
                mbar_expect_tx(bar(B_2F + s2), Lo::W2_BYTES);
                tma_load_2d(base + Lo::OFF_W2 + s2 * Lo::W2_BYTES, &tm_w2, bar(B_2F + s2), r * HB, bh * D);
                issued_2 = r + 1;
            }
            // drain: the copies this thread started must land before the CTA exits
            mbar_wait(bar(B_Q), 0, WAIT_NS);
            for (int i = max(0, issued_c - CSLOTS); i < issued_c; ++i)
                mbar_wait(bar(B_CF + i % CSLOTS), (i / CSLOTS) & 1, WAIT_NS);
            for (int r = max(0, issued_2 - 2); r < issued_2; ++r) mbar_wait(bar(B_2F + (r & 1)), (r >> 1) & 1, WAIT_NS);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t i_h = idesc_bf16_f32(128, 128, 0, 0);
            const uint32_t i_o = idesc_bf16_f32(128, D, 0, 0);
            // descriptor bases; offsets (address / 16) are added as constants
            const uint64_t dQ = sdesc_sw128(base + Lo::OFF_Q, 16, 1024);
            const uint64_t dC = sdesc_sw128(base + Lo::OFF_C, 16, 1024);
            const uint64_t dW2 = sdesc_sw128(base + Lo::OFF_W2, 16, 1024);
            const uint64_t dU = sdesc_sw128(base + Lo::OFF_U, 16, 1024);
            bool ok = mbar_wait(bar(B_Q), 0, WAIT_NS);
            if (!ok) give_up();
            auto out_mma = [&](int r) -> bool {
                const int u = r & 1;
                if (!mbar_wait(bar(B_UF + u), (r >> 1) & 1, WAIT_NS)) return false;
                if (!mbar_wait(bar(B_2F + u), (r >> 1) & 1, WAIT_NS)) return false;
                tc_fence_after();
                const uint64_t wo = (uint64_t)(u * Lo::W2_BYTES) >> 4, uo = (uint64_t)(u * BOX) >> 4;
                const uint32_t first = r > 0 ? 1u : 0u;
#pragma unroll
                for (int j = 0; j < HB / 16; ++j)
                    mma_bf16(tmem + COL_O, dU + uo + j * 2, dW2 + wo + j * 2, i_o, j > 0 ? 1u : first);
                mma_commit(bar(B_2E + u));
                mma_commit(bar(B_UE + u));
                return true;
            };
            for (int r = 0; r < R && ok && !*abort_v; ++r) {
                const int hb = r & 1;
                if (r >= 2 && !mbar_wait(bar(B_HE + hb), ((r >> 1) - 1) & 1, WAIT_NS)) { give_up(); ok = false; break; }
                const uint32_t th = tmem + COL_H13 + hb * 128;
                for (int qd = 0; qd < NQ && ok; ++qd) {
                    const int i = r * NQ + qd, s = i % CSLOTS;
                    if (!mbar_wait(bar(B_CF + s), (i / CSLOTS) & 1, WAIT_NS)) { give_up(); ok = false; break; }
                    tc_fence_after();
                    const uint64_t co = (uint64_t)(s * BOX) >> 4, qo = (uint64_t)(qd * BOX) >> 4;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        mma_bf16(th, dQ + qo + j * 2, dC + co + j * 2, i_h, (qd > 0 || j > 0) ? 1u : 0u);
                    mma_commit(bar(B_CE + s));
                }
                if (!ok) break;
                mma_commit(bar(B_HF + hb));
                if (r >= 1 && !out_mma(r - 1)) { give_up(); ok = false; break; }
            }
            if (ok && !*abort_v && R > 0 && !out_mma(R - 1)) give_up();
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
            // u = silu(h1) h3, with sigmoid(x) = 0.5 tanh(x / 2) + 0.5
            uint32_t pu[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                float uu[2];
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const float x1 = __uint_as_float(h1[j + t]);
                    const float sg = fmaf(0.5f, tanh_approx(0.5f * x1), 0.5f);
                    uu[t] = x1 * sg * __uint_as_float(h3[j + t]);
                }
                pu[j / 2] = pack_bf16(uu[0], uu[1]);
            }
            if (r >= 2 && !mbar_wait_warp(bar(B_UE + s), ((r >> 1) - 1) & 1, WAIT_NS)) { give_up(); ok = false; break; }
            unsigned char* ub = sm + Lo::OFF_U + s * BOX;
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
                // 64 contiguous bytes of this thread's row; after a transpose
                // within each quad of lanes, four lanes store one row's 64 bytes
                // together (whole 32-byte sectors per warp store)
                uint4 ch[4];
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    ch[c] = make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
                quad_transpose(ch, lane);
                const int64_t quad_tok = tok - (lane & 3);
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4)
                    if (quad_tok + k4 < a.n)
                        *reinterpret_cast<uint4*>(a.o + ((int64_t)bh * a.n_total + a.t0 + quad_tok + k4) * D + hf * (D / 2) +
                                                  h * 32 + 8 * (lane & 3)) = ch[k4];
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

template <int D>
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
    constexpr uint32_t smem = ApplyLayout<D>::SMEM_BYTES;
    cudaError_t e = cudaFuncSetAttribute(k_apply_tc<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((q.n + TT - 1) / TT), BH);
    launch_pdl(k_apply_tc<D>, grid, NTHREADS, smem, s, mq, m1, m3, m2, aa);
    g_launches++;
    g_tc_launches++;
    return cudaGetLastError();
}

cudaError_t launch_apply_tc(const lact_state* st, TokView q, void* o, cudaStream_t s) {
    if (st->cfg.d == 128) return launch_apply2_tc(st, q, o, s);
    return launch_apply_d<256>(st, q, o, s);
}

}  // namespace lact
