// Readout of the SwiGLU fast-weight memory on the sm_103a tensor cores for
// head dim 128, two query tiles per CTA:
//     o_i = W2 (silu(W1 q_i) * (W3 q_i))
// (LaCT review page, "Fast weights are temporary context memory" and "Local
// attention and nonlinear memory work together").
//
// One CTA per (head, 256 queries = two 128-query subtiles). The hidden units
// are visited in blocks r of 64; each block's weights, streamed through TMA
// rings ([W1_r ; W3_r] in 64-wide head-dim pieces, 4 slots; W2[:, r], 2
// slots), serve both subtiles, so a head's weights cross from L2 once per 256
// queries instead of once per 128. Per block and subtile s:
//   [H1 | H3]_s (TMEM, 128 cols) = Q_s . [W1_r ; W3_r]^T       (A, B K-major)
//   U_s = silu(H1) * H3 -> bf16, swizzled K-major operand       (epilogue)
//   O_s (TMEM, 128 cols) += U_s . W2[:, r]^T                    (A, B K-major)
// TMEM holds H_0, H_1, O_0, O_1 (512 columns); H is single-buffered, so the
// next block's H GEMMs wait until the epilogue has read this block's H out of
// TMEM into registers (its first step, before the arithmetic). U is
// double-buffered in shared memory. The query tiles are requested before the
// TMEM allocation.
//
// Warp roles (320 threads): warp 0 TMA, warp 1 TMEM owner + MMA issuer,
// warps 2..9 epilogue (thread = query row of both subtiles, 32 of the 64
// hidden units). Every wait is bounded; a wait that gives up sets ST_TIMEOUT
// and the CTA unwinds.
#include "lact_internal.cuh"
#include "tc_ptx.cuh"

namespace lact {

namespace {

using namespace tc;

constexpr int D = 128;
constexpr int HB = 64;
constexpr int NQ = D / 64;                       // head-dim pieces of a W block
constexpr int NSUB = 2;                          // query subtiles per CTA
constexpr int NTHREADS = 320;
constexpr int CSLOTS = 4;
constexpr uint32_t BOX = 128 * 128;              // [128 rows][64 bf16], 16 KB
constexpr uint32_t OFF_Q = 0;                    // subtile s: NQ atoms at s * NQ * BOX
constexpr uint32_t OFF_C = NSUB * NQ * BOX;      // CSLOTS pieces of [W1_r ; W3_r]
constexpr uint32_t W2_BYTES = D * 128;           // [D rows][64 hidden]
constexpr uint32_t OFF_W2 = OFF_C + CSLOTS * BOX;
constexpr uint32_t OFF_U = OFF_W2 + 2 * W2_BYTES;  // buffer u, subtile s at (u * NSUB + s) * BOX
constexpr uint32_t SMEM_BYTES = OFF_U + 2 * NSUB * BOX + 1024;
constexpr uint32_t COL_H = 0;                    // subtile s at s * 128: H1 (64) | H3 (64)
constexpr uint32_t COL_O = 256;                  // subtile s at 256 + s * 128
constexpr uint64_t WAIT_NS = 2000000000ull;

enum {
    B_Q = 0, B_CF = 1, B_CE = 1 + CSLOTS, B_2F = 1 + 2 * CSLOTS, B_2E = B_2F + 2, B_HF = B_2E + 2, B_HE,
    B_UF, B_UE = B_UF + 2, B_O = B_UE + 2, B_DRAIN, NBARS
};

struct Apply2Args {
    bf16* o;             // [BH, n_total, D], same layout as q
    int64_t n_total;
    int64_t t0;
    int64_t n;
    int dh;
    int* status;
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&p);
}

// Packed fp32 pairs (two lanes of work per instruction on sm_100 and later).
typedef unsigned long long f2;
__device__ __forceinline__ f2 f2_make(float lo, float hi) {
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_split(f2 v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f2 f2_mul(f2 a, f2 b) {
    f2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f2 f2_fma(f2 a, f2 b, f2 c) {
    f2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint32_t pack_f2(f2 v) {
    float lo, hi;
    f2_split(v, lo, hi);
    return pack_bf16(lo, hi);
}

__device__ __forceinline__ float tanh_approx(float x) {
    float r;
    asm("tanh.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__global__ void __launch_bounds__(NTHREADS, 1)
k_apply2_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_w1,
            const __grid_constant__ CUtensorMap tm_w3, const __grid_constant__ CUtensorMap tm_w2, const Apply2Args a) {
    pdl_wait();
    pdl_trigger();
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
            mbar_init(bar(B_UF + s), 8);
            mbar_init(bar(B_UE + s), 1);
        }
        mbar_init(bar(B_HF), 1);
        mbar_init(bar(B_HE), 8);
        mbar_init(bar(B_O), 1);
        mbar_init(bar(B_DRAIN), 1);
        fence_mbar_init();
        // the query tiles need no TMEM: their copies start before the allocation
        if (!skip_cta) {
            mbar_expect_tx(bar(B_Q), NSUB * NQ * BOX);
            for (int s = 0; s < NSUB; ++s) {
                const int tok = (int)(a.t0 + (int64_t)(tile * NSUB + s) * 128);
                for (int qd = 0; qd < NQ; ++qd)
                    tma_load_3d(base + OFF_Q + (s * NQ + qd) * BOX, &tm_q, bar(B_Q), qd * 64, tok, bh);
            }
        }
    }
    __syncthreads();
    if (skip_cta) return;
    if (warp == 1) {
        __syncwarp();
        tmem_alloc(smem_u32(&tmem_slot), 512);
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
            int issued_c = 0, issued_2 = 0;
            bool ok = true;
            for (int r = 0; r < R && ok && !*abort_v; ++r) {
                const int wrow = bh * a.dh + r * HB;
                for (int qd = 0; qd < NQ; ++qd) {
                    const int i = r * NQ + qd, sl = i % CSLOTS;
                    if (i >= CSLOTS && !mbar_wait(bar(B_CE + sl), ((i / CSLOTS) - 1) & 1, WAIT_NS)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    const uint32_t st = base + OFF_C + sl * BOX;
                    mbar_expect_tx(bar(B_CF + sl), BOX);
                    tma_load_2d(st, &tm_w1, bar(B_CF + sl), qd * 64, wrow);
                    tma_load_2d(st + BOX / 2, &tm_w3, bar(B_CF + sl), qd * 64, wrow);
                    issued_c = i + 1;
                }
                if (!ok) break;
                const int s2 = r & 1;
                if (r >= 2 && !mbar_wait(bar(B_2E + s2), ((r >> 1) - 1) & 1, WAIT_NS)) { give_up(); break; }
                mbar_expect_tx(bar(B_2F + s2), W2_BYTES);
                tma_load_2d(base + OFF_W2 + s2 * W2_BYTES, &tm_w2, bar(B_2F + s2), r * HB, bh * D);
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
            const uint64_t dQ = sdesc_sw128(base + OFF_Q, 16, 1024);
            const uint64_t dC = sdesc_sw128(base + OFF_C, 16, 1024);
            const uint64_t dW2 = sdesc_sw128(base + OFF_W2, 16, 1024);
            const uint64_t dU = sdesc_sw128(base + OFF_U, 16, 1024);
            bool ok = mbar_wait(bar(B_Q), 0, WAIT_NS);
            if (!ok) give_up();
            auto out_mma = [&](int r) -> bool {
                const int u = r & 1;
                if (!mbar_wait(bar(B_UF + u), (r >> 1) & 1, WAIT_NS)) return false;
                if (!mbar_wait(bar(B_2F + u), (r >> 1) & 1, WAIT_NS)) return false;
                tc_fence_after();
                const uint64_t wo = (uint64_t)(u * W2_BYTES) >> 4;
#pragma unroll
                for (int s = 0; s < NSUB; ++s) {
                    const uint64_t uo = (uint64_t)((u * NSUB + s) * BOX) >> 4;
#pragma unroll
                    for (int j = 0; j < HB / 16; ++j)
                        mma_bf16(tmem + COL_O + s * 128, dU + uo + j * 2, dW2 + wo + j * 2, i_o,
                                 (r > 0 || j > 0) ? 1u : 0u);
                }
                mma_commit(bar(B_2E + u));
                mma_commit(bar(B_UE + u));
                return true;
            };
            for (int r = 0; r < R && ok && !*abort_v; ++r) {
                // H is single-buffered: the epilogue has read block r-1 out of TMEM
                if (r >= 1 && !mbar_wait(bar(B_HE), (r - 1) & 1, WAIT_NS)) { give_up(); ok = false; break; }
                for (int qd = 0; qd < NQ && ok; ++qd) {
                    const int i = r * NQ + qd, sl = i % CSLOTS;
                    if (!mbar_wait(bar(B_CF + sl), (i / CSLOTS) & 1, WAIT_NS)) { give_up(); ok = false; break; }
                    tc_fence_after();
                    const uint64_t co = (uint64_t)(sl * BOX) >> 4;
#pragma unroll
                    for (int s = 0; s < NSUB; ++s) {
                        const uint64_t qo = (uint64_t)((s * NQ + qd) * BOX) >> 4;
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            mma_bf16(tmem + COL_H + s * 128, dQ + qo + j * 2, dC + co + j * 2, i_h,
                                     (qd > 0 || j > 0) ? 1u : 0u);
                    }
                    mma_commit(bar(B_CE + sl));
                }
                if (!ok) break;
                mma_commit(bar(B_HF));
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
        const int row = 32 * q + lane;                       // query within each subtile
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        bool ok = true;
        for (int r = 0; r < R; ++r) {
            const int u = r & 1;
            if (*abort_v || !mbar_wait_warp(bar(B_HF), r & 1, WAIT_NS)) { give_up(); ok = false; break; }
            tc_fence_after();
            // H leaves TMEM before any arithmetic, so that the next block's H
            // GEMMs overwrite it while this block's u is computed
            uint32_t hv[NSUB][2][32];
#pragma unroll
            for (int s = 0; s < NSUB; ++s) {
                tmem_ld32(lane_base + COL_H + s * 128 + hf * 32, hv[s][0]);
                tmem_ld32(lane_base + COL_H + s * 128 + 64 + hf * 32, hv[s][1]);
            }
            tmem_wait_ld();
#pragma unroll
            for (int s = 0; s < NSUB; ++s) {
                tmem_pin(hv[s][0]);
                tmem_pin(hv[s][1]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_HE));
            // u = silu(h1) h3 with sigmoid(x) = 0.5 tanh(x / 2) + 0.5, two
            // hidden units per packed fp32 instruction
            uint32_t pu[NSUB][16];
            const f2 half2 = f2_make(0.5f, 0.5f);
#pragma unroll
            for (int s = 0; s < NSUB; ++s) {
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    const f2 x1 = f2_make(__uint_as_float(hv[s][0][j]), __uint_as_float(hv[s][0][j + 1]));
                    const f2 x3 = f2_make(__uint_as_float(hv[s][1][j]), __uint_as_float(hv[s][1][j + 1]));
                    float hx0, hx1;
                    f2_split(f2_mul(x1, half2), hx0, hx1);
                    const f2 sg = f2_fma(f2_make(tanh_approx(hx0), tanh_approx(hx1)), half2, half2);
                    pu[s][j / 2] = pack_f2(f2_mul(f2_mul(x1, sg), x3));
                }
            }
            if (r >= 2 && !mbar_wait_warp(bar(B_UE + u), ((r >> 1) - 1) & 1, WAIT_NS)) { give_up(); ok = false; break; }
#pragma unroll
            for (int s = 0; s < NSUB; ++s) {
                unsigned char* ub = sm + OFF_U + (u * NSUB + s) * BOX;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    *reinterpret_cast<uint4*>(ub + sw128_offset(row, hf * 32 + c * 8)) =
                        make_uint4(pu[s][4 * c], pu[s][4 * c + 1], pu[s][4 * c + 2], pu[s][4 * c + 3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_UF + u));
        }
        if (ok && !*abort_v && mbar_wait_warp(bar(B_O), 0, WAIT_NS)) {
            tc_fence_after();
#pragma unroll
            for (int s = 0; s < NSUB; ++s) {
                const int64_t tok = (int64_t)(tile * NSUB + s) * 128 + row;
#pragma unroll
                for (int h = 0; h < D / 64; ++h) {
                    uint32_t v[32], packed[16];
                    tmem_ld32(lane_base + COL_O + s * 128 + hf * (D / 2) + h * 32, v);
                    tmem_wait_ld();
                    tmem_pin(v);
#pragma unroll
                    for (int j = 0; j < 32; j += 2)
                        packed[j / 2] = pack_bf16(__uint_as_float(v[j]), __uint_as_float(v[j + 1]));
                    // 64 contiguous bytes of this thread's row; after a transpose
                    // within each quad of lanes, four lanes store one row's 64
                    // bytes together (whole 32-byte sectors per warp store)
                    uint4 ch[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        ch[c] = make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
                    quad_transpose(ch, lane);
                    const int64_t quad_tok = tok - (lane & 3);
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4)
                        if (quad_tok + k4 < a.n)
                            *reinterpret_cast<uint4*>(a.o + ((int64_t)bh * a.n_total + a.t0 + quad_tok + k4) * D +
                                                      hf * (D / 2) + h * 32 + 8 * (lane & 3)) = ch[k4];
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
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

cudaError_t launch_apply2_tc(const lact_state* st, TokView q, void* o, cudaStream_t s) {
    const int dh = st->cfg.dh, BH = st->BH;
    CUtensorMap mq, m1, m3, m2;
    const uint64_t q_dims[3] = {(uint64_t)D, (uint64_t)q.n_total, (uint64_t)BH};
    const uint64_t q_str[2] = {(uint64_t)D * 2, (uint64_t)q.n_total * D * 2};
    const uint32_t q_box[3] = {64, 128, 1};
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
    Apply2Args aa;
    aa.o = static_cast<bf16*>(o);
    aa.n_total = q.n_total;
    aa.t0 = q.t0;
    aa.n = q.n;
    aa.dh = dh;
    aa.status = st->status;
    cudaError_t e = cudaFuncSetAttribute(k_apply2_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((q.n + NSUB * 128 - 1) / (NSUB * 128)), BH);
    launch_pdl(k_apply2_tc, grid, NTHREADS, SMEM_BYTES, s, mq, m1, m3, m2, aa);
    g_launches++;
    g_tc_launches++;
    return cudaGetLastError();
}

}  // namespace lact
