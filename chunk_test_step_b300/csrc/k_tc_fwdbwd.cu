// Per-token part of the chunk gradient on the sm_103a tensor cores (tcgen05 +
// TMA + TMEM), for the two-kernel form used at head dim 256.
//
// For the loss L = -sum_i eta_i <f_W(k_i), v_i> of the SwiGLU fast-weight
// memory f_W(x) = W2 (silu(W1 x) * (W3 x)) (LaCT review page, "Local
// attention and nonlinear memory work together"), with K, V the chunk's keys
// and values and r a block of 64 hidden units:
//   H1 = K W1_r^T, H3 = K W3_r^T, A = V W2[:, r]            (tokens x 64)
//   u'  = -eta silu(H1) H3
//   dh1 = -eta A H3 silu'(H1),  dh3 = -eta A silu(H1)
// written as bf16 rows [token][hidden] for k_wgrad_tc, which forms
// dW1 = dh1^T K, dW3 = dh3^T K, dW2 = V^T u'. At head dim 256 one 128-token
// tile of K and V is 128 KB, too large to keep resident through the gradient
// GEMMs as the fused kernel does at head dim 128; the slice's per-token
// quantities stay in L2 between the two kernels instead.
//
// One CTA per (head, hidden block, token range), persistent over its 128-token
// tiles. The block's weights stay in shared memory (96 KB): [W1_r ; W3_r]
// (128 rows x 256, K-major) and W2[:, r] (256 x 64, read MN-major). K and V
// stream through a 4-slot ring of 64-wide head-dim quarters (32 KB a slot).
// Per tile, per quarter s:
//   [H1 | H3] (TMEM, 128 cols) += K_s . [W1_r ; W3_r]_s^T     (A, B K-major)
//   A         (TMEM,  64 cols) += V_s . W2[s, r]               (A K-major, B MN-major)
// into one of two TMEM buffers, so the epilogue of a tile overlaps the GEMMs
// of the next. Warp roles (320 threads): warp 0 TMA, warp 1 TMEM + MMA issue,
// warps 2..9 the epilogue (thread = token, 32 of the 64 hidden units). Every
// wait is bounded; a wait that gives up sets ST_TIMEOUT and the CTA unwinds.
#include "lact_internal.cuh"
#include "tc_ptx.cuh"

namespace lact {

namespace {

using namespace tc;

constexpr int D = 256;         // head dim served by this kernel
constexpr int HB = 64;         // hidden units per CTA
constexpr int TT = 128;        // tokens per tile
constexpr int DS = 64;         // head-dim elements per ring slot
constexpr int NQ = D / DS;     // quarters per tile
constexpr int SLOTS = 4;
constexpr int NTHREADS = 320;
constexpr uint32_t BOX = TT * 128;                        // [128 rows][64 bf16] = 16 KB
constexpr uint32_t OFF_WC = 0;                            // NQ atoms of [W1_r (64 rows) ; W3_r (64 rows)]
constexpr uint32_t W2_BOX = DS * 128;                     // [64 d rows][64 hidden] = 8 KB
constexpr uint32_t OFF_W2 = NQ * BOX;                     // NQ boxes of W2[s, r]
constexpr uint32_t OFF_RING = OFF_W2 + NQ * W2_BOX;       // slot: K block, V block
constexpr uint32_t SLOT_BYTES = 2 * BOX;
constexpr uint32_t SMEM_BYTES = OFF_RING + SLOTS * SLOT_BYTES + 1024;
constexpr uint32_t COL_H13 = 0, COL_A = 128, BUF_COLS = 256;   // buffer b at b * 256
constexpr uint64_t WAIT_NS = 2000000000ull;

enum { B_W = 0, B_F = 1, B_E = 1 + SLOTS, B_HF = 1 + 2 * SLOTS, B_HE = B_HF + 2, B_DRAIN = B_HE + 2, NBARS };

struct FbArgs {
    const float* eta;      // [BH, n_total]
    int64_t n_total;
    int64_t t0;            // first token of the slice
    int64_t n;             // tokens in the slice
    bf16* out;             // [3][BH][slice_cap][dh]: dh1, dh3, u'
    int64_t slice_cap;
    int tiles_per_cta;
    int ntiles;
    int BH, dh;
    int* status;
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&p);
}

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
__device__ __forceinline__ float tanh_approx(float x) {
    float r;
    asm("tanh.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ uint32_t pack_f2(f2 v) {
    float lo, hi;
    f2_split(v, lo, hi);
    return pack_bf16(lo, hi);
}

__global__ void __launch_bounds__(NTHREADS, 1)
k_fwdbwd_tc(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
            const __grid_constant__ CUtensorMap tm_w1, const __grid_constant__ CUtensorMap tm_w3,
            const __grid_constant__ CUtensorMap tm_w2, const FbArgs a) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(16) unsigned char smraw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t bars[NBARS];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ int skip_cta;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = blockIdx.x, split = blockIdx.y, bh = blockIdx.z;
    const int tile_begin = split * a.tiles_per_cta;
    const int count = max(0, min(a.ntiles, tile_begin + a.tiles_per_cta) - tile_begin);
    const uint32_t base = smem_u32(sm);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };

    if (tid == 0) {
        skip_cta = (*reinterpret_cast<volatile int*>(a.status) & ST_TIMEOUT) ? 1 : 0;
        abort_flag = 0;
        mbar_init(bar(B_W), 1);
        for (int s = 0; s < SLOTS; ++s) {
            mbar_init(bar(B_F + s), 1);
            mbar_init(bar(B_E + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(B_HF + b), 1);
            mbar_init(bar(B_HE + b), 8);
        }
        mbar_init(bar(B_DRAIN), 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (skip_cta || count == 0) return;
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
    const int nsteps = count * NQ;     // ring steps: (tile, quarter)

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            // the block's weights, once
            const int wrow = bh * a.dh + r * HB;
            mbar_expect_tx(bar(B_W), NQ * BOX + NQ * W2_BOX);
            for (int qd = 0; qd < NQ; ++qd) {
                tma_load_2d(base + OFF_WC + qd * BOX, &tm_w1, bar(B_W), qd * DS, wrow);
                tma_load_2d(base + OFF_WC + qd * BOX + BOX / 2, &tm_w3, bar(B_W), qd * DS, wrow);
                tma_load_2d(base + OFF_W2 + qd * W2_BOX, &tm_w2, bar(B_W), r * HB, bh * D + qd * DS);
            }
            int issued = 0;
            for (int i = 0; i < nsteps && !*abort_v; ++i) {
                const int s = i % SLOTS, tile = i / NQ, qd = i % NQ;
                if (i >= SLOTS && !mbar_wait(bar(B_E + s), ((i / SLOTS) - 1) & 1, WAIT_NS)) { give_up(); break; }
                const uint32_t st = base + OFF_RING + s * SLOT_BYTES;
                const int tok = (int)(a.t0 + (int64_t)(tile_begin + tile) * TT);
                mbar_expect_tx(bar(B_F + s), SLOT_BYTES);
                tma_load_3d(st, &tm_k, bar(B_F + s), qd * DS, tok, bh);
                tma_load_3d(st + BOX, &tm_v, bar(B_F + s), qd * DS, tok, bh);
                issued = i + 1;
            }
            mbar_wait(bar(B_W), 0, WAIT_NS);
            for (int i = max(0, issued - SLOTS); i < issued; ++i)
                mbar_wait(bar(B_F + i % SLOTS), (i / SLOTS) & 1, WAIT_NS);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t i_13 = idesc_bf16_f32(128, 128, 0, 0);
            const uint32_t i_a = idesc_bf16_f32(128, HB, 0, 1);
            const uint64_t dK = sdesc_sw128(base + OFF_RING, 16, 1024);
            const uint64_t dV = sdesc_sw128(base + OFF_RING + BOX, 16, 1024);
            const uint64_t dWc = sdesc_sw128(base + OFF_WC, 16, 1024);
            const uint64_t dW2 = sdesc_sw128(base + OFF_W2, W2_BOX, 1024);   // MN-major
            bool ok = mbar_wait(bar(B_W), 0, WAIT_NS);
            if (!ok) give_up();
            for (int i = 0; i < nsteps && ok && !*abort_v; ++i) {
                const int s = i % SLOTS, tile = i / NQ, qd = i % NQ, b = tile & 1;
                if (qd == 0 && tile >= 2 && !mbar_wait(bar(B_HE + b), ((tile >> 1) - 1) & 1, WAIT_NS)) {
                    give_up();
                    ok = false;
                    break;
                }
                if (!mbar_wait(bar(B_F + s), (i / SLOTS) & 1, WAIT_NS)) { give_up(); ok = false; break; }
                tc_fence_after();
                const uint64_t so = (uint64_t)(s * SLOT_BYTES) >> 4;
                const uint64_t wq = (uint64_t)(qd * BOX) >> 4, w2q = (uint64_t)(qd * W2_BOX) >> 4;
                const uint32_t t13 = tmem + b * BUF_COLS + COL_H13, ta = tmem + b * BUF_COLS + COL_A;
#pragma unroll
                for (int j = 0; j < DS / 16; ++j) {
                    const uint32_t acc = (qd > 0 || j > 0) ? 1u : 0u;
                    mma_bf16(t13, dK + so + j * 2, dWc + wq + j * 2, i_13, acc);
                    mma_bf16(ta, dV + so + j * 2, dW2 + w2q + j * 128, i_a, acc);
                }
                mma_commit(bar(B_E + s));
                if (qd == NQ - 1) mma_commit(bar(B_HF + b));
            }
            mma_commit(bar(B_DRAIN));
            mbar_wait(bar(B_DRAIN), 0, WAIT_NS);
        }
    } else {
        // ------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int hf = (warp - 2) >> 2;             // hidden units [32 hf, 32 hf + 32) of the block
        const int row = 32 * q + lane;              // token within the tile
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        const size_t one = (size_t)a.BH * a.slice_cap * a.dh;
        const f2 half2 = f2_make(0.5f, 0.5f), one2 = f2_make(1.0f, 1.0f), mone2 = f2_make(-1.0f, -1.0f);
        const float* eta_h = a.eta + (int64_t)bh * a.n_total + a.t0;
        auto eta_of = [&](int t) -> float {
            const int64_t tok = (int64_t)(tile_begin + t) * TT + row;
            return (t < count && tok < a.n) ? eta_h[tok] : 0.0f;
        };
        float e_next = eta_of(0);
        for (int t = 0; t < count; ++t) {
            const int b = t & 1;
            const int64_t tok = (int64_t)(tile_begin + t) * TT + row;   // within the slice
            const float e = e_next;
            e_next = eta_of(t + 1);
            if (*abort_v || !mbar_wait_warp(bar(B_HF + b), (t >> 1) & 1, WAIT_NS)) { give_up(); break; }
            tc_fence_after();
            uint32_t h1[32], h3[32], av[32];
            tmem_ld32(lane_base + b * BUF_COLS + COL_H13 + hf * 32, h1);
            tmem_ld32(lane_base + b * BUF_COLS + COL_H13 + HB + hf * 32, h3);
            tmem_ld32(lane_base + b * BUF_COLS + COL_A + hf * 32, av);
            tmem_wait_ld();
            tmem_pin(h1);
            tmem_pin(h3);
            tmem_pin(av);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_HE + b));
            // s = sigmoid(h1) = 0.5 tanh(h1 / 2) + 0.5, silu = h1 s;
            // u' = -eta silu h3, du = -eta a, dh3 = du silu,
            // dh1 = du h3 (s + silu (1 - s))
            const f2 ne2 = f2_make(-e, -e);
            uint32_t p1[16], p3[16], pu[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                const f2 x1 = f2_make(__uint_as_float(h1[j]), __uint_as_float(h1[j + 1]));
                const f2 x3 = f2_make(__uint_as_float(h3[j]), __uint_as_float(h3[j + 1]));
                const f2 av2 = f2_make(__uint_as_float(av[j]), __uint_as_float(av[j + 1]));
                float hx0, hx1;
                f2_split(f2_mul(x1, half2), hx0, hx1);
                const f2 th = f2_make(tanh_approx(hx0), tanh_approx(hx1));
                const f2 sg = f2_fma(th, half2, half2);
                const f2 si = f2_mul(x1, sg);
                const f2 x3n = f2_mul(x3, ne2);
                const f2 du = f2_mul(av2, ne2);
                const f2 oms = f2_fma(sg, mone2, one2);
                const f2 g = f2_fma(si, oms, sg);
                pu[j / 2] = pack_f2(f2_mul(si, x3n));
                p3[j / 2] = pack_f2(f2_mul(du, si));
                p1[j / 2] = pack_f2(f2_mul(f2_mul(du, x3), g));
            }
            // Each thread holds 64 contiguous bytes of its token's row of each
            // output. After a transpose within each quad of lanes, four lanes
            // store one row's 64 bytes together: a warp store covers 8 rows in
            // whole 32-byte sectors instead of 16 bytes of each of 32 rows.
            uint4 c1[4], c3[4], cu[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                c1[c] = make_uint4(p1[4 * c], p1[4 * c + 1], p1[4 * c + 2], p1[4 * c + 3]);
                c3[c] = make_uint4(p3[4 * c], p3[4 * c + 1], p3[4 * c + 2], p3[4 * c + 3]);
                cu[c] = make_uint4(pu[4 * c], pu[4 * c + 1], pu[4 * c + 2], pu[4 * c + 3]);
            }
            quad_transpose(c1, lane);
            quad_transpose(c3, lane);
            quad_transpose(cu, lane);
            const int64_t quad_tok = tok - (lane & 3);      // token of the quad's row 0
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
                if (quad_tok + k4 < a.n) {
                    bf16* o1 = a.out + ((size_t)bh * a.slice_cap + quad_tok + k4) * a.dh + r * HB + hf * 32 +
                               8 * (lane & 3);
                    *reinterpret_cast<uint4*>(o1) = c1[k4];
                    *reinterpret_cast<uint4*>(o1 + one) = c3[k4];
                    *reinterpret_cast<uint4*>(o1 + 2 * one) = cu[k4];
                }
            }
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

bool fwdbwd_tc_supported(const lact_state* st) {
    return st->cfg.io_dtype == LACT_BF16 && st->cfg.d == D && st->cfg.dh % HB == 0 && tmap_available();
}

// Tokens [k.t0, k.t0 + k.n) (k.n <= slice_cap): dh1, dh3, u' into `inter`
// ([3][BH][slice_cap][dh] bf16).
cudaError_t launch_fwdbwd_tc(const lact_state* st, TokView k, TokView v, const float* eta, bf16* inter,
                             int64_t slice_cap, cudaStream_t s) {
    const int dh = st->cfg.dh, BH = st->BH;
    CUtensorMap mk, mv, m1, m3, m2;
    const uint64_t k_dims[3] = {(uint64_t)D, (uint64_t)k.n_total, (uint64_t)BH};
    const uint64_t k_str[2] = {(uint64_t)D * 2, (uint64_t)k.n_total * D * 2};
    const uint64_t v_dims[3] = {(uint64_t)D, (uint64_t)v.n_total, (uint64_t)BH};
    const uint64_t v_str[2] = {(uint64_t)D * 2, (uint64_t)v.n_total * D * 2};
    const uint32_t kv_box[3] = {DS, TT, 1};
    const uint64_t w13_dims[2] = {(uint64_t)D, (uint64_t)BH * dh};
    const uint64_t w13_str[1] = {(uint64_t)D * 2};
    const uint32_t w13_box[2] = {DS, HB};
    const uint64_t w2_dims[2] = {(uint64_t)dh, (uint64_t)BH * D};
    const uint64_t w2_str[1] = {(uint64_t)dh * 2};
    const uint32_t w2_box[2] = {64, DS};
    if (!make_tmap_bf16(&mk, k.p, 3, k_dims, k_str, kv_box) || !make_tmap_bf16(&mv, v.p, 3, v_dims, v_str, kv_box) ||
        !make_tmap_bf16(&m1, st->Wsh[0], 2, w13_dims, w13_str, w13_box) ||
        !make_tmap_bf16(&m3, st->Wsh[2], 2, w13_dims, w13_str, w13_box) ||
        !make_tmap_bf16(&m2, st->Wsh[1], 2, w2_dims, w2_str, w2_box))
        return cudaErrorInvalidValue;
    const int ntiles = (int)((k.n + TT - 1) / TT);
    const int units = BH * (dh / HB);
    // token splits: as many as fit in one wave (at least 2 tiles each, so
    // that a CTA's epilogue overlaps its next tile's GEMMs)
    int splits = st->num_sms / units;
    if (splits > (ntiles + 1) / 2) splits = (ntiles + 1) / 2;
    if (splits < 1) splits = 1;
    const int tpc = (ntiles + splits - 1) / splits;
    splits = (ntiles + tpc - 1) / tpc;
    FbArgs fa;
    fa.eta = eta;
    fa.n_total = k.n_total;
    fa.t0 = k.t0;
    fa.n = k.n;
    fa.out = inter;
    fa.slice_cap = slice_cap;
    fa.tiles_per_cta = tpc;
    fa.ntiles = ntiles;
    fa.BH = BH;
    fa.dh = dh;
    fa.status = st->status;
    cudaError_t e = cudaFuncSetAttribute(k_fwdbwd_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(dh / HB), (unsigned)splits, (unsigned)BH);
    launch_pdl(k_fwdbwd_tc, grid, NTHREADS, SMEM_BYTES, s, mk, mv, m1, m3, m2, fa);
    g_launches++;
    g_tc_launches++;
    return cudaGetLastError();
}

}  // namespace lact
