// Fused chunk-gradient kernel on the sm_103a tensor cores (tcgen05 + TMA +
// TMEM), bf16 io, head dim 128.
//
// For the loss L = -sum_i eta_i <f_W(k_i), v_i> of the SwiGLU fast-weight
// memory f_W(x) = W2 (silu(W1 x) * (W3 x)) (LaCT review page, "Local
// attention and nonlinear memory work together"), the chunk gradient
// decomposes over blocks r of 64 hidden units: with K, V the chunk's keys and
// values ([tokens, 128]) and eta the per-token rates,
//   H1 = K W1_r^T, H3 = K W3_r^T, A = V W2[:, r]            (forward, tokens x 64)
//   u' = -eta silu(H1) H3, du = -eta A,
//   dh1 = du H3 silu'(H1), dh3 = du silu(H1)                (registers)
//   dW1_r^T += K^T dh1, dW3_r^T += K^T dh3, dW2[:, r] += V^T u'   (weight gradients)
// so one CTA owns (hidden block r, token range, head) and never exchanges
// intermediates with another CTA. Per 128-token tile the CTA runs
// 4 GEMMs of 128x(64|128)x128 on the tensor cores:
//   fwd : [H1 | H3] (TMEM, 128 cols) = K . [W1_r ; W3_r]^T    (A K-major, B K-major)
//         A        (TMEM,  64 cols) = V . W2[:, r]            (A K-major, B MN-major)
//   grad: [dW1_r^T | dW3_r^T] (TMEM, 128 cols) += K^T . [dh1 | dh3]   (A, B MN-major)
//         dW2[:, r]          (TMEM,  64 cols) += V^T . u'             (A, B MN-major)
// The same TMA-loaded K and V tiles serve as K-major A operands in the
// forward GEMMs and as MN-major A operands in the gradient GEMMs.
//
// Warp roles (320 threads): warp 0 issues TMA loads, warp 1 owns TMEM and
// issues the MMAs (one thread), warps 2..9 are the epilogue (thread = token,
// half of the 64 hidden units each), which pulls the forward accumulators
// out of TMEM, forms dh1, dh3, u' in fp32 and writes them as bf16 into the
// swizzled operand buffer of the gradient GEMMs. Splits over tokens write
// fp32 partial sums that a separate kernel adds in a fixed order.
//
// Every mbarrier wait is bounded; a wait that gives up sets ST_TIMEOUT in the
// status word, the CTA unwinds (draining its own TMA copies and MMAs) and
// frees its TMEM.
#include "lact_internal.cuh"
#include "tc_ptx.cuh"


namespace lact {

namespace {

using namespace tc;

constexpr int D = 128;         // head dim served by this kernel
constexpr int HB = 64;         // hidden units per CTA
constexpr int TT = 128;        // tokens per tile
constexpr int STAGES = 2;      // K/V pipeline depth
constexpr int PF = 6;          // tiles of K/V prefetched into L2 ahead of their load
constexpr int NTHREADS = 320;

constexpr uint32_t BOX = TT * 128;                    // one [128 rows][64 bf16] swizzled box: 16 KB
constexpr uint32_t OFF_WCAT = 0;                      // 2 k-atoms x [W1_r rows 0-63 ; W3_r rows 64-127]
constexpr uint32_t OFF_W2 = 2 * BOX;                  // W2[:, r]: [128 d rows][64 hid]
constexpr uint32_t OFF_KV = 3 * BOX;                  // stage s: K box0, K box1, V box0, V box1
constexpr uint32_t KV_STAGE = 4 * BOX;
constexpr uint32_t OFF_B = OFF_KV + STAGES * KV_STAGE;  // dh1 | dh3 | u' (each [128 tok][64 hid])
constexpr uint32_t SMEM_TILES = OFF_B + 3 * BOX;        // 229376
constexpr uint32_t SMEM_BYTES = SMEM_TILES + 1024;      // + alignment slack

// TMEM columns
constexpr uint32_t COL_H13 = 0;     // H1 0-63, H3 64-127
constexpr uint32_t COL_A = 128;     // V W2_r
constexpr uint32_t COL_DW13 = 256;  // dW1_r^T 256-319, dW3_r^T 320-383 (lanes = d)
constexpr uint32_t COL_DW2 = 384;   // dW2[:, r] (lanes = d)
constexpr uint32_t TMEM_COLS = 512;

constexpr uint64_t WAIT_NS = 2000000000ull;   // 2 s per wait

// Barriers. K and V halves of a stage are filled and released separately: K
// is free again once the dW1/dW3 GEMMs of its tile are done, V once the dW2
// GEMMs are. The gradient operand buffer has a dh1|dh3 part and a u' part,
// likewise written and released separately.
enum {
    B_W = 0,
    B_KF = 1, B_VF = 1 + STAGES, B_KE = 1 + 2 * STAGES, B_VE = 1 + 3 * STAGES,
    B_FWDF = 1 + 4 * STAGES, B_FWDE, B_DHF, B_UF, B_DHE, B_UE, B_ACC, B_DRAIN, NBARS
};

struct GradArgs {
    const float* eta;      // [BH, n_total]
    int64_t n_total;       // tokens per head in k, v, eta
    int64_t t0;            // first token of the chunk
    int64_t n;             // tokens in the chunk
    int tiles_per_split;
    int ntiles;
    float* partial;        // [splits][3][BH][dh*d]
    int BH;
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
k_grad_tc(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
          const __grid_constant__ CUtensorMap tm_w1, const __grid_constant__ CUtensorMap tm_w3,
          const __grid_constant__ CUtensorMap tm_w2, const GradArgs a) {
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
    const uint32_t base = smem_u32(sm);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };

    const int tile_begin = split * a.tiles_per_split;
    const int tile_end = min(a.ntiles, tile_begin + a.tiles_per_split);
    const int count = max(0, tile_end - tile_begin);

    if (tid == 0) {
        skip_cta = (*reinterpret_cast<volatile int*>(a.status) & ST_TIMEOUT) ? 1 : 0;
        abort_flag = 0;
        mbar_init(bar(B_W), 1);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar(B_KF + s), 1);
            mbar_init(bar(B_VF + s), 1);
            mbar_init(bar(B_KE + s), 1);
            mbar_init(bar(B_VE + s), 1);
        }
        mbar_init(bar(B_FWDF), 1);
        mbar_init(bar(B_FWDE), 8);
        mbar_init(bar(B_DHF), 8);
        mbar_init(bar(B_UF), 8);
        mbar_init(bar(B_DHE), 1);
        mbar_init(bar(B_UE), 1);
        mbar_init(bar(B_ACC), 1);
        mbar_init(bar(B_DRAIN), 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (skip_cta) return;   // an earlier CTA's wait gave up: results are void anyway
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
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            mbar_expect_tx(bar(B_W), 3 * BOX);   // [W1_r ; W3_r] (32 KB) + W2[:, r] (16 KB)
            const int wrow = bh * a.dh + r * HB;
            for (int at = 0; at < 2; ++at) {
                tma_load_2d(base + OFF_WCAT + at * BOX, &tm_w1, bar(B_W), at * 64, wrow);
                tma_load_2d(base + OFF_WCAT + at * BOX + BOX / 2, &tm_w3, bar(B_W), at * 64, wrow);
            }
            tma_load_2d(base + OFF_W2, &tm_w2, bar(B_W), r * HB, bh * D);
            // One CTA of each group of hidden blocks (r == 0) pulls the K/V
            // tiles PF tiles ahead into L2, where the whole group finds them.
            auto prefetch = [&](int i) {
                if (r != 0 || i >= count) return;
                const int tok = (int)(a.t0 + (int64_t)(tile_begin + i) * TT);
                tma_prefetch_l2_3d(&tm_k, 0, tok, bh);
                tma_prefetch_l2_3d(&tm_k, 64, tok, bh);
                tma_prefetch_l2_3d(&tm_v, 0, tok, bh);
                tma_prefetch_l2_3d(&tm_v, 64, tok, bh);
            };
            for (int i = 0; i < PF; ++i) prefetch(i);
            int issued_k = 0, issued_v = 0;
            for (int i = 0; i < count && !*abort_v; ++i) {
                prefetch(i + PF);
                const int s = i % STAGES;
                const uint32_t ph = ((i / STAGES) - 1) & 1;
                const int tok = (int)(a.t0 + (int64_t)(tile_begin + i) * TT);
                const uint32_t st = base + OFF_KV + s * KV_STAGE;
                if (i >= STAGES && !mbar_wait(bar(B_KE + s), ph, WAIT_NS)) { give_up(); break; }
                mbar_expect_tx(bar(B_KF + s), 2 * BOX);
                tma_load_3d(st + 0 * BOX, &tm_k, bar(B_KF + s), 0, tok, bh);
                tma_load_3d(st + 1 * BOX, &tm_k, bar(B_KF + s), 64, tok, bh);
                issued_k = i + 1;
                if (i >= STAGES && !mbar_wait(bar(B_VE + s), ph, WAIT_NS)) { give_up(); break; }
                mbar_expect_tx(bar(B_VF + s), 2 * BOX);
                tma_load_3d(st + 2 * BOX, &tm_v, bar(B_VF + s), 0, tok, bh);
                tma_load_3d(st + 3 * BOX, &tm_v, bar(B_VF + s), 64, tok, bh);
                issued_v = i + 1;
            }
            // drain: the copies this thread started must land before the CTA exits
            mbar_wait(bar(B_W), 0, WAIT_NS);
            for (int i = max(0, issued_k - STAGES); i < issued_k; ++i)
                mbar_wait(bar(B_KF + i % STAGES), (i / STAGES) & 1, WAIT_NS);
            for (int i = max(0, issued_v - STAGES); i < issued_v; ++i)
                mbar_wait(bar(B_VF + i % STAGES), (i / STAGES) & 1, WAIT_NS);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t i_fwd13 = idesc_bf16_f32(128, 128, 0, 0);
            const uint32_t i_fwda = idesc_bf16_f32(128, 64, 0, 1);
            const uint32_t i_g13 = idesc_bf16_f32(128, 128, 1, 1);
            const uint32_t i_g2 = idesc_bf16_f32(128, 64, 1, 1);
            // Descriptor bases; the start-address field is the low 14 bits
            // (address / 16), so every k-step, stage and operand offset below
            // is a constant added to a base.
            const uint64_t dK = sdesc_sw128(base + OFF_KV, 16, 1024);       // K, V tiles, K-major
            const uint64_t dKT = sdesc_sw128(base + OFF_KV, BOX, 1024);     // K, V tiles, MN-major
            const uint64_t dWc = sdesc_sw128(base + OFF_WCAT, 16, 1024);    // [W1_r ; W3_r], K-major
            const uint64_t dW2 = sdesc_sw128(base + OFF_W2, BOX, 1024);     // W2[:, r], MN-major
            const uint64_t dDH = sdesc_sw128(base + OFF_B, BOX, 1024);      // [dh1 | dh3], MN-major
            const uint64_t dU = sdesc_sw128(base + OFF_B + 2 * BOX, BOX, 1024);  // u', MN-major
            constexpr uint64_t V_OFF = (2 * BOX) >> 4;
            const uint32_t t_h13 = tmem + COL_H13, t_a = tmem + COL_A;
            const uint32_t t_dw13 = tmem + COL_DW13, t_dw2 = tmem + COL_DW2;
            bool ok = mbar_wait(bar(B_W), 0, WAIT_NS);
            if (!ok) give_up();
            auto issue_g13 = [&](int i) {
                const uint64_t so = (uint64_t)((i % STAGES) * KV_STAGE) >> 4;
#pragma unroll
                for (int j = 0; j < TT / 16; ++j)
                    mma_bf16(t_dw13, dKT + so + j * 128, dDH + j * 128, i_g13, (i > 0 || j > 0) ? 1u : 0u);
                mma_commit(bar(B_KE + i % STAGES));
                mma_commit(bar(B_DHE));
            };
            auto issue_g2 = [&](int i) {
                const uint64_t so = (uint64_t)((i % STAGES) * KV_STAGE) >> 4;
#pragma unroll
                for (int j = 0; j < TT / 16; ++j)
                    mma_bf16(t_dw2, dKT + so + V_OFF + j * 128, dU + j * 128, i_g2, (i > 0 || j > 0) ? 1u : 0u);
                mma_commit(bar(B_VE + i % STAGES));
                mma_commit(bar(B_UE));
            };
            auto issue_fwd = [&](int i) {
                const uint64_t so = (uint64_t)((i % STAGES) * KV_STAGE) >> 4;
#pragma unroll
                for (int j = 0; j < D / 16; ++j) {
                    const uint64_t ko = (uint64_t)((j >> 2) * BOX + (j & 3) * 32) >> 4;
                    mma_bf16(t_h13, dK + so + ko, dWc + ko, i_fwd13, j > 0 ? 1u : 0u);
                }
#pragma unroll
                for (int j = 0; j < D / 16; ++j) {
                    const uint64_t ko = (uint64_t)((j >> 2) * BOX + (j & 3) * 32) >> 4;
                    mma_bf16(t_a, dK + so + V_OFF + ko, dW2 + j * 128, i_fwda, j > 0 ? 1u : 0u);
                }
                mma_commit(bar(B_FWDF));
            };
            // Issue whichever is ready first: the dW1/dW3 GEMMs of tile g13
            // (its dh1, dh3 are written), the dW2 GEMMs of tile g2 (its u' is
            // written), or the forward GEMMs of tile f (its K/V have landed
            // and the epilogue has read tile f-1 out of TMEM).
            int f = 0, g13 = 0, g2 = 0;
            uint64_t deadline = globaltimer_ns() + WAIT_NS;
            while (ok && g2 < count && !*abort_v) {
                bool progress = false;
                if (g13 < f && mbar_probe(bar(B_DHF), g13 & 1)) {
                    tc_fence_after();
                    issue_g13(g13++);
                    progress = true;
                }
                if (g2 < g13 && mbar_probe(bar(B_UF), g2 & 1)) {
                    tc_fence_after();
                    issue_g2(g2++);
                    progress = true;
                }
                if (f < count && (f == 0 || mbar_probe(bar(B_FWDE), (f - 1) & 1)) &&
                    mbar_probe(bar(B_KF + f % STAGES), (f / STAGES) & 1) &&
                    mbar_probe(bar(B_VF + f % STAGES), (f / STAGES) & 1)) {
                    tc_fence_after();
                    issue_fwd(f++);
                    progress = true;
                }
                if (progress) {
                    deadline = globaltimer_ns() + WAIT_NS;
                } else if (globaltimer_ns() > deadline) {
                    give_up();
                    ok = false;
                }
            }
            mma_commit(bar(B_ACC));
            // drain: every MMA issued above has completed once this commit lands
            mma_commit(bar(B_DRAIN));
            mbar_wait(bar(B_DRAIN), 0, WAIT_NS);
        }
    } else {
        // --------------------------------------------------------- epilogue
        const int q = warp & 3;                 // TMEM lane quarter of this warp
        const int hf = (warp - 2) >> 2;         // which 32 of the 64 hidden units
        const int row = 32 * q + lane;          // token within the tile / d index
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        unsigned char* bbuf = sm + OFF_B;
        const float* eta_h = a.eta + (int64_t)bh * a.n_total + a.t0;
        uint32_t boff[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) boff[c] = sw128_offset(row, hf * 32 + c * 8);
        bool ok = true;
        // eta of this thread's token, fetched two tiles ahead so the DRAM
        // latency hides behind the work of the tiles in between
        auto eta_of = [&](int i) -> float {
            const int64_t tok = (int64_t)(tile_begin + i) * TT + row;
            return (i < count && tok < a.n) ? eta_h[tok] : 0.0f;
        };
        float e_next = eta_of(0), e_next2 = eta_of(1);
        const f2 half2 = f2_make(0.5f, 0.5f), one2 = f2_make(1.0f, 1.0f), mone2 = f2_make(-1.0f, -1.0f);
        for (int i = 0; i < count; ++i) {
            const float e = e_next;
            e_next = e_next2;
            e_next2 = eta_of(i + 2);
            if (*abort_v || !mbar_wait_warp(bar(B_FWDF), i & 1, WAIT_NS)) { give_up(); ok = false; break; }
            tc_fence_after();
            uint32_t h1[32], h3[32], av[32];
            tmem_ld32(lane_base + COL_H13 + hf * 32, h1);
            tmem_ld32(lane_base + COL_H13 + 64 + hf * 32, h3);
            tmem_ld32(lane_base + COL_A + hf * 32, av);
            tmem_wait_ld();
            tmem_pin(h1);
            tmem_pin(h3);
            tmem_pin(av);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_FWDE));
            // Per hidden unit (pairs of units per instruction):
            //   s = sigmoid(h1) = 0.5 tanh(h1 / 2) + 0.5,  silu = h1 s
            //   u'  = -eta silu h3                      (dW2 operand)
            //   du  = -eta a                            (a = (W2^T v))
            //   dh3 = du silu,  dh1 = du h3 (s + silu (1 - s))
            const f2 ne2 = f2_make(-e, -e);
            uint32_t p1[16], p3[16], pu[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                const f2 x1 = f2_make(__uint_as_float(h1[j]), __uint_as_float(h1[j + 1]));
                const f2 x3 = f2_make(__uint_as_float(h3[j]), __uint_as_float(h3[j + 1]));
                const f2 av2 = f2_make(__uint_as_float(av[j]), __uint_as_float(av[j + 1]));
                float hx0, hx1;
                f2_split(f2_mul(x1, half2), hx0, hx1);
                const f2 t = f2_make(tanh_approx(hx0), tanh_approx(hx1));
                const f2 sg = f2_fma(t, half2, half2);            // sigmoid(h1)
                const f2 si = f2_mul(x1, sg);                     // silu(h1)
                const f2 x3n = f2_mul(x3, ne2);                   // -eta h3
                const f2 du = f2_mul(av2, ne2);                   // -eta a
                const f2 oms = f2_fma(sg, mone2, one2);           // 1 - s
                const f2 g = f2_fma(si, oms, sg);                 // silu'(h1)
                pu[j / 2] = pack_f2(f2_mul(si, x3n));
                p3[j / 2] = pack_f2(f2_mul(du, si));
                p1[j / 2] = pack_f2(f2_mul(f2_mul(du, x3), g));
            }
            if (i >= 1 && !mbar_wait_warp(bar(B_DHE), (i - 1) & 1, WAIT_NS)) { give_up(); ok = false; break; }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t off = boff[c];
                *reinterpret_cast<uint4*>(bbuf + off) = make_uint4(p1[4 * c], p1[4 * c + 1], p1[4 * c + 2], p1[4 * c + 3]);
                *reinterpret_cast<uint4*>(bbuf + BOX + off) =
                    make_uint4(p3[4 * c], p3[4 * c + 1], p3[4 * c + 2], p3[4 * c + 3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_DHF));
            if (i >= 1 && !mbar_wait_warp(bar(B_UE), (i - 1) & 1, WAIT_NS)) { give_up(); ok = false; break; }
#pragma unroll
            for (int c = 0; c < 4; ++c)
                *reinterpret_cast<uint4*>(bbuf + 2 * BOX + boff[c]) =
                    make_uint4(pu[4 * c], pu[4 * c + 1], pu[4 * c + 2], pu[4 * c + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_UF));
        }
        // ---- the CTA's partial dW out of TMEM
        if (ok && !*abort_v && mbar_wait_warp(bar(B_ACC), 0, WAIT_NS)) {
            tc_fence_after();
            const size_t mat = (size_t)a.BH * a.dh * D;
            float* part = a.partial + (size_t)split * 3 * mat + (size_t)bh * a.dh * D;
            if (count > 0) {
                // dW1_r^T (hf 0) or dW3_r^T (hf 1): lane = d index `row`, column = hidden unit
                float* pm = part + (hf == 0 ? 0 : 2 * mat);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t v[32];
                    tmem_ld32(lane_base + COL_DW13 + hf * 64 + half * 32, v);
                    tmem_wait_ld();
                    tmem_pin(v);
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        pm[(size_t)(r * HB + half * 32 + j) * D + row] = __uint_as_float(v[j]);
                }
                uint32_t v[32];
                tmem_ld32(lane_base + COL_DW2 + hf * 32, v);
                tmem_wait_ld();
                tmem_pin(v);
                float* p2 = part + mat + (size_t)row * a.dh + r * HB + hf * 32;
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4*>(p2 + j) = make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                                                     __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
            } else {
                float* pm = part + (hf == 0 ? 0 : 2 * mat);
                for (int j = 0; j < 64; ++j) pm[(size_t)(r * HB + j) * D + row] = 0.0f;
                float* p2 = part + mat + (size_t)row * a.dh + r * HB + hf * 32;
                for (int j = 0; j < 32; ++j) p2[j] = 0.0f;
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

bool grad_tc_supported(const lact_state* st) {
    return st->cfg.io_dtype == LACT_BF16 && st->cfg.d == D && st->cfg.dh % HB == 0 && tmap_available();
}

cudaError_t launch_grad_tc(const lact_state* st, TokView k, TokView v, const float* eta, int* slots,
                           double side_tiles, cudaStream_t s) {
    const int dh = st->cfg.dh, BH = st->BH;
    CUtensorMap mk, mv, m1, m3, m2;
    const uint64_t kv_dims[3] = {(uint64_t)D, (uint64_t)k.n_total, (uint64_t)BH};
    const uint64_t kv_str[2] = {(uint64_t)D * 2, (uint64_t)k.n_total * D * 2};
    const uint32_t kv_box[3] = {64, TT, 1};
    const uint64_t vv_dims[3] = {(uint64_t)D, (uint64_t)v.n_total, (uint64_t)BH};
    const uint64_t vv_str[2] = {(uint64_t)D * 2, (uint64_t)v.n_total * D * 2};
    const uint64_t w13_dims[2] = {(uint64_t)D, (uint64_t)BH * dh};
    const uint64_t w13_str[1] = {(uint64_t)D * 2};
    const uint32_t w13_box[2] = {64, HB};
    const uint64_t w2_dims[2] = {(uint64_t)dh, (uint64_t)BH * D};
    const uint64_t w2_str[1] = {(uint64_t)dh * 2};
    const uint32_t w2_box[2] = {64, D};
    if (!make_tmap_bf16(&mk, k.p, 3, kv_dims, kv_str, kv_box) || !make_tmap_bf16(&mv, v.p, 3, vv_dims, vv_str, kv_box) ||
        !make_tmap_bf16(&m1, st->Wsh[0], 2, w13_dims, w13_str, w13_box) ||
        !make_tmap_bf16(&m3, st->Wsh[2], 2, w13_dims, w13_str, w13_box) ||
        !make_tmap_bf16(&m2, st->Wsh[1], 2, w2_dims, w2_str, w2_box))
        return cudaErrorInvalidValue;

    const int ntiles = (int)((k.n + TT - 1) / TT);
    const int units = BH * (dh / HB);
    // Token splits (one CTA per SM; each split writes one fp32 partial per
    // unit that the reduction or Newton-Schulz reads back). Cost in units of
    // one tile's time: waves x (tiles per CTA + ~3 tiles of pipeline fill and
    // drain per CTA); when other work shares the GPU (side_tiles, e.g. the
    // chunk's readout beside it in the causal order) it takes the SMs a short
    // last wave leaves idle, so the phase ends no earlier than the SM-time of
    // both over the SM count; + ~0.5 per split for writing and re-reading
    // its partial sums. This picks one long wave where the grid allows (e.g. 48
    // units x 3 splits on 148 SMs), whole waves of shorter CTAs otherwise,
    // and few splits when a readout fills the gaps.
    int splits = 1;
    double best = 1e30;
    for (int sp = 1; sp <= kMaxSlots && sp <= ntiles; ++sp) {
        const int tps = (ntiles + sp - 1) / sp;
        const int used = (ntiles + tps - 1) / tps;
        if (used != sp) continue;
        const int64_t ctas = (int64_t)units * sp;
        const int64_t waves = (ctas + st->num_sms - 1) / st->num_sms;
        const double path = (double)waves * (tps + 3.0);
        const double shared = side_tiles > 0 ? ((double)ctas * (tps + 3.0) + side_tiles) / st->num_sms : 0.0;
        const double cost = (path > shared ? path : shared) + 0.5 * sp;
        if (cost < best - 1e-9) { best = cost; splits = sp; }
    }
    const int tps = (ntiles + splits - 1) / splits;

    GradArgs ga;
    ga.eta = eta;
    ga.n_total = k.n_total;
    ga.t0 = k.t0;
    ga.n = k.n;
    ga.tiles_per_split = tps;
    ga.ntiles = ntiles;
    ga.partial = static_cast<float*>(st->partial);
    ga.BH = BH;
    ga.dh = dh;
    ga.status = st->status;
    cudaError_t e = cudaFuncSetAttribute(k_grad_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid(dh / HB, splits, BH);
    launch_pdl(k_grad_tc, grid, NTHREADS, SMEM_BYTES, s, mk, mv, m1, m3, m2, ga);
    g_launches++;
    g_tc_launches++;
    *slots = splits;
    return cudaGetLastError();
}

}  // namespace lact
