// Weight-gradient GEMMs of the chunk gradient on the sm_103a tensor cores
// (tcgen05 + TMA + TMEM), for the two-kernel form of the chunk gradient used
// at head dim 256 (LaCT review page, "Local attention and nonlinear memory
// work together": the chunk gradient as chunk-wide GEMMs).
//
// With the per-token quantities dh1, dh3, u' (bf16, [tokens, dh], written by
// k_fwdbwd_tc) and the chunk's keys K and values V ([tokens, d]):
//   dW1 = dh1^T K      [dh x d]
//   dW3 = dh3^T K      [dh x d]
//   dW2 = V^T u'       [d x dh]
// Each is C (+)= A^T B summed over the tokens, with A and B stored
// token-major (row = token), so both are MN-major operands. One CTA computes
// a 128 x NB tile of one product for one head over the tokens of its split
// (one split here: no partial sums), with a TMA pipeline of 64-token stages
// (4 deep at NB = 256, 6 at NB = 128, in the same 192 KB) and the fp32
// accumulator in TMEM.
//
// The same kernel forms the chunk gradient of the linear fast-weight memory,
// dW = -(eta V)^T K (LaCT review page, Fig. 8: the linear state): there the
// epilogue warps scale every token row of the A tile (V) by -eta in shared
// memory before the MMAs read it, and the tokens are split over CTAs whose
// partial sums a fixed-order reduction adds.
//
// Warp roles (192 threads): warp 0 issues TMA loads, warp 1 owns TMEM and
// issues the MMAs (one thread), warps 2..5 write the tile out (thread = row
// of C). Every wait is bounded; a wait that gives up sets ST_TIMEOUT and the
// CTA unwinds.
#include "lact_internal.cuh"
#include "tc_ptx.cuh"

namespace lact {

namespace {

using namespace tc;

constexpr int TM = 128;        // rows of C per CTA
constexpr int TK = 64;         // tokens per stage
constexpr int MAXST = 6;       // stages, at most
constexpr int NBMAX = 256;     // columns of C per CTA (at most)
constexpr int NTHREADS = 192;
constexpr uint32_t BOXB = TK * 128;                       // one [64 tokens][64 elements] box: 8 KB
constexpr uint32_t A_BYTES = (TM / 64) * BOXB;            // 16 KB
constexpr uint32_t RING_BYTES = 4 * (A_BYTES + (NBMAX / 64) * BOXB);   // 192 KB: 4 stages at NB = 256
constexpr uint32_t SMEM_BYTES = RING_BYTES + 1024;
constexpr uint64_t WAIT_NS = 2000000000ull;

enum { B_F = 0, B_E = MAXST, B_S = 2 * MAXST, B_ACC = 3 * MAXST, B_DRAIN, NBARS };

// One product C (+)= A^T B of one head. The tensor maps cover all heads:
// A: (ma inner, tokens, heads), B: (nb inner, tokens, heads).
struct WProblem {
    int ma;              // columns of A = rows of C
    int nb;              // columns of B = columns of C
    int a_t0, b_t0;      // first token of the slice in A's / B's token axis
    float* c;            // C of head 0, [ma][nb] row-major; head h at c + h * ma * nb
};

struct WArgs {
    WProblem p[3];
    int tiles[3];        // tiles of each product: (ma / 128) * (nb / NB)
    int nb_tile[3];      // NB of each product: 256 or 128
    int ntok;            // tokens in the slice
    int accumulate;      // add to C instead of overwriting it
    int* status;
    const float* eta;    // nullptr, or: scale A's token rows by -eta (head h at eta + h * eta_n_total + eta_t0)
    int64_t eta_n_total, eta_t0;
    int toks_per_split;  // tokens per split (grid z); a multiple of 64
    size_t split_stride; // elements between the C of consecutive splits
};

__global__ void __launch_bounds__(NTHREADS, 1)
k_wgrad_tc(const __grid_constant__ CUtensorMap ta0, const __grid_constant__ CUtensorMap tb0,
           const __grid_constant__ CUtensorMap ta1, const __grid_constant__ CUtensorMap tb1,
           const __grid_constant__ CUtensorMap ta2, const __grid_constant__ CUtensorMap tb2, const WArgs a) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(16) unsigned char smraw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t bars[NBARS];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ int skip_cta;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.y;
    int t = blockIdx.x, which = 0;
    while (which < 2 && t >= a.tiles[which]) t -= a.tiles[which++];
    const WProblem& P = a.p[which];
    const int NB = a.nb_tile[which];
    const int n_blocks = P.nb / NB;
    const int mb = t / n_blocks, nbk = t % n_blocks;
    const CUtensorMap* tma = which == 0 ? &ta0 : which == 1 ? &ta1 : &ta2;
    const CUtensorMap* tmb = which == 0 ? &tb0 : which == 1 ? &tb1 : &tb2;
    const int split = blockIdx.z;
    const int tok0 = split * a.toks_per_split;                       // first token of this split
    const int tok1 = min(a.ntok, tok0 + a.toks_per_split);
    const int nsteps = tok1 > tok0 ? (tok1 - tok0 + TK - 1) / TK : 0;
    const bool scale = a.eta != nullptr;
    const uint32_t STAGE_BYTES = A_BYTES + (uint32_t)(NB / 64) * BOXB;
    const int STAGES = min(MAXST, (int)(RING_BYTES / STAGE_BYTES));
    const uint32_t base = smem_u32(sm);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };

    if (tid == 0) {
        skip_cta = (*reinterpret_cast<volatile int*>(a.status) & ST_TIMEOUT) ? 1 : 0;
        abort_flag = 0;
        for (int s = 0; s < MAXST; ++s) {
            mbar_init(bar(B_F + s), 1);
            mbar_init(bar(B_E + s), 1);
            mbar_init(bar(B_S + s), 4);
        }
        mbar_init(bar(B_ACC), 1);
        mbar_init(bar(B_DRAIN), 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (skip_cta) return;
    if (warp == 1) {
        __syncwarp();
        tmem_alloc(smem_u32(&tmem_slot), 256);
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
            prefetch_tmap(tma);
            prefetch_tmap(tmb);
            const uint32_t bytes = STAGE_BYTES;
            int issued = 0;
            for (int i = 0; i < nsteps && !*abort_v; ++i) {
                const int s = i % STAGES;
                if (i >= STAGES && !mbar_wait(bar(B_E + s), ((i / STAGES) - 1) & 1, WAIT_NS)) { give_up(); break; }
                const uint32_t st = base + s * STAGE_BYTES;
                mbar_expect_tx(bar(B_F + s), bytes);
                for (int c = 0; c < TM / 64; ++c)
                    tma_load_3d(st + c * BOXB, tma, bar(B_F + s), mb * TM + c * 64, P.a_t0 + tok0 + i * TK, h);
                for (int c = 0; c < NB / 64; ++c)
                    tma_load_3d(st + A_BYTES + c * BOXB, tmb, bar(B_F + s), nbk * NB + c * 64, P.b_t0 + tok0 + i * TK, h);
                issued = i + 1;
            }
            for (int i = max(0, issued - STAGES); i < issued; ++i)
                mbar_wait(bar(B_F + i % STAGES), (i / STAGES) & 1, WAIT_NS);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(TM, NB, 1, 1);
            const uint64_t dA = sdesc_sw128(base, BOXB, 1024);               // MN-major, 64-element blocks BOXB apart
            const uint64_t dB = sdesc_sw128(base + A_BYTES, BOXB, 1024);
            bool ok = true;
            for (int i = 0; i < nsteps && ok && !*abort_v; ++i) {
                const int s = i % STAGES;
                if (!mbar_wait(bar((scale ? B_S : B_F) + s), (i / STAGES) & 1, WAIT_NS)) { give_up(); ok = false; break; }
                tc_fence_after();
                const uint64_t so = (uint64_t)(s * STAGE_BYTES) >> 4;
#pragma unroll
                for (int j = 0; j < TK / 16; ++j)
                    mma_bf16(tmem, dA + so + j * 128, dB + so + j * 128, idesc, (i > 0 || j > 0) ? 1u : 0u);
                mma_commit(bar(B_E + s));
            }
            mma_commit(bar(B_ACC));
            mma_commit(bar(B_DRAIN));
            mbar_wait(bar(B_DRAIN), 0, WAIT_NS);
        }
    } else {
        // thread = row of the C tile (TMEM lane); columns in groups of 32
        const int q = warp & 3;
        const int row = 32 * q + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        if (scale) {
            // every token row of the A tile times -eta of its token (a swizzled
            // row keeps its 128 bytes in place, so a whole row scales as one)
            const int et = tid - 64;                    // 0..127: (64-element block, token row)
            const int blk = et >> 6, trow = et & 63;
            const float* eh = a.eta + (int64_t)h * a.eta_n_total + a.eta_t0;
            // eta of this thread's row, fetched one stage ahead so its DRAM
            // latency overlaps the stage's TMA
            auto eta_row = [&](int i) -> float {
                const int tok = tok0 + i * TK + trow;
                return (i < nsteps && tok < tok1) ? -eh[tok] : 0.0f;
            };
            float ne_next = eta_row(0);
            for (int i = 0; i < nsteps; ++i) {
                const int s = i % STAGES;
                const float ne = ne_next;
                ne_next = eta_row(i + 1);
                if (*abort_v || !mbar_wait_warp(bar(B_F + s), (i / STAGES) & 1, WAIT_NS)) { give_up(); break; }
                uint4* rp = reinterpret_cast<uint4*>(sm + s * STAGE_BYTES + blk * BOXB + trow * 128);
                // the 8 chunks of the row in an order rotated by lane, so that
                // the 32 rows of a warp (128 bytes apart) spread over all
                // banks; all loads first, then all stores
                uint4 x[8];
#pragma unroll
                for (int c0 = 0; c0 < 8; ++c0) x[c0] = rp[(c0 + lane) & 7];
#pragma unroll
                for (int c0 = 0; c0 < 8; ++c0) {
                    uint32_t* w = reinterpret_cast<uint32_t*>(&x[c0]);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        __nv_bfloat162 pr = *reinterpret_cast<__nv_bfloat162*>(&w[u]);
                        float2 f = __bfloat1622float2(pr);
                        pr = __floats2bfloat162_rn(f.x * ne, f.y * ne);
                        w[u] = *reinterpret_cast<uint32_t*>(&pr);
                    }
                }
#pragma unroll
                for (int c0 = 0; c0 < 8; ++c0) rp[(c0 + lane) & 7] = x[c0];
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_S + s));
            }
        }
        if (!*abort_v && mbar_wait_warp(bar(B_ACC), 0, WAIT_NS)) {
            tc_fence_after();
            float* crow = P.c + (size_t)split * a.split_stride + (size_t)h * P.ma * P.nb + (size_t)(mb * TM + row) * P.nb +
                          nbk * NB;
            for (int c0 = 0; c0 < NB; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(lane_base + c0, v);
                tmem_wait_ld();
                tmem_pin(v);
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    float4 x = make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]), __uint_as_float(v[j + 2]),
                                           __uint_as_float(v[j + 3]));
                    if (nsteps == 0) x = make_float4(0.f, 0.f, 0.f, 0.f);
                    float4* dst = reinterpret_cast<float4*>(crow + c0 + j);
                    if (a.accumulate) {
                        const float4 o = *dst;
                        x.x += o.x; x.y += o.y; x.z += o.z; x.w += o.w;
                    }
                    *dst = x;
                }
            }
        } else if (!*abort_v) {
            give_up();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

}  // namespace

// dW1 = dh1^T K, dW3 = dh3^T K, dW2 = V^T u' over one token slice, into
// out[0..2] (fp32, [BH, ...]); `inter` holds dh1, dh3, u' as [3][BH][slice_cap][dh].
cudaError_t launch_wgrad_tc(const lact_state* st, TokView k, TokView v, const bf16* inter, int64_t slice_cap,
                            bool accumulate, void* const out[3], cudaStream_t s) {
    const int d = st->cfg.d, dh = st->cfg.dh, BH = st->BH;
    const int ntok = (int)k.n;
    CUtensorMap ma[3], mb[3];
    // intermediates: (dh, ntok, BH) with the slice's own token count, so rows past it read as zero
    const uint64_t i_dims[3] = {(uint64_t)dh, (uint64_t)(ntok > 0 ? ntok : 1), (uint64_t)BH};
    const uint64_t i_str[2] = {(uint64_t)dh * 2, (uint64_t)slice_cap * dh * 2};
    const uint32_t box[3] = {64, TK, 1};
    const uint64_t x_dims[3] = {(uint64_t)d, (uint64_t)k.n_total, (uint64_t)BH};
    const uint64_t x_str[2] = {(uint64_t)d * 2, (uint64_t)k.n_total * d * 2};
    const uint64_t v_dims[3] = {(uint64_t)d, (uint64_t)v.n_total, (uint64_t)BH};
    const uint64_t v_str[2] = {(uint64_t)d * 2, (uint64_t)v.n_total * d * 2};
    const size_t inter_one = (size_t)BH * slice_cap * dh;
    bool ok = make_tmap_bf16(&ma[0], inter, 3, i_dims, i_str, box) &&                     // dh1
              make_tmap_bf16(&mb[0], k.p, 3, x_dims, x_str, box) &&                       // K
              make_tmap_bf16(&ma[1], inter + inter_one, 3, i_dims, i_str, box) &&         // dh3
              make_tmap_bf16(&mb[1], k.p, 3, x_dims, x_str, box) &&                       // K
              make_tmap_bf16(&ma[2], v.p, 3, v_dims, v_str, box) &&                       // V
              make_tmap_bf16(&mb[2], inter + 2 * inter_one, 3, i_dims, i_str, box);       // u'
    if (!ok) return cudaErrorInvalidValue;
    WArgs wa;
    const int mas[3] = {dh, dh, d}, nbs[3] = {d, d, dh};
    const int at0[3] = {0, 0, (int)v.t0}, bt0[3] = {(int)k.t0, (int)k.t0, 0};
    int total = 0;
    for (int m = 0; m < 3; ++m) {
        wa.p[m].ma = mas[m];
        wa.p[m].nb = nbs[m];
        wa.p[m].a_t0 = at0[m];
        wa.p[m].b_t0 = bt0[m];
        wa.p[m].c = static_cast<float*>(out[m == 2 ? 1 : (m == 0 ? 0 : 2)]);
        wa.nb_tile[m] = nbs[m] % 256 == 0 ? 256 : 128;
        wa.tiles[m] = (mas[m] / TM) * (nbs[m] / wa.nb_tile[m]);
        total += wa.tiles[m];
    }
    wa.ntok = ntok;
    wa.accumulate = accumulate ? 1 : 0;
    wa.status = st->status;
    wa.eta = nullptr;
    wa.eta_n_total = 0;
    wa.eta_t0 = 0;
    wa.toks_per_split = ntok > 0 ? (ntok + TK - 1) / TK * TK : TK;
    wa.split_stride = 0;
    cudaError_t e = cudaFuncSetAttribute(k_wgrad_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)total, (unsigned)BH, 1);
    launch_pdl(k_wgrad_tc, grid, NTHREADS, SMEM_BYTES, s, ma[0], mb[0], ma[1], mb[1], ma[2], mb[2], wa);
    g_launches++;
    g_tc_launches++;
    return cudaGetLastError();
}

// Linear memory (bf16 io, d = 128): partial dW = -(eta V)^T K of tokens
// [k.t0, k.t0 + k.n), one fp32 partial per token split into st->partial
// ([split][BH][d][d]); *slots receives the number of splits.
cudaError_t launch_lin_grad_tc(const lact_state* st, TokView k, TokView v, const float* eta, int* slots,
                               cudaStream_t s) {
    const int d = st->cfg.d, BH = st->BH;
    CUtensorMap mv, mk;
    const uint32_t box[3] = {64, TK, 1};
    const uint64_t k_dims[3] = {(uint64_t)d, (uint64_t)k.n_total, (uint64_t)BH};
    const uint64_t k_str[2] = {(uint64_t)d * 2, (uint64_t)k.n_total * d * 2};
    const uint64_t v_dims[3] = {(uint64_t)d, (uint64_t)v.n_total, (uint64_t)BH};
    const uint64_t v_str[2] = {(uint64_t)d * 2, (uint64_t)v.n_total * d * 2};
    if (!make_tmap_bf16(&mv, v.p, 3, v_dims, v_str, box) || !make_tmap_bf16(&mk, k.p, 3, k_dims, k_str, box))
        return cudaErrorInvalidValue;
    WArgs wa;
    wa.p[0].ma = d;
    wa.p[0].nb = d;
    wa.p[0].a_t0 = (int)v.t0;
    wa.p[0].b_t0 = (int)k.t0;
    wa.p[0].c = static_cast<float*>(st->partial);
    wa.nb_tile[0] = d % 256 == 0 ? 256 : 128;
    wa.tiles[0] = (d / TM) * (d / wa.nb_tile[0]);
    for (int m = 1; m < 3; ++m) {
        wa.p[m] = wa.p[0];
        wa.nb_tile[m] = wa.nb_tile[0];
        wa.tiles[m] = 0;
    }
    wa.ntok = (int)k.n;
    wa.accumulate = 0;
    wa.status = st->status;
    wa.eta = eta;
    wa.eta_n_total = k.n_total;
    wa.eta_t0 = k.t0;
    // token splits: about one wave of CTAs, whole 64-token stages, at most kMaxSlots
    const int64_t steps = (k.n + TK - 1) / TK;
    int64_t splits = st->num_sms / (BH * wa.tiles[0]);
    if (splits > steps) splits = steps;
    if (splits > kMaxSlots) splits = kMaxSlots;
    if (splits < 1) splits = 1;
    const int64_t sps = (steps + splits - 1) / splits;
    splits = (steps + sps - 1) / sps;
    if (splits < 1) splits = 1;
    wa.toks_per_split = (int)(sps * TK);
    wa.split_stride = (size_t)BH * d * d;
    cudaError_t e = cudaFuncSetAttribute(k_wgrad_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)wa.tiles[0], (unsigned)BH, (unsigned)splits);
    launch_pdl(k_wgrad_tc, grid, NTHREADS, SMEM_BYTES, s, mv, mk, mv, mk, mv, mk, wa);
    g_launches++;
    g_tc_launches++;
    *slots = (int)splits;
    return cudaGetLastError();
}

}  // namespace lact
