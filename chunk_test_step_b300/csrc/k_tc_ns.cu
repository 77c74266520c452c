// Muon's Newton-Schulz orthogonalisation on the sm_103a tensor cores
// (LaCT review page, "Local attention and nonlinear memory work together":
// Muon transforms each matrix gradient with Newton-Schulz iterations).
//
// One thread-block cluster per gradient matrix G (3 per head), for matrices
// whose short side is 128 and long side n <= 512 (a multiple of 128). On the
// orientation with rows <= cols (X is 128 x n):
//   X = G / (||G||_F + 1e-7)
//   repeat ns_steps times:
//     A  = Xb Xb^T             Xb = bf16(X): K-major operand, both sides   (TMEM)
//     AA = Ab Ab               Ab = bf16(A): K-major A, MN-major B        (TMEM)
//     B  = b A + c AA          fp32, from the unrounded A
//     BX = Bb Xb               Bb = bf16(B) K-major; Xb read MN-major     (TMEM)
//     X  = a X + BX            fp32
// The cluster has n/cb CTAs (cb = 256 columns each when n is a multiple of
// 256, else 128); CTA j owns columns [cb j, cb j + cb) of X. Every CTA holds
// the whole bf16 Xb in shared memory (the operand of A) and forms A, AA and B
// itself (they are small: 128 x 128); it forms only its own cb columns of BX
// and keeps its fp32 columns of X in TMEM (BX reuses the columns of A and AA,
// which are dead once B is in shared memory), so nothing of the
// iteration leaves the chip. After each update a CTA writes its new bf16
// columns into its own Xb; each half of the CTA (128 threads, whole 16 KB
// atoms) pushes its columns with one bulk copy into the Xb of every other CTA
// of the cluster (distributed shared memory) as soon as it has written them,
// completing on that CTA's mbarrier for this source. The next
// A GEMM starts on the CTA's own columns and takes each other CTA's columns
// as they land (own block first, then the others in rank order). A
// cluster-wide handshake, "every CTA's A GEMM has finished reading Xb",
// comes before anyone overwrites it.
//
// G is either the summed gradient or, when the caller skipped the split-K
// reduction, its partial slots: each CTA then adds its columns' slots in slot
// order as it reads them (the reduction kernel's order, so the result is the
// same bit for bit). The slots come into shared memory by bulk copies (TMA
// boxes where X is wide), several pieces in flight, before TMEM takes X.
//
// With `fuse` set (Muon), the CTA then applies the optimiser step to its part
// of W itself: W~ = W + scale X (X in W's orientation) and each row of W
// rescaled to its pre-update norm, W' = W~ ||W_j|| / ||W~_j|| (a row whose
// updated norm is 0 is stored as updated; a non-finite norm sets
// ST_NONFINITE), plus W' as bf16. W's tile is copied into the dead Xb during
// the last iteration; W' leaves by bulk copies. A row of W is a column of X
// when X is tall (W1, W3: its norm is a sum over the CTA's 128 lanes) and a
// row of X when X is wide (W2: the CTA's halves and the cluster's CTAs post
// partial sums, added in rank order, so every CTA finds the same factor).
// Nothing is written to G then.
//
// 256 threads: thread = row of X (TMEM lane) and half of the CTA's columns;
// thread 0 also issues the MMAs. Every mbarrier wait is bounded and its
// outcome made block-uniform; the hardware cluster barrier is used only at
// entry and exit, which every CTA reaches unconditionally.
#include "lact_internal.cuh"
#include "tc_ptx.cuh"

namespace lact {

namespace {

using namespace tc;

constexpr int M = 128;
constexpr int NMAX = 512;
constexpr int MAXCS = 4;                           // CTAs per cluster, at most (n = 512 in 128-column blocks)
constexpr int NTHREADS = 256;
constexpr uint32_t ATOM = M * 128;                 // [128 rows][64 bf16] = 16 KB
constexpr uint32_t OFF_X = 0;                      // n/64 atoms of Xb
constexpr uint32_t OFF_A = (NMAX / 64) * ATOM;     // 2 atoms of Ab
constexpr uint32_t OFF_B = OFF_A + 2 * ATOM;       // 2 atoms of Bb
// Fused update (after the iterations): W's tile and W' (fp32), W' as bf16,
// the sums of squares and the row factors.
constexpr uint32_t OFF_S32 = 0;
constexpr uint32_t S32_ROW = 1040;                 // X wide: bytes per row (1 KB + 16)
constexpr uint32_t OFF_S16 = 134144;               // after 128 rows of S32_ROW, 1 KB aligned
constexpr uint32_t S16_ROW = 528;                  // X wide: bytes per bf16 row (512 + 16)
constexpr uint32_t OFF_PN = OFF_S16 + M * S16_ROW;
constexpr uint32_t END_FUSED = OFF_PN + (4 * NMAX * 2 + NMAX) * 4;
constexpr uint32_t SMEM_BYTES = (END_FUSED > OFF_B + 2 * ATOM ? END_FUSED : OFF_B + 2 * ATOM) + 1024;
static_assert(OFF_S16 >= M * S32_ROW && 256 * M * 4 <= OFF_S16 && 256 * M * 2 <= M * S16_ROW, "fused update layout");
// Newton-Schulz input from the split-K partial slots: 16 KB pieces (32
// columns of X for one half and one slot) in a ring of NPIECE buffers.
constexpr uint32_t PIECE = M * 128;
constexpr int NPIECE = 13;
constexpr int MAXRF = 4;
static_assert(NPIECE * PIECE <= END_FUSED, "piece ring");
// TMEM: the CTA's fp32 columns of X at 0 (cb columns); from cb on, A (128)
// and AA (128), later overwritten by BX (cb).
constexpr uint32_t COL_X = 0;

// Columns of X per CTA for a long side n.
__host__ __device__ constexpr int ns_block(int n) { return n % 256 == 0 ? 256 : 128; }
constexpr uint64_t WAIT_NS = 2000000000ull;
__device__ __forceinline__ void bulk_store_s2g(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 ::"l"(reinterpret_cast<uint64_t>(dst)), "r"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_load_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t mbar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(mbar) : "memory");
}

struct NsArgs {
    float* g[3];      // gradients in place: W1 [BH,dh,d], W2 [BH,d,dh], W3 [BH,dh,d]
    const float* part;    // split-K partial slots [slots][nmat][BH][d*dh] (read when slots > 0)
    int slots;
    size_t mat;           // BH * d * dh
    int nmat;
    int BH, d, dh, n, steps;
    float a, b, c;
    // fused update (fuse != 0): in place of writing the result into g, the
    // step W~ = W + scale X, W' = W~ ||W|| / ||W~|| per row of W, and its
    // bf16 shadow, are applied here
    int fuse;
    float* W[3];
    bf16* S[3];
    float scale;
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

// Sums over the 32 lanes of a warp, for 32 columns at once: on entry v[c] is
// this lane's term for column c; on exit v[0] is the warp's sum for column
// `lane` (recursive halving: 31 shuffles in place of 32 x 5).
__device__ __forceinline__ void lane_transpose_sum(float (&v)[32], int lane) {
#pragma unroll
    for (int k = 16; k >= 1; k >>= 1) {
        const bool up = (lane & k) != 0;
#pragma unroll
        for (int m = 0; m < k; ++m) {
            const float send = up ? v[m] : v[m + k];
            const float keep = up ? v[m + k] : v[m];
            v[m] = keep + __shfl_xor_sync(0xffffffffu, send, k);
        }
    }
}

// The update and row renormalisation of the fast weights, applied to this
// CTA's columns of the Newton-Schulz result X (fp32 in TMEM), in place of a
// separate update kernel:
//   W~ = W + scale X   (X in W's orientation),   W' = W~ ||W_j|| / ||W~_j||
// for every row j of W (a row whose updated norm is 0 is stored as updated;
// a non-finite norm sets ST_NONFINITE), and W' also as bf16.
// The CTA's tile of W arrives in shared memory by bulk copies (issued once the
// last BX GEMM has read Xb), W~ replaces X in TMEM, and W' and its bf16 copy
// leave by bulk copies: fp32 at OFF_S32, bf16 at OFF_S16, each in W's own
// row order (X tall: the tile's rows are contiguous in W; X wide: one segment
// per row, rows padded by 16 bytes so that a warp's rows fall in different banks).
//  - X tall (W1, W3: rows of W are columns of X): a row of W lies in one CTA;
//    its norm is a sum over the 128 lanes (threads) of the column.
//  - X wide (W2: rows of W are rows of X): a row's norm is summed over the
//    thread's columns, the two halves of the CTA, then the CTAs of the
//    cluster (each posts its partial sums to all; all add them in rank order).
// Returns false if a bounded wait ran out.
__device__ __forceinline__ bool fused_update(const NsArgs& a, int which, int bh, bool tr, int cols, int cs,
                                             uint32_t rank, int c0, int cb, int half, int row, uint32_t lane_base,
                                             unsigned char* sm, uint32_t base, float (*upart)[M][2], uint32_t bar_u,
                                             uint32_t bar_w) {
    const int tid = threadIdx.x, lane = tid & 31, q = (tid >> 5) & 3;
    const int hc = cb / 2;
    float* Wm = a.W[which] + (size_t)bh * a.d * a.dh;
    bf16* Sm = a.S[which] + (size_t)bh * a.d * a.dh;
    float* pn = reinterpret_cast<float*>(sm + OFF_PN);        // partial sums of squares
    float* fs = pn + 4 * NMAX * 2;                            // per-row factors
    // element (row, column j) of this CTA's block of X, as W stores it
    auto s32 = [&](int j) -> float* {
        return tr ? reinterpret_cast<float*>(sm + OFF_S32) + j * M + row
                  : reinterpret_cast<float*>(sm + OFF_S32 + row * S32_ROW) + j;
    };
    if (__syncthreads_and(mbar_wait(bar_w, 0, WAIT_NS) ? 1 : 0) == 0) return false;
    // pass 1: W~ (into TMEM over X), and the sums of squares of W and W~
    float p0 = 0.f, p1 = 0.f;
    for (int h = 0; h < hc / 32; ++h) {
        const int j0 = half * hc + h * 32;                     // column within the CTA
        uint32_t v[32];
        tmem_ld32(lane_base + COL_X + j0, v);
        tmem_wait_ld();
        tmem_pin(v);
        float w[32], s0[32], s1[32];
        if (tr) {
#pragma unroll
            for (int t = 0; t < 32; ++t) w[t] = *s32(j0 + t);
        } else {
            const float4* wp = reinterpret_cast<const float4*>(s32(j0));
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const float4 x = wp[t];
                w[4 * t] = x.x; w[4 * t + 1] = x.y; w[4 * t + 2] = x.z; w[4 * t + 3] = x.w;
            }
        }
#pragma unroll
        for (int t = 0; t < 32; ++t) {
            const float tt = fmaf(a.scale, __uint_as_float(v[t]), w[t]);
            s0[t] = w[t] * w[t];
            s1[t] = tt * tt;
            v[t] = __float_as_uint(tt);
        }
        tmem_st32(lane_base + COL_X + j0, v);       // W~ over X in TMEM
        if (tr) {
            lane_transpose_sum(s0, lane);
            lane_transpose_sum(s1, lane);
            pn[(q * NMAX + j0 + lane) * 2] = s0[0];
            pn[(q * NMAX + j0 + lane) * 2 + 1] = s1[0];
        } else {
#pragma unroll
            for (int t = 0; t < 32; ++t) {
                p0 += s0[t];
                p1 += s1[t];
            }
        }
    }
    tmem_wait_st();
    if (!tr) {
        pn[(half * M + row) * 2] = p0;
        pn[(half * M + row) * 2 + 1] = p1;
    }
    __syncthreads();
    bool ok = true;
    auto factor = [&](float S0, float S1) -> float {
        const float n0 = sqrtf(S0), n1 = sqrtf(S1);
        if (!isfinite(n0) || !isfinite(n1)) atomicOr(a.status, ST_NONFINITE);
        return n1 > 0.f ? n0 / n1 : 1.f;
    };
    if (tr) {
        // column j of X = row c0 + j of W: the four lane quarters' sums
        for (int j = tid; j < cb; j += NTHREADS) {
            float S0 = 0.f, S1 = 0.f;
            for (int k = 0; k < 4; ++k) {
                S0 += pn[(k * NMAX + j) * 2];
                S1 += pn[(k * NMAX + j) * 2 + 1];
            }
            fs[j] = factor(S0, S1);
        }
    } else {
        // row `tid` of W: the CTA's two halves, posted to every CTA of the
        // cluster; each posting thread releases its own stores with its arrive
        if (tid < M) {
            const float S0 = pn[tid * 2] + pn[(M + tid) * 2], S1 = pn[tid * 2 + 1] + pn[(M + tid) * 2 + 1];
            for (int r = 0; r < cs; ++r) {
                st_cluster_f32(mapa_shared(smem_u32(&upart[rank][tid][0]), (uint32_t)r), S0);
                st_cluster_f32(mapa_shared(smem_u32(&upart[rank][tid][1]), (uint32_t)r), S1);
                mbar_arrive_cluster(mapa_shared(bar_u, (uint32_t)r));
            }
        }
        ok = __syncthreads_and(mbar_wait_cluster(bar_u, 0, WAIT_NS) ? 1 : 0) != 0;
        if (ok && tid < M) {
            float S0 = 0.f, S1 = 0.f;
            for (int r = 0; r < cs; ++r) {
                S0 += upart[r][tid][0];
                S1 += upart[r][tid][1];
            }
            fs[tid] = factor(S0, S1);
        }
    }
    __syncthreads();
    if (!ok) return false;
    // pass 2: W' = W~ f (W~ from TMEM) into the stage, and its bf16 copy
    for (int h = 0; h < hc / 32; ++h) {
        const int j0 = half * hc + h * 32;
        uint32_t v[32];
        tmem_ld32(lane_base + COL_X + j0, v);
        tmem_wait_ld();
        tmem_pin(v);
        float o[32];
        if (tr) {
            const float4* fp = reinterpret_cast<const float4*>(fs + j0);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const float4 f4 = fp[t];
                o[4 * t] = __uint_as_float(v[4 * t]) * f4.x;
                o[4 * t + 1] = __uint_as_float(v[4 * t + 1]) * f4.y;
                o[4 * t + 2] = __uint_as_float(v[4 * t + 2]) * f4.z;
                o[4 * t + 3] = __uint_as_float(v[4 * t + 3]) * f4.w;
            }
#pragma unroll
            for (int t = 0; t < 32; ++t) {
                *s32(j0 + t) = o[t];
                reinterpret_cast<bf16*>(sm + OFF_S16)[(j0 + t) * M + row] = __float2bfloat16_rn(o[t]);
            }
        } else {
            const float f = fs[row];
#pragma unroll
            for (int t = 0; t < 32; ++t) o[t] = __uint_as_float(v[t]) * f;
            float4* wp = reinterpret_cast<float4*>(s32(j0));
#pragma unroll
            for (int t = 0; t < 8; ++t) wp[t] = make_float4(o[4 * t], o[4 * t + 1], o[4 * t + 2], o[4 * t + 3]);
            uint4* sp = reinterpret_cast<uint4*>(sm + OFF_S16 + row * S16_ROW + j0 * 2);
#pragma unroll
            for (int t = 0; t < 4; ++t) sp[t] = pack8(o + 8 * t);
        }
    }
    fence_proxy_async_smem();
    __syncthreads();
    // out by bulk copies (the issuing threads wait until shared memory has been read)
    bool issued = false;
    if (tr) {
        const uint32_t w_piece = (uint32_t)(cb * M * 4 / 8), s_piece = (uint32_t)(cb * M * 2 / 8);
        if (tid < 8) {
            bulk_store_s2g(Wm + (size_t)c0 * cols + tid * (w_piece / 4), base + OFF_S32 + tid * w_piece, w_piece);
            issued = true;
        } else if (tid < 16) {
            bulk_store_s2g(Sm + (size_t)c0 * cols + (tid - 8) * (s_piece / 2), base + OFF_S16 + (tid - 8) * s_piece,
                           s_piece);
            issued = true;
        }
    } else if (tid < M) {
        bulk_store_s2g(Wm + (size_t)tid * cols + c0, base + OFF_S32 + tid * S32_ROW, (uint32_t)(cb * 4));
        bulk_store_s2g(Sm + (size_t)tid * cols + c0, base + OFF_S16 + tid * S16_ROW, (uint32_t)(cb * 2));
        issued = true;
    }
    if (issued) {
        bulk_commit();
        bulk_wait_read0();
    }
    return true;
}

__global__ void __launch_bounds__(NTHREADS, 1) k_ns_tc(const __grid_constant__ CUtensorMap tm_p, const NsArgs a) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(16) unsigned char smraw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t mbar, sync_a, sync_x[MAXCS];
    __shared__ int fail_sh;
    __shared__ uint32_t tmem_slot;
    __shared__ float red[NTHREADS / 32];
    __shared__ float norm_part[MAXCS];   // partial sums of squares, one per CTA of the cluster
    __shared__ __align__(8) uint64_t sync_u, sync_w, gbar[MAXRF];
    __shared__ float upart[MAXCS][M][2];  // fused update: each CTA's row sums of squares (rows spanning the cluster)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = a.n;
    const int cb = ns_block(n);                    // columns of X per CTA
    const int cs = n / cb;                         // CTAs in the cluster
    const uint32_t COL_A = (uint32_t)cb, COL_AA = COL_A + 128, COL_BX = COL_A;
    const uint32_t rank = cluster_rank();
    const int mi = blockIdx.x / cs, which = mi / a.BH, bh = mi % a.BH;
    const int rows = which == 1 ? a.d : a.dh, cols = which == 1 ? a.dh : a.d;
    const bool tr = rows > cols;
    float* G = a.g[which] + (size_t)bh * a.d * a.dh;
    const uint32_t base = smem_u32(sm);
    const uint32_t bar = smem_u32(&mbar);
    const uint32_t bar_a = smem_u32(&sync_a);
    auto barx = [&](int r) { return smem_u32(&sync_x[r]); };   // columns arriving from CTA r
    const int c0 = (int)rank * cb;                 // first column owned by this CTA

    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(bar_a, cs);   // one arrive per CTA of the cluster
        for (int r = 0; r < cs; ++r) mbar_init(barx(r), 1);   // own expect_tx + CTA r's bytes
        mbar_init(smem_u32(&sync_u), M * cs);   // one arrive per posting thread of each CTA
        mbar_init(smem_u32(&sync_w), 1);
        for (int g = 0; g < MAXRF; ++g) mbar_init(smem_u32(&gbar[g]), 1);
        fail_sh = 0;
        fence_mbar_init();
    }
    // barrier initialisation visible to the whole cluster before any remote arrive
    cluster_sync_all();
    if (warp == 1) {
        __syncwarp();
        tmem_alloc(smem_u32(&tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    // ---- X = G / (||G||_F + eps). Each CTA reads its own columns of G once,
    // into TMEM as fp32, summing their squares; the partial sum is posted to
    // every CTA of the cluster (every CTA adds the partials in rank order, so
    // all hold the same norm). Then each thread scales its values in TMEM and
    // writes them as bf16 into its block of Xb.
    // Thread (row, half) owns row `row` of X and hc = cb/2 of the columns.
    const int q = warp & 3, half = warp >> 2;
    const int row = 32 * q + lane;             // row of X owned by this thread
    const int hc = cb / 2;
    // 32 consecutive columns j0.. of this thread's row: element (row, j) of X
    // is G[j][row] when G is stored tall (a warp's 32 rows read 32
    // consecutive words), else G[row][j] (the thread reads 128 contiguous bytes)
    auto load32 = [&](int j0, float* x) {
        if (a.slots > 0) {
            // the split-K partial sums of this matrix, added in slot order;
            // every slot's loads are issued before the first add
            const float* P0 = a.part + (size_t)which * a.mat + (size_t)bh * a.d * a.dh;
            const size_t stride = (size_t)a.nmat * a.mat;
            float y[2][32];
#pragma unroll
            for (int t = 0; t < 32; ++t) x[t] = 0.f;
            for (int s0 = 0; s0 < a.slots; s0 += 2) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int sl = s0 + u;
                if (sl < a.slots) {
                    const float* P = P0 + (size_t)sl * stride;
                    if (tr) {
#pragma unroll
                        for (int t = 0; t < 32; ++t) y[u][t] = P[(size_t)(j0 + t) * cols + row];
                    } else {
                        const float4* gp = reinterpret_cast<const float4*>(P + (size_t)row * cols + j0);
#pragma unroll
                        for (int t = 0; t < 8; ++t) {
                            const float4 v = gp[t];
                            y[u][4 * t] = v.x; y[u][4 * t + 1] = v.y; y[u][4 * t + 2] = v.z; y[u][4 * t + 3] = v.w;
                        }
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u)
                if (s0 + u < a.slots) {
#pragma unroll
                    for (int t = 0; t < 32; ++t) x[t] += y[u][t];
                }
            }
            return;
        }
        if (tr) {
#pragma unroll
            for (int t = 0; t < 32; ++t) x[t] = G[(size_t)(j0 + t) * cols + row];
        } else {
            const float4* gp = reinterpret_cast<const float4*>(G + (size_t)row * cols + j0);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const float4 v = gp[t];
                x[4 * t] = v.x; x[4 * t + 1] = v.y; x[4 * t + 2] = v.z; x[4 * t + 3] = v.w;
            }
        }
    };
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
    float ss = 0.f;
    bool pre_ok = true;
    int g_issued = 0, g_waited = 0;     // rounds of pieces started / seen complete (thread 0's drain)
    const int S = a.slots, rounds = hc / 32, per_round = 2 * S;
    const int RF = S > 0 ? min(min(rounds, NPIECE / per_round), MAXRF) : 0;
    if (S > 0) {
        // The partial slots come into shared memory by bulk copies: a piece
        // is 32 columns of X for one half and one slot (16 KB); a round is
        // both halves' pieces of every slot; up to RF rounds are in flight.
        // Each thread adds its row's values over the slots in slot order.
        //  - X tall: the piece is 32 whole rows of G (contiguous), read
        //    [column][row] by the threads;
        //  - X wide: a TMA box of 128 rows x 32 columns, 128-byte swizzled.
        const float* P0 = a.part + (size_t)which * a.mat + (size_t)bh * a.d * a.dh;
        const size_t sstride = (size_t)a.nmat * a.mat;
        auto issue_round = [&](int k) {
            const int g = k % RF;
            const uint32_t gb = smem_u32(&gbar[g]);
            mbar_expect_tx(gb, (uint32_t)per_round * PIECE);
            for (int h = 0; h < 2; ++h)
                for (int sl = 0; sl < S; ++sl) {
                    const uint32_t dst = base + (uint32_t)(g * per_round + h * S + sl) * PIECE;
                    const int jc = c0 + h * hc + 32 * k;           // first column of X in the piece
                    if (tr) bulk_load_g2s(dst, P0 + sl * sstride + (size_t)jc * cols, PIECE, gb);
                    else tma_load_2d(dst, &tm_p, gb, jc, ((sl * a.nmat + which) * a.BH + bh) * M);
                }
        };
        if (tid == 0) {
            prefetch_tmap(&tm_p);
            for (int k = 0; k < RF; ++k) issue_round(k);
            g_issued = RF;
        }
        for (int k = 0; k < rounds; ++k) {
            const int g = k % RF;
            pre_ok = __syncthreads_and(mbar_wait(smem_u32(&gbar[g]), (uint32_t)((k / RF) & 1), WAIT_NS) ? 1 : 0) != 0;
            if (!pre_ok) break;
            g_waited = k + 1;
            float x[32];
#pragma unroll
            for (int t = 0; t < 32; ++t) x[t] = 0.f;
            for (int sl = 0; sl < S; ++sl) {
                const unsigned char* pc = sm + (uint32_t)(g * per_round + half * S + sl) * PIECE;
                if (tr) {
#pragma unroll
                    for (int t = 0; t < 32; ++t) x[t] += reinterpret_cast<const float*>(pc)[t * M + row];
                } else {
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const float4 y = *reinterpret_cast<const float4*>(pc + row * 128 + ((c ^ (row & 7)) << 4));
                        x[4 * c] += y.x; x[4 * c + 1] += y.y; x[4 * c + 2] += y.z; x[4 * c + 3] += y.w;
                    }
                }
            }
            uint32_t v[32];
#pragma unroll
            for (int t = 0; t < 32; ++t) {
                ss = fmaf(x[t], x[t], ss);
                v[t] = __float_as_uint(x[t]);
            }
            tmem_st32(lane_base + COL_X + half * hc + 32 * k, v);
            __syncthreads();                       // round k's buffers are read
            if (tid == 0 && k + RF < rounds) {
                fence_proxy_async_smem();
                issue_round(k + RF);
                g_issued = k + RF + 1;
            }
        }
    } else {
    for (int h = 0; h < hc / 32; h += 2) {
        // two 32-column pieces in flight at once
        float x0[32], x1[32];
        load32(c0 + half * hc + h * 32, x0);
        load32(c0 + half * hc + h * 32 + 32, x1);
        uint32_t v[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) {
            ss = fmaf(x0[t], x0[t], ss);
            v[t] = __float_as_uint(x0[t]);
        }
        tmem_st32(lane_base + COL_X + half * hc + h * 32, v);
#pragma unroll
        for (int t = 0; t < 32; ++t) {
            ss = fmaf(x1[t], x1[t], ss);
            v[t] = __float_as_uint(x1[t]);
        }
        tmem_st32(lane_base + COL_X + half * hc + h * 32 + 32, v);
    }
    }
    tmem_wait_st();
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    if (tid == 0) {
        float part = 0.f;
        for (int w = 0; w < NTHREADS / 32; ++w) part += red[w];
        for (int r = 0; r < cs; ++r) {
            st_cluster_f32(mapa_shared(smem_u32(&norm_part[rank]), (uint32_t)r), part);
            mbar_arrive_cluster(mapa_shared(bar_a, (uint32_t)r));
        }
    }
    bool ok = __syncthreads_and(mbar_wait_cluster(bar_a, 0, WAIT_NS) ? 1 : 0) != 0 && pre_ok;
    float tot = 0.f;
    for (int r = 0; r < cs; ++r) tot += norm_part[r];
    const float inv = 1.0f / (sqrtf(tot) + 1e-7f);
    for (int h = 0; h < hc / 32; h += 2) {
        uint32_t v[2][32];
        tmem_ld32(lane_base + COL_X + half * hc + h * 32, v[0]);
        tmem_ld32(lane_base + COL_X + half * hc + h * 32 + 32, v[1]);
        tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int j0 = half * hc + (h + u) * 32;       // within this CTA's columns
            tmem_pin(v[u]);
            float xv[32];
#pragma unroll
            for (int t = 0; t < 32; ++t) {
                xv[t] = __uint_as_float(v[u][t]) * inv;
                v[u][t] = __float_as_uint(xv[t]);
            }
            tmem_st32(lane_base + COL_X + j0, v[u]);
#pragma unroll
            for (int c = 0; c < 4; ++c)
                *reinterpret_cast<uint4*>(sm + OFF_X + atom_off(row, c0 + j0 + 8 * c)) = pack8(xv + 8 * c);
        }
    }
    tmem_wait_st();
    const uint32_t XBLOCK_BYTES = (uint32_t)(cb / 64) * ATOM;
    // The columns of each half (hc of them, whole atoms) go out to the other
    // CTAs as soon as that half's 128 threads have written them: a barrier of
    // the half, then one bulk copy per other CTA from the half's first thread.
    auto send_half = [&](bool send) {
        fence_proxy_async_smem();
        asm volatile("bar.sync %0, 128;" ::"r"(1 + half) : "memory");
        if (send && (warp & 3) == 0 && lane == 0) {
            const uint32_t src = base + OFF_X + (uint32_t)((c0 + half * hc) / 64) * ATOM;
            for (int r = 0; r < cs; ++r)
                if (r != (int)rank)
                    bulk_copy_to_cluster(mapa_shared(src, (uint32_t)r), src, XBLOCK_BYTES / 2,
                                         mapa_shared(barx((int)rank), (uint32_t)r));
        }
    };
    send_half(ok && cs > 1);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // The bytes from CTA r are counted on barx(r): send n (n = 0 at set-up,
    // then after iteration n-1) is consumed by the A GEMM of iteration n, with
    // parity n & 1. Thread 0 sets up the count of each incoming send.
    int sends = 0;                 // sends expected (thread 0's count)
    bool w_issued = false;         // the fused update's copies of W's tile were started
    int waited[MAXCS] = {0, 0, 0, 0};
    auto expect_columns = [&]() {
        if (tid == 0) {
            for (int r = 0; r < cs; ++r)
                if (r != (int)rank) mbar_expect_tx(barx(r), XBLOCK_BYTES);
            ++sends;
        }
    };
    expect_columns();

    uint32_t phase = 0;
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
    // "My A GEMM is done with Xb": thread 0 (which saw the MMA complete)
    // arrives on the barrier of every CTA of the cluster.
    // (Relaxed: the A GEMM's reads of Xb have completed, as the MMA barrier
    // showed; nothing written by this thread needs ordering before the
    // other CTAs overwrite Xb.)
    auto arrive_a_done = [&]() {
        if (tid == 0)
            for (int r = 0; r < cs; ++r)
                asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];"
                             ::"r"(mapa_shared(bar_a, (uint32_t)r)) : "memory");
    };
    // Bounded wait on a local cluster barrier, made block-uniform.
    auto cluster_wait = [&](uint32_t b, uint32_t parity) -> bool {
        return __syncthreads_and(mbar_wait_cluster(b, parity, WAIT_NS) ? 1 : 0) != 0;
    };
    const uint32_t i_xx = idesc_bf16_f32(M, M, 0, 0);
    const uint32_t i_aa = idesc_bf16_f32(M, M, 0, 1);
    const uint32_t i_bx = idesc_bf16_f32(M, cb, 0, 1);
    const uint64_t dX = sdesc_sw128(base + OFF_X, 16, 1024);      // Xb K-major
    const uint64_t dXmn = sdesc_sw128(base + OFF_X, ATOM, 1024);  // Xb MN-major
    const uint64_t dA = sdesc_sw128(base + OFF_A, 16, 1024);      // Ab K-major
    const uint64_t dAmn = sdesc_sw128(base + OFF_A, ATOM, 1024);  // Ab MN-major
    const uint64_t dB = sdesc_sw128(base + OFF_B, 16, 1024);      // Bb K-major
    for (int it = 0; it < a.steps; ++it) {
        // A = Xb Xb^T: own columns first, then each other CTA's as they land
        if (ok && tid == 0) {
            int issued = 0;
            auto issue_block = [&](int blk) {
                for (int j = blk * (cb / 16); j < (blk + 1) * (cb / 16); ++j) {
                    const uint64_t ko = (uint64_t)((j >> 2) * ATOM + (j & 3) * 32) >> 4;
                    mma_bf16(tmem + COL_A, dX + ko, dX + ko, i_xx, issued++ > 0 ? 1u : 0u);
                }
            };
            issue_block((int)rank);
            for (int r = 0; r < cs; ++r) {
                if (r == (int)rank) continue;
                if (!mbar_wait_cluster(barx(r), (uint32_t)(it & 1), WAIT_NS)) { fail_sh = 1; break; }
                ++waited[r];
                tc_fence_after();
                issue_block(r);
            }
            mma_commit(bar);
        }
        if (ok && !mma_done()) ok = false;
        if (fail_sh) ok = false;   // read after mma_done's barrier: the same in every thread
        // this CTA's last read of the other CTAs' columns of Xb in the iteration is over
        arrive_a_done();
        if (ok) {
            // Ab = bf16(A)
            {
                uint32_t v0[32], v1[32];
                tmem_ld32(lane_base + COL_A + half * 64, v0);
                tmem_ld32(lane_base + COL_A + half * 64 + 32, v1);
                tmem_wait_ld();
                tmem_pin(v0);
                tmem_pin(v1);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    float x[8];
#pragma unroll
                    for (int t = 0; t < 8; ++t) x[t] = __uint_as_float(c < 4 ? v0[8 * c + t] : v1[8 * (c - 4) + t]);
                    *reinterpret_cast<uint4*>(sm + OFF_A + atom_off(row, half * 64 + 8 * c)) = pack8(x);
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
            if (!mma_done()) ok = false;
        }
        if (ok) {
            // Bb = bf16(b A + c AA)
            uint32_t va[2][32], vaa[2][32];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                tmem_ld32(lane_base + COL_A + half * 64 + h * 32, va[h]);
                tmem_ld32(lane_base + COL_AA + half * 64 + h * 32, vaa[h]);
            }
            tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int j0 = half * 64 + h * 32;
                tmem_pin(va[h]);
                tmem_pin(vaa[h]);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float bv[8];
#pragma unroll
                    for (int t = 0; t < 8; ++t)
                        bv[t] = fmaf(a.c, __uint_as_float(vaa[h][8 * c + t]), a.b * __uint_as_float(va[h][8 * c + t]));
                    *reinterpret_cast<uint4*>(sm + OFF_B + atom_off(row, j0 + 8 * c)) = pack8(bv);
                }
            }
            sync_smem();
            // BX_j = Bb Xb[:, c0 : c0 + cb] (over the dead A and AA)
            if (tid == 0) {
                const uint64_t xo = (uint64_t)((c0 / 64) * ATOM) >> 4;
#pragma unroll
                for (int j = 0; j < M / 16; ++j) {
                    const uint64_t ko = (uint64_t)((j >> 2) * ATOM + (j & 3) * 32) >> 4;
                    mma_bf16(tmem + COL_BX, dB + ko, dXmn + xo + j * 128, i_bx, j > 0 ? 1u : 0u);
                }
                mma_commit(bar);
                if (a.fuse && it + 1 == a.steps) mbar_expect_tx(smem_u32(&sync_w), (uint32_t)(cb * M * 4));
            }
            if (!mma_done()) ok = false;
        }
        // no CTA still reads Xb with its A GEMM
        if (!cluster_wait(bar_a, (it + 1) & 1)) ok = false;
        // fused update, last iteration: every CTA's A GEMM is over (so the bulk
        // copies out of this Xb have landed) and the BX GEMM has read it, so
        // the CTA's tile of W comes into that space while X gets its last update
        if (ok && a.fuse && it + 1 == a.steps) {
            w_issued = true;
            const float* Wp = a.W[which] + (size_t)bh * a.d * a.dh;
            if (tr) {
                if (tid < 8)
                    bulk_load_g2s(base + OFF_S32 + tid * (cb * M * 4 / 8), Wp + (size_t)c0 * cols + tid * (cb * M / 8),
                                  (uint32_t)(cb * M * 4 / 8), smem_u32(&sync_w));
            } else if (tid < M) {
                bulk_load_g2s(base + OFF_S32 + tid * S32_ROW, Wp + (size_t)tid * cols + c0, (uint32_t)(cb * 4),
                              smem_u32(&sync_w));
            }
        }
        if (ok) {
            // X_j = a X_j + BX_j in TMEM; bf16(X_j) into this CTA's block of Xb
            for (int h = 0; h < hc / 32; h += 2) {
                // two 32-column pieces per TMEM round trip
                uint32_t vx[2][32], vb[2][32];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    tmem_ld32(lane_base + COL_X + half * hc + (h + u) * 32, vx[u]);
                    tmem_ld32(lane_base + COL_BX + half * hc + (h + u) * 32, vb[u]);
                }
                tmem_wait_ld();
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    tmem_pin(vx[u]);
                    tmem_pin(vb[u]);
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int j0 = half * hc + (h + u) * 32;
                    float xn[32];
#pragma unroll
                    for (int t = 0; t < 32; ++t) {
                        xn[t] = fmaf(a.a, __uint_as_float(vx[u][t]), __uint_as_float(vb[u][t]));
                        vx[u][t] = __float_as_uint(xn[t]);
                    }
                    tmem_st32(lane_base + COL_X + j0, vx[u]);
                    if (a.fuse && it + 1 == a.steps) continue;   // Xb holds W's tile now
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<uint4*>(sm + OFF_X + atom_off(row, c0 + j0 + 8 * c)) = pack8(xn + 8 * c);
                }
            }
            // (after the last iteration each CTA writes back only its own columns)
            send_half(cs > 1 && it + 1 < a.steps);
            tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (it + 1 < a.steps) expect_columns();
    }
    if (!ok) {
        if (tid == 0) atomicOr(a.status, ST_TIMEOUT);
    } else if (!a.fuse) {
        // this CTA's columns back into G's own orientation
        for (int h = 0; h < hc / 32; ++h) {
            const int j0 = half * hc + h * 32;
            uint32_t v[32];
            tmem_ld32(lane_base + COL_X + j0, v);
            tmem_wait_ld();
            tmem_pin(v);
            if (tr) {
#pragma unroll
                for (int t = 0; t < 32; ++t) G[(size_t)(c0 + j0 + t) * cols + row] = __uint_as_float(v[t]);
            } else {
                float* gr = G + (size_t)row * cols + c0 + j0;
#pragma unroll
                for (int t = 0; t < 32; t += 4)
                    *reinterpret_cast<float4*>(gr + t) = make_float4(__uint_as_float(v[t]), __uint_as_float(v[t + 1]),
                                                                    __uint_as_float(v[t + 2]), __uint_as_float(v[t + 3]));
            }
        }
    } else {
        ok = fused_update(a, which, bh, tr, cols, cs, rank, c0, cb, half, row, lane_base, sm, base, upart,
                          smem_u32(&sync_u), smem_u32(&sync_w));
        if (!ok && tid == 0) atomicOr(a.status, ST_TIMEOUT);
    }
    // every MMA has completed once this commit lands (bounded drain); after
    // an early exit from the loop, columns still on their way in are waited
    // for (bounded) before the CTA may leave
    if (tid == 0) {
        if (w_issued) mbar_wait(smem_u32(&sync_w), 0, WAIT_NS);   // W's tile copies have landed
        for (int k = g_waited; k < g_issued; ++k) mbar_wait(smem_u32(&gbar[k % RF]), (uint32_t)((k / RF) & 1), WAIT_NS);
        mma_commit(bar);
        mbar_wait(bar, phase & 1, WAIT_NS);
        for (int r = 0; r < cs; ++r)
            if (r != (int)rank)
                for (int n = waited[r]; n < sends; ++n) mbar_wait_cluster(barx(r), (uint32_t)(n & 1), WAIT_NS);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    // no CTA leaves while another may still write into its shared memory
    cluster_sync_all();
}

}  // namespace

bool ns_tc_supported(const lact_state* st) {
    const int m = st->cfg.d < st->cfg.dh ? st->cfg.d : st->cfg.dh;
    const int n = st->cfg.d < st->cfg.dh ? st->cfg.dh : st->cfg.d;
    return st->cfg.io_dtype == LACT_BF16 && m == M && n <= NMAX && n % 128 == 0;
}

cudaError_t launch_ns_tc(const lact_state* st, void* const g[3], int slots, bool fuse_update, cudaStream_t s) {
    NsArgs a;
    for (int m = 0; m < 3; ++m) {
        a.g[m] = static_cast<float*>(g[m]);
        a.W[m] = static_cast<float*>(st->W[m]);
        a.S[m] = st->Wsh[m];
    }
    if (slots < 0 || slots > kNsFusedSlots) return cudaErrorInvalidValue;   // the piece ring holds a round of 4
    a.fuse = fuse_update ? 1 : 0;
    a.scale = (float)-st->cfg.muon_lr;
    a.part = static_cast<const float*>(st->partial);
    a.slots = slots;
    a.mat = (size_t)st->BH * st->cfg.d * st->cfg.dh;
    a.nmat = st->nmat;
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
    const int cs = a.n / ns_block(a.n);
    // the partial slots as rows of n fp32 (each matrix of each slot: 128 rows)
    CUtensorMap tm_p;
    {
        const uint64_t dims[2] = {(uint64_t)a.n, (uint64_t)kMaxSlots * st->nmat * st->BH * M};
        const uint64_t str[1] = {(uint64_t)a.n * 4};
        const uint32_t box[2] = {32, M};
        if (!make_tmap_2d(&tm_p, st->partial, true, dims, str, box)) return cudaErrorInvalidValue;
    }
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)(cs * st->nmat * st->BH));
    lc.blockDim = dim3(NTHREADS);
    lc.dynamicSmemBytes = SMEM_BYTES;
    lc.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)cs;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see pdl_wait()
    at[1].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = at;
    lc.numAttrs = 2;
    e = cudaLaunchKernelEx(&lc, k_ns_tc, tm_p, a);
    g_launches++;
    g_tc_launches++;
    return e == cudaSuccess ? cudaGetLastError() : e;
}

}  // namespace lact

