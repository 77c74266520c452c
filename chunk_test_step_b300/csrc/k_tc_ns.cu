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
// same bit for bit).
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
constexpr uint32_t SMEM_BYTES = OFF_B + 2 * ATOM + 1024;
// TMEM: the CTA's fp32 columns of X at 0 (cb columns); from cb on, A (128)
// and AA (128), later overwritten by BX (cb).
constexpr uint32_t COL_X = 0;

// Columns of X per CTA for a long side n.
__host__ __device__ constexpr int ns_block(int n) { return n % 256 == 0 ? 256 : 128; }
constexpr uint64_t WAIT_NS = 2000000000ull;

struct NsArgs {
    float* g[3];      // gradients in place: W1 [BH,dh,d], W2 [BH,d,dh], W3 [BH,dh,d]
    const float* part;    // split-K partial slots [slots][nmat][BH][d*dh] (read when slots > 0)
    int slots;
    size_t mat;           // BH * d * dh
    int nmat;
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
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(16) unsigned char smraw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t mbar, sync_a, sync_x[MAXCS];
    __shared__ int fail_sh;
    __shared__ uint32_t tmem_slot;
    __shared__ float red[NTHREADS / 32];
    __shared__ float norm_part[MAXCS];   // partial sums of squares, one per CTA of the cluster

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
    bool ok = __syncthreads_and(mbar_wait_cluster(bar_a, 0, WAIT_NS) ? 1 : 0) != 0;
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
            }
            if (!mma_done()) ok = false;
        }
        // no CTA still reads Xb with its A GEMM
        if (!cluster_wait(bar_a, (it + 1) & 1)) ok = false;
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
    } else {
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
    }
    // every MMA has completed once this commit lands (bounded drain); after
    // an early exit from the loop, columns still on their way in are waited
    // for (bounded) before the CTA may leave
    if (tid == 0) {
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

cudaError_t launch_ns_tc(const lact_state* st, void* const g[3], int slots, cudaStream_t s) {
    NsArgs a;
    for (int m = 0; m < 3; ++m) a.g[m] = static_cast<float*>(g[m]);
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
    e = cudaLaunchKernelEx(&lc, k_ns_tc, a);
    g_launches++;
    g_tc_launches++;
    return e == cudaSuccess ? cudaGetLastError() : e;
}

}  // namespace lact
