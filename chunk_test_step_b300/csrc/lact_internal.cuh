// Internal declarations of liblact: state, workspace layout, kernel entry
// points and small device helpers. Not part of the public C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <atomic>
#include <vector>

#include "../../include/lact.h"

namespace lact {

typedef __nv_bfloat16 bf16;

// Sticky device status bits (workspace word 0).
enum : int { ST_NONFINITE = 1, ST_TIMEOUT = 2 };

// Device workspace, carved by ws_layout() in 256-byte aligned sections.
// "real" is the state's internal type: fp32 for bf16 io, fp64 for fp32 io.
struct WsLayout {
    size_t W[3];       // real master fast weights: W1 [BH,dh,d], W2 [BH,d,dh], W3 [BH,dh,d]
    size_t Wsh[3];     // bf16 shadows of the same, same layouts (bf16 io only)
    size_t dW[3];      // real chunk gradients (Muon: overwritten by NS output), same layouts
    size_t partial;    // real split-K partials [kMaxSlots][3][BH][dh*d]
    size_t ns[4];      // real Newton-Schulz scratch: X, X', A, B over 3*BH matrices
    size_t inter;      // bf16 per-token dh1, dh3, u' of one token slice [3][BH][slice_cap][dh] (two-kernel gradient)
    size_t mom[3];     // real momentum velocities, same layouts as W (momentum only)
    size_t status;     // int32[64]: [0] sticky status bits, [1..] diagnostics
    size_t total;
};

constexpr int kMaxSlots = 64;   // split-K partial slots
constexpr int64_t kSliceCap = 4096;   // tokens per slice of the two-kernel gradient (its intermediates stay in L2)

// Tokens per slice of the two-kernel gradient for this configuration (0 if unused).
int64_t slice_cap(const lact_config& c);

WsLayout ws_layout(const lact_config& c);

struct PhaseEvents { cudaEvent_t a, b; int phase; int launches; int tensor_launches; };

}  // namespace lact

struct lact_state {
    lact_config cfg;
    int BH;
    int nmat;                 // fast-weight matrices: 3 (SwiGLU: W1, W2, W3) or 1 (linear: W1 = W, d x d)
    bool f64;                 // internal arithmetic in fp64 (fp32 io) or fp32 (bf16 io)
    size_t rsize;             // bytes of one internal real
    char* ws;
    size_t ws_bytes;
    lact::WsLayout L;
    void* W[3];
    lact::bf16* Wsh[3];
    void* dW[3];
    void* partial;
    void* ns[4];
    lact::bf16* inter;
    void* mom[3];             // momentum velocities (nullptr unless the rule is momentum)
    int64_t slice_cap;
    int* status;
    cudaStream_t last_stream;
    cudaStream_t side;        // causal order: each chunk's readout runs here, beside its gradient
    cudaEvent_t ev_fork, ev_join;
    bool profiling;
    std::vector<lact::PhaseEvents> pending;
    std::vector<cudaEvent_t> event_pool;
    lact_profile prof;
    int num_sms;
};

namespace lact {

extern std::atomic<int64_t> g_launches;      // every kernel launch of this library
extern std::atomic<int64_t> g_tc_launches;   // launches of tcgen05 tensor-core kernels

// ------------------------------------------- programmatic dependent launch
// Every kernel of the library is launched with programmatic stream
// serialization, so the GPU may start launching it before the kernel ahead
// of it in the stream has finished. Each kernel calls pdl_wait() before it
// touches global memory: griddepcontrol.wait blocks until the previous kernel
// has completed and its writes are visible, so no kernel reads data early;
// what overlaps is the launch and the CTAs' arrival on the SMs.
// The tensor-core kernels also call pdl_trigger() at once, which lets the
// next kernel launch as soon as every CTA of theirs is running: its CTAs then
// wait in place of an SM that would otherwise idle in the last wave. The
// CUDA-core kernels leave the trigger to their exit, so that waiting CTAs
// never share an SM with their arithmetic.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = grid;
    lc.blockDim = block;
    lc.dynamicSmemBytes = smem;
    lc.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = at;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, kern, static_cast<Args&&>(args)...);
}

// ---------------------------------------------------------------- helpers
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }

// Load an io element widened to the internal real type R.
template <typename R> __device__ __forceinline__ R ld_io(const float* p, int64_t i) { return (R)p[i]; }
template <typename R> __device__ __forceinline__ R ld_io(const bf16* p, int64_t i) { return (R)__bfloat162float(p[i]); }
// Store a real as an io element (round to nearest even).
__device__ __forceinline__ void st_io(float* p, int64_t i, float x) { p[i] = x; }
__device__ __forceinline__ void st_io(float* p, int64_t i, double x) { p[i] = (float)x; }
__device__ __forceinline__ void st_io(bf16* p, int64_t i, float x) { p[i] = __float2bfloat16_rn(x); }

// Round to the nearest bf16 value (8 significant bits, ties to even), kept
// in the same type. The fp64 form rounds the fp64 value directly (no
// intermediate fp32 rounding).
__device__ __forceinline__ float round_bf16(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }
__device__ __forceinline__ double round_bf16(double x) {
    unsigned long long b = (unsigned long long)__double_as_longlong(x);
    const unsigned long long drop = 45;                 // 52 - 7 fraction bits
    const unsigned long long lsb = (b >> drop) & 1ull;
    b += (1ull << (drop - 1)) - 1ull + lsb;
    b &= ~((1ull << drop) - 1ull);
    return __longlong_as_double((long long)b);
}

__device__ __forceinline__ float fma_r(float a, float b, float c) { return fmaf(a, b, c); }
__device__ __forceinline__ double fma_r(double a, double b, double c) { return fma(a, b, c); }
__device__ __forceinline__ float exp_r(float x) { return expf(x); }
__device__ __forceinline__ double exp_r(double x) { return exp(x); }
__device__ __forceinline__ float sqrt_r(float x) { return sqrtf(x); }
__device__ __forceinline__ double sqrt_r(double x) { return sqrt(x); }

// Token-slice view of a [BH, n_total, d] tensor: tokens [t0, t0 + n) of each head.
struct TokView {
    const void* p;      // base of the whole tensor
    int64_t n_total;    // tokens per head in the tensor
    int64_t t0;         // first token of the slice
    int64_t n;          // tokens in the slice
};

// ---------------------------------------------------------------- launchers
// SIMT path (fp32 or bf16 io, any supported d, dh). Each returns a CUDA error.
cudaError_t launch_apply_simt(const lact_state* st, TokView q, void* o, cudaStream_t s);
cudaError_t launch_grad_simt(const lact_state* st, TokView k, TokView v, const float* eta,
                             int* slots_used, cudaStream_t s);
// TMA tensor maps (bf16, 128-byte swizzle); dims / strides innermost first.
bool tmap_available();
bool make_tmap_bf16(CUtensorMap* m, const void* p, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                    const uint32_t* box);
bool make_tmap_2d(CUtensorMap* m, const void* p, bool f32, const uint64_t* dims, const uint64_t* strides_bytes,
                  const uint32_t* box);

// Tensor-core (tcgen05) path: bf16 io, d = 128, dh a multiple of 64.
bool grad_tc_supported(const lact_state* st);
cudaError_t launch_grad_tc(const lact_state* st, TokView k, TokView v, const float* eta, int* slots_used,
                           double side_tiles, cudaStream_t s);
bool ns_tc_supported(const lact_state* st);
// Newton-Schulz on the gradient in g[]. With slots > 0 the gradient is not in
// g[] yet: the kernel adds the split-K partial slots 0 .. slots-1 (in that
// order, as launch_reduce does) while it reads them. Without fuse_update the
// result overwrites g[]; with it, the Muon step and row renorm are applied to
// the state's W (and bf16 shadow) from the result, and g[] is left as it was.
cudaError_t launch_ns_tc(const lact_state* st, void* const g[3], int slots, bool fuse_update, cudaStream_t s);
// Most split-K slots Newton-Schulz adds up itself (more go through launch_reduce).
constexpr int kNsFusedSlots = 4;
bool apply_tc_supported(const lact_state* st);
cudaError_t launch_apply_tc(const lact_state* st, TokView q, void* o, cudaStream_t s);
// Head dim 128: two 128-query tiles per CTA sharing every streamed weight block.
cudaError_t launch_apply2_tc(const lact_state* st, TokView q, void* o, cudaStream_t s);
// Two-kernel chunk gradient (bf16 io, head dim 256): per-token dh1, dh3, u'
// of a token slice, then the three weight-gradient GEMMs over the slice.
bool fwdbwd_tc_supported(const lact_state* st);
// Linear memory: readout (tensor cores at bf16 d = 128, else CUDA cores) and
// the chunk gradient's partial sums into st->partial (one per token split).
bool lin_tc_supported(const lact_state* st);
cudaError_t launch_lin_apply(const lact_state* st, TokView q, void* o, cudaStream_t s);
cudaError_t launch_lin_grad_simt(const lact_state* st, TokView k, TokView v, const float* eta, int* slots,
                                 cudaStream_t s);
cudaError_t launch_lin_grad_tc(const lact_state* st, TokView k, TokView v, const float* eta, int* slots,
                               cudaStream_t s);
cudaError_t launch_fwdbwd_tc(const lact_state* st, TokView k, TokView v, const float* eta, bf16* inter,
                             int64_t slice_cap, cudaStream_t s);
cudaError_t launch_wgrad_tc(const lact_state* st, TokView k, TokView v, const bf16* inter, int64_t slice_cap,
                            bool accumulate, void* const out[3], cudaStream_t s);
cudaError_t launch_reduce(const lact_state* st, int slots, bool accumulate, void* const out[3],
                          cudaStream_t s);
cudaError_t launch_newton_schulz(const lact_state* st, void* const g[3], cudaStream_t s);
// W <- renorm(W + scale D) per row, D = g, or with velocities (mom != nullptr)
// M <- beta M + g and D = M.
cudaError_t launch_update(const lact_state* st, const void* const g[3], double scale, void* const mom[3],
                          double beta, cudaStream_t s);
cudaError_t launch_shadow(const lact_state* st, cudaStream_t s);
// Raw-pointer forms of the bf16-io SIMT gradient and its reduction (no state).
cudaError_t launch_grad_simt_bf16_raw(int d, int dh, int BH, const float* W1, const float* W2, const float* W3,
                                      TokView k, TokView v, const float* eta, float* partial, int max_slots,
                                      int num_sms, int* slots, cudaStream_t s);
cudaError_t launch_reduce_f32_raw(const float* partial, int slots, size_t mat, float* o0, float* o1, float* o2,
                                  int num_sms, cudaStream_t s);
// One thread waits (bounded) on an mbarrier nobody arrives on; sets ST_TIMEOUT.
cudaError_t launch_wait_selftest(int* status, uint64_t budget_ns, cudaStream_t s);
// Element conversion between the API's fp32 buffers and internal reals.
cudaError_t launch_convert(const void* src, bool src_f64, void* dst, bool dst_f64, size_t n, int num_sms,
                           cudaStream_t s);

}  // namespace lact
