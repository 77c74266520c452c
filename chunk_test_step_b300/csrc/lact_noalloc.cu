// lact_chunk_gradient_noalloc: the chunk gradient for callers that cannot
// allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is off limits - inside a
// host callback or a custom allocator's own hooks, in a process whose memory
// pool is owned by another framework that forbids side allocations, or on a
// path that must not risk an out-of-memory failure or an implicit device
// synchronisation half-way through. Such a caller can still name its inputs
// and outputs but cannot size and hand over the workspace that lact_init_state
// needs.
//
// What it does instead: the split-K partial sums of the gradient live in
// g_scratch below, a file-scope device array of kScratchBytes (32 MiB) that
// every GPU which loads this library keeps until the process exits. The call
// runs the same CUDA-core gradient kernel and fixed-order reduction as the
// workspace path, with the weights read straight from the caller's buffers.
#include "lact_internal.cuh"

#include <mutex>

namespace lact {
namespace {

constexpr size_t kScratchBytes = 32u << 20;
constexpr int kMaxDevices = 64;

// Split-K partial sums of the no-allocation gradient. Every slot the kernel
// uses is overwritten in full before it is read, so nothing here needs to be
// cleared between calls; the contents of the last call stay behind.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};   // device address of g_scratch, per device
int g_num_sms[kMaxDevices] = {};

// Device address of g_scratch on the current device (host code may not use
// g_scratch's name as a device pointer), looked up once per device by the
// first call made with that device current, and kept. When CUDA loads
// modules lazily that first lookup also loads this file's module, array
// included, which allocates: hence the warm-up call the header asks for. The
// kept address belongs to the device's current context: after
// cudaDeviceReset the library must not be used again in the process.
lact_status scratch_for_current_device(float** out, int* num_sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LACT_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return LACT_ERR_CUDA;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return LACT_ERR_CUDA;
        g_scratch_addr[dev] = p;
        g_num_sms[dev] = sms;
    }
    *out = static_cast<float*>(g_scratch_addr[dev]);
    *num_sms = g_num_sms[dev];
    return LACT_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace
}  // namespace lact

using namespace lact;

extern "C" lact_status lact_chunk_gradient_noalloc(const lact_config* cfg, const float* d_W1, const float* d_W2,
                                                   const float* d_W3, const void* d_k, const void* d_v,
                                                   const float* d_eta, int64_t n_tok, float* d_dW1, float* d_dW2,
                                                   float* d_dW3, cudaStream_t stream) {
    if (!cfg || cfg->B < 1 || cfg->H < 1 || (int64_t)cfg->B * cfg->H > 65535) return LACT_ERR_INVALID_ARG;
    if (!(cfg->d == 32 || cfg->d == 64 || cfg->d == 128 || cfg->d == 256)) return LACT_ERR_INVALID_ARG;
    if (cfg->dh < 64 || cfg->dh > 1024 || cfg->dh % 64 != 0) return LACT_ERR_INVALID_ARG;
    if (cfg->io_dtype != LACT_BF16) return LACT_ERR_UNSUPPORTED;
    if (cfg->memory != LACT_MEM_SWIGLU) return LACT_ERR_UNSUPPORTED;   // SwiGLU memory only
    if (n_tok < 0) return LACT_ERR_INVALID_ARG;
    const void* ptrs[] = {d_W1, d_W2, d_W3, d_dW1, d_dW2, d_dW3};
    for (const void* p : ptrs)
        if (!p || !aligned16(p)) return LACT_ERR_INVALID_ARG;
    if (n_tok > 0 && (!d_k || !d_v || !d_eta || !aligned16(d_k) || !aligned16(d_v) || !aligned16(d_eta)))
        return LACT_ERR_INVALID_ARG;
    const int BH = cfg->B * cfg->H;
    const size_t mat = (size_t)BH * cfg->d * cfg->dh;
    const size_t slot_bytes = 3 * mat * sizeof(float);
    // One split-K slot must fit in the static scratch.
    if (slot_bytes > kScratchBytes) return LACT_ERR_UNSUPPORTED;
    int max_slots = (int)(kScratchBytes / slot_bytes);
    if (max_slots > kMaxSlots) max_slots = kMaxSlots;

    float* scratch = nullptr;
    int num_sms = 0;
    lact_status r = scratch_for_current_device(&scratch, &num_sms);
    if (r != LACT_OK) return r;

    int slots = 0;
    if (n_tok > 0) {
        TokView k{d_k, n_tok, 0, n_tok}, v{d_v, n_tok, 0, n_tok};
        if (launch_grad_simt_bf16_raw(cfg->d, cfg->dh, BH, d_W1, d_W2, d_W3, k, v, d_eta, scratch, max_slots,
                                      num_sms, &slots, stream) != cudaSuccess)
            return LACT_ERR_CUDA;
    }
    // slots == 0 (no tokens) writes zeros
    if (launch_reduce_f32_raw(scratch, slots, mat, d_dW1, d_dW2, d_dW3, num_sms, stream) != cudaSuccess)
        return LACT_ERR_CUDA;
    return LACT_OK;
}
