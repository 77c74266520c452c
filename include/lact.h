/*
 * lact.h - C ABI of the LaCT fast-weight chunk step on sm_103a (B300).
 *
 * The operation (per batch entry b and head h):
 *
 *   fast weights  W1, W3 : [dh, d]   W2 : [d, dh]     (fp32 master copy)
 *   readout       f_W(x) = W2 (silu(W1 x) * (W3 x))
 *   chunk loss    L = - sum_i eta_i <f_W(k_i), v_i>
 *   update        GD:   W <- W - dL/dW
 *                 Muon: W <- W - lr * NS5(dL/dW)   (per matrix)
 *   renorm        each row of W1, W2, W3 rescaled to its pre-update L2 norm
 *
 * Sources: "Test-Time Training Done Right" (arXiv 2505.23884), abstract
 * (fast weights adapted at inference, chunks of 2K to ~1M tokens, Muon);
 * the LaCT review page, sections "Fast weights are temporary context memory"
 * (queries read a small network's weights), "Local attention and nonlinear
 * memory work together" (SwiGLU memory, negative inner-product loss,
 * token-specific learning rates, GD / momentum / Muon with Newton-Schulz,
 * L2-normalised fast weights) and "Update order must respect the task"
 * (apply-then-update for causal chunks, update-then-apply for sets).
 *
 * Conventions for every call:
 *  - Pointers prefixed d_ are device pointers; the caller owns every buffer,
 *    including the workspace. The library never allocates device memory.
 *  - Tensors are dense, row-major, with the layouts given per argument.
 *    q, k, v, o are [B, H, n, d] in the state's io dtype (fp32 or bf16);
 *    eta is [B, H, n] fp32. Every device pointer must be 16-byte aligned.
 *  - Calls are asynchronous on the given stream. Shape or argument errors are
 *    returned at once and nothing is enqueued. Problems found on the device
 *    (non-finite row norms, a bounded wait that ran out) set a sticky status
 *    word that lact_sync_status() reads.
 *  - No exception or process exit crosses this interface.
 *  - A state must not be used from two host threads at once.
 *  - The compute calls (lact_chunk_apply, lact_chunk_update, lact_sequence,
 *    lact_chunk_gradient, lact_apply_gradient, lact_set_weights) enqueue only
 *    kernels, copies, event records and stream waits, so with profiling off
 *    they may be recorded by stream capture into a CUDA graph; a replay repeats the recorded work on
 *    the same buffers (the state's weights move on with each replay) and gives
 *    the same results as the direct call. Kernels are launched with
 *    programmatic stream serialization and wait for the kernel ahead of them
 *    before touching memory.
 */
#ifndef LACT_H
#define LACT_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LACT_OK = 0,
    LACT_ERR_INVALID_ARG = 1,   /* bad pointer, size, alignment or shape */
    LACT_ERR_UNSUPPORTED = 2,   /* valid request this build does not serve */
    LACT_ERR_CUDA = 3,          /* a CUDA runtime call failed */
    LACT_ERR_TIMEOUT = 4,       /* a bounded device-side wait gave up */
    LACT_ERR_NONFINITE = 5      /* a renormalised row had a non-finite norm */
} lact_status;

typedef enum { LACT_F32 = 0, LACT_BF16 = 1 } lact_dtype;
/* Update rules (review page, "Local attention and nonlinear memory work
 * together": gradient descent, momentum and Muon are the rules compared). */
typedef enum { LACT_OPT_GD = 0, LACT_OPT_MUON = 1, LACT_OPT_MOMENTUM = 2 } lact_opt;
typedef enum { LACT_CAUSAL_APPLY_THEN_UPDATE = 0, LACT_SET_UPDATE_THEN_APPLY = 1 } lact_order;
/* Fast-weight memory (review page, "Local attention and nonlinear memory work
 * together" and Fig. 8): the three-matrix SwiGLU MLP, or one linear d x d
 * matrix W read as o = W q, whose chunk gradient is -sum_i eta_i v_i k_i^T.
 * The linear memory needs dh == d and lives in the W1 slot ([.., d, d]); every
 * W2 / W3 / dW2 / dW3 argument is then unused and may be NULL. It is served
 * for fp32 io at d = 32, 64, 128 and bf16 io at d = 128. */
typedef enum { LACT_MEM_SWIGLU = 0, LACT_MEM_LINEAR = 1 } lact_memory;

typedef struct {
    int B, H;           /* batch entries and heads; every (b, h) has its own W */
    int d, dh;          /* head dim: 32, 64, 128 or 256; hidden: 64..1024, a multiple of 64 */
    lact_dtype io_dtype;/* dtype of q, k, v, o. Fast weights are held in fp32 for bf16 io and in
                           fp64 for fp32 io (the fp32 path is the accuracy path: its Muon step
                           with bf16 operand rounding must agree with an fp64 reading); the
                           weight and gradient buffers of this interface are always fp32 */
    lact_opt opt;       /* update rule */
    int ns_steps;       /* Newton-Schulz steps (Muon), 1..16; 5 in LaCT */
    double ns_a, ns_b, ns_c; /* quintic coefficients, (3.4445, -4.7750, 2.0315) */
    double muon_lr;     /* Muon step size, 0.02 */
    int64_t max_chunk;  /* most tokens one lact_chunk_update / chunk of lact_sequence may hold */
    double momentum;    /* LACT_OPT_MOMENTUM: heavy-ball coefficient beta in [0, 1), 0.9. Per
                           matrix a velocity M (zero at lact_init_state) carries across updates:
                           M <- beta M + dL/dW, then W <- renorm(W - M) */
    lact_memory memory; /* LACT_MEM_SWIGLU (W1, W2, W3) or LACT_MEM_LINEAR (W1 only) */
} lact_config;

typedef struct lact_state lact_state;   /* opaque host-side handle */

/* Per-phase device time, filled by lact_get_profile() when profiling is on. */
typedef enum {
    LACT_PHASE_APPLY = 0,    /* readout kernel(s) */
    LACT_PHASE_GRAD = 1,     /* chunk gradient: the fused kernel (head dim 128), or per token
                                slice the per-token kernel + weight-gradient GEMMs (256) */
    LACT_PHASE_REDUCE = 2,   /* split-K partial-sum reduction */
    LACT_PHASE_NS = 3,       /* Newton-Schulz (Muon); on the tensor cores (bf16 io, short
                                side 128) the same kernel also applies the update, row
                                renorm and bf16 shadow, and UPDATE then has no calls */
    LACT_PHASE_UPDATE = 4,   /* update + row renorm + bf16 shadow */
    LACT_NUM_PHASES = 5
} lact_phase;

typedef struct {
    double ms[LACT_NUM_PHASES];       /* summed device time per phase */
    int64_t launches[LACT_NUM_PHASES];/* kernel launches per phase */
    int64_t calls[LACT_NUM_PHASES];   /* timed regions per phase */
    int64_t tensor_launches[LACT_NUM_PHASES]; /* of launches[], those of tcgen05 tensor-core kernels */
} lact_profile;

/* Bytes of device workspace lact_init_state needs for this configuration
 * (0 if the configuration is invalid). */
size_t lact_workspace_bytes(const lact_config* cfg);

/* Create a state. d_workspace: caller-owned device buffer of at least
 * lact_workspace_bytes(cfg) bytes, 256-byte aligned, kept alive until
 * lact_free_state. d_W1 [H, dh, d], d_W2 [H, d, dh], d_W3 [H, dh, d] fp32:
 * the initial fast weights of each head, copied to every batch entry.
 * *out is set only on LACT_OK. */
lact_status lact_init_state(lact_state** out, const lact_config* cfg, void* d_workspace,
                            size_t ws_bytes, const float* d_W1, const float* d_W2,
                            const float* d_W3, cudaStream_t stream);

/* Readout (apply): o_i = f_W(q_i) with the current W, for n_q query tokens
 * per (b, h). d_q, d_o: [B, H, n_q, d] io dtype. n_q = 0 enqueues nothing.
 * (Review page, "Fast weights are temporary context memory": a query reads
 * the key-value relation stored in the small network's weights; "Local
 * attention and nonlinear memory work together": that network is the
 * three-matrix SwiGLU MLP.) */
lact_status lact_chunk_apply(lact_state* st, const void* d_q, int64_t n_q, void* d_o,
                             cudaStream_t stream);

/* One update of W on one chunk of n_tok tokens per (b, h) (0 <= n_tok <=
 * max_chunk): chunk gradient, optimiser step, row renorm. d_k, d_v:
 * [B, H, n_tok, d] io dtype; d_eta: [B, H, n_tok] fp32.
 * (Review page, "Local attention and nonlinear memory work together": the
 * negative inner-product loss over the chunk with token-specific learning
 * rates, the GD / momentum / Muon update and the L2-normalised result;
 * "Test-Time Training Done Right", abstract: one update per chunk of 2K to
 * ~1M tokens.) */
lact_status lact_chunk_update(lact_state* st, const void* d_k, const void* d_v,
                              const float* d_eta, int64_t n_tok, cudaStream_t stream);

/* A whole layer call (review page, "Update order must respect the task":
 * language chunks read the memory of earlier chunks and then update it;
 * a posed image set is absorbed whole before its queries are answered).
 * LACT_CAUSAL_APPLY_THEN_UPDATE: q and k/v are the same n = n_q = n_kv
 *   tokens, cut into chunks of `chunk` (the last may be shorter); each chunk
 *   is first read with the current W (into d_o), then W is updated on it.
 *   (A chunk's readout runs on a stream of the state's own, joined back into
 *   `stream` before the update; everything is complete in `stream` order.)
 * LACT_SET_UPDATE_THEN_APPLY: all n_kv input tokens form one update; they
 *   are taken in slices of `chunk` whose gradients are summed before a single
 *   optimiser step; then the n_q queries are read.
 * d_q, d_o: [B, H, n_q, d]; d_k, d_v: [B, H, n_kv, d]; d_eta: [B, H, n_kv]. */
lact_status lact_sequence(lact_state* st, lact_order order, const void* d_q, int64_t n_q,
                          const void* d_k, const void* d_v, const float* d_eta, int64_t n_kv,
                          int64_t chunk, void* d_o, cudaStream_t stream);

/* Chunk gradient only (no update): d_dW1 [B,H,dh,d], d_dW2 [B,H,d,dh],
 * d_dW3 [B,H,dh,d] fp32 receive dL/dW summed over the n_tok tokens. */
lact_status lact_chunk_gradient(lact_state* st, const void* d_k, const void* d_v,
                                const float* d_eta, int64_t n_tok, float* d_dW1,
                                float* d_dW2, float* d_dW3, cudaStream_t stream);

/* Optimiser step + row renorm from a given gradient (same layouts as above):
 * W <- renorm(W - dW) for GD, renorm(W - lr NS5(dW)) for Muon, and for
 * momentum M <- beta M + dW, W <- renorm(W - M). */
lact_status lact_apply_gradient(lact_state* st, const float* d_dW1, const float* d_dW2,
                                const float* d_dW3, cudaStream_t stream);

/* Copy the fp32 fast weights out / in: d_W1 [B,H,dh,d], d_W2 [B,H,d,dh],
 * d_W3 [B,H,dh,d]. lact_set_weights also refreshes the bf16 shadow and
 * leaves the momentum velocities as they are. */
lact_status lact_get_weights(const lact_state* st, float* d_W1, float* d_W2, float* d_W3,
                             cudaStream_t stream);
lact_status lact_set_weights(lact_state* st, const float* d_W1, const float* d_W2,
                             const float* d_W3, cudaStream_t stream);

/* The resumable state in its own precision (the master fast weights, then
 * for momentum their velocities: fp32 for bf16 io, fp64 for fp32 io), for
 * exact checkpoint / resume.
 * lact_state_bytes gives the size; export copies it to d_dst, import copies
 * it back from d_src (a buffer written by lact_export_state of a state with
 * the same configuration) and refreshes the bf16 shadow. */
size_t lact_state_bytes(const lact_state* st);
lact_status lact_export_state(const lact_state* st, void* d_dst, size_t bytes, cudaStream_t stream);
lact_status lact_import_state(lact_state* st, const void* d_src, size_t bytes, cudaStream_t stream);

/* Chunk gradient without any device allocation and without a state. The
 * method's pages have no counterpart of this call: it exists for callers that
 * cannot allocate device memory (code running inside a host callback or an
 * allocator hook, under a framework that owns the whole memory pool, or on a
 * path that must not fail for lack of memory or synchronise the device), so
 * cannot provide the workspace lact_init_state asks for.
 *
 * Computes what lact_chunk_gradient computes, for bf16 io and the SwiGLU
 * memory only (anything else returns LACT_ERR_UNSUPPORTED):
 * d_dW1 [B,H,dh,d], d_dW2 [B,H,d,dh], d_dW3 [B,H,dh,d] (fp32 outputs) from
 * the fp32 weights d_W1 [B,H,dh,d], d_W2 [B,H,d,dh], d_W3 [B,H,dh,d] and
 * d_k, d_v [B,H,n_tok,d] bf16, d_eta [B,H,n_tok] fp32 (inputs), on the
 * CUDA cores. Its split-K partial sums live in a 32 MiB array of static
 * device memory inside this library, held by every GPU that loads it until
 * the process exits; one split slot takes 12*B*H*d*dh bytes, and a problem
 * whose slot does not fit returns LACT_ERR_UNSUPPORTED before anything runs.
 * The first call on each device (with that device current) looks up the
 * array's device address and keeps it. CUDA loads a library's device code
 * lazily by default, and that first lookup is what loads the part holding
 * the array: the load allocates device memory (the array, the code) and may
 * synchronise. So make one warm-up call per device outside any path that must
 * not allocate, and before any stream capture (or run the process with
 * CUDA_MODULE_LOADING=EAGER); later calls allocate nothing. The kept address
 * belongs to the device's context: do not use this call again after
 * cudaDeviceReset. All calls share the array: two calls that may overlap on the GPU
 * (other streams, other host threads) race, so order them on one stream.
 * Nothing in it needs clearing: each call overwrites what it reads. Calls no
 * cudaMalloc, cudaFree or other allocating routine. */
lact_status lact_chunk_gradient_noalloc(const lact_config* cfg, const float* d_W1, const float* d_W2,
                                        const float* d_W3, const void* d_k, const void* d_v,
                                        const float* d_eta, int64_t n_tok, float* d_dW1, float* d_dW2,
                                        float* d_dW3, cudaStream_t stream);

/* Synchronise the state's last stream and return the sticky device status
 * (LACT_OK, LACT_ERR_TIMEOUT or LACT_ERR_NONFINITE), or LACT_ERR_CUDA. */
lact_status lact_sync_status(lact_state* st);

/* Clear the sticky device status (enqueued on `stream`), e.g. after a caller
 * has handled LACT_ERR_TIMEOUT or LACT_ERR_NONFINITE; while it is set, the
 * library's tensor-core kernels skip their work. */
lact_status lact_clear_status(lact_state* st, cudaStream_t stream);

/* Test hook of the failure path every bounded device-side wait takes: one
 * thread waits on an mbarrier that nothing arrives on, for budget_ns
 * nanoseconds (1 .. 1e10), then sets the sticky timeout status and returns;
 * lact_sync_status then reports LACT_ERR_TIMEOUT. Nothing traps or hangs. */
lact_status lact_selftest_timeout(lact_state* st, int64_t budget_ns, cudaStream_t stream);

/* Per-phase CUDA-event timing of every later call (on: 1, off: 0; turning it
 * on clears the totals). lact_get_profile synchronises and returns totals. */
lact_status lact_set_profiling(lact_state* st, int enable);
lact_status lact_get_profile(lact_state* st, lact_profile* out);

/* Kernel launches this library has made in the process so far. */
int64_t lact_launch_count(void);

const char* lact_status_str(lact_status s);

/* Free the host handle (the workspace stays the caller's). */
void lact_free_state(lact_state* st);

#ifdef __cplusplus
}
#endif
#endif /* LACT_H */
