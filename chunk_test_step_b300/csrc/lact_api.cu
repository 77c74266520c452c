// C ABI of liblact (declared in include/lact.h): argument checking, the
// workspace, the order of the phases, per-phase timing, and dispatch to the
// kernels.
//
// Orders (LaCT review page, "Update order must respect the task"):
//   causal: per chunk, read the memory with the current W, then update W;
//   set:    update W on all input tokens (one optimiser step), then read.
#include "lact_internal.cuh"

#include <new>
#include <string.h>

namespace lact {

std::atomic<int64_t> g_launches{0};
std::atomic<int64_t> g_tc_launches{0};

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static bool config_ok(const lact_config* c) {
    if (!c) return false;
    if (c->B < 1 || c->H < 1 || c->B > 65535 || c->H > 65535) return false;
    if ((int64_t)c->B * c->H > 65535) return false;
    if (!(c->d == 32 || c->d == 64 || c->d == 128 || c->d == 256)) return false;
    if (c->dh < 64 || c->dh > 1024 || c->dh % 64 != 0) return false;
    if (c->io_dtype != LACT_F32 && c->io_dtype != LACT_BF16) return false;
    if (c->opt != LACT_OPT_GD && c->opt != LACT_OPT_MUON && c->opt != LACT_OPT_MOMENTUM) return false;
    if (c->opt == LACT_OPT_MOMENTUM && !(c->momentum >= 0.0 && c->momentum < 1.0)) return false;
    if (c->opt == LACT_OPT_MUON && (c->ns_steps < 1 || c->ns_steps > 16)) return false;
    if (c->max_chunk < 1 || c->max_chunk > (1LL << 40)) return false;
    if (c->memory != LACT_MEM_SWIGLU && c->memory != LACT_MEM_LINEAR) return false;
    if (c->memory == LACT_MEM_LINEAR) {
        if (c->dh != c->d) return false;
        const bool served = c->io_dtype == LACT_F32 ? c->d <= 128 : c->d == 128;
        if (!served) return false;
    }
    return true;
}

// Fast-weight matrices of the memory: W1, W2, W3 (SwiGLU) or W1 = W (linear).
static int nmat_of(const lact_config& c) { return c.memory == LACT_MEM_LINEAR ? 1 : 3; }

int64_t slice_cap(const lact_config& c) {
    if (c.io_dtype != LACT_BF16 || c.d != 256) return 0;
    return c.max_chunk < kSliceCap ? c.max_chunk : kSliceCap;
}

// Internal real type: fp64 for fp32 io, fp32 for bf16 io.
static size_t real_size(const lact_config& c) { return c.io_dtype == LACT_F32 ? 8 : 4; }

WsLayout ws_layout(const lact_config& c) {
    WsLayout L;
    const size_t BH = (size_t)c.B * c.H;
    const size_t mat = BH * c.d * c.dh;
    const size_t rs = real_size(c);
    const int nm = nmat_of(c);
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
    for (int m = 0; m < 3; ++m) L.W[m] = take(m < nm ? mat * rs : 0);
    for (int m = 0; m < 3; ++m) L.Wsh[m] = take(m < nm && c.io_dtype == LACT_BF16 ? mat * 2 : 0);
    for (int m = 0; m < 3; ++m) L.dW[m] = take(m < nm ? mat * rs : 0);
    L.partial = take((size_t)kMaxSlots * nm * mat * rs);
    const size_t mm = (size_t)(c.d < c.dh ? c.d : c.dh);
    const size_t nn = (size_t)(c.d < c.dh ? c.dh : c.d);
    L.ns[0] = take(nm * BH * mm * nn * rs);
    L.ns[1] = take(nm * BH * mm * nn * rs);
    L.ns[2] = take(nm * BH * mm * mm * rs);
    L.ns[3] = take(nm * BH * mm * mm * rs);
    L.inter = take((size_t)3 * BH * slice_cap(c) * c.dh * 2);
    for (int m = 0; m < 3; ++m) L.mom[m] = take(c.opt == LACT_OPT_MOMENTUM && m < nm ? mat * rs : 0);
    L.status = take(64 * 4);
    L.total = off;
    return L;
}

// --------------------------------------------------------------- profiling
static cudaEvent_t get_event(lact_state* st) {
    if (!st->event_pool.empty()) {
        cudaEvent_t e = st->event_pool.back();
        st->event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

// Records a start event on construction and an end event on done().
struct PhaseTimer {
    lact_state* st;
    cudaStream_t s;
    int phase;
    cudaEvent_t a = nullptr;
    int64_t l0, t0;
    PhaseTimer(lact_state* st_, int ph, cudaStream_t s_) : st(st_), s(s_), phase(ph) {
        l0 = g_launches.load();
        t0 = g_tc_launches.load();
        if (st->profiling) {
            a = get_event(st);
            if (a) cudaEventRecord(a, s);
        }
    }
    void done() {
        if (!a) return;
        cudaEvent_t b = get_event(st);
        if (!b) { st->event_pool.push_back(a); a = nullptr; return; }
        cudaEventRecord(b, s);
        st->pending.push_back(PhaseEvents{a, b, phase, (int)(g_launches.load() - l0), (int)(g_tc_launches.load() - t0)});
        a = nullptr;
    }
};

static void drain_profile(lact_state* st) {
    for (auto& p : st->pending) {
        float ms = 0.f;
        if (cudaEventSynchronize(p.b) == cudaSuccess && cudaEventElapsedTime(&ms, p.a, p.b) == cudaSuccess) {
            st->prof.ms[p.phase] += ms;
            st->prof.launches[p.phase] += p.launches;
            st->prof.calls[p.phase] += 1;
            st->prof.tensor_launches[p.phase] += p.tensor_launches;
        }
        st->event_pool.push_back(p.a);
        st->event_pool.push_back(p.b);
    }
    st->pending.clear();
}

// ------------------------------------------------------------------ phases
static lact_status cuda_status(cudaError_t e) { return e == cudaSuccess ? LACT_OK : LACT_ERR_CUDA; }

static lact_status do_apply(lact_state* st, TokView q, void* o, cudaStream_t s) {
    if (q.n == 0) return LACT_OK;
    PhaseTimer t(st, LACT_PHASE_APPLY, s);
    cudaError_t e = st->nmat == 1          ? launch_lin_apply(st, q, o, s)
                    : apply_tc_supported(st) ? launch_apply_tc(st, q, o, s)
                                             : launch_apply_simt(st, q, o, s);
    t.done();
    return cuda_status(e);
}

// Chunk gradient of tokens [k.t0, k.t0 + k.n) into out[] (accumulate: add to it).
// With `deferred` non-null, a Muon step that follows may take the split-K sum
// over: when the tensor-core Newton-Schulz will run and the partial slots are
// few, the reduction is skipped and *deferred holds their count (else 0).
static lact_status do_grad(lact_state* st, TokView k, TokView v, const float* eta, bool accumulate,
                           void* const out[3], cudaStream_t s, int* deferred = nullptr, double side_tiles = 0.0) {
    if (deferred) *deferred = 0;
    if (k.n == 0) {
        if (!accumulate) {
            const size_t bytes = (size_t)st->BH * st->cfg.d * st->cfg.dh * st->rsize;
            for (int m = 0; m < st->nmat; ++m)
                if (cudaMemsetAsync(out[m], 0, bytes, s) != cudaSuccess) return LACT_ERR_CUDA;
        }
        return LACT_OK;
    }
    if (st->nmat == 3 && fwdbwd_tc_supported(st) && st->slice_cap > 0) {
        // two kernels per token slice; the GEMMs write (or add to) out[] directly
        PhaseTimer t(st, LACT_PHASE_GRAD, s);
        cudaError_t e = cudaSuccess;
        for (int64_t o = 0; o < k.n && e == cudaSuccess; o += st->slice_cap) {
            const int64_t n = k.n - o < st->slice_cap ? k.n - o : st->slice_cap;
            const TokView ks{k.p, k.n_total, k.t0 + o, n}, vs{v.p, v.n_total, v.t0 + o, n};
            e = launch_fwdbwd_tc(st, ks, vs, eta, st->inter, st->slice_cap, s);
            if (e == cudaSuccess) e = launch_wgrad_tc(st, ks, vs, st->inter, st->slice_cap, accumulate || o > 0, out, s);
        }
        t.done();
        return cuda_status(e);
    }
    int slots = 0;
    {
        PhaseTimer t(st, LACT_PHASE_GRAD, s);
        cudaError_t e = st->nmat == 1        ? (lin_tc_supported(st) ? launch_lin_grad_tc(st, k, v, eta, &slots, s)
                                                                     : launch_lin_grad_simt(st, k, v, eta, &slots, s))
                        : grad_tc_supported(st) ? launch_grad_tc(st, k, v, eta, &slots, side_tiles, s)
                                                : launch_grad_simt(st, k, v, eta, &slots, s);
        t.done();
        if (e != cudaSuccess) return LACT_ERR_CUDA;
    }
    if (deferred && !accumulate && out == st->dW && st->cfg.opt == LACT_OPT_MUON && ns_tc_supported(st) &&
        (grad_tc_supported(st) || (st->nmat == 1 && lin_tc_supported(st))) && slots >= 1 && slots <= kNsFusedSlots) {
        *deferred = slots;   // Newton-Schulz adds the slots while it reads them
        return LACT_OK;
    }
    PhaseTimer t(st, LACT_PHASE_REDUCE, s);
    cudaError_t e = launch_reduce(st, slots, accumulate, out, s);
    t.done();
    return cuda_status(e);
}

// Optimiser step + renorm from the gradient in g[] (Muon overwrites g[]).
// slots > 0: the gradient is still in that many split-K slots (do_grad's
// `deferred`), summed by Newton-Schulz as it reads them.
static lact_status do_step(lact_state* st, void* const g[3], cudaStream_t s, int slots = 0) {
    double scale = -1.0;
    if (st->cfg.opt == LACT_OPT_MUON) {
        PhaseTimer t(st, LACT_PHASE_NS, s);
        // on the tensor cores, Newton-Schulz applies the update + renorm to
        // its result itself (no update launch)
        const bool tc = ns_tc_supported(st);
        cudaError_t e = tc ? launch_ns_tc(st, g, slots, true, s) : launch_newton_schulz(st, g, s);
        t.done();
        if (e != cudaSuccess) return LACT_ERR_CUDA;
        if (tc) return LACT_OK;
        scale = -st->cfg.muon_lr;
    }
    PhaseTimer t(st, LACT_PHASE_UPDATE, s);
    const void* gc[3] = {g[0], g[1], g[2]};
    const bool mom = st->cfg.opt == LACT_OPT_MOMENTUM;
    cudaError_t e = launch_update(st, gc, scale, mom ? st->mom : nullptr, st->cfg.momentum, s);
    t.done();
    return cuda_status(e);
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace lact

using namespace lact;

extern "C" {

size_t lact_workspace_bytes(const lact_config* cfg) {
    if (!config_ok(cfg)) return 0;
    return ws_layout(*cfg).total;
}

// The memory's weight (or gradient) pointers: 3 for SwiGLU, W1 alone for the
// linear memory; non-null and 16-byte aligned.
static bool mats_ok(int nm, const void* a, const void* b, const void* c) {
    const void* p[3] = {a, b, c};
    for (int m = 0; m < nm; ++m)
        if (!p[m] || !aligned16(p[m])) return false;
    return true;
}

lact_status lact_init_state(lact_state** out, const lact_config* cfg, void* d_ws, size_t ws_bytes,
                            const float* d_W1, const float* d_W2, const float* d_W3, cudaStream_t s) {
    if (!out || !config_ok(cfg) || !d_ws) return LACT_ERR_INVALID_ARG;
    if (((uintptr_t)d_ws & 255u) != 0 || !mats_ok(nmat_of(*cfg), d_W1, d_W2, d_W3)) return LACT_ERR_INVALID_ARG;
    WsLayout L = ws_layout(*cfg);
    if (ws_bytes < L.total) return LACT_ERR_INVALID_ARG;
    lact_state* st = new (std::nothrow) lact_state();
    if (!st) return LACT_ERR_CUDA;
    st->cfg = *cfg;
    st->BH = cfg->B * cfg->H;
    st->nmat = nmat_of(*cfg);
    st->f64 = cfg->io_dtype == LACT_F32;
    st->rsize = real_size(*cfg);
    st->ws = static_cast<char*>(d_ws);
    st->ws_bytes = ws_bytes;
    st->L = L;
    for (int m = 0; m < 3; ++m) {
        st->W[m] = st->ws + L.W[m];
        st->Wsh[m] = reinterpret_cast<bf16*>(st->ws + L.Wsh[m]);
        st->dW[m] = st->ws + L.dW[m];
    }
    st->partial = st->ws + L.partial;
    for (int i = 0; i < 4; ++i) st->ns[i] = st->ws + L.ns[i];
    st->inter = reinterpret_cast<bf16*>(st->ws + L.inter);
    for (int m = 0; m < 3; ++m) st->mom[m] = cfg->opt == LACT_OPT_MOMENTUM ? st->ws + L.mom[m] : nullptr;
    st->slice_cap = slice_cap(*cfg);
    st->status = reinterpret_cast<int*>(st->ws + L.status);
    st->last_stream = s;
    st->profiling = false;
    memset(&st->prof, 0, sizeof(st->prof));
    int dev = 0;
    st->side = nullptr;
    st->ev_fork = st->ev_join = nullptr;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&st->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaStreamCreateWithFlags(&st->side, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&st->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&st->ev_join, cudaEventDisableTiming) != cudaSuccess) {
        if (st->ev_fork) cudaEventDestroy(st->ev_fork);
        if (st->ev_join) cudaEventDestroy(st->ev_join);
        if (st->side) cudaStreamDestroy(st->side);
        delete st;
        return LACT_ERR_CUDA;
    }
    // Per-head initial weights copied to every batch entry.
    const size_t per_head = (size_t)cfg->d * cfg->dh;
    const float* src[3] = {d_W1, d_W2, d_W3};
    cudaError_t e = cudaMemsetAsync(st->status, 0, 64 * 4, s);
    for (int m = 0; m < 3 && e == cudaSuccess; ++m)
        if (st->mom[m]) e = cudaMemsetAsync(st->mom[m], 0, per_head * cfg->B * cfg->H * st->rsize, s);
    for (int m = 0; m < st->nmat && e == cudaSuccess; ++m)
        for (int b = 0; b < cfg->B && e == cudaSuccess; ++b)
            e = launch_convert(src[m], false, static_cast<char*>(st->W[m]) + (size_t)b * cfg->H * per_head * st->rsize,
                               st->f64, (size_t)cfg->H * per_head, st->num_sms, s);
    if (e == cudaSuccess) e = launch_shadow(st, s);
    if (e != cudaSuccess) {
        cudaEventDestroy(st->ev_fork);
        cudaEventDestroy(st->ev_join);
        cudaStreamDestroy(st->side);
        delete st;
        return LACT_ERR_CUDA;
    }
    *out = st;
    return LACT_OK;
}

static lact_status check_io(const lact_state* st, const void* p, int64_t n) {
    if (!st) return LACT_ERR_INVALID_ARG;
    if (n < 0) return LACT_ERR_INVALID_ARG;
    if (n > 0 && (!p || !aligned16(p))) return LACT_ERR_INVALID_ARG;
    return LACT_OK;
}

lact_status lact_chunk_apply(lact_state* st, const void* d_q, int64_t n_q, void* d_o, cudaStream_t s) {
    lact_status r = check_io(st, d_q, n_q);
    if (r == LACT_OK) r = check_io(st, d_o, n_q);
    if (r != LACT_OK) return r;
    st->last_stream = s;
    return do_apply(st, TokView{d_q, n_q, 0, n_q}, d_o, s);
}

static lact_status check_update(const lact_state* st, const void* k, const void* v, const float* eta, int64_t n) {
    lact_status r = check_io(st, k, n);
    if (r == LACT_OK) r = check_io(st, v, n);
    if (r == LACT_OK) r = check_io(st, eta, n);
    if (r != LACT_OK) return r;
    if (n > st->cfg.max_chunk) return LACT_ERR_INVALID_ARG;
    return LACT_OK;
}

lact_status lact_chunk_update(lact_state* st, const void* d_k, const void* d_v, const float* d_eta,
                              int64_t n_tok, cudaStream_t s) {
    lact_status r = check_update(st, d_k, d_v, d_eta, n_tok);
    if (r != LACT_OK) return r;
    st->last_stream = s;
    int deferred = 0;
    r = do_grad(st, TokView{d_k, n_tok, 0, n_tok}, TokView{d_v, n_tok, 0, n_tok}, d_eta, false, st->dW, s, &deferred);
    if (r != LACT_OK) return r;
    return do_step(st, st->dW, s, deferred);
}

lact_status lact_chunk_gradient(lact_state* st, const void* d_k, const void* d_v, const float* d_eta,
                                int64_t n_tok, float* d_dW1, float* d_dW2, float* d_dW3, cudaStream_t s) {
    lact_status r = check_update(st, d_k, d_v, d_eta, n_tok);
    if (r != LACT_OK) return r;
    if (!mats_ok(st->nmat, d_dW1, d_dW2, d_dW3)) return LACT_ERR_INVALID_ARG;
    st->last_stream = s;
    r = do_grad(st, TokView{d_k, n_tok, 0, n_tok}, TokView{d_v, n_tok, 0, n_tok}, d_eta, false, st->dW, s);
    if (r != LACT_OK) return r;
    float* out[3] = {d_dW1, d_dW2, d_dW3};
    const size_t n = (size_t)st->BH * st->cfg.d * st->cfg.dh;
    for (int m = 0; m < st->nmat; ++m)
        if (launch_convert(st->dW[m], st->f64, out[m], false, n, st->num_sms, s) != cudaSuccess) return LACT_ERR_CUDA;
    return LACT_OK;
}

lact_status lact_apply_gradient(lact_state* st, const float* d_dW1, const float* d_dW2, const float* d_dW3,
                                cudaStream_t s) {
    if (!st || !mats_ok(st->nmat, d_dW1, d_dW2, d_dW3)) return LACT_ERR_INVALID_ARG;
    st->last_stream = s;
    // The Muon step works in place, so take a copy into the state's own buffer.
    const size_t n = (size_t)st->BH * st->cfg.d * st->cfg.dh;
    const float* src[3] = {d_dW1, d_dW2, d_dW3};
    for (int m = 0; m < st->nmat; ++m)
        if (launch_convert(src[m], false, st->dW[m], st->f64, n, st->num_sms, s) != cudaSuccess) return LACT_ERR_CUDA;
    return do_step(st, st->dW, s);
}

lact_status lact_sequence(lact_state* st, lact_order order, const void* d_q, int64_t n_q, const void* d_k,
                          const void* d_v, const float* d_eta, int64_t n_kv, int64_t chunk, void* d_o,
                          cudaStream_t s) {
    if (!st) return LACT_ERR_INVALID_ARG;
    if (order != LACT_CAUSAL_APPLY_THEN_UPDATE && order != LACT_SET_UPDATE_THEN_APPLY) return LACT_ERR_INVALID_ARG;
    if (chunk < 1 || chunk > st->cfg.max_chunk) return LACT_ERR_INVALID_ARG;
    lact_status r = check_io(st, d_q, n_q);
    if (r == LACT_OK) r = check_io(st, d_o, n_q);
    if (r == LACT_OK) r = check_io(st, d_k, n_kv);
    if (r == LACT_OK) r = check_io(st, d_v, n_kv);
    if (r == LACT_OK) r = check_io(st, d_eta, n_kv);
    if (r != LACT_OK) return r;
    st->last_stream = s;
    if (order == LACT_CAUSAL_APPLY_THEN_UPDATE) {
        if (n_q != n_kv) return LACT_ERR_INVALID_ARG;
        // The readout of a chunk and its gradient both read W_c and nothing
        // else of each other: the readout runs on the side stream beside the
        // gradient, and the two join before the update changes W.
        for (int64_t t0 = 0; t0 < n_kv; t0 += chunk) {
            const int64_t n = n_kv - t0 < chunk ? n_kv - t0 : chunk;
            if (cudaEventRecord(st->ev_fork, s) != cudaSuccess || cudaStreamWaitEvent(st->side, st->ev_fork, 0) != cudaSuccess)
                return LACT_ERR_CUDA;
            r = do_apply(st, TokView{d_q, n_q, t0, n}, d_o, st->side);
            if (r != LACT_OK) return r;
            if (cudaEventRecord(st->ev_join, st->side) != cudaSuccess) return LACT_ERR_CUDA;
            int deferred = 0;
            // the readout's share of the GPU beside the gradient, in tile-times of
            // the gradient kernel: a CTA per 256 queries and head takes about one
            // tile-time per 64 hidden units (measured on the 3B-shaped layer)
            const double side = (double)((n + 255) / 256) * st->BH * (st->cfg.dh / 64);
            r = do_grad(st, TokView{d_k, n_kv, t0, n}, TokView{d_v, n_kv, t0, n}, d_eta, false, st->dW, s, &deferred,
                        side);
            if (r != LACT_OK) return r;
            if (cudaStreamWaitEvent(s, st->ev_join, 0) != cudaSuccess) return LACT_ERR_CUDA;
            r = do_step(st, st->dW, s, deferred);
            if (r != LACT_OK) return r;
        }
        return LACT_OK;
    }
    // set: gradients of all slices summed, one optimiser step, then readout
    if (n_kv == 0) {
        r = do_grad(st, TokView{d_k, n_kv, 0, 0}, TokView{d_v, n_kv, 0, 0}, d_eta, false, st->dW, s);
    }
    int deferred = 0;   // (one slice only: several are summed into dW first)
    for (int64_t t0 = 0; t0 < n_kv && r == LACT_OK; t0 += chunk) {
        const int64_t n = n_kv - t0 < chunk ? n_kv - t0 : chunk;
        r = do_grad(st, TokView{d_k, n_kv, t0, n}, TokView{d_v, n_kv, t0, n}, d_eta, t0 > 0, st->dW, s,
                    n == n_kv ? &deferred : nullptr);
    }
    if (r != LACT_OK) return r;
    r = do_step(st, st->dW, s, deferred);
    if (r != LACT_OK) return r;
    return do_apply(st, TokView{d_q, n_q, 0, n_q}, d_o, s);
}

lact_status lact_get_weights(const lact_state* st, float* d_W1, float* d_W2, float* d_W3, cudaStream_t s) {
    if (!st || !mats_ok(st->nmat, d_W1, d_W2, d_W3)) return LACT_ERR_INVALID_ARG;
    const size_t n = (size_t)st->BH * st->cfg.d * st->cfg.dh;
    float* dst[3] = {d_W1, d_W2, d_W3};
    for (int m = 0; m < st->nmat; ++m)
        if (launch_convert(st->W[m], st->f64, dst[m], false, n, st->num_sms, s) != cudaSuccess) return LACT_ERR_CUDA;
    return LACT_OK;
}

lact_status lact_set_weights(lact_state* st, const float* d_W1, const float* d_W2, const float* d_W3,
                             cudaStream_t s) {
    if (!st || !mats_ok(st->nmat, d_W1, d_W2, d_W3)) return LACT_ERR_INVALID_ARG;
    st->last_stream = s;
    const size_t n = (size_t)st->BH * st->cfg.d * st->cfg.dh;
    const float* src[3] = {d_W1, d_W2, d_W3};
    for (int m = 0; m < st->nmat; ++m)
        if (launch_convert(src[m], false, st->W[m], st->f64, n, st->num_sms, s) != cudaSuccess) return LACT_ERR_CUDA;
    return cuda_status(launch_shadow(st, s));
}

// The master weights, then (momentum) their velocities.
static void* state_part(const lact_state* st, int i) { return i < st->nmat ? st->W[i] : st->mom[i - st->nmat]; }
static int state_parts(const lact_state* st) { return st->cfg.opt == LACT_OPT_MOMENTUM ? 2 * st->nmat : st->nmat; }

size_t lact_state_bytes(const lact_state* st) {
    if (!st) return 0;
    return (size_t)state_parts(st) * st->BH * st->cfg.d * st->cfg.dh * st->rsize;
}

lact_status lact_export_state(const lact_state* st, void* d_dst, size_t bytes, cudaStream_t s) {
    if (!st || !d_dst || bytes < lact_state_bytes(st)) return LACT_ERR_INVALID_ARG;
    const size_t one = lact_state_bytes(st) / state_parts(st);
    for (int m = 0; m < state_parts(st); ++m)
        if (cudaMemcpyAsync(static_cast<char*>(d_dst) + m * one, state_part(st, m), one, cudaMemcpyDeviceToDevice,
                            s) != cudaSuccess)
            return LACT_ERR_CUDA;
    return LACT_OK;
}

lact_status lact_import_state(lact_state* st, const void* d_src, size_t bytes, cudaStream_t s) {
    if (!st || !d_src || bytes != lact_state_bytes(st)) return LACT_ERR_INVALID_ARG;
    st->last_stream = s;
    const size_t one = bytes / state_parts(st);
    for (int m = 0; m < state_parts(st); ++m)
        if (cudaMemcpyAsync(state_part(st, m), static_cast<const char*>(d_src) + m * one, one,
                            cudaMemcpyDeviceToDevice, s) != cudaSuccess)
            return LACT_ERR_CUDA;
    return cuda_status(launch_shadow(st, s));
}

lact_status lact_sync_status(lact_state* st) {
    if (!st) return LACT_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(st->last_stream) != cudaSuccess) return LACT_ERR_CUDA;
    int word = 0;
    if (cudaMemcpy(&word, st->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return LACT_ERR_CUDA;
    if (word & ST_TIMEOUT) return LACT_ERR_TIMEOUT;
    if (word & ST_NONFINITE) return LACT_ERR_NONFINITE;
    return LACT_OK;
}

lact_status lact_clear_status(lact_state* st, cudaStream_t s) {
    if (!st) return LACT_ERR_INVALID_ARG;
    st->last_stream = s;
    return cuda_status(cudaMemsetAsync(st->status, 0, 64 * 4, s));
}

lact_status lact_selftest_timeout(lact_state* st, int64_t budget_ns, cudaStream_t s) {
    if (!st || budget_ns < 1 || budget_ns > 10000000000LL) return LACT_ERR_INVALID_ARG;
    st->last_stream = s;
    return cuda_status(launch_wait_selftest(st->status, (uint64_t)budget_ns, s));
}

lact_status lact_set_profiling(lact_state* st, int enable) {
    if (!st) return LACT_ERR_INVALID_ARG;
    drain_profile(st);
    memset(&st->prof, 0, sizeof(st->prof));
    st->profiling = enable != 0;
    return LACT_OK;
}

lact_status lact_get_profile(lact_state* st, lact_profile* out) {
    if (!st || !out) return LACT_ERR_INVALID_ARG;
    drain_profile(st);
    *out = st->prof;
    return LACT_OK;
}

int64_t lact_launch_count(void) { return g_launches.load(); }

const char* lact_status_str(lact_status s) {
    switch (s) {
        case LACT_OK: return "ok";
        case LACT_ERR_INVALID_ARG: return "invalid argument";
        case LACT_ERR_UNSUPPORTED: return "unsupported configuration";
        case LACT_ERR_CUDA: return "CUDA error";
        case LACT_ERR_TIMEOUT: return "device-side wait timed out";
        case LACT_ERR_NONFINITE: return "non-finite fast-weight row norm";
    }
    return "unknown status";
}

void lact_free_state(lact_state* st) {
    if (!st) return;
    drain_profile(st);
    cudaStreamSynchronize(st->side);
    cudaEventDestroy(st->ev_fork);
    cudaEventDestroy(st->ev_join);
    cudaStreamDestroy(st->side);
    for (cudaEvent_t e : st->event_pool) cudaEventDestroy(e);
    delete st;
}

}  // extern "C"
