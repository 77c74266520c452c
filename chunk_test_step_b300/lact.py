"""Python binding of liblact (include/lact.h): argument marshalling only.

Every function here has the name of the C entry point it calls and passes
plain device pointers (taken from torch tensors), sizes and the CUDA stream.
All of the chunk step runs in liblact's kernels; there is no Python or CPU
fallback: if liblact.so is missing, loading it raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblact.so")

LACT_OK, LACT_ERR_INVALID_ARG, LACT_ERR_UNSUPPORTED, LACT_ERR_CUDA, LACT_ERR_TIMEOUT, LACT_ERR_NONFINITE = range(6)
LACT_F32, LACT_BF16 = 0, 1
LACT_OPT_GD, LACT_OPT_MUON, LACT_OPT_MOMENTUM = 0, 1, 2
LACT_CAUSAL_APPLY_THEN_UPDATE, LACT_SET_UPDATE_THEN_APPLY = 0, 1
LACT_MEM_SWIGLU, LACT_MEM_LINEAR = 0, 1
PHASES = ("apply", "grad", "reduce", "ns", "update")

# Every symbol include/lact.h declares.
SYMBOLS = ("lact_workspace_bytes", "lact_init_state", "lact_chunk_apply", "lact_chunk_update",
           "lact_sequence", "lact_chunk_gradient", "lact_apply_gradient", "lact_get_weights",
           "lact_set_weights", "lact_state_bytes", "lact_export_state", "lact_import_state",
           "lact_chunk_gradient_noalloc",
           "lact_sync_status", "lact_clear_status", "lact_selftest_timeout", "lact_set_profiling", "lact_get_profile",
           "lact_launch_count", "lact_status_str", "lact_free_state")


class lact_config(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("d", ctypes.c_int), ("dh", ctypes.c_int),
                ("io_dtype", ctypes.c_int), ("opt", ctypes.c_int), ("ns_steps", ctypes.c_int),
                ("ns_a", ctypes.c_double), ("ns_b", ctypes.c_double), ("ns_c", ctypes.c_double),
                ("muon_lr", ctypes.c_double), ("max_chunk", ctypes.c_int64), ("momentum", ctypes.c_double),
                ("memory", ctypes.c_int)]


class lact_profile(ctypes.Structure):
    _fields_ = [("ms", ctypes.c_double * 5), ("launches", ctypes.c_int64 * 5), ("calls", ctypes.c_int64 * 5),
                ("tensor_launches", ctypes.c_int64 * 5)]


class LactError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {lact_status_str(status)} (status {status})")


_lib = None


def load() -> ctypes.CDLL:
    """Load liblact.so from the package directory (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"liblact.so not found at {LIB_PATH}: build it with "
                           "`python chunk_test_step_b300/build.py` (there is no fallback path)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64, cint = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    P = ctypes.POINTER
    lib.lact_workspace_bytes.argtypes = [P(lact_config)]
    lib.lact_workspace_bytes.restype = ctypes.c_size_t
    lib.lact_init_state.argtypes = [P(vp), P(lact_config), vp, ctypes.c_size_t, vp, vp, vp, vp]
    lib.lact_chunk_apply.argtypes = [vp, vp, i64, vp, vp]
    lib.lact_chunk_update.argtypes = [vp, vp, vp, vp, i64, vp]
    lib.lact_sequence.argtypes = [vp, cint, vp, i64, vp, vp, vp, i64, i64, vp, vp]
    lib.lact_chunk_gradient.argtypes = [vp, vp, vp, vp, i64, vp, vp, vp, vp]
    lib.lact_apply_gradient.argtypes = [vp, vp, vp, vp, vp]
    lib.lact_get_weights.argtypes = [vp, vp, vp, vp, vp]
    lib.lact_set_weights.argtypes = [vp, vp, vp, vp, vp]
    lib.lact_state_bytes.argtypes = [vp]
    lib.lact_state_bytes.restype = ctypes.c_size_t
    lib.lact_export_state.argtypes = [vp, vp, ctypes.c_size_t, vp]
    lib.lact_import_state.argtypes = [vp, vp, ctypes.c_size_t, vp]
    lib.lact_chunk_gradient_noalloc.argtypes = [P(lact_config), vp, vp, vp, vp, vp, vp, i64, vp, vp, vp, vp]
    lib.lact_chunk_gradient_noalloc.restype = cint
    lib.lact_sync_status.argtypes = [vp]
    lib.lact_clear_status.argtypes = [vp, vp]
    lib.lact_selftest_timeout.argtypes = [vp, i64, vp]
    lib.lact_set_profiling.argtypes = [vp, cint]
    lib.lact_get_profile.argtypes = [vp, P(lact_profile)]
    lib.lact_launch_count.argtypes = []
    lib.lact_launch_count.restype = i64
    lib.lact_status_str.argtypes = [cint]
    lib.lact_status_str.restype = ctypes.c_char_p
    lib.lact_free_state.argtypes = [vp]
    lib.lact_free_state.restype = None
    for name in ("lact_init_state", "lact_chunk_apply", "lact_chunk_update", "lact_sequence",
                 "lact_chunk_gradient", "lact_apply_gradient", "lact_get_weights", "lact_set_weights",
                 "lact_export_state", "lact_import_state",
                 "lact_sync_status", "lact_clear_status", "lact_selftest_timeout", "lact_set_profiling",
                 "lact_get_profile"):
        getattr(lib, name).restype = cint
    _lib = lib
    return lib


def _p(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _s(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st: int, what: str) -> None:
    if st != LACT_OK:
        raise LactError(st, what)


def lact_status_str(status: int) -> str:
    return load().lact_status_str(status).decode()


_OPTS = {"gd": LACT_OPT_GD, "muon": LACT_OPT_MUON, "momentum": LACT_OPT_MOMENTUM}


def make_config(B, H, d, dh, io_dtype="bf16", opt="gd", max_chunk=1 << 20, ns_steps=5,
                ns_a=3.4445, ns_b=-4.7750, ns_c=2.0315, muon_lr=0.02, momentum=0.9, memory="swiglu") -> lact_config:
    return lact_config(B, H, d, dh, LACT_BF16 if io_dtype == "bf16" else LACT_F32, _OPTS[opt], ns_steps,
                       ns_a, ns_b, ns_c, muon_lr, max_chunk, momentum,
                       LACT_MEM_LINEAR if memory == "linear" else LACT_MEM_SWIGLU)


def lact_workspace_bytes(cfg: lact_config) -> int:
    return int(load().lact_workspace_bytes(ctypes.byref(cfg)))


def lact_init_state(cfg: lact_config, workspace: torch.Tensor, W1, W2, W3, stream=None) -> int:
    h = ctypes.c_void_p()
    _check(load().lact_init_state(ctypes.byref(h), ctypes.byref(cfg), _p(workspace),
                                  workspace.numel() * workspace.element_size(), _p(W1), _p(W2), _p(W3),
                                  _s(stream)), "lact_init_state")
    return h.value


def lact_chunk_apply(st: int, q, n_q: int, o, stream=None) -> None:
    _check(load().lact_chunk_apply(st, _p(q), n_q, _p(o), _s(stream)), "lact_chunk_apply")


def lact_chunk_update(st: int, k, v, eta, n_tok: int, stream=None) -> None:
    _check(load().lact_chunk_update(st, _p(k), _p(v), _p(eta), n_tok, _s(stream)), "lact_chunk_update")


def lact_sequence(st: int, order: int, q, n_q: int, k, v, eta, n_kv: int, chunk: int, o, stream=None) -> None:
    _check(load().lact_sequence(st, order, _p(q), n_q, _p(k), _p(v), _p(eta), n_kv, chunk, _p(o), _s(stream)),
           "lact_sequence")


def lact_chunk_gradient(st: int, k, v, eta, n_tok: int, dW1, dW2, dW3, stream=None) -> None:
    _check(load().lact_chunk_gradient(st, _p(k), _p(v), _p(eta), n_tok, _p(dW1), _p(dW2), _p(dW3), _s(stream)),
           "lact_chunk_gradient")


def lact_apply_gradient(st: int, dW1, dW2, dW3, stream=None) -> None:
    _check(load().lact_apply_gradient(st, _p(dW1), _p(dW2), _p(dW3), _s(stream)), "lact_apply_gradient")


def lact_get_weights(st: int, W1, W2, W3, stream=None) -> None:
    _check(load().lact_get_weights(st, _p(W1), _p(W2), _p(W3), _s(stream)), "lact_get_weights")


def lact_set_weights(st: int, W1, W2, W3, stream=None) -> None:
    _check(load().lact_set_weights(st, _p(W1), _p(W2), _p(W3), _s(stream)), "lact_set_weights")


def lact_state_bytes(st: int) -> int:
    return int(load().lact_state_bytes(st))


def lact_export_state(st: int, dst, stream=None) -> None:
    _check(load().lact_export_state(st, _p(dst), dst.numel() * dst.element_size(), _s(stream)),
           "lact_export_state")


def lact_import_state(st: int, src, stream=None) -> None:
    _check(load().lact_import_state(st, _p(src), src.numel() * src.element_size(), _s(stream)),
           "lact_import_state")


def lact_chunk_gradient_noalloc(cfg: lact_config, W1, W2, W3, k, v, eta, n_tok: int, dW1, dW2, dW3,
                                stream=None) -> None:
    """Chunk gradient with no state and no device allocation (see include/lact.h)."""
    _check(load().lact_chunk_gradient_noalloc(ctypes.byref(cfg), _p(W1), _p(W2), _p(W3), _p(k), _p(v), _p(eta),
                                              n_tok, _p(dW1), _p(dW2), _p(dW3), _s(stream)),
           "lact_chunk_gradient_noalloc")


def lact_sync_status(st: int) -> int:
    return int(load().lact_sync_status(st))


def lact_clear_status(st: int, stream=None) -> None:
    _check(load().lact_clear_status(st, _s(stream)), "lact_clear_status")


def lact_selftest_timeout(st: int, budget_ns: int, stream=None) -> None:
    _check(load().lact_selftest_timeout(st, budget_ns, _s(stream)), "lact_selftest_timeout")


def lact_set_profiling(st: int, enable: bool) -> None:
    _check(load().lact_set_profiling(st, int(bool(enable))), "lact_set_profiling")


def lact_get_profile(st: int) -> dict:
    p = lact_profile()
    _check(load().lact_get_profile(st, ctypes.byref(p)), "lact_get_profile")
    return {name: {"ms": p.ms[i], "launches": p.launches[i], "calls": p.calls[i],
                   "tensor_launches": p.tensor_launches[i]} for i, name in enumerate(PHASES)}


def lact_launch_count() -> int:
    return int(load().lact_launch_count())


def lact_free_state(st: int) -> None:
    load().lact_free_state(st)


class LactLayer:
    """Convenience owner of one state and its torch-allocated workspace."""

    def __init__(self, cfg: lact_config, W1, W2, W3, device="cuda", stream=None):
        self.cfg = cfg
        nbytes = lact_workspace_bytes(cfg)
        if nbytes == 0:
            raise LactError(LACT_ERR_INVALID_ARG, "lact_workspace_bytes")
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.handle = lact_init_state(cfg, self.workspace, W1, W2, W3, stream)
        self.io_dtype = torch.bfloat16 if cfg.io_dtype == LACT_BF16 else torch.float32

    def weights(self, stream=None):
        """(W1, W2, W3) fp32 [B, H, ...]; for the linear memory (W, None, None)."""
        c = self.cfg
        dev = self.workspace.device
        W1 = torch.empty(c.B, c.H, c.dh, c.d, device=dev)
        if c.memory == LACT_MEM_LINEAR:
            lact_get_weights(self.handle, W1, None, None, stream)
            return W1, None, None
        W2 = torch.empty(c.B, c.H, c.d, c.dh, device=dev)
        W3 = torch.empty(c.B, c.H, c.dh, c.d, device=dev)
        lact_get_weights(self.handle, W1, W2, W3, stream)
        return W1, W2, W3

    def sequence(self, order, q, k, v, eta, chunk, o=None, stream=None):
        n_q, n_kv = q.shape[2], k.shape[2]
        if o is None:
            o = torch.empty_like(q)
        lact_sequence(self.handle, order, q, n_q, k, v, eta, n_kv, chunk, o, stream)
        return o

    def close(self):
        if self.handle:
            lact_free_state(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
