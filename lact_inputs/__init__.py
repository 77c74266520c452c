"""Seeded synthetic inputs for the LaCT fast-weight chunk step.

This module is shared by the CPU oracle and the CUDA path and holds none of
the method's arithmetic: it draws the queries, keys, values, per-token
learning rates and initial fast weights that a LaCT block's projections would
produce, with the shapes of the workloads described on the pages
(Test-Time Training Done Right, arXiv 2505.23884: abstract, 2K to ~1M-token
chunks; the LaCT review page, "View synthesis" Table 2 (48 images, ~196K
input tokens, 4K decoding tokens) and "Language modelling" Table 3
(32,768-token sequences, 2,048-token windows)).

Recipe (per workload): seed = 1234 + workload number; counter-based
SplitMix64 streams q=1, k=2, v=3, eta=4, W1=5, W2=6, W3=7;
q, k ~ N(0,1) then each token divided by its L2 norm over the head dim;
v ~ N(0,1); eta = 0.01*softplus(N(0,1)); W1, W3 ~ N(0,1)/sqrt(d),
W2 ~ N(0,1)/sqrt(dh), drawn per head and shared by every batch entry;
bf16 workloads round q, k, v to bf16 (nearest even) after the fp32 step.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, replace

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libgen.so")
_SRC = os.path.join(_HERE, "gen.c")

STREAM_Q, STREAM_K, STREAM_V, STREAM_ETA, STREAM_W1, STREAM_W2, STREAM_W3 = 1, 2, 3, 4, 5, 6, 7
BASE_SEED = 1234


def build(force: bool = False) -> str:
    """Compile gen.c into libgen.so beside it (gcc, OpenMP, no FMA contraction)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
                               "-shared", "-fPIC", "-o", _SO, _SRC, "-lm"])
    return _SO


_lib = None


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        u64, i64, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
        lib.lact_gen_draws.argtypes = [u64, u64, i64, vp]
        lib.lact_gen_splitmix_sequence.argtypes = [u64, i64, vp]
        lib.lact_gen_normal.argtypes = [u64, u64, i64, ctypes.c_double, ctypes.c_int, vp]
        lib.lact_gen_unit_rows.argtypes = [u64, u64, i64, i64, ctypes.c_int, vp]
        lib.lact_gen_eta.argtypes = [u64, u64, i64, vp]
        for f in (lib.lact_gen_draws, lib.lact_gen_splitmix_sequence, lib.lact_gen_normal,
                  lib.lact_gen_unit_rows, lib.lact_gen_eta):
            f.restype = None
        _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def draws(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _load().lact_gen_draws(seed, stream, n, _ptr(out))
    return out


def splitmix_sequence(state: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _load().lact_gen_splitmix_sequence(state, n, _ptr(out))
    return out


def normal(seed: int, stream: int, shape, scale: float = 1.0, bf16: bool = False,
           out: np.ndarray | None = None) -> np.ndarray:
    n = int(np.prod(shape))
    if out is None:
        out = np.empty(shape, dtype=np.uint16 if bf16 else np.float32)
    _load().lact_gen_normal(seed, stream, n, float(scale), int(bf16), _ptr(out))
    return out


def unit_rows(seed: int, stream: int, shape, bf16: bool = False,
              out: np.ndarray | None = None) -> np.ndarray:
    d = int(shape[-1])
    if d > 1024:
        raise ValueError("head dim above 1024 is not supported by the generator")
    rows = int(np.prod(shape[:-1]))
    if out is None:
        out = np.empty(shape, dtype=np.uint16 if bf16 else np.float32)
    _load().lact_gen_unit_rows(seed, stream, rows, d, int(bf16), _ptr(out))
    return out


def eta(seed: int, stream: int, shape, out: np.ndarray | None = None) -> np.ndarray:
    n = int(np.prod(shape))
    if out is None:
        out = np.empty(shape, dtype=np.float32)
    _load().lact_gen_eta(seed, stream, n, _ptr(out))
    return out


def bf16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float32."""
    return (a.astype(np.uint32) << 16).view(np.float32)


def as_f64(a: np.ndarray) -> np.ndarray:
    """fp32 array, or bf16 bit patterns stored as uint16, widened exactly to fp64."""
    if a.dtype == np.uint16:
        return bf16_bits_to_f32(a).astype(np.float64)
    return a.astype(np.float64)


@dataclass(frozen=True)
class Workload:
    """Shapes and settings of one synthetic workload (one LaCT layer call)."""
    number: int
    name: str
    B: int
    H: int
    d: int
    dh: int
    dtype: str          # "f32" or "bf16": dtype of q, k, v and o
    order: str          # "causal" (apply-then-update per chunk) or "set" (update-then-apply)
    opt: str            # "gd", "muon" or "momentum"
    n_kv: int           # update tokens per (b, h)
    n_q: int            # query tokens per (b, h)
    chunk: int          # tokens per update chunk
    seed: int
    ns_steps: int = 5
    ns_a: float = 3.4445
    ns_b: float = -4.7750
    ns_c: float = 2.0315
    muon_lr: float = 0.02
    momentum: float = 0.9
    memory: str = "swiglu"   # "swiglu" (W1, W2, W3) or "linear" (one d x d matrix in W1)

    @property
    def bf16(self) -> bool:
        return self.dtype == "bf16"

    def with_tokens(self, n_kv: int, n_q: int | None = None, chunk: int | None = None,
                    seed: int | None = None, **kw) -> "Workload":
        """Same layer shapes with other token counts (smaller parity cases)."""
        if n_q is None:
            n_q = n_kv if self.order == "causal" else self.n_q
        if chunk is None:
            chunk = self.chunk if self.order == "causal" else n_kv
        return replace(self, n_kv=n_kv, n_q=n_q, chunk=chunk,
                       seed=self.seed if seed is None else seed, **kw)


# The five workloads: two tiny fp32 causal layers (GD, Muon), a language-model
# shaped causal layer (32K tokens in 2,048-token chunks), the 48-view image-set
# layer (196,608 update tokens, 4,096 queries) and the million-token set layer;
# then the momentum update rule on the tiny fp32 and the language-model shapes,
# a wider causal layer in the shape of a 3B language model (24 heads of 128,
# 32,768 tokens in 4,096-token chunks, Muon); then the linear fast-weight
# memory (one d x d matrix) on the tiny fp32 and the image-set shapes.
WORKLOADS = {
    1: Workload(1, "tiny-causal-f32-gd", 1, 2, 64, 128, "f32", "causal", "gd",
                2048, 2048, 512, BASE_SEED + 1),
    2: Workload(2, "lm-causal-bf16-gd", 2, 4, 256, 512, "bf16", "causal", "gd",
                32768, 32768, 2048, BASE_SEED + 2),
    3: Workload(3, "tiny-causal-f32-muon", 1, 2, 64, 128, "f32", "causal", "muon",
                2048, 2048, 512, BASE_SEED + 3),
    4: Workload(4, "image-set-bf16-muon", 1, 6, 128, 512, "bf16", "set", "muon",
                196608, 4096, 196608, BASE_SEED + 4),
    5: Workload(5, "million-token-set-bf16-muon", 1, 8, 128, 512, "bf16", "set", "muon",
                1048576, 65536, 1048576, BASE_SEED + 5),
    6: Workload(6, "tiny-causal-f32-momentum", 1, 2, 64, 128, "f32", "causal", "momentum",
                2048, 2048, 512, BASE_SEED + 6),
    7: Workload(7, "lm-causal-bf16-momentum", 2, 4, 256, 512, "bf16", "causal", "momentum",
                32768, 32768, 2048, BASE_SEED + 7),
    8: Workload(8, "lm3b-causal-bf16-muon", 1, 24, 128, 512, "bf16", "causal", "muon",
                32768, 32768, 4096, BASE_SEED + 8),
    9: Workload(9, "tiny-causal-f32-linear-gd", 1, 2, 64, 64, "f32", "causal", "gd",
                2048, 2048, 512, BASE_SEED + 9, memory="linear"),
    10: Workload(10, "image-set-bf16-linear-muon", 1, 6, 128, 128, "bf16", "set", "muon",
                 196608, 4096, 196608, BASE_SEED + 10, memory="linear"),
}


@dataclass
class Inputs:
    q: np.ndarray      # [B,H,n_q,d]  float32, or uint16 bf16 bits
    k: np.ndarray      # [B,H,n_kv,d]
    v: np.ndarray      # [B,H,n_kv,d]
    eta: np.ndarray    # [B,H,n_kv]   float32
    W1: np.ndarray     # [H,dh,d]     float32 (shared over the batch); linear memory: [H,d,d]
    W2: np.ndarray     # [H,d,dh]     (None for the linear memory)
    W3: np.ndarray     # [H,dh,d]     (None for the linear memory)


def make_inputs(w: Workload) -> Inputs:
    s, B, H, d, dh = w.seed, w.B, w.H, w.d, w.dh
    q = unit_rows(s, STREAM_Q, (B, H, w.n_q, d), bf16=w.bf16)
    k = unit_rows(s, STREAM_K, (B, H, w.n_kv, d), bf16=w.bf16)
    v = normal(s, STREAM_V, (B, H, w.n_kv, d), bf16=w.bf16)
    et = eta(s, STREAM_ETA, (B, H, w.n_kv))
    if w.memory == "linear":
        return Inputs(q, k, v, et, normal(s, STREAM_W1, (H, d, d), scale=1.0 / np.sqrt(d)), None, None)
    W1 = normal(s, STREAM_W1, (H, dh, d), scale=1.0 / np.sqrt(d))
    W2 = normal(s, STREAM_W2, (H, d, dh), scale=1.0 / np.sqrt(dh))
    W3 = normal(s, STREAM_W3, (H, dh, d), scale=1.0 / np.sqrt(d))
    return Inputs(q, k, v, et, W1, W2, W3)
