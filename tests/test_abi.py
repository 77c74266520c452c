"""Host-side checks of liblact's C ABI that need no GPU: the library loads,
exports every symbol include/lact.h declares, sizes its workspace, and
rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

from chunk_test_step_b300 import lact as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "lact.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lact_[a-z_]+)\s*\(", src)))


def test_header_and_binding_agree():
    assert _declared() == sorted(L.SYMBOLS)


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(L.LIB_PATH)
    for name in _declared():
        assert hasattr(lib, name), name


def test_workspace_bytes():
    c = L.make_config(1, 8, 128, 512, "bf16", "muon", max_chunk=1 << 20)
    n = L.lact_workspace_bytes(c)
    mat = 8 * 128 * 512
    assert n >= 3 * mat * 4 + 3 * mat * 2 + 3 * mat * 4
    assert n < 2 << 30
    for bad in (L.make_config(0, 1, 128, 512), L.make_config(1, 1, 96, 512), L.make_config(1, 1, 128, 100),
                L.make_config(1, 1, 128, 512, max_chunk=0), L.make_config(1, 1, 128, 2048)):
        assert L.lact_workspace_bytes(bad) == 0


def test_momentum_rule_holds_its_velocities_in_the_workspace():
    gd = L.make_config(1, 8, 128, 512, "bf16", "gd", max_chunk=4096)
    mo = L.make_config(1, 8, 128, 512, "bf16", "momentum", max_chunk=4096, momentum=0.9)
    mat = 8 * 128 * 512
    assert L.lact_workspace_bytes(mo) >= L.lact_workspace_bytes(gd) + 3 * mat * 4
    for beta in (-0.1, 1.0, float("nan")):
        assert L.lact_workspace_bytes(L.make_config(1, 8, 128, 512, "bf16", "momentum", momentum=beta)) == 0


def test_bad_arguments_are_rejected_on_the_host():
    lib = L.load()
    c = L.make_config(1, 2, 64, 128, "f32", "gd", max_chunk=512)
    h = ctypes.c_void_p()
    need = L.lact_workspace_bytes(c)
    # null workspace / weights, misaligned workspace, too-small workspace
    assert lib.lact_init_state(ctypes.byref(h), ctypes.byref(c), None, need, 256, 256, 256, None) == L.LACT_ERR_INVALID_ARG
    assert lib.lact_init_state(ctypes.byref(h), ctypes.byref(c), 4096, need, None, 256, 256, None) == L.LACT_ERR_INVALID_ARG
    assert lib.lact_init_state(ctypes.byref(h), ctypes.byref(c), 4096 + 16, need, 256, 256, 256, None) == L.LACT_ERR_INVALID_ARG
    assert lib.lact_init_state(ctypes.byref(h), ctypes.byref(c), 4096, need - 1, 256, 256, 256, None) == L.LACT_ERR_INVALID_ARG
    assert lib.lact_init_state(ctypes.byref(h), ctypes.byref(c), 4096, need, 256 + 4, 256, 256, None) == L.LACT_ERR_INVALID_ARG
    assert h.value is None
    # calls on a null state
    assert lib.lact_chunk_apply(None, 256, 1, 256, None) == L.LACT_ERR_INVALID_ARG
    assert lib.lact_chunk_update(None, 256, 256, 256, 1, None) == L.LACT_ERR_INVALID_ARG
    assert lib.lact_sequence(None, 0, 256, 1, 256, 256, 256, 1, 1, 256, None) == L.LACT_ERR_INVALID_ARG
    assert lib.lact_sync_status(None) == L.LACT_ERR_INVALID_ARG


def test_status_strings():
    for s in range(6):
        assert L.lact_status_str(s)
    assert L.lact_status_str(99) == "unknown status"
