"""CPU-side checks of the C ABI: the library loads and exports every symbol
include/kda.h declares; host arithmetic and status text need no GPU."""

import ctypes
import re
from pathlib import Path

import pytest

from hybrid_linear_attention_03_gb300 import build as kbuild
from hybrid_linear_attention_03_gb300 import kda

HEADER = Path(__file__).resolve().parent.parent / "include" / "kda.h"


def declared_symbols():
    text = HEADER.read_text()
    return sorted(set(re.findall(r"KDA_API\s+[^;(]*?\b(kda_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kda.lib()


def test_header_declares_the_bound_entry_points():
    assert declared_symbols() == sorted(kda.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(str(kda.lib_path()))
    for name in declared_symbols():
        assert hasattr(raw, name), f"libkda.so does not export {name}"


def test_pool_bytes_layout_arithmetic(lib):
    # H=64, d=128, bf16: 4 MiB state + 3*64*384*2 B tail per slot, 256 B header, 256-aligned regions
    desc = kda.make_desc(256, 64, 128, 128, kda.torch.bfloat16)
    state = 256 * 64 * 128 * 128 * 4
    tail_off = (256 + state + 255) // 256 * 256
    total = (tail_off + 256 * 3 * 64 * 384 * 2 + 255) // 256 * 256
    assert kda.kda_state_pool_bytes(desc) == total


@pytest.mark.parametrize("bad", [dict(num_slots=0), dict(num_heads=0), dict(d_k=-1), dict(conv_width=3),
                                 dict(act=7)])
def test_pool_bytes_rejects_bad_descriptions(lib, bad):
    fields = dict(num_slots=4, num_heads=2, d_k=16, d_v=16, conv_width=4, act=kda.KDA_F32)
    fields.update(bad)
    desc = kda.kda_pool_desc(**fields)
    assert kda.kda_state_pool_bytes(desc) == 0


def test_status_strings(lib):
    for code in range(10):
        s = kda.kda_status_string(code)
        assert s and s != "unknown status"
    assert kda.kda_status_string(99) == "unknown status"


def test_create_rejects_null_buffer(lib):
    desc = kda.make_desc(4, 2, 16, 16, kda.torch.float32)
    h = ctypes.c_void_p()
    st = lib.kda_state_pool_create(ctypes.byref(desc), None, 1 << 20, ctypes.byref(h))
    assert st == kda.KDA_ERR_INVALID_ARG and not h.value


def test_state_transfer_rejects_null_arguments(lib):
    """Host checks of the state export / import entry points (no device call)."""
    import ctypes
    buf = (ctypes.c_uint8 * 16)()
    assert lib.kda_state_slot_bytes(None) == 0
    assert lib.kda_state_export(None, 0, ctypes.addressof(buf), 16, None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_state_import(None, 0, ctypes.addressof(buf), 16, None) == kda.KDA_ERR_INVALID_ARG


def test_binding_status_checks_name_their_entry_point():
    """Every _check(status, where) call in the binding passes exactly two
    arguments (a wrapper whose call is malformed only fails on a GPU)."""
    import ast
    tree = ast.parse(Path(kda.__file__).read_text())
    calls = [n for n in ast.walk(tree) if isinstance(n, ast.Call) and getattr(n.func, "id", None) == "_check"]
    assert calls
    for c in calls:
        assert len(c.args) == 2 and isinstance(c.args[1], ast.Constant), f"line {c.lineno}"


def test_binding_has_a_function_per_entry_point():
    """The binding is the C ABI under the same names."""
    missing = [n for n in kda.EXPORTS if not callable(getattr(kda, n, None))]
    assert not missing, missing


def test_stream_wait_rejects_bad_limits(lib):
    # checked before any CUDA call
    for bad in (-1.0, float("nan"), float("inf")):
        assert lib.kda_stream_wait(None, bad) == kda.KDA_ERR_INVALID_ARG


def test_profile_argument_errors(lib):
    """kda_profile_start / kda_profile_stop reject a bad limit and a stop with
    no profile running before touching any CUDA state."""
    assert lib.kda_profile_start(0) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_profile_start((1 << 20) + 1) == kda.KDA_ERR_INVALID_ARG
    out = kda.kda_profile()
    assert lib.kda_profile_stop(ctypes.byref(out)) == kda.KDA_ERR_INVALID_ARG


def test_state_prefetch_argument_errors(lib):
    """kda_state_prefetch rejects a null pool, a null table and a negative
    batch before launching anything."""
    assert lib.kda_state_prefetch(None, None, None, 1, None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_state_prefetch(None, None, None, -1, None) == kda.KDA_ERR_INVALID_ARG


def test_pool_flags_reject_a_null_pool_and_unknown_bits(lib):
    assert lib.kda_state_pool_set_flags(None, 0) == kda.KDA_ERR_INVALID_ARG
