"""The C ABI library loads, exports every declared symbol, and rejects bad
arguments on the host before touching a GPU."""

import ctypes
import os
import re

import pytest

from block_diffusion_masked_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    from block_diffusion_masked_gb300 import binding

    return binding.lib()


def _declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for fname in sorted(os.listdir(inc)):
        if not fname.endswith(".h"):
            continue
        text = open(os.path.join(inc, fname)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b(dfa_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert "dfa_forward" in names and "dfa_backward" in names
    for name in names:
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_version_and_error_strings(lib):
    from block_diffusion_masked_gb300 import binding as b

    assert lib.dfa_version() >= 100
    for code in (b.DFA_OK, b.DFA_EINVAL, b.DFA_EUNSUPPORTED, b.DFA_ECUDA, b.DFA_ETIMEOUT,
                 b.DFA_EDEVICE, 12345):
        assert isinstance(lib.dfa_error_string(code), bytes)


def test_host_side_argument_checks(lib):
    from block_diffusion_masked_gb300 import binding as b

    p = ctypes.c_void_p(0x1000)
    null = ctypes.c_void_p(0)
    s = ctypes.c_void_p(0)
    # unsupported head dimension, bad sizes and null pointers are refused on
    # the host, before any CUDA call.
    assert lib.dfa_forward(p, p, p, p, p, 1, 64, 2, 96, 4, s) == b.DFA_EUNSUPPORTED
    assert lib.dfa_forward(p, p, p, p, p, 1, 0, 2, 64, 4, s) == b.DFA_EINVAL
    assert lib.dfa_forward(p, p, p, p, p, 1, 64, 0, 64, 4, s) == b.DFA_EINVAL
    assert lib.dfa_forward(p, p, p, p, p, 1, 64, 2, 64, 0, s) == b.DFA_EINVAL
    assert lib.dfa_forward(p, p, p, p, p, -1, 64, 2, 64, 4, s) == b.DFA_EINVAL
    assert lib.dfa_forward(null, p, p, p, p, 1, 64, 2, 64, 4, s) == b.DFA_EINVAL
    assert lib.dfa_forward(ctypes.c_void_p(0x1008), p, p, p, p, 1, 64, 2, 64, 4, s) == b.DFA_EINVAL
    assert lib.dfa_backward(p, p, p, p, p, p, p, p, null, 1, 64, 2, 64, 4, s) == b.DFA_EINVAL
    assert lib.dfa_backward(p, p, p, p, p, p, p, p, p, 1, 64, 2, 80, 4, s) == b.DFA_EUNSUPPORTED
    assert lib.dfa_backward(p, p, p, p, p, p, p, p, p, 1, 64, 2, 96, 4, s) == b.DFA_EUNSUPPORTED
    # the causal yardstick takes any number of sequences; bad sizes are refused
    assert lib.dfa_causal_forward(p, p, p, p, p, -1, 64, 2, 64, s) == b.DFA_EINVAL
    assert lib.dfa_causal_forward(p, p, p, p, p, 3, 0, 2, 64, s) == b.DFA_EINVAL
    assert lib.dfa_causal_forward(p, p, p, p, p, 0, 64, 2, 64, s) == b.DFA_OK
    assert lib.dfa_causal_backward(p, p, p, p, p, p, p, p, null, 3, 64, 2, 64, s) == b.DFA_EINVAL
    # step API: unknown mode
    assert lib.dfa_bwd_preprocess_ex(p, p, p, p, 1, 64, 2, 64, 2, s) == b.DFA_EINVAL
    assert lib.dfa_bwd_dq_convert_ex(p, p, 1, 64, 2, 64, 5, s) == b.DFA_EINVAL
    # an empty batch is a no-op
    assert lib.dfa_forward(p, p, p, p, p, 0, 64, 2, 64, 4, s) == b.DFA_OK
    # grouped heads: kv_heads must divide heads
    assert lib.dfa_forward_gqa(p, p, p, p, p, 1, 64, 4, 3, 64, 4, s) == b.DFA_EINVAL
    assert lib.dfa_forward_gqa(p, p, p, p, p, 1, 64, 4, 0, 64, 4, s) == b.DFA_EINVAL
    assert lib.dfa_backward_gqa(p, p, p, p, p, p, p, p, p, 1, 64, 2, 4, 64, 4, s) == b.DFA_EINVAL
    # varlen: cu_seqlens must start at 0 with even, non-negative lengths
    cu = lambda *xs: (ctypes.c_int * len(xs))(*xs)  # noqa: E731
    assert lib.dfa_forward_varlen(p, p, p, p, p, cu(0, 3, 8), 2, 2, 2, 64, 4, s) == b.DFA_EINVAL
    assert lib.dfa_forward_varlen(p, p, p, p, p, cu(2, 8), 1, 2, 2, 64, 4, s) == b.DFA_EINVAL
    assert lib.dfa_forward_varlen(p, p, p, p, p, cu(0, 8, 6), 2, 2, 2, 64, 4, s) == b.DFA_EINVAL
    assert lib.dfa_forward_varlen(p, p, p, p, p, None, 1, 2, 2, 64, 4, s) == b.DFA_EINVAL
    assert lib.dfa_forward_varlen(p, p, p, p, p, cu(0, 0, 0), 2, 2, 2, 64, 4, s) == b.DFA_OK
    # backward options: unknown flag bits are refused
    assert lib.dfa_backward_ex(p, p, p, p, p, p, p, p, p, None, 1, 64, 2, 2, 64, 4, 4,
                               s) == b.DFA_EINVAL
    assert lib.dfa_bwd_main_ex(p, p, p, p, p, p, p, p, p, 1, 64, 2, 2, 64, 4, 0, 4,
                               s) == b.DFA_EINVAL
    assert lib.dfa_bwd_main_ex(p, p, p, p, p, p, p, p, p, 1, 64, 2, 2, 64, 4, 3, 2,
                               s) == b.DFA_EINVAL


def test_tile_shapes(lib):
    from block_diffusion_masked_gb300 import binding as b

    for d in (64, 128, 256):
        bm, bn, kbn, kbm = b.dfa_tile_shape(d)
        assert bm == 128 and bn in (64, 128) and kbn == 128 and kbm in (64, 128)
    with pytest.raises(b.DfaError):
        b.dfa_tile_shape(96)
