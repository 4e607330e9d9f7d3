"""The C-ABI library: builds, loads without a GPU, exports every symbol include/jfa.h
declares, and rejects bad arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

import jagged_attention_recsys_jfa_gb300 as jfa
from jagged_attention_recsys_jfa_gb300 import build as jbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "jfa.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(jfa_[a-z_]+)\s*\(", src)))


def test_header_and_binding_agree():
    assert declared_functions() == sorted(jfa.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol():
    lib = jfa.load_library()
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = os.popen(f"nm -D --defined-only {jbuild.LIB_PATH}").read()
    for name in declared_functions():
        assert re.search(rf"\bT {name}\b", out), f"{name} not exported"


def test_library_has_no_libcuda_link_dependency():
    deps = os.popen(f"ldd {jbuild.LIB_PATH}").read()
    assert "libcuda.so" not in deps


def test_workspace_size():
    lib = jfa.load_library()
    f = lib.jfa_workspace_size
    assert f(0, 8, 128, 10, 10, 0) == 0          # B < 1
    assert f(4, 8, 96, 10, 10, 0) == 0           # unsupported head dim
    a = f(4, 8, 128, 1000, 1000, 0)
    b = f(4, 8, 128, 1000, 1000, 1)
    assert a > 0 and b > a and a % 256 == 0 and b % 256 == 0
    assert f(4, 8, 128, 100000, 1000, 1) > b     # grows with the row count


def _fwd(lib, **over):
    args = dict(q=16, k=16, v=16, qo=16, ko=16, B=2, H=2, d=64, tq=10, tk=10, bias=None, scale=0.125,
                causal=0, out=16, lse=16, ws=256, wsb=1 << 30, stream=None)
    args.update(over)
    return lib.jfa_forward(args["q"], args["k"], args["v"], args["qo"], args["ko"], args["B"], args["H"],
                           args["d"], args["tq"], args["tk"], args["bias"], args["scale"], args["causal"],
                           args["out"], args["lse"], args["ws"], args["wsb"], args["stream"])


def test_host_argument_checks_return_before_any_device_work():
    lib = jfa.load_library()
    assert _fwd(lib, d=96) == 2                     # JFA_ERR_UNSUPPORTED
    assert _fwd(lib, B=0) == 1                      # JFA_ERR_INVALID_ARG
    assert _fwd(lib, scale=0.0) == 1
    assert _fwd(lib, scale=float("nan")) == 1
    assert _fwd(lib, q=18) == 1                     # misaligned
    assert _fwd(lib, qo=None) == 1
    assert _fwd(lib, ws=None) == 3                  # JFA_ERR_WORKSPACE
    assert _fwd(lib, ws=128) == 3                   # misaligned workspace
    assert _fwd(lib, wsb=100) == 3                  # too small
    bad_bias = jfa.jfa._Bias(7, 16, 16, 0)
    assert _fwd(lib, bias=ctypes.byref(bad_bias)) == 2
    big_bias = jfa.jfa._Bias(1, 16, 100000, 0)
    assert _fwd(lib, bias=ctypes.byref(big_bias)) == 1
    odd_grad = jfa.jfa._Bias(1, 16, 16, 0, 18)     # gradient table not 4-byte aligned
    assert _fwd(lib, bias=ctypes.byref(odd_grad)) == 1
    # general jagged bias (kind 2): values 16-byte aligned, block offsets 8-byte aligned,
    # no relative-position gradient, its own gradient 16-byte aligned
    assert _fwd(lib, bias=ctypes.byref(jfa.jfa._Bias(2, None, 0, 0, None, 40, 64, 100))) == 1
    assert _fwd(lib, bias=ctypes.byref(jfa.jfa._Bias(2, None, 0, 0, None, 32, 68, 100))) == 1
    assert _fwd(lib, bias=ctypes.byref(jfa.jfa._Bias(2, None, 0, 0, None, None, 64, 100))) == 1
    assert _fwd(lib, bias=ctypes.byref(jfa.jfa._Bias(2, None, 0, 0, 16, 32, 64, 100))) == 2
    assert _fwd(lib, bias=ctypes.byref(jfa.jfa._Bias(2, None, 0, 0, None, 32, 64, 100, 24))) == 1
    assert _fwd(lib, bias=ctypes.byref(jfa.jfa._Bias(2, None, 0, 0, None, 32, 64, -1))) == 1


def test_status_strings():
    lib = jfa.load_library()
    for code in range(7):
        assert lib.jfa_status_string(code)
    assert b"unknown" in lib.jfa_status_string(99)


def test_python_binding_rejects_cpu_tensors():
    import torch
    q = torch.zeros(4, 2, 64, dtype=torch.bfloat16)
    off = torch.tensor([0, 4], dtype=torch.int64)
    with pytest.raises(ValueError):
        jfa.jfa_forward(q, q, q, off, off)


def test_python_binding_checks_bias_arguments():
    import torch
    H = 2
    table = torch.zeros(H, 16)
    values = torch.zeros(H, 64, dtype=torch.bfloat16)
    boff = torch.tensor([0, 64], dtype=torch.int64)
    with pytest.raises(ValueError):   # the table must be a CUDA tensor
        jfa.jfa._bias_struct(table, 0, H)
    with pytest.raises(ValueError):   # a general bias excludes the table
        jfa.jfa._bias_struct(table, 0, H, jagged_bias=(values, boff))
    with pytest.raises(ValueError):   # and the table's gradient
        jfa.jfa._bias_struct(None, 0, H, grad=table, jagged_bias=(values, boff))
    with pytest.raises(ValueError):   # its values must be CUDA bf16 [H, plane]
        jfa.jfa._bias_struct(None, 0, H, jagged_bias=(values, boff))
    with pytest.raises(ValueError):   # a general-bias gradient needs a general bias
        jfa.jfa._bias_struct(None, 0, H, jagged_bias_grad=values)
    with pytest.raises(ValueError):   # a table gradient needs a table
        jfa.jfa._bias_struct(None, 0, H, grad=table)


def test_wait_limit_scales_with_planned_work():
    """The bounded-wait limit the planner gives each launch: 2 s for small launches, then
    32 us per tile pair of one CTA's share plus the costliest item, so a launch of any size
    stays far inside it (a correct launch's longest wait is about one CTA's share)."""
    lib = jfa.load_library()
    f = lib.jfa_wait_limit_ns
    floor, per_pair = 2_000_000_000, 32_000
    assert f(0, 152, 0) == floor
    assert f(-5, 0, -1) == floor                          # clamped arguments
    assert f(152, 152, 0) == floor + per_pair             # one pair per CTA
    assert f(153, 152, 0) == floor + 2 * per_pair         # share rounded up
    assert f(1000, 1, 7) == floor + 1007 * per_pair       # ctas < 1 would count as 1
    assert f(1000, 0, 7) == floor + 1007 * per_pair
    # the gem_self forward plans ~45k pairs over 8 heads' items on 152 CTAs: the floor
    # dominates; a launch 10^4 times larger (about 10 s of work per CTA) gets minutes
    small = f(45_000, 152, 64)
    assert floor < small < floor + 20_000_000
    big = f(450_000_000, 152, 5000)
    share_s = 450_000_000 / 152 * 1e-6                    # ~1 us per pair: ~3 s per CTA
    assert big * 1e-9 > 20 * share_s
    # monotone in each argument and capped without overflow
    assert f(10**6, 152, 10) < f(2 * 10**6, 152, 10) and f(10**6, 152, 10) < f(10**6, 152, 11)
    assert f(10**6, 76, 10) > f(10**6, 152, 10)
    assert f(2**62, 1, 2**62) == floor + 3600 * 10**9


def test_nsp_setting_round_trips_and_rejects_out_of_range():
    lib = jfa.load_library()
    prev = lib.jfa_set_nsp_max_tiles(-1)
    assert 0 <= prev <= 16
    try:
        assert lib.jfa_set_nsp_max_tiles(8) == prev
        assert lib.jfa_set_nsp_max_tiles(-1) == 8
        assert lib.jfa_set_nsp_max_tiles(17) == -1 and lib.jfa_set_nsp_max_tiles(-1) == 8
    finally:
        lib.jfa_set_nsp_max_tiles(prev)
