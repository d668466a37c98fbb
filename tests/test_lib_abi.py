"""The C-ABI library builds, loads without a GPU and exports every symbol the
header declares; host-side argument checks answer before any CUDA call."""

import ctypes
import os
import re

import pytest

from gated_deltanet_linear_tree_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "canopy.h")


@pytest.fixture(scope="module")
def lib():
    path = build.build()
    from gated_deltanet_linear_tree_gb300 import canopy
    canopy._lib = None
    return canopy.load(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)          # drop comments
    return sorted(set(re.findall(r"\b(canopy_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    from gated_deltanet_linear_tree_gb300 import canopy
    assert sorted(canopy.SIGNATURES) == names


def header_enum(prefix):
    """name -> value of every `CANOPY_<prefix>_<NAME> = <int>` enumerator."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return {m.group(1).lower(): int(m.group(2))
            for m in re.finditer(r"\bCANOPY_%s_([A-Z0-9_]+)\s*=\s*(-?\d+)" % prefix, text)}


def test_binding_enums_match_the_header():
    """The binding's solve and activation names carry the header's values."""
    from gated_deltanet_linear_tree_gb300 import canopy
    assert canopy.SOLVE == header_enum("SOLVE")
    assert canopy.ACT == header_enum("ACT")
    assert canopy.WS_REGION == header_enum("WS")
    assert canopy.PLAN == header_enum("PLAN")


def test_verify_plan(lib):
    """The dispatch the verify call follows, queried on the host: tiny trees
    over few (stream, value head) pairs take the path replay, bf16 at d = 128
    the tensor cores (one block up to 64 nodes, blocks in order beyond), fp32
    or d = 32 the CUDA cores; the forcing flags and refused combinations."""
    from gated_deltanet_linear_tree_gb300 import canopy
    vp = canopy.verify_plan
    assert vp(1, 16, 16, 16, True, 128) == "path_replay"
    assert vp(1, 16, 16, 16, True, 128, force="closed_form") == "tc_block"
    assert vp(8, 1, 16, 16, True, 128) == "tc_block"
    assert vp(8, 1, 16, 16, True, 128, force="path_replay") == "path_replay"
    assert vp(9, 1, 16, 16, True, 128, force="path_replay") == "none"     # the replay takes <= 8 nodes
    assert vp(64, 16, 16, 16, True, 128) == "tc_block"
    assert vp(65, 16, 16, 16, True, 128) == "tc_blocked"
    assert vp(256, 16, 16, 16, True, 128, lengths=True) == "tc_blocked"
    assert vp(64, 16, 16, 16, False, 128) == "fp32"
    assert vp(8, 1, 2, 2, True, 32, force="closed_form") == "fp32"
    assert vp(64, 2, 4, 4, True, 128, solve="neumann") == "tc_neumann"
    assert vp(65, 2, 4, 4, True, 128, solve="neumann") == "variant"
    assert vp(64, 2, 4, 4, True, 128, solve="split") == "variant"
    assert vp(64, 2, 4, 4, True, 128, solve="split", lengths=True) == "none"
    assert vp(64, 2, 4, 4, True, 128, solve="neumann", force="closed_form") == "none"
    assert vp(257, 2, 4, 4, True, 128) == "none"
    assert lib.canopy_verify_plan(8, 1, 4, 4, 1, 128, 128, 0, 0xC, 0) == -1     # both forcing flags


def test_workspace_offsets(lib):
    """Regions start on 256-byte boundaries, in the documented order, inside
    the workspace; unsupported sizes and regions answer (size_t)-1."""
    from gated_deltanet_linear_tree_gb300 import canopy
    bad = ctypes.c_size_t(-1).value
    for B, T, HV, d in ((16, 64, 16, 128), (3, 200, 4, 128), (1, 8, 2, 32)):
        total = lib.canopy_workspace_bytes(B, T, HV, d, d)
        offs = [lib.canopy_workspace_offset(B, T, HV, d, d, r) for r in range(6)]
        assert offs[0] == 0
        assert all(o % 256 == 0 for o in offs)
        assert offs[1] >= 4 and offs[2] >= offs[1] + B * T * HV * 4 and offs[3] >= offs[2] + B * T * 4
        assert offs[4] >= offs[3] + B * T * ((T + 31) // 32) * 4 and offs[5] >= offs[4] + B * T * 4
        assert offs[5] + B * T * HV * d * 4 <= total
    assert lib.canopy_workspace_offset(16, 257, 16, 128, 128, 1) == bad
    assert lib.canopy_workspace_offset(16, 64, 16, 128, 128, 6) == bad


def test_workspace_sizes(lib):
    n = lib.canopy_workspace_bytes(16, 64, 16, 128, 128)
    # U + l + depth + mask + order + scratch, each region 256-byte aligned
    assert n >= 16 * 64 * 16 * 128 * 4 * 3 + 2 * 16 * 16 * 64 * 64 * 4
    assert lib.canopy_workspace_bytes(16, 257, 16, 128, 128) == 0
    assert lib.canopy_workspace_bytes(16, 64, 16, 64, 64) == 0
    assert lib.canopy_workspace_bytes(0, 64, 16, 128, 128) == 0
    assert lib.canopy_workspace_bytes(1, 8, 2, 32, 32) > 0
    assert lib.canopy_snapshot_bytes(16, 64, 16, 128, 128) == 16 * 64 * 16 * 128 * 128 * 4


def test_status_strings_and_version(lib):
    assert lib.canopy_status_string(0) == b"ok"
    assert lib.canopy_status_string(3).startswith(b"unsupported")
    assert lib.canopy_version() >= 1


def _verify(lib, ptrs, T=64, B=1, H=1, HV=None, d=128, in_dt=1, solve=0, o_dt=0, flags=0, scale=1.0,
            lengths=None):
    q, k, v, g, be, S0, par, o, ws = ptrs
    HV = H if HV is None else HV
    return lib.canopy_tree_verify(q, k, v, in_dt, g, be, S0, par, lengths, T, B, H, HV, d, d, scale, solve, o,
                                  o_dt, ws, flags, None)


def test_host_argument_errors(lib):
    # Every case returns before any CUDA call: fake pointers are never dereferenced.
    good = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(9)]
    null = list(good)
    null[0] = None
    assert _verify(lib, null) == 1                                  # null pointer
    mis = list(good)
    mis[2] = ctypes.c_void_p(0x10008)
    assert _verify(lib, mis) == 1                                   # misaligned
    assert _verify(lib, good, T=257) == 3                           # T too large
    assert _verify(lib, good, T=0) == 1
    assert _verify(lib, good, d=64) == 3                            # unsupported head size
    assert _verify(lib, good, in_dt=7) == 1                         # bad enum
    assert _verify(lib, good, solve=5) == 1
    assert _verify(lib, good, solve=4) == 1
    for solve in (1, 2, 3):                                         # variants: bf16 and d = 128 only
        assert _verify(lib, good, solve=solve, in_dt=0) == 3
        assert _verify(lib, good, solve=solve, d=32) == 3
    assert _verify(lib, good, flags=0x10) == 1                      # unknown flag
    assert _verify(lib, good, flags=0x20) == 1
    assert _verify(lib, good, flags=0xC) == 1                       # closed form and path replay forced at once
    assert _verify(lib, good, flags=0x8, solve=1) == 1              # forcing flags: forward substitution only
    assert _verify(lib, good, flags=0x8, T=9) == 3                  # the path replay takes at most 8 nodes
    assert _verify(lib, good, H=2, HV=3) == 1                       # value heads not a multiple of key heads
    assert _verify(lib, good, H=2, HV=1) == 1
    assert _verify(lib, good, scale=float("nan")) == 1
    assert _verify(lib, good, scale=float("inf")) == 1
    assert _verify(lib, good, lengths=ctypes.c_void_p(0x10004)) == 1   # misaligned lengths
    for solve in (1, 2, 3):                                         # the variants take no lengths
        assert _verify(lib, good, solve=solve, lengths=good[0]) == 3
    assert lib.canopy_commit(None, good[1], good[2], good[3], good[5], None, 1, 64, 1, 1, 1, 128, 128, good[4], 0,
                             None) == 1
    assert lib.canopy_commit(good[0], good[1], good[2], good[3], None, None, 1, 64, 1, 1, 1, 128, 128, good[4], 0,
                             None) == 1
    assert lib.canopy_commit(good[0], good[1], good[2], good[3], good[5], None, 1, 300, 1, 1, 1, 128, 128, good[4], 0,
                             None) == 3
    assert lib.canopy_commit(good[0], good[1], good[2], good[3], good[5], None, 1, 64, 1, 1, 1, 128, 128, good[4], 4,
                             None) == 1
    assert lib.canopy_commit(good[0], good[1], good[2], good[3], good[5], None, 1, 64, 1, 4, 6, 128, 128, good[4], 0,
                             None) == 1
    assert lib.canopy_commit(good[0], good[1], good[2], good[3], good[5], ctypes.c_void_p(0x10004), 1, 64, 1, 1, 1,
                             128, 128, good[4], 0, None) == 1                 # misaligned lengths
    assert lib.canopy_tree_prep(good[0], good[1], 0, 1, 1, good[2], None) == 3
    # tree convolution (x, dtype, state, weight, bias, parent, T, B, C, K, act, y, err): every case is
    # refused on the host before a launch
    assert lib.canopy_tree_conv(None, 1, good[1], good[2], None, good[3], 16, 2, 64, 4, 1, good[4], None, None) == 1
    assert lib.canopy_tree_conv(good[0], 1, good[1], good[2], None, good[3], 16, 2, 64, 4, 7, good[4], None,
                                None) == 1                                          # bad activation
    assert lib.canopy_tree_conv(good[0], 1, good[1], good[2], None, good[3], 16, 2, 62, 4, 1, good[4], None,
                                None) == 3                                          # C not a multiple of 4
    assert lib.canopy_tree_conv(good[0], 1, good[1], good[2], None, good[3], 16, 2, 64, 9, 1, good[4], None,
                                None) == 3                                          # K > 8
    assert lib.canopy_tree_conv(good[0], 1, good[1], good[2], None, good[3], 16, 2, 64, 1, 1, good[4], None,
                                None) == 1                                          # K < 2
    assert lib.canopy_conv_commit(good[0], good[1], 1, good[2], good[3], good[4], 300, 2, 64, 4, None, None) == 3
    assert lib.canopy_conv_commit(good[0], None, 1, good[2], good[3], good[4], 16, 2, 64, 4, None, None) == 1
    err = ctypes.c_int32(0)
    assert lib.canopy_read_device_error(None, ctypes.byref(err), None) == 1
    assert lib.canopy_workspace_init(None, 16, None) == 1


def test_binding_fails_loudly_without_library(tmp_path):
    from gated_deltanet_linear_tree_gb300 import canopy
    saved = canopy._lib
    canopy._lib = None
    try:
        with pytest.raises(canopy.CanopyError):
            canopy.load(str(tmp_path / "missing.so"))
    finally:
        canopy._lib = saved
