"""Thin ctypes binding of libcanopy.so (include/canopy.h).

Argument marshalling only: every step of the path runs in the library's
CUDA kernels.  Tensors are torch CUDA tensors (torch provides device memory
and the current stream); the calls are enqueued on
``torch.cuda.current_stream()`` and return without synchronising.  If the
library has not been built, loading fails loudly: there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcanopy.so")

OK, ERR_ARG, ERR_TREE, ERR_UNSUPPORTED, ERR_CUDA = 0, 1, 2, 3, 4
F32, BF16 = 0, 1
SOLVE = {"fwdsub": 0, "neumann": 1, "squaring": 2, "split": 3}
DEVERR_TREE, DEVERR_GATE, DEVERR_ACCEPTED, DEVERR_TIMEOUT, DEVERR_LENGTH = 0x1, 0x2, 0x4, 0x8, 0x10
VERIFY_INPUTS_READY = 0x1
VERIFY_STATE_READY = 0x2
VERIFY_CLOSED_FORM = 0x4
VERIFY_PATH_REPLAY = 0x8
PLAN = {"none": -1, "path_replay": 0, "tc_block": 1, "tc_neumann": 2, "tc_blocked": 3, "fp32": 4, "variant": 5}
FORCE = {None: 0, "closed_form": VERIFY_CLOSED_FORM, "path_replay": VERIFY_PATH_REPLAY}
COMMIT_STATE_READY = 0x1
ACT = {"none": 0, "silu": 1}
WS_REGION = {"err": 0, "l": 1, "depth": 2, "mask": 3, "order": 4, "u": 5}

# name -> (restype, argtypes); mirrors include/canopy.h
_P, _I, _S, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
SIGNATURES = {
    "canopy_workspace_bytes": (_S, [_I, _I, _I, _I, _I]),
    "canopy_workspace_init": (_I, [_P, _S, _P]),
    "canopy_workspace_offset": (_S, [_I, _I, _I, _I, _I, _I]),
    "canopy_tree_prep": (_I, [_P, _P, _I, _I, _I, _P, _P]),
    "canopy_tree_verify": (_I, [_P, _P, _P, _I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _I,
                                _P, ctypes.c_uint, _P]),
    "canopy_verify_plan": (_I, [_I, _I, _I, _I, _I, _I, _I, _I, ctypes.c_uint, _I]),
    "canopy_commit": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, ctypes.c_uint, _P]),
    "canopy_snapshot_bytes": (_S, [_I, _I, _I, _I, _I]),
    "canopy_serial_replay": (_I, [_P, _P, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _I, _P, _P,
                                  _P]),
    "canopy_serial_replay_static": (_I, [_P, _P, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _I, _P,
                                         _P]),
    "canopy_tree_conv": (_I, [_P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P]),
    "canopy_conv_commit": (_I, [_P, _P, _I, _P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "canopy_read_device_error": (_I, [_P, ctypes.POINTER(ctypes.c_int32), _P]),
    "canopy_status_string": (ctypes.c_char_p, [_I]),
    "canopy_version": (_I, []),
}

_lib = None


class CanopyError(RuntimeError):
    pass


def load(path: str = LIB_PATH):
    """Load the shared library (no CUDA call is made by loading)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise CanopyError(f"{path} is missing: build it with gated_deltanet_linear_tree_gb300.build.build()")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(status: int, what: str):
    if status != OK:
        msg = load().canopy_status_string(status).decode()
        raise CanopyError(f"{what}: {msg} (status {status})")


def _ptr(t: torch.Tensor):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise CanopyError(f"unsupported dtype {t.dtype}")


def _need(t: torch.Tensor, name: str, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise CanopyError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise CanopyError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise CanopyError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise CanopyError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def workspace_bytes(B: int, T: int, HV: int, d: int) -> int:
    """Workspace bytes for B streams of T nodes and HV value heads."""
    return int(load().canopy_workspace_bytes(B, T, HV, d, d))


def workspace(B: int, T: int, HV: int, d: int, device="cuda") -> torch.Tensor:
    n = workspace_bytes(B, T, HV, d)
    if n == 0:
        raise CanopyError("unsupported sizes for the workspace")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    _check(load().canopy_workspace_init(_ptr(ws), n, _stream()), "canopy_workspace_init")
    return ws


def workspace_views(ws, B: int, T: int, HV: int, d: int) -> dict:
    """Views of the workspace regions a caller may read (canopy_ws_region):
    l fp32 [B, T, HV], depth int32 [B, T], mask int32 [B, T, ceil(T/32)]
    (the uint32 words' bits), order int32 [B, T], U fp32 [B, T, HV, d]."""
    _need(ws, "workspace", torch.uint8)
    W = (T + 31) // 32
    shapes = {"l": ((B, T, HV), torch.float32), "depth": ((B, T), torch.int32),
              "mask": ((B, T, W), torch.int32), "order": ((B, T), torch.int32),
              "u": ((B, T, HV, d), torch.float32)}
    out = {}
    for name, (shape, dt) in shapes.items():
        off = int(load().canopy_workspace_offset(B, T, HV, d, d, WS_REGION[name]))
        n = 1
        for x in shape:
            n *= x
        if off == ctypes.c_size_t(-1).value or off + 4 * n > ws.numel():
            raise CanopyError(f"workspace too small or sizes unsupported for region {name}")
        out[name] = ws[off:off + 4 * n].view(dt).view(shape)
    return out


def tree_prep(parent, g, ws):
    B, T = parent.shape
    HV = g.shape[-1]
    _need(parent, "parent", torch.int32)
    _need(g, "g", torch.float32, (B, T, HV))
    _check(load().canopy_tree_prep(_ptr(parent), _ptr(g), T, B, HV, _ptr(ws), _stream()), "canopy_tree_prep")


def _heads(q, k, v, g, beta, S0, parent):
    """Check the shapes of one verify call's inputs: q, k [B, T, H, dk]
    (key heads), v [B, T, HV, dv], g, beta [B, T, HV], S0 [B, HV, dv, dk]."""
    _need(q, "q")
    B, T, H, dk = q.shape
    _need(k, "k", q.dtype, q.shape)
    _need(v, "v", q.dtype)
    if v.dim() != 4 or v.shape[:2] != q.shape[:2]:
        raise CanopyError(f"v must have shape ({B}, {T}, HV, dv), got {tuple(v.shape)}")
    HV, dv = v.shape[2], v.shape[3]
    if HV % H:
        raise CanopyError(f"value heads {HV} are not a multiple of key heads {H}")
    _need(g, "g", torch.float32, (B, T, HV))
    _need(beta, "beta", torch.float32, (B, T, HV))
    _need(S0, "S0", torch.float32, (B, HV, dv, dk))
    _need(parent, "parent", torch.int32, (B, T))
    return B, T, H, HV, dk, dv


def _lengths(lengths, B):
    if lengths is None:
        return None
    _need(lengths, "lengths", torch.int32, (B,))
    return _ptr(lengths)


def verify(q, k, v, g, beta, S0, parent, ws, solve: str = "fwdsub", o_dtype=torch.float32, out=None,
           inputs_ready: bool = False, state_ready: bool = False, scale: float = 1.0, lengths=None, force=None):
    """o [B, T, HV, dv] for every node of every stream's tree; q and k carry
    H key heads, v, g, beta and S0 HV value heads (a multiple of H), and
    scale multiplies q.  solve: "fwdsub" (every size and dtype), or
    "neumann", "squaring", "split" (bf16 q/k/v, dk = dv = 128).  inputs_ready: q, k, v, g, beta and parent are not
    written by the kernel launched just before this call on the current
    stream (CANOPY_VERIFY_INPUTS_READY); state_ready (with inputs_ready): nor
    is S0 (CANOPY_VERIFY_STATE_READY).  lengths: int32 [B] CUDA tensor of
    per-stream tree sizes (ragged batches), or None for T everywhere; rows of
    o past a stream's length are left as they were.  force: None (the
    library's dispatch), "closed_form" or "path_replay" (forward substitution
    only; the path replay takes trees of up to 8 nodes)."""
    B, T, H, HV, dk, dv = _heads(q, k, v, g, beta, S0, parent)
    _need(ws, "workspace", torch.uint8)
    if out is None:
        out = torch.empty((B, T, HV, dv), dtype=o_dtype, device=q.device)
    _need(out, "o", None, (B, T, HV, dv))
    st = load().canopy_tree_verify(_ptr(q), _ptr(k), _ptr(v), _dt(q), _ptr(g), _ptr(beta), _ptr(S0),
                                   _ptr(parent), _lengths(lengths, B), T, B, H, HV, dk, dv, float(scale),
                                   SOLVE[solve], _ptr(out), _dt(out),
                                   _ptr(ws), (VERIFY_INPUTS_READY if inputs_ready else 0)
                                   | (VERIFY_STATE_READY if state_ready else 0) | FORCE[force], _stream())
    _check(st, "canopy_tree_verify")
    return out


def verify_plan(T: int, B: int, H: int, HV: int, bf16: bool, d: int, solve: str = "fwdsub", force=None,
                lengths: bool = False) -> str:
    """Which path canopy_tree_verify takes for these sizes (a PLAN name)."""
    code = load().canopy_verify_plan(T, B, H, HV, BF16 if bf16 else F32, d, d, SOLVE[solve], FORCE[force],
                                     int(bool(lengths)))
    return {v: k for k, v in PLAN.items()}[code]


def commit(accepted, S0, k, parent, ws, out=None, state_ready: bool = False, lengths=None):
    """S_new [B, HV, dv, dk] for the accepted node of every stream, from the
    preceding verify call's k (H key heads), parent and workspace.
    state_ready: S0, accepted, k and parent are not written by the kernel
    launched just before this call on the current stream
    (CANOPY_COMMIT_STATE_READY).  lengths: the verify call's, or None."""
    _need(S0, "S0", torch.float32)
    _need(parent, "parent", torch.int32)
    _need(k, "k")
    B, HV, dv, dk = S0.shape
    if parent.dim() != 2 or parent.shape[0] != B:
        raise CanopyError(f"parent must have shape ({B}, T), got {tuple(parent.shape)}")
    T = parent.shape[1]
    if k.dim() != 4 or k.shape[0] != B or k.shape[1] != T or k.shape[3] != dk or HV % k.shape[2]:
        raise CanopyError(f"k must have shape ({B}, {T}, H, {dk}) with H dividing {HV}, got {tuple(k.shape)}")
    H = k.shape[2]
    _need(accepted, "accepted", torch.int32, (B,))
    if out is None:
        out = torch.empty_like(S0)
    _need(out, "S_new", torch.float32, S0.shape)
    st = load().canopy_commit(_ptr(accepted), _ptr(S0), _ptr(out), _ptr(k), _ptr(parent), _lengths(lengths, B),
                              _dt(k), T, B, H, HV, dk, dv, _ptr(ws), COMMIT_STATE_READY if state_ready else 0,
                              _stream())
    _check(st, "canopy_commit")
    return out


def snapshot_bytes(B: int, T: int, HV: int, d: int) -> int:
    return int(load().canopy_snapshot_bytes(B, T, HV, d, d))


def serial_replay(q, k, v, g, beta, S0, parent, ws, snapshot=None, o_dtype=torch.float32, out=None,
                  scale: float = 1.0):
    B, T, H, HV, dk, dv = _heads(q, k, v, g, beta, S0, parent)
    if snapshot is None:
        snapshot = torch.empty(snapshot_bytes(B, T, HV, dk), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty((B, T, HV, dv), dtype=o_dtype, device=q.device)
    _need(out, "o", None, (B, T, HV, dv))
    st = load().canopy_serial_replay(_ptr(q), _ptr(k), _ptr(v), _dt(q), _ptr(g), _ptr(beta), _ptr(S0),
                                     _ptr(parent), T, B, H, HV, dk, dv, float(scale), _ptr(out), _dt(out),
                                     _ptr(snapshot), _ptr(ws), _stream())
    _check(st, "canopy_serial_replay")
    return out


def serial_replay_static(q, k, v, g, beta, S0, parent, err=None, o_dtype=torch.float32, out=None,
                         scale: float = 1.0):
    """Serial replay whose snapshots live in the library's fixed device array
    (no workspace, no snapshot buffer); err is an optional int32 CUDA tensor
    of one element that receives the device error bits (OR-ed)."""
    B, T, H, HV, dk, dv = _heads(q, k, v, g, beta, S0, parent)
    if out is None:
        out = torch.empty((B, T, HV, dv), dtype=o_dtype, device=q.device)
    _need(out, "o", None, (B, T, HV, dv))
    errp = _ptr(err) if err is not None else None
    st = load().canopy_serial_replay_static(_ptr(q), _ptr(k), _ptr(v), _dt(q), _ptr(g), _ptr(beta), _ptr(S0),
                                            _ptr(parent), T, B, H, HV, dk, dv, float(scale), _ptr(out), _dt(out),
                                            errp, _stream())
    _check(st, "canopy_serial_replay_static")
    return out


def tree_conv(x, conv_state, weight, parent, bias=None, act: str = "silu", err=None, out=None):
    """Tree-aware short causal convolution: y [B, T, C] in x's dtype.
    x [B, T, C] (bf16 or fp32); conv_state fp32 [B, C, K-1]; weight fp32
    [C, K]; bias fp32 [C] or None; parent int32 [B, T]; err an optional int32
    CUDA tensor of one element that receives device error bits (OR-ed)."""
    _need(x, "x")
    B, T, C = x.shape
    _need(weight, "weight", torch.float32)
    if weight.dim() != 2 or weight.shape[0] != C:
        raise CanopyError(f"weight must have shape ({C}, K), got {tuple(weight.shape)}")
    K = weight.shape[1]
    _need(conv_state, "conv_state", torch.float32, (B, C, K - 1))
    _need(parent, "parent", torch.int32, (B, T))
    if bias is not None:
        _need(bias, "bias", torch.float32, (C,))
    if out is None:
        out = torch.empty_like(x)
    _need(out, "y", x.dtype, x.shape)
    st = load().canopy_tree_conv(_ptr(x), _dt(x), _ptr(conv_state), _ptr(weight),
                                 _ptr(bias) if bias is not None else None, _ptr(parent), T, B, C, K, ACT[act],
                                 _ptr(out), _ptr(err) if err is not None else None, _stream())
    _check(st, "canopy_tree_conv")
    return out


def conv_commit(accepted, x, parent, conv_state, out=None, err=None):
    """The convolution state after accepting node accepted[b] of every
    stream's tree: [B, C, K-1] fp32 (out may be conv_state itself)."""
    _need(x, "x")
    B, T, C = x.shape
    _need(conv_state, "conv_state", torch.float32)
    if conv_state.dim() != 3 or conv_state.shape[:2] != (B, C):
        raise CanopyError(f"conv_state must have shape ({B}, {C}, K-1), got {tuple(conv_state.shape)}")
    K = conv_state.shape[2] + 1
    _need(accepted, "accepted", torch.int32, (B,))
    _need(parent, "parent", torch.int32, (B, T))
    if out is None:
        out = torch.empty_like(conv_state)
    _need(out, "conv_state_new", torch.float32, conv_state.shape)
    st = load().canopy_conv_commit(_ptr(accepted), _ptr(x), _dt(x), _ptr(parent), _ptr(conv_state), _ptr(out), T, B,
                                   C, K, _ptr(err) if err is not None else None, _stream())
    _check(st, "canopy_conv_commit")
    return out


def read_device_error(ws) -> int:
    """Synchronise the current stream, return and clear the device error word."""
    err = ctypes.c_int32(0)
    _check(load().canopy_read_device_error(_ptr(ws), ctypes.byref(err), _stream()), "canopy_read_device_error")
    return int(err.value)
