"""Shared helpers for the GPU parity tests: move seeded numpy inputs to the
device, call the library, and measure errors the way the tolerances are
stated (max |x - x_ref| / rms(x_ref) over the whole tensor of one call)."""

import numpy as np
import torch

import oracle

TOL_BF16 = 1e-2   # bf16-input tensor-core path
TOL_F32 = 1e-4    # fp32 path


def rel_err(x, ref) -> float:
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.abs(x - ref).max() / np.sqrt((ref ** 2).mean()))


def to_device(inp, bf16: bool):
    """Inputs dict (numpy) -> CUDA tensors; q/k/v as bf16 (values already
    bf16-representable) or fp32."""
    qdt = torch.bfloat16 if bf16 else torch.float32
    d = {}
    for n in ("q", "k", "v"):
        d[n] = torch.from_numpy(inp[n]).to(device="cuda", dtype=qdt).contiguous()
    for n in ("g", "beta", "S0"):
        d[n] = torch.from_numpy(inp[n]).to(device="cuda", dtype=torch.float32).contiguous()
    d["parent"] = torch.from_numpy(inp["parent"].astype(np.int32)).to("cuda").contiguous()
    return d


def oracle_outputs(inp, keep_states=False, scale=1.0):
    return oracle.replay_batch(inp["parent"], inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                               inp["S0"], keep_states=keep_states, scale=scale)


def run_verify(canopy, dev, solve="fwdsub", o_dtype=torch.float32, ws=None, scale=1.0):
    B, T, HV, d = dev["v"].shape
    if ws is None:
        ws = canopy.workspace(B, T, HV, d)
    o = canopy.verify(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["S0"], dev["parent"], ws,
                      solve=solve, o_dtype=o_dtype, scale=scale)
    err = canopy.read_device_error(ws)
    return o, ws, err


def page_metrics(x, ref):
    """The canopy page's own error measures ("Hard constraints", oracle
    parity): the largest absolute difference, and the relative Frobenius
    norm ||x - ref||_F / ||ref||_F over the whole tensor."""
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    d = x - ref
    return float(np.abs(d).max()), float(np.sqrt((d ** 2).sum() / (ref ** 2).sum()))
