"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs.

Tolerances (canopy page, "Hard constraints", oracle parity; restated as
max |o - o_ref| / rms(o_ref) over one call's whole output): 1e-2 on the
bf16-input tensor-core path, 1e-4 on the fp32 path.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from synth import trees
from tests.gpu_helpers import TOL_BF16, TOL_F32, oracle_outputs, page_metrics, rel_err, run_verify, to_device

pytestmark = pytest.mark.gpu


def _inputs(T, fam, B=2, H=4, d=128, bf16=True, seed=0):
    rng = np.random.default_rng(seed + 7919 * T)
    parents = [trees.family(fam, T, rng) for _ in range(B)]
    return synth.make_inputs(parents, H, d, d, bf16, case=90, rnd=seed)


def test_case0_tiny_fp32(lib):
    inp = synth.config_inputs(0)
    o_ref, _ = oracle_outputs(inp)
    o, ws, err = run_verify(lib, to_device(inp, bf16=False))
    assert err == 0
    assert rel_err(o.cpu().numpy(), o_ref) <= TOL_F32


def test_case1_qwen_layer_batch1(lib):
    inp = synth.config_inputs(1)
    o_ref, _ = oracle_outputs(inp)
    o, ws, err = run_verify(lib, to_device(inp, bf16=True))
    assert err == 0
    e = rel_err(o.cpu().numpy(), o_ref)
    print("case1 bf16 err", e)
    assert e <= TOL_BF16


def test_case2_batched_both_tiers(lib):
    inp = synth.config_inputs(2)
    o_ref, _ = oracle_outputs(inp)
    o, ws, err = run_verify(lib, to_device(inp, bf16=True))
    assert err == 0
    eb = rel_err(o.cpu().numpy(), o_ref)
    o32, _, err = run_verify(lib, to_device(inp, bf16=False))
    assert err == 0
    ea = rel_err(o32.cpu().numpy(), o_ref)
    print("case2 errors: bf16 tensor-core", eb, "fp32", ea)
    assert eb <= TOL_BF16
    assert ea <= TOL_F32
    # the page's own measures ("Hard constraints", oracle parity): bf16 relative
    # Frobenius <= 1e-2; fp32 max-abs <= 1e-4 and relative Frobenius <= 1e-5
    mb, fb = page_metrics(o.cpu().numpy(), o_ref)
    ma, fa = page_metrics(o32.cpu().numpy(), o_ref)
    print(f"case2 page metrics: bf16 max_abs {mb:.3e} rel_fro {fb:.3e}; fp32 max_abs {ma:.3e} rel_fro {fa:.3e}")
    assert fb <= 1e-2
    assert ma <= 1e-4 and fa <= 1e-5


TC_T = [1, 2, 3, 8, 15, 16, 17, 31, 33, 48, 63, 64]
BIG_T = [65, 100, 127, 128, 129, 200, 255, 256]


@pytest.mark.parametrize("fam", ["chain", "top2", "top4", "top8", "skewed", "random"])
@pytest.mark.parametrize("T", TC_T + BIG_T)
def test_shapes_bf16(lib, fam, T):
    inp = _inputs(T, fam)
    o_ref, _ = oracle_outputs(inp)
    o, _, err = run_verify(lib, to_device(inp, bf16=True))
    assert err == 0
    assert rel_err(o.cpu().numpy(), o_ref) <= TOL_BF16


@pytest.mark.parametrize("fam", ["chain", "top2", "top4", "skewed", "random"])
@pytest.mark.parametrize("T", [1, 2, 5, 16, 33, 64])
def test_neumann_variant(lib, fam, T):
    """The finite Neumann series solve (canopy page, "Design decisions") gives
    outputs and, through commit, pseudo-values that match the oracle."""
    inp = _inputs(T, fam)
    o_ref, S_ref = oracle_outputs(inp, keep_states=True)
    dev = to_device(inp, bf16=True)
    on, ws_n, err = run_verify(lib, dev, solve="neumann")
    assert err == 0
    assert rel_err(on.cpu().numpy(), o_ref) <= TOL_BF16
    B = dev["q"].shape[0]
    acc = torch.full((B,), T - 1, dtype=torch.int32, device="cuda")
    Sn = lib.commit(acc, dev["S0"], dev["k"], dev["parent"], ws_n)
    assert lib.read_device_error(ws_n) == 0
    assert rel_err(Sn.cpu().numpy(), S_ref[:, T - 1]) <= TOL_BF16


@pytest.mark.parametrize("fam", ["chain", "top4", "random"])
@pytest.mark.parametrize("T", [1, 3, 17, 64, 65, 256])
def test_shapes_fp32(lib, fam, T):
    inp = _inputs(T, fam, bf16=False)
    o_ref, _ = oracle_outputs(inp)
    o, _, err = run_verify(lib, to_device(inp, bf16=False))
    assert err == 0
    on = o.cpu().numpy()
    assert rel_err(on, o_ref) <= TOL_F32
    ma, fa = page_metrics(on, o_ref)
    print(f"FP32PAGE {fam} {T} max_abs {ma:.3e} rel_fro {fa:.3e}")
    assert ma <= 1e-4 and fa <= 1e-5


def test_small_gates_chain_stays_finite(lib):
    """64-node chain with alpha = 0.05 (the page's stability case) and a
    random tree with alpha down to 0.01."""
    for T, fam, amin in ((64, "chain", 0.05), (64, "random", 0.01), (256, "chain", 0.05)):
        inp = _inputs(T, fam)
        inp["g"] = np.full_like(inp["g"], amin) if fam == "chain" else \
            np.random.default_rng(3).uniform(amin, 1.0, inp["g"].shape).astype(np.float32)
        o_ref, _ = oracle_outputs(inp)
        o, _, err = run_verify(lib, to_device(inp, bf16=True))
        on = o.cpu().numpy()
        assert err == 0 and np.isfinite(on).all()
        assert rel_err(on, o_ref) <= TOL_BF16


def test_bf16_output(lib):
    """o written as bf16: the rounding of the result to bf16 (at most half an
    ulp, 2^-8 of the value) is allowed on top of the tolerance, as the
    KBench verify task's bound adds a bf16 half-ulp."""
    inp = synth.config_inputs(2)
    o_ref, _ = oracle_outputs(inp)
    o, _, err = run_verify(lib, to_device(inp, bf16=True), o_dtype=torch.bfloat16)
    assert err == 0
    ob = o.float().cpu().numpy().astype(np.float64)
    excess = np.maximum(np.abs(ob - o_ref) - 2.0 ** -8 * np.abs(o_ref), 0.0)
    assert excess.max() / np.sqrt((o_ref ** 2).mean()) <= TOL_BF16
    # and the plain metric is within the tolerance plus the largest rounding step
    assert rel_err(ob, o_ref) <= TOL_BF16 + 2.0 ** -8 * np.abs(o_ref).max() / np.sqrt((o_ref ** 2).mean())


def test_relabelling_gives_permuted_outputs(lib):
    inp = _inputs(64, "random", B=1)
    p = inp["parent"][0]
    o1, _, _ = run_verify(lib, to_device(inp, bf16=True))
    for order in (trees.dfs_preorder(p), trees.level_order(p)):
        inp2 = dict(inp)
        inp2["parent"] = trees.relabel(p, order)[None]
        for n in ("q", "k", "v", "g", "beta"):
            inp2[n] = np.ascontiguousarray(inp[n][:, order])
        o2, _, err = run_verify(lib, to_device(inp2, bf16=True))
        assert err == 0
        assert rel_err(o2.cpu().numpy(), o1.cpu().numpy()[:, order]) <= TOL_BF16


def test_identical_siblings(lib):
    p = np.array([-1, 0, 1, 2, 2, 1, 5, 5], dtype=np.int32)
    inp = synth.make_inputs([p], 4, 128, 128, True)
    for src, dst in ((2, 5), (3, 6), (4, 7)):
        for n in ("q", "k", "v", "g", "beta"):
            inp[n][:, dst] = inp[n][:, src]
    o, _, err = run_verify(lib, to_device(inp, bf16=True))
    o = o.cpu().numpy()
    assert err == 0
    for src, dst in ((2, 5), (3, 6), (4, 7)):
        assert np.abs(o[:, src] - o[:, dst]).max() <= 1e-5 * np.abs(o).max()


def test_beta_zero(lib):
    inp = _inputs(40, "random")
    inp["beta"][:] = 0
    o, ws, err = run_verify(lib, to_device(inp, bf16=True))
    assert err == 0
    l = np.stack([oracle.cumulative_log_gate(inp["parent"][b], inp["g"][b]) for b in range(2)])
    expect = np.exp(l)[..., None] * np.einsum("bhvd,bthd->bthv", inp["S0"].astype(np.float64),
                                              inp["q"].astype(np.float64))
    assert rel_err(o.cpu().numpy(), expect) <= TOL_BF16


def test_deterministic_and_guarded(lib):
    inp = synth.config_inputs(2)
    dev = to_device(inp, bf16=True)
    B, T, H, d = dev["q"].shape
    n = B * T * H * d
    buf = torch.full((n + 128,), 7.25, dtype=torch.float32, device="cuda")
    ws = lib.workspace(B, T, H, d)
    outs = []
    for _ in range(2):
        out = buf[64:64 + n].view(B, T, H, d)
        lib.verify(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["S0"], dev["parent"], ws, out=out)
        torch.cuda.synchronize()
        outs.append(out.clone())
    assert lib.read_device_error(ws) == 0
    assert torch.equal(outs[0], outs[1])
    assert (buf[:64] == 7.25).all() and (buf[64 + n:] == 7.25).all()


@pytest.mark.parametrize("state_ready", [False, True])
def test_inputs_ready_overlap_back_to_back(lib, state_ready):
    """With inputs_ready (and state_ready: S0 read early as well),
    back-to-back verifies (each may start while the previous one finishes,
    reading its own inputs early) give the same bits as calls that wait, for
    several input sets sharing nothing."""
    sets = []
    for s in range(3):
        inp = synth.config_inputs(2, rnd=s)
        dev = to_device(inp, bf16=True)
        B, T, H, d = dev["q"].shape
        dev["ws"] = lib.workspace(B, T, H, d)
        sets.append((inp, dev))
    ref = []
    for inp, dev in sets:
        o = lib.verify(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["S0"], dev["parent"], dev["ws"])
        torch.cuda.synchronize()
        ref.append(o.clone())
    outs = []
    for rep in range(3):
        for inp, dev in sets:
            outs.append(lib.verify(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["S0"], dev["parent"],
                                   dev["ws"], inputs_ready=True, state_ready=state_ready))
    torch.cuda.synchronize()
    for idx, o in enumerate(outs):
        assert torch.equal(o, ref[idx % len(sets)])
    for inp, dev in sets:
        assert lib.read_device_error(dev["ws"]) == 0
    o_ref, _ = oracle_outputs(sets[0][0])
    assert rel_err(outs[0].cpu().numpy(), o_ref) <= TOL_BF16


def _gva_inputs(T, fam, H, HV, bf16=True, B=2, seed=0):
    """q and k for H key heads, v, g, beta and S0 for HV value heads (the
    canopy page's grouped value attention layout)."""
    rng = np.random.default_rng(seed + 131 * T)
    parents = [trees.family(fam, T, rng) for _ in range(B)]
    ik = synth.make_inputs(parents, H, 128, 128, bf16, case=92, rnd=seed)
    iv = synth.make_inputs(parents, HV, 128, 128, bf16, case=93, rnd=seed)
    return dict(iv, q=ik["q"], k=ik["k"])


@pytest.mark.parametrize("bf16", [True, False])
@pytest.mark.parametrize("T,fam", [(16, "top4"), (64, "random"), (100, "chain"), (256, "random")])
def test_grouped_value_heads_and_scale(lib, T, fam, bf16):
    """HV = 2H value heads on H key heads and the FLA scale 1/sqrt(dk) on q:
    o and, through the commit, the accepted state match the oracle."""
    H, HV = 2, 4
    inp = _gva_inputs(T, fam, H, HV, bf16)
    sc = 1.0 / np.sqrt(128.0)
    o_ref, S_ref = oracle_outputs(inp, keep_states=True, scale=sc)
    dev = to_device(inp, bf16)
    o, ws, err = run_verify(lib, dev, scale=sc)
    assert err == 0
    tol = TOL_BF16 if bf16 else TOL_F32
    assert rel_err(o.cpu().numpy(), o_ref) <= tol
    acc = torch.tensor([T - 1, T // 2], dtype=torch.int32, device="cuda")
    Sn = lib.commit(acc, dev["S0"], dev["k"], dev["parent"], ws)
    assert lib.read_device_error(ws) == 0
    ref = np.stack([S_ref[0, T - 1], S_ref[1, T // 2]])
    assert rel_err(Sn.cpu().numpy(), ref) <= tol


@pytest.mark.parametrize("T", [8, 64])
def test_grouped_value_heads_neumann_and_serial(lib, T):
    H, HV = 1, 4
    inp = _gva_inputs(T, "top2", H, HV, True, seed=1)
    sc = 0.5
    o_ref, _ = oracle_outputs(inp, scale=sc)
    dev = to_device(inp, True)
    on, _, err = run_verify(lib, dev, solve="neumann", scale=sc)
    assert err == 0
    assert rel_err(on.cpu().numpy(), o_ref) <= TOL_BF16
    ws = lib.workspace(2, T, HV, 128)
    os_ = lib.serial_replay(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["S0"], dev["parent"], ws,
                            scale=sc)
    assert lib.read_device_error(ws) == 0
    assert rel_err(os_.cpu().numpy(), o_ref) <= TOL_F32
    if T <= 16:  # the library's fixed snapshot array holds 32 MiB
        ost = lib.serial_replay_static(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["S0"],
                                       dev["parent"], scale=sc)
        assert torch.equal(ost, os_)


def test_grouped_value_heads_bad_shapes_refused(lib):
    inp = _gva_inputs(16, "top4", 2, 4, True)
    dev = to_device(inp, True)
    ws = lib.workspace(2, 16, 4, 128)
    v3 = dev["v"][:, :, :3].contiguous()
    with pytest.raises(lib.CanopyError):
        lib.verify(dev["q"], dev["k"], v3, dev["g"][:, :, :3].contiguous(), dev["beta"][:, :, :3].contiguous(),
                   dev["S0"][:, :3].contiguous(), dev["parent"], ws)


@pytest.mark.parametrize("B,HV", [(2, 4), (16, 16)])
@pytest.mark.parametrize("T,fam", [(1, "chain"), (2, "chain"), (3, "top2"), (3, "chain")])
def test_tiny_trees_both_sides_of_the_dispatch(lib, B, HV, T, fam):
    """Below the crossover (one node, or up to three with few stream-head
    pairs) the verify replays root paths; above it, the closed form: both
    give the oracle's o, and the commit after either gives its state."""
    inp = _gva_inputs(T, fam, 2, HV, True, B=B, seed=3)
    sc = 0.25
    o_ref, S_ref = oracle_outputs(inp, keep_states=True, scale=sc)
    dev = to_device(inp, True)
    o, ws, err = run_verify(lib, dev, scale=sc)
    assert err == 0
    assert rel_err(o.cpu().numpy(), o_ref) <= TOL_BF16
    acc = torch.full((B,), T - 1, dtype=torch.int32, device="cuda")
    Sn = lib.commit(acc, dev["S0"], dev["k"], dev["parent"], ws)
    assert lib.read_device_error(ws) == 0
    assert rel_err(Sn.cpu().numpy(), S_ref[:, T - 1]) <= TOL_BF16
