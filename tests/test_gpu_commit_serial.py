"""GPU parity for commit and the serial replay, device error reporting, and the
verify/commit round trip (canopy page, "M5: Commit kernel and the full
round")."""

import numpy as np
import pytest
import torch

import oracle
import synth
from synth import trees
from tests.gpu_helpers import TOL_BF16, TOL_F32, oracle_outputs, page_metrics, rel_err, run_verify, to_device

pytestmark = pytest.mark.gpu


def _inputs(T, fam, B=3, H=4, d=128, bf16=True, seed=0):
    rng = np.random.default_rng(seed + 31 * T)
    parents = [trees.family(fam, T, rng) for _ in range(B)]
    return synth.make_inputs(parents, H, d, d, bf16, case=91, rnd=seed)


@pytest.mark.parametrize("bf16", [True, False])
@pytest.mark.parametrize("T,fam", [(16, "top4"), (64, "random"), (64, "chain"), (100, "random"),
                                   (256, "skewed")])
def test_commit_matches_replay_state(lib, T, fam, bf16):
    inp = _inputs(T, fam, bf16=bf16)
    _, S_ref = oracle_outputs(inp, keep_states=True)
    dev = to_device(inp, bf16)
    B = inp["parent"].shape[0]
    o, ws, err = run_verify(lib, dev)
    assert err == 0
    rng = np.random.default_rng(T)
    for trial in range(3):
        acc = np.array([rng.choice(trees.leaves(inp["parent"][b])) if trial < 2 else rng.integers(0, T)
                        for b in range(B)], dtype=np.int32)
        S_new = lib.commit(torch.from_numpy(acc).cuda(), dev["S0"], dev["k"], dev["parent"], ws)
        assert lib.read_device_error(ws) == 0
        ref = np.stack([S_ref[b, acc[b]] for b in range(B)])
        assert rel_err(S_new.cpu().numpy(), ref) <= (TOL_BF16 if bf16 else TOL_F32)


def test_commit_nothing_accepted_and_in_place(lib):
    inp = _inputs(32, "random")
    dev = to_device(inp, True)
    o, ws, err = run_verify(lib, dev)
    acc = torch.full((3,), -1, dtype=torch.int32, device="cuda")
    S_new = lib.commit(acc, dev["S0"], dev["k"], dev["parent"], ws)
    assert torch.equal(S_new, dev["S0"])
    # in place: S_new aliases S0
    _, S_ref = oracle_outputs(inp, keep_states=True)
    acc = torch.tensor([5, 9, 31], dtype=torch.int32, device="cuda")
    S = dev["S0"].clone()
    lib.commit(acc, S, dev["k"], dev["parent"], ws, out=S)
    ref = np.stack([S_ref[b, a] for b, a in enumerate([5, 9, 31])])
    assert rel_err(S.cpu().numpy(), ref) <= TOL_BF16


@pytest.mark.parametrize("bf16", [True, False])
@pytest.mark.parametrize("T,fam", [(1, "chain"), (8, "top2"), (64, "random"), (64, "chain"), (65, "skewed"),
                                   (256, "random"), (256, "top8")])
def test_serial_replay_matches_oracle(lib, T, fam, bf16):
    inp = _inputs(T, fam, bf16=bf16)
    o_ref, _ = oracle_outputs(inp)
    dev = to_device(inp, bf16)
    B, T_, H, d = dev["q"].shape
    ws = lib.workspace(B, T, H, d)
    o = lib.serial_replay(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["S0"], dev["parent"], ws)
    assert lib.read_device_error(ws) == 0
    assert rel_err(o.cpu().numpy(), o_ref) <= TOL_F32          # fp32 state on the given inputs


def test_serial_tiny_case(lib):
    inp = synth.config_inputs(0)
    o_ref, _ = oracle_outputs(inp)
    dev = to_device(inp, False)
    ws = lib.workspace(1, 8, 2, 32)
    o = lib.serial_replay(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["S0"], dev["parent"], ws)
    assert rel_err(o.cpu().numpy(), o_ref) <= TOL_F32


def test_tiny_case_commit_every_node(lib):
    """The tiny fp32 case (dk = dv = 32): the state committed at every node
    equals the oracle's state of that node."""
    inp = synth.config_inputs(0)
    _, S_ref = oracle_outputs(inp, keep_states=True)
    dev = to_device(inp, False)
    o, ws, err = run_verify(lib, dev)
    assert err == 0
    T = inp["parent"].shape[1]
    for a in range(T):
        S_new = lib.commit(torch.tensor([a], dtype=torch.int32, device="cuda"), dev["S0"], dev["k"], dev["parent"], ws)
        assert lib.read_device_error(ws) == 0
        assert rel_err(S_new.cpu().numpy(), S_ref[:, a]) <= TOL_F32


@pytest.mark.parametrize("T", [16, 64, 128])
def test_device_error_flags(lib, T):
    """Bad trees and gates are reported through the error word, never by a
    trap; the kernels sanitise what they read, so nothing is out of bounds."""
    inp = _inputs(T, "random", B=2)
    dev = to_device(inp, True)
    bad = dev["parent"].clone()
    bad[1, T - 1] = T - 1                                  # parent[i] = i
    dev2 = dict(dev, parent=bad)
    _, ws, err = run_verify(lib, dev2)
    assert err & 0x1
    bad0 = dev["parent"].clone()
    bad0[0, 0] = 0                                         # root with a parent
    _, ws, err = run_verify(lib, dict(dev, parent=bad0))
    assert err & 0x1
    g = dev["g"].clone()
    g[0, T // 2, 1] = 0.0                                  # gate 0: log undefined
    _, ws, err = run_verify(lib, dict(dev, g=g))
    assert err & 0x2
    _, ws, err = run_verify(lib, dev)
    assert err == 0
    acc = torch.tensor([T, -5], dtype=torch.int32, device="cuda")
    lib.commit(acc, dev["S0"], dev["k"], dev["parent"], ws)
    assert lib.read_device_error(ws) & 0x4
    s = lib.workspace(2, T, 4, 128)
    lib.serial_replay(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["S0"], bad, s)
    assert lib.read_device_error(s) & 0x1


@pytest.mark.parametrize("T", [16, 64, 200])
def test_commit_on_sanitised_tree(lib, T):
    """A tree with bad parents is reported by the verify and read as the
    sanitised tree (a parent outside [0, i) becomes 0); the commit walks the
    same sanitised path, so its state is the oracle's for that tree."""
    inp = _inputs(T, "chain" if T == 200 else "random", B=2)
    bad = inp["parent"].copy()
    bad[0, T - 1] = T + 7                                  # out of range
    bad[1, T // 2] = T // 2                                # parent[i] = i
    fixed = bad.copy()
    fixed[0, T - 1] = 0
    fixed[1, T // 2] = 0
    dev = to_device(dict(inp, parent=bad), True)
    _, ws, err = run_verify(lib, dev)
    assert err & 0x1
    _, S_ref = oracle_outputs(dict(inp, parent=fixed), keep_states=True)
    acc = np.array([T - 1, T - 1], dtype=np.int32)
    S_new = lib.commit(torch.from_numpy(acc).cuda(), dev["S0"], dev["k"], dev["parent"], ws)
    ref = np.stack([S_ref[b, acc[b]] for b in range(2)])
    assert rel_err(S_new.cpu().numpy(), ref) <= TOL_BF16


def _round_trip(lib, B, T, H, rounds, bf16, replay_streams):
    """Verify a fresh tree, accept a random root-to-leaf path, commit it into
    S0 in fp32; the oracle carries its own fp64 state from the same S0.
    Every stream's o is checked every round against the oracle's closed form
    (carried over all heads at once), and the streams replay_streams(r)
    against the replay itself.  Returns the per-round errors."""
    S_dev = None
    S_orc = None
    curve = []
    for r in range(rounds):
        inp = synth.config_inputs(4, rnd=r, B=B, T=T, H=H, bf16=bf16)
        if r == 0:
            S_orc = inp["S0"].astype(np.float64)
            S_dev = torch.from_numpy(inp["S0"]).cuda()
        inp["S0"] = S_orc
        dev = to_device(inp, bf16)
        dev["S0"] = S_dev
        ws = lib.workspace(B, T, H, 128)
        o = lib.verify(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], S_dev, dev["parent"], ws)
        rng = synth.stream_seed(4, r, 999)
        acc = np.array([rng.choice(trees.leaves(inp["parent"][b])) for b in range(B)], dtype=np.int32)
        lib.commit(torch.from_numpy(acc).cuda(), S_dev, dev["k"], dev["parent"], ws, out=S_dev)
        assert lib.read_device_error(ws) == 0
        on = o.cpu().numpy()
        o_cf = np.stack([oracle.closed_form_heads(inp["parent"][b], inp["q"][b], inp["k"][b], inp["v"][b],
                                                  inp["g"][b], inp["beta"][b], S_orc[b])[0] for b in range(B)])
        e_o = rel_err(on, o_cf)
        for b in replay_streams(r):
            o_ref, _ = oracle.replay(inp["parent"][b], inp["q"][b], inp["k"][b], inp["v"][b], inp["g"][b],
                                     inp["beta"][b], S_orc[b], keep_states=False)
            e_o = max(e_o, rel_err(on[b], o_ref))
        # the oracle's own state: replay only the accepted path
        for b in range(B):
            path = oracle.root_path(inp["parent"][b], int(acc[b]))
            chain = np.arange(-1, len(path) - 1, dtype=np.int32)
            _, S_path = oracle.replay(chain, inp["q"][b][path], inp["k"][b][path], inp["v"][b][path],
                                      inp["g"][b][path], inp["beta"][b][path], S_orc[b], keep_states=True)
            S_orc[b] = S_path[-1]
        Sd = S_dev.cpu().numpy()
        curve.append((e_o, rel_err(Sd, S_orc), *page_metrics(on, o_cf), *page_metrics(Sd, S_orc)))
    return np.array(curve)


def _print_curve(tag, curve):
    """The error growth curve (canopy page, "M5": record it): per round, the
    o and state errors as max/rms, then the page's max-abs and relative
    Frobenius for o and for the state."""
    print(f"{tag} round o_err S_err o_max_abs o_rel_fro S_max_abs S_rel_fro")
    for r, row in enumerate(curve):
        print(f"{tag} {r} " + " ".join(f"{x:.3e}" for x in row))


def test_round_trip_100_rounds(lib):
    """Batched round trip: B=16, H=16, T=128, 100 rounds; o and the state
    checked every round for every stream (o against the closed form on all
    streams and against the replay on one rotating stream)."""
    curve = _round_trip(lib, 16, 128, 16, 100, True, lambda r: [r % 16])
    _print_curve("RT100", curve)
    assert curve[:, 0].max() <= TOL_BF16 and curve[:, 1].max() <= TOL_BF16
    assert curve[:, 3].max() <= TOL_BF16 and curve[:, 5].max() <= TOL_BF16   # bf16: relative Frobenius


def test_round_trip_fp32_20_rounds(lib):
    curve = _round_trip(lib, 4, 64, 4, 20, False, lambda r: range(4))
    _print_curve("RT32", curve)
    assert curve[:, 0].max() <= TOL_F32 and curve[:, 1].max() <= TOL_F32
    # the page's fp32 measures: max-abs <= 1e-4 and relative Frobenius <= 1e-5
    assert curve[:, 2].max() <= 1e-4 and curve[:, 4].max() <= 1e-4
    assert curve[:, 3].max() <= 1e-5 and curve[:, 5].max() <= 1e-5


def test_overlapped_verify_commit_steps(lib):
    """verify(inputs_ready, state_ready) then commit(state_ready), back to back over
    rotating input sets (each kernel may start while the one before it
    finishes), give the same bits as the waiting calls."""
    sets = []
    for s in range(3):
        inp = synth.config_inputs(2, rnd=s)
        dev = to_device(inp, bf16=True)
        B, T, H, d = dev["q"].shape
        dev["ws"] = lib.workspace(B, T, H, d)
        dev["acc"] = torch.full((B,), T - 1 - s, dtype=torch.int32, device="cuda")
        sets.append(dev)

    def run(overlap):
        outs = []
        for rep in range(2):
            for dev in sets:
                o = lib.verify(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["S0"], dev["parent"],
                               dev["ws"], inputs_ready=overlap, state_ready=overlap)
                Sn = lib.commit(dev["acc"], dev["S0"], dev["k"], dev["parent"], dev["ws"], state_ready=overlap)
                outs.append((o, Sn))
        torch.cuda.synchronize()
        return outs

    ref = run(False)
    got = run(True)
    for (o0, s0), (o1, s1) in zip(ref, got):
        assert torch.equal(o0, o1) and torch.equal(s0, s1)
    for dev in sets:
        assert lib.read_device_error(dev["ws"]) == 0
