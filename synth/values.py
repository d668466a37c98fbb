"""Per-node activations and committed state, seeded.

Value recipe (canopy page, "Design decisions" and "The gated delta rule"; the
tiny oracle case fixes the distributions, the other cases reuse them):
  q, k    ~ N(0, 1), then L2-normalised per (token, head)
  v       ~ N(0, 1)
  alpha   = exp(-softplus(z)), z ~ N(0, 1)     (decay gate, in (0, 1))
  beta    = sigmoid(z),        z ~ N(0, 1)     (write strength, in (0, 1))
  S0      ~ N(0, 0.1^2) in fp32, shape [B, H, dv, dk] (0.1 read as the std)
For the bf16-input tier, q, k and v are rounded to bf16 (round to nearest
even) and every consumer sees exactly those rounded values; alpha, beta and S0
stay fp32.  Seeds are (case, round, stream) triples.
"""

from __future__ import annotations

import numpy as np


def stream_seed(case: int, rnd: int, stream: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(case), int(rnd), int(stream)]))


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even); returned as fp32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    bits = (bits + 0x7FFF + lsb) & 0xFFFF0000
    return bits.astype(np.uint32).view(np.float32)


def _unit_rows(x: np.ndarray) -> np.ndarray:
    n = np.sqrt((x.astype(np.float64) ** 2).sum(-1, keepdims=True))
    return (x / n).astype(np.float32)


def _softplus(z):
    return np.logaddexp(0.0, z)


def make_stream(rng: np.random.Generator, T: int, H: int, dk: int, dv: int,
                bf16: bool, s0_std: float = 0.1):
    q = _unit_rows(rng.standard_normal((T, H, dk)).astype(np.float32))
    k = _unit_rows(rng.standard_normal((T, H, dk)).astype(np.float32))
    v = rng.standard_normal((T, H, dv)).astype(np.float32)
    alpha = np.exp(-_softplus(rng.standard_normal((T, H)))).astype(np.float32)
    beta = (1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))).astype(np.float32)
    S0 = (s0_std * rng.standard_normal((H, dv, dk))).astype(np.float32)
    if bf16:
        q, k, v = round_bf16(q), round_bf16(k), round_bf16(v)
    return q, k, v, alpha, beta, S0


def make_inputs(parents, H: int, dk: int, dv: int, bf16: bool, case: int = 0,
                rnd: int = 0, s0_std: float = 0.1):
    """Inputs for B streams with the given parent arrays (all of length T).

    Returns a dict of numpy arrays: parent int32 [B,T]; q, k fp32 [B,T,H,dk];
    v fp32 [B,T,H,dv]; g (= alpha) and beta fp32 [B,T,H]; S0 fp32 [B,H,dv,dk].
    With bf16=True, q/k/v hold bf16-representable values.
    """
    parents = [np.asarray(p, dtype=np.int32) for p in parents]
    B, T = len(parents), parents[0].size
    out = {"parent": np.stack(parents)}
    cols = {n: [] for n in ("q", "k", "v", "g", "beta", "S0")}
    for b in range(B):
        rng = stream_seed(case, rnd, 1000 + b)
        q, k, v, a, be, S0 = make_stream(rng, T, H, dk, dv, bf16, s0_std)
        for n, x in zip(cols, (q, k, v, a, be, S0)):
            cols[n].append(x)
    for n, xs in cols.items():
        out[n] = np.ascontiguousarray(np.stack(xs))
    return out


def make_aligned_inputs(parents, H: int, dk: int, dv: int, bf16: bool, case: int = 0,
                        rnd: int = 0, beta_range=(0.4, 0.6), alpha_range=(0.8, 1.0)):
    """Inputs whose keys are all alike: one unit key per (stream, head),
    repeated at every node; beta and alpha uniform over the given ranges; q,
    v and S0 as in ``make_inputs``.

    With random keys in 128 dimensions k_i.k_j is about 0.09, so the deep
    terms (-G)^m R of the series the solves sum fall below any tolerance
    after two or three steps; with one key per stream they stay near
    (beta alpha)^m times the number of paths, so a solve that drops an
    ancestor or a round changes the output visibly.  Same dict layout as
    ``make_inputs``."""
    parents = [np.asarray(p, dtype=np.int32) for p in parents]
    B, T = len(parents), parents[0].size
    out = {"parent": np.stack(parents)}
    cols = {n: [] for n in ("q", "k", "v", "g", "beta", "S0")}
    for b in range(B):
        rng = stream_seed(case, rnd, 5000 + b)
        q = _unit_rows(rng.standard_normal((T, H, dk)).astype(np.float32))
        k1 = _unit_rows(rng.standard_normal((1, H, dk)).astype(np.float32))
        k = np.ascontiguousarray(np.broadcast_to(k1, (T, H, dk)))
        v = rng.standard_normal((T, H, dv)).astype(np.float32)
        alpha = rng.uniform(alpha_range[0], alpha_range[1], (T, H)).astype(np.float32)
        beta = rng.uniform(beta_range[0], beta_range[1], (T, H)).astype(np.float32)
        S0 = (0.1 * rng.standard_normal((H, dv, dk))).astype(np.float32)
        if bf16:
            q, k, v = round_bf16(q), round_bf16(k), round_bf16(v)
        for n, x in zip(cols, (q, k, v, alpha, beta, S0)):
            cols[n].append(x)
    for n, xs in cols.items():
        out[n] = np.ascontiguousarray(np.stack(xs))
    return out
