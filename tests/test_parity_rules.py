"""The acceptance rule itself (tests/parity.py), on the CPU: planted route and
expert mistakes are rejected, legal near-tie choices are accepted."""
import numpy as np
import pytest

import parity
import synth


def _setup(m=6, N=40, seed=2):
    q = synth.normal_bf16((1, 1, N, 64), seed, 0)
    rng = np.random.default_rng(seed)
    lq = rng.standard_normal((1, 1, m, 64))
    logits = (lq[0, 0] @ synth.bf16_to_f64(q[0, 0]).T).T / 8.0  # [N, m]
    return q, lq, logits


def _oracle_multi(logits, s):
    order = np.argsort(-logits, axis=1, kind="stable")
    ts = -np.sort(-logits, axis=1)
    gap = ts[:, s - 1] - ts[:, s] if s < logits.shape[1] else np.full(len(logits), np.inf)
    return order[:, :s].astype(np.int32), gap


def test_routes_multi_accepts_the_oracle():
    q, lq, lg = _setup()
    r, gap = _oracle_multi(lg, 2)
    parity.check_routes_multi(q, lq, r.copy(), r, gap, np.arange(len(r)), {})


def test_routes_multi_rejects_a_wrong_set():
    q, lq, lg = _setup()
    r, gap = _oracle_multi(lg, 2)
    t = int(np.argmax(gap))  # the clearest cut
    bad = r.copy()
    third = int(np.argsort(-lg[t], kind="stable")[2])
    bad[t, 1] = third
    with pytest.raises(AssertionError):
        parity.check_routes_multi(q, lq, bad, r, gap, np.arange(len(r)), {})


def test_routes_multi_rejects_a_wrong_order():
    q, lq, lg = _setup()
    r, gap = _oracle_multi(lg, 2)
    inner = lg[np.arange(len(r)), r[:, 0]] - lg[np.arange(len(r)), r[:, 1]]
    t = int(np.argmax(inner))  # first and second far apart
    assert inner[t] > 1e-2
    bad = r.copy()
    bad[t] = bad[t, ::-1]
    with pytest.raises(AssertionError):
        parity.check_routes_multi(q, lq, bad, r, gap, np.arange(len(r)), {})


def test_routes_multi_rejects_duplicates():
    q, lq, lg = _setup()
    r, gap = _oracle_multi(lg, 2)
    bad = r.copy()
    bad[0, 1] = bad[0, 0]
    with pytest.raises(AssertionError):
        parity.check_routes_multi(q, lq, bad, r, gap, np.arange(len(r)), {})


def test_routes_multi_accepts_a_near_tie_at_the_cut():
    """Landmarks 2 and 5 made equal (to 1e-6 in logit) for every query: where
    they straddle the cut, either may be taken."""
    q, lq, lg = _setup()
    lq = lq.copy()
    lq[0, 0, 5] = lq[0, 0, 2] + 1e-7
    lg = (lq[0, 0] @ synth.bf16_to_f64(q[0, 0]).T).T / 8.0
    r, gap = _oracle_multi(lg, 2)
    alt = r.copy()
    swapped = 0
    for t in range(len(r)):
        if r[t, 1] in (2, 5) and r[t, 0] not in (2, 5) and gap[t] < 1e-3:
            alt[t, 1] = 7 - r[t, 1]  # the other of the pair
            swapped += 1
    parity.check_routes_multi(q, lq, alt, r, gap, np.arange(len(r)), {})
    assert swapped > 0


def test_outputs_rule():
    rep = {}
    ref = np.zeros((4, 64))
    parity.check_outputs(ref + 1e-3, ref, rep)
    with pytest.raises(AssertionError):
        parity.check_outputs(ref + 3e-3, ref, {})  # mean-abs above 2e-3
    bad = ref.copy()
    bad[0, 0] = 0.05
    with pytest.raises(AssertionError):
        parity.check_outputs(bad, ref, {})  # max-abs above 2e-2


def test_experts_rule(orc):
    q, k, v = synth.make_inputs("tiny")
    ora = orc.forward(q, k, v, 14, 14, 25, 25)
    lq = ora["lq"].reshape(1, 25, 64)
    e = ora["expert_idx"].reshape(1, 25, 25)
    gap = ora["gap"].reshape(1, 25)
    kf = k.reshape(1, 196, 64)
    parity.check_experts(orc, lq, kf, e.copy(), e, gap, {})
    i = int(np.argmax(gap[0]))
    bad = e.copy()
    outside = np.setdiff1d(np.arange(196), bad[0, i])
    bad[0, i, -1] = outside[-1]
    bad[0, i] = np.sort(bad[0, i])
    with pytest.raises(AssertionError):
        parity.check_experts(orc, lq, kf, bad, e, gap, {})
