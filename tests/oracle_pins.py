"""Pins for the fp64 oracle: checks against facts that do not come from the
oracle itself. Each pin takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees. test_oracle_pins.py runs them on the real oracle;
test_oracle_mutants.py runs them on deliberately broken copies and expects a
failure from at least one.

What pins what:
  * windows            hand-worked window tables (tests/golden/windows.json)
  * landmarks          torch adaptive_avg_pool1d/2d in float64 (library
                       routine); m=1 gives the mean query; m=N in 2-D gives Q
  * scores             numpy matmul
  * top-k              brute-force ranking by counting, with planted exact ties
  * LV                 scipy softmax attention of each landmark over all keys
  * routing            numpy argmax (first index on ties) and sorted margins
  * attention          k=N reduces the method to plain softmax attention over
                       [Lq; K] with values [LV; V], whatever the routes
  * weights            softmax weights sum to 1
  * permutation        permuting K,V rows permutes the experts' indices and
                       leaves LV, routes and outputs unchanged
  * hand example       a 4-token, d=2 case worked out in closed form
  * routing-only       k=N gives plain softmax attention over K, V; k<N
                       gives softmax attention over the routed keys alone
  * s experts/query    top-s routes against a stable numpy argsort (planted
                       exact tie); outputs against a brute-force softmax over
                       the shared pairs and the Python set union of the s
                       experts; s=1 is the one-expert forward; s=m with k=N
                       is plain softmax attention over [Lq; K]
  * gradients          the torch restatement of the forward pass equals the
                       C++ oracle; its autograd gradients match central
                       finite differences (torch.autograd.gradcheck)
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
from scipy.special import softmax

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _f64(a):
    return synth.bf16_to_f64(a)


def _rand(shape, seed, tag, scale=1.0):
    return synth.normal_bf16(shape, seed, tag, scale)


def pin_window_tables(o):
    g = json.load(open(os.path.join(GOLDEN, "windows.json")))
    for key, gh, p in (("14->5", 14, 5), ("32->7", 32, 7), ("40->7", 40, 7)):
        bounds = g["axis_bounds"][key]
        for i in range(p * p):
            r, c = divmod(i, p)
            (y0, y1), (x0, x1) = bounds[r], bounds[c]
            want = [y * gh + x for y in range(y0, y1) for x in range(x0, x1)]
            got = o.window(gh * gh, gh, gh, p * p, i).tolist()
            assert got == want, f"{key} window {i}: {got} != {want}"
    od = g["one_d"]
    for i, (a, b) in enumerate(od["bounds"]):
        assert o.window(od["N"], 0, 0, od["m"], i).tolist() == list(range(a, b))
    for i in range(64):  # divisible case: exactly N/m tokens each
        assert o.window(4096, 0, 0, 64, i).tolist() == list(range(64 * i, 64 * i + 64))


def pin_landmarks_adaptive_pool(o):
    import torch
    import torch.nn.functional as F

    q = _rand((2, 3, 196, 64), 11, 0)
    lq = o.landmarks(q, 14, 14, 25)
    t = torch.from_numpy(_f64(q)).reshape(6, 14, 14, 64).permute(0, 3, 1, 2)
    ref = F.adaptive_avg_pool2d(t, (5, 5)).permute(0, 2, 3, 1).reshape(2, 3, 25, 64).numpy()
    assert np.max(np.abs(lq - ref)) < 1e-12
    q = _rand((1, 2, 1600, 64), 12, 0)
    lq = o.landmarks(q, 40, 40, 49)
    t = torch.from_numpy(_f64(q)).reshape(2, 40, 40, 64).permute(0, 3, 1, 2)
    ref = F.adaptive_avg_pool2d(t, (7, 7)).permute(0, 2, 3, 1).reshape(1, 2, 49, 64).numpy()
    assert np.max(np.abs(lq - ref)) < 1e-12
    q = _rand((1, 2, 1000, 64), 13, 0)  # 1-D, m does not divide N
    lq = o.landmarks(q, 0, 0, 7)
    t = torch.from_numpy(_f64(q)).reshape(2, 1000, 64).permute(0, 2, 1)
    ref = F.adaptive_avg_pool1d(t, 7).permute(0, 2, 1).reshape(1, 2, 7, 64).numpy()
    assert np.max(np.abs(lq - ref)) < 1e-12


def pin_landmarks_special(o):
    q = _rand((1, 2, 196, 64), 14, 0)
    mean = _f64(q).mean(axis=2, keepdims=True)
    assert np.max(np.abs(o.landmarks(q, 0, 0, 1) - mean)) < 1e-12
    assert np.max(np.abs(o.landmarks(q, 14, 14, 1) - mean)) < 1e-12
    assert np.array_equal(o.landmarks(q, 14, 14, 196), _f64(q))  # m = N: one token per window


def pin_scores(o):
    q, k = _rand((2, 1, 300, 64), 15, 0), _rand((2, 1, 300, 64), 15, 1)
    lq = o.landmarks(q, 0, 0, 10)
    for bh in range(2):
        ref = (lq.reshape(2, 10, 64)[bh] @ _f64(k).reshape(2, 300, 64)[bh].T) / 8.0
        for i in (0, 9):
            assert np.max(np.abs(o.scores(lq, k, bh, i) - ref[i])) < 1e-12


def _brute_topk(s, kk):
    """Key j is selected iff fewer than kk keys beat it, where j' beats j when
    s[j'] > s[j], or s[j'] == s[j] and j' < j."""
    n = len(s)
    sel = []
    for j in range(n):
        beats = sum(1 for jj in range(n) if s[jj] > s[j] or (s[jj] == s[j] and jj < j))
        if beats < kk:
            sel.append(j)
    order = sorted(range(n), key=lambda j: (-s[j], j))
    gap = s[order[kk - 1]] - s[order[kk]] if kk < n else math.inf
    return sel, gap


def pin_topk_bruteforce(o):
    N = 40
    q, k, v = _rand((1, 2, N, 64), 16, 0), _rand((1, 2, N, 64), 16, 1), _rand((1, 2, N, 64), 16, 2)
    k = k.copy()
    k[0, 0, 7] = k[0, 0, 3]  # exact ties: duplicate rows...
    k[0, 0, 30] = k[0, 0, 3]
    k[0, 1, 5] = 0  # ...and zero rows (score exactly 0)
    k[0, 1, 25] = 0
    lq = o.landmarks(q, 0, 0, 4)
    for kk in (1, 2, 3, 7, 20, N - 1, N):
        _, e, gap = o.scan(lq, k, v, kk)
        for bh in range(2):
            for i in range(4):
                s = o.scores(lq, k, bh, i).tolist()
                sel, g = _brute_topk(s, kk)
                assert e[bh, i].tolist() == sel, (kk, bh, i)
                assert g == gap[bh, i] or (math.isinf(g) and math.isinf(gap[bh, i]))
    # a landmark equal to a duplicated key direction: force the tie to straddle the cut
    lq2 = np.zeros((1, 2, 4, 64))
    lq2[0, 0, :] = _f64(k[0, 0, 3])
    _, e, gap = o.scan(lq2, k, v, 2)
    s = o.scores(lq2, k, 0, 0).tolist()
    sel, _ = _brute_topk(s, 2)
    assert e[0, 0].tolist() == sel and sel == [3, 7]


def pin_lv_textbook(o):
    q, k, v = _rand((1, 3, 257, 64), 17, 0), _rand((1, 3, 257, 64), 17, 1, 2.0), _rand((1, 3, 257, 64), 17, 2)
    lq = o.landmarks(q, 0, 0, 5) * 4.0  # sharper softmax
    lv, _, _ = o.scan(lq, k, v, 3, want_idx=False, want_gap=False)
    K, V = _f64(k).reshape(3, 257, 64), _f64(v).reshape(3, 257, 64)
    for bh in range(3):
        w = softmax(lq.reshape(3, 5, 64)[bh] @ K[bh].T / 8.0, axis=-1)
        assert np.max(np.abs(lv[bh] - w @ V[bh])) < 1e-12


def pin_route_argmax(o):
    q = _rand((2, 2, 150, 64), 18, 0)
    lq = o.landmarks(q, 0, 0, 6)
    r, g = o.route(q, lq)
    t = np.einsum("bhnc,bhic->bhni", _f64(q), lq) / 8.0
    assert np.array_equal(r.reshape(2, 2, 150), np.argmax(t, axis=-1))
    ts = np.sort(t, axis=-1)
    assert np.max(np.abs(g.reshape(2, 2, 150) - (ts[..., -1] - ts[..., -2]))) < 1e-12
    which = np.array([0, 151, 599])
    r2, _ = o.route(q, lq, which=which)
    assert np.array_equal(r2, r.reshape(-1)[which])


def pin_attention_k_equals_n(o):
    N, m = 60, 4
    q, k, v = _rand((1, 2, N, 64), 19, 0, 2.0), _rand((1, 2, N, 64), 19, 1), _rand((1, 2, N, 64), 19, 2)
    r = o.forward(q, k, v, 0, 0, m, N)
    assert np.array_equal(r["expert_idx"][0], np.broadcast_to(np.arange(N), (2, m, N)))
    Q, K, V = _f64(q)[0], _f64(k)[0], _f64(v)[0]
    for h in range(2):
        keys = np.concatenate([r["lq"][0, h], K[h]])
        vals = np.concatenate([r["lv"][0, h], V[h]])
        w = softmax(Q[h] @ keys.T / 8.0, axis=-1)
        assert np.max(np.abs(r["out"][0, h] - w @ vals)) < 1e-12
    # with every key in every expert the routes cannot matter
    other = (r["route"] + 1) % m
    out2, _ = o.attend(q, r["lq"], r["lv"], k, v, r["expert_idx"], other)
    assert np.max(np.abs(out2 - r["out"].reshape(2, N, 64))) < 1e-12


def pin_routing_only(o):
    """The routing-only ablation (no shared pairs): with k = N every query
    attends to all keys, so the output is plain softmax attention over K, V
    (whatever the routes); with k < N it is softmax attention over the routed
    expert's keys alone, and its weights sum to 1."""
    N, m = 60, 4
    q, k, v = _rand((1, 2, N, 64), 23, 0, 2.0), _rand((1, 2, N, 64), 23, 1), _rand((1, 2, N, 64), 23, 2)
    r = o.forward(q, k, v, 0, 0, m, N, shared=False)
    Q, K, V = _f64(q)[0], _f64(k)[0], _f64(v)[0]
    for h in range(2):
        w = softmax(Q[h] @ K[h].T / 8.0, axis=-1)
        assert np.max(np.abs(r["out"][0, h] - w @ V[h])) < 1e-12
    assert np.max(np.abs(r["wsum"] - 1.0)) < 1e-12
    kk = 7
    r = o.forward(q, k, v, 0, 0, m, kk, shared=False)
    for h in range(2):
        for n in (0, 17, 59):
            sel = r["expert_idx"][0, h, r["route"][0, h, n]]
            w = softmax(Q[h, n] @ K[h, sel].T / 8.0)
            assert np.max(np.abs(r["out"][0, h, n] - w @ V[h, sel])) < 1e-12
    # the shared branch does change the result
    full = o.forward(q, k, v, 0, 0, m, kk)
    assert np.max(np.abs(full["out"] - r["out"])) > 1e-3


def pin_route_multi(o):
    """Top-s routes: the first s entries of a stable descending sort of the
    logits (equal logits keep index order), and the s-th/(s+1)-th margin."""
    q = _rand((2, 2, 150, 64), 31, 0)
    lq = o.landmarks(q, 0, 0, 9)
    lq[:, :, 6] = lq[:, :, 2]  # an exact tie between landmarks 2 and 6 for every query
    t = np.einsum("bhnc,bhic->bhni", _f64(q), lq) / 8.0
    order = np.argsort(-t, axis=-1, kind="stable")
    ts = -np.sort(-t, axis=-1)
    for s_ in (1, 2, 3, 9):
        r, g = o.route_multi(q, lq, s_)
        assert np.array_equal(r.reshape(2, 2, 150, s_), order[..., :s_])
        want = ts[..., s_ - 1] - ts[..., s_] if s_ < 9 else np.full((2, 2, 150), np.inf)
        assert np.all(g.reshape(2, 2, 150) == want) or np.max(np.abs(g.reshape(2, 2, 150) - want)) < 1e-12
    # where landmark 2 or 6 is taken and the other falls inside the cut too,
    # 2 comes first
    r, _ = o.route_multi(q, lq, 9)
    pos = {i: np.argmax(r == i, axis=-1) for i in (2, 6)}
    assert np.all(pos[2] < pos[6])
    r1, _ = o.route_multi(q, lq, 1)
    r0, _ = o.route(q, lq)
    assert np.array_equal(r1[..., 0], r0)


def pin_attend_multi_union(o):
    """s experts per query: one softmax over the m shared pairs and the set
    union of the s experts' keys, computed here by brute force (Python sets,
    numpy softmax). The inputs make the experts overlap, so counting a shared
    key twice would fail."""
    N, m, kk, s_ = 48, 6, 8, 3
    q, k, v = synth.make_inputs(dict(B=1, H=2, N=N, d=64, grid_h=0, grid_w=0, m=m, k=kk, recipe="clusters",
                                     clusters=3))
    r = o.forward_multi(q, k, v, 0, 0, m, kk, s_)
    Q, K, V = _f64(q)[0], _f64(k)[0], _f64(v)[0]
    overlaps = 0
    for h in range(2):
        for n in range(N):
            union = sorted(set(int(j) for u in range(s_) for j in r["expert_idx"][0, h, r["route"][0, h, n, u]]))
            overlaps += len(union) < s_ * kk
            keys = np.concatenate([r["lq"][0, h], K[h, union]])
            vals = np.concatenate([r["lv"][0, h], V[h, union]])
            w = softmax(keys @ Q[h, n] / 8.0)
            assert np.max(np.abs(r["out"][0, h, n] - w @ vals)) < 1e-12
    assert overlaps > N // 2, overlaps
    assert np.max(np.abs(r["wsum"] - 1.0)) < 1e-12


def pin_multi_reductions(o):
    """s = 1 is the one-expert forward pass; s = m with k = N takes every key
    once, which is plain softmax attention over [Lq; K] with values [LV; V]."""
    q, k, v = synth.make_inputs("tiny")
    one = o.forward(q, k, v, 14, 14, 25, 25)
    mul = o.forward_multi(q, k, v, 14, 14, 25, 25, 1)
    assert np.array_equal(mul["route"][..., 0], one["route"])
    assert np.max(np.abs(mul["out"] - one["out"])) < 1e-12
    N, m = 40, 4
    q, k, v = _rand((1, 2, N, 64), 37, 0, 2.0), _rand((1, 2, N, 64), 37, 1), _rand((1, 2, N, 64), 37, 2)
    r = o.forward_multi(q, k, v, 0, 0, m, N, m)
    Q, K, V = _f64(q)[0], _f64(k)[0], _f64(v)[0]
    for h in range(2):
        w = softmax(Q[h] @ np.concatenate([r["lq"][0, h], K[h]]).T / 8.0, axis=-1)
        assert np.max(np.abs(r["out"][0, h] - w @ np.concatenate([r["lv"][0, h], V[h]]))) < 1e-12


def pin_grad_forward_matches(o):
    """The differentiable restatement of the forward pass used for gradients
    (oracle/mita_grad.py, torch float64) gives the C++ oracle's outputs for
    the C++ oracle's own experts and routes, 1-D and 2-D."""
    from oracle import mita_grad

    for cfg in ("tiny", dict(B=1, H=2, N=300, d=64, grid_h=0, grid_w=0, m=7, k=11, recipe="iid")):
        c = synth.CONFIGS[cfg] if isinstance(cfg, str) else cfg
        q, k, v = synth.make_inputs(c)
        r = o.forward(q, k, v, c["grid_h"], c["grid_w"], c["m"], c["k"])
        out = mita_grad.forward(o, q, k, v, c["grid_h"], c["grid_w"], c["m"], r["expert_idx"], r["route"])
        assert np.max(np.abs(out - r["out"])) < 1e-12


def pin_grad_finite_differences(o):
    """Gradients of the restated forward pass against central finite
    differences (torch.autograd.gradcheck) on a small problem with fixed,
    overlapping experts and every expert routed to."""
    import torch

    from oracle import mita_grad

    rng = np.random.default_rng(3)
    N, d, m, kk = 12, 4, 3, 5
    W = mita_grad.pooling_matrix(o, N, 0, 0, m)
    eidx = np.sort(np.stack([rng.choice(N, kk, replace=False) for _ in range(m)]), axis=1)[None]
    route = (np.arange(N) % m)[None]
    Q, K, V = (torch.from_numpy(rng.standard_normal((1, N, d))).requires_grad_(True) for _ in range(3))
    assert torch.autograd.gradcheck(lambda a, b, c: mita_grad.forward_fixed(W, a, b, c, eidx, route), (Q, K, V),
                                    eps=1e-6, atol=1e-7, rtol=1e-6)


def pin_weights_sum_to_one(o):
    q, k, v = synth.make_inputs("tiny")
    r = o.forward(q, k, v, 14, 14, 25, 25)
    assert np.max(np.abs(r["wsum"] - 1.0)) < 1e-12


def pin_permutation(o):
    N = 128
    q, k, v = _rand((1, 2, N, 64), 20, 0), _rand((1, 2, N, 64), 20, 1), _rand((1, 2, N, 64), 20, 2)
    rng = np.random.default_rng(5)
    pi = rng.permutation(N)
    kp, vp = k[:, :, pi], v[:, :, pi]  # row j of the permuted inputs is row pi[j]
    a = o.forward(q, k, v, 0, 0, 8, 10)
    b = o.forward(q, kp, vp, 0, 0, 8, 10)
    inv = np.argsort(pi)
    mapped = np.sort(inv[a["expert_idx"]], axis=-1)  # old key j now sits at inv[j]
    assert np.array_equal(mapped, b["expert_idx"])
    assert np.array_equal(a["route"], b["route"])
    assert np.max(np.abs(a["lv"] - b["lv"])) < 1e-12
    assert np.max(np.abs(a["out"] - b["out"])) < 1e-12


def pin_hand_example(o):
    """N=4 tokens, d=2, 1-D windows of 2 (m=2), k=1; tau = 1/sqrt(2).

    Q = (2,0),(0,0),(0,4),(0,0) -> Lq_0 = (1,0), Lq_1 = (0,2).
    K = (1,0),(0,1),(-1,0),(0,0);  V = (1,0),(0,1),(0,0),(0,0).
    Landmark 0 logits (t,0,-t,0): expert {0}, gap t,
        LV_0 = (e^t, 1) / (e^t + e^-t + 2).
    Landmark 1 logits (0,2t,0,0): expert {1}, gap 2t,
        LV_1 = (1, e^2t) / (3 + e^2t).
    Routes: q0 -> 0 (margin 2t); q1, q3 tie at 0 -> 0 (margin 0); q2 -> 1 (8t).
    Outputs (one softmax over [Lq_0, Lq_1, routed key]):
        q0: logits (2t, 0, 2t)  -> (e^2t LV_0 + LV_1 + e^2t v0) / (2 e^2t + 1)
        q1, q3: all 0           -> (LV_0 + LV_1 + v0) / 3
        q2: logits (0, 8t, 4t)  -> (LV_0 + e^8t LV_1 + e^4t v1) / (1 + e^8t + e^4t)
    """
    t = 1.0 / math.sqrt(2.0)
    bf = lambda rows: synth.f64_to_bf16(np.array(rows, dtype=np.float64)).reshape(1, 1, 4, 2)
    q = bf([[2, 0], [0, 0], [0, 4], [0, 0]])
    k = bf([[1, 0], [0, 1], [-1, 0], [0, 0]])
    v = bf([[1, 0], [0, 1], [0, 0], [0, 0]])
    r = o.forward(q, k, v, 0, 0, 2, 1)
    e = math.exp
    lv0 = np.array([e(t), 1.0]) / (e(t) + e(-t) + 2)
    lv1 = np.array([1.0, e(2 * t)]) / (3 + e(2 * t))
    v0, v1 = np.array([1.0, 0.0]), np.array([0.0, 1.0])
    assert np.array_equal(r["lq"][0, 0], [[1.0, 0.0], [0.0, 2.0]])
    assert r["expert_idx"][0, 0].tolist() == [[0], [1]]
    assert np.allclose(r["gap"][0, 0], [t, 2 * t], rtol=0, atol=1e-15)
    assert np.allclose(r["lv"][0, 0], [lv0, lv1], rtol=0, atol=1e-15)
    assert r["route"][0, 0].tolist() == [0, 0, 1, 0]
    assert np.allclose(r["rgap"][0, 0], [2 * t, 0, 8 * t, 0], rtol=0, atol=1e-14)
    want = np.array([
        (e(2 * t) * lv0 + lv1 + e(2 * t) * v0) / (2 * e(2 * t) + 1),
        (lv0 + lv1 + v0) / 3,
        (lv0 + e(8 * t) * lv1 + e(4 * t) * v1) / (1 + e(8 * t) + e(4 * t)),
        (lv0 + lv1 + v0) / 3,
    ])
    assert np.max(np.abs(r["out"][0, 0] - want)) < 1e-14


ALL_PINS = [
    pin_grad_forward_matches,
    pin_grad_finite_differences,
    pin_route_multi,
    pin_attend_multi_union,
    pin_multi_reductions,
    pin_routing_only,
    pin_window_tables,
    pin_landmarks_adaptive_pool,
    pin_landmarks_special,
    pin_scores,
    pin_topk_bruteforce,
    pin_lv_textbook,
    pin_route_argmax,
    pin_attention_k_equals_n,
    pin_weights_sum_to_one,
    pin_permutation,
    pin_hand_example,
]
