"""Parity of the CUDA backward pass (mita_backward) with the fp64 gradient
oracle (oracle/mita_grad.py), both conditioned on the experts and routes the
CUDA forward pass chose.

Bound: every element of dQ, dK, dV within 1e-2 of the largest magnitude of
that oracle gradient. Derivation: the tensor-core kernels multiply bf16
operands with fp32 accumulation. The inputs (Q, K, V, dO) are bf16 already;
what gets rounded to bf16 on the way are the softmax weights p and the
products ds = p (dP - Delta) of both attentions, and dLV (an operand of the
landmark attention's products), each by at most 2^-9 relative, and the
shared keys are the bf16 landmark queries the forward pass itself uses. So
every term of a gradient sum carries a relative error of at most about
2^-8, and the sums' errors are those of independent roundings: a few 2^-8
of the sum of the terms' magnitudes, which, for these softmax-weighted sums,
stays within a small multiple of the largest gradient magnitude. 1e-2 is
about 2.5 x 2^-8. Shapes the tensor-core kernels do not cover (m > 256, an
expert list longer than 512 keys) run in fp32 on the CUDA cores, well
inside the same bound.
"""
import numpy as np
import pytest

import parity
import synth

pytestmark = pytest.mark.gpu

RTOL_MAX = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch

    import mixture_top_forward_gb300 as M

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    M.load(build_if_missing=False)


def _run(orc, q, k, v, gh, gw, m, kk, seed=11):
    import torch

    import mixture_top_forward_gb300 as M
    from oracle import mita_grad

    B, H, N, d = q.shape
    dout = synth.normal_bf16((B, H, N, d), seed, 7)
    Q, K, V, dO = (parity.to_device(x) for x in (q, k, v, dout))
    _, eidx, route = M.mita_forward(Q, K, V, gh, gw, m, kk)
    dq, dk, dv = M.mita_backward(Q, K, V, dO, gh, gw, m, kk, eidx, route)
    torch.cuda.synchronize()
    assert M.mita_sync_status() == 0
    e, r = eidx.cpu().numpy(), route.cpu().numpy()
    ref = mita_grad.grads(orc, q, k, v, dout, gh, gw, m, e, r)
    rep = {}
    # a gradient that cancels to ~0 (a single token's dQ) keeps the rounding
    # of terms as large as the other gradients: floor the bound at 1e-2 of it
    # taken at the largest gradient magnitude of the three
    floor = 1e-2 * RTOL_MAX * max(float(np.abs(o).max()) for o in ref)
    for name, g, o in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        g = g.cpu().numpy().astype(np.float64)
        scale = float(np.abs(o).max())
        err = float(np.abs(g - o).max())
        rep[name] = (err, scale)
        assert err <= RTOL_MAX * scale + floor, f"{name}: max error {err:.3g} vs scale {scale:.3g}"
    return rep


@pytest.mark.parametrize("name", ["tiny", "seg1024"])
def test_backward_configs(orc, name):
    c = synth.CONFIGS[name]
    q, k, v = synth.make_inputs(name)
    print(name, _run(orc, q, k, v, c["grid_h"], c["grid_w"], c["m"], c["k"]))


def _rand(B, H, N, seed, scale=2.0):
    return [synth.normal_bf16((B, H, N, 64), seed, t, scale if t < 2 else 1.0) for t in range(3)]


@pytest.mark.parametrize("B,H,N,gh,gw,m,k", [
    (2, 3, 1000, 0, 0, 7, 13),       # ragged windows, key chunks and items
    (1, 2, 196, 14, 14, 25, 196),    # k = N: every key in every expert
    (2, 2, 300, 0, 0, 1, 5),         # m = 1
    (1, 1, 1, 0, 0, 1, 1),           # a single token
    (1, 2, 2500, 50, 50, 16, 1024),  # 2-D 4x4 landmarks, k = MITA_MAX_K
    (1, 2, 8192, 0, 0, 64, 64),      # many items per expert, several landmark-side chunks
    (1, 1, 3000, 0, 0, 300, 40),     # m > 256: several landmark tiles
])
def test_backward_edge_shapes(orc, B, H, N, gh, gw, m, k):
    q, kk_, v = _rand(B, H, N, 700 + N + m + k)
    print(_run(orc, q, kk_, v, gh, gw, m, k))


@pytest.mark.parametrize("heads", [(0, 5)])
def test_backward_long64k_sampled_heads(orc, heads):
    """The full long64k problem (8 heads, N = 65536, m = k = 256) through
    mita_backward, checked on whole heads against the oracle run on each head
    alone (the heads are independent problems)."""
    import torch

    import mixture_top_forward_gb300 as M
    from oracle import mita_grad

    c = synth.CONFIGS["long64k"]
    q, k, v = synth.make_inputs("long64k")
    dout = synth.normal_bf16(q.shape, 11, 7)
    Q, K, V, dO = (parity.to_device(x) for x in (q, k, v, dout))
    args = (c["grid_h"], c["grid_w"], c["m"], c["k"])
    _, eidx, route = M.mita_forward(Q, K, V, *args)
    dq, dk, dv = M.mita_backward(Q, K, V, dO, *args, eidx, route)
    torch.cuda.synchronize()
    assert M.mita_sync_status() == 0
    e, r = eidx.cpu().numpy(), route.cpu().numpy()
    got = [g.cpu().numpy().astype(np.float64) for g in (dq, dk, dv)]
    for h in heads:
        sl = (slice(0, 1), slice(h, h + 1))
        ref = mita_grad.grads(orc, q[sl], k[sl], v[sl], dout[sl], *args[:3], e[sl], r[sl])
        floor = 1e-2 * RTOL_MAX * max(float(np.abs(o).max()) for o in ref)
        for name, g, o in zip(("dQ", "dK", "dV"), got, ref):
            scale = float(np.abs(o).max())
            err = float(np.abs(g[sl] - o).max())
            print(h, name, err, scale)
            assert err <= RTOL_MAX * scale + floor, f"head {h} {name}: max error {err:.3g} vs scale {scale:.3g}"


def test_backward_rejects_bad_routes():
    """A route outside [0, m) is left out and reported by mita_sync_status."""
    import torch

    import mixture_top_forward_gb300 as M

    q, k, v = _rand(1, 1, 256, 9)
    Q, K, V = (parity.to_device(x) for x in (q, k, v))
    _, eidx, route = M.mita_forward(Q, K, V, 0, 0, 4, 8)
    route[0, 0, 5] = 4
    M.mita_backward(Q, K, V, Q, 0, 0, 4, 8, eidx, route)
    torch.cuda.synchronize()
    assert M.mita_sync_status() == M.MITA_ERR_INVALID_ARG
    assert M.mita_sync_status() == 0  # the report clears the status
