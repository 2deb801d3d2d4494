"""Out-of-bounds writes on a GPU: every output buffer (out, expert_idx,
route) sits inside a larger one whose guard regions hold a fixed byte
pattern. After the call the guards must be unchanged, and the outputs must
equal those of a call with plain buffers, bit for bit. The cases cover the
forward pass's kernel paths: the fused short head, dense rows with one key
list per warpgroup, the row-loaded and the producer-loaded shared key
lists, a speculative scan after a pilot level, ragged 1-D windows and a
2-D landmark grid; each through the one-expert, routing-only and s = 2
entry points.
"""
import pytest

import parity
import synth

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes of guard on each side (a multiple of 16: outputs stay 16-byte aligned)
PATTERN = 0x5A

CASES = [
    ("fused short head", dict(B=1, H=1, N=196, gh=14, gw=14, m=25, k=25)),
    ("ragged 1-D windows", dict(B=2, H=3, N=1000, gh=0, gw=0, m=7, k=13)),
    ("dense rows, list per warpgroup", dict(B=2, H=2, N=4096, gh=0, gw=0, m=64, k=64)),
    ("2-D landmark grid", dict(B=2, H=2, N=1600, gh=40, gw=40, m=49, k=49)),
    ("pilot level, speculative scan", dict(B=1, H=2, N=65536, gh=0, gw=0, m=64, k=64)),
    ("row-loaded shared list", dict(B=1, H=2, N=16384, gh=0, gw=0, m=128, k=128)),
    ("producer-loaded shared list", dict(B=1, H=1, N=65536, gh=0, gw=0, m=16, k=128)),
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch

    import mixture_top_forward_gb300 as M

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    M.load(build_if_missing=False)


def _guarded(numel, dtype):
    """A buffer of numel elements with GUARD pattern bytes on each side; returns
    (the whole buffer, the interior view)."""
    import torch

    item = torch.empty(0, dtype=dtype).element_size()
    g = GUARD // item
    buf = torch.empty(numel + 2 * g, dtype=dtype, device="cuda")
    buf.view(torch.uint8).fill_(PATTERN)
    return buf, buf[g:g + numel]


def _guards_intact(buf):
    import torch

    b = buf.view(torch.uint8)
    return bool((b[:GUARD] == PATTERN).all()) and bool((b[-GUARD:] == PATTERN).all())


@pytest.mark.parametrize("entry", ["forward", "routed", "multi"])
@pytest.mark.parametrize("name,c", CASES, ids=[n for n, _ in CASES])
def test_outputs_stay_in_bounds(name, c, entry):
    import torch

    import mixture_top_forward_gb300 as M

    B, H, N, gh, gw, m, k = c["B"], c["H"], c["N"], c["gh"], c["gw"], c["m"], c["k"]
    s = 2 if entry == "multi" else 1
    q = synth.normal_bf16((B, H, N, 64), 61, 0)
    kk = synth.normal_bf16((B, H, N, 64), 61, 1)
    v = synth.normal_bf16((B, H, N, 64), 61, 2)
    Q, K, V = parity.to_device(q), parity.to_device(kk), parity.to_device(v)

    def call(out=None, eidx=None, route=None):
        if entry == "forward":
            return M.mita_forward(Q, K, V, gh, gw, m, k, out=out, expert_idx=eidx, route=route)
        if entry == "routed":
            return M.mita_forward_routed(Q, K, V, gh, gw, m, k, out=out, expert_idx=eidx, route=route)
        return M.mita_forward_multi(Q, K, V, gh, gw, m, k, s, out=out, expert_idx=eidx, route=route)

    ob, out = _guarded(B * H * N * 64, torch.bfloat16)
    eb, eidx = _guarded(B * H * m * k, torch.int32)
    rb, route = _guarded(B * H * N * s, torch.int32)
    rshape = (B, H, N) if s == 1 else (B, H, N, s)
    got = call(out.view(B, H, N, 64), eidx.view(B, H, m, k), route.view(*rshape))
    torch.cuda.synchronize()
    assert M.mita_sync_status() == 0, M.mita_last_error()
    for buf, what in ((ob, "out"), (eb, "expert_idx"), (rb, "route")):
        assert _guards_intact(buf), f"{name}: a write landed outside {what}"
    ref = call()
    torch.cuda.synchronize()
    assert M.mita_sync_status() == 0, M.mita_last_error()
    for a, b in zip(got, ref):
        assert torch.equal(a.reshape(-1).view(torch.int16 if a.dtype == torch.bfloat16 else a.dtype),
                           b.reshape(-1).view(torch.int16 if b.dtype == torch.bfloat16 else b.dtype))
