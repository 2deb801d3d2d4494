"""The library's device-side status and its workspace, on a GPU.

* The bounded-wait path: mita_selftest_wait runs a kernel whose wait nothing
  completes; the wait gives up after its limit, mita_sync_status reports
  MITA_ERR_TIMEOUT once and MITA_OK after that, and the next forward pass on
  the same stream is exact again. Nothing hangs, traps or faults.
* A pending non-timeout code (mita_backward's index check) does not affect a
  forward pass enqueued after it on the same stream.
* The workspace grows in stream order: a call that needs a larger workspace,
  enqueued behind a long stretch of work on the same stream, returns without
  waiting for that work, and every result on that stream matches the oracle.
"""
import time

import numpy as np
import pytest

import parity
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch

    import mixture_top_forward_gb300 as M

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    M.load(build_if_missing=False)


def _stage(stream, q, k, v):
    """Device copies of q, k, v, made on `stream` (a torch stream)."""
    import torch

    with torch.cuda.stream(stream):
        return parity.to_device(q), parity.to_device(k), parity.to_device(v)


def _forward_on(stream, dev, gh, gw, m, kk):
    """mita_forward_aux's outputs for the device inputs `dev` = (Q, K, V),
    enqueued on `stream` (a torch stream); the outputs are made on that
    stream too, and nothing here waits for it."""
    import torch

    import mixture_top_forward_gb300 as M

    Q, K, V = dev
    with torch.cuda.stream(stream):
        B, H, N, d = Q.shape
        out = torch.empty_like(Q)
        e = torch.empty((B, H, m, kk), dtype=torch.int32, device="cuda")
        r = torch.empty((B, H, N), dtype=torch.int32, device="cuda")
        lq = torch.empty((B, H, m, d), dtype=torch.float32, device="cuda")
        lv = torch.empty_like(lq)
    lib = M.load()
    rc = lib.mita_forward_aux(Q.data_ptr(), K.data_ptr(), V.data_ptr(), B, H, N, d, gh, gw, m, kk, out.data_ptr(),
                              e.data_ptr(), r.data_ptr(), lq.data_ptr(), lv.data_ptr(), stream.cuda_stream)
    assert rc == 0, M.mita_last_error()
    return dict(keep=(Q, K, V), out=out, e=e, r=r, lq=lq, lv=lv)


def _as_gpu_result(res):
    import torch

    out = synth.bf16_to_f64(res["out"].view(torch.int16).cpu().numpy().view(np.uint16))
    return dict(out=out, expert_idx=res["e"].cpu().numpy(), route=res["r"].cpu().numpy(),
                lq=res["lq"].cpu().numpy().astype(np.float64), lv=res["lv"].cpu().numpy().astype(np.float64))


def test_timeout_path_reports_and_recovers(orc):
    import torch

    import mixture_top_forward_gb300 as M

    s = torch.cuda.Stream()
    assert M.mita_sync_status(s) == 0
    M.mita_selftest_wait(2000, stream=s)  # 2 ms
    assert M.mita_sync_status(s) == M.MITA_ERR_TIMEOUT
    assert "wait gave up" in M.mita_last_error()
    assert M.mita_sync_status(s) == 0  # reported once, then cleared
    q, k, v = synth.make_inputs("tiny")
    res = _forward_on(s, _stage(s, q, k, v), 14, 14, 25, 25)
    assert M.mita_sync_status(s) == 0
    print(parity.full_parity(orc, q, k, v, 14, 14, 25, 25, gpu=_as_gpu_result(res)))


def test_selftest_rejects_bad_limits():
    import mixture_top_forward_gb300 as M

    for bad in (0, -5, 2000001):
        with pytest.raises(M.MitaError) as ex:
            M.mita_selftest_wait(bad)
        assert ex.value.code == M.MITA_ERR_INVALID_ARG


def test_pending_index_error_does_not_poison_the_forward_pass(orc):
    """mita_backward flags an out-of-range route in the stream's status word;
    a forward pass enqueued after it (no mita_sync_status in between) must
    still run to completion and match the oracle."""
    import torch

    import mixture_top_forward_gb300 as M

    s = torch.cuda.Stream()
    q, k, v = synth.make_inputs("seg1024")
    gh, gw, m, kk = 32, 32, 49, 49
    dev = _stage(s, q, k, v)
    first = _forward_on(s, dev, gh, gw, m, kk)
    with torch.cuda.stream(s):
        dO = first["keep"][0].clone()
        bad = first["r"].clone()
        bad[0, 0, 5] = m  # out of range
        M.mita_backward(*first["keep"], dO, gh, gw, m, kk, first["e"], bad, stream=s)
    res = _forward_on(s, dev, gh, gw, m, kk)
    s.synchronize()
    print(parity.full_parity(orc, q, k, v, gh, gw, m, kk, gpu=_as_gpu_result(res)))
    assert M.mita_sync_status(s) == M.MITA_ERR_INVALID_ARG
    assert M.mita_sync_status(s) == 0


def test_workspace_grows_in_stream_order(orc):
    """On a fresh workspace: a small problem, then ~0.2 s
    of matrix products, then a larger problem whose workspace must grow, then
    the small one again. The growing call returns long before the products
    finish (no host synchronisation), and all three results are exact."""
    import torch

    import mixture_top_forward_gb300 as M

    torch.cuda.synchronize()
    M.mita_release_workspace()  # torch hands out pooled stream handles: start every workspace afresh
    s = torch.cuda.Stream()
    small = ("tiny", 14, 14, 25, 25)
    large = ("seg1600", 40, 40, 49, 49)
    need_small = M.mita_workspace_bytes(1, 1, 196, 64, 14, 14, 25, 25)
    c = synth.CONFIGS["seg1600"]
    need_large = M.mita_workspace_bytes(c["B"], c["H"], c["N"], 64, 40, 40, 49, 49)
    assert need_large > 2 * need_small
    data = {n: synth.make_inputs(n) for n in ("tiny", "seg1600")}
    # inputs staged first: a copy from pageable host memory would wait for the stream
    dev = {n: _stage(s, *data[n]) for n in data}
    with torch.cuda.stream(s):
        a = torch.randn(8192, 8192, device="cuda", dtype=torch.bfloat16)
    r1 = _forward_on(s, dev["tiny"], *small[1:])
    s.synchronize()
    with torch.cuda.stream(s):
        for _ in range(300):  # ~1 TFLOP each
            a = a @ a
            a = a / a.abs().amax().clamp(min=1.0)
    t0 = time.perf_counter()
    r2 = _forward_on(s, dev["seg1600"], *large[1:])
    t_call = time.perf_counter() - t0
    t1 = time.perf_counter()
    r3 = _forward_on(s, dev["tiny"], *small[1:])
    s.synchronize()
    t_gpu = time.perf_counter() - t1 + t_call
    assert M.mita_sync_status(s) == 0
    # the growing call returned well before the stream drained
    assert t_call < 0.5 * t_gpu, (t_call, t_gpu)
    for (name, gh, gw, m, kk), res in ((small, r1), (large, r2), (small, r3)):
        q, k, v = data[name]
        print(name, parity.full_parity(orc, q, k, v, gh, gw, m, kk, gpu=_as_gpu_result(res)))
