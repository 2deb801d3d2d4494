"""The C-ABI library on the host: it loads, exports every function the header
declares, and rejects bad arguments before touching a device."""
import ctypes

import pytest

import mixture_top_forward_gb300 as M

FAKE = 0x100000  # 16-byte aligned, never dereferenced: validation fails first


@pytest.fixture(scope="module")
def lib():
    M.build()
    return M.load()


def test_exports_every_declared_function(lib):
    names = M.declared_functions()
    assert {"mita_forward", "mita_forward_aux", "mita_forward_host", "mita_last_error",
            "mita_release_workspace"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def _fwd(lib, B=1, H=1, N=196, d=64, gh=14, gw=14, m=25, k=25, q=FAKE, kp=FAKE, v=FAKE, out=FAKE, e=FAKE, r=FAKE):
    return lib.mita_forward(q, kp, v, B, H, N, d, gh, gw, m, k, out, e, r, None)


@pytest.mark.parametrize("kw,code", [
    (dict(d=65), M.MITA_ERR_UNSUPPORTED),
    (dict(d=128), M.MITA_ERR_UNSUPPORTED),
    (dict(m=0), M.MITA_ERR_INVALID_ARG),
    (dict(m=197), M.MITA_ERR_INVALID_ARG),
    (dict(k=0), M.MITA_ERR_INVALID_ARG),
    (dict(k=197), M.MITA_ERR_INVALID_ARG),
    (dict(m=24), M.MITA_ERR_UNSUPPORTED),            # non-square m with a 2-D grid
    (dict(gh=14, gw=13), M.MITA_ERR_INVALID_ARG),     # grid does not tile N
    (dict(gh=0, gw=14), M.MITA_ERR_INVALID_ARG),
    (dict(N=0), M.MITA_ERR_INVALID_ARG),
    (dict(B=-1), M.MITA_ERR_INVALID_ARG),
    (dict(N=4096, gh=0, gw=0, m=1025), M.MITA_ERR_UNSUPPORTED),
    (dict(N=4096, gh=0, gw=0, k=1025), M.MITA_ERR_UNSUPPORTED),
    (dict(q=0), M.MITA_ERR_INVALID_ARG),
    (dict(out=0), M.MITA_ERR_INVALID_ARG),
    (dict(q=FAKE + 8), M.MITA_ERR_INVALID_ARG),      # misaligned
])
def test_rejects_bad_arguments(lib, kw, code):
    assert _fwd(lib, **kw) == code
    assert M.mita_last_error() != ""


def test_empty_problem_is_a_no_op(lib):
    assert _fwd(lib, B=0) == M.MITA_OK
    assert _fwd(lib, H=0, q=0, out=0) == M.MITA_OK


def test_workspace_bytes(lib):
    assert M.mita_workspace_bytes(1, 1, 196, 64, 14, 14, 25, 25) > 0
    assert M.mita_workspace_bytes(1, 1, 196, 65, 14, 14, 25, 25) == 0
    small = M.mita_workspace_bytes(1, 8, 65536, 64, 0, 0, 256, 256)
    big = M.mita_workspace_bytes(1, 8, 1 << 20, 64, 0, 0, 256, 256)
    assert 0 < small < big < 2 << 30


def test_stage_names(lib):
    names = [M.mita_stage_name(i) for i in range(7)]
    assert names == ["pool", "pilot", "scan", "select", "route", "group", "expert"]
    assert M.mita_stage_name(7) is None


def _multi(lib, s, B=1, H=1, N=196, d=64, gh=14, gw=14, m=25, k=25, q=FAKE, out=FAKE):
    return lib.mita_forward_multi(q, FAKE, FAKE, B, H, N, d, gh, gw, m, k, s, out, FAKE, FAKE, None)


@pytest.mark.parametrize("kw,code", [
    (dict(s=0), M.MITA_ERR_INVALID_ARG),
    (dict(s=26), M.MITA_ERR_INVALID_ARG),               # s > m
    (dict(s=9, N=4096, gh=0, gw=0, m=64), M.MITA_ERR_INVALID_ARG),  # s > MITA_MAX_S
    (dict(s=2, d=32), M.MITA_ERR_UNSUPPORTED),
    (dict(s=2, q=0), M.MITA_ERR_INVALID_ARG),
    (dict(s=2, out=FAKE + 4), M.MITA_ERR_INVALID_ARG),  # misaligned
])
def test_multi_rejects_bad_arguments(lib, kw, code):
    assert _multi(lib, **kw) == code
    assert M.mita_last_error() != ""


def _bwd(lib, B=1, H=1, N=196, d=64, gh=14, gw=14, m=25, k=25, dO=FAKE, e=FAKE, dq=FAKE):
    return lib.mita_backward(FAKE, FAKE, FAKE, dO, B, H, N, d, gh, gw, m, k, e, FAKE, dq, FAKE, FAKE, None)


@pytest.mark.parametrize("kw,code", [
    (dict(d=128), M.MITA_ERR_UNSUPPORTED),
    (dict(m=0), M.MITA_ERR_INVALID_ARG),
    (dict(k=197), M.MITA_ERR_INVALID_ARG),
    (dict(m=24), M.MITA_ERR_UNSUPPORTED),
    (dict(dO=0), M.MITA_ERR_INVALID_ARG),
    (dict(e=0), M.MITA_ERR_INVALID_ARG),
    (dict(dq=FAKE + 8), M.MITA_ERR_INVALID_ARG),       # misaligned
])
def test_backward_rejects_bad_arguments(lib, kw, code):
    assert _bwd(lib, **kw) == code
    assert M.mita_last_error() != ""


def test_variants_empty_problem_is_a_no_op(lib):
    assert _multi(lib, 2, B=0) == M.MITA_OK
    assert _bwd(lib, B=0) == M.MITA_OK
    assert lib.mita_forward_routed(FAKE, FAKE, FAKE, 0, 1, 196, 64, 14, 14, 25, 25, FAKE, FAKE, FAKE, None) == M.MITA_OK


def _ceil(a, b):
    return -(-a // b)


@pytest.mark.parametrize("N,m,k,pilots,dense_main", [
    # N = 1M: a dense first level of 4 t = 8192 samples (t = 8 k), one
    # filtered level 16x larger (32768 = N/32, the cap), then every key
    (1 << 20, 256, 256, [(8192, 128, True), (32768, 32, False)], False),
    # 256K: the first level (8192 = N/32) is the last one
    (1 << 18, 256, 256, [(8192, 32, True)], False),
    # 64K: the dense first level is capped at N/16 = 4096 samples
    (1 << 16, 256, 256, [(4096, 16, True)], False),
    # the LRA shape: a sample could only pass one key in 8, so no pilots and
    # the main scan writes every logit and ranks whole rows
    (4096, 64, 64, [], True),
])
def test_plan_info_pilot_schedule(lib, N, m, k, pilots, dense_main):
    """The landmark scan's schedule (mita_plan_info): the pilot levels'
    sample sizes and strides, the main scan over every key, and the
    speculative threshold's rank j = ceil(2 k S / N) + 8 (S: the last pilot's
    samples), used only when below k."""
    info = M.mita_plan_info(1, 8, N, 64, 0, 0, m, k)
    assert info["levels"][:-1] == pilots
    assert info["levels"][-1] == (N, 1, dense_main)
    assert info["dense_main"] == dense_main
    if pilots:
        S = pilots[-1][0]
        j = _ceil(2 * k * S, N) + 8
        assert info["spec_j"] == (j if j < k else 0)
        # every level's keys are a strided sample of the head's N keys
        for s, stride, _ in pilots:
            assert s == _ceil(N, stride)
    else:
        assert info["spec_j"] == 0


def test_plan_info_rejects_bad_shapes(lib):
    assert M.mita_plan_info(1, 1, 196, 65, 14, 14, 25, 25) is None  # d != 64
    assert M.mita_plan_info(0, 1, 196, 64, 14, 14, 25, 25) is None  # empty


@pytest.mark.parametrize("N", [1000, 4096, 8192, 40000, 65536, 1 << 18, 1 << 20, 1 << 22])
@pytest.mark.parametrize("m,k", [(16, 16), (64, 64), (256, 256), (300, 70), (64, 1024)])
def test_plan_info_invariants(lib, N, m, k):
    """Over a sweep of shapes: each level samples keys at a stride (the
    last is the main scan over every key, stride 1), later levels sample
    more keys at smaller strides, every level holds at least k keys, the
    filtered pilot levels stay within N/32 and the dense first one within
    N/8, and the speculative rank follows j = ceil(2 k S / N) + 8 when below
    k (0 otherwise, and whenever the main scan ranks whole rows)."""
    if k > N or m > N:
        return
    info = M.mita_plan_info(1, 2, N, 64, 0, 0, m, k)
    assert info is not None
    lv = info["levels"]
    assert lv[-1][0] == N and lv[-1][1] == 1
    for (s, stride, _) in lv:
        assert s == _ceil(N, stride) and s >= min(k, N)
    for a, b in zip(lv, lv[1:]):
        assert a[0] < b[0] and a[1] > b[1]
    pilots = lv[:-1]
    for i, (s, stride, dense) in enumerate(pilots):
        assert s <= N // 8
        if i > 0:
            assert not dense and s <= N // 32
    if info["dense_main"] or not pilots:
        assert info["spec_j"] == 0
    else:
        j = _ceil(2 * k * pilots[-1][0], N) + 8
        assert info["spec_j"] == (j if j < k else 0)
