"""mita_forward_noalloc: the forward pass for callers that may not allocate
device memory (a framework that hands out all device memory from its own
pool, or a latency-critical loop that cannot take the device-wide
synchronisation of cudaMalloc/cudaFree). It runs on a static device scratch
array instead of the library's workspace.

The checks: through the C ABI, two calls in a row give the same routes and
expert sets as mita_forward and outputs within the parity tolerances
(max-abs 2e-2, mean-abs 2e-3); the second call starts from whatever the
first left in the shared array, and a second shape follows the first. A
shape too large for the array is refused before anything runs. This file is
collected last on purpose and depends on no other test."""
import pytest

import parity
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixture_top_forward_gb300 as M

    M.load(build_if_missing=False)
    return M


@pytest.mark.parametrize("name", ["deit", "seg1600", "tiny"])
def test_noalloc_matches_forward_on_two_calls(M, name):
    """Also checks the property the entry point exists for: with every buffer
    made beforehand and the library's own workspace released, two calls leave
    the device's free memory (cudaMemGetInfo) exactly as it was. One call
    runs first, since the static array itself is placed on the device when
    the library's module is first used there."""
    import torch

    c = synth.CONFIGS[name]
    q, k, v = synth.make_inputs(c)
    Q, K, V = parity.to_device(q), parity.to_device(k), parity.to_device(v)
    args = (c["grid_h"], c["grid_w"], c["m"], c["k"])
    ref_out, ref_e, ref_r = M.mita_forward(Q, K, V, *args)
    out = torch.empty_like(Q)
    e = torch.empty_like(ref_e)
    r = torch.empty_like(ref_r)
    M.mita_forward_noalloc(Q, K, V, *args, out=out, expert_idx=e, route=r)
    torch.cuda.synchronize()
    M.mita_release_workspace()
    for _ in range(2):
        out.fill_(0)
        e.fill_(-1)
        r.fill_(-1)
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        M.mita_forward_noalloc(Q, K, V, *args, out=out, expert_idx=e, route=r)
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0
        assert torch.equal(e, ref_e)
        assert torch.equal(r, ref_r)
        err = (out.float() - ref_out.float()).abs()
        assert err.max().item() <= parity.OUT_MAX and err.mean().item() <= parity.OUT_MEAN
    assert M.mita_sync_status() == 0


def test_noalloc_refuses_shapes_beyond_its_scratch(M):
    import ctypes

    lib = M.load()
    c = synth.CONFIGS["long64k"]
    need = M.mita_workspace_bytes(c["B"], c["H"], c["N"], 64, 0, 0, c["m"], c["k"])
    assert need > (64 << 20)
    p = ctypes.c_void_p(0x100000)
    rc = lib.mita_forward_noalloc(p, p, p, c["B"], c["H"], c["N"], 64, 0, 0, c["m"], c["k"], p, p, p, None)
    assert rc == M.MITA_ERR_UNSUPPORTED
    assert "MITA_NOALLOC_SCRATCH_BYTES" in M.mita_last_error()
