"""Parity of the CUDA path with the fp64 oracle (acceptance rule in parity.py).

Small configs and edge cases are compared element by element with the full
oracle; the large configs run in exactly the launch configuration bench.py
times (mita_forward on the whole problem) and are checked on a few heads:
every landmark's expert set and shared-expert value, and routes and outputs of
sampled queries."""
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


def _cfg_args(name):
    c = synth.CONFIGS[name]
    return c["grid_h"], c["grid_w"], c["m"], c["k"]


@pytest.mark.parametrize("name", ["tiny", "deit", "seg1024", "seg1600"])
def test_config_full_oracle(orc, name):
    q, k, v = synth.make_inputs(name)
    rep = parity.full_parity(orc, q, k, v, *_cfg_args(name))
    print(name, rep)


@pytest.mark.parametrize("name,heads,nq", [
    ("lra", (0, 131, 255), 4096),
    ("long64k", (0, 7), 8192),
    ("long256k", (0, 5), 8192),
    ("long1m", (3,), 8192),
])
def test_config_sampled(orc, name, heads, nq):
    q, k, v = synth.make_inputs(name)
    gpu = parity.run_gpu(q, k, v, *_cfg_args(name), full_out=False)
    rep = parity.sampled_parity(orc, q, k, v, *_cfg_args(name), gpu, heads, nq)
    print(name, rep)


def _rand(B, H, N, seed, scale=1.0):
    """Q and K at `scale` (sharper softmaxes), V at unit scale: outputs stay
    below 4 in magnitude, where bf16's half-ulp is below the 2e-2 bound."""
    return [synth.normal_bf16((B, H, N, 64), seed, t, scale if t < 2 else 1.0) for t in range(3)]


@pytest.mark.parametrize("B,H,N,gh,gw,m,k", [
    (2, 3, 1000, 0, 0, 7, 13),      # ragged windows and tiles
    (1, 2, 196, 14, 14, 25, 196),   # k = N: every key in every expert
    (1, 2, 196, 14, 14, 196, 3),    # m = N: one token per window
    (2, 2, 300, 0, 0, 1, 5),        # m = 1: one landmark, every route 0
    (1, 3, 777, 0, 0, 33, 1),       # k = 1
    (1, 1, 1, 0, 0, 1, 1),          # a single token
    (1, 2, 5000, 0, 0, 300, 700),   # several landmark tiles, k > 512
    (3, 1, 2500, 50, 50, 16, 1024), # 2-D 4x4 landmarks, k = MITA_MAX_K
    # one shared key list per CTA loaded by the row warps (few items per expert)
    (1, 2, 8192, 0, 0, 128, 128),   # two heads: the shared rows reload
    (2, 1, 3000, 0, 0, 96, 200),    # ragged: k not a multiple of 4, windows of 31-32
    # heads short enough for the one-kernel-per-head pass (N <= 256, m <= 32)
    (2, 2, 256, 0, 0, 32, 256),     # its largest N and m, k = N
    (1, 3, 255, 0, 0, 32, 100),     # ragged key blocks and windows
    (2, 1, 256, 16, 16, 16, 40),    # 2-D 16x16 grid onto 4x4 landmarks
    (1, 2, 129, 0, 0, 3, 7),        # a second query tile of one row
])
def test_edge_shapes(orc, B, H, N, gh, gw, m, k):
    q, kk_, v = _rand(B, H, N, 100 + N + m + k, 2.0)
    rep = parity.full_parity(orc, q, kk_, v, gh, gw, m, k)
    print(rep)


def _routed_args(name):
    """The routing-only ablation at the MiTA config's budget: each expert
    holds k' = m + k keys (the shared pairs' share goes to routed keys)."""
    gh, gw, m, k = _cfg_args(name)
    return gh, gw, m, min(m + k, synth.CONFIGS[name]["N"])


@pytest.mark.parametrize("name", ["tiny", "deit", "seg1024"])
def test_routed_config_full_oracle(orc, name):
    q, k, v = synth.make_inputs(name)
    rep = parity.full_parity(orc, q, k, v, *_routed_args(name), shared=False)
    print(name, rep)


@pytest.mark.parametrize("name,heads,nq", [
    ("long64k", (0, 7), 8192),
    ("long1m", (3,), 8192),
])
def test_routed_config_sampled(orc, name, heads, nq):
    q, k, v = synth.make_inputs(name)
    args = _routed_args(name)
    gpu = parity.run_gpu(q, k, v, *args, full_out=False, shared=False)
    rep = parity.sampled_parity(orc, q, k, v, *args, gpu, heads, nq, shared=False)
    print(name, rep)


@pytest.mark.parametrize("B,H,N,gh,gw,m,k", [
    (2, 3, 1000, 0, 0, 7, 13),      # ragged windows and tiles
    (1, 2, 196, 14, 14, 25, 196),   # k = N: full softmax attention for every query
    (2, 2, 300, 0, 0, 1, 5),        # m = 1: every query in one expert
    (1, 3, 777, 0, 0, 33, 1),       # k = 1: each output is one value row
    (1, 1, 1, 0, 0, 1, 1),          # a single token
    (3, 1, 2500, 50, 50, 16, 1024), # k = MITA_MAX_K
])
def test_routed_edge_shapes(orc, B, H, N, gh, gw, m, k):
    q, kk_, v = _rand(B, H, N, 300 + N + m + k, 2.0)
    rep = parity.full_parity(orc, q, kk_, v, gh, gw, m, k, shared=False)
    print(rep)


def test_routed_differs_from_mita(orc):
    """Same experts and routes on both entry points; the outputs differ (the
    shared pairs are gone), so the ablation is not MiTA under another name."""
    import torch

    import mixture_top_forward_gb300 as M

    q, k, v = synth.make_inputs("seg1024")
    Q, K, V = parity.to_device(q), parity.to_device(k), parity.to_device(v)
    a = M.mita_forward(Q, K, V, 32, 32, 49, 49)
    b = M.mita_forward_routed(Q, K, V, 32, 32, 49, 49)
    torch.cuda.synchronize()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    diff = (a[0].float() - b[0].float()).abs().mean().item()
    assert diff > 1e-2, diff


@pytest.mark.parametrize("name", ["seg1024", "ragged"])
def test_full_attention_comparator(orc, name):
    """The fused-SDPA baseline bench.py times is plain softmax attention: the
    oracle's routing-only mode with one landmark and k = N (every query
    attends to every key) gives the same outputs."""
    import torch

    import bench

    if name == "ragged":
        q, k, v = _rand(1, 3, 1000, 77, 2.0)
    else:
        q, k, v = synth.make_inputs(name)
    out, backend = bench.sdpa_full(parity.to_device(q), parity.to_device(k), parity.to_device(v))
    torch.cuda.synchronize()
    got = synth.bf16_to_f64(out.contiguous().view(torch.int16).cpu().numpy().view(np.uint16))
    N = q.shape[2]
    ref = orc.forward(q, k, v, 0, 0, 1, N, shared=False)["out"]
    rep = {"backend": backend}
    parity.check_outputs(got, ref, rep)
    print(name, rep)


@pytest.mark.parametrize("name,s", [("tiny", 2), ("deit", 2), ("seg1024", 3)])
def test_multi_config_full_oracle(orc, name, s):
    q, k, v = synth.make_inputs(name)
    rep = parity.full_parity_multi(orc, q, k, v, *_cfg_args(name), s)
    print(name, s, rep)


@pytest.mark.parametrize("name,s,heads,nq", [
    ("long64k", 2, (0, 7), 4096),
    ("long1m", 2, (3,), 4096),
])
def test_multi_config_sampled(orc, name, s, heads, nq):
    q, k, v = synth.make_inputs(name)
    args = _cfg_args(name)
    gpu = parity.run_gpu_multi(q, k, v, *args, s, full_out=False)
    rep = parity.sampled_parity_multi(orc, q, k, v, *args, s, gpu, heads, nq)
    print(name, rep)


@pytest.mark.parametrize("B,H,N,gh,gw,m,k,s", [
    (2, 3, 1000, 0, 0, 7, 13, 3),      # ragged windows and tiles
    (1, 2, 196, 14, 14, 25, 196, 2),   # k = N: both experts hold every key (all duplicates)
    (2, 2, 300, 0, 0, 4, 5, 4),        # s = m: every expert for every query
    (1, 1, 1, 0, 0, 1, 1, 1),          # a single token
    (3, 1, 2500, 50, 50, 16, 1024, 2), # k = MITA_MAX_K
    (1, 2, 5000, 0, 0, 300, 70, 8),    # s = MITA_MAX_S, several landmark tiles
])
def test_multi_edge_shapes(orc, B, H, N, gh, gw, m, k, s):
    q, kk_, v = _rand(B, H, N, 500 + N + m + k + s, 2.0)
    rep = parity.full_parity_multi(orc, q, kk_, v, gh, gw, m, k, s)
    print(rep)


@pytest.mark.parametrize("s", [2, 3])
def test_multi_tensor_core_clustered(orc, s):
    """Clustered keys make the experts of nearby landmarks overlap heavily, so
    the later passes mask many keys; N >= 32 m takes the tensor-core passes."""
    cfg = dict(B=2, H=2, N=8192, d=64, grid_h=0, grid_w=0, m=64, k=64, recipe="clusters", clusters=8)
    q, k, v = synth.make_inputs(cfg, seed=5)
    rep = parity.full_parity_multi(orc, q, k, v, 0, 0, 64, 64, s)
    print(s, rep)


def test_multi_s1_is_mita():
    """s = 1 through the s-expert entry point is the one-expert forward pass."""
    import torch

    import mixture_top_forward_gb300 as M

    q, k, v = synth.make_inputs("seg1024")
    Q, K, V = parity.to_device(q), parity.to_device(k), parity.to_device(v)
    a = M.mita_forward(Q, K, V, 32, 32, 49, 49)
    b = M.mita_forward_multi(Q, K, V, 32, 32, 49, 49, 1)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]) and torch.equal(a[2], b[2].reshape(a[2].shape))


def test_multi_rejects_bad_s():
    import torch

    import mixture_top_forward_gb300 as M

    Q = torch.zeros((1, 1, 64, 64), dtype=torch.bfloat16, device="cuda")
    for s in (0, 5, M_MAX_S + 1):
        with pytest.raises(M.MitaError) as ei:
            M.mita_forward_multi(Q, Q, Q, 0, 0, 4 if s == 5 else 16, 8, s)
        assert ei.value.code == M.MITA_ERR_INVALID_ARG


M_MAX_S = 8  # MITA_MAX_S in mita.h


def test_ascending_scores_force_compaction(orc):
    """Scores that grow along the sequence make every key beat the running
    threshold, so every chunk buffer overflows and compacts repeatedly."""
    B, H, N, m, k = 1, 2, 40000, 4, 64
    q = synth.normal_bf16((B, H, N, 64), 7, 0, 0.1)
    q = synth.f64_to_bf16(synth.bf16_to_f64(q) + 1.0)  # queries (and landmarks) near the all-ones direction
    ramp = np.linspace(-2.0, 2.0, N)[None, None, :, None]
    noise = synth.bf16_to_f64(synth.normal_bf16((B, H, N, 64), 7, 1, 0.01))
    kk_ = synth.f64_to_bf16(ramp + noise)
    v = synth.normal_bf16((B, H, N, 64), 7, 2)
    rep = parity.full_parity(orc, q, kk_, v, 0, 0, m, k)
    print(rep)


def test_exact_ties_go_to_lower_index(orc):
    """Duplicated key rows tie exactly; the lower index must win. With every
    row repeated 8 times, k = 12 cuts through the second-best group of ties."""
    B, H, N, m, k = 1, 1, 4096, 8, 12
    q, kk_, v = _rand(B, H, N, 31)
    kk_ = kk_.copy()
    src = np.arange(0, N, 8)
    for r in range(1, 8):  # every key row repeated 8 times in a row
        kk_[:, :, src + r] = kk_[:, :, src]
    gpu = parity.run_gpu(q, kk_, v, 0, 0, m, k)
    ora = orc.forward(q, kk_, v, 0, 0, m, k)
    # ties are exact, so each expert must be the oracle's (same tie rule)
    assert np.array_equal(gpu["expert_idx"], ora["expert_idx"])
    parity.full_parity(orc, q, kk_, v, 0, 0, m, k, gpu=gpu)


def test_all_scores_tied_in_dense_rows(orc):
    """Every key row identical: each landmark's N logits tie exactly, so its
    expert is the k lowest indices. On this short, ragged sequence the select
    ranks whole logit rows, and every key survives its threshold (the path
    that ranks the whole row)."""
    B, H, N, m, k = 1, 2, 2999, 16, 100
    q, kk_, v = _rand(B, H, N, 37)
    kk_ = np.repeat(kk_[:, :, :1], N, axis=2).copy()
    gpu = parity.run_gpu(q, kk_, v, 0, 0, m, k)
    assert np.array_equal(gpu["expert_idx"], np.broadcast_to(np.arange(k, dtype=np.int32), (B, H, m, k)))
    parity.full_parity(orc, q, kk_, v, 0, 0, m, k, gpu=gpu)


def test_empty_batch():
    import torch

    import mixture_top_forward_gb300 as M

    Q = torch.empty((0, 4, 196, 64), dtype=torch.bfloat16, device="cuda")
    out, e, r = M.mita_forward(Q, Q, Q, 14, 14, 25, 25)
    assert out.shape == Q.shape and e.shape == (0, 4, 25, 25) and r.shape == (0, 4, 196)


def test_host_entry_point_matches_device(orc):
    import torch

    import mixture_top_forward_gb300 as M

    q, k, v = synth.make_inputs("tiny")
    out_h, e_h, r_h = M.mita_forward_host(q, k, v, 14, 14, 25, 25)
    out_d, e_d, r_d = M.mita_forward(parity.to_device(q), parity.to_device(k), parity.to_device(v), 14, 14, 25, 25)
    torch.cuda.synchronize()
    assert np.array_equal(out_h, out_d.view(torch.int16).cpu().numpy().view(np.uint16))
    assert np.array_equal(e_h, e_d.cpu().numpy()) and np.array_equal(r_h, r_d.cpu().numpy())


def test_host_entry_point_pipelined_groups():
    """Large inputs go through the host entry point in head groups (copies
    overlapping the forward pass): same experts and routes as one device-side
    call on all heads, outputs within bf16 rounding (the groups' scans split
    the keys into other chunks, so LV's merge order differs)."""
    import torch

    import mixture_top_forward_gb300 as M

    q, k, v = synth.make_inputs("lra")  # 256 heads, 402 MB of inputs: 8 groups of 32 heads
    c = synth.CONFIGS["lra"]
    args = (c["grid_h"], c["grid_w"], c["m"], c["k"])
    out_h, e_h, r_h = M.mita_forward_host(q, k, v, *args)
    out_d, e_d, r_d = M.mita_forward(parity.to_device(q), parity.to_device(k), parity.to_device(v), *args)
    torch.cuda.synchronize()
    assert np.array_equal(e_h, e_d.cpu().numpy()) and np.array_equal(r_h, r_d.cpu().numpy())
    o_d = out_d.view(torch.int16).cpu().numpy().view(np.uint16)
    err = np.abs(synth.bf16_to_f64(out_h) - synth.bf16_to_f64(o_d))
    assert err.max() <= 2e-2 and err.mean() <= 2e-4


def test_repeatable(orc):
    """Two calls give bit-identical results (no order-dependent arithmetic)."""
    import torch

    import mixture_top_forward_gb300 as M

    q, k, v = synth.make_inputs("seg1024")
    Q, K, V = parity.to_device(q), parity.to_device(k), parity.to_device(v)
    a = M.mita_forward(Q, K, V, 32, 32, 49, 49)
    b = M.mita_forward(Q, K, V, 32, 32, 49, 49)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_pilot_blind_spot_forces_compaction(orc):
    """Every key at an odd index outscores every key at an even index. At
    N = 65536 the pilot samples are strided by even steps, so they see only
    the weaker half and leave a low threshold: the main scan's candidate
    buffers overflow and must compact, and the result must still be exact."""
    B, H, N, m, k = 1, 1, 65536, 4, 64
    noise = synth.bf16_to_f64(synth.normal_bf16((B, H, N, 64), 41, 0))
    q = synth.f64_to_bf16(1.0 + 0.1 * noise)
    sign = np.where(np.arange(N) % 2 == 1, 1.0, -1.0)[None, None, :, None]
    kn = synth.bf16_to_f64(synth.normal_bf16((B, H, N, 64), 41, 1))
    kk_ = synth.f64_to_bf16(0.5 * sign + 0.05 * kn)
    v = synth.normal_bf16((B, H, N, 64), 41, 2)
    rep = parity.full_parity(orc, q, kk_, v, 0, 0, m, k)
    print(rep)


def test_pilot_records_in_every_group(orc):
    """Keys at indices 32, 64, 96 (mod 128) outscore the rest. At N = 65536
    and k = 16 the first pilot level (512 samples, every 128th key) sees only
    weak ones, so the second (every 32nd key) finds three quarters of its
    samples above that threshold, in every 8-sample group: each group goes
    out as a record (64 per chunk of 512 samples, within the 96 a landmark
    may keep), the select expands them all, and the result must still be
    exact."""
    B, H, N, m, k = 1, 1, 65536, 4, 16
    noise = synth.bf16_to_f64(synth.normal_bf16((B, H, N, 64), 43, 0))
    q = synth.f64_to_bf16(1.0 + 0.1 * noise)
    idx = np.arange(N) % 128
    sign = np.where((idx == 32) | (idx == 64) | (idx == 96), 1.0, -1.0)[None, None, :, None]
    kn = synth.bf16_to_f64(synth.normal_bf16((B, H, N, 64), 43, 1))
    kk_ = synth.f64_to_bf16(0.5 * sign + 0.05 * kn)
    v = synth.normal_bf16((B, H, N, 64), 43, 2)
    rep = parity.full_parity(orc, q, kk_, v, 0, 0, m, k)
    print(rep)


def test_speculative_threshold_falls_back(orc):
    """Keys at indices 0 (mod 32), the pilot's samples at N = 65536 (one
    level of 2048 samples), outscore the rest, so the head's best keys are
    all sample keys: the speculative threshold (the sample key of rank
    2 k / 32 + 8 = 12) leaves only 12 keys above it, every landmark keeps
    fewer than k candidates, and the head is scanned again from the k-th
    best sample key; the result must still be exact."""
    B, H, N, m, k = 1, 2, 65536, 4, 64
    noise = synth.bf16_to_f64(synth.normal_bf16((B, H, N, 64), 47, 0))
    q = synth.f64_to_bf16(1.0 + 0.1 * noise)
    sign = np.where(np.arange(N) % 32 == 0, 1.0, -1.0)[None, None, :, None]
    kn = synth.bf16_to_f64(synth.normal_bf16((B, H, N, 64), 47, 1))
    kk_ = synth.f64_to_bf16(0.5 * sign + 0.05 * kn)
    v = synth.normal_bf16((B, H, N, 64), 47, 2)
    rep = parity.full_parity(orc, q, kk_, v, 0, 0, m, k)
    print(rep)


# --- mita_forward_split: the shared branch folded into the routing kernel ---
def _run_split(q, k, v, gh, gw, m, kk, full_out=True):
    """mita_forward_split's outputs; Lq and LV (not returned by that entry
    point) from mita_forward_aux, whose first two stages are the same."""
    import torch

    import mixture_top_forward_gb300 as M

    Q, K, V = parity.to_device(q), parity.to_device(k), parity.to_device(v)
    _, _, _, lq, lv = M.mita_forward_aux(Q, K, V, gh, gw, m, kk)
    out, eidx, route = M.mita_forward_split(Q, K, V, gh, gw, m, kk)
    torch.cuda.synchronize()
    assert M.mita_sync_status() == 0
    if full_out:
        out = synth.bf16_to_f64(out.view(torch.int16).cpu().numpy().view(np.uint16))
    return dict(out=out, expert_idx=eidx.cpu().numpy(), route=route.cpu().numpy(),
                lq=lq.cpu().numpy().astype(np.float64), lv=lv.cpu().numpy().astype(np.float64))


@pytest.mark.parametrize("name", ["tiny", "deit", "seg1024", "seg1600"])
def test_split_config_full_oracle(orc, name):
    q, k, v = synth.make_inputs(name)
    rep = parity.full_parity(orc, q, k, v, *_cfg_args(name), gpu=_run_split(q, k, v, *_cfg_args(name)))
    print(name, rep)


@pytest.mark.parametrize("name,heads,nq", [("lra", (0, 200), 4096), ("long64k", (0, 6), 8192)])
def test_split_config_sampled(orc, name, heads, nq):
    q, k, v = synth.make_inputs(name)
    gpu = _run_split(q, k, v, *_cfg_args(name), full_out=False)
    rep = parity.sampled_parity(orc, q, k, v, *_cfg_args(name), gpu, heads, nq)
    print(name, rep)


@pytest.mark.parametrize("B,H,N,gh,gw,m,k", [
    (2, 3, 1000, 0, 0, 7, 13),      # ragged windows and tiles, m_pad < m + 16
    (2, 2, 300, 0, 0, 1, 5),        # one landmark
    (1, 2, 4096, 0, 0, 200, 100),   # two landmark halves in the shared product
    (1, 2, 196, 14, 14, 196, 3),    # m = N
])
def test_split_edge_shapes(orc, B, H, N, gh, gw, m, k):
    q, kk_, v = _rand(B, H, N, 300 + N + m + k, 2.0)
    rep = parity.full_parity(orc, q, kk_, v, gh, gw, m, k, gpu=_run_split(q, kk_, v, gh, gw, m, k))
    print(rep)


def test_split_matches_forward():
    """Same routes and expert sets as mita_forward, outputs within the
    parity tolerances of each other."""
    import torch

    import mixture_top_forward_gb300 as M

    q, k, v = synth.make_inputs("seg1600")
    Q, K, V = parity.to_device(q), parity.to_device(k), parity.to_device(v)
    a = M.mita_forward(Q, K, V, *_cfg_args("seg1600"))
    b = M.mita_forward_split(Q, K, V, *_cfg_args("seg1600"))
    torch.cuda.synchronize()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    err = (a[0].float() - b[0].float()).abs()
    assert err.max().item() <= parity.OUT_MAX and err.mean().item() <= parity.OUT_MEAN
