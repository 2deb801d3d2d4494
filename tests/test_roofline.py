"""The benchmark's roofline numerator against FLOP counts the pages print.

Per head, the pass costs 4 m N d FLOPs for the landmark scan (scores and the
shared-expert values) and 4 N (m+k) d for the query-expert attention; full
attention costs 4 N^2 d. Substituted into DeiT-S and ViT-S+CBT (12 layers,
embedding 384 = 6 heads x 64), the saving must turn the pages' full-attention
totals into their MiTA totals (tests/golden/cost_model.json; the pages count
multiply-accumulates)."""
import json
import os

import bench

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "cost_model.json")


def test_cost_model_reproduces_the_pages():
    for c in json.load(open(GOLDEN))["cases"]:
        D, L, N = c["embed_dim"], c["layers"], c["tokens"]
        cfg = dict(B=1, H=D // 64, N=N, m=c["m"], k=c["k"])
        mita_flops = bench.work(cfg)["total"]["flops"] * L
        full_flops = 4 * N * N * D * L
        saving_gmac = (full_flops - mita_flops) / 2 / 1e9
        assert abs(c["full_gflops"] - saving_gmac - c["mita_gflops"]) <= c["tolerance_gflops"], c["name"]


def test_bytes_formula():
    c = dict(B=1, H=8, N=1 << 20, m=256, k=256)
    w = bench.work(c)["total"]
    # Q, K, V read once and O written (4 x 128 MiB per head) plus m*k gathered K and V rows
    assert w["bytes"] == 8 * (4 * (1 << 20) * 128 + 256 * 256 * 2 * 128)
    assert w["flops"] == 8 * (4 * 256 * (1 << 20) * 64 + 4 * (1 << 20) * 512 * 64)


def test_variant_numerators():
    """The routing-only ablation's scan forms logits only (2 m N d) and its
    experts hold k keys (4 N k d); s routed experts count m + s k keys per
    query (an upper bound); s = 1 and shared are the headline numerator."""
    c = dict(B=1, H=2, N=4096, m=64, k=128)
    BH, N, m, k, d = 2, 4096, 64, 128, 64
    base = bench.work(c)
    assert bench.work(c, s=1) == base and bench.work(c, shared=True) == base
    r = bench.work(c, shared=False)
    assert r["scan"]["flops"] == BH * 2 * m * N * d
    assert r["expert"]["flops"] == BH * 4 * N * k * d
    assert r["total"]["flops"] == r["scan"]["flops"] + r["expert"]["flops"]
    for s in (2, 3):
        w = bench.work(c, s=s)
        assert w["expert"]["flops"] == BH * 4 * N * (m + s * k) * d
        assert w["total"]["flops"] == w["scan"]["flops"] + w["expert"]["flops"]
        assert w["expert"]["flops"] > base["expert"]["flops"]
