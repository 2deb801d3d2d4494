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
