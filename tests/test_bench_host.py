"""Host-side accounting of bench.py (no GPU): the algorithmic FLOPs and bytes
behind every roofline fraction, the roofline time itself, the committed ncu
traffic lookup and the tile-plan predicate, each against numbers worked out
by hand for the Mixtral shape (hidden 4096, expert width 14336, 8 experts,
top-2)."""
import json
import os

import pytest

import bench

D, FFN, E, K = 4096, 14336, 8, 2
EXPERT_BYTES = 3 * D * FFN * 2  # one expert's W1, W3, W2 in bf16: 352,321,536


def test_layer_flops_per_token():
    """6 d ffn FLOPs per expert row (three d x ffn products, 2 FLOPs per
    multiply-add), two rows per token, plus 2 d E for the router."""
    flops, _ = bench.algorithmic(1, D, FFN, E, K, n_touched=2)
    assert flops == 2 * 6 * D * FFN + 2 * D * E
    assert flops == 704_643_072 + 65_536


def test_layer_bytes_decode():
    """Decode T=16 touching all 8 experts: the whole layer's weights once,
    W_g, x in, out, fp32 logits."""
    _, b = bench.algorithmic(16, D, FFN, E, K, n_touched=8)
    assert EXPERT_BYTES == 352_321_536
    assert b == 8 * EXPERT_BYTES + D * E * 2 + 2 * 16 * D * 2 + 16 * E * 4
    assert b == 2_818_900_480


def test_layer_capacity_rows_count_kept_rows_only():
    f_all, _ = bench.algorithmic(100, D, FFN, E, K, n_touched=8)
    f_cap, _ = bench.algorithmic(100, D, FFN, E, K, n_touched=8, rows=150)
    assert f_all - f_cap == 50 * 6 * D * FFN


def test_roofline_time_decode_and_prefill():
    """max(bytes / HBM, FLOPs / tensor peak) with the measured peaks: decode
    is HBM-bound (435.1 us), prefill T=4096 tensor-bound (1643 us)."""
    hbm, tc = 6478.9e9, 1756.8e12
    f, b = bench.algorithmic(16, D, FFN, E, K, n_touched=8)
    assert b / hbm > f / tc
    assert b / hbm * 1e6 == pytest.approx(435.09, abs=0.01)
    f, b = bench.algorithmic(4096, D, FFN, E, K, n_touched=8)
    assert f / tc > b / hbm
    assert f / tc * 1e6 == pytest.approx(1643.1, abs=0.5)


def test_gate_up_launch_accounting():
    """Gate/up GEMM at decode: W1 and W3 of 8 experts, 32 grouped rows in,
    32 hidden rows out."""
    f, b = bench.gemm1_algorithmic(32, D, FFN, 8)
    assert f == 4 * 32 * D * FFN
    assert b == 8 * 2 * D * FFN * 2 + 32 * D * 2 + 32 * FFN * 2 == 1_880_227_840


def test_backward_accounting():
    """16 T k d ffn FLOPs (gate/up again 4, Z 2, dX 4, three weight gradients
    6) plus 4 T d E for the router; bytes: W1/W3 twice, W2 once, fp32 weight
    gradients of every expert, x, dout, dx, W_g and its gradient."""
    f, b = bench.backward_algorithmic(4096, D, FFN, E, K, n_touched=8)
    assert f == 7_697_118_265_344
    assert b == 8 * 5 * D * FFN * 2 + 8 * 3 * D * FFN * 4 + 3 * 4096 * D * 2 + E * D * 6


def test_traffic_lookup_follows_the_kernel_sources(monkeypatch):
    """ncu traffic is reported only for the kernel sources it was taken on."""
    path = os.path.join(bench.ROOT, "profiles", "ncu_traffic.json")
    with open(path) as f:
        rec = json.load(f)
    ent = rec["gate_up_decode"]
    assert ent["bytes_per_launch"] == ent["dram_bytes_read"] + ent["dram_bytes_write"]
    if ent["source_hash"] == bench.gemm_source_hash():
        assert bench.recorded_traffic("gate_up_decode") == ent["bytes_per_launch"]
    monkeypatch.setattr(bench, "gemm_source_hash", lambda: "0" * 16)
    assert bench.recorded_traffic("gate_up_decode") is None
    assert bench.recorded_traffic("no such kernel") is None


def test_pair_plan_predicate(monkeypatch):
    """CTA pairs from 128 rows per expert on average (T = 512 at top-2 of 8)."""
    monkeypatch.delenv("MOE_PLAN_WIDE", raising=False)
    monkeypatch.delenv("MOE_PLAN_PAIR", raising=False)
    assert not bench.uses_pairs(511, K, E)
    assert bench.uses_pairs(512, K, E)
    monkeypatch.setenv("MOE_PLAN_PAIR", "0")
    assert not bench.uses_pairs(4096, K, E)


def test_config_is_the_same_for_both_arms():
    """Both arms print config_record(...) of the same workload: the shape and
    the workload's name only, nothing a run observes (routing)."""
    import argparse
    ns = argparse.Namespace(T=0, E=0, k=0)
    for name in ("decode", "prefill", "skewed"):
        cfg, over = bench.workload_cfg(ns, name)
        a = bench.config_record(name, cfg, over, 1)
        b = bench.config_record(name, dict(cfg), list(over), 1)
        assert a == b
        assert set(a) == {"workload", "T", "d", "ffn", "E", "k", "tokens_per_gpu",
                          "parallelism", "l2"}
        assert (a["d"], a["ffn"], a["E"], a["k"]) == (D, FFN, E, K)
    cfg, over = bench.workload_cfg(argparse.Namespace(T=1024, E=0, k=0), "decode")
    assert cfg["T"] == 1024 and over == ["T=1024"]
    assert "T=1024" in bench.config_record("decode", cfg, over, 1)["workload"]
