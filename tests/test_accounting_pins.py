"""The bench's FLOP and byte accounting against the worked examples the pages print."""

import os

import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _fixture(name):
    vals = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = (x.strip() for x in line.split("=", 1))
            vals[k] = float(v)
    return vals


def test_mla_cost_formula_section_7_2():
    """FLOPs per MTP request at 3K: 3072 x (576 + 512) x 128 x 2 x 2, giving 6.2 us per BS."""
    g = _fixture("p1_s7_2_mla_cost.txt")
    L = int(g["seq_len"])
    assert W.D_ROW == g["d_score"] and W.D_LATENT == g["d_out"] and W.NUM_HEADS == g["heads"]
    # Our count is per visible key: the first MTP token sees one key fewer (causal), so it
    # is smaller than the printed formula by exactly one key's worth of work.
    ours = W.flops([L], s_q=int(g["query_tokens"]))
    printed = L * (g["d_score"] + g["d_out"]) * g["heads"] * g["flop_per_mac"] * g["query_tokens"]
    per_key = g["flop_per_mac"] * g["heads"] * (g["d_score"] + g["d_out"])
    assert printed - ours == per_key
    us = printed / (g["peak_flops"] * g["utilisation"] * g["overlap_derate"]) * 1e6
    assert abs(us - g["printed_us_per_bs"]) < 0.05


def test_kv_memory_section_3_2_1():
    """72 requests x 4K tokens x 61 layers of 576 bf16 values is close to 20 GB."""
    g = _fixture("p1_s3_2_1_kv_memory.txt")
    per_layer = W.cache_bytes([int(g["seq_len"])] * int(g["concurrent"]))
    total_gb = per_layer * g["layers"] / 1e9
    assert abs(total_gb - g["printed_gb"]) / g["printed_gb"] < 0.05
    assert W.cache_bytes([1]) == 1152


def test_workload_shapes():
    assert W.workload("tiny").seq_lens and sorted(W.workload("tiny").seq_lens) == [1, 63, 64, 200]
    m = W.workload("mixed")
    assert m.batch == 64 and m.seq_lens.count(20480) == 26 and m.seq_lens.count(400) == 38
    t = W.workload("mtp")
    assert t.s_q == 2 and t.batch == 128 and min(t.seq_lens) >= 1024 and max(t.seq_lens) <= 8192
    assert W.cache_bytes(W.workload("uniform").seq_lens) == 64 * 4096 * 1152
