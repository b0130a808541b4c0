"""The benchmark's work model against the numbers the pages print and brute force."""
import json
import os

import pytest

from global_causal_gqa_gb300 import accounting as acc

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "kv_bytes.json")


def test_decode_bytes_per_token_table():
    g = json.load(open(GOLDEN))
    for row in g["decode_mib_per_token"]:
        b = acc.kv_bytes_per_token(row["L"], row["Hkv"], 128, 4096, 2048)
        assert b == row["mib"] * 2 ** 20, row


def test_capacity_table():
    g = json.load(open(GOLDEN))
    models = {
        "PLaMo 3 31B": [(8, 8, 128, 0), (56, 8, 128, 2048)],
        "Gemma 4 31B": [(10, 4, 512, 0), (50, 16, 256, 1024)],
    }
    for row in g["capacity_mib"]:
        b = acc.kv_capacity_bytes(models[row["model"]], row["N"])
        assert b == row["mib"] * 2 ** 20, row


@pytest.mark.parametrize("T,S,W", [(1, 1, 0), (7, 7, 0), (7, 7, 3), (10, 25, 4), (33, 33, 33),
                                   (33, 33, 34), (5, 9, 9), (64, 64, 1), (50, 80, 100)])
def test_unmasked_pairs_brute_force(T, S, W):
    n = 0
    for t in range(T):
        qp = S - T + t
        for kp in range(S):
            if kp <= qp and (W <= 0 or qp - kp < W):
                n += 1
    assert acc.unmasked_pairs(T, S, W) == n


def test_workload_flops():
    # B=2, T=S=8192, Hq=64, d=128, W=2048: 14,681,088 pairs per head, 962.1 GFLOP
    assert acc.unmasked_pairs(8192, 8192, 2048) == 14_681_088
    assert round(acc.prefill_flops(2, 64, 8192, 8192, 128, 2048) / 1e9, 1) == 962.1
    assert round(acc.prefill_flops(1, 64, 32768, 32768, 128, 0) / 1e12, 3) == 17.593
