"""Seeded input generators: determinism, shapes, and the peaked-row recipe."""
import math

import torch

import fa_workloads as W


def test_inputs_are_deterministic_bf16():
    w = W.WORKLOADS["gqa8k"].with_(B=1, N=200)
    a, b = W.make_inputs(w), W.make_inputs(w)
    for key in ("q", "k", "v", "dout"):
        assert a[key].dtype == torch.bfloat16
        assert torch.equal(a[key], b[key])
    assert a["q"].shape == (1, 200, 32, 128) and a["k"].shape == (1, 200, 8, 128)
    # Q, K, V scaled by 0.5; dO is N(0, 1)
    assert 0.4 < a["q"].float().std().item() < 0.6
    assert 0.9 < a["dout"].float().std().item() < 1.1


def test_peaked_rows_recipe():
    w = W.WORKLOADS["gqa32k_peaked"].with_(N=1000)
    x = W.make_inputs(w, with_dout=False)
    pos = W.peaked_positions(w)
    npk = math.ceil(0.01 * 1000)
    for (b, h), idx in pos.items():
        assert idx.numel() == npk and idx.unique().numel() == npk
        norms = x["k"][b, :, h].float().norm(dim=-1)
        mask = torch.zeros(1000, dtype=torch.bool)
        mask[idx] = True
        # peaked rows are ~8x the typical norm (~sqrt(128))
        assert norms[mask].min() > 4 * norms[~mask].median()
    assert math.ceil(0.01 * 32768) == 328


def test_nominal_flop_formula():
    w = W.WORKLOADS["gpt2s"]
    assert W.fwd_flops(w) == 4 * 16 * 12 * 2048 ** 2 * 64
    assert W.bwd_flops(w) == 2.5 * W.fwd_flops(w)
    c = W.WORKLOADS["mqa128k"]
    assert W.fwd_flops(c) == 4 * 16 * 131072 ** 2 * 128 / 2
