"""The seeded input generators: determinism, shapes and the outlier recipe."""
import math

import torch

import synth


def test_deterministic_and_shapes():
    a = synth.make_inputs(synth.SMALL)
    b = synth.make_inputs(synth.SMALL)
    assert len(a["partials"]) == 2
    for x, y in zip(a["partials"] + [a["residual"], a["gamma"]], b["partials"] + [b["residual"], b["gamma"]]):
        assert x.dtype == torch.bfloat16 and torch.equal(x.view(torch.int16), y.view(torch.int16))
    assert a["partials"][0].shape == (4, 256) and a["gamma"].shape == (256,)
    c = synth.make_inputs(synth.SMALL, seed=1)
    assert not torch.equal(a["partials"][0], c["partials"][0])


def test_distribution_roughly_matches_recipe():
    w = synth.DECODE_8B
    x = synth.make_inputs(w)
    p = torch.stack([t.float() for t in x["partials"]])
    assert abs(p.std().item() - 0.5) < 0.01
    assert abs(x["residual"].float().std().item() - 1.0) < 0.02
    assert abs(x["gamma"].float().mean().item() - 1.0) < 0.01
    assert abs(x["gamma"].float().std().item() - 0.1) < 0.01


def test_outliers_exact_count():
    w = synth.NVFP4.with_(T=8, d=1024)
    x = synth.make_inputs(w)
    base = synth.make_inputs(w.with_(outlier_frac=0.0))
    k = math.floor(0.01 * 8 * 1024)
    for p, q in zip(x["partials"], base["partials"]):
        changed = (p.float() != q.float()).sum().item()
        # a drawn zero stays zero; otherwise every chosen position changes
        assert k - 2 <= changed <= k
        ratio = (p.float()[p != q] / q.float()[p != q])
        assert torch.allclose(ratio, torch.full_like(ratio, 50.0), rtol=1e-2)


def test_bits_round_trip():
    x = synth.random_bf16((3, 16), 1.0, seed=3)
    assert torch.equal(synth.from_bits(synth.bits(x)).view(torch.int16), x.view(torch.int16))
