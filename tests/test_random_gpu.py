"""Seeded random sweep over the argument space, every case against the
oracle: ranks (1..16, odd counts included), T (0..700), d (any multiple of 8
up to 9216; 16 or 64 when the output needs it), element type, residual
present or not, output pattern (norm, sum only, NVFP4 given / dynamic, 128x4
scales, FP8) and forced kernel form (row, cluster, TMA-fed, cooperative
grid). The cases are drawn once from a fixed
seed, so a failure names a reproducible case."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import assert_close_to_ref, assert_nvfp4_bit_exact, lib, oracle_rows, to_device

pytestmark = pytest.mark.gpu


def _cases(n_cases=200, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n_cases):
        n = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 11, 16]))
        T = int(rng.choice([0, 1, 2, 3, 5, 8, 13, 31, 33, 47, 64, 100, 153, 229, 300, 700]))
        mode = str(rng.choice(["norm", "norm", "sum", "nvfp4_given", "nvfp4_dyn", "nvfp4_128x4", "fp8"]))
        step = 64 if mode == "nvfp4_128x4" else (16 if mode.startswith("nvfp4") else 8)
        d = int(step * rng.integers(1, 9216 // step + 1))
        if n * T * d > 40_000_000:  # keep the oracle quick
            T = max(1, 40_000_000 // (n * d))
        residual = bool(rng.random() < 0.8)
        dtype = "fp16" if rng.random() < 0.25 else "bf16"
        force = str(rng.choice(["auto", "auto", "auto", "row", "cluster", "stream", "grid"]))
        out.append((i, n, T, d, mode, residual, dtype, force))
    return out


@pytest.mark.parametrize("case", _cases(), ids=lambda c: f"c{c[0]}-N{c[1]}-T{c[2]}-d{c[3]}-{c[4]}-{c[6]}-{c[7]}")
def test_random_case(case):
    i, n, T, d, mode, residual, dtype, force = case
    tp = lib()
    dt = torch.float16 if dtype == "fp16" else torch.bfloat16
    w = synth.Workload(f"random {i}", n, T, d, 1e-5, 0.5, seed=1000 + i)
    inputs = synth.make_inputs(w, dtype=dt)
    if not residual:
        inputs = dict(inputs, residual=None)
    dev = to_device(inputs)
    flags = {"auto": 0, "row": tp.TPAR_FORCE_ROW, "cluster": tp.TPAR_FORCE_CLUSTER,
             "stream": tp.TPAR_FORCE_STREAM, "grid": tp.TPAR_FORCE_GRID}[force]
    if force == "grid" and not (mode in ("nvfp4_dyn", "nvfp4_128x4") and d <= 8192 and
                                -(-T // torch.cuda.get_device_properties(0).multi_processor_count) * d * 2 <= 200 * 1024):
        flags = 0  # the cooperative path: dynamic-scale NVFP4 whose rows fit on chip
    if force == "cluster" and d < 32:
        flags = 0  # rows too short to split
    if force == "stream" and mode == "fp8":
        flags = 0  # the TMA-fed kernel has no FP8 output
    rows = np.arange(T) if T <= 64 else np.unique(np.concatenate([[0, T - 1],
                                                                  np.random.default_rng(i).choice(T, 24)]))
    g = torch.tensor([0.05], dtype=torch.float32, device="cuda")
    if mode == "sum":
        out = tp.allreduce_sum(dev["partials"], dev["residual"], flags=flags)
        torch.cuda.synchronize()
        if T:
            ref = oracle_rows(inputs, rows, w.eps, residual=residual)
            assert_close_to_ref(out[rows], ref["h"], f"case {i} sum")
    elif mode == "fp8":
        out = tp.fused_rmsnorm_fp8(dev["partials"], dev["residual"], dev["gamma"], w.eps, flags=flags)
        torch.cuda.synchronize()
        if T:
            ref = oracle_rows(inputs, rows, w.eps, residual=residual)
            assert_close_to_ref(out["out_norm"][rows], ref["y"], f"case {i} fp8 out_norm")
            oc, os_ = oracle.fp8_quantize(synth.bits(out["out_norm"]), dtype=dtype)
            assert np.array_equal(out["codes"].cpu().numpy(), oc) and np.float32(out["scale"].item()) == os_
    else:
        nv = mode.startswith("nvfp4")
        given = mode == "nvfp4_given"
        out = tp.fused_rmsnorm(dev["partials"], dev["residual"], dev["gamma"], w.eps, nvfp4=nv,
                               global_scale=g if given else None, scales_128x4=mode == "nvfp4_128x4",
                               flags=flags)
        torch.cuda.synchronize()
        if T:
            ref = oracle_rows(inputs, rows, w.eps, residual=residual)
            assert_close_to_ref(out["out_norm"][rows], ref["y"], f"case {i} out_norm")
            assert_close_to_ref(out["out_residual"][rows], ref["h"], f"case {i} out_residual")
            if nv:
                assert_nvfp4_bit_exact(out["out_norm"], out["codes"], out["scales"], out["global_scale"],
                                       given=float(np.float32(0.05)) if given else None, what=f"case {i}",
                                       scales_128x4=mode == "nvfp4_128x4")
    assert tp.tpar_device_error(torch.cuda.current_device()) == 0
