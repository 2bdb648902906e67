"""The no-allocation unfused entry point, tpar_unfused_rmsnorm_noalloc.

It serves callers that cannot allocate device memory: code running while a
framework owns the device allocator, plugins whose contract forbids
allocating, code that may first run inside a CUDA-graph capture (where
cudaMalloc is not allowed), latency-critical paths that cannot pay for an
allocation's synchronisation. Such callers cannot pass the `reduced` scratch
tensor the ordinary unfused entry point needs, so this variant keeps that
scratch (and the dynamic NVFP4 scale's accumulator) in a static device array
inside the library.

The GPU test drives it through the C ABI for two calls in a row, with
different inputs (so a stale scratch from the first call would show), and
checks each against the ordinary unfused entry point on the same inputs:
bf16 outputs within the tolerance the other tests use, NVFP4 codes, scales
and global scale bit for bit. This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import ATOL, RTOL, lib, to_device


def _noalloc(tp, dev, w, nvfp4):
    T, d = w.T, w.d
    out_n = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    out_r = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    codes = scales = g = None
    if nvfp4:
        codes = torch.empty((T, d // 2), dtype=torch.uint8, device="cuda")
        scales = torch.empty((T, d // 16), dtype=torch.uint8, device="cuda")
        g = torch.empty((1,), dtype=torch.float32, device="cuda")
    tp.tpar_unfused_rmsnorm_noalloc(
        [p.data_ptr() for p in dev["partials"]], w.n_ranks, dev["residual"].data_ptr(),
        dev["gamma"].data_ptr(), w.eps, T, d, out_n.data_ptr(), out_r.data_ptr(),
        codes.data_ptr() if nvfp4 else 0, scales.data_ptr() if nvfp4 else 0,
        g.data_ptr() if nvfp4 else 0, 0, torch.cuda.current_stream().cuda_stream)
    return {"out_norm": out_n, "out_residual": out_r, "codes": codes, "scales": scales, "global_scale": g}


def _within_tolerance(got, ref, what):
    a = got.double()
    b = ref.double()
    bad = (a - b).abs() > RTOL * b.abs() + ATOL
    assert not bool(bad.any()), f"{what}: {int(bad.sum())} elements outside the tolerance"


@pytest.mark.gpu
def test_noalloc_matches_the_unfused_entry_point_twice_in_a_row():
    tp = lib()
    cases = [(synth.DECODE_8B, False), (synth.NVFP4.with_(T=64, d=2048, seed=3), True),
             (synth.PREFILL.with_(T=96, seed=4), False)]
    for w, nvfp4 in cases:
        dev = to_device(synth.make_inputs(w))
        got = _noalloc(tp, dev, w, nvfp4)
        want = tp.unfused_rmsnorm(dev["partials"], dev["residual"], dev["gamma"], w.eps, nvfp4=nvfp4)
        torch.cuda.synchronize()
        _within_tolerance(got["out_residual"], want["out_residual"], f"{w.name} out_residual")
        _within_tolerance(got["out_norm"], want["out_norm"], f"{w.name} out_norm")
        if nvfp4:
            assert torch.equal(got["codes"], want["codes"])
            assert torch.equal(got["scales"], want["scales"])
            assert got["global_scale"].item() == want["global_scale"].item()


@pytest.mark.gpu
def test_noalloc_refuses_sizes_beyond_its_scratch():
    tp = lib()
    d = 8192
    T = tp.TPAR_NOALLOC_MAX_ELEMENTS // d + 1
    base = 0x7F0000000000  # never dereferenced: the size check comes first
    st = tp.tpar_unfused_rmsnorm_noalloc([base] * 2, 2, 0, base, 1e-5, T, d, base, base, 0, 0, 0, 0, 0,
                                         check=False)
    assert st == 6  # TPAR_ERR_SCRATCH_TOO_SMALL
    assert "exceeds" in tp.tpar_status_string(6)


def test_noalloc_host_checks_without_gpu():
    from residual_rmsnorm_gb300 import build
    build.build()
    import residual_rmsnorm_gb300 as tp
    base, mb = 0x7F0000000000, 1 << 20
    parts = [base + r * 4 * mb for r in range(4)]
    call = lambda T, d, flags: tp.tpar_unfused_rmsnorm_noalloc(
        parts, 4, base + 64 * mb, base + 96 * mb, 1e-5, T, d, base + 128 * mb, base + 160 * mb,
        0, 0, 0, flags, 0, check=False)
    assert call(8, 4096, tp.TPAR_DRY_RUN) == 0
    assert call(tp.TPAR_NOALLOC_MAX_ELEMENTS // 4096, 4096, tp.TPAR_DRY_RUN) == 0
    assert call(tp.TPAR_NOALLOC_MAX_ELEMENTS // 4096 + 1, 4096, tp.TPAR_DRY_RUN) == 6
    assert call(8, 12, tp.TPAR_DRY_RUN) == 1
    assert call(0, 4096, 0) == 0
