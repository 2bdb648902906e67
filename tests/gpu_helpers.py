"""Shared helpers of the GPU parity tests (imported only by tests/)."""
import numpy as np
import pytest
import torch

import oracle
import synth

# bf16 outputs vs the oracle's unrounded fp64 value, elementwise
RTOL, ATOL = 1e-2, 1e-3


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def lib():
    need_gpu()
    import os
    import residual_rmsnorm_gb300 as tp
    from residual_rmsnorm_gb300 import build
    build.build(debug=os.environ.get("TPAR_DEBUG") == "1")
    tp.library()
    tp.tpar_init(torch.cuda.current_device())
    return tp


def dtype_name(t: torch.Tensor) -> str:
    return "fp16" if t.dtype == torch.float16 else "bf16"


def assert_close_to_ref(got_bf16: torch.Tensor, ref64: np.ndarray, what: str, extra=None):
    got = oracle.to_float64(synth.bits(got_bf16), dtype_name(got_bf16))
    assert got.shape == ref64.shape, (got.shape, ref64.shape)
    with np.errstate(invalid="ignore"):
        err = np.abs(got - ref64)
        bound = RTOL * np.abs(ref64) + ATOL
        if extra is not None:
            bound = bound + extra
        # within the bound (false for any NaN), or NaN exactly where the
        # reference is NaN, or the same infinity
        ok = (err <= bound) | (np.isnan(got) & np.isnan(ref64)) | (np.isinf(got) & (got == ref64))
    bad = ~ok
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                             f"first {idx.tolist()}: got {got[bad][:5]}, want {ref64[bad][:5]}")


def oracle_rows(inputs, rows, eps, residual=True):
    """Oracle outputs for the selected rows (rows are independent), in the
    inputs' element type."""
    sel = lambda t: synth.bits(t[rows])
    parts = [sel(p) for p in inputs["partials"]]
    res = sel(inputs["residual"]) if residual and inputs.get("residual") is not None else None
    return oracle.fused_rmsnorm(parts, res, synth.bits(inputs["gamma"]), eps,
                                dtype=dtype_name(inputs["gamma"]))


def to_device(inputs, dev="cuda"):
    return {"partials": [p.to(dev) for p in inputs["partials"]],
            "residual": None if inputs["residual"] is None else inputs["residual"].to(dev),
            "gamma": inputs["gamma"].to(dev)}


def assert_nvfp4_bit_exact(out_norm: torch.Tensor, codes, scales, g, given=None, what="nvfp4",
                           scales_128x4=False, sf_fill=0):
    """The oracle quantiser run on the kernel's own normed tensor. With
    ``scales_128x4`` the kernel's scales are the flat 128x4 tiled layout,
    whose padding rows must still hold ``sf_fill``."""
    oc, os_, og = oracle.nvfp4_quantize(synth.bits(out_norm), global_scale=given, dtype=dtype_name(out_norm))
    if scales_128x4:
        os_ = oracle.nvfp4_scales_128x4(os_, fill=sf_fill)
    gc = codes.cpu().numpy()
    gs = scales.cpu().numpy()
    gg = np.float32(g.item()) if isinstance(g, torch.Tensor) else np.float32(g)
    if not np.array_equal(os_, gs):
        bad = np.argwhere(os_ != gs)[:5].tolist()
        raise AssertionError(f"{what}: {int((os_ != gs).sum())} scale bytes differ, first {bad}")
    if not np.array_equal(oc, gc):
        bad = np.argwhere(oc != gc)[:5].tolist()
        raise AssertionError(f"{what}: {int((oc != gc).sum())} code bytes differ, first {bad}: "
                             f"got {[hex(gc[tuple(b)]) for b in bad]}, want {[hex(oc[tuple(b)]) for b in bad]}")
    assert og == gg, (what, og, gg)


# The unfused path rounds the rank sum s to bf16 before adding the residual
# (the all-reduce result is a bf16 tensor in HBM). That one extra rounding
# moves h by at most half a bf16 ulp of s, <= 2^-8 |s|, which near
# cancellation (|h| << |s|) exceeds the fused tolerance. The derived extra
# bound per element: 2^-8 * sum_r |P_r| for h, and the same times
# |gamma| / sqrt(ms + eps) for y.
def unfused_extra_tolerance(inputs, ref, eps):
    dt = dtype_name(inputs["gamma"])
    s_abs = sum(np.abs(oracle.to_float64(synth.bits(p), dt)) for p in inputs["partials"])
    eh = (2.0 ** -8 if dt == "bf16" else 2.0 ** -11) * s_abs
    gam = np.abs(oracle.to_float64(synth.bits(inputs["gamma"]), dt))
    ms = np.mean(ref["h"] ** 2, axis=1, keepdims=True)
    ey = eh * gam[None, :] / np.sqrt(ms + float(np.float32(eps))) * 1.01
    return eh, ey
