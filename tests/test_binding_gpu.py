"""The PyTorch binding refuses tensors the C ABI cannot check for itself
(shapes, element types, devices of caller-supplied outputs and scales)
before anything launches: a wrong-sized output would otherwise be written
past its end."""
import pytest
import torch

import synth
from gpu_helpers import lib, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def call():
    tp = lib()
    w = synth.DECODE_8B.with_(T=4, d=1024)
    dev = to_device(synth.make_inputs(w))
    return tp, w, dev


def test_caller_outputs_of_the_wrong_shape_or_type(call):
    tp, w, dev = call
    T, d = dev["partials"][0].shape
    short = torch.empty((T - 1, d), dtype=torch.bfloat16, device="cuda")
    half = torch.empty((T, d), dtype=torch.float16, device="cuda")
    strided = torch.empty((d, T), dtype=torch.bfloat16, device="cuda").t()
    for bad in (short, half, strided):
        for kw in ("reduced", "out_norm", "out_residual"):
            with pytest.raises((ValueError, TypeError)):
                tp.unfused_rmsnorm(dev["partials"], dev["residual"], dev["gamma"], w.eps, **{kw: bad})
        for kw in ("out_norm", "out_residual"):
            with pytest.raises((ValueError, TypeError)):
                tp.fused_rmsnorm(dev["partials"], dev["residual"], dev["gamma"], w.eps, **{kw: bad})
        with pytest.raises((ValueError, TypeError)):
            tp.fused_rmsnorm_fp8(dev["partials"], dev["residual"], dev["gamma"], w.eps, out_residual=bad)
        with pytest.raises((ValueError, TypeError)):
            tp.allreduce_sum(dev["partials"], dev["residual"], out=bad)
    torch.cuda.synchronize()


def test_scales_must_be_one_fp32_element_on_the_device(call):
    tp, w, dev = call
    x = dev["partials"][0]
    bad = [torch.tensor([0.5], dtype=torch.bfloat16, device="cuda"),
           torch.tensor([0.5, 0.5], dtype=torch.float32, device="cuda"),
           torch.tensor([0.5], dtype=torch.float32)]
    for s in bad:
        with pytest.raises(ValueError):
            tp.fp8_quantize(x, scale=s)
        with pytest.raises(ValueError):
            tp.fused_rmsnorm_fp8(dev["partials"], dev["residual"], dev["gamma"], w.eps, scale=s)
        with pytest.raises(ValueError):
            tp.nvfp4_quantize(x, global_scale=s)
        with pytest.raises(ValueError):
            tp.fused_rmsnorm(dev["partials"], dev["residual"], dev["gamma"], w.eps, nvfp4=True, global_scale=s)


def test_inputs_of_the_wrong_rank_count_or_place(call):
    tp, w, dev = call
    with pytest.raises(ValueError):
        tp.fused_rmsnorm([], dev["residual"], dev["gamma"], w.eps)
    with pytest.raises(ValueError):
        tp.unfused_rmsnorm([], dev["residual"], dev["gamma"], w.eps)
    with pytest.raises(ValueError):
        tp.fused_rmsnorm(dev["partials"], dev["residual"], None, w.eps)
    with pytest.raises(ValueError):
        tp.nvfp4_quantize(dev["partials"][0].reshape(-1))
    with pytest.raises(ValueError):  # pageable host memory: no CPU compute path
        tp.fused_rmsnorm(dev["partials"], dev["residual"].cpu(), dev["gamma"], w.eps)


@pytest.mark.skipif(torch.cuda.device_count() < 2, reason="needs a second GPU")
def test_tensors_on_another_device(call):
    tp, w, dev = call
    other = dev["residual"].to("cuda:1")
    with pytest.raises(ValueError):
        tp.fused_rmsnorm(dev["partials"], other, dev["gamma"], w.eps)
