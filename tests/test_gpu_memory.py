"""Device memory high-water of the library's calls.

Page "PyTorch + HIP fused bias + GELU on Hygon DCU" (s7, s9) reports an op's
memory cost as the allocator's peak during one call minus the peak before
it.  The C ABI allocates nothing, so with every output (and the backward's
workspace) passed in, repeated calls of every entry point must leave both
torch's allocated peak and the device's free memory exactly where they were.
"""
import pytest
import torch

import window_gather_swin_gb300 as wgs
from window_gather_swin_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def _inputs(dtype):
    st = synth.TINY_PADDED
    a, b, x, bias = synth.tiny_block(seed=3, stage=st)
    a, b = a.to(dtype).to(DEV), b.to(dtype).to(DEV)
    idx = wgs.build_window_index(st.grid, synth.WINDOW, synth.SHIFT, device=DEV)
    inv = wgs.build_window_inverse(st.grid, synth.WINDOW, synth.SHIFT, device=DEV)
    reg = wgs.build_shift_regions(st.grid, synth.WINDOW, synth.SHIFT, device=DEV)
    n_win = idx.numel() // 144
    sc, sb = synth.attention_logits(n_win, 2, 144, 1, seed=3, dtype=dtype)
    x, bias = x.to(DEV), bias.to(DEV)
    rows, width = x.shape
    ws = torch.empty(max(wgs.gelu_bwd_workspace_bytes(rows, width), 16), dtype=torch.uint8,
                     device=DEV)
    t = dict(a=a, b=b, idx=idx, inv=inv, reg=reg, sc=sc.to(DEV), sb=sb.to(DEV), x=x, bias=bias,
             gy=torch.ones_like(x), ws=ws)
    # every output, allocated once
    t.update(y=torch.empty_like(a), r=torch.empty_like(a),
             g=torch.empty(idx.numel(), a.shape[1], dtype=dtype, device=DEV),
             z=torch.empty_like(x), gx=torch.empty_like(x), gb=torch.empty_like(bias),
             bm=torch.empty_like(t["sc"]))
    return t


def _every_call(t, eps=1e-5):
    wgs.ln_fwd(t["a"], eps, out=t["y"])
    wgs.residual_add_ln_fwd(t["a"], t["b"], eps, residual_out=t["r"], out=t["y"])
    wgs.window_gather(t["a"], t["idx"], out=t["g"])
    wgs.norm_gather(t["a"], t["idx"], eps, out=t["g"])
    wgs.residual_add_norm_gather(t["a"], t["b"], t["idx"], eps, residual_out=t["r"], out=t["g"])
    wgs.window_reverse_add_ln_fwd(t["a"], t["g"], t["inv"], eps, residual_out=t["r"], out=t["y"])
    wgs.bias_gelu_tanh(t["x"], t["bias"], out=t["z"])
    wgs.bias_gelu_tanh_bwd(t["gy"], t["x"], t["bias"], grad_x=t["gx"], grad_bias=t["gb"],
                           workspace=t["ws"])
    wgs.window_bias_mask_add(t["sc"], t["sb"], None, t["reg"], -100.0, out=t["bm"])


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_calls_with_given_outputs_allocate_no_device_memory(dtype):
    t = _inputs(dtype)
    _every_call(t)                      # first calls: runtime queries and module loading
    torch.cuda.synchronize(DEV)
    torch.cuda.reset_peak_memory_stats(DEV)
    allocated = torch.cuda.memory_allocated(DEV)
    free_before = torch.cuda.mem_get_info(DEV)[0]
    for _ in range(3):
        _every_call(t)
    torch.cuda.synchronize(DEV)
    assert torch.cuda.max_memory_allocated(DEV) == allocated    # incremental peak: 0 bytes
    assert torch.cuda.mem_get_info(DEV)[0] == free_before       # nothing outside torch either
    wgs.check_error(DEV)
