"""The binding's typical use, call by call (the same statements as the usage example
users copy): the activation alone, the one-launch FFN, routed experts with the
combine, a training step, MX experts.  Each result has its documented shape and no
kernel records a device-side failure."""
import pytest
import torch

import situ_glu_activation_gb300 as situ

pytestmark = pytest.mark.gpu


def test_usage_example_runs(cuda_dev):
    x = torch.randn(16384, 2048, device="cuda").bfloat16()              # tokens x model width
    w_gate_up = (torch.randn(6144, 2048, device="cuda") / 2048 ** 0.5).bfloat16()  # [2I, M]
    w_down = (torch.randn(2048, 3072, device="cuda") / 3072 ** 0.5).bfloat16()     # [M, I]

    h = situ.situ_glu_act(x @ w_gate_up.T)                  # the activation alone: [R, I]
    y = situ.situ_ffn_forward(x, w_gate_up, w_down)         # the whole FFN, one launch: [R, M]

    # Routed experts: ids [T, k] -> per-(token, slot) outputs [T, k, M], then the combine.
    ids = torch.randint(0, 64, (16384, 8), device="cuda", dtype=torch.int32)
    wgu_e = (torch.randn(64, 6144, 2048, device="cuda") / 2048 ** 0.5).bfloat16()
    wd_e = (torch.randn(64, 2048, 3072, device="cuda") / 3072 ** 0.5).bfloat16()
    offsets, token_index = situ.situ_moe_build_index(ids, 64)
    y_slots = situ.situ_moe_grouped_forward(x, offsets, token_index, wgu_e, wd_e, k_eff=8)
    out = situ.situ_moe_combine(y_slots, torch.full((16384, 8), 0.125, device="cuda"))

    # Training: forward keeping the pre-activation, then the backward.
    y, gu, h = situ.situ_ffn_forward_train(x, w_gate_up, w_down)
    dx, dw_gate_up, dw_down = situ.situ_ffn_backward(x, w_gate_up, w_down, gu, h,
                                                     torch.ones_like(y))

    # MX experts: weights quantized once, activations quantized in the call.
    wq = situ.mx_quantize_weights(w_gate_up, situ.MX_GATE_UP, situ.MX_E2M1)   # MXFP4
    wdq = situ.mx_quantize_weights(w_down, situ.MX_DOWN, situ.MX_E2M1)
    y_mx = situ.situ_ffn_forward_mxfp8(x, wq, wdq)

    torch.cuda.synchronize()
    assert tuple(h.shape) == (16384, 3072) and tuple(gu.shape) == (16384, 6144)
    assert tuple(y.shape) == (16384, 2048)
    assert tuple(y_slots.shape) == (16384, 8, 2048)
    assert tuple(out.shape) == (16384, 2048)
    assert tuple(dx.shape) == (16384, 2048)
    assert tuple(dw_gate_up.shape) == (6144, 2048) and tuple(dw_down.shape) == (2048, 3072)
    assert tuple(y_mx.shape) == (16384, 2048)
    assert situ.device_status(clear=True) == 0
