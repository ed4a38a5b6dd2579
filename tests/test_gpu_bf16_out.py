"""The bf16-output entry point: every output is the float32 result rounded once to bf16
(round to nearest even), on every path (decode, decode passes, prefill with and without K slices,
and with the gate/up projection's last round split along K)."""
import numpy as np
import pytest

import workloads
from tests.gpu_util import dev, lib, to_dev, torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("H,I,m,xdt", [(1024, 2816, 1, "f32"), (512, 1536, 8, "bf16"), (1024, 768, 16, "f32"),
                                        (512, 768, 48, "bf16"), (2304, 1280, 300, "bf16"), (4096, 2048, 64, "bf16"),
                                        (2048, 10240, 32, "bf16")])
def test_bf16_output_is_the_rounded_float32_output(H, I, m, xdt):
    c = workloads.small_config(H, I, m, xdt, ("channels", 0.01, 50.0))
    wg, wu, wd = [to_dev(a) for a in workloads.weights(c)]
    _, xb = workloads.activations(c)
    x = to_dev(xb)
    ws = torch.empty(lib().ffn_q4k_workspace_bytes(m, H, I), dtype=torch.uint8, device=dev())
    y32 = lib().ffn_q4k_swiglu_ex(x, wg, wu, wd, ws).cpu().numpy()
    y16 = torch.full((m, H), float("nan"), dtype=torch.bfloat16, device=dev())
    lib().ffn_q4k_swiglu_ex_y(x, wg, wu, wd, ws, y16)
    torch.cuda.synchronize()
    got = y16.view(torch.int16).cpu().numpy().view(np.uint16)
    want = workloads.f32_to_bf16_bits(y32).reshape(m, H)
    same = got == want
    # an exact zero may carry either sign (a chunk sum 0 + (-0) is +0)
    zero = (y32 == 0) & ((got & 0x7FFF) == 0)
    assert np.all(same | zero)
    assert lib().q4k_check_device_error() == 0


def test_bf16_output_rejects_other_dtypes():
    c = workloads.small_config(256, 512, 1)
    wg, wu, wd = [to_dev(a) for a in workloads.weights(c)]
    x = torch.zeros((1, 256), dtype=torch.float32, device=dev())
    ws = torch.empty(lib().ffn_q4k_workspace_bytes(1, 256, 512), dtype=torch.uint8, device=dev())
    with pytest.raises(TypeError):
        lib().ffn_q4k_swiglu_ex_y(x, wg, wu, wd, ws, torch.empty((1, 256), dtype=torch.float16, device=dev()))
