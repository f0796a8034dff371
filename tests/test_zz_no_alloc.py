"""The allocation-free down projection entry point (runs last in the suite).

moe_gather_qmm_down_unsort_noalloc serves callers that cannot call cudaMalloc
(an inference-runtime plugin whose execute step must not allocate, a program
with no allocator to lend a workspace): it keeps its fp32 accumulator in a
fixed array inside the library instead of a caller workspace.  Here it is
called through the C ABI twice in a row and compared with the workspace
entry point, moe_gather_qmm_down_unsort, on the same inputs; the second call
shows that the shared array is cleared between calls.
"""
import numpy as np
import pytest

import synth
from _util import bf16_to_f64, excess, to_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import moe_expert_bit_gb300 as mq  # noqa: E402


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill_uniform"])
def test_noalloc_matches_workspace_entry_point_twice(name):
    d = synth.make(name)
    dev = to_device(d)
    E, H, I, T, k = d["E"], d["H"], d["I"], d["T"], d["k"]
    assert T * H <= mq.NOALLOC_MAX_Y_ELEMENTS
    b = mq.moe_layer(dev["x"], dev["topk_ids"], dev["topk_weights"], dev, E, tile_m=128)
    torch.cuda.synchronize()
    assert int(b.routing.status.item()) == 0
    y_ref = bf16_to_f64(b.y)
    for _ in range(2):
        y = torch.full((T, H), 5.0, dtype=torch.bfloat16, device="cuda")
        mq.moe_gather_qmm_down_unsort_noalloc(b.h, dev["Wd"], dev["Sd"], dev["Bd"], b.routing,
                                              dev["topk_weights"], H, I, y)
        torch.cuda.synchronize()
        assert int(b.routing.status.item()) == 0
        assert excess(bf16_to_f64(y), y_ref) <= 1.0
    assert np.abs(y_ref).max() > 0


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_noalloc_deterministic_equals_workspace_entry_point_bitwise(name):
    """The fixed-order un-sort through the built-in array gives the same bits as through a
    caller workspace (same variant, same inputs)."""
    d = synth.make(name)
    dev = to_device(d)
    E, H, I, T, k = d["E"], d["H"], d["I"], d["T"], d["k"]
    b = mq.moe_layer(dev["x"], dev["topk_ids"], dev["topk_weights"], dev, E, tile_m=128,
                     variant=mq.VARIANT_GEMV, deterministic=True)
    torch.cuda.synchronize()
    assert int(b.routing.status.item()) == 0
    for _ in range(2):
        y = torch.full((T, H), 5.0, dtype=torch.bfloat16, device="cuda")
        mq.moe_gather_qmm_down_unsort_noalloc(b.h, dev["Wd"], dev["Sd"], dev["Bd"], b.routing,
                                              dev["topk_weights"], H, I, y, mq.VARIANT_GEMV,
                                              deterministic=True)
        torch.cuda.synchronize()
        assert int(b.routing.status.item()) == 0
        assert torch.equal(y.view(torch.int16), b.y.view(torch.int16))


def test_noalloc_rejects_sizes_beyond_its_array():
    T, k, E, H, I = 4096, 1, 4, 2048, 64  # T * H = 8 Mi elements > 4 Mi
    r = mq.Routing(T, k, E, 32)
    h = torch.zeros(T * k, I, dtype=torch.bfloat16, device="cuda")
    Wd = torch.zeros(E, H, I // 8, dtype=torch.int32, device="cuda")
    Sd = torch.zeros(E, H, I // 64, dtype=torch.bfloat16, device="cuda")
    tw = torch.zeros(T, k, dtype=torch.float32, device="cuda")
    y = torch.zeros(T, H, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mq.MoeError) as ei:
        mq.moe_gather_qmm_down_unsort_noalloc(h, Wd, Sd, Sd, r, tw, H, I, y)
    assert ei.value.status == mq.MOE_ERR_UNSUPPORTED
    assert "exceeds" in str(ei.value)
