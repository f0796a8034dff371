"""GPU parity of the one-launch decode layer (moe_layer_fused) against the fp64 oracle and
against the four calls: routing state bit for bit, h and y within the bound of tests/_util.py.
"""
import numpy as np
import pytest

import oracle
import synth
from _util import bf16_to_f64, excess, to_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import moe_expert_bit_gb300 as mq  # noqa: E402


def run_fused(d, tile_m=128, dev=None, buffers=None):
    dev = dev or to_device(d)
    b = buffers or mq.MoeLayerBuffers(d["T"], d["k"], d["E"], d["H"], d["I"], tile_m)
    mq.moe_layer(dev["x"], dev["topk_ids"], dev["topk_weights"], dev, d["E"], tile_m=tile_m,
                 buffers=b, fused=True)
    torch.cuda.synchronize()
    return b


def check_routing(b, d, tile_m):
    st, sid, perm, counts = oracle.sort_assignments(d["topk_ids"], d["E"])
    r = b.routing
    assert int(r.status.item()) == 0
    assert np.array_equal(r.sorted_ids.cpu().numpy(), sid)
    assert np.array_equal(r.perm.cpu().numpy(), perm)
    assert np.array_equal(r.counts.cpu().numpy(), counts)
    st, off, tiles, tc = oracle.build_expert_tiles(sid, d["E"], tile_m)
    assert np.array_equal(r.offsets.cpu().numpy(), off)
    assert int(r.tile_count.item()) == tc
    assert np.array_equal(r.tiles.cpu().numpy()[:3 * tc].reshape(-1, 3), tiles)


def check_outputs(b, d):
    ref = oracle.layer(d)
    out_rows = np.isin(np.arange(d["T"]), d["outlier_rows"])
    slot_rows = out_rows[ref["perm"] // d["k"]]
    assert excess(bf16_to_f64(b.h), ref["h"], slot_rows) <= 1.0
    assert excess(bf16_to_f64(b.y), ref["y"], out_rows) <= 1.0
    return ref


@pytest.mark.parametrize("name", ["tiny", "decode"])
@pytest.mark.parametrize("tile_m", [16, 128])
def test_fused_layer_matches_oracle(name, tile_m):
    d = synth.make(name)
    b = run_fused(d, tile_m)
    check_routing(b, d, tile_m)
    check_outputs(b, d)


@pytest.mark.parametrize("E,H,I,T,k", [
    (5, 192, 128, 37, 3),      # ragged, 3 K-groups, odd group counts
    (1, 128, 64, 1, 1),        # one assignment
    (8, 256, 128, 64, 1),      # the most token rows it stages
    (4, 128, 64, 16, 4),       # tiles of ~16 rows: several passes per tile in both phases
    (16, 512, 320, 32, 8),     # A = 256, the most assignments it takes
])
def test_fused_layer_custom_shapes(E, H, I, T, k):
    d = synth.make_custom(E, H, I, T, k, seed=3)
    b = run_fused(d, 32)
    check_routing(b, d, 32)
    check_outputs(b, d)


def test_fused_equals_four_calls_and_leaves_workspace_zero():
    d = synth.make("decode")
    dev = to_device(d)
    b = run_fused(d, dev=dev)
    ref = mq.moe_layer(dev["x"], dev["topk_ids"], dev["topk_weights"], dev, d["E"],
                       variant=mq.VARIANT_GEMV)
    torch.cuda.synchronize()
    # same partition of every dot product: h bit for bit; y up to the order of the atomics
    assert torch.equal(b.h, ref.h)
    y0, y1 = bf16_to_f64(b.y), bf16_to_f64(ref.y)
    assert np.abs(y0 - y1).max() <= 2e-2 * max(1.0, np.abs(y1).max())
    for key in ("sorted_ids", "perm", "counts", "offsets", "tile_count"):
        assert torch.equal(getattr(b.routing, key), getattr(ref.routing, key)), key
    n_zero = d["T"] * d["H"] + d["H"] // 16  # accumulator and counters (then the barrier)
    assert int(torch.count_nonzero(b.y_acc[:n_zero]).item()) == 0
    # a second call on the same buffers gives the same routing and h, and y within atomics
    b2 = run_fused(d, dev=dev, buffers=b)
    assert torch.equal(b2.h, ref.h)
    assert np.abs(bf16_to_f64(b2.y) - y1).max() <= 2e-2 * max(1.0, np.abs(y1).max())
    assert int(torch.count_nonzero(b2.y_acc[:n_zero]).item()) == 0
    # the count of finished CTAs (after the counters): one per CTA per call
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert int(b2.y_acc[n_zero:n_zero + 2].view(torch.int64).item()) == 2 * n_sm


def test_fused_zero_router_weight_gives_exact_zero():
    d = synth.make("decode")
    d["topk_weights"][1, :] = 0.0
    b = run_fused(d)
    assert torch.count_nonzero(b.y[1].float()).item() == 0
    check_outputs(b, d)


def test_fused_bad_routing_leaves_outputs_untouched():
    d = synth.make("decode")
    d["topk_ids"][2, 3] = d["E"] + 5
    dev = to_device(d)
    b = mq.MoeLayerBuffers(d["T"], d["k"], d["E"], d["H"], d["I"], 128)
    b.h.fill_(7.0)
    b.y.fill_(3.0)
    mq.moe_layer(dev["x"], dev["topk_ids"], dev["topk_weights"], dev, d["E"], buffers=b,
                 fused=True)
    torch.cuda.synchronize()
    assert int(b.routing.status.item()) == mq.MOE_ERR_RANGE
    assert int(b.routing.tile_count.item()) == 0
    assert bool((b.h == 7.0).all()) and bool((b.y == 3.0).all())
    assert int(torch.count_nonzero(b.y_acc).item()) == 0


def test_fused_refuses_calls_beyond_it():
    d = synth.make_custom(3, 256, 192, 300, 2, seed=1)
    dev = to_device(d)
    with pytest.raises(mq.MoeError) as ei:
        mq.moe_layer(dev["x"], dev["topk_ids"], dev["topk_weights"], dev, d["E"], fused=True)
    assert ei.value.status == mq.MOE_ERR_UNSUPPORTED
