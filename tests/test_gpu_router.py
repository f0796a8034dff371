"""GPU parity of the router's top-k + softmax and of the route from logits (the step before
the sort), against the fp64 oracle.

Ids are compared bit for bit (the selection compares the fp32 logits themselves, exact in
any precision); weights within 2e-6 (fp32 exp and division against the fp64 softmax rounded
to fp32); the routing state that follows bit for bit against the oracle's sort and tiles of
the same ids.  Both launch shapes of moe_route_logits are covered: one CTA for calls of at
most 64 tokens, the router over every SM then the sort for larger calls.
"""
import math

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

W_TOL = 2e-6


def route(logits, k, E, tile_m=128):
    T = logits.shape[0]
    lg = torch.from_numpy(np.ascontiguousarray(logits, np.float32)).cuda()
    ids = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), -7.0, dtype=torch.float32, device="cuda")
    r = mq.Routing(T, k, E, tile_m)
    mq.moe_route_logits(lg, k, tile_m, ids, w, r)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy(), r


def check_route(logits, k, E, tile_m=128):
    st, ids_ref, w_ref = oracle.router_topk(logits, k)
    assert st == oracle.OK
    ids, w, r = route(logits, k, E, tile_m)
    assert int(r.status.item()) == 0
    assert np.array_equal(ids, ids_ref)
    assert np.max(np.abs(w.astype(np.float64) - w_ref)) <= W_TOL
    st, sid, perm, counts = oracle.sort_assignments(ids_ref, E)
    assert np.array_equal(r.sorted_ids.cpu().numpy(), sid)
    assert np.array_equal(r.perm.cpu().numpy(), perm)
    assert np.array_equal(r.counts.cpu().numpy(), counts)
    st, off, tiles, tc = oracle.build_expert_tiles(sid, E, tile_m)
    assert np.array_equal(r.offsets.cpu().numpy(), off)
    assert int(r.tile_count.item()) == tc
    assert np.array_equal(r.tiles.cpu().numpy()[:3 * tc].reshape(-1, 3), tiles)
    return ids, w, r


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill_uniform", "prefill_skewed",
                                  "prefill_zipf"])
def test_route_logits_of_the_workloads(name):
    d = synth.make(name)
    check_route(d["router_logits"], d["k"], d["E"])


@pytest.mark.parametrize("T,E,k,tile_m,seed", [
    (1, 1, 1, 16, 0),          # one token, one expert
    (37, 5, 3, 32, 1),         # ragged
    (64, 256, 32, 64, 2),      # the most experts and the largest k, one launch
    (65, 256, 32, 128, 3),     # just past the one-launch bound
    (300, 33, 4, 16, 4),       # experts not a multiple of 32
])
def test_route_logits_shapes_with_ties(T, E, k, tile_m, seed):
    rng = np.random.default_rng(seed)
    logits = (np.round(rng.normal(size=(T, E)) * 2) / 2).astype(np.float32)  # many ties
    check_route(logits, k, E, tile_m)


def test_signed_zeros_are_equal_logits():
    """-0 and +0 are the same logit: the lower expert id comes first, whichever sign."""
    row = np.array([[-0.0, 0.0, -0.0, -1.0, 0.0]], np.float32)
    ids, w, _ = check_route(row, 4, 5)
    assert list(ids[0]) == [0, 1, 2, 4]


def test_minus_infinity_logits_are_chosen_last_with_zero_weight():
    T, E, k = 70, 16, 6
    rng = np.random.default_rng(9)
    logits = rng.normal(size=(T, E)).astype(np.float32)
    logits[:, 4:] = -np.inf  # four finite logits per token, k = 6
    ids, w, _ = check_route(logits, k, E)
    assert np.all(w[:, 4:] == 0.0) and np.all(np.sort(ids[:, :4], axis=1) == np.arange(4))


@pytest.mark.parametrize("T", [8, 200])
@pytest.mark.parametrize("bad", [math.nan, math.inf])
def test_bad_logits_raise_range_and_stop_the_route(T, bad):
    E, k = 64, 4
    logits = np.random.default_rng(1).normal(size=(T, E)).astype(np.float32)
    logits[T // 2, 7] = bad
    ids, w, r = route(logits, k, E)
    assert int(r.status.item()) == mq.MOE_ERR_RANGE
    assert int(r.tile_count.item()) == 0
    assert np.all(ids[T // 2] == -7)  # that token's outputs are not written


def test_router_alone_equals_the_oracle():
    d = synth.make("prefill_zipf")
    T, E, k = d["T"], d["E"], d["k"]
    lg = torch.from_numpy(d["router_logits"]).cuda()
    ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mq.moe_router_topk(lg, k, ids, w, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    st, ids_ref, w_ref = oracle.router_topk(d["router_logits"], k)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    assert np.max(np.abs(w.cpu().numpy().astype(np.float64) - w_ref)) <= W_TOL


@pytest.mark.parametrize("name", ["decode", "tiny"])
def test_layer_from_logits_matches_the_oracle(name):
    """Route from logits, then the two projections: y against the oracle's layer on the
    router's own ids and weights."""
    d = dict(synth.make(name))
    dev = to_device(d)
    T, E, k, H, I = d["T"], d["E"], d["k"], d["H"], d["I"]
    b = mq.MoeLayerBuffers(T, k, E, H, I, 128)
    lg = torch.from_numpy(d["router_logits"]).cuda()
    ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    mq.moe_route_logits(lg, k, 128, ids, w, b.routing)
    mq.moe_gather_qmm_glu(dev["x"], dev["Wgu"], dev["Sgu"], dev["Bgu"], b.routing, H, I, b.h)
    mq.moe_gather_qmm_down_unsort(b.h, dev["Wd"], dev["Sd"], dev["Bd"], b.routing, w, H, I,
                                  b.y_acc, b.y)
    torch.cuda.synchronize()
    assert int(b.routing.status.item()) == 0
    st, ids_ref, w_ref = oracle.router_topk(d["router_logits"], k)
    d["topk_ids"], d["topk_weights"] = ids_ref, w_ref
    ref = oracle.layer(d)
    assert excess(bf16_to_f64(b.y), ref["y"]) <= 1.0
