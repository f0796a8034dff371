"""The seeded input generator: determinism and the workload properties it promises."""
import numpy as np
import pytest

import oracle
import synth
from _util import bf16_bits


def test_counter_generator_is_deterministic_and_streams_differ():
    a = synth.normals(0, 1, 1000)
    b = synth.normals(0, 1, 1000)
    c = synth.normals(0, 2, 1000)
    assert np.array_equal(a, b)
    assert not np.allclose(a, c)
    assert abs(a.mean()) < 0.15 and abs(a.std() - 1.0) < 0.1


def test_quantisation_round_trip_is_within_half_a_step():
    packed, s, b = synth.quantized_weights(0, 77, 2, 16, 256)
    W = oracle.dequant_matrix(packed.reshape(32, 32), s.reshape(32, 4), b.reshape(32, 4))
    # regenerate the fp32 weights the quantiser saw
    w = synth.normals(0, 77, 2 * 16 * 256, std=synth.WEIGHT_STD).astype(np.float32)
    w = w.astype(np.float64).reshape(32, 256)
    step = synth.bf16_bits_to_f64(s).reshape(32, 4).repeat(64, axis=1)
    # half a step, plus slack for the bf16 rounding of scale and bias
    assert np.all(np.abs(W - w) <= 0.5 * step + 2.0**-8 * (np.abs(w) + 16 * step) + 1e-12)


def test_workload_shapes_and_routers():
    d = synth.make("tiny")
    assert d["x"].shape == (32, 128) and d["topk_ids"].shape == (32, 2)
    assert d["Wgu"].shape == (8, 128, 16) and d["Sgu"].shape == (8, 128, 2)
    assert d["Wd"].shape == (8, 128, 8) and d["Sd"].shape == (8, 128, 1)
    for t in range(d["T"]):
        assert len(set(d["topk_ids"][t].tolist())) == 2
    assert np.allclose(d["topk_weights"].sum(1), 1.0, atol=1e-6)
    assert np.all(np.diff(d["topk_weights"], axis=1) <= 0)  # descending logits


def test_zipf_router_leaves_at_least_eight_experts_empty():
    ids, w = synth.router("prefill_zipf", 2048, 128, 8)
    counts = np.bincount(ids.ravel(), minlength=128)
    assert (counts == 0).sum() >= 8
    assert counts.sum() == 16384
    assert counts.max() > 8 * counts[counts > 0].min()  # heavy head
    assert all(len(set(r.tolist())) == 8 for r in ids)


@pytest.mark.parametrize("activation", ["gelu_tanh", "silu"])
def test_activation_grid_isolates_the_gate_activation(activation):
    """The grid layer's gate pre-activations are the given values and its up ones 1.0, so the
    oracle's h is the activation at those values alone (exactly), and y is zero."""
    bits = bf16_bits(np.linspace(-12.0, 12.0, 128))
    d = synth.activation_grid(bits)
    ref = oracle.layer(d, activation=activation)
    z = synth.bf16_bits_to_f64(bits)
    f = oracle.gelu_tanh if activation == "gelu_tanh" else oracle.silu
    assert np.array_equal(ref["h"][0], f(z))
    assert not np.any(ref["y"])
    with pytest.raises(ValueError):
        synth.activation_grid(bits[:100])
