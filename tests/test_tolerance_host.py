"""The comparison bars of the GPU parity tests, checked on the CPU against the
oracle itself: the combine-propagation allowance covers exactly what one-ulp
differences in the BF16 y rows do to the output, and the plain bar does not."""
import numpy as np
import pytest

import oracle
import synth
from tests import gpu_util as gu


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


def _one_ulp_neighbours(bits: np.ndarray, rng) -> np.ndarray:
    """Each BF16 value moved one ulp up or down in magnitude (random), zeros kept."""
    b = np.asarray(bits, np.uint16).astype(np.int32)
    step = rng.choice([-1, 1], size=b.shape)
    mag = b & 0x7FFF
    moved = np.where(mag == 0, b, (b & 0x8000) | np.clip(mag + step, 1, 0x7F7F))
    return moved.astype(np.uint16)


def test_combine_propagation_bound_covers_one_ulp_y_differences():
    w = synth.Workload("tol", T=64, K=256, N=128, E=8, topk=4, bits=2, g13=128, g2=128,
                       scale_lo=0.5, scale_hi=2.0, zipf_s=0.0)
    inp = synth.make_all(w, 3)
    out, _, y = oracle.forward(inp["x"], inp["ids"], inp["weights"], inp["w13_packed"], inp["w13_scales"],
                               inp["w2_packed"], inp["w2_scales"], bits=w.bits, group_size=w.g13,
                               swiglu_limit=w.swiglu_limit, return_intermediates=True)
    bound = gu.y_ulp_bound(y, inp["weights"])
    rng = np.random.default_rng(0)
    worst_plain = 0.0
    for _ in range(4):
        y2 = _one_ulp_neighbours(y, rng)
        part = oracle.combine_partial(inp["ids"], inp["weights"], y2, (0, w.E))
        out2 = oracle.sum_partials([part])
        s = gu.compare_bf16(out2, out, "one-ulp y neighbours", y_bound=bound)
        assert s["beyond"] == 0, s
        plain = gu.compare_bf16(out2, out, "plain bar")
        worst_plain = max(worst_plain, plain["max_abs_excess"])
    # the mechanism is real: without the allowance some outputs leave the plain bar
    assert worst_plain > 0.0


def test_combine_propagation_bound_rejects_a_two_ulp_error_in_out():
    w = synth.Workload("tol2", T=32, K=256, N=128, E=4, topk=2, bits=2, g13=128, g2=128,
                       scale_lo=0.5, scale_hi=2.0, zipf_s=0.0)
    inp = synth.make_all(w, 5)
    out, _, y = oracle.forward(inp["x"], inp["ids"], inp["weights"], inp["w13_packed"], inp["w13_scales"],
                               inp["w2_packed"], inp["w2_scales"], bits=w.bits, group_size=w.g13,
                               swiglu_limit=w.swiglu_limit, return_intermediates=True)
    bound = gu.y_ulp_bound(y, inp["weights"])
    r = gu.bf16_bits_to_f64(out)
    i = int(np.argmax(np.abs(r)))
    bad = out.copy().reshape(-1)
    # move the largest output (scales of 0.5-2 make it large) by enough ulps to
    # exceed every allowance
    u = gu.ulp_of(r.reshape(-1)[i])
    need = max(gu.MAX_ABS, bound.reshape(-1)[i] + 2 * gu.ulp_of(abs(r.reshape(-1)[i]) + bound.reshape(-1)[i])) / u
    bad[i] = np.uint16(int(bad[i]) + int(np.ceil(need)) + 1)
    s = gu.compare_bf16(bad.reshape(out.shape), out, "planted", y_bound=bound)
    assert s["beyond"] == 1, s
