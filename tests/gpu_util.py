"""Helpers for the GPU parity tests: host inputs -> device tensors, oracle
runs on the host, and the comparison metrics with the tolerances of the
path (routing indices and packed words: bit-exact; BF16 tensors: relative
L2 <= 1e-3, and max-abs <= 2e-2 where the BF16 spacing of the reference
value is finer than that -- an element whose reference has a BF16 ulp above
2e-2 (|ref| >= 4) may differ by that one ulp, the smallest difference BF16
can express there; at most 0.1 % of the elements may need that allowance).

For the forward's output, where the oracle's y is at hand, an element may
also differ by as much as a one-ulp difference in the BF16 y of each of its
top-k slots moves it, plus the two final roundings: B + ulp(|out| + B) with
B = sum_j |w_j| ulp(y_j) (y is rounded to BF16 before the combine on both
sides, and a y computed with fp32 sums may land one ulp from the fp64 one;
each rounding of out moves it by at most half the BF16 spacing where it
lands); at most 1e-5 of the elements may need that."""
from __future__ import annotations

import numpy as np
import torch

MAX_ABS = 2e-2
REL_L2 = 1e-3


def bf16_bits_to_f64(bits) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def to_dev(inp: dict, device="cuda") -> dict:
    return dict(
        x=dev_bf16(inp["x"], device),
        topk_ids=torch.from_numpy(np.ascontiguousarray(inp["ids"], np.int32)).to(device),
        topk_weights=torch.from_numpy(np.ascontiguousarray(inp["weights"], np.float32)).to(device),
        w13_packed=torch.from_numpy(inp["w13_packed"]).to(device),
        w13_scales=torch.from_numpy(inp["w13_scales"]).to(device),
        w2_packed=torch.from_numpy(inp["w2_packed"]).to(device),
        w2_scales=torch.from_numpy(inp["w2_scales"]).to(device),
    )


def ulp_of(v: np.ndarray) -> np.ndarray:
    """One BF16 ulp of each value (the spacing above |v|)."""
    return np.ldexp(1.0, np.frexp(np.maximum(np.abs(v), 2.0 ** -126))[1] - 8)


def y_ulp_bound(y_ref_bits, weights) -> np.ndarray:
    """Per output element [tokens, K]: sum_j |w_j| ulp(y_j) over the token's
    top-k slots, y_ref in slot order [tokens * topk, K], weights [tokens, topk]."""
    w = np.abs(np.asarray(weights, np.float64))
    y = bf16_bits_to_f64(y_ref_bits).reshape(w.shape[0], w.shape[1], -1)
    return np.einsum("tj,tjk->tk", w, ulp_of(y))


def compare_bf16(got_bits, ref_bits, what: str = "", y_bound=None) -> dict:
    g = bf16_bits_to_f64(got_bits)
    r = bf16_bits_to_f64(ref_bits)
    assert g.shape == r.shape, (g.shape, r.shape)
    d = np.abs(g - r)
    denom = np.sqrt(np.sum(r * r))
    rel = float(np.sqrt(np.sum(d * d)) / denom) if denom > 0 else float(np.sqrt(np.sum(d * d)))
    gi = np.asarray(got_bits, np.uint16).astype(np.int32)
    ri = np.asarray(ref_bits, np.uint16).astype(np.int32)
    # ulp distance of bf16 patterns (same sign assumed for nearby values)
    ulp = np.abs(gi - ri)
    # one BF16 ulp of each reference value (spacing above |ref|)
    ulp_ref = ulp_of(r)
    allowed = np.maximum(MAX_ABS, ulp_ref)
    propagated = 0
    if y_bound is not None:
        # the combine's propagation of one-ulp differences in y (see the module docstring)
        B = np.asarray(y_bound, np.float64).reshape(r.shape)
        wider = np.maximum(allowed, B + ulp_of(np.abs(r) + B))
        propagated = int(((d > allowed) & (d <= wider)).sum())
        allowed = wider
    stats = dict(what=what, n=int(g.size), max_abs=float(d.max()) if d.size else 0.0, rel_l2=rel,
                 max_abs_excess=float((d - allowed).max()) if d.size else 0.0,
                 # elements inside the bar only through the one-ulp allowance for |ref| >= 4
                 widened=int((d > MAX_ABS).sum()),
                 propagated=propagated,
                 beyond=int((d > allowed).sum()),
                 exact=float((ulp == 0).mean()) if ulp.size else 1.0,
                 le1ulp=float((ulp <= 1).mean()) if ulp.size else 1.0,
                 nonfinite=int((~np.isfinite(g)).sum()))
    return stats


# At most this fraction of the elements may rely on the one-ulp allowance,
# and at most MAX_PROPAGATED_FRAC on the combine's propagation of y's ulps.
MAX_WIDENED_FRAC = 1e-3
MAX_PROPAGATED_FRAC = 1e-5


def assert_close(got_bits, ref_bits, what: str = "", max_abs=MAX_ABS, rel_l2=REL_L2, y_bound=None) -> dict:
    s = compare_bf16(got_bits, ref_bits, what, y_bound=y_bound)
    print(s)
    assert s["nonfinite"] == 0, s
    assert s["rel_l2"] <= rel_l2, s
    if max_abs == MAX_ABS:
        assert s["max_abs_excess"] <= 0.0, s
        assert s["widened"] <= MAX_WIDENED_FRAC * s["n"], s
        assert s["propagated"] <= MAX_PROPAGATED_FRAC * s["n"], s
    else:
        assert s["max_abs"] <= max_abs, s
    return s
