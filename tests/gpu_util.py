"""Helpers for the GPU parity tests: host inputs -> device tensors, oracle
runs on the host, and the comparison metrics with the tolerances of the
path (routing indices and packed words: bit-exact; BF16 tensors: relative
L2 <= 1e-3, and max-abs <= 2e-2 where the BF16 spacing of the reference
value is finer than that -- an element whose reference has a BF16 ulp above
2e-2 (|ref| >= 4) may differ by that one ulp, the smallest difference BF16
can express there; at most 0.1 % of the elements may need that allowance)."""
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


def compare_bf16(got_bits, ref_bits, what: str = "") -> dict:
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
    ulp_ref = np.ldexp(1.0, np.frexp(np.maximum(np.abs(r), 2.0 ** -126))[1] - 8)
    allowed = np.maximum(MAX_ABS, ulp_ref)
    stats = dict(what=what, n=int(g.size), max_abs=float(d.max()) if d.size else 0.0, rel_l2=rel,
                 max_abs_excess=float((d - allowed).max()) if d.size else 0.0,
                 # elements inside the bar only through the one-ulp allowance for |ref| >= 4
                 widened=int((d > MAX_ABS).sum()),
                 beyond=int((d > allowed).sum()),
                 exact=float((ulp == 0).mean()) if ulp.size else 1.0,
                 le1ulp=float((ulp <= 1).mean()) if ulp.size else 1.0,
                 nonfinite=int((~np.isfinite(g)).sum()))
    return stats


# At most this fraction of the elements may rely on the one-ulp allowance.
MAX_WIDENED_FRAC = 1e-3


def assert_close(got_bits, ref_bits, what: str = "", max_abs=MAX_ABS, rel_l2=REL_L2) -> dict:
    s = compare_bf16(got_bits, ref_bits, what)
    print(s)
    assert s["nonfinite"] == 0, s
    assert s["rel_l2"] <= rel_l2, s
    if max_abs == MAX_ABS:
        assert s["max_abs_excess"] <= 0.0, s
        assert s["widened"] <= MAX_WIDENED_FRAC * s["n"], s
    else:
        assert s["max_abs"] <= max_abs, s
    return s
