"""Tolerances and comparison helpers for GPU-vs-oracle parity.

Attention outputs (bf16 inputs, fp32 accumulation): max-abs <= 1e-2 and mean-abs <= 1e-3
against the fp64 oracle, plus a relative-L2 guard <= 1e-2 so that a near-zero output
cannot pass on small-magnitude workloads. The float32 path is held to 1e-4 max-abs.

Stress cases outside the named workloads (entries scaled so that outputs reach several
units) add a relative term RTOL * |ref| to both bounds: the bf16 output alone rounds with
relative error up to 2^-9, and the bf16 probabilities fed to the value product add about
as much again, so RTOL = 2^-7 keeps a 2x margin over both.
"""
import numpy as np
import torch

MAX_ABS = 1e-2
MEAN_ABS = 1e-3
REL_L2 = 1e-2
RTOL_STRESS = 2.0 ** -7


def to_np(t):
    return t.detach().to("cpu", torch.float64).numpy() if isinstance(t, torch.Tensor) else np.asarray(t)


def assert_attn_close(gpu, ref, max_abs=MAX_ABS, mean_abs=MEAN_ABS, rel_l2=REL_L2, what="",
                      rtol=0.0):
    g = to_np(gpu).astype(np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    d = np.abs(g - r)
    mx, mn = float(d.max()), float(d.mean())
    rl = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30))
    ok_elem = bool(np.all(d <= max_abs + rtol * np.abs(r)))
    ok_mean = mn <= mean_abs + rtol * float(np.abs(r).mean())
    assert ok_elem and ok_mean and rl <= rel_l2, \
        f"{what}: max-abs {mx:.3e} mean-abs {mn:.3e} rel-l2 {rl:.3e} (rtol {rtol})"
    return mx, mn, rl
