"""Helpers shared by the parity tests: tolerances and comparisons against the oracle."""
import numpy as np
import torch

# Tolerances (fixed by the target: fp32 max-abs 1e-4; bf16 max-abs 2e-2 and relative L2 <= 5e-3).
F32_MAX_ABS = 1e-4
BF16_MAX_ABS = 2e-2
BF16_REL_L2 = 5e-3


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def errors(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    diff = got - ref
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    denom = float(np.linalg.norm(ref))
    rel_l2 = float(np.linalg.norm(diff) / denom) if denom > 0 else float(np.linalg.norm(diff))
    return max_abs, rel_l2


def assert_close(got, ref, dtype, what, max_abs=None, rel_l2=None, stored_bf16=False):
    """fp32: max-abs <= 1e-4.  bf16: max-abs <= 2e-2 and relative L2 <= 5e-3.

    stored_bf16: the result is stored in bfloat16, whose rounding alone moves a value x by up to
    2^-8 |x|; each element may then differ by 2e-2 + 2^-8 |ref|."""
    if stored_bf16:
        got = np.asarray(got, np.float64)
        ref = np.asarray(ref, np.float64)
        excess = np.abs(got - ref) - (BF16_MAX_ABS + np.abs(ref) * 2.0 ** -8)
        worst = float(excess.max()) if excess.size else 0.0
        assert worst <= 0, f"{what}: bf16-stored element off by {worst:.3e} beyond 2e-2 + 2^-8|x|"
        _, rl = errors(got, ref)
        assert rl <= BF16_REL_L2, f"{what}: rel-L2 {rl:.3e} > {BF16_REL_L2}"
        return worst, rl
    ma, rl = errors(got, ref)
    if dtype == torch.float32:
        lim = F32_MAX_ABS if max_abs is None else max_abs
        assert ma <= lim, f"{what}: max-abs {ma:.3e} > {lim:.1e}"
    else:
        lim_a = BF16_MAX_ABS if max_abs is None else max_abs
        lim_r = BF16_REL_L2 if rel_l2 is None else rel_l2
        assert ma <= lim_a and rl <= lim_r, f"{what}: max-abs {ma:.3e} (<= {lim_a}), rel-L2 {rl:.3e} (<= {lim_r})"
    return ma, rl
