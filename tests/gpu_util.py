"""Helpers shared by the GPU tests: device upload, tolerances, comparisons."""
from __future__ import annotations

import numpy as np

# The bar for bf16 outputs against the fp64 oracle (elementwise over B*Hq*D).
MAX_ABS = 2e-2
MEAN_ABS = 2e-3
# The bar between the tiled and the one-shot path, both in fp32 before rounding.
TILED_VS_ONESHOT = 1e-3
# Regression guard on the kernel's own arithmetic: beyond the half bf16 step
# the output rounding may cost, the fp32 path adds at most ~2^-17 * max|v|
# (softmax weights enter P.V as bf16 hi + lo parts, exact to 2^-17 relative;
# |v| <= ~6 for the N(0,1) draws of the workloads), about 4.6e-5.  Measured:
# a few 1e-6.  Dropping the lo part alone would cost ~2^-9 relative.
EXCESS_GUARD = 5e-5

# Achieved errors of every oracle comparison in this session (printed at the
# end of the run by conftest.py; report only).
ERROR_LOG: list = []


def dev(a: np.ndarray):
    """numpy -> CUDA tensor; uint16 arrays are bf16 bit patterns."""
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_f64(t) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def upload(w):
    return dict(q=dev(w.q), k_pool=dev(w.k_pool), v_pool=dev(w.v_pool),
                block_table=dev(w.block_table), seq_lens=dev(w.seq_lens))


def context_for(w, max_seqs=None, tile_capacity=64):
    import paged_gqa_decode_05_gb300 as pda
    return pda.Context(max_seqs=max_seqs or max(w.B, 1), num_q_heads=w.Hq, num_kv_heads=w.Hkv,
                       head_dim=w.D, block_size=w.block_size, tile_capacity=tile_capacity)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values (8 significant bits) around each |x| (0 at 0)."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    e = np.frexp(x)[1]
    return np.where(x > 0, np.ldexp(1.0, e - 8), 0.0)


def bf16_rn(x: np.ndarray) -> np.ndarray:
    """x rounded to the nearest bf16 value, ties to even (normal range)."""
    x = np.asarray(x, dtype=np.float64)
    q = bf16_ulp(x)
    return np.where(q > 0, np.round(x / np.where(q > 0, q, 1.0)) * q, 0.0)


def rounding_report(got: np.ndarray, ref: np.ndarray) -> dict:
    """How the output relates to the correctly rounded oracle value:
    the fraction equal to bf16_rn(ref), the largest distance from it in bf16
    steps, and the largest error beyond the half step the output rounding
    itself may cost (what the kernel's fp32 arithmetic added)."""
    if got.size == 0:
        return {"exact_frac": 1.0, "max_steps": 0.0, "excess": 0.0}
    rn = bf16_rn(ref)
    step = bf16_ulp(np.maximum(np.abs(got), np.abs(ref)))
    dist = np.abs(got - rn)
    steps = np.where(step > 0, dist / np.where(step > 0, step, 1.0), 0.0)
    excess = np.abs(got - ref) - 0.5 * step
    return {"exact_frac": float(np.mean(got == rn)), "max_steps": float(steps.max()),
            "excess": float(max(excess.max(), 0.0))}


def assert_close_to_oracle(got: np.ndarray, ref: np.ndarray, what: str = "", rounded: bool = True):
    """The task's bar (max |err| <= 2e-2, mean |err| <= 2e-3), and the
    regression guard EXCESS_GUARD on the error beyond the output rounding (on
    the whole error for fp32 outputs, rounded=False).  The achieved errors, and
    for bf16 outputs their relation to bf16_rn(ref), are logged."""
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    rec = {"what": what, "max": mx, "mean": mean}
    if rounded:
        rec.update(rounding_report(got, ref))
    ERROR_LOG.append(rec)
    assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{what}: max|err|={mx:.3e} mean|err|={mean:.3e}"
    excess = rec["excess"] if rounded else mx
    assert excess <= EXCESS_GUARD, f"{what}: error beyond the output rounding {excess:.3e}"
    return mx, mean
