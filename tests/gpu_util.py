"""Helpers shared by the GPU tests: device upload, tolerances, comparisons."""
from __future__ import annotations

import numpy as np

# The bar for bf16 outputs against the fp64 oracle (elementwise over B*Hq*D).
MAX_ABS = 2e-2
MEAN_ABS = 2e-3
# The bar between the tiled and the one-shot path, both in fp32 before rounding.
TILED_VS_ONESHOT = 1e-3


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


def assert_close_to_oracle(got: np.ndarray, ref: np.ndarray, what: str = ""):
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{what}: max|err|={mx:.3e} mean|err|={mean:.3e}"
    return mx, mean
