"""Shared helpers of the GPU parity tests (no method arithmetic here)."""
import os

import numpy as np
import pytest

try:
    import torch
except Exception:  # pragma: no cover
    torch = None

# Tolerances of the parity tests: fp32 scores and m / l
# within 1e-3 relative; bf16 attention outputs within 2e-2 max-abs; block
# tables, compacted bytes and selection on identical scores bit-exact.
REL_ML = 1e-3
REL_S = 1e-3
ABS_S = 1e-30
ABS_O = 2e-2


def need_gpu():
    if torch is None or not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def kvs_lib():
    need_gpu()
    from layer_wise_kv_gb300 import build, kvs
    build.build()
    kvs.library()
    return kvs


def dev_bf16(bits: np.ndarray):
    """bf16 bit patterns (uint16) -> CUDA bf16 tensor with the same bits."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.cuda()


def host_bits(t) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_f64(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_m(got, ref):
    err = np.abs(got - ref) / np.maximum(1.0, np.abs(ref))
    assert err.max() <= REL_ML, f"m: worst relative error {err.max():.3e}"


def check_rel(got, ref, rel, absol=0.0, what=""):
    err = np.abs(got - ref)
    bound = rel * np.abs(ref) + absol
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} values outside {rel} relative; worst "
                           f"{(err / np.maximum(np.abs(ref), 1e-300)).max():.3e}")


def check_kept(gpu_idx, ref_idx, ref_scores, n, k, recent):
    """Kept sets equal except swaps among keys whose oracle score lies within
    1e-3 relative of the k-th kept score (the selection runs on the GPU's own
    fp32 scores, which differ from the fp64 ones by rounding)."""
    g, r = set(gpu_idx.tolist()), set(ref_idx.tolist())
    assert len(g) == len(gpu_idx) == len(ref_idx)
    assert list(gpu_idx) == sorted(gpu_idx)
    if k >= n:
        assert g == r
        return 0
    assert set(range(n - recent, n)) <= g
    cand = ref_scores[: n - recent]
    kth = np.sort(cand)[::-1][k - recent - 1]
    diff = g ^ r
    for i in diff:
        assert abs(ref_scores[i] - kth) <= 1e-3 * kth, (i, ref_scores[i], kth)
    return len(diff)
