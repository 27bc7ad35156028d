"""Shared helpers for the parity tests (no arithmetic of the method here)."""

import numpy as np
import pytest
import torch

# Tolerances on the normwise relative error max|x - ref| / max|ref|.
TOL_DECODE = 1e-5    # FP32 decode and decode_k against the FP64 oracle
TOL_PREFILL = 2e-3   # tensor-core chunked prefill (TF32 and FP16 operands) or FP32 SIMT


def rel_err(x, ref) -> float:
    x = np.asarray(x.detach().double().cpu().numpy() if isinstance(x, torch.Tensor) else x,
                   dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    assert np.all(np.isfinite(x)), "non-finite values in the GPU result"
    den = np.abs(ref).max()
    return float(np.abs(x - ref).max() / (den if den > 0 else 1.0))


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def kda():
    need_gpu()
    import gated_delta_rule_prepare_gb300 as K
    return K
