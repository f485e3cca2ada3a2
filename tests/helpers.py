"""Shared helpers for the GPU parity tests (test infrastructure only)."""
import numpy as np
import torch

import oracle

# Tolerances of the numeric contract: |logp_gpu - logp_oracle| <= 1e-3 absolute;
# gradient relative L2 error <= 2e-3 (GPU bf16 converted to fp64 against the
# unrounded fp64 oracle, over the whole tensor).
LOGP_ATOL = 1e-3
GRAD_REL_L2 = 2e-3


def dev():
    return torch.device("cuda:0")


def f64(t):
    """exact float64 copy of a bf16 / fp32 tensor (CPU numpy)."""
    if t.dtype == torch.bfloat16:
        return oracle.bf16_bits_to_f64(t.detach().cpu())
    return t.detach().cpu().double().numpy()


def rel_l2(gpu, ref):
    g = f64(gpu) if isinstance(gpu, torch.Tensor) else gpu
    num = np.linalg.norm((g - ref).ravel())
    den = np.linalg.norm(ref.ravel())
    return num / den


def same_bits(a, b):
    return torch.equal(a.contiguous().view(torch.int32) if a.dtype == torch.float32 else
                       a.contiguous().view(torch.int16),
                       b.contiguous().view(torch.int32) if b.dtype == torch.float32 else
                       b.contiguous().view(torch.int16))
