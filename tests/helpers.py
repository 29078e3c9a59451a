"""Shared helpers for the GPU parity tests (marshalling and comparisons only)."""
import numpy as np
import torch

import workloads as W


def rel_l2(x, y):
    """||x - y||_2 / ||y||_2 over the whole tensor in fp64 (absolute if ||y|| = 0)."""
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    ny = np.linalg.norm(y)
    d = np.linalg.norm(x - y)
    return float(d / ny) if ny > 0 else float(d)


def dev_tensor(a, dtype, device="cuda"):
    """Stored workload array (bf16 bits or fp32) -> CUDA tensor of that dtype."""
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device)


def i32(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(device)


def to_np(t):
    return t.float().cpu().numpy().astype(np.float64)


def wid(case, name):
    return W.widen(case[name], case["dtype"])


def tol_out(dtype):
    """Outputs: rel-L2 5e-3 from bf16 inputs, 1e-4 when everything is fp32."""
    return 5e-3 if dtype == "bf16" else 1e-4


TOL_STATE = 1e-4  # fp32 states and snapshots


def worst_seq_head(x, y, cu_seqlens):
    """Largest rel-L2 over the (sequence, head) blocks of [T, H, d] rows: a wrong
    sequence or head cannot hide inside the whole-tensor figure."""
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    cu = np.asarray(cu_seqlens)
    worst = 0.0
    for n in range(len(cu) - 1):
        a, b = int(cu[n]), int(cu[n + 1])
        if b > a:
            for h in range(x.shape[1]):
                worst = max(worst, rel_l2(x[a:b, h], y[a:b, h]))
    return worst


def worst_state(x, y):
    """Largest rel-L2 over the 128 x 128 state blocks of two arrays shaped
    [..., 128, 128] (one block per slot / snapshot and head)."""
    x = np.asarray(x, np.float64).reshape(-1, 128 * 128)
    y = np.asarray(y, np.float64).reshape(-1, 128 * 128)
    return max((rel_l2(a, b) for a, b in zip(x, y)), default=0.0)
