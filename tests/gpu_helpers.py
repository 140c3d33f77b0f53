"""Shared helpers for the GPU tests: device upload and error metrics.

Error metrics (output scale): relRMSE = RMS(O - O_ref) / RMS(O_ref) and
relMax = max |O - O_ref| / max |O_ref| over the compared elements.
"""
import numpy as np
import torch


def to_dev(*xs):
    return [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in xs]


def rel_errors(o_gpu, o_ref):
    o_gpu = np.asarray(o_gpu, np.float64)
    o_ref = np.asarray(o_ref, np.float64)
    d = o_gpu - o_ref
    rmse = float(np.sqrt(np.mean(d * d)) / max(np.sqrt(np.mean(o_ref * o_ref)), 1e-300))
    rmax = float(np.max(np.abs(d)) / max(np.max(np.abs(o_ref)), 1e-300))
    return rmse, rmax


def gather_rows(o, rows):
    """Rows (flat (b*H + h)*S + i indices) of a [B,H,S,D] device tensor, as float64 numpy."""
    D = o.shape[-1]
    flat = o.reshape(-1, D)
    idx = torch.as_tensor(rows, device=o.device, dtype=torch.long)
    return flat.index_select(0, idx).double().cpu().numpy()
