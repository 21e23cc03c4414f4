"""Helpers shared by the GPU parity tests: host<->device marshalling and the
tolerance check |y - y_ref| <= tol, element by element."""
import numpy as np
import torch

import synth


def dev_weight(w: synth.QuantWeight, device="cuda"):
    codes = torch.from_numpy(np.ascontiguousarray(w.codes).view(np.int32)).to(device)
    return (codes, torch.from_numpy(np.ascontiguousarray(w.scales)).to(device),
            torch.from_numpy(np.ascontiguousarray(w.biases)).to(device))


def dev16(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float16)).to(device)


def plain_tol(bound):
    """Tolerance of a plain matvec: 2e-3 * (sum |w||x| (+ |r|)) + 1e-5."""
    return 2e-3 * bound + 1e-5


def check(y_gpu, y_ref, tol, what):
    y = y_gpu.detach().float().cpu().numpy().astype(np.float64).reshape(np.shape(y_ref))
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    err = np.abs(y - y_ref)
    ratio = err / tol
    bad = int(np.count_nonzero(ratio > 1.0))
    worst = float(ratio.max()) if ratio.size else 0.0
    assert bad == 0, (f"{what}: {bad} of {ratio.size} outputs outside tolerance "
                      f"(worst |err|/tol = {worst:.3g} at {np.unravel_index(ratio.argmax(), ratio.shape)})")
    return worst
