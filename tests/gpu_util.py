"""Helpers shared by the GPU tests and the smoke check: host <-> device copies
with the same bits, library weight structs over device tensors, the parity
tolerance."""
import numpy as np

from speculative_decode_verification_gb300 import binding as B

# spec tolerance for floating point: max |gpu - oracle| <= 1e-3 * rms(oracle)
TOL = 1e-3


def dev(a):
    import torch

    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16))
    elif a.dtype == np.uint32:
        t = torch.from_numpy(a.view(np.int32))
    else:
        t = torch.from_numpy(a)
    return t.cuda()


def host(t, dtype=None):
    a = t.detach().cpu().numpy()
    if dtype is not None:
        a = a.view(dtype)
    return a


class DevQ4:
    """A Q4Matrix (synth) copied to the device in the row layout (`rows`), and
    its tiled form for the compute calls (`struct`, kept alive by `tiled`):
    gate_up / down for an expert's gate/up or down matrix, else dense."""

    def __init__(self, vf, m, gate_up=False, down=False):
        self.packed, self.scales, self.biases = dev(m.packed), dev(m.scales), dev(m.biases)
        if m.packed.ndim == 3:
            self.rows = B.q4_experts(self.packed, self.scales, self.biases)
        else:
            self.rows = B.q4_weight(self.packed, self.scales, self.biases)
        self.tiled = vf.tile(self.rows, gate_up=gate_up, down=down)
        self.struct = self.tiled.struct


def rel_err(gpu, ref):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref * ref))
    return float(np.max(np.abs(gpu - ref)) / rms) if rms > 0 else float(np.max(np.abs(gpu - ref)))


def assert_close(gpu, ref, tol=TOL, what=""):
    e = rel_err(gpu, ref)
    assert e <= tol, f"{what}: max|gpu-oracle|/rms(oracle) = {e:.3e} > {tol:.1e}"
    return e


def bf16_to_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
