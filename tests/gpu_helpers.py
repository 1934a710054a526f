"""Helpers shared by the GPU parity tests (upload/download of bf16 bit patterns, tolerance)."""
import numpy as np


def to_dev_bf16(bits):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def bf16_to_f64(t):
    import torch
    u = t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return (u.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_bits(t):
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def tol_bound(ref):
    """Tolerance for bf16-in / fp32-accumulate outputs: 1e-2 * max|ref| + 1e-3."""
    return 1e-2 * float(np.max(np.abs(ref))) + 1e-3


def assert_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = float(np.max(np.abs(got - ref))) if got.size else 0.0
    bound = tol_bound(ref) if ref.size else 0.0
    assert err <= bound, f"{what}: max|gpu-ref| = {err:.3e} > {bound:.3e}"
    return err, bound


def workspace(nbytes):
    import torch
    return torch.zeros(max(int(nbytes), 16), dtype=torch.uint8, device="cuda")
