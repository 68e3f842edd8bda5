"""Helpers shared by the GPU parity tests: numpy <-> torch transfer of bf16
bit patterns, the tolerance check, and device buffers for one problem."""
import numpy as np

ATOL = 2e-2
RTOL = 1e-2


def to_dev(a, dtype=None):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    t = torch.from_numpy(a)
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def bits(t) -> np.ndarray:
    """bf16 CUDA tensor -> uint16 numpy bit patterns."""
    import torch
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_f64(b) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def assert_close(gpu, ref, what="", atol=ATOL, rtol=RTOL):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU values"
    err = np.abs(gpu - ref)
    bad = err > atol + rtol * np.abs(ref)
    if np.any(bad):
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tol; max err "
                             f"{err.max():.3e}; first {idx.tolist()} gpu {gpu[bad][:5]} "
                             f"ref {ref[bad][:5]}")


def rel_rms_err(gpu, ref):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.sqrt(np.mean((gpu - ref) ** 2)) / max(np.sqrt(np.mean(ref ** 2)), 1e-30))
