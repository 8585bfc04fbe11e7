"""Helpers for the GPU parity tests: device copies (torch as the allocator) and
the comparison metrics the tolerances are stated in."""
import numpy as np


def _torch_dtype(dtype):
    import torch
    return {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[dtype]


def dev(a, dtype="f32"):
    t = __import__("torch").from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(_torch_dtype(dtype)).cuda()


def host(t):
    import torch
    torch.cuda.synchronize()
    return t.float().cpu().numpy().astype(np.float64)


def empty(shape, dtype="f32"):
    import torch
    return torch.zeros(shape, dtype=_torch_dtype(dtype), device="cuda")


def max_rel_floor(got, ref, floor):
    """max_i |got_i - ref_i| / max(|ref_i|, floor)"""
    got = np.asarray(got, dtype=np.float64).reshape(-1)
    ref = np.asarray(ref, dtype=np.float64).reshape(-1)
    return float(np.max(np.abs(got - ref) / np.maximum(np.abs(ref), floor))) if ref.size else 0.0


def rel_to_max(got, ref, floor=1e-6):
    """max |got - ref| / max(max|ref|, floor): an all-zero reference (e.g. the
    exact dQ of a one-position sequence) is compared in absolute terms."""
    got = np.asarray(got, dtype=np.float64).reshape(-1)
    ref = np.asarray(ref, dtype=np.float64).reshape(-1)
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), floor))


def cosine(a, b):
    a = np.asarray(a, dtype=np.float64).reshape(-1)
    b = np.asarray(b, dtype=np.float64).reshape(-1)
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    if na == 0 and nb == 0:
        return 1.0
    return float(a @ b / (na * nb))
