"""Shared test helpers: move generated bf16 bits to the device and compare."""
import numpy as np


def to_dev_bf16(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def weights_to_dev(wbits: dict) -> dict:
    return {k: to_dev_bf16(v) for k, v in wbits.items()}


def err_scale(got, ref) -> float:
    """max|got - ref| / max|ref| (the GEMM gate of the metalgemm ledger)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))


def cosine(a, b) -> float:
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b)))
