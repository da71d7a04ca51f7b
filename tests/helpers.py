"""Shared helpers for the tests: host<->device conversion and the acceptance
tolerance for bf16 outputs (relative Frobenius error <= 5e-3 and max-abs error
<= 1e-2 * max|y_ref|, against the float64 oracle)."""

import numpy as np

REL_FRO = 5e-3
REL_MAX = 1e-2


def to_dev_bf16(bits_u16):
    import torch

    a = np.ascontiguousarray(bits_u16, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()


def to_dev(a, dtype=None):
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def bf16_dev_to_bits(t):
    import torch

    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_dev_to_f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def packed_dev_to_u32(t):
    return t.detach().cpu().numpy().view(np.uint32)


def errors(y, y_ref):
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    err = y - y_ref
    fro = np.linalg.norm(err) / max(np.linalg.norm(y_ref), 1e-300)
    mx = np.max(np.abs(err)) / max(np.max(np.abs(y_ref)), 1e-300) if y.size else 0.0
    return fro, mx


def assert_bf16_close(y_dev, y_ref, what=""):
    fro, mx = errors(bf16_dev_to_f64(y_dev), y_ref)
    assert fro <= REL_FRO and mx <= REL_MAX, f"{what}: rel_fro={fro:.3e} rel_max={mx:.3e}"
    return fro, mx
