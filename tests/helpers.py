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


class Guarded:
    """A device output tensor placed between two sentinel bands of a larger
    buffer (the stand-in for an out-of-bounds checker): after the call,
    check() asserts that no byte of either band changed. The tensor itself is
    pre-filled with the same pattern, so elements a kernel never writes also
    stand out against the oracle."""

    BAND = 4096
    PATTERN = 0xA5

    def __init__(self, shape, dtype):
        import torch

        self.shape = tuple(int(d) for d in shape)
        item = torch.empty((), dtype=dtype).element_size()
        self.nbytes = int(np.prod(self.shape, dtype=np.int64)) * item
        body = (self.nbytes + 15) // 16 * 16
        self.raw = torch.full((self.BAND + body + self.BAND,), self.PATTERN, dtype=torch.uint8, device="cuda")
        self.t = self.raw[self.BAND:self.BAND + self.nbytes].view(dtype).view(self.shape)

    def check(self, what=""):
        import torch

        torch.cuda.synchronize()
        lo = self.raw[:self.BAND]
        hi = self.raw[self.BAND + self.nbytes:]
        bad_lo = int((lo != self.PATTERN).sum())
        bad_hi = int((hi != self.PATTERN).sum())
        assert bad_lo == 0 and bad_hi == 0, f"{what}: {bad_lo} bytes before and {bad_hi} after the output changed"
