"""Helpers for the GPU parity tests: host<->device conversion of the shared
synthetic inputs, guarded output buffers (canary words around every output
the kernels write, checked after the call), and the error norm."""
import numpy as np

GUARD = 4096  # bytes of canary on each side
CANARY = 0x5A


def torch():
    import torch as _t
    return _t


def dev_bf16(bits):
    """numpy uint16 bf16 bit patterns -> CUDA bf16 tensor (same bits)."""
    t = torch()
    a = np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)
    return t.from_numpy(a).cuda().view(t.bfloat16)


def dev(arr):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(arr)).cuda()


class Guarded:
    """A device tensor with CANARY bytes before and after it."""

    def __init__(self, shape, dtype, fill=0):
        t = torch()
        self.shape, self.dtype = tuple(shape), dtype
        n = int(np.prod(shape)) if len(shape) else 1
        itemsize = t.empty(0, dtype=dtype).element_size()
        self.nbytes = n * itemsize
        self.raw = t.full((GUARD + self.nbytes + GUARD,), CANARY, dtype=t.uint8, device="cuda")
        body = self.raw[GUARD:GUARD + self.nbytes]
        self.t = body.view(dtype).view(self.shape)
        if fill is not None:
            self.t.fill_(fill)

    def check(self):
        t = torch()
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.nbytes:]
        assert bool((head == CANARY).all()), "write before the start of a device buffer"
        assert bool((tail == CANARY).all()), "write past the end of a device buffer"

    def numpy(self):
        self.check()
        return self.t.cpu().numpy()


def rel_err(y, ref):
    """max_i |y_i - ref_i| / max_i |ref_i| (the FFN parity norm)."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.max(np.abs(ref))
    if den == 0:
        return float(np.max(np.abs(y)))
    return float(np.max(np.abs(y - ref)) / den)


TOL = 2e-2  # max relative error of FFN outputs (bf16 weights, fp32 accumulation)


class _CAI:
    def __init__(self, ptr, shape, typestr):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr, "data": (int(ptr), False),
                                         "version": 2, "strides": None}


def device_view(ptr, shape, typestr):
    """A torch view of library-owned device memory (typestr like '<i4', '|u1', '<u2')."""
    return torch().as_tensor(_CAI(ptr, shape, typestr), device="cuda")


def u16_of(t):
    """bf16/int16 device tensor -> numpy uint16 bit patterns."""
    return t.contiguous().view(torch().int16).cpu().numpy().view(np.uint16)
