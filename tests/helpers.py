"""Shared test plumbing: the oracle's workload adapter (oracle.from_workload)
under the names the tests use, the oracle thread count, and guard bands around
GPU output buffers.  Nothing here computes attention or quantises."""
import os

import torch

from oracle.from_workload import ODT, OCACHE, bits, np_i32, np_i64  # noqa: F401
from oracle.from_workload import attention as oracle_attention  # noqa: F401
from oracle.from_workload import cache_after_step as oracle_cache_after_step  # noqa: F401


# oracle threads for full-size comparisons: every host core
ALL_CORES = os.cpu_count() or 8

GUARD_BYTES = 4096
# quiet-NaN patterns written into a guarded buffer (output and bands alike)
_CANARY = {torch.float32: (torch.int32, 0x7FC0DEAD), torch.float16: (torch.int16, 0x7E5A),
           torch.bfloat16: (torch.int16, 0x7FDA)}


class GuardedOut:
    """An output buffer with GUARD_BYTES of canary bytes on each side.

    The output and both bands start as a NaN bit pattern, so an element the
    kernel never writes stays NaN (and fails parity) and a write past either end
    of the output changes a band; check() asserts both bands are untouched."""

    def __init__(self, shape, dtype, device):
        ity, pat = _CANARY[dtype]
        esz = torch.empty((), dtype=dtype).element_size()
        self.g = GUARD_BYTES // esz
        self.n = 1
        for x in shape:
            self.n *= int(x)
        self.pattern = pat
        self.buf = torch.full((self.n + 2 * self.g,), pat, dtype=ity, device=device).view(dtype)
        self.out = self.buf[self.g:self.g + self.n].view(tuple(shape))

    def refill(self):
        ity, _ = _CANARY[self.out.dtype]
        self.buf.view(ity).fill_(self.pattern)

    def check(self):
        ity, _ = _CANARY[self.out.dtype]
        raw = self.buf.view(ity)
        head, tail = raw[:self.g], raw[self.g + self.n:]
        bad = int((head != self.pattern).sum()) + int((tail != self.pattern).sum())
        assert bad == 0, f"{bad} guard-band elements around the output were overwritten"


def guard(st):
    """Give a DecodeStep a guarded output buffer (same shape and dtype); returns
    the guard, whose check() the caller runs after the step."""
    g = GuardedOut(st.out.shape, st.out.dtype, st.out.device)
    st.out = g.out
    return g
