"""Ordering rules of weight-page movement (oracle; test infrastructure).

PagedWeight, Sec. 3.1: an offload first lowers the committed bitwidth q_i in the page
table and then moves the unneeded pages to CPU memory; a reload first moves the pages
back and raises q_i only once they are GPU-resident.  Sec. 3.3 / Fig. 4: inference keeps
running at the lowered bitwidth while the copy is in flight, and a raise is committed
after the reload lands.

A page is one bit-plane together with its LUT state; its state is GPU-resident,
CPU-resident or in transfer (Sec. 3.1).  This model tracks one block.
"""
from __future__ import annotations

GPU, CPU, TO_CPU, TO_GPU = "gpu", "cpu", "to_cpu", "to_gpu"


class StateError(Exception):
    pass


class BlockPages:
    def __init__(self, bits, bmax: int, q: int):
        self.bits = list(bits)
        self.bmax = bmax
        self.q = q
        self.pending = None          # reload target waiting for its pages
        self.state = [GPU if p < q else CPU for p in range(bmax)]

    def offload(self, q_new: int):
        if q_new not in self.bits or q_new >= self.q:
            raise StateError("offload needs a lower supported bitwidth")
        if self.pending is not None or any(self.state[p] != GPU for p in range(q_new, self.q)):
            raise StateError("pages to offload are not all GPU-resident")
        old = self.q
        self.q = q_new                      # lower the committed bitwidth first ...
        for p in range(q_new, old):         # ... then move the pages out
            self.state[p] = TO_CPU

    def reload(self, q_new: int):
        if q_new not in self.bits or q_new <= self.q:
            raise StateError("reload needs a higher supported bitwidth")
        if self.pending is not None or any(self.state[p] in (TO_CPU, TO_GPU) for p in range(self.q, q_new)):
            raise StateError("a page of the range is in transfer")
        for p in range(self.q, q_new):      # move the pages in; q stays where it is
            if self.state[p] == CPU:
                self.state[p] = TO_GPU
        self.pending = q_new

    def copies_landed(self):
        for p in range(self.bmax):
            if self.state[p] == TO_CPU:
                self.state[p] = CPU
            elif self.state[p] == TO_GPU:
                self.state[p] = GPU

    def commit(self) -> int:
        """Raise q to a pending reload target once its pages are resident; returns 0/1."""
        if self.pending is None:
            return 0
        if all(self.state[p] == GPU for p in range(self.q, self.pending)):
            self.q = self.pending
            self.pending = None
            return 1
        return 0

    def set_bits(self, q_new: int):
        if q_new not in self.bits:
            raise StateError("unsupported bitwidth")
        if any(self.state[p] != GPU for p in range(q_new)):
            raise StateError("a page below the new bitwidth is not GPU-resident")
        self.q = q_new
