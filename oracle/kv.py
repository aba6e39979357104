"""KV-block accounting coupled to the weight pages (oracle; test infrastructure).

PagedWeight, Sec. 3.2 (Eq. 7): the planner's pressure is measured in KV blocks -- the
allocator wants T_blk free blocks of B_KV bytes and has F_blk -- and the byte target D is
max(0, T_blk + 1 - F_blk) * B_KV.  Sec. 3.3 (asynchronous page movement): while serving, the
planner follows the free KV blocks, the allocator's headroom and the KV growth that is still
pending, and the GPU pages that a finished offload retires become headroom that KV blocks
can take.

The pages give no formula for how those three signals make F_blk.  Readings taken here:

* One device budget of S bytes is shared by the weight pages the GPU holds (W bytes: the
  resident pages and any page still in transfer or not yet retired) and the KV blocks.
* Capacity: C = floor(max(0, S - W) / B) blocks.  Headroom: H = S - W - U * B bytes, with U
  the blocks that requests hold.
* Pending growth: a request may announce how many blocks it is about to need (p_r, which
  replaces its previous announcement); their sum P counts as taken.
* The free blocks the planner reads: F_blk = C - U - P.  It is negative when the weights or
  the announcements overcommit the budget.
* Growing request r by n blocks first draws on r's own announcement, c = min(n, p_r); the
  other n - c blocks must fit in F_blk.  A grow is all or nothing.  A release returns all of
  r's blocks and drops its announcement.
* Block ids are logical, in [0, floor(S / B)), and the lowest free id is granted first.

Parity: pinned by a hand-worked sequence (tests/golden/kv_hand.json) computed from these
readings; the pages print no numbers for it.
"""
from __future__ import annotations


class KVError(Exception):
    pass


class KVAllocator:
    def __init__(self, budget_bytes: int, block_bytes: int):
        if budget_bytes < 0 or block_bytes <= 0:
            raise KVError("budget must be >= 0 and the block size > 0")
        self.S = int(budget_bytes)
        self.B = int(block_bytes)
        self.W = 0
        self.n_ids = self.S // self.B
        self.free_ids = set(range(self.n_ids))
        self.held = {}      # request -> list of block ids, in the order granted
        self.announced = {}  # request -> blocks announced

    # ---- the three signals and F_blk
    def set_weight_bytes(self, w: int):
        if w < 0:
            raise KVError("weight bytes must be >= 0")
        self.W = int(w)

    def capacity(self) -> int:
        return max(0, self.S - self.W) // self.B

    def used(self) -> int:
        return sum(len(ids) for ids in self.held.values())

    def pending(self) -> int:
        return sum(self.announced.values())

    def free_blocks(self) -> int:
        return self.capacity() - self.used() - self.pending()

    def headroom(self) -> int:
        return self.S - self.W - self.used() * self.B

    def stats(self) -> dict:
        return {"budget_bytes": self.S, "block_bytes": self.B, "weight_bytes": self.W,
                "capacity_blocks": self.capacity(), "used_blocks": self.used(),
                "pending_blocks": self.pending(), "free_blocks": self.free_blocks(),
                "headroom_bytes": self.headroom()}

    # ---- requests
    def announce(self, r: int, n: int):
        if n < 0:
            raise KVError("announced blocks must be >= 0")
        if n == 0:
            self.announced.pop(r, None)
        else:
            self.announced[r] = int(n)

    def grow(self, r: int, n: int) -> list:
        if n < 0:
            raise KVError("blocks to grow must be >= 0")
        own = self.announced.get(r, 0)
        c = min(n, own)
        if n - c > self.free_blocks():
            raise KVError("not enough free KV blocks")
        ids = sorted(self.free_ids)[:n]
        for i in ids:
            self.free_ids.remove(i)
        self.held.setdefault(r, []).extend(ids)
        self.announce(r, own - c)
        return ids

    def release(self, r: int) -> int:
        ids = self.held.pop(r, [])
        self.free_ids.update(ids)
        self.announced.pop(r, None)
        return len(ids)

    def request(self, r: int):
        """(blocks held, blocks announced) of request r."""
        return len(self.held.get(r, [])), self.announced.get(r, 0)

    def blocks(self, r: int) -> list:
        return list(self.held.get(r, []))
