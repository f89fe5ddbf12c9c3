"""Host-tier admission and eviction for the block repository (test infrastructure:
only tests/, the smoke check and the bench's CPU baseline use this package).

KVMem: Virtualizing Million-Token Agent Workspaces on a Consumer GPU, §4.4
(retrieval-aware hierarchical reuse): host memory holds a bounded set of
blocks; admission and eviction weigh both recent retrieval and cumulative
retrieval frequency, so that often-recalled blocks stay in host memory across
short idle periods, while the rest are demoted to the next tier.

The pages give no formula.  The reading taken here is LRFU (D. Lee et al.,
"LRFU: A Spectrum of Policies that Subsumes the Least Recently Used and Least
Frequently Used Policies", IEEE Transactions on Computers 50(12), 2001): each
block's combined recency and frequency value at step t is

    CRF_t(b) = sum over the steps t_i at which b was referenced of 2^(-lam * (t - t_i)),

with lam in [0, 1] (lam = 0: reference counts, LFU; lam = 1: the last reference
dominates, LRU).  A step first creates its new blocks (their K / V land in host
memory by stage-out: resident, one reference each), then references every
selected block: a selected block that is not resident is a host miss (a read
from the lower tier) and becomes resident.  Then, while more than `capacity`
blocks are host-resident, the resident block with the smallest CRF_t that was
not selected in this step is demoted (ties: the lower block id first).

Written as the definition: the CRF is recomputed from the full reference
history, with no incremental update.
"""
from __future__ import annotations


class HostTier:
    def __init__(self, capacity: int, lam: float):
        self.capacity = int(capacity)
        self.lam = float(lam)
        self.t = 0
        self.refs: dict[int, list[int]] = {}
        self.resident: set[int] = set()
        self.n_blocks = 0

    def crf(self, b: int, t: int) -> float:
        return sum(2.0 ** (-self.lam * (t - ti)) for ti in self.refs.get(b, []))

    def step(self, ids, n_blocks: int):
        """One step: blocks [previous n_blocks, n_blocks) are created, `ids` are
        retrieved.  Returns (hits, misses, demoted ids in demotion order)."""
        self.t += 1
        t = self.t
        created = list(range(self.n_blocks, n_blocks))
        self.n_blocks = max(self.n_blocks, n_blocks)
        ids = [int(b) for b in ids]
        for b in created:
            self.refs.setdefault(b, []).append(t)
            self.resident.add(b)
        hits = sum(1 for b in ids if b in self.resident)
        misses = len(ids) - hits
        for b in ids:
            self.refs.setdefault(b, []).append(t)
            self.resident.add(b)
        protected = set(ids)
        demoted = []
        while len(self.resident) > self.capacity:
            cands = [b for b in self.resident if b not in protected]
            if not cands:
                break
            victim = min(cands, key=lambda b: (self.crf(b, t), b))
            self.resident.remove(victim)
            demoted.append(victim)
        return hits, misses, demoted
