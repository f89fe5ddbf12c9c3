"""Pins of the host-tier policy oracle (oracle/tier.py) against policies it must
reduce to, plus planted mistakes that the pins catch.

- lam = 0: every reference weighs 1, so the policy is LFU (reference counts,
  ties to the lower id), checked against a plain counting simulation.
- lam = 1: with one reference per step after a step that only creates the
  blocks, the last reference dominates, so the policy is LRU, checked against a
  plain last-use simulation.
- The property the pages give: an often-recalled block survives a short idle
  period under a frequency-weighted lam, where LRU demotes it.
- Invariants: hits + misses = references, referenced blocks end resident, the
  resident count stays at the capacity.
"""
import numpy as np
import pytest

import oracle.tier as tier


def _lfu_brute(capacity, seq, n_per_step):
    count, resident, out = {}, set(), []
    prev_n = 0
    for ids, n_blocks in zip(seq, n_per_step):
        created = range(prev_n, n_blocks)
        prev_n = n_blocks
        for b in created:
            count[b] = count.get(b, 0) + 1
            resident.add(b)
        hits = sum(1 for b in ids if b in resident)
        for b in ids:
            count[b] = count.get(b, 0) + 1
            resident.add(b)
        dem = []
        while len(resident) > capacity:
            victim = min((b for b in resident if b not in set(ids)), key=lambda b: (count[b], b))
            resident.remove(victim)
            dem.append(victim)
        out.append((hits, len(ids) - hits, dem))
    return out


def _lru_brute(capacity, seq, n_per_step):
    last, resident, out = {}, set(), []
    prev_n = 0
    for t, (ids, n_blocks) in enumerate(zip(seq, n_per_step), start=1):
        created = range(prev_n, n_blocks)
        prev_n = n_blocks
        for b in set(created) | set(ids):
            last[b] = t
        resident |= set(created)
        hits = sum(1 for b in ids if b in resident)
        resident |= set(ids)
        dem = []
        while len(resident) > capacity:
            victim = min((b for b in resident if b not in set(ids)), key=lambda b: (last[b], b))
            resident.remove(victim)
            dem.append(victim)
        out.append((hits, len(ids) - hits, dem))
    return out


def pin_lfu(mod):
    """The history grows by two blocks a step, so creation counts as a reference."""
    rng = np.random.default_rng(20)
    for trial in range(20):
        C = int(rng.integers(8, 20))
        ns = [10 + 2 * k for k in range(25)]
        seq = [sorted(rng.choice(n, size=int(rng.integers(1, 6)), replace=False).tolist())
               for n in ns]
        t = mod.HostTier(C, 0.0)
        got = [t.step(ids, n) for ids, n in zip(seq, ns)]
        assert got == _lfu_brute(C, seq, ns), trial


def pin_lru(mod):
    """One event per step -- a step creates one block or selects one block --
    so every block's last event has its own step."""
    rng = np.random.default_rng(21)
    for trial in range(20):
        C = int(rng.integers(5, 15))
        seq, ns, n = [[]], [10], 10
        for k in range(60):
            if k % 2:
                n += 1
                seq.append([])
            else:
                seq.append([int(rng.integers(0, n))])
            ns.append(n)
        t = mod.HostTier(C, 1.0)
        got = [t.step(ids, nb) for ids, nb in zip(seq, ns)]
        assert got == _lru_brute(C, seq, ns), trial


def pin_frequency_protection(mod):
    """Block 0 is recalled in 10 steps, then idles for 3 steps while 3 other
    blocks are recalled once each; capacity 3 with 4 live blocks forces one
    demotion per idle step.  LRU (lam = 1) demotes block 0; a frequency-weighted
    lam keeps it."""
    def run(lam):
        t = mod.HostTier(3, lam)
        t.step([], 1)                       # block 0 created
        for _ in range(9):
            t.step([0], 1)
        t.step([], 4)                       # blocks 1..3 created
        for b in (1, 2, 3):
            t.step([b], 4)
        return 0 in t.resident
    assert run(0.1) and not run(1.0)


def pin_invariants(mod):
    rng = np.random.default_rng(22)
    t = mod.HostTier(12, 0.3)
    N = 5
    for step in range(60):
        N += int(rng.integers(0, 3))
        ids = sorted(rng.choice(N, size=min(N, int(rng.integers(1, 8))), replace=False).tolist())
        before = set(t.resident) | set(range(t.n_blocks, N))   # new blocks arrive resident
        h, m, d = t.step(ids, N)
        assert h + m == len(ids) and h == len(before & set(ids))
        assert set(ids) <= t.resident and len(t.resident) == min(12, len(t.resident))
        assert not (set(d) & set(ids))


PINS = [pin_lfu, pin_lru, pin_frequency_protection, pin_invariants]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_tier_pin(pin):
    pin(tier)


class _NoDecay(tier.HostTier):
    def crf(self, b, t):
        return float(len(self.refs.get(b, [])))


class _EvictLargest(tier.HostTier):
    def crf(self, b, t):
        return -super().crf(b, t)


class _HigherIdFirst(tier.HostTier):
    def step(self, ids, n_blocks):
        self.t += 1
        t = self.t
        created = list(range(self.n_blocks, n_blocks))
        self.n_blocks = max(self.n_blocks, n_blocks)
        ids = [int(b) for b in ids]
        for b in created:
            self.refs.setdefault(b, []).append(t)
            self.resident.add(b)
        hits = sum(1 for b in ids if b in self.resident)
        for b in ids:
            self.refs.setdefault(b, []).append(t)
            self.resident.add(b)
        dem = []
        while len(self.resident) > self.capacity:
            victim = min((b for b in self.resident if b not in set(ids)),
                         key=lambda b: (self.crf(b, t), -b))
            self.resident.remove(victim)
            dem.append(victim)
        return hits, len(ids) - hits, dem


class _CreationNotAReference(tier.HostTier):
    def step(self, ids, n_blocks):
        self.t += 1
        t = self.t
        created = list(range(self.n_blocks, n_blocks))
        self.n_blocks = max(self.n_blocks, n_blocks)
        ids = [int(b) for b in ids]
        for b in created:
            self.resident.add(b)
        hits = sum(1 for b in ids if b in self.resident)
        for b in ids:
            self.refs.setdefault(b, []).append(t)
            self.resident.add(b)
        dem = []
        while len(self.resident) > self.capacity:
            victim = min((b for b in self.resident if b not in set(ids)),
                         key=lambda b: (self.crf(b, t), b))
            self.resident.remove(victim)
            dem.append(victim)
        return hits, len(ids) - hits, dem


@pytest.mark.parametrize("mutant", [_NoDecay, _EvictLargest, _HigherIdFirst,
                                    _CreationNotAReference], ids=lambda m: m.__name__)
def test_tier_mutant_is_caught(mutant):
    class Mod:
        HostTier = mutant
    failed = 0
    for pin in PINS:
        try:
            pin(Mod)
        except AssertionError:
            failed += 1
    assert failed, mutant.__name__
