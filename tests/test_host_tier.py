"""The library's host-tier policy (kvm_tier_*, host-only C++) against the
oracle's LRFU definition (oracle/tier.py) on random step sequences: hits,
misses and the demoted ids in order, step by step, and the resident set.

lam = 0 and lam = 1 make every CRF a sum of powers of two, exact in double on
both sides.  For other lam the library keeps CRF incrementally and the oracle
recomputes the sum, so a choice between two blocks whose values differ by a
rounding may legitimately go either way; there the test checks that a first
disagreement is such a near-tie and ends the sequence."""
import numpy as np
import pytest

import oracle.tier as tier


@pytest.fixture(scope="module")
def kvm():
    import paged_kv_cache_meank_gb300 as kvm
    from paged_kv_cache_meank_gb300 import build
    build.build()
    return kvm


def _sequence(rng, steps, start, grow, per_step):
    n, seq = start, []
    for _ in range(steps):
        n += int(rng.integers(0, grow + 1))
        k = min(n, int(rng.integers(1, per_step + 1)))
        # skewed reuse: low ids recalled more often
        p = 1.0 / (1.0 + np.arange(n)) ** 0.7
        ids = sorted(rng.choice(n, size=k, replace=False, p=p / p.sum()).tolist())
        seq.append((ids, n))
    return seq


@pytest.mark.parametrize("lam", [0.0, 1.0, 0.3, 0.05])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tier_matches_the_oracle(kvm, lam, seed):
    rng = np.random.default_rng(100 + seed)
    cap = int(rng.integers(20, 60))
    seq = _sequence(rng, 80, 30, 4, 12)
    lib = kvm.HostTier(cap, lam)
    ref = tier.HostTier(cap, lam)
    for step, (ids, n) in enumerate(seq):
        got = lib.step(ids, n)
        want = ref.step(ids, n)
        if got != want:
            assert lam not in (0.0, 1.0), (step, got, want)
            # only a near-tie may differ: the first differing victims' CRFs agree
            g, w = got[2], want[2]
            i = next(k for k in range(min(len(g), len(w))) if g[k] != w[k])
            a, b = ref.crf(g[i], ref.t), ref.crf(w[i], ref.t)
            assert abs(a - b) <= 1e-12 * max(a, b), (step, a, b)
            return
        res = lib.resident(n)
        assert set(np.flatnonzero(res).tolist()) == ref.resident, step


def test_tier_rejects_bad_input(kvm):
    with pytest.raises(kvm.KvmError):
        kvm.HostTier(0, 0.5)
    with pytest.raises(kvm.KvmError):
        kvm.HostTier(10, 1.5)
    t = kvm.HostTier(10, 0.5)
    t.step([0, 1], 5)
    for ids, n in (([1, 1], 5), ([7], 5), ([0], 3)):    # repeated, out of range, shrinking
        with pytest.raises(kvm.KvmError):
            t.step(ids, n)
    assert t.step([2], 5)[0] == 1                          # state unchanged by the errors
