"""Seeded workload recipes: shapes, distributions and the EPLB map invariants."""
import numpy as np
import pytest

from combine_dp_gather_gb300 import synth
from conftest import ints, read_golden


@pytest.mark.parametrize("row", read_golden("trivial_map.txt"))
def test_trivial_map_golden(row):
    E, P, p2l = int(row[0]), int(row[1]), ints(row[2])
    l2p, nrep, got = synth.trivial_map(E, P)
    assert got.tolist() == p2l
    for e in range(E):
        assert sorted(l2p[e, : nrep[e]].tolist()) == [s for s in range(P) if p2l[s] == e]


def test_eplb_map_invariants():
    spec = synth.spec_eplb()
    counts = synth.eplb_expected_counts(spec)
    assert counts.sum() == spec.T * spec.k
    l2p, nrep, p2l = synth.eplb_map(counts, 32, 16)
    assert len(p2l) == 288 and int(nrep.sum()) == 288 and (nrep >= 1).all()
    hottest = sorted(range(256), key=lambda e: (-counts[e], e))[:32]
    assert sorted(np.nonzero(nrep == 2)[0].tolist()) == sorted(hottest)
    per_range = p2l.reshape(16, 18)
    for e in np.nonzero(nrep == 2)[0]:
        ranges = [s // 18 for s in l2p[e, :2]]
        assert ranges[0] != ranges[1]          # replicas on different simulated ranks
    for e in range(256):
        for x in range(nrep[e]):
            assert p2l[l2p[e, x]] == e
    # packing is balanced far better than the unreplicated trivial layout
    load = np.array([sum(counts[e] / nrep[e] for e in row) for row in per_range])
    triv = np.array([counts[r * 16:(r + 1) * 16].sum() for r in range(16)])
    assert load.max() / load.mean() < triv.max() / triv.mean()


def test_decode_counts_have_idle_replica():
    for seed in range(20):
        c = synth.decode_counts(seed)
        assert len(c) == 8 and min(c) == 0 and max(c) <= 64


def test_sweep_requests_from_allowed_set():
    for mix in synth.SWEEP_MIXES:
        r = synth.sweep_requests(mix)
        assert len(r) == 16 and set(r) <= {0, 4, 8, 24}


def test_zipf_bias_ranks():
    b = synth.zipf_bias(256, 1.1, 0)
    rank = synth.popularity_rank(256, 0)
    hot = int(np.argmin(rank))
    assert b[hot] == 0.0 and np.all(b <= 0)
    # probability ratio between rank 0 and rank 9 is 10**s
    e9 = int(np.nonzero(rank == 9)[0][0])
    assert np.isclose(np.exp(b[hot] - b[e9]), 10 ** 1.1, rtol=1e-6)


def test_generators_reproducible_and_shaped():
    spec = synth.spec_tiny()
    a = synth.hidden_states(spec)
    b = synth.hidden_states(spec)
    assert [t.shape[0] for t in a] == spec.counts
    assert all((x == y).all() for x, y in zip(a, b))
    wgu, wd = synth.expert_weights(spec)
    assert tuple(wgu.shape) == (8, 256, 256) and tuple(wd.shape) == (8, 256, 128)
    assert abs(float(wgu.std()) - 0.02) < 1e-3
