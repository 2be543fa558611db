"""The oracle-filtered episode generator used by the GPU parity cases (tests/helpers.py:
oracle_checked_dag) produces the mount kinds the episode presets never make: spans of an
ancestor's tokens past the fork point and further disjoint spans of a producer the lineage
already mounted (both legal: they show no token twice)."""
from helpers import mount_kinds, oracle_checked_dag


def _checked_dag(oracle_mod, seed, **kw):
    ep = oracle_checked_dag(oracle_mod, seed, **kw)
    return ep, mount_kinds(ep)


def test_checked_dags_hold_ancestor_and_repeated_mounts(oracle_mod):
    """Seeds 600-611 (those of the GPU parity cases on these episodes) hold spans of an
    ancestor's tokens past the fork point and second spans of an already mounted producer."""
    anc = rep = 0
    for seed in range(600, 612):
        _, (a, r) = _checked_dag(oracle_mod, seed, page_size=16, max_segments=12, max_len=80)
        anc, rep = anc + a, rep + r
    assert anc >= 4 and rep >= 4, (anc, rep)


