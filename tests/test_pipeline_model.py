"""The attention kernel's barrier protocol, run as a random-schedule model on the CPU.

The model is in tests/_pipeline_model.py.  It covers both ring forms:

- split K and V rings for three slots or fewer;
- one combined ring otherwise.

It covers 64- and 128-key tiles, ragged and tiny S, repeated units on one CTA, and units whose two
query tiles cover the same rows (two heads of one KV group, equal tile counts).  A planted
mistake in the K/V release rule must be caught.
"""
import random

import pytest

from _pipeline_model import simulate

SEQ = [1, 63, 64, 65, 128, 129, 255, 256, 257, 385, 700]


def _cases():
    for S in SEQ:
        for BN in (64, 128):
            for stages in (2, 3, 4, 5, 8):
                for seed in range(3):
                    rnd = random.Random(seed * 7919 + S * 31 + BN + stages)
                    r0s = list(range(0, S, 256))
                    units = [rnd.choice(r0s) for _ in range(rnd.randint(1, 4))]
                    yield S, BN, stages, units, seed
                    # head-pair units: both query tiles on the same 128 rows (equal tile counts)
                    rows = list(range(0, S, 128))
                    pairs = [(r, r) for r in (rnd.choice(rows) for _ in range(rnd.randint(1, 4)))]
                    yield S, BN, stages, pairs, seed


def test_every_schedule_is_clean():
    bad = []
    for S, BN, stages, units, seed in _cases():
        errs = simulate(S, BN, stages, units, seed)
        if errs:
            bad.append((S, BN, stages, units, seed, errs[:2]))
    assert not bad, bad[:5]


def test_a_steady_block_that_never_releases_q1_is_caught():
    # with head-pair units query tile 1 ends inside the steady-state block, which must then release
    # its Q buffer (the next unit's Q1 load waits for that release)
    caught = sum(bool(simulate(S, BN, stages, units, seed, steady_without_q1_release=True))
                 for S, BN, stages, units, seed in _cases() if isinstance(units[0], tuple))
    assert caught > 0


def test_a_wrong_release_rule_is_caught():
    caught = sum(bool(simulate(S, BN, stages, units, seed, wrong_release=True))
                 for S, BN, stages, units, seed in _cases())
    assert caught > 0


@pytest.mark.parametrize("stages", [2, 3, 4, 5])
def test_long_units_on_one_cta(stages):
    # several full-length units back to back (the deferred last PVs cross every boundary)
    assert simulate(2048, 128, stages, [1792, 1536, 0, 1024], seed=stages) == []


@pytest.mark.parametrize("stages", [2, 3, 4, 5])
def test_long_head_pair_units_on_one_cta(stages):
    # head-pair units end both query tiles on the same K/V tile; mixed with row-pair units
    assert simulate(2048, 128, stages, [(1920, 1920), (1792, 1792), (0, 0), 1024, (640, 640)], seed=stages) == []
