"""The decode kernels' mbarrier hand-offs on a random-schedule model
(tests/barrier_model.py), with the ring shapes the kernels use.

Every shape must finish every schedule with no problem. The schedules include
ones where a PV issuer or a producer runs far behind the other roles. Two
shapes the kernels used to have serve as controls, so the model is shown able
to catch each kind of fault:
- one hand-off barrier for two P buffers: a PV issuer two phases behind waits
  forever;
- an odd pair ring fed by per-pair producers: a slot is reloaded before its
  PV has freed it."""
import pytest

from barrier_model import run

SKEWS = [None, {"PV0": 0.02}, {"PV1": 0.02}, {"PV0": 0.01, "LD1": 0.2}, {"PV1": 0.01, "LD0": 0.2},
         {"PV0": 0.005, "S": 3.0, "LD0": 3.0}]

# (name, blocks per tile, ring slots, rope slots, producers, P buffers)
SHAPES = [
    ("folded 16 rows", 4, 11, 2, 2, 2),
    ("folded 32 rows", 4, 10, 1, 2, 2),
    ("cluster TMA 16 rows", 2, 5, 3, 1, 2),
    ("cluster TMA 32 rows", 2, 5, 2, 1, 2),
    ("cluster TMA 64 rows", 2, 4, 1, 1, 1),
    ("cluster load/convert 16 rows", 2, 4, 3, 2, 2),
    ("cluster load/convert 32 rows", 2, 4, 2, 2, 2),
    ("cluster load/convert 64 rows", 2, 4, 1, 2, 1),
]


def failures(seeds, **shape):
    out = []
    for w in SKEWS:
        for seed in range(seeds):
            e = run(seed, weights=w, **shape)
            if e:
                out.append((w, seed, e[0]))
    return out


@pytest.mark.parametrize("name,KB,R,RR,producers,PB", SHAPES, ids=[s[0] for s in SHAPES])
def test_kernel_shapes_survive_skew(name, KB, R, RR, producers, PB):
    bad = failures(40, KB=KB, R=R, RR=RR, producers=producers, PB=PB, H=2)
    assert not bad, bad[:3]


def test_one_handoff_barrier_deadlocks():
    bad = failures(40, KB=4, R=11, RR=2, producers=2, PB=2, H=1)
    assert any("deadlock" in e for _, _, e in bad)
    # with a single P buffer the softmax waits for PV(i - 1) before handing
    # over tile i, so one barrier is enough
    assert not failures(20, KB=2, R=4, RR=1, producers=1, PB=1, H=1)


def test_odd_ring_with_per_pair_producers_reloads_early():
    bad = failures(40, KB=2, R=5, RR=3, producers=2, PB=2, H=2)
    assert any("unfreed" in e for _, _, e in bad)
