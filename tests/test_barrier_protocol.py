"""The decode kernels' mbarrier hand-offs on random-schedule models
(tests/barrier_model.py for one CTA, tests/barrier_model_pair.py for the
cluster kernel's CTA pair, tests/barrier_model_mc.py for the 65..128-row
pair of 64-row CTAs that share tiles through multicast copies), with the
shapes the kernels use.

Every shape must finish every schedule with no problem. The schedules include
ones where a PV issuer, a producer or one CTA's softmax runs far behind the
other roles. Controls show that the models catch each kind of fault:
- one hand-off barrier for two P buffers, which the kernels used to have: a
  PV issuer two phases behind waits forever;
- an odd pair ring fed by per-pair producers, which the kernels also used to
  have: a slot is reloaded before its PV has freed it;
- the cluster kernel without the wait that protects its score staging: P
  overwrites the staged scores before the bulk copy has read them;
- a multicast pair whose slots are released by one CTA's products only: a
  copy lands in the peer's slot while the peer still reads it."""
import pytest

from barrier_model import run
from barrier_model_mc import run_mc
from barrier_model_pair import run_pair

SKEWS = [None, {"PV0": 0.02}, {"PV1": 0.02}, {"PV0": 0.01, "LD1": 0.2}, {"PV1": 0.01, "LD0": 0.2},
         {"PV0": 0.005, "S": 3.0, "LD0": 3.0}]

# (name, blocks per tile, ring slots, rope slots, producers, P buffers, rope read first (the
#  folded kernel's order: S reads the rope first and frees it early, the producers load it
#  first), fp8 rows widened in place by one expander per block)
SHAPES = [
    ("folded 16 rows", 4, 11, 2, 2, 2, True, False),
    ("folded 32 rows", 4, 10, 1, 2, 2, True, False),
    ("folded 64 rows (two score buffers)", 4, 8, 1, 2, 1, True, False),
    ("folded latent 256, 16 rows", 2, 11, 2, 2, 2, True, False),
    ("folded latent 256, 32 rows", 2, 10, 2, 2, 2, True, False),
    ("folded latent 768, 16 rows", 6, 11, 1, 2, 2, True, False),
    ("folded latent 1792 (one CTA of a pair), 16 rows", 7, 9, 2, 2, 2, True, False),
    ("folded fp8 64 rows (two score buffers)", 4, 8, 1, 1, 1, True, True),
    ("folded fp8 16 rows", 4, 11, 2, 1, 2, True, True),
    ("folded fp8 32 rows", 4, 10, 1, 1, 2, True, True),
    ("folded 64 rows, rope read last", 4, 8, 1, 2, 1, False, False),
    ("folded fp8 64 rows, rope read last", 4, 8, 1, 1, 1, False, True),
    ("cluster TMA 16 rows", 2, 5, 3, 1, 2, False, False),
    ("cluster TMA 32 rows", 2, 5, 2, 1, 2, False, False),
    ("cluster load/convert 16 rows", 2, 4, 3, 2, 2, False, False),
    ("cluster load/convert 32 rows", 2, 4, 2, 2, 2, False, False),
    ("cluster load/convert 64 rows", 2, 4, 1, 2, 1, False, False),
    ("cluster fp8 64 rows", 2, 4, 1, 1, 1, False, False),
]


def failures(seeds, **shape):
    out = []
    for w in SKEWS:
        for seed in range(seeds):
            e = run(seed, weights=w, **shape)
            if e:
                out.append((w, seed, e[0]))
    return out


# the transposed 64-row kernels: eleven K-block slots, two rope slots, one score buffer
# (and twelve with one rope slot, measured slower: the rope reload then waits for the
# previous tile's score product)
SHAPES_ONE_S = [
    ("folded 64 rows, transposed scores", 4, 11, 2, 2, 1, True, False),
    ("folded fp8 64 rows, transposed scores", 4, 11, 2, 1, 1, True, True),
    ("folded 64 rows, transposed scores, one rope slot", 4, 12, 1, 2, 1, True, False),
]


@pytest.mark.parametrize("name,KB,R,RR,producers,PB,rope_first,expand", SHAPES_ONE_S, ids=[s[0] for s in SHAPES_ONE_S])
def test_one_score_buffer_shapes_survive_skew(name, KB, R, RR, producers, PB, rope_first, expand):
    bad = failures(40, KB=KB, R=R, RR=RR, producers=producers, PB=PB, H=2, rope_first=rope_first, expand=expand, SB=1)
    assert not bad, bad[:3]


@pytest.mark.parametrize("name,KB,R,RR,producers,PB,rope_first,expand", SHAPES, ids=[s[0] for s in SHAPES])
def test_kernel_shapes_survive_skew(name, KB, R, RR, producers, PB, rope_first, expand):
    bad = failures(40, KB=KB, R=R, RR=RR, producers=producers, PB=PB, H=2, rope_first=rope_first, expand=expand)
    assert not bad, bad[:3]


def test_seven_slots_at_64_rows_would_be_sound_but_serial():
    """Seven K-block slots at 64 rows pass the model too; the kernel takes
    eight for speed (with seven, a tile's last block reuses the previous
    tile's first slot, so loads wait for the previous tile's value product)."""
    assert not failures(20, KB=4, R=7, RR=1, producers=2, PB=1, H=2)


def test_too_small_a_ring_reloads_early():
    """Control: six K-block slots with two rope slots at 64 rows lose a slot."""
    bad = failures(40, KB=4, R=6, RR=2, producers=2, PB=1, H=2)
    assert any("unfreed" in e for _, _, e in bad)


def test_one_handoff_barrier_deadlocks():
    bad = failures(40, KB=4, R=11, RR=2, producers=2, PB=2, H=1)
    assert any("deadlock" in e for _, _, e in bad)
    # with a single P buffer the softmax waits for PV(i - 1) before handing
    # over tile i, so one barrier is enough
    assert not failures(20, KB=2, R=4, RR=1, producers=1, PB=1, H=1)


def test_odd_ring_with_per_pair_producers_reloads_early():
    bad = failures(40, KB=2, R=5, RR=3, producers=2, PB=2, H=2)
    assert any("unfreed" in e for _, _, e in bad)


PAIR_SKEWS = [None, {"PV0_0": 0.02}, {"PV1_1": 0.02}, {"SM0": 0.05}, {"SM1": 0.05, "PV0_0": 0.1}, {"LD0": 0.05},
              {"S1": 0.05}, {"EX0": 0.05}]

# (name, pair slots, rope slots, P buffers, split softmax columns, score staging in the P buffer,
#  fp8 pool: TMA-landed codes widened in place by the expand warps)
PAIR_SHAPES = [
    ("16 rows", 5, 3, 2, False, False, False),
    ("32 rows", 5, 2, 2, True, True, False),
    ("64 rows", 4, 1, 1, True, False, False),
    ("16 rows, load/convert warps", 4, 3, 2, False, False, False),
    ("32 rows, load/convert warps", 4, 2, 2, True, True, False),
    ("16 rows, fp8", 5, 3, 2, False, False, True),
    ("32 rows, fp8", 5, 2, 2, True, True, True),
    ("64 rows, fp8", 4, 1, 1, True, False, True),
]


def pair_failures(seeds, **shape):
    out = []
    for w in PAIR_SKEWS:
        for seed in range(seeds):
            e = run_pair(seed, weights=w, **shape)
            if e:
                out.append((w, seed, e[0]))
    return out


@pytest.mark.parametrize("name,R,RR,PB,split,send_in_p,fp8", PAIR_SHAPES, ids=[s[0] for s in PAIR_SHAPES])
def test_cluster_exchanges_survive_skew(name, R, RR, PB, split, send_in_p, fp8):
    bad = pair_failures(20, R=R, RR=RR, PB=PB, split=split, send_in_p=send_in_p, fp8=fp8)
    assert not bad, bad[:3]


def test_score_staging_needs_the_peer_to_have_read_it():
    """At 32 rows the partial scores are staged in the tile's P buffer; writing
    P before the peer has consumed them (its xfree arrive) lets P overwrite the
    staging before the bulk copy has read it."""
    bad = pair_failures(20, R=5, RR=2, PB=2, split=True, send_in_p=True, skip_xfree_before_p=True)
    assert any("source changed" in e for _, _, e in bad)


MC_SKEWS = [None, {"PV00": 0.02}, {"PV11": 0.02}, {"SM1": 0.05}, {"S0": 0.02, "LD11": 3.0},
            {"LD00": 0.05, "PV10": 0.1}, {"PV01": 0.01, "LD10": 0.2}]


def mc_failures(seeds, **shape):
    out = []
    for w in MC_SKEWS:
        for seed in range(seeds):
            e = run_mc(seed, weights=w, **shape)
            if e:
                out.append((w, seed, e[0]))
    return out


def test_multicast_pair_at_128_rows_survives_skew():
    """The 65..128-row pair: eleven K-block slots and two rope slots per CTA
    (the 64-row transposed kernel's ring), each CTA copying its half of every
    block and its rope half into both CTAs, both CTAs' products releasing
    each slot."""
    bad = mc_failures(30, KB=4, R=11, RR=2)
    assert not bad, bad[:3]


def test_multicast_slot_released_by_one_cta_reloads_early():
    bad = mc_failures(20, KB=4, R=11, RR=2, empty_count=1)
    assert any("still in use" in e for _, _, e in bad)


def test_multicast_rope_released_by_one_cta_reloads_early():
    bad = mc_failures(20, KB=4, R=11, RR=2, rope_count=1)
    assert any("unconsumed rope slot" in e for _, _, e in bad)
