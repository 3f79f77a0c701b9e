"""Input generators: the DynaSpec position-aware budget.

The per-position shortlist workload draws k_c(t) clusters at draft step t.
The DynaSpec summary (§ Method 3) prints k_c(t) = k_max for t in {0, 1} and
floor(k_max / ((t + 1) * 2)) for t >= 2; the generator also keeps at least
one cluster per step (an empty list would leave the drafter nothing to
propose).  The values below are worked out by hand from that formula.
"""
from speculative_decoding_verification_sampling_gb300 import synth


def test_budget_kmax_8():
    # t = 2: 8 // 6 = 1; t = 3: 8 // 8 = 1; t = 4, 5: 8 // 10 = 8 // 12 = 0 -> floor of 1
    assert synth.dynaspec_budget(8, 6) == [8, 8, 1, 1, 1, 1]


def test_budget_kmax_64():
    # 64 // 6 = 10, 64 // 8 = 8, 64 // 10 = 6, 64 // 12 = 5, 64 // 14 = 4
    assert synth.dynaspec_budget(64, 7) == [64, 64, 10, 8, 6, 5, 4]


def test_budget_short_drafts():
    assert synth.dynaspec_budget(8, 1) == [8]
    assert synth.dynaspec_budget(3, 3) == [3, 3, 1]


def test_per_position_lists_follow_the_budget():
    cfg = synth.shortlist_per_position(B=2, K=4, V=4096, n_clusters=64, seed=3)
    assert cfg["shortlist_len"] == [8 * 64, 8 * 64, 64, 64]
