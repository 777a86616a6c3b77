"""The edge-flux checker every parity test relies on (oracle/check.py), on crafted histograms.

A count may move only across the adjacent edge, and only for pairs within 1e-6 rad of it, so the
net flow across edge K is bounded by the oracle's counts of such pairs just below it (up to
near_below[K] may move up) and just above it (up to near_above[K] may move down). A flow beyond
either bound, a move across two edges, or a different total must fail.
"""
import numpy as np

from oracle import check


def _hist(*counts):
    return np.array(counts, np.uint64)


def _near(nb, **at):
    a = np.zeros(nb + 1, np.uint64)
    for k, v in at.items():
        a[int(k[1:])] = v
    return a


def test_identical_histograms_pass_and_move_nothing():
    o = _hist(5, 7, 9, 11)
    rep = check.edge_flux(o, o, _near(4), _near(4))
    assert rep.ok and rep.moved_pairs == 0 and rep.bins_differing == 0 and not rep.violations


def test_one_pair_up_across_an_edge_needs_a_pair_just_below_it():
    o = _hist(5, 7, 9, 11)
    f = _hist(5, 6, 10, 11)  # one count from bin 1 to bin 2: across edge 2
    assert check.edge_flux(f, o, _near(4, e2=1), _near(4)).ok
    assert not check.edge_flux(f, o, _near(4), _near(4)).ok  # nothing near edge 2
    assert not check.edge_flux(f, o, _near(4), _near(4, e2=1)).ok  # near it, but on the wrong side
    assert not check.edge_flux(f, o, _near(4, e1=1, e3=1), _near(4)).ok  # near other edges only
    rep = check.edge_flux(f, o, _near(4), _near(4))
    assert rep.violations[0][0] == 2 and rep.moved_pairs == 1 and rep.bins_differing == 2


def test_one_pair_down_across_an_edge_needs_a_pair_just_above_it():
    o = _hist(5, 7, 9, 11)
    f = _hist(5, 8, 8, 11)  # one count from bin 2 to bin 1: across edge 2
    assert check.edge_flux(f, o, _near(4), _near(4, e2=1)).ok
    assert not check.edge_flux(f, o, _near(4, e2=1), _near(4)).ok


def test_flows_are_bounded_by_the_counts_near_the_edge():
    o = _hist(10, 10, 10)
    f = _hist(7, 13, 10)  # three counts up across edge 1
    assert check.edge_flux(f, o, _near(3, e1=3), _near(3)).ok
    assert not check.edge_flux(f, o, _near(3, e1=2), _near(3)).ok


def test_a_move_across_two_edges_fails_unless_both_edges_allow_it():
    o = _hist(10, 10, 10, 10)
    f = _hist(9, 10, 11, 10)  # one count from bin 0 to bin 2: across edges 1 and 2
    assert not check.edge_flux(f, o, _near(4, e1=1), _near(4)).ok
    assert not check.edge_flux(f, o, _near(4, e2=1), _near(4)).ok
    # counts alone cannot tell this from two separate one-edge moves, which the rule allows
    assert check.edge_flux(f, o, _near(4, e1=1, e2=1), _near(4)).ok


def test_totals_must_agree():
    o = _hist(5, 7, 9)
    assert not check.edge_flux(_hist(5, 7, 10), o, _near(3, e1=9, e2=9), _near(3, e1=9, e2=9)).ok
    assert not check.edge_flux(_hist(5, 7, 8), o, _near(3, e1=9, e2=9), _near(3, e1=9, e2=9)).ok


def test_last_bin_and_the_edges_beyond_it():
    # the flow into the last bin crosses the last interior edge; edge nb (the top) takes no flow
    o = _hist(4, 4, 4)
    f = _hist(4, 3, 5)
    assert check.edge_flux(f, o, _near(3, e2=1), _near(3)).ok
    assert not check.edge_flux(f, o, _near(3, e3=1), _near(3)).ok
