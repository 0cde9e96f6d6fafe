"""Pins of the layerwise prefill oracle (readings R14-R16 of oracle/layerwise.py;
"Layerwise and Sparse KV Cache Offloading Design", section 3, and the FlashOffloading
explainer's prefill paragraph)."""
import numpy as np
import pytest

from oracle import layerwise as LW


def test_pages_four_trays_for_78_layers():
    # the explainer: four trays hold about 4/78, or 5.1%, of a fully resident design
    n_phys, phys = LW.plan(78, independent=(0,), n_shared=3)
    assert n_phys == 4
    assert round(100 * LW.footprint_ratio(78, n_phys), 1) == 5.1
    assert phys[0] == 0  # tray B0 stays bound to the first layer
    assert sorted(set(phys[1:])) == [1, 2, 3]  # B1..B3 rotate


def test_hand_derived_round_robin():
    # six layers, layer 0 independent, two shared buffers: layers 1..5 -> 1, 2, 1, 2, 1
    assert LW.plan(6, (0,), 2) == (3, [0, 1, 2, 1, 2, 1])
    # independent layers 0 and 3, three shared: reusable 1, 2, 4, 5 -> 2, 3, 4, 2
    assert LW.plan(6, (0, 3), 3) == (5, [0, 2, 3, 1, 4, 2])


def test_more_shared_buffers_than_reusable_layers():
    # physical = I + min(B, R): B beyond R adds nothing
    assert LW.plan(3, (0,), 5) == (3, [0, 1, 2])
    assert LW.plan(1, (0,), 4) == (1, [0])
    assert LW.plan(4, (), 4) == (4, [0, 1, 2, 3])


def test_no_independent_layers_and_bad_plans():
    assert LW.plan(5, (), 2) == (2, [0, 1, 0, 1, 0])
    with pytest.raises(ValueError):
        LW.plan(4, (0,), 0)  # reusable layers without a shared buffer
    with pytest.raises(ValueError):
        LW.plan(4, (7,), 2)


@pytest.mark.parametrize("n,ind,b", [(78, (0,), 3), (61, (0, 60), 4), (10, (), 3), (24, (0, 1), 2)])
def test_plan_invariants(n, ind, b):
    n_phys, phys = LW.plan(n, ind, b)
    assert all(0 <= x < n_phys for x in phys)
    ded = [phys[l] for l in ind]
    assert len(set(ded)) == len(ded)  # a dedicated buffer each
    reusable = [l for l in range(n) if l not in ind]
    assert not set(ded) & {phys[l] for l in reusable}  # never shared with a reusable layer
    if min(b, len(reusable)) >= 2:  # consecutive reusable layers alternate buffers
        assert all(phys[x] != phys[y] for x, y in zip(reusable, reusable[1:]))
    # every shared buffer serves layers evenly (round robin)
    counts = np.bincount([phys[l] for l in reusable], minlength=n_phys)[len(ind):]
    if len(reusable):
        assert counts.max() - counts.min() <= 1


def test_digest_and_passes_hand_derived():
    o = LW.LayerwiseOracle(2, 4, row_elems=2)
    o.fill_prefix(np.array([[[1, 2]], [[3, 0xFFFF]]], dtype=np.uint16))  # L = 1
    d = o.forward(np.array([[[5, 6], [7, 8]], [[9, 10], [11, 12]]], dtype=np.uint16))
    assert d == [3, 3 + 65535]  # unsigned bit patterns
    assert o.length == 3
    d = o.forward(np.array([[[1, 1]], [[0, 0]]], dtype=np.uint16))
    assert d == [1 + 2 + 5 + 6 + 7 + 8, 3 + 65535 + 9 + 10 + 11 + 12]
    assert o.host[0, :4].tolist() == [[1, 2], [5, 6], [7, 8], [1, 1]]
    with pytest.raises(ValueError):
        o.forward(np.zeros((2, 1, 2), np.uint16))  # past max_tokens


def test_empty_prefix_pass():
    o = LW.LayerwiseOracle(3, 8, row_elems=4)
    d = o.forward(np.ones((3, 2, 4), np.uint16))
    assert d == [0, 0, 0] and o.length == 2
