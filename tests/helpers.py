"""Test helpers that are independent of both the oracle and the CUDA path.

Exact integer-valued inputs (so that every fp32 partial sum is exact and the
score is the plain integer dot product), an explicit-list LRU model, and the
state invariants of the residency table.
"""
import numpy as np


def int_bf16(values):
    """bf16 bit patterns of small integers (exact)."""
    v = np.asarray(values, dtype=np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16)


def rand_int_bf16(rng, shape, lo=-3, hi=3):
    ints = rng.integers(lo, hi + 1, size=shape)
    return ints.astype(np.int64), int_bf16(ints)


def exact_topk(int_scores, visible, k):
    """Plain full sort by (score desc, token asc); returns (tokens, scores) padded with -1/-inf."""
    order = sorted(range(visible), key=lambda t: (-int(int_scores[t]), t))[:k]
    toks = order + [-1] * (k - len(order))
    scs = [float(int_scores[t]) for t in order] + [-np.inf] * (k - len(order))
    return toks, scs


class ListLRU:
    """Residency shelf kept as an explicit recency list (least recent first).

    Initially every slot is free and the list is 0..C-1.  On each step the
    slots used by the step (hits and filled misses) are moved to the most
    recent end, in slot order; victims are taken from the least recent end,
    skipping slots that hold a token of this step.  Misses are filled in
    token order.
    """

    def __init__(self, capacity):
        self.C = capacity
        self.order = list(range(capacity))
        self.slot_tok = [-1] * capacity
        self.tok_slot = {}

    def step(self, wanted):
        wanted = set(wanted)
        if len(wanted) > self.C:
            return None
        hits = {t for t in wanted if t in self.tok_slot}
        misses = sorted(wanted - hits)
        hit_slots = {self.tok_slot[t] for t in hits}
        victims = [s for s in self.order if s not in hit_slots][: len(misses)]
        for t, s in zip(misses, victims):
            old = self.slot_tok[s]
            if old >= 0:
                del self.tok_slot[old]
            self.slot_tok[s] = t
            self.tok_slot[t] = s
        touched = sorted(hit_slots | set(victims))
        touched_set = set(touched)
        self.order = [s for s in self.order if s not in touched_set] + touched
        return list(zip(misses, victims))


def check_residency_invariants(cache_slots, slot_token, last_use, stamp, length):
    """Mutual inverse, occupancy counts, stamps bounded.  Raises AssertionError."""
    cache_slots = np.asarray(cache_slots)
    slot_token = np.asarray(slot_token)
    C = slot_token.shape[0]
    occ = np.nonzero(slot_token >= 0)[0]
    res = np.nonzero(cache_slots >= 0)[0]
    assert len(occ) == len(res), "occupied slots != resident tokens"
    assert np.all(cache_slots[slot_token[occ]] == occ), "slot_token -> cache_slots not inverse"
    assert np.all(slot_token[cache_slots[res]] == res), "cache_slots -> slot_token not inverse"
    assert np.all(res < length), "resident token beyond length"
    assert np.all(cache_slots[res] < C)
    assert np.all(np.asarray(last_use, dtype=np.int64) <= stamp), "last_use beyond stamp"
