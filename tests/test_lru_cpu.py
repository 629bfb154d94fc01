"""CPU checks of the recency index behind the pool's eviction under pressure
(slora_lru_*): least recently used first, held (pinned) adapters never chosen, and a
randomized comparison with a plain Python list model of the same policy.  No GPU."""
import shutil

import numpy as np
import pytest

import rank_delta_paged_gb300 as rdp
from rank_delta_paged_gb300 import build as B

pytestmark = pytest.mark.skipif(shutil.which(B.NVCC) is None, reason="nvcc not available")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    rdp.lib()


@pytest.fixture
def lru():
    h = rdp.slora_lru_create()
    yield h
    rdp.slora_lru_destroy(h)


def test_order_of_insertion_then_touch(lru):
    for a in range(5):
        rdp.slora_lru_insert(lru, a)
    assert rdp.slora_lru_victims(lru) == [0, 1, 2, 3, 4]
    rdp.slora_lru_touch(lru, 1)
    rdp.slora_lru_touch(lru, 0)
    assert rdp.slora_lru_victims(lru) == [2, 3, 4, 1, 0]
    rdp.slora_lru_insert(lru, 3)            # already present: no change of recency
    assert rdp.slora_lru_victims(lru) == [2, 3, 4, 1, 0]
    assert rdp.slora_lru_victims(lru, max_out=2) == [2, 3]
    assert rdp.slora_lru_victims(lru, exclude=[3, 4]) == [2, 1, 0]


def test_pinned_ids_are_never_victims_and_keep_their_recency(lru):
    for a in range(4):
        rdp.slora_lru_insert(lru, a)
    rdp.slora_lru_pin(lru, 1)
    rdp.slora_lru_pin(lru, 1)                # two holds
    assert rdp.slora_lru_victims(lru) == [0, 2, 3]
    rdp.slora_lru_unpin(lru, 1)
    assert rdp.slora_lru_victims(lru) == [0, 2, 3]
    rdp.slora_lru_unpin(lru, 1)
    assert rdp.slora_lru_victims(lru) == [0, 1, 2, 3]   # back at its place: pinning is not use
    rdp.slora_lru_pin(lru, 2)
    rdp.slora_lru_touch(lru, 2)              # use while held
    rdp.slora_lru_unpin(lru, 2)
    assert rdp.slora_lru_victims(lru) == [0, 1, 3, 2]


def test_errors_change_nothing(lru):
    rdp.slora_lru_insert(lru, 7)
    rdp.slora_lru_pin(lru, 7)
    for fn, arg in ((rdp.slora_lru_remove, 7), (rdp.slora_lru_remove, 8), (rdp.slora_lru_touch, 8),
                    (rdp.slora_lru_pin, 8), (rdp.slora_lru_unpin, 8)):
        with pytest.raises(rdp.SloraError) as ei:
            fn(lru, arg)
        assert ei.value.status == 1
    rdp.slora_lru_unpin(lru, 7)
    with pytest.raises(rdp.SloraError):
        rdp.slora_lru_unpin(lru, 7)          # no hold left
    assert rdp.slora_lru_victims(lru) == [7]
    rdp.slora_lru_remove(lru, 7)
    assert rdp.slora_lru_victims(lru) == []


class ListModel:
    """The policy written out plainly: a list in order of last use, hold counts."""

    def __init__(self):
        self.order, self.pins = [], {}

    def insert(self, a):
        if a not in self.pins:
            self.order.append(a)
            self.pins[a] = 0

    def remove(self, a):
        if a not in self.pins or self.pins[a] > 0:
            return False
        self.order.remove(a)
        del self.pins[a]
        return True

    def touch(self, a):
        if a not in self.pins:
            return False
        self.order.remove(a)
        self.order.append(a)
        return True

    def pin(self, a):
        if a not in self.pins:
            return False
        self.pins[a] += 1
        return True

    def unpin(self, a):
        if self.pins.get(a, 0) == 0:
            return False
        self.pins[a] -= 1
        return True

    def victims(self, exclude):
        return [a for a in self.order if self.pins[a] == 0 and a not in exclude]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_random_operations_match_the_list_model(lru, seed):
    rng = np.random.default_rng(seed)
    model = ListModel()
    ops = {"insert": rdp.slora_lru_insert, "remove": rdp.slora_lru_remove, "touch": rdp.slora_lru_touch,
           "pin": rdp.slora_lru_pin, "unpin": rdp.slora_lru_unpin}
    for step in range(600):
        name = rng.choice(list(ops))
        a = int(rng.integers(0, 24))
        want = getattr(model, name)(a)
        want = True if want is None else want
        try:
            ops[name](lru, a)
            got = True
        except rdp.SloraError:
            got = False
        assert got == want, (step, name, a)
        if step % 25 == 0:
            ex = [int(v) for v in rng.integers(0, 24, size=3)]
            assert rdp.slora_lru_victims(lru, exclude=ex) == model.victims(set(ex)), step
    assert rdp.slora_lru_victims(lru) == model.victims(set())
