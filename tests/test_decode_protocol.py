"""The tensor-core decode's barrier protocol, run under random interleavings
on the CPU (`tests/decode_protocol_model.py`): every completion order gives
no deadlock, no aliased parity wait and no buffer overwritten while it is
still needed; and each planted mistake is caught."""
import pytest

from tests import decode_protocol_model as M

TILE_COUNTS = list(range(1, 25)) + [53, 81]


@pytest.mark.parametrize("ntiles", TILE_COUNTS)
def test_protocol_holds_under_random_completion_order(ntiles):
    for seed in range(25):
        M.run(ntiles, seed)


@pytest.mark.parametrize("mutation", M.MUTATIONS)
def test_planted_protocol_mistake_is_caught(mutation):
    for ntiles in (3, 5, 8, 12, 17, 24, 53):
        for seed in range(60):
            try:
                M.run(ntiles, seed, mutation)
            except M.ProtocolError:
                return
    pytest.fail("no interleaving exposed the planted mistake %r" % mutation)
