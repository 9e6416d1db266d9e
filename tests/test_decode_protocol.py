"""The tensor-core decode's barrier protocol, run under random interleavings
on the CPU (`tests/decode_protocol_model.py`), in both of its forms (bf16
cache: each CTA loads what it needs and only P crosses the cluster; fp8
cache: each CTA forwards the half of the tile its peer lacks): every
completion order gives no deadlock, no aliased
parity wait and no buffer overwritten while it is still needed; and each
planted mistake is caught."""
import pytest

from tests import decode_protocol_model as M

TILE_COUNTS = list(range(1, 25)) + [53, 81]


FORMS = [True, False]
FORM_IDS = ["bf16_decoupled", "fp8_copied_recv"]


@pytest.mark.parametrize("decoupled", FORMS, ids=FORM_IDS)
@pytest.mark.parametrize("ntiles", TILE_COUNTS)
def test_protocol_holds_under_random_completion_order(ntiles, decoupled):
    for seed in range(25):
        M.run(ntiles, seed, decoupled=decoupled)


@pytest.mark.parametrize("mutation,decoupled", [(m, f) for m, form in M.MUTATIONS.items() for f in FORMS
                                                if form is None or form == f])
def test_planted_protocol_mistake_is_caught(mutation, decoupled):
    for ntiles in (3, 5, 8, 12, 17, 24, 53):
        for seed in range(60):
            try:
                M.run(ntiles, seed, mutation, decoupled=decoupled)
            except M.ProtocolError:
                return
    pytest.fail("no interleaving exposed the planted mistake %r" % mutation)


@pytest.mark.parametrize("decoupled", FORMS, ids=FORM_IDS)
@pytest.mark.parametrize("own,recv", [(8, 3), (9, 2)])
def test_other_splits_of_the_value_rings_hold(monkeypatch, own, recv, decoupled):
    # the value CTA's own and receive rings share one region; the kernel's
    # split is 7 + 4, and these fit the same region
    monkeypatch.setattr(M, "K_OWN", own)
    monkeypatch.setattr(M, "K_RECV", recv)
    for ntiles in (1, 2, 5, 9, 16, 23, 54):
        for seed in range(15):
            M.run(ntiles, seed, decoupled=decoupled)


@pytest.mark.parametrize("decoupled", FORMS, ids=FORM_IDS)
def test_receive_ring_deeper_than_the_p_slots_is_caught(monkeypatch, decoupled):
    # With more receive slots than P slots, the receive warp's p_ok arrival
    # for tile j + 4 can land in tile j's open phase (its receive slot no
    # longer waits for PV(j)), so PV(j) could start before O is rescaled for
    # tile j.  A build with these ring sizes gave wrong outputs on the GPU;
    # the kernel now asserts kRecv <= kPSlots at compile time.
    monkeypatch.setattr(M, "K_OWN", 6)
    monkeypatch.setattr(M, "K_RECV", 5)
    for ntiles in (6, 9, 17, 54):
        for seed in range(40):
            try:
                M.run(ntiles, seed, decoupled=decoupled)
            except M.ProtocolError as e:
                assert "mixes arrivals" in str(e)
                return
    pytest.fail("the early p_ok arrival was not caught")
