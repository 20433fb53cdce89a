"""Pins of the EP pack / combine oracle (CPU only)."""
import numpy as np

from collective_communication_schedules_gb300 import inputs
from oracle import ep
from tests import pins


def test_pack_matches_brute_force():
    pins.check_ep_pack_brute(ep.pack, np.random.default_rng(0))


def test_pack_agrees_with_the_input_generator_layout():
    w = inputs.EP_DISPATCH
    routing = inputs.ep_routing(2, 64, w["experts"], w["topk"], w["zipf"], seed_base=77)
    x = inputs.normal_bf16(64 * 16, 78).reshape(64, 16)
    for r in range(2):
        send, perm, _, counts = ep.pack(x, routing[r], w["experts"], 2)
        gsend, order, gcounts = inputs.ep_pack(routing[r], x, w["experts"], 2)
        assert np.array_equal(send, gsend)
        assert np.array_equal(counts, gcounts * 16)
        assert np.array_equal(perm, order[:, 0] * w["topk"] + order[:, 1])


def test_combine_matches_scalar_brute_force():
    pins.check_ep_combine_scalar(ep.pack, ep.combine, np.random.default_rng(1))


def test_combine_topk1_unit_weight_is_identity():
    pins.check_ep_combine_identity(ep.pack, ep.combine, np.random.default_rng(2))


def test_combine_golden_cases():
    pins.check_ep_combine_golden(ep.combine)


def test_combine_within_the_error_bound():
    pins.check_ep_combine_error_bound(ep.pack, ep.combine, np.random.default_rng(3))
