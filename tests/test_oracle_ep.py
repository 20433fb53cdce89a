"""Pins of the EP pack / combine oracle (CPU only)."""
import numpy as np

from collective_communication_schedules_gb300 import inputs
from oracle import ep
from tests import pins


def test_pack_matches_brute_force():
    pins.check_ep_pack_brute(ep.pack, np.random.default_rng(0))


def test_pack_agrees_with_a_four_key_sort():
    w = inputs.EP_DISPATCH
    routing = inputs.ep_routing(2, 64, w["experts"], w["topk"], w["zipf"], seed_base=77)
    x = inputs.normal_bf16(64 * 16, 78).reshape(64, 16)
    for r in range(2):
        pins.check_ep_pack_four_key_sort(ep.pack, x, routing[r], w["experts"], 2)


def test_combine_matches_scalar_brute_force():
    pins.check_ep_combine_scalar(ep.pack, ep.combine, np.random.default_rng(1))


def test_combine_topk1_unit_weight_is_identity():
    pins.check_ep_combine_identity(ep.pack, ep.combine, np.random.default_rng(2))


def test_combine_golden_cases():
    pins.check_ep_combine_golden(ep.combine)


def test_combine_within_the_error_bound():
    pins.check_ep_combine_error_bound(ep.pack, ep.combine, np.random.default_rng(3))
