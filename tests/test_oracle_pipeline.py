"""Pins of the 1F1B pipeline workload oracle (CPU only)."""
import numpy as np

from oracle import pipeline
from tests import pins


def test_1f1b_shape():
    pins.check_1f1b_shape(pipeline.one_f_one_b)


def test_closed_form_xor():
    pins.check_pipeline_closed_form(pipeline.simulate, np.random.default_rng(0))


def test_the_pipeline_driver_issues_the_oracle_order():
    """The GPU pipeline driver's per-stage operation order (host logic, no GPU) is the oracle's 1F1B."""
    from collective_communication_schedules_gb300.pipeline import stage_order
    for p in range(1, 9):
        for m in range(1, 17):
            assert stage_order(p, m) == pipeline.one_f_one_b(p, m), (p, m)
