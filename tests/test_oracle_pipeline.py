"""Pins of the 1F1B pipeline workload oracle (CPU only)."""
import numpy as np

from oracle import pipeline
from tests import pins


def test_1f1b_shape():
    pins.check_1f1b_shape(pipeline.one_f_one_b)


def test_closed_form_xor():
    pins.check_pipeline_closed_form(pipeline.simulate, np.random.default_rng(0))
