import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# A stream held at a device-count all-to-all's start flag blocks the hardware
# work queue it is mapped to, and CUDA maps streams onto
# CUDA_DEVICE_MAX_CONNECTIONS queues (8 by default): the host proxy's copy
# streams can land on the held stream's queue and then wait for the watchdog
# (seen in about 3 of 10 fresh processes at 8 queues, none at 32).  Set before
# any CUDA context exists.
os.environ.setdefault("CUDA_DEVICE_MAX_CONNECTIONS", "32")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload (runs in the gpu tier)")
