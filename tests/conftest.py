import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running oracle case")


@pytest.fixture(scope="session")
def tiny_decoder():
    from synthetic import SHAPES, make_weights, weights_to_numpy
    from oracle.decoder import Decoder
    shape = SHAPES["tiny"]
    return Decoder(shape, weights_to_numpy(make_weights(shape, seed=1)))
