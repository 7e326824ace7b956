"""Shared pytest configuration.

Tests marked ``gpu`` need a CUDA device and the compiled library; everything
else runs on the CPU (oracle pins, host-side logic, library symbol checks).
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the compiled libgdn")
    config.addinivalue_line("markers", "slow: larger CPU cases")
