"""Test configuration: the ``gpu`` marker and import paths.

``-m "not gpu"`` runs on any machine (oracle pins, host logic, ABI exports);
``-m gpu`` needs a CUDA device and a built library.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
for p in (ROOT, os.path.join(ROOT, "tests")):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the built liblse")
