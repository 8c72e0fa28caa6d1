import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running case")


@pytest.fixture(params=["auto", "split"])
def decode_impl(request, monkeypatch):
    """auto: small batches take the decode's one-launch path (one CTA per
    (sequence, kv head)), larger ones the split-KV path; split: every call
    takes the split-KV path (PKV_DECODE_IMPL=split)."""
    if request.param == "split":
        monkeypatch.setenv("PKV_DECODE_IMPL", "split")
    else:
        monkeypatch.delenv("PKV_DECODE_IMPL", raising=False)
    return request.param
