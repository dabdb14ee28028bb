"""Failure path without a GPU fault: a bounded device wait that nothing will
complete gives up, records a timeout in the status word, and the context keeps
working."""
import pytest
import torch

from . import _gpu as G

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    b = G.nk()
    assert b.nvfp4kv_get_device_status() == 0
    b.nvfp4kv_debug_wait_timeout(2_000_000)        # 2 ms limit
    assert b.nvfp4kv_get_device_status() == -5
    assert b.nvfp4kv_get_device_status() == 0      # read clears
    x = torch.ones(1024, device=G.dev())
    assert float(x.sum()) == 1024.0                # the context is still usable
