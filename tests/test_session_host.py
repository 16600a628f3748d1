"""Host-side checks of the session module (no GPU needed)."""

import pytest

from paged_fp8_kv_gb300 import synthetic as syn
from paged_fp8_kv_gb300.session import StagedPipeline


def test_pipeline_depth_is_checked_before_any_device_work():
    w = syn.config(1)
    for depth in (0, -1):
        with pytest.raises(ValueError):
            StagedPipeline(w, depth=depth, device="cpu")
