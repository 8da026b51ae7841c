"""HostPipeline argument checks that need no GPU."""
import pytest

import w8a8_int8_linear_gb300 as w8a8


def test_host_pipeline_rejects_zero_depth():
    with pytest.raises(ValueError, match="depth"):
        w8a8.HostPipeline(lambda X, Y: None, (1, 16), (1, 16), "cpu", depth=0)
