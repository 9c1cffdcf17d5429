"""The bounded-wait watchdog, exercised without any fault: a self-test
kernel waits on an mbarrier nobody arrives on; the wait runs out after its
limit, records ATTN_ERR_TIMEOUT in the library's device word and returns.
The context stays usable and the status word is cleared once read."""
import pytest
import torch

import attn_inputs as ai
import warp_specialized_gb300 as ws
from attn_check import compare, run_gpu

pytestmark = pytest.mark.gpu


def test_watchdog_reports_timeout_and_context_survives():
    ws.load_library(build_if_missing=True)
    assert ws.attn_fwd_status() == 0
    assert ws.attn_watchdog_selftest(2000) == 6          # ATTN_ERR_TIMEOUT
    assert ws.attn_fwd_status() == 0                     # cleared when read
    inp = ai.make_inputs(1, 2, 256, 128, "bf16", seed=3)  # the device still works
    o, lse = run_gpu(inp, False)
    compare(inp, False, o, lse)
