"""Bounded device waits: a kernel whose mbarrier is never signalled gives up
after its limit, records FP8FG_ERR_TIMEOUT in the device status word and
returns; the context stays usable.  No fault, trap or hang is involved."""
from __future__ import annotations

import time

import numpy as np
import pytest
import torch

from fp8_fine_grained_act_gb300 import binding as fb
from fp8_fine_grained_act_gb300 import synth
from gpu_util import dev_bf16, host

pytestmark = pytest.mark.gpu


def test_wait_times_out_and_reports(gpu_device):
    fb.fp8fg_last_device_status()                            # clear
    t0 = time.perf_counter()
    assert fb.fp8fg_selftest_watchdog(2_000_000) == 0        # 2 ms limit
    assert fb.fp8fg_last_device_status() == fb.FP8FG_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 5.0
    assert fb.fp8fg_last_device_status() == 0                # read clears it
    # the context still works
    x = synth.activations_random_outliers(np.random.default_rng(0), 4, 128)
    q, s = fb.fp8_quant_act_1x128(dev_bf16(x, gpu_device))
    torch.cuda.synchronize()
    assert host(s).shape == (1, 4)
