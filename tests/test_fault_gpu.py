"""Failure detection on the GPU without a fault: a kernel whose data never
arrives must give up its bounded waits, report RA_ERR_TIMEOUT through the
device status word, and leave the device usable."""
import time

import pytest
import torch

from gpu_helpers import TOL, fwd_full_check
from ring_attention_fwd_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


def test_withheld_tile_times_out_cleanly_and_device_stays_usable(fwd_kernel):
    import ring_attention_fwd_gb300 as ra
    L = ra.binding.lib()
    inp = {k: v.cuda() for k, v in make_inputs(1, 2, 1024, 128, seed=41).items()}
    ra.check_device_status()                       # start from a clean status word
    assert L.ra_set_wait_test(1) == 0
    t0 = time.time()
    ra.fwd(inp["q"], inp["k"], inp["v"], 4, True, "contiguous")
    with pytest.raises(ra.RingAttnError) as ei:
        ra.check_device_status()
    elapsed = time.time() - t0
    assert ei.value.code == ra.binding.RA_ERR_TIMEOUT and "timed out" in str(ei.value)
    assert elapsed < 30, elapsed                   # bounded: ~2 s wait limit plus a short drain
    ra.check_device_status()                       # the word was cleared; no CUDA error is pending
    # the switch was one-shot: the next call is normal and correct
    eo, el = fwd_full_check(ra, make_inputs(1, 2, 512, 128, seed=42), 2, True, "striped", "bf16")
    assert eo <= TOL["bf16"]["o"] and el <= TOL["bf16"]["lse"]
