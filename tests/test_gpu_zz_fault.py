"""Failure detection without a GPU fault: every device wait of the library is bounded.

hq_selftest_bounded_wait launches one warp that waits, through the kernels' own bounded mbarrier
wait, on a barrier that nothing completes.  The wait must give up (about one second), record
bit 0 in the device fault word that hq_read_fault returns, and leave the context usable: a
quantization right after it is bit-exact and records no fault.  (The file name sorts last so
that the fault word it sets, then clears, is not seen by other tests.)
"""
import time

import numpy as np
import pytest
import torch

import hadamard_rotation_gb300 as hq
import oracle
from hadamard_rotation_gb300 import synth

pytestmark = pytest.mark.gpu


def read_fault(clear):
    return hq.hq_read_fault(clear=clear)


@pytest.mark.parametrize("unit", [0, 1])  # NVFP4/MXFP4 unit, INT8 unit
def test_bounded_wait_gives_up_and_is_reported(unit):
    from hadamard_rotation_gb300 import build

    build.build()
    oracle.build()
    hq.load()
    assert read_fault(clear=True) == 0            # nothing recorded before
    t0 = time.perf_counter()
    hq.hq_selftest_bounded_wait(unit)
    fault = read_fault(clear=True)                  # synchronises: the wait has ended
    elapsed = time.perf_counter() - t0
    assert fault == 1, fault
    assert 0.5 < elapsed < 30.0, elapsed            # gave up after about a second
    assert read_fault(clear=False) == 0             # cleared
    # the context is still usable: a quantization right after is exact and fault-free
    x_host = synth.generate(synth.WORKLOADS["tiny_f32_128x256"])
    q, s, sg, amax = hq.quantize_nvfp4(x_host.cuda(), 16)
    torch.cuda.synchronize()
    oq, os_, _, _ = oracle.quantize(synth.as_oracle_array(x_host), 16)
    assert np.array_equal(q.cpu().numpy(), oq) and np.array_equal(s.cpu().numpy(), os_)
    assert read_fault(clear=False) == 0
