"""The bench's pipelined end-to-end steps (GPU): every step copies its inputs
in from pinned host memory and its results back, with two device buffer sets
and copy streams overlapping neighbouring steps.  The results that reach the
host must be, bit for bit, what one step computes on the device."""
import pytest
import torch

import bench

pytestmark = pytest.mark.gpu


def test_fused_layer_e2e_steps_match_the_device_step():
    R = bench.RUNNERS["fused_layer"]()
    try:
        R.step()
        torch.cuda.synchronize()
        ref = [y.cpu() for y in R.y]
        R.e2e_setup()
        for _ in range(3):                       # both buffer sets, and one reused
            R.e2e_step()
        torch.cuda.synchronize()
        for m in range(4):
            assert torch.equal(R._p_down[f"y{m}"], ref[m]), m
        assert R.pool.check_device_status() == 0
    finally:
        R.pool.close()


def test_prefill_e2e_steps_match_the_device_step():
    # y is read-modify-written: every e2e step uploads y0 again, so every step's
    # result is y0 + delta, what one device step gives from y0
    R = bench.RUNNERS["prefill_sgmv"]()
    try:
        R.e2e_setup()                            # host copies of x and y0
        R.step()
        torch.cuda.synchronize()
        ref = [y.cpu() for y in R.y]
        for _ in range(3):
            R.e2e_step()
        torch.cuda.synchronize()
        for m in range(4):
            assert torch.equal(R._p_down[f"y{m}"], ref[m]), m
        assert R.pool.check_device_status() == 0
    finally:
        R.pool.close()
