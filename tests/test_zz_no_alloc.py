"""lora_layer_forward_noalloc against lora_layer_forward (GPU).

Some callers cannot allocate device memory (a fixed-arena serving runtime, a
decode loop that must not call cudaMalloc because it synchronises the
device, a C plugin without an allocator).  lora_layer_forward_noalloc serves
them from a fixed scratch array inside the library.  This test calls it
through the C ABI twice in a row, on two different batches that share the
one scratch array, and checks that each result has exactly the bits of the
workspace-taking entry point (both run the same kernels with the same fixed
reduction orders; only where the scratch lives differs) and that both launch
the same number of kernels.  It lives in its own file, named to be collected
last.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

from segmented_gathered_rank_gb300 import harness as H  # noqa: E402
from segmented_gathered_rank_gb300 import inputs as I  # noqa: E402
from segmented_gathered_rank_gb300 import lora as L  # noqa: E402


def _both(dp, w, seed_layer):
    ss, sa = H.int_tensor(w.seg_starts), H.int_tensor(w.seg_adapter)
    x = H.to_device(w.x(0, seed_layer), w.dtype)
    Wd = H.to_device(w.W(0, seed_layer), w.dtype)
    h_out = w.matrices[0].h_out
    y_ref = torch.full((w.T, h_out), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(L.lora_layer_forward_workspace_size(dp.handle, 0, w.S, w.T), dtype=torch.uint8, device="cuda")
    n0 = L.lora_launch_count()
    L.lora_layer_forward(dp.handle, 0, x, Wd, y_ref, ss, sa, w.S, w.T, ws)
    n1 = L.lora_launch_count()
    y = torch.full((w.T, h_out), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.lora_layer_forward_noalloc(dp.handle, 0, x, Wd, y, ss, sa, w.S, w.T)
    n2 = L.lora_launch_count()
    torch.cuda.synchronize()
    return H.to_host(y), H.to_host(y_ref), n1 - n0, n2 - n1


def test_noalloc_matches_workspace_entry_point_twice():
    w = I.random_case(71, T=700, lengths=[300, 0, 1, 399], h_in=1024, h_out=512, ranks=[16, 128, 8])
    with H.DevicePool(w) as dp:
        for call in range(2):   # second call reuses the scratch the first one left behind
            y, y_ref, launches_ref, launches = _both(dp, w, seed_layer=call)
            assert not np.isnan(y).any()
            assert np.array_equal(y, y_ref), call
            assert launches == launches_ref > 0, call
        assert dp.check_device_status() == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    w = I.random_case(72, T=64, lengths=[64], h_in=256, h_out=256, ranks=[128])
    with H.DevicePool(w) as dp:
        T = L.LORA_NOALLOC_SCRATCH_BYTES // (4 * w.max_rank)     # v alone fills the scratch; the plan does not fit
        x = torch.zeros((T, 256), dtype=torch.bfloat16, device="cuda")
        Wd = torch.zeros((256, 256), dtype=torch.bfloat16, device="cuda")
        y = torch.zeros((T, 256), dtype=torch.bfloat16, device="cuda")
        ss = H.int_tensor([0, T])
        sa = H.int_tensor([0])
        n0 = L.lora_launch_count()
        with pytest.raises(L.LoraError) as e:
            L.lora_layer_forward_noalloc(dp.handle, 0, x, Wd, y, ss, sa, 1, T)
        assert e.value.status == L.LORA_ERR_ARG
        assert L.lora_launch_count() == n0
