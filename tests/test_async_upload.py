"""Asynchronous adapter upload (GPU): uploads enqueued on one stream while
lora_layer_forward runs on another, a replacement ordered after its readers,
a kernel launched on the upload's own stream right after it, the prefetch
list, and pages of asynchronously unloaded adapters reused.  Every result is
checked against the CPU oracle.

Source: S-LoRA slide 9 (adapters copied to the GPU asynchronously while a
batch computes) and "Multi-LoRA Serving - S-LoRA/Punica Batching, Adapter
Hot-Swap & Memory", section "Memory: slots, tiers and paging" (host tier
plus prefetch).
"""
import dataclasses

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

import oracle  # noqa: E402
from segmented_gathered_rank_gb300 import harness as H  # noqa: E402
from segmented_gathered_rank_gb300 import inputs as I  # noqa: E402
from segmented_gathered_rank_gb300 import lora as L  # noqa: E402
from tests.parity import TOL_Y, oracle_delta, rel_err, token_ids  # noqa: E402

RANKS = [16, 8, 32, 16, 128, 16, 8, 32, 16, 128]     # adapters 0-4 resident first, 5-9 uploaded later


def _workload(seed, ids, T=700, lengths=None):
    w = I.random_case(seed, T=T, lengths=lengths or [256, 128, 1, 1, 1, 313], h_in=1024, h_out=512, ranks=RANKS)
    w.seg_adapter = np.array(ids, np.int32)
    return w


def _prep(dp, w):
    """Device inputs of one layer call (ready when this returns)."""
    t = dict(ss=H.int_tensor(w.seg_starts), sa=H.int_tensor(w.seg_adapter), x=H.to_device(w.x(0), w.dtype),
             W=H.to_device(w.W(0), w.dtype),
             ws=torch.empty(L.lora_layer_forward_workspace_size(dp.handle, 0, w.S, w.T), dtype=torch.uint8,
                            device="cuda"),
             y=torch.full((w.T, 512), float("nan"), dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    return t


def _run(dp, w, t, stream):
    L.lora_layer_forward(dp.handle, 0, t["x"], t["W"], t["y"], t["ss"], t["sa"], w.S, w.T, t["ws"], stream=stream)
    return t["y"]


def _layer(dp, w, stream):
    """Enqueue lora_layer_forward on `stream`; returns (y, keep-alive tensors)."""
    t = _prep(dp, w)
    return _run(dp, w, t, stream), t


def _check_layer(w, y, ad=None):
    tok = token_ids(w)
    ad = ad or oracle.adapters_for(w, 0, ids=range(w.n_adapters))
    ref, st = oracle.layer(w.x(0), w.W(0), tok, ad, 512)
    assert st == 0
    got = H.to_host(y)
    assert not np.isnan(got).any()
    assert rel_err(got, ref) <= TOL_Y[w.dtype]


def _upload(dp, w, a, stream, seed_shift=0):
    at, b = w.adapter(a, 0, layer=seed_shift)
    L.lora_pool_load_async(dp.handle, a, 0, int(w.ranks[a]), float(w.scales[a]), 1024, 512,
                           H.host_array(at, w.dtype), H.host_array(b, w.dtype), stream=stream)
    return at, b


def test_upload_while_layer_runs_on_another_stream():
    w1 = _workload(81, [0, 1, 2, 3, 4, 0])
    w2 = _workload(81, [5, 6, 7, 8, 9, 5])        # same adapter population, the other half
    with H.DevicePool(w1, load_ids=range(5), spare_pages=2 * int(np.sum(RANKS[5:]))) as dp:
        s_a, s_b = torch.cuda.Stream(), torch.cuda.Stream()
        t1, t2 = _prep(dp, w1), _prep(dp, w2)
        y1 = _run(dp, w1, t1, s_a)                           # batch 1 on stream A
        for a in range(5, 10):                               # uploads on stream B, beside it
            _upload(dp, w2, a, s_b)
        # the workspace a layer call needs grows with the adapter ids loaded on the matrix
        t2["ws"] = torch.empty(L.lora_layer_forward_workspace_size(dp.handle, 0, w2.S, w2.T), dtype=torch.uint8,
                               device="cuda")
        y2 = _run(dp, w2, t2, s_b)                           # batch 2, after them on stream B
        torch.cuda.synchronize()
        assert dp.check_device_status() == 0
        _check_layer(w1, y1)
        _check_layer(w2, y2)


def test_replacement_ordered_after_its_readers():
    w = _workload(82, [0, 1, 2, 3, 4, 0])
    with H.DevicePool(w, load_ids=range(5), spare_pages=2 * 128) as dp:
        s_a, s_b = torch.cuda.Stream(), torch.cuda.Stream()
        y_old, keep = _layer(dp, w, s_a)                     # reads adapter 4 (rank 128) as loaded
        done = torch.cuda.Event()
        done.record(s_a)
        s_b.wait_event(done)                                 # the replacement waits for its readers
        at_new, b_new = _upload(dp, w, 4, s_b, seed_shift=7)
        y_new, keep2 = _layer(dp, w, s_b)
        torch.cuda.synchronize()
        assert dp.check_device_status() == 0
        _check_layer(w, y_old)
        entries = {a: (int(w.ranks[a]), float(w.scales[a]), *w.adapter(a, 0)) for a in range(5)}
        entries[4] = (128, float(w.scales[4]), at_new, b_new)
        _check_layer(w, y_new, oracle.Adapters(w.n_adapters, entries))
        # the replaced adapter's pages are back once the stream has passed the update
        assert L.lora_pool_free_pages(dp.handle) == dp.n_pages - 2 * int(np.sum(RANKS[:5]))


def test_kernel_right_after_upload_on_the_same_stream_sees_it():
    # BGMV reads page tables before it waits for the kernel ahead of it in its
    # stream; the upload ends with a copy, so the record it reads is the new one
    w = I.random_case(83, T=256, decode=True, ranks=[16, 16, 64, 8], h_in=1024, h_out=1024)
    w.token_adapter[:] = np.arange(256) % 4
    w.seg_adapter = w.token_adapter.copy()
    with H.DevicePool(w, load_ids=[0, 1], spare_pages=2 * (64 + 8)) as dp:
        s = torch.cuda.Stream()
        x = H.to_device(w.x(0), w.dtype)
        y0 = w.y0(0)
        y = H.to_device(y0, w.dtype)
        tok = H.int_tensor(w.token_adapter)
        torch.cuda.synchronize()
        for a in (2, 3):
            at, b = w.adapter(a)
            L.lora_pool_load_async(dp.handle, a, 0, int(w.ranks[a]), float(w.scales[a]), 1024, 1024,
                                   H.host_array(at, w.dtype), H.host_array(b, w.dtype), stream=s)
        L.lora_bgmv(dp.handle, 0, x, y, tok, w.T, stream=s)
        torch.cuda.synchronize()
        assert dp.check_device_status() == 0
        ref, st = oracle_delta(w, 0, y0, ids=range(4))
        assert st == 0 and rel_err(H.to_host(y), ref) <= TOL_Y[w.dtype]


def test_prefetch_list_uploads_only_missing_adapters():
    w = _workload(84, [5, 6, 7, 8, 9, 2])
    with H.DevicePool(w, load_ids=[2, 5, 6], spare_pages=2 * int(np.sum(RANKS[7:]))) as dp:
        s = torch.cuda.Stream()
        keep, entries = [], []
        for a in range(5, 10):
            at, b = (H.host_array(t, w.dtype) for t in w.adapter(a))
            keep += [at, b]
            entries.append((a, 0, int(w.ranks[a]), float(w.scales[a]), 1024, 512, at, b))
        assert L.lora_pool_prefetch(dp.handle, entries, stream=s) == 3      # 5 and 6 are resident
        assert L.lora_pool_prefetch(dp.handle, entries, stream=s) == 0      # now all are
        y, keep2 = _layer(dp, w, s)
        torch.cuda.synchronize()
        assert dp.check_device_status() == 0
        _check_layer(w, y, oracle.adapters_for(w, 0, ids=[2, 5, 6, 7, 8, 9]))


def test_unload_async_pages_serve_a_later_upload():
    w = _workload(85, [0, 1, 2, 3, 1, 0], lengths=[256, 128, 1, 1, 1, 313])
    # room for adapters 0-4 only: the upload of 9 (rank 128) needs the pages of 4 (rank 128)
    with H.DevicePool(w, load_ids=range(5), spare_pages=0) as dp:
        s = torch.cuda.Stream()
        free0 = L.lora_pool_free_pages(dp.handle)
        L.lora_pool_unload_async(dp.handle, 4, 0, stream=s)
        at, b = _upload(dp, w, 9, s)                        # waits for the retired pages if it must
        wd = dataclasses.replace(w, seg_adapter=np.array([0, 1, 2, 3, 9, 0], np.int32))
        y, keep = _layer(dp, wd, s)
        torch.cuda.synchronize()
        assert dp.check_device_status() == 0
        _check_layer(wd, y, oracle.adapters_for(wd, 0, ids=[0, 1, 2, 3, 9]))
        assert L.lora_pool_free_pages(dp.handle) == free0
        with pytest.raises(L.LoraError) as e:
            L.lora_pool_unload_async(dp.handle, 4, 0, stream=s)
        assert e.value.status == L.LORA_ERR_NOT_LOADED
