"""GPU parity: every entry point against the CPU oracle on seeded inputs.

Covers the five workloads at full size (the fused layer on sampled rows of
q and o, and on every row of k), small randomized ragged cases, integer
probes compared bit for bit, and the edge cases: empty segments, tokens
without an adapter, invalid ids, bad segment tables, rank-0 and zero-B
adapters computed through every entry point (their rows keep the base or y0
output bit for bit), T = 0, pool exhaustion and page reuse.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU, skipped there
    pytest.skip("needs a GPU", allow_module_level=True)

import oracle  # noqa: E402
from segmented_gathered_rank_gb300 import harness as H  # noqa: E402
from segmented_gathered_rank_gb300 import inputs as I  # noqa: E402
from segmented_gathered_rank_gb300 import lora as L  # noqa: E402
from tests.parity import (TOL_V, TOL_Y, oracle_delta, oracle_v, rel_err, sample_rows,  # noqa: E402
                          written_mask)


def _tables(w):
    return H.int_tensor(w.seg_starts), H.int_tensor(w.seg_adapter)


def run_sgmv(w, m=0, zero_y0=False):
    """shrink then expand on one matrix; returns (v, y, device status)."""
    with H.DevicePool(w, matrices=[m]) as dp:
        ss, sa = _tables(w)
        x = H.to_device(w.x(m), w.dtype)
        y0 = np.zeros((w.T, w.matrices[m].h_out), np.float32) if zero_y0 else w.y0(m)
        y = H.to_device(y0, w.dtype)
        ld_v = w.max_rank
        v = torch.full((w.T, ld_v), float("nan"), dtype=torch.float32, device="cuda")
        L.lora_sgmv_shrink(dp.handle, 0, x, v, ld_v, ss, sa, w.S, w.T)
        L.lora_sgmv_expand(dp.handle, 0, v, ld_v, y, ss, sa, w.S, w.T)
        word = dp.check_device_status()
        return H.to_host(v), H.to_host(y), y0, word


def run_bgmv(w, m=0, zero_y0=False):
    with H.DevicePool(w, matrices=[m]) as dp:
        ids = w.token_adapter if w.token_adapter is not None else w.seg_adapter
        tok = H.int_tensor(ids)
        x = H.to_device(w.x(m), w.dtype)
        y0 = np.zeros((w.T, w.matrices[m].h_out), np.float32) if zero_y0 else w.y0(m)
        y = H.to_device(y0, w.dtype)
        L.lora_bgmv(dp.handle, 0, x, y, tok, w.T)
        word = dp.check_device_status()
        return H.to_host(y), y0, word


def run_layer(w, m=0, zero_w=False):
    with H.DevicePool(w, matrices=[m]) as dp:
        ss, sa = _tables(w)
        x = H.to_device(w.x(m), w.dtype)
        Wh = np.zeros((w.matrices[m].h_out, w.matrices[m].h_in), np.float32) if zero_w else w.W(m)
        Wd = H.to_device(Wh, w.dtype)
        y = torch.full((w.T, w.matrices[m].h_out), float("nan"), dtype=H.torch_dtype(w.dtype), device="cuda")
        ws_bytes = L.lora_layer_forward_workspace_size(dp.handle, 0, w.S, w.T)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        L.lora_layer_forward(dp.handle, 0, x, Wd, y, ss, sa, w.S, w.T, ws)
        word = dp.check_device_status()
        return H.to_host(y), Wh, word


def check_sgmv(w, m=0, rows=None):
    for zero in (True, False):
        v, y, y0, word = run_sgmv(w, m, zero_y0=zero)
        assert word == 0
        vr, st = oracle_v(w, m, w.max_rank)
        assert st == 0
        mask = written_mask(w, w.max_rank)
        assert not np.isnan(v[mask]).any()
        assert rel_err(v[mask], vr[mask]) <= TOL_V[w.dtype]
        yr, st = oracle_delta(w, m, y0)
        assert st == 0
        e = rel_err(y, yr)
        assert e <= TOL_Y[w.dtype], (zero, e)


def check_bgmv(w, m=0):
    for zero in (True, False):
        y, y0, word = run_bgmv(w, m, zero_y0=zero)
        assert word == 0
        yr, st = oracle_delta(w, m, y0)
        assert st == 0
        e = rel_err(y, yr)
        assert e <= TOL_Y[w.dtype], (zero, e)


# ---------------------------------------------------------------------------
# The five workloads
# ---------------------------------------------------------------------------
def test_tiny_sgmv_f32():
    check_sgmv(I.tiny_sgmv())


def test_tiny_layer_f32():
    w = I.tiny_sgmv()
    y, Wh, word = run_layer(w)
    assert word == 0
    yr, st = oracle_delta(w, 0, None, W=Wh)
    assert st == 0 and rel_err(y, yr) <= TOL_Y[w.dtype]


def test_decode_bgmv_full():
    check_bgmv(I.decode_bgmv())


def test_decode_batch_as_unit_segments():
    check_sgmv(I.decode_bgmv())


@pytest.mark.parametrize("m", [0, 1])   # q (4096 -> 4096) and k (4096 -> 1024)
def test_prefill_sgmv_full(m):
    check_sgmv(I.prefill_sgmv(), m)


@pytest.mark.parametrize("m", [0, 47])
def test_encoder_mixed_rank_full(m):
    check_sgmv(I.encoder_mixed_rank(), m)


def test_encoder_mixed_rank_bgmv():
    """The same mixed-rank batch through BGMV, one adapter id per token (MBGMV)."""
    w = I.encoder_mixed_rank()
    w.token_adapter = np.repeat(w.seg_adapter, np.diff(w.seg_starts)).astype(np.int32)
    check_bgmv(w, 5)


def _fused_rows(w):
    rng = np.random.default_rng(1)
    rows = set()
    for s in range(4):
        lo, hi = int(w.seg_starts[s]), int(w.seg_starts[s + 1])
        rows.update({lo, lo + 1, lo + 127, lo + 128, hi - 1})
    rows.update(rng.integers(0, 4096, 24).tolist())
    dec = np.arange(4096, 4608)
    rows.update(rng.choice(dec, 40, replace=False).tolist())
    rows.update(dec[w.seg_adapter[4:] == 0][:8].tolist())   # the rank-128 adapter at decode
    rows.add(4607)
    return np.array(sorted(rows), np.int32)


@pytest.mark.parametrize("m", [0, 1, 3])
def test_fused_layer_sampled(m):
    w = I.fused_layer()
    rows = _fused_rows(w)
    y, Wh, word = run_layer(w, m)
    assert word == 0
    yr, st = oracle_delta(w, m, None, rows=rows, W=Wh)
    assert st == 0
    assert rel_err(y[rows], yr) <= TOL_Y[w.dtype]


def test_fused_layer_k_every_row():
    """The k projection (4096 -> 1024) of the fused workload on all 4608 rows:
    every M-tile of the GEMM, every decode row and the rank-128 adapter's rows
    are compared, so a scheduling slip confined to some rows cannot hide."""
    w = I.fused_layer()
    y, Wh, word = run_layer(w, 1)
    assert word == 0 and not np.isnan(y).any()
    yr, st = oracle_delta(w, 1, None, W=Wh)
    assert st == 0
    assert rel_err(y, yr) <= TOL_Y[w.dtype]


def test_fused_layer_delta_alone():
    w = I.fused_layer()
    rows = _fused_rows(w)
    y, Wh, word = run_layer(w, 0, zero_w=True)
    assert word == 0
    yr, st = oracle_delta(w, 0, None, rows=rows)
    assert st == 0
    assert rel_err(y[rows], yr) <= TOL_Y[w.dtype]


# ---------------------------------------------------------------------------
# Small randomized cases: ragged segments (some empty), ragged ranks,
# tokens without an adapter, T off the tile grid.
# ---------------------------------------------------------------------------
RANDOM = [
    dict(seed=1, T=1, lengths=[1]),
    dict(seed=2, T=77, lengths=[0, 30, 0, 47, 0]),
    dict(seed=3, T=300, none_fraction=0.3),
    dict(seed=4, T=257, h_in=72, h_out=40),
    dict(seed=5, T=513, h_in=1024, h_out=520, ranks=[8, 64, 16, 32, 1]),
    dict(seed=6, T=129, dtype=I.F32, h_in=96, h_out=128),
    dict(seed=7, T=1000, h_in=4096, h_out=1024, ranks=[16, 128, 16, 4]),
    # every adapter above rank 64 and segments of 128+ rows: the tensor-core shrink's segment tiles
    dict(seed=8, T=640, lengths=[512, 0, 127, 1], h_in=512, h_out=256, ranks=[128, 96]),
]


@pytest.mark.parametrize("case", RANDOM, ids=lambda c: f"seed{c['seed']}")
def test_random_sgmv(case):
    check_sgmv(I.random_case(**case))


@pytest.mark.parametrize("case", RANDOM, ids=lambda c: f"seed{c['seed']}")
def test_random_bgmv(case):
    c = dict(case)
    c.pop("lengths", None)
    check_bgmv(I.random_case(decode=True, **c))


@pytest.mark.parametrize("case", RANDOM, ids=lambda c: f"seed{c['seed']}")
def test_random_layer(case):
    w = I.random_case(**case)
    y, Wh, word = run_layer(w)
    assert word == 0
    yr, st = oracle_delta(w, 0, None, W=Wh)
    assert st == 0 and rel_err(y, yr) <= TOL_Y[w.dtype]


# ---------------------------------------------------------------------------
# Integer probes: every partial sum exact -> bit-exact agreement.
# ---------------------------------------------------------------------------
PROBES = [
    dict(seed=11, T=40, lengths=[10, 0, 30], h_in=64, h_out=48, ranks=[4, 8]),
    dict(seed=12, T=300, lengths=[128, 1, 0, 171], h_in=512, h_out=256, ranks=[16, 2, 32], none_fraction=0.2),
    dict(seed=13, T=260, lengths=[130, 130], h_in=4096, h_out=1024, ranks=[16, 128]),
]


def _exact(a):
    return np.array_equal(np.asarray(a, np.float64), np.round(np.asarray(a, np.float64)))


@pytest.mark.parametrize("dtype", [I.BF16, I.F32])
@pytest.mark.parametrize("case", PROBES, ids=lambda c: f"seed{c['seed']}")
def test_integer_probe_bitexact(case, dtype):
    w = I.integer_probe(dtype=dtype, **case)
    v, y, y0, word = run_sgmv(w)
    assert word == 0
    vr, _ = oracle_v(w, 0, w.max_rank)
    mask = written_mask(w, w.max_rank)
    assert _exact(vr[mask]) and np.array_equal(v[mask], vr[mask])
    yr, _ = oracle_delta(w, 0, y0)
    assert _exact(yr) and np.max(np.abs(yr)) <= 256
    assert np.array_equal(y, yr)
    yl, Wh, word = run_layer(w)
    assert word == 0
    ylr, _ = oracle_delta(w, 0, None, W=Wh)
    assert _exact(ylr) and np.max(np.abs(ylr)) <= 256
    assert np.array_equal(yl, ylr)
    wd = I.integer_probe(dtype=dtype, **case)
    wd.token_adapter = np.repeat(wd.seg_adapter, np.diff(wd.seg_starts)).astype(np.int32)
    yb, y0b, word = run_bgmv(wd)
    assert word == 0
    assert np.array_equal(yb, yr)


# ---------------------------------------------------------------------------
# Edge cases and faults (host-made; nothing traps)
# ---------------------------------------------------------------------------
def test_invalid_ids_are_flagged_and_skipped():
    w = I.random_case(21, T=64, lengths=[16, 16, 16, 16], n_adapters=3, ranks=[4, 8, 4])
    w.seg_adapter = np.array([0, 5, 1, 2], np.int32)       # 5 >= max_adapters
    with H.DevicePool(w, load_ids=[0, 1]) as dp:             # 2 is not loaded
        ss, sa = _tables(w)
        x = H.to_device(w.x(), w.dtype)
        y0 = w.y0()
        y = H.to_device(y0, w.dtype)
        v = torch.zeros((w.T, w.max_rank), dtype=torch.float32, device="cuda")
        L.lora_sgmv_shrink(dp.handle, 0, x, v, w.max_rank, ss, sa, w.S, w.T)
        L.lora_sgmv_expand(dp.handle, 0, v, w.max_rank, y, ss, sa, w.S, w.T)
        rc, word = L.lora_get_error(dp.handle)
        assert rc == L.LORA_ERR_DEVICE_INDEX and word == L.LORA_DEV_BAD_ADAPTER
        assert L.lora_get_error(dp.handle) == (L.LORA_OK, 0)     # cleared
        yh = H.to_host(y)
        assert np.array_equal(yh[16:32], y0[16:32]) and np.array_equal(yh[48:64], y0[48:64])
        yr, st = oracle_delta(w, 0, y0, ids=[0, 1])
        assert st == oracle.ERR_ADAPTER
        assert rel_err(yh, yr) <= TOL_Y[w.dtype]


def test_bad_segment_table_is_flagged():
    w = I.random_case(22, T=32, lengths=[16, 16], n_adapters=2, ranks=[4, 4])
    with H.DevicePool(w) as dp:
        x = H.to_device(w.x(), w.dtype)
        v = torch.zeros((w.T, w.max_rank), dtype=torch.float32, device="cuda")
        for bad in ([0, 20, 16], [1, 16, 32], [0, 16, 31]):
            ss = H.int_tensor(bad)
            sa = H.int_tensor(w.seg_adapter)
            L.lora_sgmv_shrink(dp.handle, 0, x, v, w.max_rank, ss, sa, 2, 32)
            rc, word = L.lora_get_error(dp.handle)
            assert rc == L.LORA_ERR_DEVICE_INDEX and word & L.LORA_DEV_BAD_SEGMENTS


def test_zero_tokens_and_host_errors():
    w = I.random_case(23, T=16, lengths=[16], n_adapters=1, ranks=[4])
    with H.DevicePool(w) as dp:
        x = H.to_device(w.x(), w.dtype)
        y = H.to_device(w.y0(), w.dtype)
        v = torch.zeros((16, w.max_rank), dtype=torch.float32, device="cuda")
        ss, sa = _tables(w)
        n0 = L.lora_launch_count()
        L.lora_sgmv_shrink(dp.handle, 0, x, v, w.max_rank, ss, sa, 1, 0)
        L.lora_bgmv(dp.handle, 0, x, y, sa, 0)
        assert L.lora_launch_count() == n0
        with pytest.raises(L.LoraError) as e:
            L.lora_sgmv_shrink(dp.handle, 0, x, v, w.max_rank - 1, ss, sa, 1, 16)
        assert e.value.status == L.LORA_ERR_RANK
        with pytest.raises(L.LoraError) as e:
            L.lora_sgmv_shrink(dp.handle, 3, x, v, w.max_rank, ss, sa, 1, 16)
        assert e.value.status == L.LORA_ERR_ARG
        with pytest.raises(L.LoraError) as e:
            L.lora_bgmv(dp.handle, 0, None, y, sa, 16)
        assert e.value.status == L.LORA_ERR_ARG


def test_pool_lifecycle():
    h_in = h_out = 256
    pool = L.lora_pool_create(L.LORA_BF16, 256, 40, 16, 2, 4)
    try:
        rng = np.random.default_rng(0)

        def arr(r, h):
            return I.bf16_bits(I.round_to_bf16(rng.normal(size=(r, h)).astype(np.float32)))

        assert L.lora_pool_free_pages(pool) == 40
        L.lora_pool_load(pool, 0, 0, 8, 1.0, h_in, h_out, arr(8, h_in), arr(8, h_out))
        assert L.lora_pool_free_pages(pool) == 24
        L.lora_pool_load(pool, 1, 1, 0, 1.0, h_in, h_out, None, None)            # rank 0
        assert L.lora_pool_free_pages(pool) == 24
        with pytest.raises(L.LoraError) as e:
            L.lora_pool_load(pool, 2, 0, 16, 1.0, h_in, h_out, arr(16, h_in), arr(16, h_out))
        assert e.value.status == L.LORA_ERR_POOL_FULL
        assert L.lora_pool_free_pages(pool) == 24
        with pytest.raises(L.LoraError) as e:
            L.lora_pool_load(pool, 2, 0, 17, 1.0, h_in, h_out, arr(17, h_in), arr(17, h_out))
        assert e.value.status == L.LORA_ERR_RANK
        with pytest.raises(L.LoraError) as e:
            L.lora_pool_load(pool, 2, 0, 4, 1.0, 128, h_out, arr(4, 128), arr(4, h_out))
        assert e.value.status == L.LORA_ERR_SHAPE
        with pytest.raises(L.LoraError) as e:
            L.lora_pool_unload(pool, 3, 0)
        assert e.value.status == L.LORA_ERR_NOT_LOADED
        L.lora_pool_load(pool, 0, 0, 4, 1.0, h_in, h_out, arr(4, h_in), arr(4, h_out))   # replace
        assert L.lora_pool_free_pages(pool) == 32
        L.lora_pool_unload(pool, 0, 0)
        assert L.lora_pool_free_pages(pool) == 40
        L.lora_pool_load(pool, 2, 0, 16, 1.0, h_in, h_out, arr(16, h_in), arr(16, h_out))
        assert L.lora_pool_free_pages(pool) == 8
    finally:
        L.lora_pool_destroy(pool)


def test_reloaded_pages_serve_the_new_adapter():
    """Unload + load reuses pages; results follow the newly loaded weights."""
    w = I.random_case(24, T=50, lengths=[25, 25], n_adapters=2, ranks=[8, 8])
    with H.DevicePool(w, spare_pages=0) as dp:
        L.lora_pool_unload(dp.handle, 1, 0)
        w2 = I.random_case(25, T=50, lengths=[25, 25], n_adapters=2, ranks=[8, 8])
        at, b = w2.adapter(1)
        L.lora_pool_load(dp.handle, 1, 0, 8, float(w.scales[1]), 256, 256, H.host_array(at, w.dtype),
                         H.host_array(b, w.dtype))
        ss, sa = _tables(w)
        x = H.to_device(w.x(), w.dtype)
        y = H.to_device(np.zeros((50, 256), np.float32), w.dtype)
        v = torch.zeros((50, w.max_rank), dtype=torch.float32, device="cuda")
        L.lora_sgmv_shrink(dp.handle, 0, x, v, w.max_rank, ss, sa, w.S, w.T)
        L.lora_sgmv_expand(dp.handle, 0, v, w.max_rank, y, ss, sa, w.S, w.T)
        assert dp.check_device_status() == 0
        a0 = w.adapter(0)
        ad = oracle.Adapters(2, {0: (8, float(w.scales[0]), *a0), 1: (8, float(w.scales[1]), at, b)})
        from tests.parity import token_ids
        yr, st = oracle.layer(w.x(), None, token_ids(w), ad, 256)
        assert st == 0 and rel_err(H.to_host(y), yr) <= TOL_Y[w.dtype]


def test_bgmv_zipf_decode_hot_rank128_adapter():
    """The fused-layer workload's 512 decode tokens alone: Zipf(1.0) ids over
    128 adapters, adapter 0 (the hottest) at rank 128 -- many tokens per
    adapter and ranks above one chunk."""
    import dataclasses
    w = I.fused_layer()
    ids = w.seg_adapter[4:].copy()
    wd = dataclasses.replace(w, T=512, seg_starts=np.arange(513, dtype=np.int32), seg_adapter=ids,
                             token_adapter=ids.copy())
    assert (ids == 0).sum() > 16
    for m in (0, 1):
        check_bgmv(wd, m)


def test_bgmv_all_tokens_one_adapter_and_none():
    w = I.random_case(31, T=200, decode=True, n_adapters=3, ranks=[32, 8, 16], h_in=512, h_out=512)
    w.token_adapter[:] = 1
    w.token_adapter[::7] = -1
    w.seg_adapter = w.token_adapter.copy()
    check_bgmv(w)


# ---------------------------------------------------------------------------
# Determinism: every reduction order is fixed (K splits of the tensor-core
# shrink are added in split order, warp partials in warp order), so repeated
# calls on the same inputs give the same bits.
# ---------------------------------------------------------------------------
def test_repeated_calls_are_bit_identical():
    # uniform 128-row tiles of a rank-128 and a rank-16 adapter (tensor-core shrink and
    # GEMM-fused term), one-token segments (plan work list), a long rank-96 segment
    w = I.random_case(41, T=700, lengths=[256, 128, 1, 1, 1, 313], h_in=1024, h_out=512, ranks=[128, 16, 96])
    ys = [run_layer(w)[0] for _ in range(2)]
    assert not np.isnan(ys[0]).any() and np.array_equal(ys[0], ys[1])
    vs = [run_sgmv(w)[0] for _ in range(2)]
    mask = written_mask(w, w.max_rank)
    assert np.array_equal(vs[0][mask], vs[1][mask])


def test_fused_layer_bit_identical_across_calls_and_streams():
    """The full fused workload (4608 tokens, decode rows of the rank-128
    adapter among them): repeated calls on workspaces filled with different
    bytes, and the four projections issued at once on four streams with their
    own workspaces, give bit-identical outputs.  Token order inside an
    adapter's list follows per-segment atomics, so this also checks that no
    row's rounding depends on which work item it lands in."""
    w = I.fused_layer()
    with H.DevicePool(w) as dp:
        ss, sa = _tables(w)
        xs = {0: H.to_device(w.x(0), w.dtype), 3: H.to_device(w.x(3), w.dtype)}
        Ws = [H.to_device(w.W(m), w.dtype) for m in range(4)]
        ws_bytes = max(L.lora_layer_forward_workspace_size(dp.handle, m, w.S, w.T) for m in range(4))

        def call(m, y, fill, stream=None, ws=None):
            if ws is None:
                ws = torch.full((ws_bytes,), fill, dtype=torch.uint8, device="cuda")
            L.lora_layer_forward(dp.handle, m, xs[0 if m < 3 else 3], Ws[m], y, ss, sa, w.S, w.T, ws, stream=stream)
            return ws

        def new_y(m):
            return torch.full((w.T, w.matrices[m].h_out), float("nan"), dtype=torch.bfloat16, device="cuda")

        ref = []
        for m in range(4):
            y = new_y(m)
            call(m, y, 0)
            torch.cuda.synchronize()
            ref.append(y.clone())
        assert not any(torch.isnan(y).any().item() for y in ref)
        for fill in (0xff, 0x3c):
            for m in (0, 3):
                y = new_y(m)
                call(m, y, fill)
                torch.cuda.synchronize()
                assert torch.equal(y, ref[m]), (fill, m)
        streams = [torch.cuda.Stream() for _ in range(4)]
        ys = [new_y(m) for m in range(4)]
        # every buffer is filled before the event the four streams wait on
        wss = [torch.full((ws_bytes,), 0x7f, dtype=torch.uint8, device="cuda") for _ in range(4)]
        start = torch.cuda.Event()
        start.record()
        for m in range(4):
            streams[m].wait_event(start)
            call(m, ys[m], None, streams[m], wss[m])
        torch.cuda.synchronize()
        for m in range(4):
            assert torch.equal(ys[m], ref[m]), m
        assert dp.check_device_status() == 0


def test_sgmv_projections_on_concurrent_streams_match_sequential():
    """The prefill workload's four projections (shrink + expand each), issued
    at once on four streams with a v buffer each, give bit for bit what the
    same calls give one after another on one stream: the calls share only
    read-only state (pool, segment table)."""
    w = I.prefill_sgmv()
    with H.DevicePool(w) as dp:
        ss, sa = _tables(w)
        xs = {0: H.to_device(w.x(0), w.dtype), 3: H.to_device(w.x(3), w.dtype)}
        y0 = [H.to_device(w.y0(m), w.dtype) for m in range(4)]

        def run(m, y, v, stream=None):
            L.lora_sgmv_shrink(dp.handle, m, xs[0 if m < 3 else 3], v, w.max_rank, ss, sa, w.S, w.T, stream=stream)
            L.lora_sgmv_expand(dp.handle, m, v, w.max_rank, y, ss, sa, w.S, w.T, stream=stream)

        vs = [torch.zeros((w.T, w.max_rank), dtype=torch.float32, device="cuda") for _ in range(4)]
        ref = [y.clone() for y in y0]
        for m in range(4):
            run(m, ref[m], vs[m])
        torch.cuda.synchronize()
        ys = [y.clone() for y in y0]
        vs2 = [torch.full((w.T, w.max_rank), float("nan"), dtype=torch.float32, device="cuda") for _ in range(4)]
        streams = [torch.cuda.Stream() for _ in range(4)]
        start = torch.cuda.Event()
        start.record()
        for m in range(4):
            streams[m].wait_event(start)
            run(m, ys[m], vs2[m], streams[m])
        torch.cuda.synchronize()
        for m in range(4):
            assert torch.equal(ys[m], ref[m]), m
        assert dp.check_device_status() == 0


def test_layer_in_cuda_graph_on_side_stream_matches_eager():
    # The layer call forks part of its work onto an internal stream and joins it back:
    # captured into a CUDA graph on a non-default stream and replayed, it must give
    # exactly what the eager call gives (and the oracle's answer), and it must leave
    # nothing unjoined (capture would fail).
    w = I.random_case(43, T=700, lengths=[256, 128, 1, 1, 1, 313], h_in=1024, h_out=512, ranks=[128, 16, 96])
    with H.DevicePool(w, matrices=[0]) as dp:
        ss, sa = _tables(w)
        x = H.to_device(w.x(0), w.dtype)
        Wh = w.W(0)
        Wd = H.to_device(Wh, w.dtype)
        ws = torch.empty(L.lora_layer_forward_workspace_size(dp.handle, 0, w.S, w.T), dtype=torch.uint8,
                         device="cuda")
        y_eager = torch.full((w.T, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        L.lora_layer_forward(dp.handle, 0, x, Wd, y_eager, ss, sa, w.S, w.T, ws)
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        y_graph = torch.full((w.T, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                L.lora_layer_forward(dp.handle, 0, x, Wd, y_graph, ss, sa, w.S, w.T, ws,
                                     stream=torch.cuda.current_stream())
        for _ in range(2):
            y_graph.fill_(float("nan"))
            g.replay()
        torch.cuda.synchronize()
        word = dp.check_device_status()
    ye, yg = H.to_host(y_eager), H.to_host(y_graph)
    assert word == 0
    assert not np.isnan(yg).any() and np.array_equal(ye, yg)
    yr, st = oracle_delta(w, 0, None, W=Wh)
    assert st == 0 and rel_err(yg, yr) <= TOL_Y[w.dtype]


def test_layer_more_items_than_plan_threads():
    # 2600 one-token segments over 1500 adapters of mixed rank: over 1024 items and
    # over 1024 work items, so every plan loop and scan runs more than one round
    ranks = np.tile(np.array([4, 16, 32, 64, 8], np.int32), 300)
    w = I.random_case(51, T=2600, decode=True, ranks=ranks, h_in=256, h_out=256)
    y, Wh, word = run_layer(w)
    assert word == 0
    yr, st = oracle_delta(w, 0, None, W=Wh)
    assert st == 0 and rel_err(y, yr) <= TOL_Y[w.dtype]


def test_layer_one_segment_every_tile_fused():
    # one 1000-token segment of one rank-64 adapter: every M-tile, the ragged last one too,
    # is fused into the GEMM (two rounds each), the plan's tile flags are read from global
    # memory (more tiles than its shared staging holds), and no row is left for the unit
    # kernels (empty work list)
    w = I.random_case(52, T=1000, lengths=[1000], n_adapters=1, ranks=[64], h_in=512, h_out=256)
    y, Wh, word = run_layer(w)
    assert word == 0
    yr, st = oracle_delta(w, 0, None, W=Wh)
    assert st == 0 and rel_err(y, yr) <= TOL_Y[w.dtype]


# ---------------------------------------------------------------------------
# Rank-0 and zero-B adapters.  Their merged weight is W itself (S-LoRA slide 5,
# W' = W + AB with AB = 0), so their rows must come out as the base product
# (layer) or as y0 (SGMV, BGMV), bit for bit, while the other rows of the same
# batch still match the oracle.  The batch gives the rank-0 adapter two whole
# 128-row M-tiles and the zero-B adapter one (the GEMM's tile flags and its
# fused adapter rounds see them), plus one-token segments of both mixed with
# ordinary adapters (the plan's work units and the expand).
# ---------------------------------------------------------------------------
_DEGEN_RANKS = [16, 0, 128, 16, 8]      # adapter 1: rank 0; adapter 3: B = 0
_DEGEN_ZERO_B = (3,)
_DEGEN_IDS = (1, 3, 2)                  # the three whole tiles


def _degenerate_case(seed, dtype=I.BF16, decode=False):
    ragged = [37, 1, 1, 1, 90, 1, 1, 0, 64, 1, 1, 1, 13, 1, 1, 200, 1, 1, 1, 1]
    ragged_ids = [1, 3, 0, 4, 2, -1, 1, 3, 3, 1, 0, 2, 4, 3, 1, 1, 2, 3, 0, 1]
    lengths = [256, 128, 128] + ragged
    T = int(sum(lengths))
    w = I.random_case(seed, T=T, lengths=lengths, h_in=512, h_out=256, ranks=_DEGEN_RANKS, dtype=dtype)
    w.seg_adapter = np.array(list(_DEGEN_IDS) + ragged_ids, np.int32)
    w.zero_b = _DEGEN_ZERO_B
    if decode:
        tok = np.repeat(w.seg_adapter, np.diff(w.seg_starts)).astype(np.int32)
        w.seg_starts = np.arange(T + 1, dtype=np.int32)
        w.seg_adapter = tok.copy()
        w.token_adapter = tok
    return w


def _degenerate_rows(w):
    tok = np.repeat(w.seg_adapter, np.diff(w.seg_starts))
    keep = (tok == 1) | (tok == 3) | (tok < 0)
    assert keep.sum() > 384 and (~keep).sum() > 200
    return keep


@pytest.mark.parametrize("dtype", [I.BF16, I.F32])
def test_rank0_and_zero_b_sgmv(dtype):
    w = _degenerate_case(61, dtype)
    keep = _degenerate_rows(w)
    v, y, y0, word = run_sgmv(w)
    assert word == 0
    yh0 = H.to_host(H.to_device(y0, w.dtype))
    assert np.array_equal(y[keep], yh0[keep])
    yr, st = oracle_delta(w, 0, y0)
    assert st == 0 and rel_err(y, yr) <= TOL_Y[w.dtype]
    vr, _ = oracle_v(w, 0, w.max_rank)
    mask = written_mask(w, w.max_rank)
    assert rel_err(v[mask], vr[mask]) <= TOL_V[w.dtype]


@pytest.mark.parametrize("dtype", [I.BF16, I.F32])
def test_rank0_and_zero_b_bgmv(dtype):
    w = _degenerate_case(62, dtype, decode=True)
    keep = _degenerate_rows(w)
    y, y0, word = run_bgmv(w)
    assert word == 0
    yh0 = H.to_host(H.to_device(y0, w.dtype))
    assert np.array_equal(y[keep], yh0[keep])
    yr, st = oracle_delta(w, 0, y0)
    assert st == 0 and rel_err(y, yr) <= TOL_Y[w.dtype]


@pytest.mark.parametrize("dtype", [I.BF16, I.F32])
def test_rank0_and_zero_b_layer(dtype):
    w = _degenerate_case(63, dtype)
    keep = _degenerate_rows(w)
    y, Wh, word = run_layer(w)
    assert word == 0 and not np.isnan(y).any()
    yr, st = oracle_delta(w, 0, None, W=Wh)
    assert st == 0 and rel_err(y, yr) <= TOL_Y[w.dtype]
    # the same batch with no adapter at all: the base product alone
    import dataclasses
    wb = dataclasses.replace(w, seg_adapter=np.full_like(w.seg_adapter, -1))
    y_base, _, word = run_layer(wb)
    assert word == 0
    assert np.array_equal(y[keep], y_base[keep])
    # delta alone (W = 0): those rows are exactly zero
    yd, _, word = run_layer(w, zero_w=True)
    assert word == 0
    assert np.array_equal(yd[keep], np.zeros_like(yd[keep]))
    ydr, _ = oracle_delta(w, 0, None)
    assert rel_err(yd, ydr) <= TOL_Y[w.dtype]


def test_rank0_and_zero_b_decode_layer():
    """One-token segments only: every row goes through the plan's units."""
    w = _degenerate_case(64, I.BF16, decode=True)
    keep = _degenerate_rows(w)
    yd, _, word = run_layer(w, zero_w=True)
    assert word == 0
    assert np.array_equal(yd[keep], np.zeros_like(yd[keep]))
    ydr, st = oracle_delta(w, 0, None)
    assert st == 0 and rel_err(yd, ydr) <= TOL_Y[w.dtype]


# ---------------------------------------------------------------------------
# BGMV launch modes.  The grid follows the batch: a pool whose adapter-id range
# is large next to the batch runs the compacted mode (persistent clusters over
# the items of the adapters present); batches above the clustered kernels'
# limit run on the per-token kernel.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("T", [256, 2048])      # compacted mode; its largest batch
def test_bgmv_2048_adapter_pool(T):
    ranks = np.tile(np.array([16, 8, 32, 16], np.int32), 512)             # 2048 adapters
    w = I.random_case(111, T=T, decode=True, ranks=ranks, h_in=1024, h_out=1024)
    used = set(w.used_adapters().tolist())
    assert len(used) > 200
    with H.DevicePool(w, matrices=[0], filler=lambda a: a not in used) as dp:
        tok = H.int_tensor(w.token_adapter)
        x = H.to_device(w.x(0), w.dtype)
        y0 = w.y0(0)
        y = H.to_device(y0, w.dtype)
        L.lora_bgmv(dp.handle, 0, x, y, tok, w.T)
        word = dp.check_device_status()
    assert word == 0
    yr, st = oracle_delta(w, 0, y0)
    assert st == 0 and rel_err(H.to_host(y), yr) <= TOL_Y[w.dtype]


@pytest.mark.parametrize("n_adapters", [40, 600])
def test_bgmv_batch_above_the_clustered_limit(n_adapters):
    ranks = np.tile(np.array([16, 64, 8, 0, 32], np.int32), n_adapters // 5)
    w = I.random_case(112 + n_adapters, T=5000, decode=True, ranks=ranks, h_in=512, h_out=256)
    w.token_adapter[::13] = -1
    w.seg_adapter = w.token_adapter.copy()
    check_bgmv(w)


@pytest.mark.parametrize("dtype", [I.BF16])
def test_bgmv_compacted_integer_probe_bitexact(dtype):
    ranks = np.tile(np.array([4, 8, 16, 2], np.int32), 50)               # 200 ids for 64 tokens
    w = I.integer_probe(seed=113, T=64, lengths=[1] * 64, h_in=256, h_out=128, ranks=ranks, dtype=dtype)
    w.token_adapter = np.repeat(w.seg_adapter, np.diff(w.seg_starts)).astype(np.int32)
    y, y0, word = run_bgmv(w)
    assert word == 0
    yr, _ = oracle_delta(w, 0, y0)
    assert _exact(yr) and np.array_equal(y, yr)
