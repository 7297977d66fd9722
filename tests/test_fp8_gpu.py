"""FP8 base product (GPU): the row quantiser bit for bit against the oracle's,
and lora_layer_forward_fp8 (e4m3 base on the tensor cores, bf16 adapters)
against the oracle: the FP8 base of oracle/fp8.py plus the bf16 low-rank term
of the plain oracle, within the bf16 output tolerance.

Source: "Multi-LoRA Serving - S-LoRA/Punica Batching, Adapter Hot-Swap &
Memory", failure assumptions and "Operating it" (FP8 base, bf16 adapters).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

import oracle  # noqa: E402
from oracle import fp8 as F  # noqa: E402
from segmented_gathered_rank_gb300 import harness as H  # noqa: E402
from segmented_gathered_rank_gb300 import inputs as I  # noqa: E402
from segmented_gathered_rank_gb300 import lora as L  # noqa: E402
from tests.parity import TOL_Y, rel_err, token_ids  # noqa: E402


def _quantize_gpu(x_host, dtype=I.BF16):
    T, h = x_host.shape
    x = H.to_device(x_host, dtype)
    q = torch.empty((T, h), dtype=torch.uint8, device="cuda")
    sx = torch.empty(T, dtype=torch.float32, device="cuda")
    L.lora_quantize_e4m3(x, T, h, q, sx)
    torch.cuda.synchronize()
    return q.cpu().numpy(), sx.cpu().numpy()


def test_quantizer_bit_exact():
    rng = np.random.default_rng(91)
    x = rng.normal(0, 1, (40, 512)).astype(np.float32)
    x[3] = 0.0                                                  # a row of zeros
    x[5] *= 1e-6                                                # small, large and spiky rows
    x[7] *= 3e3
    x[9, 17] = 80.0
    x[11] = x[11] * 2.0 ** -125                                  # largest magnitude below 2^-120: zero codes
    x[13] = x[13] / np.max(np.abs(x[13])) * 2.0 ** -119          # just above: 448 / a stays finite
    x = I.round_to_bf16(x)
    q, sx = _quantize_gpu(x)
    q_ref, sx_ref = F.quantize_rows(x)
    assert np.array_equal(sx, sx_ref)
    assert np.array_equal(q, q_ref)


def _run_fp8(w, m=0, zero_w=False):
    with H.DevicePool(w, matrices=[m]) as dp:
        mat = w.matrices[m]
        ss, sa = H.int_tensor(w.seg_starts), H.int_tensor(w.seg_adapter)
        x = H.to_device(w.x(m), w.dtype)
        codes, s_w = w.W_e4m3(m)
        if zero_w:
            codes = np.zeros_like(codes)
        W8 = torch.from_numpy(codes).cuda()
        y = torch.full((w.T, mat.h_out), float("nan"), dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(L.lora_layer_forward_fp8_workspace_size(dp.handle, 0, w.S, w.T), dtype=torch.uint8,
                         device="cuda")
        L.lora_layer_forward_fp8(dp.handle, 0, x, W8, s_w, y, ss, sa, w.S, w.T, ws)
        word = dp.check_device_status()
        return H.to_host(y), codes, s_w, word


def _oracle_fp8(w, m, codes, s_w, rows=None):
    x = w.x(m)
    q, sx = F.quantize_rows(x)
    base = F.base(q, sx, codes, s_w, rows=rows)
    tok = token_ids(w)
    ad = oracle.adapters_for(w, m)
    rr = np.arange(w.T, dtype=np.int32) if rows is None else np.asarray(rows, np.int32)
    delta, st = oracle.layer(x, None, tok, ad, w.matrices[m].h_out, rows=rr)
    assert st == 0
    return base + delta, delta


FP8_CASES = [
    dict(seed=92, T=700, lengths=[256, 128, 1, 1, 1, 313], h_in=1024, h_out=512, ranks=[128, 16, 96]),
    dict(seed=93, T=333, lengths=[200, 0, 5, 128], h_in=512, h_out=384, ranks=[16, 64, 8, 128]),
    dict(seed=94, T=300, h_in=256, h_out=256, none_fraction=0.3),
    dict(seed=95, T=129, lengths=[129], h_in=128, h_out=96, ranks=[32]),
]


@pytest.mark.parametrize("case", FP8_CASES, ids=lambda c: f"seed{c['seed']}")
def test_fp8_layer_matches_oracle(case):
    w = I.random_case(**case)
    y, codes, s_w, word = _run_fp8(w)
    assert word == 0 and not np.isnan(y).any()
    ref, _ = _oracle_fp8(w, 0, codes, s_w)
    assert rel_err(y, ref) <= TOL_Y[w.dtype]


@pytest.mark.parametrize("case", FP8_CASES[:2], ids=lambda c: f"seed{c['seed']}")
def test_fp8_layer_delta_alone(case):
    # W8 = 0: only the low-rank term remains, in fused tiles through the FP8
    # accumulator (divided by s_x s_w on the way in, multiplied on the way out)
    w = I.random_case(**case)
    y, codes, s_w, word = _run_fp8(w, zero_w=True)
    assert word == 0
    _, delta = _oracle_fp8(w, 0, codes, s_w)
    assert rel_err(y, delta) <= TOL_Y[w.dtype]


def test_fp8_fused_layer_k_every_row():
    """The fused workload's k projection (4096 -> 1024, 4608 rows) with an FP8 base."""
    w = I.fused_layer()
    y, codes, s_w, word = _run_fp8(w, 1)
    assert word == 0 and not np.isnan(y).any()
    ref, _ = _oracle_fp8(w, 1, codes, s_w)
    assert rel_err(y, ref) <= TOL_Y[w.dtype]


def test_fp8_shape_and_argument_errors():
    w = I.random_case(96, T=64, lengths=[64], h_in=192, h_out=256, ranks=[8])
    with H.DevicePool(w) as dp:
        x = H.to_device(w.x(), w.dtype)
        W8 = torch.zeros((256, 192), dtype=torch.uint8, device="cuda")
        y = torch.zeros((64, 256), dtype=torch.bfloat16, device="cuda")
        ss, sa = H.int_tensor(w.seg_starts), H.int_tensor(w.seg_adapter)
        ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
        with pytest.raises(L.LoraError) as e:                  # h_in not a multiple of 128
            L.lora_layer_forward_fp8(dp.handle, 0, x, W8, 1.0, y, ss, sa, 1, 64, ws)
        assert e.value.status == L.LORA_ERR_SHAPE
