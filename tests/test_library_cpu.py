"""The C-ABI library without a GPU: it loads, exports what the header
declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

from segmented_gathered_rank_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ctypes.CDLL(build.LIB)


def _declared():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            with open(os.path.join(ROOT, "include", h)) as f:
                text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
            names |= set(re.findall(r"\b(lora_[a-z_0-9]+)\s*\(", text))
    return names


def test_header_declares_the_boundary():
    need = {"lora_pool_create", "lora_pool_destroy", "lora_pool_load", "lora_pool_unload", "lora_sgmv_shrink",
            "lora_sgmv_expand", "lora_bgmv", "lora_layer_forward", "lora_get_error", "lora_strerror"}
    assert need <= _declared()


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in sorted(_declared()) if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_names_match_header():
    from segmented_gathered_rank_gb300 import lora
    assert set(lora.EXPORTS) == _declared()
    for n in lora.EXPORTS:
        assert callable(getattr(lora, n))


def test_host_argument_checks(lib):
    from segmented_gathered_rank_gb300 import lora as L
    P = ctypes.c_void_p
    h = P()
    assert L._lib.lora_pool_create(None, 1, 4096, 8, 16, 1, 1) == L.LORA_ERR_ARG
    assert L._lib.lora_pool_create(ctypes.byref(h), 7, 4096, 8, 16, 1, 1) == L.LORA_ERR_ARG   # dtype
    assert L._lib.lora_pool_create(ctypes.byref(h), 1, 100, 8, 16, 1, 1) == L.LORA_ERR_ARG    # page % 8
    assert L._lib.lora_pool_create(ctypes.byref(h), 1, 4096, 0, 16, 1, 1) == L.LORA_ERR_ARG
    assert L._lib.lora_pool_create(ctypes.byref(h), 1, 4096, 8, 0, 1, 1) == L.LORA_ERR_ARG
    assert L._lib.lora_pool_create(ctypes.byref(h), 1, 4096, 8, 2048, 1, 1) == L.LORA_ERR_ARG
    assert h.value is None
    z = P(0)
    assert L._lib.lora_pool_load(None, 0, 0, 4, 1.0, 8, 8, None, None, z) == L.LORA_ERR_ARG
    assert L._lib.lora_sgmv_shrink(None, 0, None, None, 16, None, None, 1, 1, z) == L.LORA_ERR_ARG
    assert L._lib.lora_sgmv_expand(None, 0, None, 16, None, None, None, 1, 1, z) == L.LORA_ERR_ARG
    assert L._lib.lora_bgmv(None, 0, None, None, None, 1, z) == L.LORA_ERR_ARG
    assert L._lib.lora_layer_forward(None, 0, None, None, None, None, None, 1, 1, None, 0, z) == L.LORA_ERR_ARG
    assert L._lib.lora_layer_forward_workspace_size(None, 0, 1, 1) == 0
    assert L._lib.lora_pool_unload(None, 0, 0) == L.LORA_ERR_ARG
    assert L._lib.lora_pool_free_pages(None) == -1
    assert L._lib.lora_pool_destroy(None) == L.LORA_OK
    assert L.lora_get_error(None)[0] == L.LORA_ERR_ARG


def test_create_without_a_device_reports_cuda_error(lib):
    pytest.importorskip("torch")
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    from segmented_gathered_rank_gb300 import lora as L
    h = ctypes.c_void_p()
    assert L._lib.lora_pool_create(ctypes.byref(h), 1, 4096, 8, 16, 1, 1) == L.LORA_ERR_CUDA
    assert h.value is None


def test_strerror_covers_every_code(lib):
    from segmented_gathered_rank_gb300 import lora as L
    codes = [L.LORA_OK, L.LORA_ERR_ARG, L.LORA_ERR_POOL_FULL, L.LORA_ERR_RANK, L.LORA_ERR_NOT_LOADED,
             L.LORA_ERR_CUDA, L.LORA_ERR_DEVICE_INDEX, L.LORA_ERR_SHAPE]
    texts = [L.lora_strerror(c) for c in codes]
    assert len(set(texts)) == len(texts) and "unknown status" not in texts
    assert L.lora_strerror(12345) == "unknown status"


def test_async_upload_host_checks(lib):
    from segmented_gathered_rank_gb300 import lora as L
    z = ctypes.c_void_p(0)
    assert L._lib.lora_pool_load_async(None, 0, 0, 4, 1.0, 8, 8, None, None, z) == L.LORA_ERR_ARG
    assert L._lib.lora_pool_unload_async(None, 0, 0, z) == L.LORA_ERR_ARG
    assert L._lib.lora_pool_prefetch(None, None, 0, z) == L.LORA_ERR_ARG

