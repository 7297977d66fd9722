"""Host-side plumbing: put a generated workload into a device pool.

Moves data only (adapters into the paged pool through ``lora_pool_load``,
activations and tables into device tensors); all arithmetic runs in the CUDA
library.  Used by the tests, the benchmark and the smoke check.
"""
from __future__ import annotations

import numpy as np
import torch

from . import inputs as I
from . import lora as L


def torch_dtype(dtype: str):
    return torch.bfloat16 if dtype == I.BF16 else torch.float32


def host_array(a: np.ndarray, dtype: str) -> np.ndarray:
    """Host buffer in the pool's element type (bf16 as uint16 encodings)."""
    return I.bf16_bits(a) if dtype == I.BF16 else np.ascontiguousarray(a, np.float32)


def to_device(a: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """Exact device copy of bf16-representable (or fp32) values."""
    if dtype == I.BF16:
        bits = I.bf16_bits(a).view(np.int16)
        return torch.from_numpy(bits).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device)


def to_host(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def int_tensor(a, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(device)


class DevicePool:
    """A pool holding adapters of ``workload`` for the listed matrices.

    Pool matrix index ``layer * len(matrices) + i`` holds workload matrix
    ``matrices[i]`` of copy ``layer``.  ``load_ids`` defaults to every
    adapter of the workload.  Adapters for which ``filler(a)`` is true are
    loaded with zero weights of their own rank: they occupy their pages like
    any other adapter but skip drawing values no token reads.
    """

    def __init__(self, w: I.Workload, matrices=None, layers: int = 1, load_ids=None, spare_pages: int = 64,
                 stream=None, filler=None):
        self.w = w
        self.filler = filler
        self._zeros = {}
        self.matrices = list(range(len(w.matrices))) if matrices is None else list(matrices)
        self.layers = layers
        self.load_ids = np.arange(w.n_adapters) if load_ids is None else np.asarray(load_ids)
        per_matrix = int(2 * w.ranks[self.load_ids].sum())
        self.n_pages = per_matrix * len(self.matrices) * layers + spare_pages
        self.dtype_code = L.LORA_BF16 if w.dtype == I.BF16 else L.LORA_F32
        self.handle = L.lora_pool_create(self.dtype_code, w.page_elems, self.n_pages, w.max_rank,
                                         len(self.matrices) * layers, w.n_adapters)
        try:
            for layer in range(layers):
                for i, m in enumerate(self.matrices):
                    self.load_matrix(layer, i, m, stream)
            torch.cuda.synchronize()
        except Exception:
            self.close()
            raise

    def index(self, layer: int, i: int) -> int:
        return layer * len(self.matrices) + i

    def load_matrix(self, layer, i, m, stream=None):
        mat = self.w.matrices[m]
        for a in self.load_ids.tolist():
            if self.filler is not None and self.filler(a):
                r = int(self.w.ranks[a])
                key = (r, mat.h_in, mat.h_out)
                if key not in self._zeros:
                    self._zeros[key] = (np.zeros((r, mat.h_in), np.float32), np.zeros((r, mat.h_out), np.float32))
                at, b = self._zeros[key]
            else:
                at, b = self.w.adapter(a, m, layer)
            L.lora_pool_load(self.handle, a, self.index(layer, i), int(self.w.ranks[a]), float(self.w.scales[a]),
                             mat.h_in, mat.h_out, host_array(at, self.w.dtype), host_array(b, self.w.dtype),
                             stream=stream)

    def close(self):
        if getattr(self, "handle", None):
            L.lora_pool_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def check_device_status(self) -> int:
        rc, word = L.lora_get_error(self.handle)
        if rc not in (L.LORA_OK, L.LORA_ERR_DEVICE_INDEX):
            raise L.LoraError(rc, "lora_get_error")
        return word
