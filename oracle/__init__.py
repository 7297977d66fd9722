"""CPU oracle for the multi-LoRA mixed-batch adapter update.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The library under
``segmented_gathered_rank_gb300`` never imports this package, and this package
imports nothing from it.

The arithmetic lives in ``lora_oracle.c`` (plain C, double precision, loops
written from the definition on "Multi-LoRA Serving - S-LoRA/Punica Batching,
Adapter Hot-Swap & Memory", section "The kernel trick: gather, do not
merge").  This module compiles it with gcc and marshals numpy arrays into it.

Parity status of each function (what pins it is in ``tests/test_oracle.py``):
  token_adapters  pinned: brute-force segment cases, invalid-table cases
  shrink          pinned: numpy matrix product on small data, integer probes
  expand          pinned: numpy matrix product on small data, integer probes
  layer           pinned: the page's worked example (merged == gathered,
                  34 distinct adapters), merged-weight invariant, rank-0 /
                  zero-B base identity, segment permutation, pure-Python brute
                  force on tiny inputs, integer one-hot probes
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import numpy as np

_DIR = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_DIR, "lora_oracle.c")
LIB = os.path.join(_DIR, "liblora_oracle.so")

ERR_SEGMENTS = 1
ERR_ADAPTER = 2
ERR_RANK = 4

_lib = None


def build(force: bool = False, src: str = SRC, out: str = LIB) -> str:
    """Compile the oracle with gcc (OpenMP when available). Returns the .so path."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("no C compiler found to build the oracle")
    base = [cc, "-O2", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC", "-std=c11"]
    tmp = out + ".tmp"
    r = subprocess.run(base + ["-fopenmp", "-o", tmp, src], capture_output=True, text=True)
    if r.returncode != 0:
        r = subprocess.run(base + ["-o", tmp, src], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("oracle build failed:\n" + r.stderr)
    os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load (building if needed) the oracle library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _bind(lib):
    P = ctypes.c_void_p
    I = ctypes.c_int
    lib.orc_num_threads.restype = I
    lib.orc_token_adapters.argtypes = [I, P, P, I, P]
    lib.orc_shrink.argtypes = [I, I, P, P, I, P, P, P, I, P, I, P]
    lib.orc_expand.argtypes = [I, I, P, I, P, I, P, P, P, P, I, P, P]
    lib.orc_layer.argtypes = [I, I, I, P, P, P, I, P, P, P, P, P, P, I, P, P]
    for f in (lib.orc_token_adapters, lib.orc_shrink, lib.orc_expand, lib.orc_layer):
        f.restype = I
    return lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def num_threads(lib=None) -> int:
    return (lib or load()).orc_num_threads()


class Adapters:
    """Adapters packed in the oracle's dense layout.

    ``entries`` maps adapter id -> (rank, scale, A_T [rank x h_in],
    B [rank x h_out]).  Ids in ``0..n-1`` that are not given are marked not
    loaded (rank -1), so a token that names one is reported, never read.
    """

    def __init__(self, n: int, entries: dict):
        self.n = int(n)
        self.rank = np.full(max(self.n, 1), -1, np.int32)
        self.scale = np.zeros(max(self.n, 1), np.float64)
        self.at_off = np.zeros(max(self.n, 1), np.int64)
        self.b_off = np.zeros(max(self.n, 1), np.int64)
        at_parts, b_parts, at_pos, b_pos = [], [], 0, 0
        for a, (r, s, at, b) in sorted(entries.items()):
            at = _f64(at).reshape(int(r), -1) if r else np.zeros((0, 0))
            b = _f64(b).reshape(int(r), -1) if r else np.zeros((0, 0))
            self.rank[a] = int(r)
            self.scale[a] = float(s)
            self.at_off[a] = at_pos
            self.b_off[a] = b_pos
            at_parts.append(at.ravel())
            b_parts.append(b.ravel())
            at_pos += at.size
            b_pos += b.size
        self.AT = np.concatenate(at_parts + [np.zeros(1)])
        self.B = np.concatenate(b_parts + [np.zeros(1)])


def token_adapters(seg_starts, seg_adapter, T: int, lib=None):
    """(status, per-token adapter ids) from a segment table."""
    lib = lib or load()
    ss, sa = _i32(seg_starts), _i32(seg_adapter)
    out = np.full(max(T, 1), -7, np.int32)
    st = lib.orc_token_adapters(len(sa), _p(ss), _p(sa), int(T), _p(out))
    return st, out[:T]


def _rows(rows, T):
    return np.arange(T, dtype=np.int32) if rows is None else _i32(rows)


def shrink(x, token_adapter, ad: Adapters, ld_v: int, rows=None, lib=None):
    """(v [n_rows x ld_v] float64 (NaN where not written), status)."""
    lib = lib or load()
    x = _f64(x)
    T, h_in = x.shape
    rows = _rows(rows, T)
    v = np.full((len(rows), ld_v), np.nan)
    st = lib.orc_shrink(T, h_in, _p(x), _p(_i32(token_adapter)), ad.n, _p(ad.rank), _p(ad.AT),
                        _p(ad.at_off), len(rows), _p(rows), ld_v, _p(v))
    return v, st


def expand(v, token_adapter, ad: Adapters, y0, rows=None, T=None, lib=None):
    """(y = y0 + scale * v.B per row, status); y0 and v are given per listed row."""
    lib = lib or load()
    v = _f64(v)
    y = _f64(y0).copy()
    T = int(T if T is not None else len(token_adapter))
    rows = _rows(rows, T)
    st = lib.orc_expand(T, y.shape[1], _p(v), v.shape[1], _p(_i32(token_adapter)), ad.n, _p(ad.rank),
                        _p(ad.scale), _p(ad.B), _p(ad.b_off), len(rows), _p(rows), _p(y))
    return y, st


def layer(x, W, token_adapter, ad: Adapters, h_out: int, y0=None, rows=None, lib=None):
    """(y = y0 + x.W^T + scale * (x.A_T^T).B per listed row, status).

    ``W`` may be None (no base term); ``y0`` defaults to zeros.
    """
    lib = lib or load()
    x = _f64(x)
    T, h_in = x.shape
    rows = _rows(rows, T)
    y = np.zeros((len(rows), h_out)) if y0 is None else _f64(y0).copy()
    Wd = None if W is None else _f64(W)
    st = lib.orc_layer(T, h_in, h_out, _p(x), _p(Wd), _p(_i32(token_adapter)), ad.n, _p(ad.rank),
                       _p(ad.scale), _p(ad.AT), _p(ad.at_off), _p(ad.B), _p(ad.b_off),
                       len(rows), _p(rows), _p(y))
    return y, st


def adapters_for(workload, m: int = 0, ids=None, layer: int = 0) -> Adapters:
    """Pack the adapters ``ids`` (default: those the batch uses) of one matrix
    of a generated workload."""
    if ids is None:
        ids = workload.used_adapters()
    entries = {}
    for a in np.asarray(ids).tolist():
        at, b = workload.adapter(a, m, layer)
        entries[a] = (int(workload.ranks[a]), float(workload.scales[a]), at, b)
    return Adapters(workload.n_adapters, entries)
