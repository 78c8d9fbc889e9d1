"""fp64 CPU oracle for the dense attention forward -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline / reference leg
of ``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls it, and the two share no
code: this package holds its own C source (``attn_oracle.c``), compiled with
gcc into ``oracle/_build/``.

Functions
---------
attn_fwd        plain definition, every row            (parity pinned)
attn_fwd_rows   plain definition, selected rows         (parity pinned: same C row routine)
attn_probs      materialised softmax of one head        (parity pinned)
attn_bwd        gradients dQ, dK, dV of the definition  (parity pinned)
online.*        the pages' tiled online-softmax steps   (parity pinned, see online.py)

What the plain definition is and where it comes from is stated in the header of
``attn_oracle.c``.  The pins are in ``tests/test_oracle.py``: the library
routine ``torch.nn.functional.scaled_dot_product_attention`` in float64,
brute force with exactly rounded sums (``math.fsum``) on tiny inputs, and closed
forms (constant V, one dominant key, zero scale, permutation and duplication of
the key/value rows).

Inputs are BF16 bit patterns (numpy ``uint16``) in ``[B, H, S, D]`` layout.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, f"liboracle_{platform.machine()}.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile attn_oracle.c with gcc (OpenMP, fp64, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, f64, i32 = ctypes.c_int64, ctypes.c_double, ctypes.c_int
            vp = ctypes.c_void_p
            lib.oracle_attn_fwd.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, f64, i32, vp, vp, i32]
            lib.oracle_attn_fwd.restype = i32
            lib.oracle_attn_fwd_rows.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, f64, i32,
                                                 vp, vp, i64, vp, vp, i32]
            lib.oracle_attn_fwd_rows.restype = i32
            lib.oracle_attn_probs.argtypes = [vp, vp, i64, i64, i64, f64, i32, vp]
            lib.oracle_attn_probs.restype = i32
            lib.oracle_attn_bwd.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, f64, i32,
                                            vp, vp, vp, i32]
            lib.oracle_attn_bwd.restype = i32
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = i32
            _lib = lib
    return _lib


def _bits(a) -> np.ndarray:
    """Accept a numpy uint16 array or a torch bfloat16 CPU tensor; return contiguous uint16."""
    if hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        import torch
        a = a.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected BF16 bit patterns (uint16), got {a.dtype}")
    return a


def max_threads() -> int:
    """Threads the OpenMP runtime of the oracle uses."""
    return int(_load().oracle_max_threads())


def attn_fwd(q, k, v, scale: float, nthreads: int = 0, causal: bool = False):
    """O [B,H,Sq,D] and LSE [B,H,Sq] in fp64 from BF16 q [B,H,Sq,D], k/v [B,H,Sk,D].

    causal: query i attends keys j <= i (top-left aligned)."""
    q, k, v = _bits(q), _bits(k), _bits(v)
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    if k.shape != (B, H, Sk, D) or v.shape != (B, H, Sk, D):
        raise ValueError("shape mismatch")
    o = np.empty((B, H, Sq, D), dtype=np.float64)
    lse = np.empty((B, H, Sq), dtype=np.float64)
    rc = _load().oracle_attn_fwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, B, H, Sq, Sk, D,
                                 float(scale), int(bool(causal)), o.ctypes.data, lse.ctypes.data,
                                 int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_fwd failed: {rc}")
    return o, lse


def attn_fwd_rows(q, k, v, scale: float, bh_idx, row_idx, nthreads: int = 0,
                  causal: bool = False):
    """Selected output rows: (O [n,D], LSE [n]) for flattened heads bh_idx and query rows row_idx."""
    q, k, v = _bits(q), _bits(k), _bits(v)
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    bh_idx = np.ascontiguousarray(bh_idx, dtype=np.int64)
    row_idx = np.ascontiguousarray(row_idx, dtype=np.int64)
    n = bh_idx.shape[0]
    if row_idx.shape[0] != n:
        raise ValueError("index length mismatch")
    o = np.empty((n, D), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    rc = _load().oracle_attn_fwd_rows(q.ctypes.data, k.ctypes.data, v.ctypes.data, B, H, Sq, Sk,
                                      D, float(scale), int(bool(causal)), bh_idx.ctypes.data,
                                      row_idx.ctypes.data, n,
                                      o.ctypes.data, lse.ctypes.data, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_fwd_rows failed: {rc}")
    return o, lse


def attn_probs(q_head, k_head, scale: float, causal: bool = False):
    """Materialised P = softmax(scale * q k^T) of one head, q [Sq,D], k [Sk,D]."""
    q, k = _bits(q_head), _bits(k_head)
    Sq, D = q.shape
    Sk = k.shape[0]
    p = np.empty((Sq, Sk), dtype=np.float64)
    rc = _load().oracle_attn_probs(q.ctypes.data, k.ctypes.data, Sq, Sk, D, float(scale),
                                   int(bool(causal)), p.ctypes.data)
    if rc != 0:
        raise RuntimeError(f"oracle_attn_probs failed: {rc}")
    return p


def attn_bwd(q, k, v, do, scale: float, causal: bool = False, nthreads: int = 0):
    """(dQ [B,H,Sq,D], dK [B,H,Sk,D], dV [B,H,Sk,D]) in fp64 for upstream gradient do = dL/dO."""
    q, k, v, do = _bits(q), _bits(k), _bits(v), _bits(do)
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    if k.shape != (B, H, Sk, D) or v.shape != (B, H, Sk, D) or do.shape != q.shape:
        raise ValueError("shape mismatch")
    dq = np.empty((B, H, Sq, D), dtype=np.float64)
    dk = np.empty((B, H, Sk, D), dtype=np.float64)
    dv = np.empty((B, H, Sk, D), dtype=np.float64)
    rc = _load().oracle_attn_bwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, do.ctypes.data, B, H,
                                 Sq, Sk, D, float(scale), int(bool(causal)), dq.ctypes.data,
                                 dk.ctypes.data, dv.ctypes.data, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_bwd failed: {rc}")
    return dq, dk, dv
