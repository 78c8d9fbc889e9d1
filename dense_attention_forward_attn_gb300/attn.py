"""Python binding of the C ABI in include/attn_fwd.h (ctypes; marshalling only).

Every step of the attention forward runs in the CUDA library; this module
checks tensor dtypes/shapes, allocates outputs with PyTorch, passes raw
pointers and the current CUDA stream, and maps status codes to exceptions.
There is no fallback: if the library is missing or the device is not a
GB300, the call raises.
"""
from __future__ import annotations

import ctypes
import math
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = -1
ATTN_ERR_UNSUPPORTED = -2
ATTN_ERR_ARCH = -3
ATTN_ERR_CUDA = -4
ATTN_ERR_TOO_LARGE = -5
ATTN_FLAG_CAUSAL = 1
ATTN_FLAG_BSHD = 2
ATTN_FLAG_SOFT_EXP2 = 4           # forward: 4 of 16 P columns by polynomial exp2 (Chapter 9)
ATTN_FLAG_TEST_WITHHOLD = 0x100   # test hook: see include/attn_fwd.h


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class _Plan(ctypes.Structure):
    _fields_ = [("work_items", ctypes.c_int64), ("grid", ctypes.c_int), ("threads", ctypes.c_int),
                ("q_tiles", ctypes.c_int), ("kv_tiles", ctypes.c_int), ("kv_stages", ctypes.c_int),
                ("smem_bytes", ctypes.c_int), ("tmem_cols", ctypes.c_int)]


EXPORTS = ("attn_fwd", "attn_fwd_ex", "attn_fwd_ws", "attn_fwd_workspace", "attn_fwd_segment",
           "attn_fwd_host", "attn_fwd_host_workspace", "attn_fwd_host_chunking", "attn_bwd",
           "attn_bwd_noalloc", "attn_status_string", "attn_fwd_plan", "attn_fwd_work_item",
           "attn_fwd_schedule", "attn_device_status")


def lib_path() -> str:
    return _build.lib_path()


def _bind(lib):
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp]
    lib.attn_fwd.restype = i32
    lib.attn_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, vp]
    lib.attn_fwd_ex.restype = i32
    sz = ctypes.c_size_t
    lib.attn_fwd_ws.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, vp, sz, vp]
    lib.attn_fwd_ws.restype = i32
    lib.attn_fwd_workspace.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.POINTER(sz)]
    lib.attn_fwd_workspace.restype = i32
    ipp = ctypes.POINTER(i32)
    lib.attn_fwd_segment.argtypes = [i32, i32, i32, i64, i32, i32, ipp, ipp, ipp, ipp, ipp]
    lib.attn_fwd_segment.restype = i32
    lib.attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, vp, sz, vp]
    lib.attn_fwd_host.restype = i32
    lib.attn_fwd_host_workspace.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.POINTER(sz)]
    lib.attn_fwd_host_workspace.restype = i32
    lib.attn_fwd_host_chunking.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.POINTER(i64),
                                           ctypes.POINTER(i64)]
    lib.attn_fwd_host_chunking.restype = i32
    lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32,
                             i32, vp]
    lib.attn_bwd.restype = i32
    lib.attn_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                     f32, i32, vp]
    lib.attn_bwd_noalloc.restype = i32
    lib.attn_status_string.argtypes = [i32]
    lib.attn_status_string.restype = ctypes.c_char_p
    lib.attn_fwd_plan.argtypes = [i32, i32, i32, i32, i32, i32, i32, ctypes.POINTER(_Plan)]
    lib.attn_fwd_plan.restype = i32
    ip = ctypes.POINTER(i32)
    lib.attn_fwd_work_item.argtypes = [i64, i32, i32, i32, i32, i32, ip, ip, ip, ip]
    lib.attn_fwd_work_item.restype = i32
    lib.attn_fwd_schedule.argtypes = [i32, i32, i32, i64, i32]
    lib.attn_fwd_schedule.restype = i32
    lib.attn_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint), i32]
    lib.attn_device_status.restype = i32
    return lib


def library(path: str | None = None):
    """Load (once) the CUDA library; raises if it has not been built."""
    global _lib
    with _lock:
        if path is not None:
            return _bind(ctypes.CDLL(path))
        if _lib is None:
            p = lib_path()
            try:
                _lib = _bind(ctypes.CDLL(p))
            except OSError as e:
                raise RuntimeError(f"attention CUDA library not loadable at {p} ({e}); "
                                   "build it with dense_attention_forward_attn_gb300.build.build()") from e
    return _lib


def status_string(status: int) -> str:
    return library().attn_status_string(int(status)).decode()


def _flags(causal: bool, layout: str = "bhsd", soft_exp2: bool = False) -> int:
    if layout not in ("bhsd", "bshd"):
        raise ValueError("layout must be 'bhsd' ([B,H,S,D]) or 'bshd' ([B,S,H,D])")
    return ((ATTN_FLAG_CAUSAL if causal else 0) | (ATTN_FLAG_BSHD if layout == "bshd" else 0)
            | (ATTN_FLAG_SOFT_EXP2 if soft_exp2 else 0))


def plan(B: int, H: int, Sq: int, Sk: int, D: int = 128, num_sms: int = 0,
         causal: bool = False) -> dict:
    p = _Plan()
    rc = library().attn_fwd_plan(B, H, Sq, Sk, D, _flags(causal), num_sms, ctypes.byref(p))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_plan")
    return {f: getattr(p, f) for f, _ in _Plan._fields_}


def work_item(item: int, B: int, H: int, Sq: int, Sk: int | None = None, causal: bool = False):
    """(bh, first Q tile, KV tiles of Q tile 0, KV tiles of Q tile 1 or 0)."""
    bh, qt0, n0, n1 = (ctypes.c_int() for _ in range(4))
    rc = library().attn_fwd_work_item(item, B, H, Sq, Sq if Sk is None else Sk, _flags(causal),
                                      ctypes.byref(bh), ctypes.byref(qt0), ctypes.byref(n0),
                                      ctypes.byref(n1))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_work_item")
    return bh.value, qt0.value, n0.value, n1.value


def schedule(cta: int, rnd: int, grid: int, work_items: int, causal: bool = False) -> int:
    """Work item CTA `cta` runs in its rnd-th turn, -1 when it has none left."""
    return int(library().attn_fwd_schedule(cta, rnd, grid, work_items, _flags(causal)))


def segment(cta: int, rnd: int, grid: int, work_items: int, kv_tiles: int, causal: bool = False):
    """The turn `rnd` of CTA `cta` under attn_fwd_ws's schedule: None when the CTA has no more,
    else (item, first KV tile, KV tile count or -1 for the whole item, split slot or -1, part)."""
    out = [ctypes.c_int() for _ in range(5)]
    rc = library().attn_fwd_segment(cta, rnd, grid, work_items, kv_tiles, _flags(causal),
                                    *(ctypes.byref(x) for x in out))
    if rc < 0:
        raise AttnError(rc, "attn_fwd_segment")
    return tuple(x.value for x in out) if rc == 1 else None


def workspace_bytes(B: int, H: int, Sq: int, Sk: int, D: int = 128, causal: bool = False,
                    layout: str = "bhsd", soft_exp2: bool = False) -> int:
    """Workspace attn_fwd_ws needs for this problem on the current device (0: none)."""
    n = ctypes.c_size_t(0)
    rc = library().attn_fwd_workspace(B, H, Sq, Sk, D, _flags(causal, layout, soft_exp2),
                                      ctypes.byref(n))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_workspace")
    return int(n.value)


def workspace_for(q, k, causal: bool = False, layout: str = "bhsd", soft_exp2: bool = False):
    """A device workspace for fwd_into(..., workspace=...) with these q/k, or None if the call
    does not need one.  Allocated from PyTorch's caching allocator on q's device."""
    import torch
    B, H, Sq, Sk, D = _dims(q, k, layout)
    n = workspace_bytes(B, H, Sq, Sk, D, causal, layout, soft_exp2)
    return torch.empty(n, dtype=torch.uint8, device=q.device) if n else None


def host_chunking(B: int, H: int, Sq: int, Sk: int, num_sms: int, causal: bool = False,
                  layout: str = "bhsd"):
    """(units per chunk, chunks) of the host-buffer forward; units are heads ([B,H,S,D]) or
    batch entries ([B,S,H,D]); the last chunk takes the remainder."""
    per, n = ctypes.c_int64(), ctypes.c_int64()
    rc = library().attn_fwd_host_chunking(B, H, Sq, Sk, _flags(causal, layout), num_sms,
                                          ctypes.byref(per), ctypes.byref(n))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_host_chunking")
    return per.value, n.value


def device_status(clear: bool = False) -> int:
    w = ctypes.c_uint(0)
    rc = library().attn_device_status(ctypes.byref(w), 1 if clear else 0)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_device_status")
    return int(w.value)


def _check(t, name):
    import torch
    if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or t.dim() != 4:
        raise TypeError(f"{name} must be a 4-D torch.bfloat16 tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (row-major)")


def _dims(q, k, layout):
    """(B, H, Sq, Sk, D) from q and k in the given layout."""
    if layout == "bshd":
        B, Sq, H, D = q.shape
        return B, H, Sq, k.shape[1], D
    B, H, Sq, D = q.shape
    return B, H, Sq, k.shape[2], D


def fwd_into(q, k, v, o, lse=None, scale: float | None = None, stream=None,
             causal: bool = False, layout: str = "bhsd", soft_exp2: bool = False,
             workspace=None) -> None:
    """Device tensors only: write softmax(scale q k^T) v into `o` (and LSE into `lse`).

    layout "bhsd": q/o [B,H,Sq,D], k/v [B,H,Sk,D]; "bshd": q/o [B,Sq,H,D], k/v [B,Sk,H,D].
    lse is [B,H,Sq] either way.  soft_exp2: ATTN_FLAG_SOFT_EXP2 (off by default).
    workspace: None calls attn_fwd_ex (whole work items only); a uint8 CUDA tensor (from
    workspace_for) calls attn_fwd_ws, which evens out the persistent grid's last rounds.
    """
    import torch
    flags = _flags(causal, layout, soft_exp2)
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o")):
        _check(t, n)
    B, H, Sq, Sk, D = _dims(q, k, layout)
    kv_shape = (B, Sk, H, D) if layout == "bshd" else (B, H, Sk, D)
    if tuple(k.shape) != kv_shape or tuple(v.shape) != kv_shape or tuple(o.shape) != tuple(q.shape):
        raise ValueError("shape mismatch between q, k, v, o")
    if lse is not None and (lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, Sq)
                            or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous float32 tensor [B, H, Sq]")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    lse_ptr = lse.data_ptr() if lse is not None else None
    if workspace is None:
        rc = library().attn_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse_ptr,
                                   B, H, Sq, Sk, D, float(scale), flags, stream)
    else:
        if (not isinstance(workspace, torch.Tensor) or not workspace.is_cuda
                or workspace.device != q.device or not workspace.is_contiguous()):
            raise ValueError("workspace must be a contiguous CUDA tensor on q's device")
        rc = library().attn_fwd_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse_ptr,
                                   B, H, Sq, Sk, D, float(scale), flags, workspace.data_ptr(),
                                   workspace.numel() * workspace.element_size(), stream)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd")


def fwd(q, k, v, scale: float | None = None, return_lse: bool = True, causal: bool = False,
        layout: str = "bhsd", soft_exp2: bool = False):
    """Attention forward.  q [B,H,Sq,D], k/v [B,H,Sk,D] (or [B,S,H,D] with layout="bshd"),
    BF16 contiguous.  Returns (o in q's layout, lse [B,H,Sq] or None).

    CUDA tensors: runs on the current stream through attn_fwd_ws (with a workspace from
    PyTorch's caching allocator when the schedule needs one), returns (o, lse) on the device.
    CPU tensors: attn_fwd_host -- the library copies the inputs to the current
    CUDA device in chunks (pinned host memory, pinned here first if needed),
    overlapping the copies with the kernel, copies O and LSE back into pinned
    CPU tensors and this call returns them once they are complete.
    """
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n)
    B, H, Sq, Sk, D = _dims(q, k, layout)
    if not q.is_cuda:
        return _fwd_host(q, k, v, B, H, Sq, Sk, D, scale, return_lse, causal, layout, soft_exp2)
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device) if return_lse else None
    ws = workspace_for(q, k, causal, layout, soft_exp2)
    fwd_into(q, k, v, o, lse, scale, causal=causal, layout=layout, soft_exp2=soft_exp2,
             workspace=ws)   # None: the call has no split rounds, attn_fwd_ex
    return o, lse


_side_streams = {}


def _flop_per_byte(pb):
    """Tensor-core work per byte copied for one host-buffer problem: 4*Sq*Sk*D FLOP (half with
    the causal mask) over the BF16 Q, K, V in and O out."""
    try:
        B, H, Sq, Sk, D = _dims(pb["q"], pb["k"], pb.get("layout", "bhsd"))
    except (ValueError, TypeError, AttributeError, KeyError):
        return 0.0   # malformed; the enqueue reports it
    flop = 4.0 * Sq * Sk * D * (0.5 if pb.get("causal", False) else 1.0)
    return flop / max(1, 2 * D * (2 * Sq + 2 * Sk))


def batch_order(problems):
    """The order fwd_host_batch enqueues problems in by default: most tensor work per copied byte
    first (stable for ties)."""
    return sorted(range(len(problems)), key=lambda i: -_flop_per_byte(problems[i]))


def fwd_host_batch(problems, order=None):
    """Several host-buffer forwards at once: each problem is a dict with q, k, v (CPU BF16) and
    optional scale, causal, layout, soft_exp2, return_lse.  Each goes through attn_fwd_host on its
    own side stream (after the work already on the current stream); the library's copies run in the
    order the problems are enqueued, so by default the problems with the most tensor work per
    copied byte go first: their kernels then run while the copies of the others stream in,
    instead of after the last copy.  `order` (a permutation of range(len(problems))) overrides
    that.  Returns [(o, lse)] (pinned CPU tensors) in the problems' order, once all are
    complete."""
    import torch
    order = batch_order(problems) if order is None else list(order)
    if sorted(order) != list(range(len(problems))):
        raise ValueError("order must be a permutation of the problem indices")
    dev = torch.device("cuda", torch.cuda.current_device())
    cur = torch.cuda.current_stream(dev)
    streams = _side_streams.setdefault(dev.index, [])
    while len(streams) < len(problems):
        streams.append(torch.cuda.Stream(dev))
    pending = [None] * len(problems)
    for i, st in zip(order, streams):
        pb = problems[i]
        st.wait_stream(cur)
        with torch.cuda.stream(st):
            pending[i] = _fwd_host_enqueue(pb["q"], pb["k"], pb["v"], pb.get("scale"),
                                           pb.get("return_lse", True), pb.get("causal", False),
                                           pb.get("layout", "bhsd"), pb.get("soft_exp2", False))
    for st in streams[:len(problems)]:
        cur.wait_stream(st)
    cur.synchronize()
    return [(o, lse) for o, lse, _keep in pending]


def _fwd_host(q, k, v, B, H, Sq, Sk, D, scale, return_lse, causal, layout, soft_exp2=False):
    import torch
    o, lse, keep = _fwd_host_enqueue(q, k, v, scale, return_lse, causal, layout, soft_exp2)
    torch.cuda.current_stream().synchronize()
    del keep
    return o, lse


def _fwd_host_enqueue(q, k, v, scale, return_lse, causal, layout, soft_exp2=False):
    """Enqueue attn_fwd_host on the current stream; returns (o, lse, keep) -- keep (the device
    workspace and the pinned inputs) must stay referenced until the stream has finished the
    call, since the library's copies are not tracked by PyTorch's allocators."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n)
    B, H, Sq, Sk, D = _dims(q, k, layout)
    if k.is_cuda or v.is_cuda:
        raise ValueError("q, k, v must all be CPU tensors or all CUDA tensors")
    kv_shape = (B, Sk, H, D) if layout == "bshd" else (B, H, Sk, D)
    if tuple(k.shape) != kv_shape or tuple(v.shape) != kv_shape:
        raise ValueError("shape mismatch between q, k, v")
    flags = _flags(causal, layout, soft_exp2)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    q, k, v = (t if t.is_pinned() else t.pin_memory() for t in (q, k, v))
    lib = library()
    ws = ctypes.c_size_t()
    rc = lib.attn_fwd_host_workspace(B, H, Sq, Sk, D, flags, ctypes.byref(ws))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_host_workspace")
    dev = torch.device("cuda", torch.cuda.current_device())
    work = torch.empty(max(ws.value, 1), dtype=torch.uint8, device=dev)
    o = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=True)
    lse = torch.empty((B, H, Sq), dtype=torch.float32, pin_memory=True) if return_lse else None
    stream = torch.cuda.current_stream(dev)
    rc = lib.attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                           lse.data_ptr() if lse is not None else None, B, H, Sq, Sk, D,
                           float(scale), flags, work.data_ptr(), ws.value, stream.cuda_stream)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_host")
    return o, lse, (work, q, k, v)


def bwd(q, k, v, o, dout, lse, scale: float | None = None, causal: bool = False,
        layout: str = "bhsd"):
    """Backward of fwd (device tensors, BF16; layout "bhsd": q/o/dout [B,H,Sq,D], k/v [B,H,Sk,D];
    "bshd": [B,S,H,D]; lse [B,H,Sq] fp32 from fwd either way).

    Returns (dq, dk, dv), BF16 in the shapes of q, k, v.  Runs on the current stream.
    """
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dout, "dout")):
        _check(t, n)
    flags = _flags(causal, layout)
    B, H, Sq, Sk, D = _dims(q, k, layout)
    kv_shape = (B, Sk, H, D) if layout == "bshd" else (B, H, Sk, D)
    if tuple(v.shape) != kv_shape or tuple(k.shape) != kv_shape:
        raise ValueError("k and v must have the same shape")
    if tuple(o.shape) != tuple(q.shape) or tuple(dout.shape) != tuple(q.shape):
        raise ValueError("o and dout must have q's shape")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, Sq) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 tensor [B, H, Sq]")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    delta = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    stream = torch.cuda.current_stream(q.device).cuda_stream
    rc = library().attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
                            lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                            delta.data_ptr(), B, H, Sq, Sk, D, float(scale), flags, stream)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_bwd")
    return dq, dk, dv
