"""ctypes binding of libringattn.so (include/ringattn.h).  Argument marshalling only: every step of
the computation runs in the library's CUDA kernels.  torch is used for device memory and streams.

The library is loaded on first use from this package's directory; if it has not been built the
call raises RingAttnError (there is no fallback of any kind).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libringattn.so")

RA_OK, RA_ERR_INVALID_ARG, RA_ERR_UNSUPPORTED, RA_ERR_CUDA, RA_ERR_NO_DEVICE, RA_ERR_TIMEOUT = range(6)
LAYOUTS = {"contiguous": 0, "zigzag": 1, "striped": 2}
PATHS = {1: "simt", 2: "tcgen05"}
RA_DEVICE_TIMEOUT = 1
RA_DEVICE_LAYOUT = 2

_lock = threading.Lock()
_lib = None

EXPORTS = (
    "ring_attn_fwd", "ring_attn_ring_step_fwd", "ring_attn_lse_merge", "ring_attn_fwd_stepwise",
    "ring_attn_fwd_stepwise_workspace_size", "ring_attn_bwd", "ring_attn_bwd_workspace_size",
    "ring_attn_shard_tiles", "ring_attn_fwd_path", "ring_attn_bwd_path", "ring_attn_device_status",
    "ring_attn_last_error", "ring_attn_abi_version", "ring_attn_bwd_static_scratch",
    "ring_attn_bwd_static_scratch_capacity", "ring_attn_fwd_tile_visits", "ring_attn_bwd_tile_visits",
    "ring_attn_rope", "ring_attn_ulysses_a2a", "ring_attn_ulysses_fwd", "ring_attn_ulysses_workspace_size",
    "ring_attn_ulysses_bwd", "ring_attn_ulysses_bwd_workspace_size", "ring_attn_fwd_host",
    "ring_attn_ring_step_fwd_accumulate",
    "ring_attn_fwd_host_workspace_size", "ring_attn_selftest_bounded_wait", "ring_attn_device_check",
    "ring_attn_block_fwd", "ring_attn_block_bwd", "ring_attn_bwd_preprocess", "ring_attn_f32_zero",
    "ring_attn_f32_add", "ring_attn_f32_convert", "ring_attn_block_rope", "ring_attn_fwd_f32out",
    "ring_attn_bwd_f32out", "ring_attn_bwd_preprocess_f32out",
)


class RingAttnError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"libringattn status {status}: {msg}")
        self.status = status


def library():
    """The loaded ctypes library (raises RingAttnError if it is missing)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RingAttnError(-1, f"{LIB_PATH} is missing: build it with "
                                    "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(LIB_PATH)
        P, I, LL, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_size_t
        lib.ring_attn_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, I, P]
        lib.ring_attn_fwd_f32out.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, I, P]
        lib.ring_attn_ring_step_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, P]
        lib.ring_attn_lse_merge.argtypes = [P, P, P, P, LL, I, P]
        lib.ring_attn_fwd_stepwise.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, I, P, SZ, P]
        lib.ring_attn_fwd_stepwise_workspace_size.argtypes = [I, I, I, I]
        lib.ring_attn_fwd_stepwise_workspace_size.restype = SZ
        lib.ring_attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, P, SZ, I, I, I, I, I, I, I, I,
                                      I, P]
        lib.ring_attn_bwd_f32out.argtypes = lib.ring_attn_bwd.argtypes
        lib.ring_attn_bwd_preprocess_f32out.argtypes = [P, P, P, LL, I, I, P]
        lib.ring_attn_bwd_workspace_size.argtypes = [I, I, I, I, I, I]
        lib.ring_attn_bwd_workspace_size.restype = SZ
        lib.ring_attn_shard_tiles.argtypes = [I, I, I, I, I, P]
        lib.ring_attn_fwd_path.argtypes = [I, I, I, I, I, I, I, I, I, P]
        lib.ring_attn_bwd_path.argtypes = [I, I, I, I, I, I, I, I, I, P]
        lib.ring_attn_device_status.argtypes = [P, P]
        lib.ring_attn_device_check.argtypes = [P]
        lib.ring_attn_device_check.restype = ctypes.c_int
        lib.ring_attn_block_fwd.argtypes = [P, P, P, P, P] + [I] * 12 + [P]
        lib.ring_attn_block_fwd.restype = ctypes.c_int
        lib.ring_attn_block_bwd.argtypes = [P] * 9 + [I] * 12 + [P]
        lib.ring_attn_block_bwd.restype = ctypes.c_int
        lib.ring_attn_bwd_preprocess.argtypes = [P, P, P, LL, I, I, P]
        lib.ring_attn_bwd_preprocess.restype = ctypes.c_int
        lib.ring_attn_f32_zero.argtypes = [P, LL, P]
        lib.ring_attn_f32_zero.restype = ctypes.c_int
        lib.ring_attn_f32_add.argtypes = [P, P, LL, P]
        lib.ring_attn_f32_add.restype = ctypes.c_int
        lib.ring_attn_f32_convert.argtypes = [P, P, LL, I, P]
        lib.ring_attn_f32_convert.restype = ctypes.c_int
        lib.ring_attn_block_rope.argtypes = [P, I, I, I, I, I, I, I, I, ctypes.c_double, I, P]
        lib.ring_attn_block_rope.restype = ctypes.c_int
        lib.ring_attn_last_error.argtypes = []
        lib.ring_attn_last_error.restype = ctypes.c_char_p
        lib.ring_attn_abi_version.argtypes = []
        lib.ring_attn_bwd_static_scratch.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I,
                                                     I, I, I, P]
        lib.ring_attn_bwd_static_scratch.restype = ctypes.c_int
        lib.ring_attn_fwd_tile_visits.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, I, P, P]
        lib.ring_attn_fwd_tile_visits.restype = ctypes.c_int
        lib.ring_attn_bwd_tile_visits.argtypes = [P, P, P, P, P, P, P, P, P, I, P, SZ, I, I, I, I, I,
                                                  I, I, I, I, P, P]
        lib.ring_attn_bwd_tile_visits.restype = ctypes.c_int
        lib.ring_attn_rope.argtypes = [P, I, I, I, I, I, I, I, ctypes.c_double, I, P]
        lib.ring_attn_rope.restype = ctypes.c_int
        lib.ring_attn_ulysses_a2a.argtypes = [P, P, I, I, I, I, I, I, I, I, P]
        lib.ring_attn_ulysses_a2a.restype = ctypes.c_int
        lib.ring_attn_ulysses_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, I, P, SZ, P]
        lib.ring_attn_ulysses_fwd.restype = ctypes.c_int
        lib.ring_attn_ulysses_workspace_size.argtypes = [I, I, I, I, I, I]
        lib.ring_attn_ulysses_workspace_size.restype = SZ
        lib.ring_attn_ulysses_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, P, SZ, I, I, I, I, I, I, I, I, I, P]
        lib.ring_attn_ulysses_bwd.restype = ctypes.c_int
        lib.ring_attn_ulysses_bwd_workspace_size.argtypes = [I, I, I, I, I, I, I, I]
        lib.ring_attn_ulysses_bwd_workspace_size.restype = SZ
        lib.ring_attn_fwd_host.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, I, P, SZ, P]
        lib.ring_attn_fwd_host.restype = ctypes.c_int
        lib.ring_attn_fwd_host_workspace_size.argtypes = [I, I, I, I, I]
        lib.ring_attn_fwd_host_workspace_size.restype = SZ
        lib.ring_attn_selftest_bounded_wait.argtypes = [ctypes.c_ulonglong, P, P]
        lib.ring_attn_selftest_bounded_wait.restype = ctypes.c_int
        lib.ring_attn_ring_step_fwd_accumulate.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, P]
        lib.ring_attn_ring_step_fwd_accumulate.restype = ctypes.c_int
        lib.ring_attn_bwd_static_scratch_capacity.argtypes = []
        lib.ring_attn_bwd_static_scratch_capacity.restype = SZ
        for name in EXPORTS:
            f = getattr(lib, name)
            if f.restype is ctypes.c_int or name in ("ring_attn_fwd", "ring_attn_ring_step_fwd",
                                                     "ring_attn_lse_merge", "ring_attn_fwd_stepwise",
                                                     "ring_attn_bwd", "ring_attn_shard_tiles",
                                                     "ring_attn_fwd_path", "ring_attn_bwd_path",
                                                     "ring_attn_device_status",
                                                     "ring_attn_abi_version"):
                f.restype = ctypes.c_int
        _lib = lib
        return lib


def _check(status):
    if status != RA_OK:
        msg = library().ring_attn_last_error().decode(errors="replace")
        raise RingAttnError(status, msg)


def _dtype_code(dt):
    if dt == torch.float32:
        return 0
    if dt == torch.bfloat16:
        return 1
    raise ValueError(f"unsupported dtype {dt}")


def _layout(layout):
    return LAYOUTS[layout] if isinstance(layout, str) else int(layout)


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _dims(q, k):
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q must be [B,H,L,d] and k, v [B,Hkv,L,d]")
    B, H, L, d = q.shape
    Hkv = k.shape[1]
    return int(B), int(H), int(Hkv), int(L), int(d)


def _need(t, name, device, shape=None, dtype=None):
    """The library takes raw pointers and trusts the sizes it is given: every tensor is checked here
    (device, layout, shape, dtype) before its pointer is passed."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda or t.device != device:
        raise ValueError(f"{name} must be a CUDA tensor on {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, not {tuple(t.shape)}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, not {t.dtype}")


def _need_qkv(q, k, v):
    """q [B,H,L,d], k and v [B,Hkv,L,d] of q's dtype, all on q's device; returns (B, H, Hkv, L, d)."""
    B, H, Hkv, L, d = _dims(q, k)
    _need(q, "q", q.device)
    _dtype_code(q.dtype)
    _need(k, "k", q.device, (B, Hkv, L, d), q.dtype)
    _need(v, "v", q.device, (B, Hkv, L, d), q.dtype)
    return B, H, Hkv, L, d


def _need_workspace(ws, need, device):
    _need(ws, "workspace", device)
    if ws.dtype != torch.uint8 or ws.numel() < need:
        raise ValueError(f"workspace must be a uint8 tensor of at least {need} bytes")


def fwd_path(B, H, Hkv, L, d, n_shards, causal, layout, dtype):
    out = ctypes.c_int(0)
    _check(library().ring_attn_fwd_path(B, H, Hkv, L, d, n_shards, int(causal), _layout(layout),
                                        _dtype_code(dtype), ctypes.byref(out)))
    return PATHS[out.value]


def bwd_path(B, H, Hkv, L, d, n_shards, causal, layout, dtype):
    out = ctypes.c_int(0)
    _check(library().ring_attn_bwd_path(B, H, Hkv, L, d, n_shards, int(causal), _layout(layout),
                                        _dtype_code(dtype), ctypes.byref(out)))
    return PATHS[out.value]


def _visits(n_shards, device):
    return torch.zeros((n_shards, n_shards), dtype=torch.int64, device=device)


def fwd(q, k, v, n_shards, causal=True, layout="zigzag", out=None, lse=None, stream=None):
    """Ring Attention forward.  Returns (out [B,H,L,d] q.dtype, lse [B,H,L] float32)."""
    return _fwd(q, k, v, n_shards, causal, layout, out, lse, None, stream)


def fwd_tile_visits(q, k, v, n_shards, causal=True, layout="zigzag", stream=None):
    """ring_attn_fwd_tile_visits: the forward plus the count of (256-row query block, 128-row K/V
    tile) pairs computed per (query shard, key shard).  Returns (out, lse, visits [n, n] int64)."""
    visits = _visits(n_shards, q.device)
    out, lse = _fwd(q, k, v, n_shards, causal, layout, None, None, visits, stream)
    return out, lse, visits


def _fwd(q, k, v, n_shards, causal, layout, out, lse, visits, stream):
    B, H, Hkv, L, d = _need_qkv(q, k, v)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, L), dtype=torch.float32, device=q.device)
    _need(out, "out", q.device, q.shape, q.dtype)
    _need(lse, "lse", q.device, (B, H, L), torch.float32)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Hkv, L, d, int(n_shards),
            int(causal), _layout(layout), _dtype_code(q.dtype))
    if visits is None:
        _check(library().ring_attn_fwd(*args, _stream(stream, q.device)))
    else:
        _check(library().ring_attn_fwd_tile_visits(*args, _ptr(visits), _stream(stream, q.device)))
    return out, lse


def fwd_host(q, k, v, n_shards, causal=True, layout="zigzag", out=None, lse=None, workspace=None, device=None,
             stream=None):
    """ring_attn_fwd_host: q, k, v are CPU tensors (page-locked for overlap); returns CPU (out, lse).
    The copies in and out overlap the compute of other kv-head groups."""
    B, H, Hkv, L, d = _dims(q, k)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    _dtype_code(q.dtype)
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    if lse is None:
        lse = torch.empty((B, H, L), dtype=torch.float32, pin_memory=True)
    for t, nm, shape, dt in ((q, "q", q.shape, q.dtype), (k, "k", (B, Hkv, L, d), q.dtype),
                             (v, "v", (B, Hkv, L, d), q.dtype), (out, "out", q.shape, q.dtype),
                             (lse, "lse", (B, H, L), torch.float32)):
        if not isinstance(t, torch.Tensor) or t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{nm} must be a contiguous CPU tensor")
        if tuple(t.shape) != tuple(shape) or t.dtype != dt:
            raise ValueError(f"{nm} must be {dt} of shape {tuple(shape)}")
    need = int(library().ring_attn_fwd_host_workspace_size(H, Hkv, L, d, _dtype_code(q.dtype)))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _need_workspace(workspace, need, dev)
    _check(library().ring_attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Hkv, L, d,
                                        int(n_shards), int(causal), _layout(layout), _dtype_code(q.dtype),
                                        _ptr(workspace), workspace.numel(), _stream(stream, dev)))
    return out, lse


def ring_step_fwd(q, k, v, n_shards, step, causal=True, layout="zigzag", o_part=None,
                  lse_part=None, stream=None):
    """One ring step for all shards.  Returns (o_part float32 [B,H,L,d], lse_part [B,H,L])."""
    B, H, Hkv, L, d = _need_qkv(q, k, v)
    if o_part is None:
        o_part = torch.empty((B, H, L, d), dtype=torch.float32, device=q.device)
    if lse_part is None:
        lse_part = torch.empty((B, H, L), dtype=torch.float32, device=q.device)
    _need(o_part, "o_part", q.device, (B, H, L, d), torch.float32)
    _need(lse_part, "lse_part", q.device, (B, H, L), torch.float32)
    _check(library().ring_attn_ring_step_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o_part),
                                             _ptr(lse_part), B, H, Hkv, L, d, int(n_shards),
                                             int(step), int(causal), _layout(layout),
                                             _dtype_code(q.dtype), _stream(stream, q.device)))
    return o_part, lse_part


def ring_step_fwd_accumulate(q, k, v, n_shards, step, o_acc, lse_acc, causal=True, layout="zigzag", stream=None):
    """ring_attn_ring_step_fwd_accumulate: fold ring step `step` into (o_acc float32 [B,H,L,d],
    lse_acc [B,H,L]) in place.  Returns (o_acc, lse_acc)."""
    B, H, Hkv, L, d = _need_qkv(q, k, v)
    _need(o_acc, "o_acc", q.device, (B, H, L, d), torch.float32)
    _need(lse_acc, "lse_acc", q.device, (B, H, L), torch.float32)
    _check(library().ring_attn_ring_step_fwd_accumulate(_ptr(q), _ptr(k), _ptr(v), _ptr(o_acc), _ptr(lse_acc), B, H,
                                                        Hkv, L, d, int(n_shards), int(step), int(causal),
                                                        _layout(layout), _dtype_code(q.dtype),
                                                        _stream(stream, q.device)))
    return o_acc, lse_acc


def lse_merge(o_acc, lse_acc, o_part, lse_part, stream=None):
    """In-place merge of a partial (o_part, lse_part) into (o_acc, lse_acc); float32 tensors."""
    if o_acc.dim() < 1 or tuple(lse_acc.shape) != tuple(o_acc.shape[:-1]):
        raise ValueError("lse_acc must have the shape of o_acc without its last dimension")
    d = int(o_acc.shape[-1])
    rows = int(lse_acc.numel())
    _need(o_acc, "o_acc", o_acc.device, None, torch.float32)
    _need(lse_acc, "lse_acc", o_acc.device, None, torch.float32)
    _need(o_part, "o_part", o_acc.device, o_acc.shape, torch.float32)
    _need(lse_part, "lse_part", o_acc.device, lse_acc.shape, torch.float32)
    _check(library().ring_attn_lse_merge(_ptr(o_acc), _ptr(lse_acc), _ptr(o_part), _ptr(lse_part),
                                         rows, d, _stream(stream, o_acc.device)))
    return o_acc, lse_acc


def fwd_stepwise(q, k, v, n_shards, causal=True, layout="zigzag", out=None, lse=None,
                 workspace=None, stream=None):
    """The ring forward run as n ring-step launches, each folding its block into the running
    result (same results as fwd)."""
    B, H, Hkv, L, d = _need_qkv(q, k, v)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, L), dtype=torch.float32, device=q.device)
    _need(out, "out", q.device, q.shape, q.dtype)
    _need(lse, "lse", q.device, (B, H, L), torch.float32)
    need = int(library().ring_attn_fwd_stepwise_workspace_size(B, H, L, d))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _need_workspace(workspace, need, q.device)
    _check(library().ring_attn_fwd_stepwise(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H,
                                            Hkv, L, d, int(n_shards), int(causal),
                                            _layout(layout), _dtype_code(q.dtype),
                                            _ptr(workspace), workspace.numel(),
                                            _stream(stream, q.device)))
    return out, lse


def bwd_workspace_size(B, H, Hkv, L, d, grad_dtype=torch.float32):
    return int(library().ring_attn_bwd_workspace_size(B, H, Hkv, L, d, _dtype_code(grad_dtype)))


def bwd(q, k, v, out, lse, dout, n_shards, causal=True, layout="zigzag",
        grad_dtype=torch.float32, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Ring Attention backward.  Returns (dq, dk, dv) in grad_dtype."""
    return _bwd(q, k, v, out, lse, dout, n_shards, causal, layout, grad_dtype, dq, dk, dv,
                workspace, None, stream)


def bwd_tile_visits(q, k, v, out, lse, dout, n_shards, causal=True, layout="zigzag",
                    grad_dtype=torch.float32, stream=None):
    """ring_attn_bwd_tile_visits: the backward plus the count of (128-row query tile, 128-row K/V
    tile) pairs computed per (query shard, key shard).  Returns (dq, dk, dv, visits [n, n] int64)."""
    visits = _visits(n_shards, q.device)
    dq, dk, dv = _bwd(q, k, v, out, lse, dout, n_shards, causal, layout, grad_dtype, None, None,
                      None, None, visits, stream)
    return dq, dk, dv, visits


def _need_bwd_args(q, k, v, out, lse, dout, grad_dtype, out_dtype=None):
    B, H, Hkv, L, d = _need_qkv(q, k, v)
    _need(out, "out", q.device, q.shape, q.dtype if out_dtype is None else out_dtype)
    _need(lse, "lse", q.device, (B, H, L), torch.float32)
    _need(dout, "dout", q.device, q.shape, q.dtype)
    _dtype_code(grad_dtype)
    return B, H, Hkv, L, d


def _need_grads(dq, dk, dv, device, dims, grad_dtype):
    B, H, Hkv, L, d = dims
    _need(dq, "dq", device, (B, H, L, d), grad_dtype)
    _need(dk, "dk", device, (B, Hkv, L, d), grad_dtype)
    _need(dv, "dv", device, (B, Hkv, L, d), grad_dtype)


def _bwd(q, k, v, out, lse, dout, n_shards, causal, layout, grad_dtype, dq, dk, dv, workspace,
         visits, stream, out_f32=False):
    B, H, Hkv, L, d = _need_bwd_args(q, k, v, out, lse, dout, grad_dtype,
                                     torch.float32 if out_f32 else None)
    if dq is None:
        dq = torch.empty((B, H, L, d), dtype=grad_dtype, device=q.device)
    if dk is None:
        dk = torch.empty((B, Hkv, L, d), dtype=grad_dtype, device=q.device)
    if dv is None:
        dv = torch.empty((B, Hkv, L, d), dtype=grad_dtype, device=q.device)
    _need_grads(dq, dk, dv, q.device, (B, H, Hkv, L, d), grad_dtype)
    need = bwd_workspace_size(B, H, Hkv, L, d, grad_dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _need_workspace(workspace, need, q.device)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
            _ptr(dv), _dtype_code(grad_dtype), _ptr(workspace), workspace.numel(), B, H, Hkv, L, d,
            int(n_shards), int(causal), _layout(layout), _dtype_code(q.dtype))
    if out_f32:
        _check(library().ring_attn_bwd_f32out(*args, _stream(stream, q.device)))
    elif visits is None:
        _check(library().ring_attn_bwd(*args, _stream(stream, q.device)))
    else:
        _check(library().ring_attn_bwd_tile_visits(*args, _ptr(visits), _stream(stream, q.device)))
    return dq, dk, dv


def fwd_f32out(q, k, v, n_shards, causal=True, layout="zigzag", out=None, lse=None, stream=None):
    """ring_attn_fwd_f32out: the forward with out in float32 -- the output before it is rounded to
    q's dtype.  Returns (out [B,H,L,d] float32, lse [B,H,L] float32)."""
    B, H, Hkv, L, d = _need_qkv(q, k, v)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, L), dtype=torch.float32, device=q.device)
    _need(out, "out", q.device, q.shape, torch.float32)
    _need(lse, "lse", q.device, (B, H, L), torch.float32)
    _check(library().ring_attn_fwd_f32out(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Hkv, L, d,
                                          int(n_shards), int(causal), _layout(layout), _dtype_code(q.dtype),
                                          _stream(stream, q.device)))
    return out, lse


def bwd_f32out(q, k, v, out, lse, dout, n_shards, causal=True, layout="zigzag",
               grad_dtype=torch.float32, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """ring_attn_bwd_f32out: the backward with out in float32 (from fwd_f32out), so that D is taken from
    the unrounded output.  Returns (dq, dk, dv) in grad_dtype."""
    return _bwd(q, k, v, out, lse, dout, n_shards, causal, layout, grad_dtype, dq, dk, dv,
                workspace, None, stream, out_f32=True)


def bwd_static_scratch(q, k, v, out, lse, dout, n_shards, causal=True, layout="zigzag",
                       grad_dtype=torch.float32, dq=None, dk=None, dv=None, stream=None):
    """ring_attn_bwd_static_scratch: the backward with the library's static scratch (no workspace
    argument; the C call allocates nothing).  Returns (dq, dk, dv) in grad_dtype."""
    B, H, Hkv, L, d = _need_bwd_args(q, k, v, out, lse, dout, grad_dtype)
    if dq is None:
        dq = torch.empty((B, H, L, d), dtype=grad_dtype, device=q.device)
    if dk is None:
        dk = torch.empty((B, Hkv, L, d), dtype=grad_dtype, device=q.device)
    if dv is None:
        dv = torch.empty((B, Hkv, L, d), dtype=grad_dtype, device=q.device)
    _need_grads(dq, dk, dv, q.device, (B, H, Hkv, L, d), grad_dtype)
    _check(library().ring_attn_bwd_static_scratch(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
        _dtype_code(grad_dtype), B, H, Hkv, L, d, int(n_shards), int(causal), _layout(layout),
        _dtype_code(q.dtype), _stream(stream, q.device)))
    return dq, dk, dv


def bwd_static_scratch_capacity():
    return int(library().ring_attn_bwd_static_scratch_capacity())


def shard_tiles(L, n_shards, causal=True, layout="zigzag", tile=128):
    """Host-only: per query shard, the (query tile, key tile) pairs with a visible pair."""
    arr = (ctypes.c_longlong * n_shards)()
    _check(library().ring_attn_shard_tiles(int(L), int(n_shards), int(causal), _layout(layout),
                                           int(tile), arr))
    return [int(x) for x in arr]


def rope(x, n_shards, layout="zigzag", base=10000.0, inverse=False, stream=None):
    """ring_attn_rope: rotary position embedding of x [B, H, L, d] (bf16 or float32) in place, each row
    by its natural position under the layout; inverse=True turns the other way (for gradients).
    Returns x."""
    if x.dim() != 4:
        raise ValueError("x must be [B, H, L, d]")
    _need(x, "x", x.device)
    B, H, L, d = (int(s) for s in x.shape)
    _check(library().ring_attn_rope(_ptr(x), B, H, L, d, int(n_shards), _layout(layout), _dtype_code(x.dtype),
                                    float(base), int(bool(inverse)), _stream(stream, x.device)))
    return x


def ulysses_a2a(src, n_shards, layout="contiguous", direction=0, dst=None, stream=None):
    """ring_attn_ulysses_a2a.  direction 0: src [n, B, S, H, d] (token split) -> [n, B, H/n, L, d]
    (head split); direction 1 the reverse.  A 4-D src [n, B, S, H] (lse) moves rows of one float."""
    _need(src, "src", src.device)
    if direction == 0:
        if src.dim() == 5:
            n, B, S, H, d = (int(s) for s in src.shape)
            shape = (n, B, H // n, n * S, d)
        else:
            n, B, S, H = (int(s) for s in src.shape)
            d = 1
            shape = (n, B, H // n, n * S)
    else:
        if src.dim() == 5:
            n, B, Hn, L, d = (int(s) for s in src.shape)
            S, H = L // n, Hn * n
            shape = (n, B, S, H, d)
        else:
            n, B, Hn, L = (int(s) for s in src.shape)
            S, H, d = L // n, Hn * n, 1
            shape = (n, B, S, H)
    if n != n_shards:
        raise ValueError("the leading dimension of src must be n_shards")
    if dst is None:
        dst = torch.empty(shape, dtype=src.dtype, device=src.device)
    _need(dst, "dst", src.device, shape, src.dtype)
    _check(library().ring_attn_ulysses_a2a(_ptr(src), _ptr(dst), B, H, n * S, d, n, _layout(layout),
                                           _dtype_code(src.dtype), int(direction), _stream(stream, src.device)))
    return dst


def _need_ulysses_qkv(q, k, v, n_shards):
    """q [n, B, S, H, d], k and v [n, B, S, Hkv, d] of q's dtype; returns (n, B, S, H, Hkv, d)."""
    for t, nm in ((q, "q"), (k, "k"), (v, "v")):
        if not isinstance(t, torch.Tensor) or t.dim() != 5:
            raise ValueError(f"{nm} must be [n, B, S, heads, d]")
    n, B, S, H, d = (int(s) for s in q.shape)
    Hkv = int(k.shape[3])
    if n != n_shards:
        raise ValueError("the leading dimension of q must be n_shards")
    _need(q, "q", q.device)
    _dtype_code(q.dtype)
    _need(k, "k", q.device, (n, B, S, Hkv, d), q.dtype)
    _need(v, "v", q.device, (n, B, S, Hkv, d), q.dtype)
    return n, B, S, H, Hkv, d


def ulysses_fwd(q, k, v, n_shards, causal=True, layout="contiguous", out=None, lse=None, workspace=None,
                stream=None):
    """ring_attn_ulysses_fwd: q [n, B, S, H, d], k and v [n, B, S, Hkv, d] (token split).  Returns
    (out [n, B, S, H, d], lse [n, B, S, H] float32)."""
    n, B, S, H, Hkv, d = _need_ulysses_qkv(q, k, v, n_shards)
    L = n * S
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((n, B, S, H), dtype=torch.float32, device=q.device)
    _need(out, "out", q.device, q.shape, q.dtype)
    _need(lse, "lse", q.device, (n, B, S, H), torch.float32)
    need = int(library().ring_attn_ulysses_workspace_size(B, H, Hkv, L, d, _dtype_code(q.dtype)))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _need_workspace(workspace, need, q.device)
    _check(library().ring_attn_ulysses_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Hkv, L, d, n,
                                           int(causal), _layout(layout), _dtype_code(q.dtype), _ptr(workspace),
                                           workspace.numel(), _stream(stream, q.device)))
    return out, lse


def ulysses_bwd(q, k, v, out, lse, dout, n_shards, causal=True, layout="contiguous", grad_dtype=torch.float32,
                workspace=None, stream=None):
    """ring_attn_ulysses_bwd: token-split inputs as for ulysses_fwd (plus out, lse from it and dout
    [n, B, S, H, d]).  Returns (dq, dk, dv) in the token split, grad_dtype."""
    n, B, S, H, Hkv, d = _need_ulysses_qkv(q, k, v, n_shards)
    L = n * S
    _need(out, "out", q.device, q.shape, q.dtype)
    _need(lse, "lse", q.device, (n, B, S, H), torch.float32)
    _need(dout, "dout", q.device, q.shape, q.dtype)
    _dtype_code(grad_dtype)
    dq = torch.empty(q.shape, dtype=grad_dtype, device=q.device)
    dk = torch.empty(k.shape, dtype=grad_dtype, device=q.device)
    dv = torch.empty(v.shape, dtype=grad_dtype, device=q.device)
    need = int(library().ring_attn_ulysses_bwd_workspace_size(B, H, Hkv, L, d, n, _dtype_code(q.dtype),
                                                              _dtype_code(grad_dtype)))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _need_workspace(workspace, need, q.device)
    _check(library().ring_attn_ulysses_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq),
                                           _ptr(dk), _ptr(dv), _dtype_code(grad_dtype), _ptr(workspace),
                                           workspace.numel(), B, H, Hkv, L, d, n, int(causal), _layout(layout),
                                           _dtype_code(q.dtype), _stream(stream, q.device)))
    return dq, dk, dv


def selftest_bounded_wait(limit_ns=2_000_000, stream=None, device=None):
    """ring_attn_selftest_bounded_wait: a GPU wait that nothing completes runs out after limit_ns.
    Returns the kernel's report (1: gave up, 2: completed); the status word then has the timeout bit."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    flag = torch.zeros(4, dtype=torch.int32, device=dev)
    _check(library().ring_attn_selftest_bounded_wait(int(limit_ns), _ptr(flag), _stream(stream, dev)))
    return int(flag[0].item())


def device_status(stream=None, device=None):
    """Reads and clears the device status word (bit RA_DEVICE_TIMEOUT: a bounded wait ran out)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    st = ctypes.c_uint(0)
    _check(library().ring_attn_device_status(ctypes.byref(st), _stream(stream, dev)))
    return int(st.value)


def device_check(stream=None, device=None):
    """ring_attn_device_check: synchronises the stream, reads and clears the device status word and
    raises RingAttnError (status RA_ERR_TIMEOUT) if a bounded wait inside a kernel ran out."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    _check(library().ring_attn_device_check(_stream(stream, dev)))


# ------------------------------------------------------------------------------------------------
# One device of the multi-device ring: local shard buffers of S = L / n_shards rows per head
# ------------------------------------------------------------------------------------------------
def _need_block(q, k, v, n_shards, shard_q, shard_kv):
    """q [B,H,S,d] (shard shard_q's rows), k and v [B,Hkv,S,d] (shard shard_kv's rows), same dtype and
    device; returns (B, H, Hkv, S, d, L = n_shards * S)."""
    B, H, Hkv, S, d = _need_qkv(q, k, v)
    n = int(n_shards)
    if n < 1 or not (0 <= int(shard_q) < n and 0 <= int(shard_kv) < n):
        raise ValueError("shard indices must lie in [0, n_shards)")
    return B, H, Hkv, S, d, n * S


def block_fwd(q, k, v, o_acc, lse_acc, n_shards, shard_q, shard_kv, accumulate, causal=True, layout="zigzag",
              stream=None):
    """ring_attn_block_fwd: block attention of the local query shard shard_q against the K/V block of
    shard shard_kv, written to (accumulate=False) or folded into (accumulate=True) the running state
    o_acc [B,H,S,d] float32 (normalised output) and lse_acc [B,H,S] float32.  Returns (o_acc, lse_acc)."""
    B, H, Hkv, S, d, L = _need_block(q, k, v, n_shards, shard_q, shard_kv)
    _need(o_acc, "o_acc", q.device, (B, H, S, d), torch.float32)
    _need(lse_acc, "lse_acc", q.device, (B, H, S), torch.float32)
    _check(library().ring_attn_block_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o_acc), _ptr(lse_acc), B, H, Hkv, L, d,
                                         int(n_shards), int(shard_q), int(shard_kv), int(bool(accumulate)),
                                         int(causal), _layout(layout), _dtype_code(q.dtype),
                                         _stream(stream, q.device)))
    return o_acc, lse_acc


def block_bwd(q, k, v, dout, lse, D, dq_acc, dk, dv, n_shards, shard_q, shard_kv, accumulate_kv, causal=True,
              layout="zigzag", stream=None):
    """ring_attn_block_bwd: the gradient contributions of the pairs (query of shard shard_q, key of shard
    shard_kv): added into dq_acc [B,H,S,d] float32; added into (accumulate_kv=True) or stored to dk, dv
    [B,Hkv,S,d] float32.  lse and D [B,H,S] float32 are the query rows' full log-sum-exp and
    rowsum(dout * out).  Returns (dq_acc, dk, dv)."""
    B, H, Hkv, S, d, L = _need_block(q, k, v, n_shards, shard_q, shard_kv)
    _need(dout, "dout", q.device, q.shape, q.dtype)
    _need(lse, "lse", q.device, (B, H, S), torch.float32)
    _need(D, "D", q.device, (B, H, S), torch.float32)
    _need(dq_acc, "dq_acc", q.device, (B, H, S, d), torch.float32)
    _need(dk, "dk", q.device, (B, Hkv, S, d), torch.float32)
    _need(dv, "dv", q.device, (B, Hkv, S, d), torch.float32)
    _check(library().ring_attn_block_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(lse), _ptr(D), _ptr(dq_acc),
                                         _ptr(dk), _ptr(dv), B, H, Hkv, L, d, int(n_shards), int(shard_q),
                                         int(shard_kv), int(bool(accumulate_kv)), int(causal), _layout(layout),
                                         _dtype_code(q.dtype), _stream(stream, q.device)))
    return dq_acc, dk, dv


def bwd_preprocess(out, dout, D=None, stream=None):
    """ring_attn_bwd_preprocess: D = rowsum(out * dout) over the last dimension, float32.  out may be
    float32 while dout is bf16 (ring_attn_bwd_preprocess_f32out: the unrounded output)."""
    _need(out, "out", out.device)
    _dtype_code(dout.dtype)
    f32out = out.dtype == torch.float32 and dout.dtype != torch.float32
    _need(dout, "dout", out.device, out.shape, dout.dtype if f32out else out.dtype)
    if D is None:
        D = torch.empty(out.shape[:-1], dtype=torch.float32, device=out.device)
    _need(D, "D", out.device, out.shape[:-1], torch.float32)
    d = int(out.shape[-1])
    call = library().ring_attn_bwd_preprocess_f32out if f32out else library().ring_attn_bwd_preprocess
    _check(call(_ptr(out), _ptr(dout), _ptr(D), int(D.numel()), d, _dtype_code(dout.dtype),
                _stream(stream, out.device)))
    return D


def f32_zero(x, stream=None):
    """ring_attn_f32_zero: x (float32) = 0.  Returns x."""
    _need(x, "x", x.device, None, torch.float32)
    _check(library().ring_attn_f32_zero(_ptr(x), int(x.numel()), _stream(stream, x.device)))
    return x


def f32_add(acc, part, stream=None):
    """ring_attn_f32_add: acc += part (float32, same shape).  Returns acc."""
    _need(acc, "acc", acc.device, None, torch.float32)
    _need(part, "part", acc.device, acc.shape, torch.float32)
    _check(library().ring_attn_f32_add(_ptr(acc), _ptr(part), int(acc.numel()), _stream(stream, acc.device)))
    return acc


def f32_convert(src, dtype, dst=None, stream=None):
    """ring_attn_f32_convert: src (float32) converted to dtype (float32 or bfloat16).  Returns dst."""
    _need(src, "src", src.device, None, torch.float32)
    if dst is None:
        dst = torch.empty(src.shape, dtype=dtype, device=src.device)
    _need(dst, "dst", src.device, src.shape, dtype)
    _check(library().ring_attn_f32_convert(_ptr(src), _ptr(dst), int(src.numel()), _dtype_code(dtype),
                                           _stream(stream, src.device)))
    return dst


def block_rope(x, n_shards, shard, layout="zigzag", base=10000.0, inverse=False, stream=None):
    """ring_attn_block_rope: rotary position embedding, in place, of one device's shard x [B, H, S, d]
    (shard `shard` of n_shards; bf16 or float32), each row by its natural position in the whole
    sequence.  Returns x."""
    if x.dim() != 4:
        raise ValueError("x must be [B, H, S, d]")
    _need(x, "x", x.device)
    B, H, S, d = (int(t) for t in x.shape)
    n = int(n_shards)
    if not 0 <= int(shard) < n:
        raise ValueError("shard must lie in [0, n_shards)")
    _check(library().ring_attn_block_rope(_ptr(x), B, H, n * S, d, n, int(shard), _layout(layout),
                                          _dtype_code(x.dtype), float(base), int(bool(inverse)),
                                          _stream(stream, x.device)))
    return x
