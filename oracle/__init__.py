"""Float64 CPU oracle for Ring Attention -- TEST INFRASTRUCTURE ONLY.

The arithmetic lives in ``ring_oracle.c`` (plain C, float64, optional OpenMP); this module compiles it
with gcc on first use and wraps its functions with numpy arrays.  Only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import this package.  The
CUDA product path (``sequence_sharded_exact_gb300``) never imports it, and the two share no code.

Every function follows the pages' definition of exact softmax attention cut into ring shards (see
the header of ``ring_oracle.c`` for the passages and the readings taken where the pages are silent).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ring_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_ring_oracle.so")
_lock = threading.Lock()
_lib = None

LAYOUTS = {"contiguous": 0, "zigzag": 1, "striped": 2}


def build(force: bool = False) -> str:
    """Compile ring_oracle.c into _ring_oracle.so (gcc, -O2, no fast-math, no FMA contraction)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-fopenmp",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        Lg = ctypes.c_long
        lib.oracle_natural_position.argtypes = [Lg, Lg, I, I]
        lib.oracle_natural_position.restype = Lg
        common = [P, P, P, I, I, I, Lg, I, I, I, I]
        lib.oracle_attn_fwd_rows.argtypes = common + [Lg, P, P, P]
        lib.oracle_attn_fwd.argtypes = common + [P, P]
        lib.oracle_ring_fwd.argtypes = common + [P, P, P]
        bcommon = [P, P, P, P, I, I, I, Lg, I, I, I, I]
        given = [P, P, P, P, P, I, I, I, Lg, I, I, I, I]  # q, k, v, dout, out (or NULL), ...
        lib.oracle_attn_bwd_dq_rows.argtypes = given + [Lg, P, P]
        lib.oracle_attn_bwd_dkv_rows.argtypes = given + [Lg, P, P, P]
        lib.oracle_attn_bwd.argtypes = bcommon + [P, P, P]
        lib.oracle_block_fwd.argtypes = [P, P, P, I, I, I, Lg, I, I, I, I, I, I, P, P]
        lib.oracle_block_bwd.argtypes = [P, P, P, P, P, P, I, I, I, Lg, I, I, I, I, I, I, P, P, P]
        lib.oracle_shard_tiles.argtypes = [Lg, I, I, I, I, P]
        lib.oracle_rope.argtypes = [P, Lg, Lg, I, I, I, ctypes.c_double, I, P]
        lib.oracle_num_threads.argtypes = []
        for f in ("oracle_attn_fwd_rows", "oracle_attn_fwd", "oracle_ring_fwd",
                  "oracle_attn_bwd_dq_rows", "oracle_attn_bwd_dkv_rows", "oracle_attn_bwd",
                  "oracle_shard_tiles", "oracle_rope", "oracle_num_threads", "oracle_block_fwd",
                  "oracle_block_bwd"):
            getattr(lib, f).restype = I
        _lib = lib
        return lib


def _f32(a):
    """Contiguous float32 numpy copy of a numpy array or torch tensor (bf16 upcasts exactly)."""
    if hasattr(a, "detach"):
        a = a.detach().to("cpu")
        if str(a.dtype) != "torch.float32":
            a = a.float()
        a = a.contiguous().numpy()
    return np.ascontiguousarray(a, dtype=np.float32)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(st, what):
    if st != 0:
        raise ValueError(f"oracle: {what} failed with status {st}")


def _layout(layout):
    return LAYOUTS[layout] if isinstance(layout, str) else int(layout)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def natural_position(r, L, n, layout):
    """Natural sequence position of buffer row r."""
    return int(_load().oracle_natural_position(int(r), int(L), int(n), _layout(layout)))


def attn_fwd(q, k, v, n, causal, layout):
    """Exact attention for every row.  q [B,H,L,d], k/v [B,Hkv,L,d] -> (out [B,H,L,d], lse [B,H,L])."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, H, L, d = q.shape
    Hkv = k.shape[1]
    out = np.empty((B, H, L, d), np.float64)
    lse = np.empty((B, H, L), np.float64)
    _check(_load().oracle_attn_fwd(_ptr(q), _ptr(k), _ptr(v), B, H, Hkv, L, d, int(n), int(causal),
                                   _layout(layout), _ptr(out), _ptr(lse)), "attn_fwd")
    return out, lse


def attn_fwd_rows(q, k, v, n, causal, layout, rows):
    """Exact attention for selected rows; rows are flat indices (b*H + h)*L + r.
    Returns (out [nrows,d], lse [nrows])."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, H, L, d = q.shape
    Hkv = k.shape[1]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((rows.size, d), np.float64)
    lse = np.empty((rows.size,), np.float64)
    _check(_load().oracle_attn_fwd_rows(_ptr(q), _ptr(k), _ptr(v), B, H, Hkv, L, d, int(n),
                                        int(causal), _layout(layout), rows.size, _ptr(rows),
                                        _ptr(out), _ptr(lse)), "attn_fwd_rows")
    return out, lse


def ring_fwd(q, k, v, n, causal, layout):
    """The n-step ring walk with the page's online-softmax update.
    Returns (out, lse, pairs[n,n]) where pairs[i,j] counts visible (query,key) pairs of step (i,j)."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, H, L, d = q.shape
    Hkv = k.shape[1]
    out = np.empty((B, H, L, d), np.float64)
    lse = np.empty((B, H, L), np.float64)
    pairs = np.zeros((n, n), np.int64)
    _check(_load().oracle_ring_fwd(_ptr(q), _ptr(k), _ptr(v), B, H, Hkv, L, d, int(n), int(causal),
                                   _layout(layout), _ptr(out), _ptr(lse), _ptr(pairs)), "ring_fwd")
    return out, lse, pairs


def attn_bwd(q, k, v, dout, n, causal, layout):
    """Gradients of sum(out * dout) w.r.t. q, k, v for every row: (dq, dk, dv) float64."""
    q, k, v, dout = _f32(q), _f32(k), _f32(v), _f32(dout)
    B, H, L, d = q.shape
    Hkv = k.shape[1]
    dq = np.empty((B, H, L, d), np.float64)
    dk = np.empty((B, Hkv, L, d), np.float64)
    dv = np.empty((B, Hkv, L, d), np.float64)
    _check(_load().oracle_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), B, H, Hkv, L, d, int(n),
                                   int(causal), _layout(layout), _ptr(dq), _ptr(dk), _ptr(dv)),
           "attn_bwd")
    return dq, dk, dv


def _given_out(out, shape):
    """The output array whose rows give D, as float32 (a bf16 tensor upcasts exactly), or None."""
    if out is None:
        return None
    o = _f32(out)
    if o.shape != shape:
        raise ValueError(f"out of shape {o.shape}, expected {shape}")
    return o


def attn_bwd_dq_rows(q, k, v, dout, n, causal, layout, rows, out=None):
    """dQ for selected query rows (flat (b*H + h)*L + r) -> [nrows, d].

    out: None (D = <dO, O> with the forward definition's O) or an output [B, H, L, d] whose rows give
    D instead -- the output a backward receives as its input (the forward's stored, rounded result),
    read as given, like the rounded q, k, v."""
    q, k, v, dout = _f32(q), _f32(k), _f32(v), _f32(dout)
    B, H, L, d = q.shape
    Hkv = k.shape[1]
    og = _given_out(out, q.shape)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    dq = np.empty((rows.size, d), np.float64)
    _check(_load().oracle_attn_bwd_dq_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(dout),
                                           None if og is None else _ptr(og), B, H, Hkv, L, d,
                                           int(n), int(causal), _layout(layout), rows.size,
                                           _ptr(rows), _ptr(dq)), "attn_bwd_dq_rows")
    return dq


def attn_bwd_dkv_rows(q, k, v, dout, n, causal, layout, keys, out=None):
    """dK, dV for selected key rows (flat (b*Hkv + g)*L + t) -> ([nkeys, d], [nkeys, d]).

    out: as in attn_bwd_dq_rows (D from the given output's rows, or from the forward definition)."""
    q, k, v, dout = _f32(q), _f32(k), _f32(v), _f32(dout)
    B, H, L, d = q.shape
    Hkv = k.shape[1]
    og = _given_out(out, q.shape)
    keys = np.ascontiguousarray(keys, dtype=np.int64)
    dk = np.empty((keys.size, d), np.float64)
    dv = np.empty((keys.size, d), np.float64)
    _check(_load().oracle_attn_bwd_dkv_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(dout),
                                            None if og is None else _ptr(og), B, H, Hkv, L, d,
                                            int(n), int(causal), _layout(layout), keys.size,
                                            _ptr(keys), _ptr(dk), _ptr(dv)), "attn_bwd_dkv_rows")
    return dk, dv


def shard_tiles(L, n, causal, layout, tile=128):
    """Per query shard, the number of (query tile, key tile) pairs holding a visible pair."""
    out = np.zeros((n,), np.int64)
    _check(_load().oracle_shard_tiles(int(L), int(n), int(causal), _layout(layout), int(tile),
                                      _ptr(out)), "shard_tiles")
    return out


def rope(x, n, layout, base=10000.0, inverse=False):
    """Rotary position embedding of every row of x [..., L, d] by its natural position (float64)."""
    x = _f32(x)
    L, d = x.shape[-2], x.shape[-1]
    nheads = int(np.prod(x.shape[:-2])) if x.ndim > 2 else 1
    y = np.empty(x.shape, np.float64)
    _check(_load().oracle_rope(_ptr(x), nheads, L, d, int(n), _layout(layout), float(base), int(bool(inverse)),
                               _ptr(y)), "rope")
    return y


def _f64(a):
    """Contiguous float64 numpy copy of a numpy array or torch tensor."""
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").double().contiguous().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def block_fwd(q_i, k_j, v_j, L, n, causal, layout, i, j):
    """One device's block: attention of shard i's rows (q_i [B,H,S,d]) restricted to the keys of
    shard j (k_j, v_j [B,Hkv,S,d]).  Returns (o_part [B,H,S,d] normalised by the block's own sum,
    lse_part [B,H,S]; -inf where the row sees nothing of the block)."""
    q_i, k_j, v_j = _f32(q_i), _f32(k_j), _f32(v_j)
    B, H, S, d = q_i.shape
    Hkv = k_j.shape[1]
    o = np.empty((B, H, S, d), np.float64)
    lse = np.empty((B, H, S), np.float64)
    _check(_load().oracle_block_fwd(_ptr(q_i), _ptr(k_j), _ptr(v_j), B, H, Hkv, int(L), d, int(n), int(causal),
                                    _layout(layout), int(i), int(j), _ptr(o), _ptr(lse)), "block_fwd")
    return o, lse


def block_bwd(q_i, k_j, v_j, dout_i, lse_i, D_i, L, n, causal, layout, i, j):
    """The gradient contributions of the pairs (query of shard i, key of shard j), with P from the
    query rows' full lse_i and D_i = <dO, O> ([B,H,S], float64).  Returns (dq_part [B,H,S,d],
    dk_part [B,Hkv,S,d], dv_part [B,Hkv,S,d])."""
    q_i, k_j, v_j, dout_i = _f32(q_i), _f32(k_j), _f32(v_j), _f32(dout_i)
    lse_i, D_i = _f64(lse_i), _f64(D_i)
    B, H, S, d = q_i.shape
    Hkv = k_j.shape[1]
    dq = np.empty((B, H, S, d), np.float64)
    dk = np.empty((B, Hkv, S, d), np.float64)
    dv = np.empty((B, Hkv, S, d), np.float64)
    _check(_load().oracle_block_bwd(_ptr(q_i), _ptr(k_j), _ptr(v_j), _ptr(dout_i), _ptr(lse_i), _ptr(D_i), B, H,
                                    Hkv, int(L), d, int(n), int(causal), _layout(layout), int(i), int(j), _ptr(dq),
                                    _ptr(dk), _ptr(dv)), "block_bwd")
    return dq, dk, dv
