"""CPU-only checks of the C ABI: the library loads without a GPU, exports every declared entry
point, rejects bad arguments before touching CUDA, and its host-side shard scheduler agrees with
the oracle's brute-force tile counter."""
import ctypes
import os
import re

import pytest
import torch

import oracle
from sequence_sharded_exact_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ringattn.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ring_attn_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return binding.library()


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("ring_attn_fwd", "ring_attn_bwd", "ring_attn_ring_step_fwd", "ring_attn_lse_merge",
                 "ring_attn_shard_tiles", "ring_attn_last_error"):
        assert want in names
    assert set(names) == set(binding.EXPORTS), "binding and header disagree"


def test_binding_constants_match_the_header():
    """The binding's status, layout, dtype, path and device-status codes are the header's."""
    src = open(HEADER).read()
    defs = {m.group(1): int(m.group(2)) for m in re.finditer(r"#define (RA_\w+) (\d+)u?\b", src)}
    for name in ("RA_OK", "RA_ERR_INVALID_ARG", "RA_ERR_UNSUPPORTED", "RA_ERR_CUDA", "RA_ERR_NO_DEVICE",
                 "RA_ERR_TIMEOUT", "RA_DEVICE_TIMEOUT", "RA_DEVICE_LAYOUT"):
        assert getattr(binding, name) == defs[name], name
    assert binding.LAYOUTS == {"contiguous": defs["RA_LAYOUT_CONTIGUOUS"], "zigzag": defs["RA_LAYOUT_ZIGZAG"],
                               "striped": defs["RA_LAYOUT_STRIPED"]}
    assert binding.PATHS == {defs["RA_PATH_SIMT"]: "simt", defs["RA_PATH_TCGEN05"]: "tcgen05"}
    assert binding._dtype_code(torch.float32) == defs["RA_F32"]
    assert binding._dtype_code(torch.bfloat16) == defs["RA_BF16"]


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert lib.ring_attn_abi_version() == 1


def _fwd(lib, **kw):
    a = dict(q=16, k=16, v=16, out=16, lse=16, B=1, H=2, Hkv=1, L=1024, d=128, n=4, causal=1,
             layout=1, dtype=1)
    a.update(kw)
    P = ctypes.c_void_p
    return lib.ring_attn_fwd(P(a["q"]), P(a["k"]), P(a["v"]), P(a["out"]), P(a["lse"]), a["B"],
                             a["H"], a["Hkv"], a["L"], a["d"], a["n"], a["causal"], a["layout"],
                             a["dtype"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=0), binding.RA_ERR_INVALID_ARG),
    (dict(k=8), binding.RA_ERR_INVALID_ARG),           # not 16-byte aligned
    (dict(H=3, Hkv=2), binding.RA_ERR_INVALID_ARG),    # H % Hkv
    (dict(L=1000, n=3), binding.RA_ERR_INVALID_ARG),   # L % n
    (dict(L=1026, n=6), binding.RA_ERR_INVALID_ARG),   # zigzag needs L % 2n
    (dict(d=96), binding.RA_ERR_UNSUPPORTED),
    (dict(layout=7), binding.RA_ERR_INVALID_ARG),
    (dict(dtype=5), binding.RA_ERR_INVALID_ARG),
    (dict(causal=2), binding.RA_ERR_INVALID_ARG),
    (dict(B=0), binding.RA_ERR_INVALID_ARG),                   # empty problem
    (dict(L=0), binding.RA_ERR_INVALID_ARG),
    (dict(B=256, H=32, Hkv=8, L=1 << 20, n=8), binding.RA_ERR_UNSUPPORTED),  # 2^40 elements of q
])
def test_argument_errors_before_any_cuda_call(lib, kw, status):
    assert _fwd(lib, **kw) == status
    assert lib.ring_attn_last_error().decode()


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device answer")
def test_no_device_answer(lib):
    assert _fwd(lib) == binding.RA_ERR_NO_DEVICE


def test_path_selection():
    assert binding.fwd_path(1, 32, 8, 131072, 128, 8, True, "zigzag", torch.bfloat16) == "tcgen05"
    assert binding.fwd_path(2, 8, 8, 8192, 128, 8, True, "contiguous", torch.bfloat16) == "tcgen05"
    assert binding.fwd_path(1, 1, 1, 256, 64, 4, False, "contiguous", torch.float32) == "simt"
    assert binding.fwd_path(1, 2, 2, 384, 128, 3, True, "zigzag", torch.bfloat16) == "simt"
    assert binding.fwd_path(1, 2, 2, 512, 64, 2, True, "zigzag", torch.bfloat16) == "simt"  # chunks of 128
    assert binding.fwd_path(1, 8, 2, 2048, 64, 4, True, "zigzag", torch.bfloat16) == "tcgen05"
    assert binding.bwd_path(1, 8, 2, 2048, 64, 4, True, "zigzag", torch.bfloat16) == "tcgen05"
    assert binding.bwd_path(1, 2, 2, 512, 64, 4, True, "zigzag", torch.bfloat16) == "simt"  # chunks of 64
    assert binding.bwd_path(1, 8, 2, 2048, 64, 4, True, "zigzag", torch.float32) == "simt"
    # striped: the tensor-core paths need shards of whole 256-row (forward) / 128-row (backward) tiles
    assert binding.fwd_path(1, 32, 8, 131072, 128, 8, True, "striped", torch.bfloat16) == "tcgen05"
    assert binding.fwd_path(1, 2, 2, 384, 128, 3, True, "striped", torch.bfloat16) == "simt"
    assert binding.bwd_path(1, 2, 2, 384, 128, 3, True, "striped", torch.bfloat16) == "tcgen05"
    assert binding.bwd_path(1, 2, 2, 600, 128, 3, True, "striped", torch.bfloat16) == "simt"


@pytest.mark.parametrize("L,n,T", [(8192, 8, 128), (32768, 8, 128), (1000, 5, 64), (384, 3, 128),
                                   (4096, 16, 128), (96, 4, 7)])
@pytest.mark.parametrize("layout", ["contiguous", "zigzag", "striped"])
@pytest.mark.parametrize("causal", [True, False])
def test_shard_tiles_match_oracle(L, n, T, layout, causal):
    if layout == "zigzag" and L % (2 * n):
        pytest.skip("zigzag needs L % 2n == 0")
    got = binding.shard_tiles(L, n, causal, layout, T)
    assert got == oracle.shard_tiles(L, n, causal, layout, T).tolist()


def test_shard_tiles_workloads():
    assert binding.shard_tiles(8192, 8, True, "contiguous") == [36 + 64 * i for i in range(8)]
    assert binding.shard_tiles(131072, 8, True, "zigzag") == [65600] * 8
    assert binding.shard_tiles(65536, 16, True, "zigzag") == [8208] * 16
    # striped, S = L / n rows per shard in s = S / 128 tiles: every pair of shards meets in a
    # triangle of s (s + 1) / 2 tiles
    assert binding.shard_tiles(131072, 8, True, "striped") == [8 * 128 * 129 // 2] * 8
    assert binding.shard_tiles(65536, 16, True, "striped") == [16 * 32 * 33 // 2] * 16


def test_workspace_sizes(lib):
    assert binding.bwd_workspace_size(1, 32, 8, 65536, 128, torch.float32) >= 32 * 65536 * 4
    assert binding.bwd_workspace_size(1, 32, 8, 65536, 128, torch.bfloat16) >= 32 * 65536 * 129 * 4
    assert lib.ring_attn_fwd_stepwise_workspace_size(1, 2, 1024, 128) >= 2 * 1024 * 128 * 4


def test_ring_step_accumulate_argument_errors(lib):
    """The folded ring step refuses a step outside [0, n_shards) and NULL running buffers before
    any CUDA call."""
    P = ctypes.c_void_p
    ptrs = [P(256)] * 5
    f = lib.ring_attn_ring_step_fwd_accumulate
    assert f(*ptrs, 1, 2, 2, 1024, 128, 4, 4, 1, 1, 1, None) == binding.RA_ERR_INVALID_ARG
    assert "step" in lib.ring_attn_last_error().decode()
    assert f(*ptrs, 1, 2, 2, 1024, 128, 4, -1, 1, 1, 1, None) == binding.RA_ERR_INVALID_ARG
    assert f(*ptrs[:3], None, P(256), 1, 2, 2, 1024, 128, 4, 0, 1, 1, 1, None) == binding.RA_ERR_INVALID_ARG


def test_tile_visits_argument_errors(lib):
    """The counted entry points refuse a NULL counter, and problems off the tensor-core path,
    before any CUDA call."""
    P = ctypes.c_void_p
    ptrs = [P(256)] * 5
    st = lib.ring_attn_fwd_tile_visits(*ptrs, 1, 2, 2, 1024, 128, 4, 1, 1, 1, None, None)
    assert st == binding.RA_ERR_INVALID_ARG
    # chunks of 128 rows take the forward's CUDA-core path (its tensor-core tiles are 256 rows),
    # which does not count tiles
    st = lib.ring_attn_fwd_tile_visits(*ptrs, 1, 2, 2, 1024, 64, 4, 1, 1, 1, P(256), None)
    assert st == binding.RA_ERR_UNSUPPORTED
    assert "tensor-core" in lib.ring_attn_last_error().decode()
    bptrs = [P(256)] * 9
    st = lib.ring_attn_bwd_tile_visits(*bptrs, 0, P(256), 1 << 20, 1, 2, 2, 600, 128, 3, 1, 1, 1,
                                       P(256), None)
    assert st == binding.RA_ERR_UNSUPPORTED
    st = lib.ring_attn_bwd_tile_visits(*bptrs, 0, P(256), 1 << 20, 1, 2, 2, 1024, 128, 4, 1, 1, 1,
                                       None, None)
    assert st == binding.RA_ERR_INVALID_ARG


def test_rope_argument_errors(lib):
    P = ctypes.c_void_p
    # base must be positive and finite; d in {64, 128}; x not NULL -- all before any CUDA call
    assert lib.ring_attn_rope(P(256), 1, 2, 1024, 128, 4, 1, 1, 0.0, 0, None) == binding.RA_ERR_INVALID_ARG
    assert lib.ring_attn_rope(P(256), 1, 2, 1024, 128, 4, 1, 1, float("inf"), 0, None) == binding.RA_ERR_INVALID_ARG
    assert lib.ring_attn_rope(P(256), 1, 2, 1024, 96, 4, 1, 1, 10000.0, 0, None) == binding.RA_ERR_UNSUPPORTED
    assert lib.ring_attn_rope(None, 1, 2, 1024, 128, 4, 1, 1, 10000.0, 0, None) == binding.RA_ERR_INVALID_ARG
    assert lib.ring_attn_rope(P(256), 1, 2, 1020, 128, 4, 1, 1, 10000.0, 0, None) == binding.RA_ERR_INVALID_ARG


def test_ulysses_head_divisibility_and_workspace(lib):
    """Ulysses splits the heads across the shards: H and Hkv must divide by n (checked before any
    CUDA call).  The workspace holds the head-split q, k, v, out and lse."""
    P = ctypes.c_void_p
    ptrs = [P(256)] * 5
    st = lib.ring_attn_ulysses_fwd(*ptrs, 1, 12, 4, 1024, 128, 8, 1, 0, 1, P(256), 1 << 30, None)
    assert st == binding.RA_ERR_INVALID_ARG and "multiples of n_shards" in lib.ring_attn_last_error().decode()
    st = lib.ring_attn_ulysses_fwd(*ptrs, 1, 16, 4, 1024, 128, 8, 1, 0, 1, P(256), 1 << 30, None)
    assert st == binding.RA_ERR_INVALID_ARG  # Hkv = 4 < 8 shards
    st = lib.ring_attn_ulysses_a2a(P(256), P(512), 1, 6, 1024, 128, 4, 0, 1, 0, None)
    assert st == binding.RA_ERR_INVALID_ARG
    st = lib.ring_attn_ulysses_a2a(P(256), P(512), 1, 8, 1024, 3, 4, 0, 1, 0, None)
    assert st == binding.RA_ERR_INVALID_ARG  # 3 bf16 = 6 bytes per row
    B, H, Hkv, L, d = 1, 32, 8, 131072, 128
    want = 2 * B * H * L * d * 2 + 2 * B * Hkv * L * d * 2 + B * H * L * 4
    assert binding.library().ring_attn_ulysses_workspace_size(B, H, Hkv, L, d, 1) == want
    # backward: head-split q, out, dout, k, v, lse, dq, dk, dv, plus the inner backward's workspace
    # for n problems of H/n query heads (float32 gradients here)
    n = 8
    lib = binding.library()
    inner = lib.ring_attn_bwd_workspace_size(n * B, H // n, Hkv // n, L, d, 0)
    want_b = (3 * B * H * L * d * 2 + 2 * B * Hkv * L * d * 2 + B * H * L * 4 + B * H * L * d * 4
              + 2 * B * Hkv * L * d * 4 + inner)
    got_b = lib.ring_attn_ulysses_bwd_workspace_size(B, H, Hkv, L, d, n, 1, 0)
    assert want_b <= got_b <= want_b + 10 * 256
    assert lib.ring_attn_ulysses_bwd_workspace_size(B, 12, Hkv, L, d, n, 1, 0) == 0  # 12 heads over 8


def test_fwd_host_argument_errors(lib):
    P = ctypes.c_void_p
    need = lib.ring_attn_fwd_host_workspace_size(32, 8, 131072, 128, 1)
    # per slot: q and out of 4 heads (2 x 128 MiB), k and v (2 x 32 MiB), lse (2 MiB); two slots
    assert need == 2 * (2 * 4 * 131072 * 128 * 2 + 2 * 131072 * 128 * 2 + 4 * 131072 * 4)
    ptrs = [P(4096)] * 5
    st = lib.ring_attn_fwd_host(P(4096), None, P(4096), P(4096), P(4096), 1, 32, 8, 131072, 128, 8, 1, 1, 1,
                                P(256), need, None)
    assert st == binding.RA_ERR_INVALID_ARG
    st = lib.ring_attn_fwd_host(*ptrs, 1, 32, 8, 131072, 128, 8, 1, 1, 1, P(256), need - 1, None)
    assert st == binding.RA_ERR_INVALID_ARG and "workspace too small" in lib.ring_attn_last_error().decode()


def test_selftest_bounded_wait_argument_errors(lib):
    P = ctypes.c_void_p
    assert lib.ring_attn_selftest_bounded_wait(10, P(256), None) == binding.RA_ERR_INVALID_ARG
    assert lib.ring_attn_selftest_bounded_wait(10**9, P(256), None) == binding.RA_ERR_INVALID_ARG
    assert lib.ring_attn_selftest_bounded_wait(10**6, None, None) == binding.RA_ERR_INVALID_ARG


def test_device_check_reports_its_codes(lib):
    """ring_attn_device_check turns the device status word into a status code (RA_ERR_TIMEOUT when
    a bounded wait ran out; exercised on the GPU by test_gpu_failure_detection).  Without a device it
    says so before touching the word."""
    if torch.cuda.is_available():
        pytest.skip("the GPU side is covered by test_gpu_failure_detection")
    assert lib.ring_attn_device_check(None) == binding.RA_ERR_NO_DEVICE
    st = ctypes.c_uint(7)
    assert lib.ring_attn_device_status(ctypes.byref(st), None) == binding.RA_ERR_NO_DEVICE
    assert st.value == 7  # untouched on failure


def test_block_calls_check_their_arguments(lib):
    """The per-device block calls refuse bad shard indices, flags, counts and pointers before any
    CUDA call (so these run without a GPU)."""
    P = ctypes.c_void_p
    ok16 = P(16)

    def fwd(i=1, j=0, acc=0, L=4096, n=4, ptr=ok16):
        return lib.ring_attn_block_fwd(ptr, ok16, ok16, ok16, ok16, 1, 2, 1, L, 128, n, i, j, acc, 1, 1, 1, None)

    def bwd(i=1, j=0, acc=0):
        return lib.ring_attn_block_bwd(*([ok16] * 9), 1, 2, 1, 4096, 128, 4, i, j, acc, 1, 1, 1, None)

    for st in (fwd(i=4), fwd(j=-1), fwd(acc=2), fwd(L=4100), fwd(ptr=P(8)), fwd(ptr=None), bwd(i=-1), bwd(j=4),
               bwd(acc=3)):
        assert st == binding.RA_ERR_INVALID_ARG
    assert "shard indices" in lib.ring_attn_last_error().decode() or "must be 0 or 1" in lib.ring_attn_last_error().decode()
    LL = ctypes.c_longlong
    assert lib.ring_attn_f32_zero(ok16, LL(-1), None) == binding.RA_ERR_INVALID_ARG
    assert lib.ring_attn_f32_add(ok16, P(8), LL(4), None) == binding.RA_ERR_INVALID_ARG
    assert lib.ring_attn_f32_convert(ok16, ok16, LL(4), 7, None) == binding.RA_ERR_INVALID_ARG
    assert lib.ring_attn_bwd_preprocess(ok16, ok16, ok16, LL(4), 0, 1, None) == binding.RA_ERR_INVALID_ARG
    assert lib.ring_attn_bwd_preprocess_f32out(ok16, ok16, ok16, LL(-1), 128, 1, None) == binding.RA_ERR_INVALID_ARG
    assert lib.ring_attn_bwd_preprocess_f32out(ok16, ok16, ok16, LL(4), 128, 9, None) == binding.RA_ERR_INVALID_ARG
    assert lib.ring_attn_bwd_preprocess_f32out(ok16, P(8), ok16, LL(4), 128, 1, None) == binding.RA_ERR_INVALID_ARG
    assert lib.ring_attn_bwd_preprocess_f32out(None, None, None, LL(0), 128, 1, None) == binding.RA_OK
    # an empty count enqueues nothing and needs no device
    assert lib.ring_attn_f32_zero(None, LL(0), None) == binding.RA_OK
    assert lib.ring_attn_f32_convert(None, None, LL(0), 1, None) == binding.RA_OK


@pytest.mark.parametrize("kw,status", [
    (dict(q=0), binding.RA_ERR_INVALID_ARG),
    (dict(out=8), binding.RA_ERR_INVALID_ARG),
    (dict(d=96), binding.RA_ERR_UNSUPPORTED),
    (dict(L=1026, n=6), binding.RA_ERR_INVALID_ARG),
])
def test_float32_output_calls_check_their_arguments_first(lib, kw, status):
    """ring_attn_fwd_f32out / ring_attn_bwd_f32out share the forward's and the backward's checks."""
    a = dict(q=16, k=16, v=16, out=16, lse=16, B=1, H=2, Hkv=1, L=1024, d=128, n=4, causal=1, layout=1, dtype=1)
    a.update(kw)
    P = ctypes.c_void_p
    assert lib.ring_attn_fwd_f32out(P(a["q"]), P(a["k"]), P(a["v"]), P(a["out"]), P(a["lse"]), a["B"], a["H"],
                                    a["Hkv"], a["L"], a["d"], a["n"], a["causal"], a["layout"], a["dtype"],
                                    None) == status
    ws = 256
    assert lib.ring_attn_bwd_f32out(P(a["q"]), P(a["k"]), P(a["v"]), P(a["out"]), P(a["lse"]), P(16), P(16),
                                    P(16), P(16), 0, P(ws), ctypes.c_size_t(1 << 40), a["B"], a["H"], a["Hkv"],
                                    a["L"], a["d"], a["n"], a["causal"], a["layout"], a["dtype"], None) == status
