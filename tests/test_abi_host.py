"""Host-side checks of the C ABI (no GPU): the library loads, exports every
function include/q4.h declares, computes the packed size exactly like the
oracle's closed form, and rejects bad arguments before touching a device."""
import ctypes
import os
import re

import pytest

import bit_row_speculative_gb300 as q4
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(q4_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_exports_every_declared_symbol():
    lib = q4.lib()
    declared = declared_functions()
    assert "q4_matmul" in declared and "q4_packed_bytes" in declared
    for name in declared:
        assert hasattr(lib, name), name
    assert declared == set(q4.SYMBOLS)


@pytest.mark.parametrize("N,K", [(256, 512), (14336, 5120), (34816, 5120), (5120, 17408), (16640, 5120),
                                 (5120, 6144), (248320, 5120), (1, 64), (7, 192), (0, 64), (3, 100),
                                 (1, 0), (1 << 40, 1 << 40), ((1 << 58) + 1, 64)])
def test_packed_bytes_matches_oracle(N, K):
    assert q4.packed_bytes(N, K) == oracle.packed_bytes(N, K)


def test_status_strings():
    for code, name in [(0, "Q4_OK"), (1, "Q4_ERR_INVALID_ARG"), (6, "Q4_ERR_TIMEOUT"), (7, "Q4_ERR_OVERFLOW")]:
        assert q4.status_name(code) == name


@pytest.mark.parametrize("args,status", [
    ((0, 16, 1, 256, 512, 16), q4.Q4_ERR_INVALID_ARG),        # null x
    ((16, 0, 1, 256, 512, 16), q4.Q4_ERR_INVALID_ARG),        # null W
    ((16, 16, 1, 256, 512, 0), q4.Q4_ERR_INVALID_ARG),        # null y
    ((16, 16, 0, 256, 512, 16), q4.Q4_ERR_INVALID_ARG),       # M = 0
    ((16, 16, 33, 256, 512, 16), q4.Q4_ERR_INVALID_ARG),      # M = 33
    ((16, 16, 1, 0, 512, 16), q4.Q4_ERR_INVALID_ARG),         # N = 0
    ((16, 16, 1, 256, 96, 16), q4.Q4_ERR_UNSUPPORTED_SHAPE),  # K % 64 != 0
    ((16, 16, 1, 256, 0, 16), q4.Q4_ERR_UNSUPPORTED_SHAPE),   # K = 0
    ((16, 16, 1, 1 << 40, 1 << 40, 16), q4.Q4_ERR_OVERFLOW),  # packed size overflows
    ((8, 16, 1, 256, 512, 16), q4.Q4_ERR_MISALIGNED),         # x misaligned
    ((16, 24, 1, 256, 512, 16), q4.Q4_ERR_MISALIGNED),        # W misaligned
])
def test_argument_errors_return_before_launch(args, status):
    lib = q4.lib()
    rc = lib.q4_matmul(*args, None)
    assert rc == status, (rc, lib.q4_last_error())
    assert lib.q4_last_error().decode() != ""


def _layers(spec):
    """ctypes q4_layer array from (W address, N, K, glue) tuples."""
    arr = (q4.Layer * len(spec))()
    for i, (w, N, K, g) in enumerate(spec):
        arr[i] = q4.Layer(w, N, K, g)
    return arr


def test_decode_workspace_size():
    lib = q4.lib()
    spec = [(16, 2048, 512, q4.GLUE_SWIGLU_RMSNORM), (16, 1280, 1024, q4.GLUE_RMSNORM), (16, 300, 576, q4.GLUE_NONE)]
    arr = _layers(spec)
    need = lib.q4_decode_step_workspace_bytes(ctypes.addressof(arr), 3, 16)
    # widest intermediate y: 16 x 2048 fp32; widest intermediate x: 16 x 1024 bf16 (each rounded to 256 bytes)
    assert need == 16 * 2048 * 4 + 16 * 1024 * 2
    assert lib.q4_decode_step_workspace_bytes(ctypes.addressof(arr), 1, 16) == 0
    assert lib.q4_decode_step_workspace_bytes(None, 3, 16) == 0
    assert lib.q4_decode_step_workspace_bytes(ctypes.addressof(arr), 3, 33) == 0


@pytest.mark.parametrize("spec,ws,status", [
    ([(16, 2000, 512, q4.GLUE_SWIGLU_RMSNORM), (16, 300, 1000, q4.GLUE_NONE)], 1 << 20,
     q4.Q4_ERR_UNSUPPORTED_SHAPE),                                              # K of layer 1 not a multiple of 64
    ([(16, 2048, 512, q4.GLUE_SWIGLU_RMSNORM), (16, 300, 512, q4.GLUE_NONE)], 1 << 20,
     q4.Q4_ERR_INVALID_ARG),                                                    # SwiGLU needs N == 2 * next K
    ([(16, 2048, 512, q4.GLUE_RMSNORM), (16, 300, 4096, q4.GLUE_NONE)], 1 << 20,
     q4.Q4_ERR_INVALID_ARG),                                                    # RMSNORM: next K > N
    ([(16, 2048, 512, q4.GLUE_NONE), (16, 300, 512, q4.GLUE_NONE)], 1 << 20,
     q4.Q4_ERR_INVALID_ARG),                                                    # no glue between layers
    ([(16, 2048, 512, 7), (16, 300, 512, q4.GLUE_NONE)], 1 << 20,
     q4.Q4_ERR_INVALID_ARG),                                                    # unknown glue kind
    ([(16, 2048, 512, q4.GLUE_RMSNORM), (16, 300, 512, q4.GLUE_NONE)], 64,
     q4.Q4_ERR_INVALID_ARG),                                                    # workspace too small
    ([(16, 2048, 512, q4.GLUE_RMSNORM), (24, 300, 512, q4.GLUE_NONE)], 1 << 20,
     q4.Q4_ERR_MISALIGNED),                                                     # W of layer 1 misaligned
])
def test_decode_step_rejects_bad_lists_before_launch(spec, ws, status):
    lib = q4.lib()
    buf = ctypes.create_string_buffer(256)
    p = (ctypes.addressof(buf) + 15) & ~15
    arr = _layers([(p if w == 16 else p + 8, N, K, g) for w, N, K, g in spec])
    rc = lib.q4_decode_step(ctypes.addressof(arr), len(spec), p, 4, p, ws, p, None)
    assert rc == status, (rc, lib.q4_last_error())
    assert lib.q4_last_error().decode() != ""


@pytest.mark.parametrize("M,n_prev,K,kind,status", [
    (4, 640, 700, q4.GLUE_RMSNORM, q4.Q4_ERR_INVALID_ARG),              # K > N_prev
    (4, 640, 300, q4.GLUE_SWIGLU_RMSNORM, q4.Q4_ERR_INVALID_ARG),       # N_prev != 2K
    (4, 640, 320, 3, q4.Q4_ERR_INVALID_ARG),                            # unknown kind
    (0, 640, 320, q4.GLUE_RMSNORM, q4.Q4_ERR_INVALID_ARG),              # M = 0
    (4, 640, 100, q4.GLUE_RMSNORM, q4.Q4_ERR_UNSUPPORTED_SHAPE),        # K not a multiple of 64
])
def test_glue_rejects_bad_arguments(M, n_prev, K, kind, status):
    lib = q4.lib()
    buf = ctypes.create_string_buffer(64)
    p = (ctypes.addressof(buf) + 15) & ~15
    assert lib.q4_glue(p, M, n_prev, K, kind, p, None) == status


@pytest.mark.parametrize("limit", [0, -5, (1 << 32) + 1])
def test_wait_check_rejects_bad_limits(limit):
    lib = q4.lib()
    assert lib.q4_check_wait_timeout(limit, None) == q4.Q4_ERR_INVALID_ARG
    assert "limit_cycles" in lib.q4_last_error().decode()


@pytest.mark.parametrize("M,N,k,T,p,align,status", [
    (0, 100, 8, 1.0, 1.0, 0, q4.Q4_ERR_INVALID_ARG),
    (33, 100, 8, 1.0, 1.0, 0, q4.Q4_ERR_INVALID_ARG),
    (2, 100, 0, 1.0, 1.0, 0, q4.Q4_ERR_INVALID_ARG),
    (2, 100, 33, 1.0, 1.0, 0, q4.Q4_ERR_INVALID_ARG),
    (2, 5, 8, 1.0, 1.0, 0, q4.Q4_ERR_INVALID_ARG),
    (2, 100, 8, 0.0, 1.0, 0, q4.Q4_ERR_INVALID_ARG),
    (2, 100, 8, float("nan"), 1.0, 0, q4.Q4_ERR_INVALID_ARG),
    (2, 100, 8, 1.0, 0.0, 0, q4.Q4_ERR_INVALID_ARG),
    (2, (1 << 20) + 1, 8, 1.0, 1.0, 0, q4.Q4_ERR_UNSUPPORTED_SHAPE),
    (2, 100, 8, 1.0, 1.0, 4, q4.Q4_ERR_MISALIGNED),
])
def test_topk_rejects_bad_arguments(M, N, k, T, p, align, status):
    lib = q4.lib()
    rc = lib.q4_topk_probs(16 + align, M, N, k, T, p, 16, 16, None)
    assert rc == status, (rc, lib.q4_last_error())


@pytest.mark.parametrize("V,R,rows,align,status", [
    (0, 256, 7, 0, q4.Q4_ERR_INVALID_ARG),
    (1 << 31, 256, 7, 0, q4.Q4_ERR_INVALID_ARG),
    (100, 0, 7, 0, q4.Q4_ERR_UNSUPPORTED_SHAPE),
    (100, 12, 7, 0, q4.Q4_ERR_UNSUPPORTED_SHAPE),
    (100, 264, 7, 0, q4.Q4_ERR_UNSUPPORTED_SHAPE),
    (100, 256, 0, 0, q4.Q4_ERR_INVALID_ARG),
    (100, 256, (1 << 20) + 1, 0, q4.Q4_ERR_INVALID_ARG),
    (100, 256, 7, 8, q4.Q4_ERR_MISALIGNED),
])
def test_edges_rejects_bad_arguments(V, R, rows, align, status):
    lib = q4.lib()
    rc = lib.q4_draft_select_edges(16 + align, 16, V, R, 16, 16, 16, rows, 16, None)
    assert rc == status, (rc, lib.q4_last_error())


def test_edges_rejects_null_pointers():
    lib = q4.lib()
    assert lib.q4_draft_select_edges(16, None, 100, 256, 16, 16, 16, 7, 16, None) == q4.Q4_ERR_INVALID_ARG


def test_status_names_cover_every_code():
    lib = q4.lib()
    for code in range(0, 9):
        assert lib.q4_status_string(code).decode().startswith("Q4_")
        assert lib.q4_status_string(code).decode() != "Q4_ERR_UNKNOWN"


def test_noalloc_rejects_more_than_16_rows():
    lib = q4.lib()
    rc = lib.q4_matmul_noalloc(16, 16, 17, 256, 512, 16, None)
    assert rc == q4.Q4_ERR_INVALID_ARG, (rc, lib.q4_last_error())


def test_fused_head_rejects_bad_arguments():
    lib = q4.lib()
    ok = (16, 16, 4, 256, 512, 8, 1.0, 1.0, 16, 16, None)
    assert lib.q4_lm_head_topk(*ok[:2], 33, *ok[3:]) == q4.Q4_ERR_INVALID_ARG            # M = 33
    assert lib.q4_lm_head_topk(*ok[:5], 0, *ok[6:]) == q4.Q4_ERR_INVALID_ARG             # top_k = 0
    assert lib.q4_lm_head_topk(*ok[:3], 4, *ok[4:]) == q4.Q4_ERR_INVALID_ARG             # N < top_k
    assert lib.q4_lm_head_topk(*ok[:4], 96, *ok[5:]) == q4.Q4_ERR_UNSUPPORTED_SHAPE      # K % 64
    assert lib.q4_lm_head_topk(*ok[:6], 0.0, *ok[7:]) == q4.Q4_ERR_INVALID_ARG           # temperature
    assert lib.q4_lm_head_topk(*ok[:8], 24, *ok[9:]) == q4.Q4_ERR_MISALIGNED             # idx
    assert lib.q4_lm_head_topk(None, *ok[1:]) == q4.Q4_ERR_INVALID_ARG
