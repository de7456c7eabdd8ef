"""The C-ABI library: it loads without a GPU, exports every symbol the header
declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

import delta_rule_linear_qdelta_gb300 as qd
from delta_rule_linear_qdelta_gb300 import build as qd_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qdelta.h")


@pytest.fixture(scope="module")
def lib():
    qd_build.build()
    return qd.load_library()


def header_functions():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"QD_API\s+[\w\s\*]+?\b(\w+)\s*\(", txt)))


def test_header_declares_the_entry_points():
    names = header_functions()
    assert set(names) == set(qd.EXPORTS), names


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name


def test_null_and_misaligned_pointers_rejected(lib):
    P = ctypes.c_void_p
    good = P(256)
    st = lib.qdelta_fwd(None, good, good, None, good, None, None, good, None,
                        1, 8, 1, 64, 64, 64, qd.QD_BF16, None, 0, None)
    assert st == qd.QD_ERR_ARG and "NULL" in qd.qd_last_error()
    st = lib.qdelta_fwd(P(258), good, good, None, good, None, None, good, None,
                        1, 8, 1, 64, 64, 64, qd.QD_BF16, None, 0, None)
    assert st == qd.QD_ERR_ARG and "aligned" in qd.qd_last_error()
    st = lib.qdelta_step(good, good, good, good, None, None, None, good, 1, 1, 64, 64, qd.QD_BF16, None)
    assert st == qd.QD_ERR_ARG


@pytest.mark.parametrize("dk,dv,chunk,dt,code", [(48, 64, 64, 1, 2), (64, 256, 64, 1, 2), (64, 64, 32, 1, 2),
                                                  (64, 64, 64, 7, 2)])
def test_unsupported_shapes_rejected(lib, dk, dv, chunk, dt, code):
    g = ctypes.c_void_p(256)
    st = lib.qdelta_fwd(g, g, g, None, g, None, None, g, None, 1, 8, 1, dk, dv, chunk, dt, None, 0, None)
    assert st == code, qd.qd_last_error()
    st = lib.qed_fwd(g, g, g, g, g, g, g, None, g, None, 1, 8, 1, dk, dv, chunk, dt, None, 0, None)
    assert st == code, qd.qd_last_error()


def test_negative_sizes_rejected_and_empty_batch_is_a_noop(lib):
    g = ctypes.c_void_p(256)
    assert lib.qdelta_fwd(g, g, g, None, g, None, None, g, None, -1, 8, 1, 64, 64, 64, 1, None, 0, None) == qd.QD_ERR_ARG
    # B = 0: nothing to do, no device call
    assert lib.qdelta_fwd(None, None, None, None, None, None, None, None, None, 0, 8, 4, 64, 64, 64, 1,
                          None, 0, None) == qd.QD_OK
    assert lib.qdelta_step(None, None, None, None, None, None, None, None, 0, 4, 64, 64, 1, None) == qd.QD_OK


def test_python_binding_refuses_cpu_tensors(lib):
    import torch
    x = torch.zeros(1, 4, 1, 16, dtype=torch.bfloat16)
    gt = torch.zeros(1, 4, 1, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        qd.qdelta_fwd(x, x, x, gt, gt, gt)


def _cpu_calls():
    """Every Python entry point, called with CPU tensors of valid shapes and dtypes."""
    import torch
    bf, f32 = torch.bfloat16, torch.float32
    B, T, H, d, N = 1, 4, 1, 16, 2
    x = lambda *s, dt=bf: torch.zeros(*s, dtype=dt)
    tok, gate, st = x(B, T, H, d), x(B, T, H), x(B, H, d, d, dt=f32)
    stok, sgate, sst = x(N, H, d), x(N, H), x(N, H, d, d, dt=f32)
    lam_h = x(H, dt=f32)
    return {
        "qdelta_fwd": lambda: qd.qdelta_fwd(tok, tok, tok, gate, gate, gate, st),
        "qdelta_fwd prologue": lambda: qd.qdelta_fwd(tok, tok, tok, gate, gate, gate, st, prologue=True),
        "qdelta_fwd_static_scratch": lambda: qd.qdelta_fwd_static_scratch(tok, tok, tok, gate, gate, gate, st),
        "qdelta_bwd": lambda: qd.qdelta_bwd(tok, tok, tok, gate, gate, gate, st, tok, st),
        "qdelta_bwd prologue": lambda: qd.qdelta_bwd(tok, tok, tok, gate, gate, gate, st, tok, st, prologue=True),
        "qed_fwd": lambda: qd.qed_fwd(tok, tok, tok, tok, tok, tok, lam_h, st),
        "qed_fwd nogate": lambda: qd.qed_fwd(tok, tok, tok, tok, tok, tok, lam_h, st, variant="nogate"),
        "eda_fwd": lambda: qd.eda_fwd(tok, tok, tok, tok, gate, st),
        "qdelta_step": lambda: qd.qdelta_step(sst, stok, stok, stok, sgate, sgate, sgate),
        "qdelta_step prologue": lambda: qd.qdelta_step(sst, stok, stok, stok, sgate, sgate, sgate, prologue=True),
        "qed_step": lambda: qd.qed_step(sst, stok, stok, stok, stok, stok, stok, lam_h),
    }


@pytest.mark.parametrize("name", sorted(_cpu_calls()))
def test_every_entry_point_refuses_cpu_tensors(lib, name):
    """No entry point has a CPU path: host tensors are refused before any launch."""
    with pytest.raises(ValueError, match="CUDA"):
        _cpu_calls()[name]()


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        qd.load_library(str(tmp_path / "nope.so"))


def test_qed_arms_and_step_arguments_checked(lib):
    g = ctypes.c_void_p(256)
    # unknown arm, rand without z_h, misaligned z_h
    st = lib.qed_fwd_variant(g, g, g, g, g, g, g, None, g, None, 1, 8, 1, 64, 64, 64, qd.QD_BF16, 7, None,
                             None, 0, None)
    assert st == qd.QD_ERR_ARG and "variant" in qd.qd_last_error()
    st = lib.qed_fwd_variant(g, g, g, g, g, g, g, None, g, None, 1, 8, 1, 64, 64, 64, qd.QD_BF16,
                             qd.QED_VARIANTS["rand"], None, None, 0, None)
    assert st == qd.QD_ERR_ARG and "z_h" in qd.qd_last_error()
    st = lib.qed_fwd_variant(g, g, g, g, g, g, g, None, g, None, 1, 8, 1, 64, 64, 64, qd.QD_BF16,
                             qd.QED_VARIANTS["rand"], ctypes.c_void_p(260), None, 0, None)
    assert st == qd.QD_ERR_ARG and "aligned" in qd.qd_last_error()
    # the decode step: NULL gate, unknown arm, unsupported head dim; empty batch is a no-op
    st = lib.qed_step(g, g, g, g, None, g, g, g, g, 1, 1, 64, 64, qd.QD_BF16, 0, None, None)
    assert st == qd.QD_ERR_ARG and "NULL" in qd.qd_last_error()
    st = lib.qed_step(g, g, g, g, g, g, g, g, g, 1, 1, 64, 64, qd.QD_BF16, 9, None, None)
    assert st == qd.QD_ERR_ARG
    st = lib.qed_step(g, g, g, g, g, g, g, g, g, 1, 1, 48, 64, qd.QD_BF16, 0, None, None)
    assert st == qd.QD_ERR_UNSUPPORTED
    st = lib.qed_step(g, g, g, g, g, g, g, g, g, 1, 1, 64, 64, qd.QD_BF16, qd.QED_VARIANTS["rand"], None, None)
    assert st == qd.QD_ERR_ARG and "z_h" in qd.qd_last_error()
    assert lib.qed_step(None, None, None, None, None, None, None, None, None, 0, 4, 64, 64, 1, 0, None,
                        None) == qd.QD_OK


def test_prologue_entry_points_checked(lib):
    g = ctypes.c_void_p(256)
    # missing b_logit, misaligned q_raw, unsupported head dim; empty batch is a no-op
    st = lib.qdelta_fwd_prologue(g, g, g, None, None, None, None, g, None, 1, 8, 1, 64, 64, 64, qd.QD_BF16,
                                 None, 0, None)
    assert st == qd.QD_ERR_ARG and "qdelta_fwd_prologue" in qd.qd_last_error()
    st = lib.qdelta_fwd_prologue(ctypes.c_void_p(258), g, g, None, g, None, None, g, None, 1, 8, 1, 64, 64, 64,
                                 qd.QD_BF16, None, 0, None)
    assert st == qd.QD_ERR_ARG and "aligned" in qd.qd_last_error()
    st = lib.qdelta_fwd_prologue(g, g, g, None, g, None, None, g, None, 1, 8, 1, 48, 64, 64, qd.QD_BF16,
                                 None, 0, None)
    assert st == qd.QD_ERR_UNSUPPORTED
    assert lib.qdelta_fwd_prologue(None, None, None, None, None, None, None, None, None, 0, 8, 4, 64, 64, 64, 1,
                                   None, 0, None) == qd.QD_OK
    st = lib.qdelta_step_prologue(g, g, g, g, None, None, None, g, 1, 1, 64, 64, qd.QD_BF16, None)
    assert st == qd.QD_ERR_ARG and "qdelta_step_prologue" in qd.qd_last_error()
    assert lib.qdelta_step_prologue(None, None, None, None, None, None, None, None, 0, 4, 64, 64, 1,
                                    None) == qd.QD_OK


def test_backward_arguments_checked(lib):
    g = ctypes.c_void_p(256)
    args = lambda **kw: [kw.get(n, g) for n in ("q", "k", "v", "alpha", "beta", "lam", "S0", "dO", "dS",
                                               "dq", "dk", "dv", "dal", "dbe", "dla", "dS0")]
    # missing dbeta, misaligned dq, unsupported head dim, missing workspace
    st = lib.qdelta_bwd(*args(dbe=None), 1, 8, 1, 64, 64, 64, qd.QD_BF16, g, 1 << 30, None)
    assert st == qd.QD_ERR_ARG and "qdelta_bwd" in qd.qd_last_error()
    st = lib.qdelta_bwd(*args(dq=ctypes.c_void_p(260)), 1, 8, 1, 64, 64, 64, qd.QD_BF16, g, 1 << 30, None)
    assert st == qd.QD_ERR_ARG and "aligned" in qd.qd_last_error()
    st = lib.qdelta_bwd(*args(), 1, 8, 1, 48, 64, 64, qd.QD_BF16, g, 1 << 30, None)
    assert st == qd.QD_ERR_UNSUPPORTED
    need = lib.qdelta_bwd_workspace_bytes(1, 8, 1, 64, 64, 64, qd.QD_BF16)
    assert need == 2 * 64 * 64 * 4
    st = lib.qdelta_bwd(*args(), 1, 8, 1, 64, 64, 64, qd.QD_BF16, g, need - 16, None)
    assert st == qd.QD_ERR_WORKSPACE
    assert lib.qdelta_bwd_workspace_bytes(2, 130, 3, 128, 64, 64, qd.QD_F32) == 2 * 2 * 3 * 3 * 64 * 128 * 4
    assert lib.qdelta_bwd_workspace_bytes(2, 0, 3, 128, 64, 64, qd.QD_F32) == 0
    # empty batch: no device call
    assert lib.qdelta_bwd(*([None] * 16), 0, 8, 4, 64, 64, 64, 1, None, 0, None) == qd.QD_OK


def test_eda_arguments_checked(lib):
    g = ctypes.c_void_p(256)
    st = lib.eda_fwd(g, g, g, None, None, None, g, None, 1, 8, 1, 64, 64, 64, qd.QD_BF16, g, 1 << 30, None)
    assert st == qd.QD_ERR_ARG and "eda_fwd" in qd.qd_last_error()
    st = lib.eda_fwd(g, g, g, g, ctypes.c_void_p(258), None, g, None, 1, 8, 1, 64, 64, 64, qd.QD_BF16, g, 1 << 30,
                     None)
    assert st == qd.QD_ERR_ARG and "aligned" in qd.qd_last_error()
    assert lib.eda_workspace_bytes(1, 8, 1, 64, 64, 64, qd.QD_BF16) == 0
    st = lib.eda_fwd(g, g, g, g, None, None, g, None, 1, 8, 1, 48, 64, 64, qd.QD_BF16, None, 0, None)
    assert st == qd.QD_ERR_UNSUPPORTED
    assert lib.eda_fwd(None, None, None, None, None, None, None, None, 0, 8, 4, 64, 64, 64, 1, None, 0,
                       None) == qd.QD_OK


def test_bounded_wait_selftest_limit_checked(lib):
    assert lib.qd_selftest_bounded_wait(0, None) == qd.QD_ERR_ARG
    assert lib.qd_selftest_bounded_wait(2000000, None) == qd.QD_ERR_ARG


def test_prologue_backward_arguments_checked(lib):
    g = ctypes.c_void_p(256)
    args = lambda **kw: [kw.get(n, g) for n in ("q", "k", "v", "a", "b", "l", "S0", "dO", "dS",
                                               "dq", "dk", "dv", "da", "db", "dl", "dS0")]
    st = lib.qdelta_bwd_prologue(*args(b=None), 1, 8, 1, 64, 64, 64, qd.QD_BF16, g, 1 << 30, None)
    assert st == qd.QD_ERR_ARG and "qdelta_bwd_prologue" in qd.qd_last_error()
    need = lib.qdelta_bwd_prologue_workspace_bytes(1, 8, 1, 64, 64, 64, qd.QD_BF16)
    assert need > lib.qdelta_bwd_workspace_bytes(1, 8, 1, 64, 64, 64, qd.QD_BF16)
    st = lib.qdelta_bwd_prologue(*args(), 1, 8, 1, 64, 64, 64, qd.QD_BF16, g, need - 16, None)
    assert st == qd.QD_ERR_WORKSPACE
    assert lib.qdelta_bwd_prologue(*([None] * 16), 0, 8, 4, 64, 64, 64, 1, None, 0, None) == qd.QD_OK


def test_static_scratch_checks_arguments_before_any_device_call(lib):
    """Sizes that would take the segment scan (and so the fixed scratch array) still
    get QD_ERR_ARG for a NULL or misaligned pointer, from the host checks alone."""
    P = ctypes.c_void_p
    g = P(256)
    st = lib.qdelta_fwd_static_scratch(None, g, g, None, g, None, None, g, None, 1, 4096, 2, 128, 128, 64,
                                       qd.QD_BF16, None)
    assert st == qd.QD_ERR_ARG and "NULL" in qd.qd_last_error()
    st = lib.qdelta_fwd_static_scratch(g, g, P(264), None, g, None, None, g, None, 1, 4096, 2, 128, 128, 64,
                                       qd.QD_BF16, None)
    assert st == qd.QD_ERR_ARG and "aligned" in qd.qd_last_error()
    st = lib.qdelta_fwd_static_scratch(g, g, g, None, g, None, None, g, None, 1, 4096, 2, 128, 128, 32,
                                       qd.QD_BF16, None)
    assert st == qd.QD_ERR_UNSUPPORTED


@pytest.mark.parametrize("B,T,H", [(2, 130, 3), (8, 2048, 16), (4, 4096, 8)])
def test_qed_workspace_covers_derived_operands_and_counters(lib, B, T, H):
    """The tensor-core QED path keeps four bf16 [B][T][H][128] operand arrays, e^{G_C} per
    chunk and channel in fp32, and one 32-bit hand-over counter per chunk and stream
    (rounded up to 256 bytes); these sizes take no segment states."""
    nch = (T + 63) // 64
    derived = 4 * B * T * H * 128 * 2 + B * H * nch * 128 * 4
    counters = (B * H * nch * 4 + 255) // 256 * 256
    assert lib.qed_workspace_bytes(B, T, H, 128, 128, 64, qd.QD_BF16) == derived + counters
    # the CUDA-core paths (fp32, head dim 64) and a chunk other than 64 need none
    assert lib.qed_workspace_bytes(B, T, H, 128, 128, 64, qd.QD_F32) == 0
    assert lib.qed_workspace_bytes(B, T, H, 64, 64, 64, qd.QD_BF16) == 0
    assert lib.qed_workspace_bytes(B, T, H, 128, 128, 32, qd.QD_BF16) == 0


def test_eda_workspace_for_the_tensor_core_path(lib):
    """bf16 at d_k = d_v = 128 takes the tensor-core path: the fp16 sub-token keys
    [B][2T+1][H][128], three compact fp16 [B][T][H][128] arrays (r_t, v_t, o'_2t), the
    sub-tokens' bf16 strengths and c_t (fp32 [B][T][H]), each rounded up to 256 bytes; a
    call without it is refused before any device work."""
    r = lambda n: (n + 255) // 256 * 256
    for B, T, H in [(2, 150, 2), (8, 2048, 16)]:
        n = B * (2 * T + 1) * H
        want = r(n * 128 * 2) + 3 * r(B * T * H * 128 * 2) + r(n * 2) + r(B * T * H * 4)
        assert lib.eda_workspace_bytes(B, T, H, 128, 128, 64, qd.QD_BF16) == want
        assert lib.eda_workspace_bytes(B, T, H, 128, 128, 64, qd.QD_F32) == 0
        assert lib.eda_workspace_bytes(B, T, H, 128, 64, 64, qd.QD_BF16) == 0
    g = ctypes.c_void_p(256)
    st = lib.eda_fwd(g, g, g, g, None, None, g, None, 1, 8, 1, 128, 128, 64, qd.QD_BF16, None, 0, None)
    assert st == qd.QD_ERR_WORKSPACE and "eda_fwd" in qd.qd_last_error()
    need = lib.eda_workspace_bytes(1, 8, 1, 128, 128, 64, qd.QD_BF16)
    st = lib.eda_fwd(g, g, g, g, None, None, g, None, 1, 8, 1, 128, 128, 64, qd.QD_BF16, g, need - 16, None)
    assert st == qd.QD_ERR_WORKSPACE
