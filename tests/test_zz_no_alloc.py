"""qdelta_fwd_static_scratch, the entry point for callers that cannot allocate
device memory at call time (a caller with only input and output pointers and no
device allocator, or a serving loop whose memory is reserved up front and must
not call cudaMalloc mid-step).  Called through the C ABI and checked against
qdelta_fwd, which takes a caller workspace, on two calls in a row.  Both run the
same kernels on the same inputs, so their outputs must agree bit for bit; one of
them is also held to the fp64 oracle at the bf16 tolerance.  The sizes used take
the segment scan, so the library's fixed scratch array is really used."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

REL, ABS = 5e-3, 2e-2          # the bf16 tolerance of the parity tests
STATIC_SCRATCH = 24 << 20      # the library's fixed scratch array


@pytest.fixture(scope="module")
def qd():
    import delta_rule_linear_qdelta_gb300 as m
    from delta_rule_linear_qdelta_gb300 import build
    build.build()
    m.load_library()
    assert torch.cuda.is_available()
    return m


def _dev(x, dtype=torch.bfloat16):
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x)).to("cuda", dtype)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _close(got, ref, what):
    got, ref = got.double().cpu().numpy(), ref.double().cpu().numpy()
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    mx = np.abs(got - ref).max()
    assert rel <= REL and mx <= ABS, f"{what}: rel L2 {rel:.3e}, max abs {mx:.3e}"


def test_static_scratch_matches_workspace_forward_two_calls(qd):
    B, T, H, D = 1, 4096, 2, 128
    need = qd.qdelta_workspace_bytes(B, T, H, D, D)
    assert 0 < need <= STATIC_SCRATCH
    lib = qd.load_library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for seed in (301, 302):                      # two calls in a row, different inputs
        d = synth.qdelta_inputs(B, T, H, D, D, seed=seed, dtype="bf16", mode="qdelta", s0_var=0.01)
        q, k, v = _dev(d["q"]), _dev(d["k"]), _dev(d["v"])
        a, b, lm = _dev(d["alpha"]), _dev(d["beta"]), _dev(d["lam"])
        S0 = _dev(d["S0"], torch.float32)
        o_ref, S_ref = qd.qdelta_fwd(q, k, v, a, b, lm, S0)
        o = torch.empty_like(o_ref)
        S = torch.empty_like(S_ref)
        st = lib.qdelta_fwd_static_scratch(_p(q), _p(k), _p(v), _p(a), _p(b), _p(lm), _p(S0), _p(o), _p(S),
                                           B, T, H, D, D, 64, qd.QD_BF16, stream)
        assert st == qd.QD_OK, qd.qd_last_error()
        assert qd.last_launch_count() == 4       # the segment scan ran on the static scratch
        torch.cuda.synchronize()
        assert qd.qd_device_status() == qd.QD_OK
        assert torch.equal(o, o_ref), f"o (call {seed}) differs from qdelta_fwd's"
        assert torch.equal(S, S_ref), f"S_final (call {seed}) differs from qdelta_fwd's"
        if seed == 301:                          # and against the fp64 oracle
            o64, S64 = oracle.qdelta_fwd(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["lam"], d["S0"])
            _close(o, torch.from_numpy(o64), f"o vs oracle (call {seed})")
            _close(S, torch.from_numpy(S64), f"S_final vs oracle (call {seed})")


def test_static_scratch_rejects_sizes_beyond_its_array(qd):
    B, T, H, D = 1, 4096, 72, 128                # 72 heads in 2 segments: 144 segment-heads
    need = qd.qdelta_workspace_bytes(B, T, H, D, D)
    if need <= STATIC_SCRATCH:
        pytest.skip("this GPU cuts these sizes into fewer segments")
    lib = qd.load_library()
    x = torch.empty(256, dtype=torch.uint8, device="cuda")
    st = lib.qdelta_fwd_static_scratch(_p(x), _p(x), _p(x), None, _p(x), None, None, _p(x), None,
                                       B, T, H, D, D, 64, qd.QD_BF16, None)
    assert st == qd.QD_ERR_WORKSPACE and "24 MiB" in qd.qd_last_error()
