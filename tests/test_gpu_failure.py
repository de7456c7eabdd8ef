"""Failure detection on the GPU without a GPU fault.

A bounded wait that can never complete (an mbarrier nothing arrives on) must give up
after its limit, record the timeout, and leave the context usable: the next status
query reports QD_ERR_TIMEOUT once, and the library's kernels still compute correctly
afterwards.  No trap, no fault, no unbounded spin is involved.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qd():
    import delta_rule_linear_qdelta_gb300 as m
    from delta_rule_linear_qdelta_gb300 import build
    build.build()
    m.load_library()
    assert torch.cuda.is_available()
    return m


def test_bounded_wait_gives_up_and_context_stays_usable(qd):
    lib = qd.load_library()
    assert qd.qd_device_status() == qd.QD_OK
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.qd_selftest_bounded_wait(20000, stream) == qd.QD_OK      # a 20 ms limit
    assert qd.qd_device_status() == qd.QD_ERR_TIMEOUT
    assert "bounded wait" in qd.qd_last_error()
    assert qd.qd_device_status() == qd.QD_OK                             # reported once, then cleared
    d = synth.qdelta_inputs(1, 150, 2, 128, 128, seed=91, dtype="bf16", mode="qdelta", s0_var=0.01)
    cu = lambda x, dt=torch.bfloat16: None if x is None else torch.from_numpy(np.ascontiguousarray(x)).to("cuda", dt)
    o, S = qd.qdelta_fwd(cu(d["q"]), cu(d["k"]), cu(d["v"]), cu(d["alpha"]), cu(d["beta"]), cu(d["lam"]),
                         cu(d["S0"], torch.float32))
    assert qd.qd_device_status() == qd.QD_OK
    o_ref, S_ref = oracle.qdelta_fwd(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["lam"], d["S0"])
    rel = np.linalg.norm(o.float().cpu().numpy() - o_ref) / np.linalg.norm(o_ref)
    assert rel <= 5e-3
