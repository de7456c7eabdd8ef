"""GPU vs oracle parity, through the C ABI (via the thin binding).

Tolerances (element by element against the fp64 oracle on identical inputs):
  bf16 inputs, fp32 accumulation: relative L2 <= 5e-3 and max abs <= 2e-2
  fp32 path:                       relative L2 <= 1e-5
Small cases compare every output; the full-size workloads run on the GPU in the
same launch configuration the bench times and compare every (b, h) stream over
the full sequence, stream by stream and as a whole.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

BF16_REL, BF16_ABS, F32_REL = 5e-3, 2e-2, 1e-5


@pytest.fixture(scope="module")
def qd():
    import delta_rule_linear_qdelta_gb300 as m
    from delta_rule_linear_qdelta_gb300 import build
    build.build()
    m.load_library()
    assert torch.cuda.is_available()
    return m


def dev(x, dtype=torch.bfloat16):
    if x is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(x)).to("cuda", dtype)


def tdt(d):
    return torch.bfloat16 if d["dtype"] == "bf16" else torch.float32


def check(got, ref, dtype, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    mx = np.abs(got - ref).max() if got.size else 0.0
    if dtype == "bf16":
        assert rel <= BF16_REL and mx <= BF16_ABS, f"{what}: rel L2 {rel:.3e}, max abs {mx:.3e}"
    else:
        assert rel <= F32_REL, f"{what}: rel L2 {rel:.3e}, max abs {mx:.3e}"
    return rel, mx


def run_qdelta(qd, d):
    dt = tdt(d)
    o, S = qd.qdelta_fwd(dev(d["q"], dt), dev(d["k"], dt), dev(d["v"], dt), dev(d["alpha"], dt),
                         dev(d["beta"], dt), dev(d["lam"], dt), dev(d["S0"], torch.float32))
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), S.cpu().numpy()


def run_qed(qd, d, variant="full"):
    dt = tdt(d)
    z = dev(d["z"], torch.float32) if variant == "rand" else None
    o, S = qd.qed_fwd(dev(d["q"], dt), dev(d["k"], dt), dev(d["v"], dt), dev(d["g"], dt), dev(d["b"], dt),
                      dev(d["w"], dt), dev(d["lam_h"], torch.float32), dev(d["S0"], torch.float32),
                      variant=variant, z=z)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), S.cpu().numpy()


def sel(x, pairs, gate=False):
    """Stack streams (b, h) of [B,T,H,...] into [n,T,1,...] for the oracle."""
    if x is None:
        return None
    return np.stack([x[b, :, h] for b, h in pairs])[:, :, None]


# ------------------------------------------------------------------ Q-Delta

def test_tiny_fp32_full(qd):
    name, d = synth.tiny_fp32()
    o, S = run_qdelta(qd, d)
    o_ref, S_ref = oracle.qdelta_fwd(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["lam"], d["S0"])
    check(o, o_ref, "f32", name + " o")
    check(S, S_ref, "f32", name + " S")


@pytest.mark.parametrize("mode", ["qdelta", "gdn", "deltanet"])
def test_bf16_small_all_outputs(qd, mode):
    d = synth.qdelta_inputs(2, 200, 3, 128, 128, seed=21, dtype="bf16", mode=mode, s0_var=0.01)
    o, S = run_qdelta(qd, d)
    o_ref, S_ref = oracle.qdelta_fwd(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["lam"], d["S0"])
    check(o, o_ref, "bf16", f"{mode} o")
    check(S, S_ref, "bf16", f"{mode} S")


@pytest.mark.parametrize("alpha_mu", [-0.45, 0.3, 2.0])
def test_qdelta_strong_decay(qd, alpha_mu):
    """Log-decay per token about -0.5, -0.85 and -2.1 (chunk sums near -31, -55 and
    -136): chunks on both sides of the tensor-core kernel's switch between folding
    kappa into Z^T and scaling K, and past the range where e^{-l_i} stays finite."""
    d = synth.qdelta_inputs(2, 200, 3, 128, 128, seed=23, dtype="bf16", mode="qdelta", alpha_mu=alpha_mu,
                            s0_var=0.01)
    o, S = run_qdelta(qd, d)
    o_ref, S_ref = oracle.qdelta_fwd(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["lam"], d["S0"])
    check(o, o_ref, "bf16", f"strong decay {alpha_mu} o")
    check(S, S_ref, "bf16", f"strong decay {alpha_mu} S")


@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 100, 191])
@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_ragged_lengths(qd, T, dt):
    d = synth.qdelta_inputs(1, T, 2, 128, 128, seed=30 + T, dtype=dt, mode="qdelta", s0_var=0.01)
    o, S = run_qdelta(qd, d)
    o_ref, S_ref = oracle.qdelta_fwd(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["lam"], d["S0"])
    check(o, o_ref, dt, f"T={T} o")
    check(S, S_ref, dt, f"T={T} S")


@pytest.mark.parametrize("dk,dv", [(16, 16), (32, 64), (64, 32), (64, 64), (128, 64), (64, 128)])
def test_head_dims_fp32(qd, dk, dv):
    d = synth.qdelta_inputs(2, 130, 2, dk, dv, seed=40 + dk + dv, dtype="f32", mode="qdelta", s0_var=0.01)
    o, S = run_qdelta(qd, d)
    o_ref, S_ref = oracle.qdelta_fwd(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["lam"], d["S0"])
    check(o, o_ref, "f32", f"dk={dk} dv={dv} o")
    check(S, S_ref, "f32", f"dk={dk} dv={dv} S")


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 64), (64, 128)])
def test_head_dims_bf16(qd, dk, dv):
    d = synth.qdelta_inputs(2, 150, 2, dk, dv, seed=45 + dk + dv, dtype="bf16", mode="qdelta", s0_var=0.01)
    o, S = run_qdelta(qd, d)
    o_ref, S_ref = oracle.qdelta_fwd(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["lam"], d["S0"])
    check(o, o_ref, "bf16", f"dk={dk} dv={dv} o")
    check(S, S_ref, "bf16", f"dk={dk} dv={dv} S")


def check_every_stream(o, o_ref, S, S_ref, name):
    """Each (b, h) stream of o [B,T,H,dv] and S [B,H,dv,dk] on its own, then the whole:
    an error confined to one CTA's stream cannot hide in the others' norm."""
    Bn, _, Hn, _ = o.shape
    for b in range(Bn):
        for h in range(Hn):
            check(o[b, :, h], o_ref[b, :, h], "bf16", f"{name} o stream (b={b}, h={h})")
            check(S[b, h], S_ref[b, h], "bf16", f"{name} S stream (b={b}, h={h})")
    check(o, o_ref, "bf16", name + " o")
    check(S, S_ref, "bf16", name + " S")


@pytest.mark.parametrize("mode", ["qdelta", "gdn", "deltanet"])
def test_layer_1p3b_full_size_every_stream(qd, mode):
    """B=8, H=16, T=2048, d=128 bf16: the benchmarked workload in the launch
    configuration the bench times; all 128 streams against the oracle."""
    name, d = synth.layer_1p3b(mode)
    o, S = run_qdelta(qd, d)
    o_ref, S_ref = oracle.qdelta_fwd(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["lam"])
    check_every_stream(o, o_ref, S, S_ref, name)


def test_long_context_full_size_every_stream(qd):
    """B=1, H=16, T=32768, mean alpha 0.995, S0 ~ N(0, 0.01) (the segment scan); all
    16 heads against the oracle."""
    name, d = synth.long_context()
    o, S = run_qdelta(qd, d)
    o_ref, S_ref = oracle.qdelta_fwd(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["lam"], d["S0"])
    check_every_stream(o, o_ref, S, S_ref, name)


@pytest.mark.parametrize("mode", ["qdelta", "deltanet"])
def test_segmented_long_sequence_all_outputs(qd, mode):
    """B=1, H=2, T=4096: few streams and a long sequence take the segment scan
    (several segments in parallel, stitched by their linear state maps)."""
    d = synth.qdelta_inputs(1, 4096, 2, 128, 128, seed=55, dtype="bf16", mode=mode, s0_var=0.01)
    assert qd.qdelta_workspace_bytes(1, 4096, 2, 128, 128) > 0
    o, S = run_qdelta(qd, d)
    assert qd.last_launch_count() == 4
    o_ref, S_ref = oracle.qdelta_fwd(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["lam"], d["S0"])
    check(o, o_ref, "bf16", f"segmented {mode} o")
    check(S, S_ref, "bf16", f"segmented {mode} S")


def test_split_call_carries_state_in_place(qd):
    """fwd(T1) then fwd(T2, S0 = S_T1) equals one fwd(T1+T2); S0 aliases S_final."""
    d = synth.qdelta_inputs(2, 300, 2, 128, 128, seed=50, dtype="bf16", mode="qdelta", s0_var=0.01)
    dt = torch.bfloat16
    o_ref, S_ref = oracle.qdelta_fwd(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["lam"], d["S0"])
    S = dev(d["S0"], torch.float32)
    outs = []
    for a, b in ((0, 100), (100, 300)):   # split at a non-multiple of the chunk
        sl = lambda x: None if x is None else x[:, a:b]
        o, _ = qd.qdelta_fwd(dev(sl(d["q"]), dt), dev(sl(d["k"]), dt), dev(sl(d["v"]), dt),
                             dev(sl(d["alpha"]), dt), dev(sl(d["beta"]), dt), dev(sl(d["lam"]), dt), S, S_final=S)
        outs.append(o.float().cpu().numpy())
    torch.cuda.synchronize()
    check(np.concatenate(outs, axis=1), o_ref, "bf16", "split o")
    check(S.cpu().numpy(), S_ref, "bf16", "split S")


def test_empty_sequence_and_batch(qd):
    S0 = torch.randn(2, 3, 64, 64, device="cuda")
    z = torch.empty(2, 0, 3, 64, device="cuda", dtype=torch.bfloat16)
    zg = torch.empty(2, 0, 3, device="cuda", dtype=torch.bfloat16)
    o, S = qd.qdelta_fwd(z, z, z, zg, zg, zg, S0)
    torch.cuda.synchronize()
    assert o.shape == (2, 0, 3, 64) and torch.equal(S, S0)
    o, S = qd.qdelta_fwd(z, z, z, None, zg, None, None)
    torch.cuda.synchronize()
    assert torch.count_nonzero(S) == 0


def test_deterministic(qd):
    d = synth.qdelta_inputs(1, 300, 4, 128, 128, seed=60, dtype="bf16", mode="qdelta")
    o1, S1 = run_qdelta(qd, d)
    o2, S2 = run_qdelta(qd, d)
    assert np.array_equal(o1, o2) and np.array_equal(S1, S2)


# ---------------------------------------------------------------------- QED

@pytest.mark.parametrize("T,dt", [(1, "bf16"), (70, "bf16"), (200, "bf16"), (130, "f32")])
def test_qed_small_all_outputs(qd, T, dt):
    d = synth.qed_inputs(2, T, 2, 128, 128, seed=70 + T, dtype=dt, s0_var=0.01)
    o, S = run_qed(qd, d)
    o_ref, S_ref = oracle.qed_fwd(d["q"], d["k"], d["v"], d["g"], d["b"], d["w"], d["lam_h"], d["S0"])
    check(o, o_ref, dt, f"qed T={T} o")
    check(S, S_ref, dt, f"qed T={T} S")


@pytest.mark.parametrize("B,H", [(2, 2), (1, 160)])
def test_qed_fused_and_two_launch_paths(qd, B, H):
    # One cooperative launch (the derive step on the SMs the B*H chains leave free) when
    # B*H + 8 <= SMs; the derive kernel and then the chain kernel otherwise.
    d = synth.qed_inputs(B, 130, H, 128, 128, seed=90 + H, dtype="bf16", s0_var=0.01)
    o, S = run_qed(qd, d)
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    assert qd.last_launch_count() == (1 if B * H + 8 <= nsm else 2)
    o_ref, S_ref = oracle.qed_fwd(d["q"], d["k"], d["v"], d["g"], d["b"], d["w"], d["lam_h"], d["S0"])
    check(o, o_ref, "bf16", f"qed B={B} H={H} o")
    check(S, S_ref, "bf16", f"qed B={B} H={H} S")


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 64)])
def test_qed_head_dims_bf16(qd, dk, dv):
    d = synth.qed_inputs(2, 150, 2, dk, dv, seed=75 + dk + dv, dtype="bf16", s0_var=0.01)
    o, S = run_qed(qd, d)
    o_ref, S_ref = oracle.qed_fwd(d["q"], d["k"], d["v"], d["g"], d["b"], d["w"], d["lam_h"], d["S0"])
    check(o, o_ref, "bf16", f"qed dk={dk} dv={dv} o")
    check(S, S_ref, "bf16", f"qed dk={dk} dv={dv} S")


def test_qed_strong_decay(qd):
    """Per-channel log-decay near -0.5 per token (about -32 summed over a chunk): the
    factored decay of the tensor-core kernel still inside its fp32 range."""
    d = synth.qed_inputs(2, 200, 2, 128, 128, seed=78, dtype="bf16", g_mu=-0.3, s0_var=0.01)
    o, S = run_qed(qd, d)
    o_ref, S_ref = oracle.qed_fwd(d["q"], d["k"], d["v"], d["g"], d["b"], d["w"], d["lam_h"], d["S0"])
    check(o, o_ref, "bf16", "qed strong decay o")
    check(S, S_ref, "bf16", "qed strong decay S")


def test_qed_split_call_carries_state_in_place(qd):
    d = synth.qed_inputs(2, 300, 2, 128, 128, seed=79, dtype="bf16", s0_var=0.01)
    bf = torch.bfloat16
    o_ref, S_ref = oracle.qed_fwd(d["q"], d["k"], d["v"], d["g"], d["b"], d["w"], d["lam_h"], d["S0"])
    S = dev(d["S0"], torch.float32)
    outs = []
    for a, b in ((0, 130), (130, 300)):
        sl = lambda x: x[:, a:b]
        o, _ = qd.qed_fwd(dev(sl(d["q"]), bf), dev(sl(d["k"]), bf), dev(sl(d["v"]), bf), dev(sl(d["g"]), bf),
                          dev(sl(d["b"]), bf), dev(sl(d["w"]), bf), dev(d["lam_h"], torch.float32), S, S_final=S)
        outs.append(o.float().cpu().numpy())
    torch.cuda.synchronize()
    check(np.concatenate(outs, axis=1), o_ref, "bf16", "qed split o")
    check(S.cpu().numpy(), S_ref, "bf16", "qed split S")


def test_qed_lambda_zero_is_gdn2(qd):
    """lam_h = 0 reduces QED to GDN-2; compared with the oracle at lam_h = 0."""
    d = synth.qed_inputs(1, 150, 2, 64, 64, seed=80, dtype="f32")
    d["lam_h"] = np.zeros_like(d["lam_h"])
    o, S = run_qed(qd, d)
    o_ref, S_ref = oracle.qed_fwd(d["q"], d["k"], d["v"], d["g"], d["b"], d["w"], d["lam_h"])
    check(o, o_ref, "f32", "gdn2 o")
    check(S, S_ref, "f32", "gdn2 S")


def test_qed_segmented_long_sequence_all_outputs(qd):
    """B=1, H=2, T=2048 with an initial state: few streams and a long sequence take
    the segment scan for QED too (its transposed state also maps linearly)."""
    d = synth.qed_inputs(1, 2048, 2, 128, 128, seed=57, dtype="bf16", s0_var=0.01)
    assert qd.qed_workspace_bytes(1, 2048, 2, 128, 128) > 0
    o, S = run_qed(qd, d)
    assert qd.last_launch_count() == 5    # the operand derivation, three segment passes, the combine
    o_ref, S_ref = oracle.qed_fwd(d["q"], d["k"], d["v"], d["g"], d["b"], d["w"], d["lam_h"], d["S0"])
    check(o, o_ref, "bf16", "segmented qed o")
    check(S, S_ref, "bf16", "segmented qed S")


@pytest.mark.parametrize("variant", ["nogate", "nogate_noproj", "rand"])
@pytest.mark.parametrize("dt,dh", [("f32", 64), ("bf16", 128)])
def test_qed_ablation_arms_all_outputs(qd, variant, dt, dh):
    """The QED notes' ablation arms (Table 1) on the CUDA-core path (fp32, d=64) and
    the tensor-core path (bf16, d=128): 2 full chunks + a ragged tail, initial state."""
    d = synth.qed_inputs(2, 150, 2, dh, dh, seed=61, dtype=dt, s0_var=0.01)
    o, S = run_qed(qd, d, variant)
    o_ref, S_ref = oracle.qed_fwd_variant(d["q"], d["k"], d["v"], d["g"], d["b"], d["w"], d["lam_h"], variant,
                                          d["z"], d["S0"])
    check(o, o_ref, dt, f"qed {variant} {dt} o")
    check(S, S_ref, dt, f"qed {variant} {dt} S")


def test_qed_full_size_every_stream(qd):
    """B=4, H=8, T=4096, d=128 bf16 (the QED bench workload); all 32 streams against
    the oracle."""
    name, d = synth.qed_gdn2()
    o, S = run_qed(qd, d)
    o_ref, S_ref = oracle.qed_fwd(d["q"], d["k"], d["v"], d["g"], d["b"], d["w"], d["lam_h"])
    check_every_stream(o, o_ref, S, S_ref, name)


# ------------------------------------------------------------------- decode

def test_decode_small_all_outputs(qd):
    d = synth.decode_inputs(3, 2, 128, 128, 20, seed=90)
    S = dev(d["S0"], torch.float32)
    S_ref = d["S0"].astype(np.float64).copy()
    for t in range(20):
        o = qd.qdelta_step(S, dev(d["q"][t]), dev(d["k"][t]), dev(d["v"][t]), dev(d["alpha"][t]),
                           dev(d["beta"][t]), dev(d["lam"][t]))
        o_ref = oracle.qdelta_step(S_ref, d["q"][t], d["k"][t], d["v"][t], d["alpha"][t], d["beta"][t],
                                   d["lam"][t])
        check(o.float().cpu().numpy(), o_ref, "bf16", f"step {t} o")
    check(S.cpu().numpy(), S_ref, "f32", "decode S")


@pytest.mark.parametrize("dk,dv", [(16, 16), (32, 64), (64, 128)])
def test_decode_head_dims_fp32(qd, dk, dv):
    d = synth.decode_inputs(2, 3, dk, dv, 5, seed=91, dtype="f32")
    S = dev(d["S0"], torch.float32)
    S_ref = d["S0"].astype(np.float64).copy()
    for t in range(5):
        o = qd.qdelta_step(S, dev(d["q"][t], torch.float32), dev(d["k"][t], torch.float32),
                           dev(d["v"][t], torch.float32), None, dev(d["beta"][t], torch.float32), None)
        o_ref = oracle.qdelta_step(S_ref, d["q"][t], d["k"][t], d["v"][t], None, d["beta"][t], None)
        check(o.cpu().numpy(), o_ref, "f32", f"step {t} o")
    check(S.cpu().numpy(), S_ref, "f32", "decode S")


def test_decode_512x16_100_steps_sampled(qd):
    """N=512 x H=16, 128x128 fp32 state, 100 consecutive steps in place; 96 heads
    followed by the oracle step by step."""
    name, d = synth.decode_512x16()
    S = dev(d["S0"], torch.float32)
    heads = [(n, h) for n in (0, 1, 77, 255, 256, 400, 510, 511) for h in range(0, 16, 4)] + \
            [(n, h) for n in (3, 300) for h in range(16)] + [(100 + i, i % 16) for i in range(32)]
    ns = np.array([n for n, _ in heads])
    hs = np.array([h for _, h in heads])
    S_ref = d["S0"][ns, hs].astype(np.float64)[:, None].copy()
    tok = lambda x, t: x[t][ns, hs][:, None]
    q_d, k_d, v_d = dev(d["q"]), dev(d["k"]), dev(d["v"])
    a_d, b_d, l_d = dev(d["alpha"]), dev(d["beta"]), dev(d["lam"])
    for t in range(100):
        o = qd.qdelta_step(S, q_d[t], k_d[t], v_d[t], a_d[t], b_d[t], l_d[t])
        o_ref = oracle.qdelta_step(S_ref, tok(d["q"], t), tok(d["k"], t), tok(d["v"], t), tok(d["alpha"], t),
                                   tok(d["beta"], t), tok(d["lam"], t))
        if t % 10 == 9:
            got = o[torch.from_numpy(ns).cuda(), torch.from_numpy(hs).cuda()].float().cpu().numpy()[:, None]
            check(got, o_ref, "bf16", f"{name} step {t} o")
    got = S[torch.from_numpy(ns).cuda(), torch.from_numpy(hs).cuda()].cpu().numpy()[:, None]
    check(got, S_ref, "f32", name + " S after 100 steps")


def test_step_sequence_matches_forward(qd):
    d = synth.qdelta_inputs(2, 40, 2, 64, 64, seed=95, dtype="f32", mode="qdelta", s0_var=0.01)
    f = torch.float32
    o_fwd, S_fwd = qd.qdelta_fwd(dev(d["q"], f), dev(d["k"], f), dev(d["v"], f), dev(d["alpha"], f),
                                 dev(d["beta"], f), dev(d["lam"], f), dev(d["S0"], f))
    S = dev(d["S0"], f)
    outs = []
    for t in range(40):
        outs.append(qd.qdelta_step(S, dev(d["q"][:, t], f), dev(d["k"][:, t], f), dev(d["v"][:, t], f),
                                   dev(d["alpha"][:, t], f), dev(d["beta"][:, t], f), dev(d["lam"][:, t], f)))
    o_step = torch.stack(outs, dim=1)
    torch.cuda.synchronize()
    check(o_step.cpu().numpy(), o_fwd.cpu().numpy(), "f32", "step vs fwd o")
    check(S.cpu().numpy(), S_fwd.cpu().numpy(), "f32", "step vs fwd S")


# ---------------------------------------------------------------- prologue

def run_prologue(qd, d, use_alpha=True, use_lam=True):
    dt = tdt(d)
    o, S = qd.qdelta_fwd(dev(d["q"], dt), dev(d["k"], dt), dev(d["v"], dt),
                         dev(d["alpha"], dt) if use_alpha else None, dev(d["beta"], dt),
                         dev(d["lam"], dt) if use_lam else None, dev(d["S0"], torch.float32), prologue=True)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), S.cpu().numpy()


@pytest.mark.parametrize("dt,dh,use_alpha,use_lam", [("bf16", 128, True, True), ("bf16", 128, False, False),
                                                     ("f32", 64, True, True), ("f32", 32, True, False)])
def test_prologue_forward_all_outputs(qd, dt, dh, use_alpha, use_lam):
    """Forward from projections and logits (feature map and gates inside the kernel),
    tensor-core (bf16, d=128) and CUDA-core (fp32) paths: 2 full chunks + a ragged tail."""
    d = synth.qdelta_raw_inputs(2, 150, 2, dh, dh, seed=63, dtype=dt, s0_var=0.01)
    o, S = run_prologue(qd, d, use_alpha, use_lam)
    o_ref, S_ref = oracle.qdelta_fwd_prologue(d["q"], d["k"], d["v"], d["alpha"] if use_alpha else None, d["beta"],
                                              d["lam"] if use_lam else None, d["S0"])
    check(o, o_ref, dt, f"prologue {dt} o")
    check(S, S_ref, dt, f"prologue {dt} S")


def test_prologue_segmented_long_sequence(qd):
    """B=1, H=2, T=4096 from projections through the segment scan (all passes apply
    the prologue)."""
    d = synth.qdelta_raw_inputs(1, 4096, 2, 128, 128, seed=64, dtype="bf16", s0_var=0.01)
    o, S = run_prologue(qd, d)
    assert qd.last_launch_count() == 4
    o_ref, S_ref = oracle.qdelta_fwd_prologue(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["lam"], d["S0"])
    check(o, o_ref, "bf16", "segmented prologue o")
    check(S, S_ref, "bf16", "segmented prologue S")


@pytest.mark.parametrize("dt,dh", [("f32", 64), ("bf16", 128)])
def test_prologue_decode_steps(qd, dt, dh):
    """Decode steps from projections and logits: 12 steps against the oracle's prologue
    forward run token by token with the state carried."""
    d = synth.qdelta_raw_inputs(3, 12, 2, dh, dh, seed=65, dtype=dt, s0_var=0.01)
    tt = torch.bfloat16 if dt == "bf16" else torch.float32
    S = dev(d["S0"], torch.float32)
    S_ref = d["S0"].astype(np.float64).copy()
    for t in range(12):
        sl = slice(t, t + 1)
        o = qd.qdelta_step(S, dev(d["q"][:, t], tt), dev(d["k"][:, t], tt), dev(d["v"][:, t], tt),
                           dev(d["alpha"][:, t], tt), dev(d["beta"][:, t], tt), dev(d["lam"][:, t], tt), prologue=True)
        o_ref, S_ref = oracle.qdelta_fwd_prologue(d["q"][:, sl], d["k"][:, sl], d["v"][:, sl], d["alpha"][:, sl],
                                                  d["beta"][:, sl], d["lam"][:, sl], S_ref)
        check(o.float().cpu().numpy(), o_ref[:, 0], dt, f"prologue step {t} o")
    check(S.cpu().numpy(), S_ref, "f32", "prologue decode S")


def _qed_step_call(qd, S, d, t, dt, variant):
    z = dev(d["z"], torch.float32) if variant == "rand" else None
    return qd.qed_step(S, dev(d["q"][t], dt), dev(d["k"][t], dt), dev(d["v"][t], dt), dev(d["g"][t], dt),
                       dev(d["b"][t], dt), dev(d["w"][t], dt), dev(d["lam_h"], torch.float32), variant=variant, z=z)


@pytest.mark.parametrize("variant", ["full", "nogate", "nogate_noproj", "rand"])
@pytest.mark.parametrize("dt,dh", [("f32", 64), ("bf16", 128), ("f32", 16)])
def test_qed_decode_steps_all_outputs(qd, variant, dt, dh):
    """QED decode step (the T = 1 recurrence, state in place) for every arm: 20 steps
    from a random state, each step's output and the final state against the oracle."""
    d = synth.qed_decode_inputs(3, 2, dh, dh, 20, seed=92, dtype=dt)
    tt = torch.bfloat16 if dt == "bf16" else torch.float32
    S = dev(d["S0"], torch.float32)
    S_ref = d["S0"].astype(np.float64).copy()
    for t in range(20):
        o = _qed_step_call(qd, S, d, t, tt, variant)
        o_ref = oracle.qed_step(S_ref, d["q"][t], d["k"][t], d["v"][t], d["g"][t], d["b"][t], d["w"][t],
                                d["lam_h"], variant, d["z"])
        check(o.float().cpu().numpy(), o_ref, dt, f"qed step {t} o")
    check(S.cpu().numpy(), S_ref, "f32", "qed decode S")


def test_qed_decode_64x8_30_steps(qd):
    """64 sequences x 8 heads, 128x128 fp32 state, bf16 tokens, 30 steps in place:
    every head against the oracle."""
    d = synth.qed_decode_inputs(64, 8, 128, 128, 30, seed=93)
    S = dev(d["S0"], torch.float32)
    S_ref = d["S0"].astype(np.float64).copy()
    for t in range(30):
        o = _qed_step_call(qd, S, d, t, torch.bfloat16, "full")
        o_ref = oracle.qed_step(S_ref, d["q"][t], d["k"][t], d["v"][t], d["g"][t], d["b"][t], d["w"][t],
                                d["lam_h"], "full")
        if t % 10 == 9:
            check(o.float().cpu().numpy(), o_ref, "bf16", f"qed 64x8 step {t} o")
    check(S.cpu().numpy(), S_ref, "f32", "qed 64x8 S after 30 steps")


def test_qed_step_sequence_matches_forward(qd):
    """T QED decode steps equal one QED forward over the T tokens (fp32, d=64)."""
    d = synth.qed_inputs(2, 40, 2, 64, 64, seed=96, dtype="f32", s0_var=0.01)
    f = torch.float32
    o_fwd, S_fwd = qd.qed_fwd(dev(d["q"], f), dev(d["k"], f), dev(d["v"], f), dev(d["g"], f), dev(d["b"], f),
                              dev(d["w"], f), dev(d["lam_h"], f), dev(d["S0"], f))
    S = dev(d["S0"], f)
    outs = []
    for t in range(40):
        outs.append(qd.qed_step(S, dev(d["q"][:, t], f), dev(d["k"][:, t], f), dev(d["v"][:, t], f),
                                dev(d["g"][:, t], f), dev(d["b"][:, t], f), dev(d["w"][:, t], f),
                                dev(d["lam_h"], f)))
    o_step = torch.stack(outs, dim=1)
    torch.cuda.synchronize()
    check(o_step.cpu().numpy(), o_fwd.cpu().numpy(), "f32", "qed step vs fwd o")
    check(S.cpu().numpy(), S_fwd.cpu().numpy(), "f32", "qed step vs fwd S")


def test_device_status_ok(qd):
    assert qd.qd_device_status() == qd.QD_OK


# ---------------------------------------------------------------- backward

GRAD_NAMES = ("dq", "dk", "dv", "dalpha", "dbeta", "dlam", "dS0")


def check_grad(got, ref, dtype, what):
    """As check(), with the bf16 max-abs bound scaled by the gradient's own magnitude:
    gradients come out in the input dtype, whose rounding alone is 2^-9 of |value|."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    mx = np.abs(got - ref).max() if got.size else 0.0
    if dtype == "bf16":
        bound = BF16_ABS * max(1.0, np.abs(ref).max())
        assert rel <= BF16_REL and mx <= bound, f"{what}: rel L2 {rel:.3e}, max abs {mx:.3e} (bound {bound:.3e})"
    else:
        assert rel <= F32_REL, f"{what}: rel L2 {rel:.3e}, max abs {mx:.3e}"
    return rel, mx


def run_bwd(qd, d, c, want_dS0=True):
    dt = tdt(d)
    g = qd.qdelta_bwd(dev(d["q"], dt), dev(d["k"], dt), dev(d["v"], dt), dev(d["alpha"], dt), dev(d["beta"], dt),
                      dev(d["lam"], dt), dev(d["S0"], torch.float32), dev(c["dO"], dt),
                      dev(c["dS_final"], torch.float32), want_dS0=want_dS0)
    torch.cuda.synchronize()
    return {n: None if x is None else x.float().cpu().numpy() for n, x in g.items()}


@pytest.mark.parametrize("dt,dk,dv,mode", [("f32", 64, 64, "qdelta"), ("f32", 64, 64, "gdn"),
                                           ("f32", 64, 64, "deltanet"), ("f32", 32, 16, "qdelta"),
                                           ("f32", 128, 128, "qdelta"), ("bf16", 128, 128, "qdelta"),
                                           ("bf16", 64, 32, "gdn"), ("bf16", 16, 16, "qdelta")])
def test_backward_all_gradients(qd, dt, dk, dv, mode):
    """Every gradient against the oracle's adjoint: 2 full chunks + a ragged tail,
    carried S0 and an incoming dS_final."""
    d = synth.qdelta_inputs(2, 150, 2, dk, dv, seed=71, dtype=dt, mode=mode, s0_var=0.01)
    c = synth.cotangents(2, 150, 2, dk, dv, seed=71, dtype=dt)
    g = run_bwd(qd, d, c)
    assert qd.last_launch_count() == 3
    ref = oracle.qdelta_bwd(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["lam"], d["S0"], c["dO"],
                            c["dS_final"])
    for name in GRAD_NAMES:
        if ref[name] is None:
            assert g[name] is None, name
            continue
        check_grad(g[name], ref[name], dt, f"{dt} {mode} {name}")


@pytest.mark.parametrize("T", [1, 63, 64, 65, 100, 128])
def test_backward_edge_lengths_without_state(qd, T):
    """T = 1, one short chunk, exactly one chunk, one past it, a ragged second chunk, two
    chunks; S0 = 0 and dS_final = 0."""
    d = synth.qdelta_inputs(1, T, 3, 64, 64, seed=72, dtype="f32", mode="qdelta")
    c = synth.cotangents(1, T, 3, 64, 64, seed=72, dtype="f32", final_state=False)
    g = run_bwd(qd, d, c)
    ref = oracle.qdelta_bwd(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["lam"], None, c["dO"])
    for name in GRAD_NAMES:
        check_grad(g[name], ref[name], "f32", f"T={T} {name}")


def test_backward_empty_sequence_passes_state_gradient(qd):
    d = synth.qdelta_inputs(2, 0, 2, 64, 64, seed=73, dtype="f32", mode="qdelta")
    c = synth.cotangents(2, 0, 2, 64, 64, seed=73, dtype="f32")
    g = run_bwd(qd, d, c)
    assert qd.last_launch_count() == 0
    np.testing.assert_array_equal(g["dS0"], c["dS_final"])


def test_backward_full_size_every_stream(qd):
    """The 1.3B-layer workload (B=8, H=16, T=2048, d=128, bf16) in one call; every
    gradient of every (b, h) stream compared with the oracle over the whole sequence,
    stream by stream and as a whole."""
    _, d = synth.layer_1p3b()
    B, T, H = 8, 2048, 16
    c = synth.cotangents(B, T, H, 128, 128, seed=74, dtype="bf16")
    g = run_bwd(qd, d, c)
    ref = oracle.qdelta_bwd(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["lam"], None, c["dO"],
                            c["dS_final"])
    for name in GRAD_NAMES:
        got, r = g[name], ref[name]
        for b in range(B):
            for h in range(H):
                gs, rs = (got[b, h], r[b, h]) if name == "dS0" else (got[b, :, h], r[b, :, h])
                check_grad(gs, rs, "bf16", f"full-size {name} stream (b={b}, h={h})")
        check_grad(got, r, "bf16", f"full-size {name}")


# ---------------------------------------------------------------- EDA

def run_eda(qd, d):
    dt = tdt(d)
    o, S = qd.eda_fwd(dev(d["q"], dt), dev(d["k"], dt), dev(d["v"], dt), dev(d["e"], dt), dev(d["beta"], dt),
                      dev(d["S0"], torch.float32))
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), S.cpu().numpy()


@pytest.mark.parametrize("dt,dh,erase,beta", [("bf16", 128, "random", True), ("bf16", 128, "query", False),
                                              ("f32", 64, "random", True), ("f32", 32, "query", False),
                                              ("f32", 16, "random", False), ("bf16", 64, "query", True)])
def test_eda_forward_all_outputs(qd, dt, dh, erase, beta):
    """EDA, bf16 and fp32 inputs, random erase directions and the page's e = q/|q|:
    150 tokens (9 staged tiles + a ragged one), carried S0."""
    d = synth.eda_inputs(2, 150, 2, dh, dh, seed=81, dtype=dt, erase=erase, beta=beta, s0_var=0.01)
    o, S = run_eda(qd, d)
    # bf16 at d = 128: sub-token pass, the fp16 tensor-core forward, read-out; else the recurrence
    assert qd.last_launch_count() == (3 if (dt, dh) == ("bf16", 128) else 1)
    o_ref, S_ref = oracle.eda_fwd(d["q"], d["k"], d["v"], d["e"], d["beta"], d["S0"])
    check(o, o_ref, dt, f"eda {dt} {erase} o")
    check(S, S_ref, dt, f"eda {dt} {erase} S")


@pytest.mark.parametrize("dt,dk,dv", [("bf16", 128, 16), ("bf16", 64, 128), ("f32", 128, 64), ("f32", 32, 128)])
def test_eda_rectangular_state(qd, dt, dk, dv):
    """EDA with d_k != d_v: the kernel spreads state rows (d_v) over threads and the
    columns (d_k) over the threads of a row independently, one to four rows a thread."""
    d = synth.eda_inputs(2, 70, 3, dk, dv, seed=83, dtype=dt, erase="random", s0_var=0.01)
    o, S = run_eda(qd, d)
    o_ref, S_ref = oracle.eda_fwd(d["q"], d["k"], d["v"], d["e"], d["beta"], d["S0"])
    check(o, o_ref, dt, f"eda {dt} dk={dk} dv={dv} o")
    check(S, S_ref, dt, f"eda {dt} dk={dk} dv={dv} S")


@pytest.mark.parametrize("erase", ["random", "query"])
def test_eda_full_size_every_stream(qd, erase):
    """The bench's EDA workload (B=8, H=16, T=2048, d=128, bf16, beta = sigmoid(N(0,1)),
    carried S0) on the tensor-core path: every (b, h) stream against the oracle."""
    d = synth.eda_inputs(8, 2048, 16, 128, 128, seed=84, dtype="bf16", erase=erase, s0_var=0.01)
    o, S = run_eda(qd, d)
    assert qd.last_launch_count() == 3
    o_ref, S_ref = oracle.eda_fwd(d["q"], d["k"], d["v"], d["e"], d["beta"], d["S0"])
    check_every_stream(o, o_ref, S, S_ref, f"eda full {erase}")


def test_eda_tensor_core_short_and_empty_sequences(qd):
    """T = 1 and T = 63 (one ragged chunk of 3 and of 127 sub-tokens), and T = 0 (the
    final state is S0) on the tensor-core path."""
    for T in (1, 63):
        d = synth.eda_inputs(1, T, 3, 128, 128, seed=85 + T, dtype="bf16", erase="query", s0_var=0.01)
        o, S = run_eda(qd, d)
        o_ref, S_ref = oracle.eda_fwd(d["q"], d["k"], d["v"], d["e"], d["beta"], d["S0"])
        check(o, o_ref, "bf16", f"eda T={T} o")
        check(S, S_ref, "bf16", f"eda T={T} S")
    d = synth.eda_inputs(1, 1, 3, 128, 128, seed=90, dtype="bf16", s0_var=0.01)
    z = torch.empty(1, 0, 3, 128, dtype=torch.bfloat16, device="cuda")
    S0 = dev(d["S0"], torch.float32)
    o, S = qd.eda_fwd(z, z, z, z, None, S0)
    torch.cuda.synchronize()
    assert o.shape == (1, 0, 3, 128)
    np.testing.assert_array_equal(S.cpu().numpy(), d["S0"])


def test_eda_long_sequence_query_erase(qd):
    """B=1, H=2, T=2048 with e = q: the state carried over the whole sequence."""
    d = synth.eda_inputs(1, 2048, 2, 128, 128, seed=82, dtype="bf16", erase="query", s0_var=0.01)
    o, S = run_eda(qd, d)
    o_ref, S_ref = oracle.eda_fwd(d["q"], d["k"], d["v"], d["e"], d["beta"], d["S0"])
    check(o, o_ref, "bf16", "eda long o")
    check(S, S_ref, "bf16", "eda long S")


@pytest.mark.parametrize("dt,dh,cut", [("f32", 64, 64), ("f32", 64, 90), ("bf16", 128, 128)])
def test_backward_split_call_chains_state_gradient(qd, dt, dh, cut):
    """The state gradient is the backward's carry: the backward of tokens [cut, T) with
    S0 = S_cut and the incoming dS_final, then the backward of [0, cut) with its dS0 as
    dS_final, gives the one-call gradients (chunk-aligned and unaligned cuts)."""
    T = 200
    d = synth.qdelta_inputs(1, T, 2, dh, dh, seed=75, dtype=dt, mode="qdelta", s0_var=0.01)
    c = synth.cotangents(1, T, 2, dh, dh, seed=75, dtype=dt)
    tt = tdt(d)
    cu = lambda x, a, b: None if x is None else dev(x[:, a:b], tt)
    whole = run_bwd(qd, d, c)
    _, S_cut = qd.qdelta_fwd(cu(d["q"], 0, cut), cu(d["k"], 0, cut), cu(d["v"], 0, cut), cu(d["alpha"], 0, cut),
                             cu(d["beta"], 0, cut), cu(d["lam"], 0, cut), dev(d["S0"], torch.float32))
    g2 = qd.qdelta_bwd(cu(d["q"], cut, T), cu(d["k"], cut, T), cu(d["v"], cut, T), cu(d["alpha"], cut, T),
                       cu(d["beta"], cut, T), cu(d["lam"], cut, T), S_cut, cu(c["dO"], cut, T),
                       dev(c["dS_final"], torch.float32))
    g1 = qd.qdelta_bwd(cu(d["q"], 0, cut), cu(d["k"], 0, cut), cu(d["v"], 0, cut), cu(d["alpha"], 0, cut),
                       cu(d["beta"], 0, cut), cu(d["lam"], 0, cut), dev(d["S0"], torch.float32),
                       cu(c["dO"], 0, cut), g2["dS0"])
    torch.cuda.synchronize()
    for name in ("dq", "dk", "dv", "dalpha", "dbeta", "dlam"):
        joined = np.concatenate([g1[name].float().cpu().numpy(), g2[name].float().cpu().numpy()], axis=1)
        check_grad(joined, whole[name], "f32" if dt == "f32" else "bf16", f"split {name}")
    check_grad(g1["dS0"].cpu().numpy(), whole["dS0"], "f32" if dt == "f32" else "bf16", "split dS0")


def test_backward_and_eda_deterministic(qd):
    """Repeated calls give bitwise-identical results (no atomics, no order-dependent sums)."""
    d = synth.qdelta_inputs(2, 150, 2, 128, 128, seed=76, dtype="bf16", mode="qdelta", s0_var=0.01)
    c = synth.cotangents(2, 150, 2, 128, 128, seed=76, dtype="bf16")
    a, b = run_bwd(qd, d, c), run_bwd(qd, d, c)
    for name in GRAD_NAMES:
        assert np.array_equal(a[name], b[name]), name
    e = synth.eda_inputs(2, 150, 2, 128, 128, seed=77, dtype="bf16", s0_var=0.01)
    o1, S1 = run_eda(qd, e)
    o2, S2 = run_eda(qd, e)
    assert np.array_equal(o1, o2) and np.array_equal(S1, S2)


@pytest.mark.parametrize("dt,dh,gates", [("bf16", 128, "all"), ("f32", 64, "all"), ("f32", 32, "beta_only")])
def test_prologue_backward_all_gradients(qd, dt, dh, gates):
    """Backward from projections and logits against the oracle's chain rule through the
    prologue: 2 full chunks + a ragged tail, carried S0 and dS_final."""
    d = synth.qdelta_raw_inputs(2, 150, 2, dh, dh, seed=78, dtype=dt, s0_var=0.01)
    if gates == "beta_only":
        d["alpha"], d["lam"] = None, None
    c = synth.cotangents(2, 150, 2, dh, dh, seed=78, dtype=dt)
    tt = tdt(d)
    g = qd.qdelta_bwd(dev(d["q"], tt), dev(d["k"], tt), dev(d["v"], tt), dev(d["alpha"], tt), dev(d["beta"], tt),
                      dev(d["lam"], tt), dev(d["S0"], torch.float32), dev(c["dO"], tt),
                      dev(c["dS_final"], torch.float32), prologue=True)
    torch.cuda.synchronize()
    assert qd.last_launch_count() == 5
    ref = oracle.qdelta_bwd_prologue(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["lam"], d["S0"], c["dO"],
                                     c["dS_final"])
    for name in GRAD_NAMES:
        if ref[name] is None:
            assert g[name] is None, name
            continue
        check_grad(g[name].float().cpu().numpy(), ref[name], dt, f"prologue bwd {dt} {name}")
