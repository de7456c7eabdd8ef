"""Seeded synthetic inputs for the Q-Delta / QED chunked forward and decode step.

This module is shared by the tests, the bench and the callers of the oracle.  It
holds none of the method's arithmetic: only a counter-based random stream
(SplitMix64, Steele, Lea & Flood 2014), Box-Muller normals, the input
distributions of the workloads and round-to-nearest-even to bf16/fp32.

Every tensor of a workload draws from its own stream, keyed by (seed, stream id),
so a tensor's values do not depend on which other tensors were drawn or in what
order.  All arrays are returned as float32 numpy arrays whose values are exactly
representable in the requested input dtype ("bf16" or "f32"); the GPU path and
the oracle consume the very same values.

Distributions (the workloads of the Q-Delta and QED reading notes; the model
shapes stand in for their 340M-1.3B models and 2K-32K contexts):
  q, k   ~ N(0,1), then L2-normalised per token (in fp64, before rounding)
  v      ~ N(0,1)
  beta   = sigmoid(N(0,1));  lambda = sigmoid(N(0,1))
  alpha  = exp(-softplus(N(mu, 0.5))), mu = -4 (alpha ~ 0.98) unless a mean alpha
           is requested, in which case mu is found by bisection on 1e6 fp64 draws
  QED:   g = -softplus(N(-5, 0.5)) per key channel; b, w = sigmoid(N(0,1));
         lambda_h ~ U(0,1) per head; the rand arm's z_h ~ N(0,1) per head, unit length
  S0     ~ N(0, s0_var) when an initial state is requested (variance, not std)
"""
from __future__ import annotations

import math

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Fixed stream ids per tensor name.
STREAMS = {
    "q": 1, "k": 2, "v": 3, "alpha": 4, "beta": 5, "lam": 6, "S0": 7,
    "g": 8, "b": 9, "w": 10, "lam_h": 11, "alpha_mu": 12, "z": 13, "dO": 14, "dS": 15, "e": 16,
}

_BLOCK = 1 << 22


def _mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function (bijective finaliser), on uint64 arrays."""
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def _base(seed: int, stream: int) -> np.uint64:
    key = np.array([(int(seed) & 0xFFFFFFFF) << 32 | (int(stream) & 0xFFFFFFFF)], dtype=np.uint64)
    return _mix64(_mix64(key))[0]


def splitmix64(seed: int, stream: int, start: int, n: int) -> np.ndarray:
    """Outputs start..start+n-1 of the SplitMix64 sequence seeded by (seed, stream)."""
    idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        x = _base(seed, stream) + idx * _GOLDEN
    return _mix64(x)


def uniform(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """n fp64 uniforms in the open interval (0, 1): (top 53 bits + 0.5) / 2^53."""
    out = np.empty(n, dtype=np.float64)
    for s in range(0, n, _BLOCK):
        m = min(_BLOCK, n - s)
        bits = splitmix64(seed, stream, start + s, m) >> np.uint64(11)
        out[s:s + m] = (bits.astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)
    return out


def normal(seed: int, stream: int, n: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """n fp64 normals by Box-Muller on consecutive uniform pairs (u1, u2)."""
    out = np.empty(n, dtype=np.float64)
    pairs_per_block = _BLOCK // 2
    for p0 in range(0, (n + 1) // 2, pairs_per_block):
        np_ = min(pairs_per_block, (n + 1) // 2 - p0)
        u = uniform(seed, stream, 2 * np_, start=2 * p0)
        r = np.sqrt(-2.0 * np.log(u[0::2]))
        th = (2.0 * math.pi) * u[1::2]
        z = np.empty(2 * np_, dtype=np.float64)
        z[0::2] = r * np.cos(th)
        z[1::2] = r * np.sin(th)
        lo = 2 * p0
        hi = min(n, lo + 2 * np_)
        out[lo:hi] = z[: hi - lo]
    return out * std + mean


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round to the input dtype: "f32" (RNE to fp32) or "bf16" (RNE fp32 -> bf16).

    Returns float32 values exactly representable in that dtype."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    if dtype == "f32":
        return f
    if dtype != "bf16":
        raise ValueError(f"unknown dtype {dtype!r}")
    b = f.view(np.uint32)
    with np.errstate(over="ignore"):
        r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def _softplus(x):
    return np.logaddexp(0.0, x)


def _unit_rows(x: np.ndarray) -> np.ndarray:
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def alpha_mu_for_mean(mean_alpha: float, std: float = 0.5, seed: int = 0) -> float:
    """mu such that E[exp(-softplus(N(mu, std)))] = mean_alpha, by bisection over
    1e6 fixed fp64 draws."""
    z = normal(seed, STREAMS["alpha_mu"], 1_000_000)
    lo, hi = -30.0, 10.0
    for _ in range(60):
        mid = 0.5 * (lo + hi)
        m = np.mean(np.exp(-_softplus(mid + std * z)))
        if m > mean_alpha:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def qdelta_inputs(B: int, T: int, H: int, dk: int, dv: int, seed: int, dtype: str = "bf16",
                  mode: str = "qdelta", alpha_mu: float = -4.0, s0_var: float | None = None) -> dict:
    """Inputs of one Q-Delta forward in the boundary layout.

    mode: "qdelta" (alpha, beta, lambda), "gdn" (lambda absent = 0) or
    "deltanet" (alpha absent = 1, lambda absent = 0).  Absent gates are None.
    Shapes: q, k [B,T,H,dk]; v [B,T,H,dv]; gates [B,T,H]; S0 [B,H,dv,dk] fp32."""
    n_tok = B * T * H
    q = _unit_rows(normal(seed, STREAMS["q"], n_tok * dk).reshape(B, T, H, dk))
    k = _unit_rows(normal(seed, STREAMS["k"], n_tok * dk).reshape(B, T, H, dk))
    v = normal(seed, STREAMS["v"], n_tok * dv).reshape(B, T, H, dv)
    beta = _sigmoid(normal(seed, STREAMS["beta"], n_tok)).reshape(B, T, H)
    out = {"q": round_to(q, dtype), "k": round_to(k, dtype), "v": round_to(v, dtype),
           "beta": round_to(beta, dtype), "alpha": None, "lam": None, "S0": None,
           "dtype": dtype, "shape": (B, T, H, dk, dv)}
    if mode in ("qdelta", "gdn"):
        a = np.exp(-_softplus(normal(seed, STREAMS["alpha"], n_tok, mean=alpha_mu, std=0.5)))
        out["alpha"] = round_to(a.reshape(B, T, H), dtype)
    elif mode != "deltanet":
        raise ValueError(f"unknown mode {mode!r}")
    if mode == "qdelta":
        lam = _sigmoid(normal(seed, STREAMS["lam"], n_tok)).reshape(B, T, H)
        out["lam"] = round_to(lam, dtype)
    if s0_var is not None:
        s0 = normal(seed, STREAMS["S0"], B * H * dv * dk, std=math.sqrt(s0_var))
        out["S0"] = round_to(s0.reshape(B, H, dv, dk), "f32")
    return out


def eda_inputs(B: int, T: int, H: int, dk: int, dv: int, seed: int, dtype: str = "bf16", erase: str = "random",
               beta: bool = True, s0_var: float | None = None) -> dict:
    """Inputs of one EDA forward: q, k unit rows and v ~ N(0,1) as for Q-Delta; the erase
    direction e a unit N(0,1) row ("random") or e = q ("query", the page's e = q/|q|);
    beta = sigmoid(N(0,1)) or None (the page's unit step)."""
    d = qdelta_inputs(B, T, H, dk, dv, seed, dtype, mode="deltanet", s0_var=s0_var)
    if erase == "query":
        e = d["q"].copy()
    elif erase == "random":
        e = round_to(_unit_rows(normal(seed, STREAMS["e"], B * T * H * dk).reshape(B, T, H, dk)), dtype)
    else:
        raise ValueError(f"unknown erase {erase!r}")
    return {"q": d["q"], "k": d["k"], "v": d["v"], "e": e, "beta": d["beta"] if beta else None, "S0": d["S0"],
            "dtype": dtype, "shape": (B, T, H, dk, dv)}


def cotangents(B: int, T: int, H: int, dk: int, dv: int, seed: int, dtype: str = "bf16",
               final_state: bool = True) -> dict:
    """Incoming gradients of one backward: dO [B,T,H,dv] ~ N(0,1) in the input dtype
    and dS_final [B,H,dv,dk] ~ N(0,1) fp32 (None unless final_state)."""
    dO = round_to(normal(seed, STREAMS["dO"], B * T * H * dv).reshape(B, T, H, dv), dtype)
    dS = round_to(normal(seed, STREAMS["dS"], B * H * dv * dk).reshape(B, H, dv, dk), "f32") if final_state else None
    return {"dO": dO, "dS_final": dS}


def qdelta_raw_inputs(B: int, T: int, H: int, dk: int, dv: int, seed: int, dtype: str = "bf16",
                      alpha_mu: float = -4.0, s0_var: float | None = None) -> dict:
    """Inputs of one Q-Delta forward from projections (the prologue entry points): the
    draws of qdelta_inputs before their maps, i.e. q_raw, k_raw ~ N(0,1) (not
    normalised), a_logit ~ N(alpha_mu, 0.5), b_logit, l_logit ~ N(0,1); v, S0 as there."""
    n_tok = B * T * H
    out = {
        "q": round_to(normal(seed, STREAMS["q"], n_tok * dk).reshape(B, T, H, dk), dtype),
        "k": round_to(normal(seed, STREAMS["k"], n_tok * dk).reshape(B, T, H, dk), dtype),
        "v": round_to(normal(seed, STREAMS["v"], n_tok * dv).reshape(B, T, H, dv), dtype),
        "alpha": round_to(normal(seed, STREAMS["alpha"], n_tok, mean=alpha_mu, std=0.5).reshape(B, T, H), dtype),
        "beta": round_to(normal(seed, STREAMS["beta"], n_tok).reshape(B, T, H), dtype),
        "lam": round_to(normal(seed, STREAMS["lam"], n_tok).reshape(B, T, H), dtype),
        "S0": None, "dtype": dtype, "shape": (B, T, H, dk, dv),
    }
    if s0_var is not None:
        s0 = normal(seed, STREAMS["S0"], B * H * dv * dk, std=math.sqrt(s0_var))
        out["S0"] = round_to(s0.reshape(B, H, dv, dk), "f32")
    return out


def qed_inputs(B: int, T: int, H: int, dk: int, dv: int, seed: int, dtype: str = "bf16",
               g_mu: float = -5.0, s0_var: float | None = None) -> dict:
    """Inputs of one QED forward: q, k [B,T,H,dk]; v [B,T,H,dv]; g, b [B,T,H,dk];
    w [B,T,H,dv]; lam_h [H] fp32; S0 [B,H,dv,dk] fp32 (QED's K x V state stored
    transposed, as [dv][dk])."""
    n_tok = B * T * H
    q = _unit_rows(normal(seed, STREAMS["q"], n_tok * dk).reshape(B, T, H, dk))
    k = _unit_rows(normal(seed, STREAMS["k"], n_tok * dk).reshape(B, T, H, dk))
    v = normal(seed, STREAMS["v"], n_tok * dv).reshape(B, T, H, dv)
    g = -_softplus(normal(seed, STREAMS["g"], n_tok * dk, mean=g_mu, std=0.5)).reshape(B, T, H, dk)
    b = _sigmoid(normal(seed, STREAMS["b"], n_tok * dk)).reshape(B, T, H, dk)
    w = _sigmoid(normal(seed, STREAMS["w"], n_tok * dv)).reshape(B, T, H, dv)
    lam_h = uniform(seed, STREAMS["lam_h"], H)
    z = _unit_rows(normal(seed, STREAMS["z"], H * dk).reshape(H, dk))
    out = {"q": round_to(q, dtype), "k": round_to(k, dtype), "v": round_to(v, dtype),
           "g": round_to(g, dtype), "b": round_to(b, dtype), "w": round_to(w, dtype),
           "lam_h": round_to(lam_h, "f32"), "z": round_to(z, "f32"), "S0": None, "dtype": dtype,
           "shape": (B, T, H, dk, dv)}
    if s0_var is not None:
        s0 = normal(seed, STREAMS["S0"], B * H * dv * dk, std=math.sqrt(s0_var))
        out["S0"] = round_to(s0.reshape(B, H, dv, dk), "f32")
    return out


def decode_inputs(N: int, H: int, dk: int, dv: int, steps: int, seed: int, dtype: str = "bf16",
                  s0_var: float | None = 0.01) -> dict:
    """Inputs of `steps` consecutive decode steps: tokens q, k [steps,N,H,dk],
    v [steps,N,H,dv], gates [steps,N,H]; state S0 [N,H,dv,dk] fp32."""
    d = qdelta_inputs(steps, 1, N * H, dk, dv, seed, dtype, mode="qdelta")
    out = {
        "q": d["q"].reshape(steps, N, H, dk), "k": d["k"].reshape(steps, N, H, dk),
        "v": d["v"].reshape(steps, N, H, dv), "alpha": d["alpha"].reshape(steps, N, H),
        "beta": d["beta"].reshape(steps, N, H), "lam": d["lam"].reshape(steps, N, H),
        "S0": None, "dtype": dtype, "shape": (N, H, dk, dv, steps),
    }
    if s0_var is not None:
        s0 = normal(seed, STREAMS["S0"], N * H * dv * dk, std=math.sqrt(s0_var))
        out["S0"] = round_to(s0.reshape(N, H, dv, dk), "f32")
    return out


def qed_decode_inputs(N: int, H: int, dk: int, dv: int, steps: int, seed: int, dtype: str = "bf16",
                      s0_var: float | None = 0.01) -> dict:
    """Inputs of `steps` consecutive QED decode steps: q, k, g, b [steps,N,H,dk],
    v, w [steps,N,H,dv]; lam_h [H], z [H,dk] fp32; state S0 [N,H,dv,dk] fp32."""
    d = qed_inputs(steps, 1, N * H, dk, dv, seed, dtype)
    out = {key: d[key].reshape(steps, N, H, -1) for key in ("q", "k", "v", "g", "b", "w")}
    # one lambda_h / z_h per head: the first H of the N*H drawn
    out.update({"lam_h": d["lam_h"][:H].copy(), "z": d["z"][:H].copy(), "S0": None, "dtype": dtype,
                "shape": (N, H, dk, dv, steps)})
    if s0_var is not None:
        s0 = normal(seed, STREAMS["S0"], N * H * dv * dk, std=math.sqrt(s0_var))
        out["S0"] = round_to(s0.reshape(N, H, dv, dk), "f32")
    return out


# The workloads, by what they are.  Each returns (name, inputs).
def tiny_fp32():
    """Tiny Q-Delta forward in fp32: B=1, H=2, T=256, d=64, S0 = 0, seed 0."""
    return "qdelta_fp32_B1_H2_T256_d64", qdelta_inputs(1, 256, 2, 64, 64, seed=0, dtype="f32")


def layer_1p3b(mode: str = "qdelta", T: int = 2048, B: int = 8):
    """1.3B-model layer shape, bf16: B=8, H=16, T=2048, d=128, seed 1."""
    return (f"{mode}_bf16_B{B}_H16_T{T}_d128",
            qdelta_inputs(B, T, 16, 128, 128, seed=1, dtype="bf16", mode=mode))


def long_context(T: int = 32768):
    """Long-context Q-Delta, bf16: B=1, H=16, T=32768, d=128, mean alpha 0.995,
    S0 ~ N(0, 0.01), seed 2."""
    mu = alpha_mu_for_mean(0.995)
    return (f"qdelta_bf16_B1_H16_T{T}_d128_meanalpha0.995",
            qdelta_inputs(1, T, 16, 128, 128, seed=2, dtype="bf16", mode="qdelta",
                          alpha_mu=mu, s0_var=0.01))


def qed_gdn2(T: int = 4096, B: int = 4):
    """QED over GDN-2, bf16: B=4, H=8, T=4096, d=128, seed 3."""
    return f"qed_bf16_B{B}_H8_T{T}_d128", qed_inputs(B, T, 8, 128, 128, seed=3, dtype="bf16")


def decode_512x16(steps: int = 100, N: int = 512):
    """Decode: N=512 sequences x H=16, fp32 128x128 state, bf16 tokens, seed 4."""
    return (f"qdelta_step_bf16_N{N}_H16_d128_steps{steps}",
            decode_inputs(N, 16, 128, 128, steps, seed=4, dtype="bf16"))
