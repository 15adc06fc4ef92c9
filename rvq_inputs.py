"""Seeded synthetic inputs for residual vector quantisation (RVQ) tests and benchmarks.

This module is shared by the CPU oracle's tests and by the CUDA path's tests and
benchmark.  It makes data only; it holds none of the RVQ encode/decode arithmetic.

Generator
---------
Every tensor is drawn from a counter-based splitmix64 stream (Steele, Lea and
Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014; finaliser
constants as published by Vigna for SplitMix64):

    mix(z) = z ^= z >> 30; z *= 0xBF58476D1CE4E5B9;
             z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31
    word(key, i) = mix(key + (i + 1) * 0x9E3779B97F4A7C15)      (mod 2^64)
    key(seed, tensor) = mix(seed * 0x100000001B3 + tensor)

so element ``i`` of tensor ``tensor`` is a pure function of (seed, tensor, i).
Any row of any tensor can be regenerated on its own, on the CPU (numpy) or on a
CUDA device (torch); the integer words are bit-identical on both.

* uniform  u(i)  = ((word(i) >> 11) + 1) * 2^-53, in (0, 1]
* gaussian g(i)  = sqrt(-2 ln u(2i)) * cos(2 pi u(2i+1))   (Box-Muller, float64)
* code     c(i)  = ((word(i) >> 32) * K) >> 32, uniform in [0, K)

Gaussians are formed in float64 and rounded once to float32.

Workloads
---------
The workloads are the RVQ shapes of the OmniVoice codec (8 stages,
1024 entries of dimension 64 at 25 Hz; omnivoice.cpp ARCHITECTURE.md, sections
"GGUF layout" and "RVQ codec") and of the MOSS audio tokenizer (32 stages at
12.5 Hz; moss-tts.cpp AGENTS.md, "What this project is").  Weights follow the
PyTorch (out, in) layouts printed in the "RVQ codec" section:

    w_in     [Q][d][D]   N(0, 1/D)   (standard deviation 1/sqrt(fan_in))
    codebook [Q][K][d]   N(0, 1) * scale_q  (scale_q = decay^q)
    w_out    [Q][D][d]   N(0, 1/d)
    b_in     [Q][d], b_out [Q][D]    N(0, 1) * bias_scale, only when asked for

Frames x are [N][D] with N = B*T.  "gauss" workloads draw x ~ N(0, 1).
"planted" workloads draw codes c[n][q] uniformly and form
x[n] = sum_q w_out[q] @ codebook[q][c[n][q]] + sigma * g: that sum is the
workload's definition of its input, formed here in float64 with a library
matmul and rounded once to float32.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB
KEY_MUL = 0x100000001B3
MASK64 = (1 << 64) - 1

# Tensor identifiers inside one seed.
T_W_IN, T_CODEBOOK, T_W_OUT, T_CODES, T_X, T_B_IN, T_B_OUT = 1, 2, 3, 4, 5, 6, 7
T_FC_W, T_FC_B, T_FC2_W, T_FC2_B = 8, 9, 10, 11

BASE_SEED = 20261202


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    D: int
    Q: int
    K: int
    d: int
    kind: str            # "gauss" | "planted" | "decode"
    sigma: float = 0.0   # planted noise standard deviation
    cb_decay: float = 1.0
    seed: int = BASE_SEED
    metric: str = "l2"   # "l2" | "cosine" (argmin between L2-normalised vectors)
    fc_in: int = 0       # with an fc Linear layer (fc_in -> D) before the quantizer: its input width
    fc_out: int = 0      # with an fc2 Linear layer (D -> fc_out) after decode: its output width

    @property
    def D_in(self) -> int:
        return self.fc_in or self.D

    @property
    def D_out(self) -> int:
        return self.fc_out or self.D

    @property
    def N(self) -> int:
        return self.B * self.T

    def describe(self) -> str:
        return (f"{self.name}: B={self.B} T={self.T} N={self.N} D={self.D} Q={self.Q} "
                f"K={self.K} d={self.d} kind={self.kind} sigma={self.sigma} "
                f"cb_decay={self.cb_decay} seed={self.seed} metric={self.metric}"
                + (f" fc={self.fc_in}->{self.D}" if self.fc_in else "")
                + (f" fc2={self.D}->{self.fc_out}" if self.fc_out else ""))


WORKLOADS = [
    Workload("tiny", 1, 250, 256, 8, 1024, 64, "gauss", seed=BASE_SEED + 0),
    Workload("omnivoice", 16, 750, 1024, 8, 1024, 64, "planted", sigma=0.05, seed=BASE_SEED + 1),
    Workload("decode_only", 64, 750, 1024, 8, 1024, 64, "decode", seed=BASE_SEED + 2),
    Workload("moss_deep", 32, 375, 768, 32, 1024, 64, "gauss", cb_decay=0.8, seed=BASE_SEED + 3),
    Workload("large_batch", 256, 750, 1024, 8, 1024, 64, "planted", sigma=0.2, seed=BASE_SEED + 4),
    # ten books of 4096 entries (the Audio8 codec, audio.cpp
    # docs/models/audio8_tts.md); the latent sizes D, d are not given there,
    # so D=1024, d=64 as in the other shapes
    Workload("k4096_q10", 16, 750, 1024, 10, 4096, 64, "planted", sigma=0.05, seed=BASE_SEED + 5),
    # the MOSS tokenizer's quantizer: 32 books of 1024 entries, argmin between
    # L2-normalised vectors in an 8-dim code space (moss-tts.cpp AGENTS.md,
    # gotchas 9 and 12); the latent size is not given there, D=768 as moss_deep
    Workload("moss_lfq", 32, 375, 768, 32, 1024, 8, "gauss", cb_decay=0.8, seed=BASE_SEED + 6, metric="cosine"),
    # the OmniVoice codec with the Linear layers around its quantizer
    # (omnivoice.cpp ARCHITECTURE.md, "Audio tokenizer": fc 1024 -> 1024 before
    # the RVQ encode, fc2 1024 -> 256 after the RVQ decode)
    Workload("omnivoice_fc", 16, 750, 1024, 8, 1024, 64, "gauss", seed=BASE_SEED + 7, fc_in=1024, fc_out=256),
]
WORKLOAD_BY_NAME = {w.name: w for w in WORKLOADS}


# ----------------------------------------------------------------------------
# numpy backend (reference definition)
# ----------------------------------------------------------------------------

def _mix_np(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.uint64, copy=True)
    z ^= z >> np.uint64(30)
    z *= np.uint64(MIX1)
    z ^= z >> np.uint64(27)
    z *= np.uint64(MIX2)
    z ^= z >> np.uint64(31)
    return z


def _mix_int(z: int) -> int:
    z &= MASK64
    z ^= z >> 30
    z = (z * MIX1) & MASK64
    z ^= z >> 27
    z = (z * MIX2) & MASK64
    z ^= z >> 31
    return z


def stream_key(seed: int, tensor: int) -> int:
    return _mix_int((seed * KEY_MUL + tensor) & MASK64)


def words_np(key: int, idx: np.ndarray) -> np.ndarray:
    """splitmix64 words for counters idx (uint64 array)."""
    with np.errstate(over="ignore"):
        z = np.uint64(key) + (idx.astype(np.uint64) + np.uint64(1)) * np.uint64(GAMMA)
    return _mix_np(z)


def uniform_np(key: int, idx: np.ndarray) -> np.ndarray:
    w = words_np(key, idx)
    return ((w >> np.uint64(11)) + np.uint64(1)).astype(np.float64) * (2.0 ** -53)


def gaussian_np(key: int, idx: np.ndarray) -> np.ndarray:
    idx = idx.astype(np.uint64)
    u1 = uniform_np(key, idx * np.uint64(2))
    u2 = uniform_np(key, idx * np.uint64(2) + np.uint64(1))
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)


def codes_np(key: int, idx: np.ndarray, K: int) -> np.ndarray:
    w = words_np(key, idx)
    return (((w >> np.uint64(32)) * np.uint64(K)) >> np.uint64(32)).astype(np.int32)


def _gauss_block(seed: int, tensor: int, start: int, count: int) -> np.ndarray:
    idx = np.arange(start, start + count, dtype=np.uint64)
    return gaussian_np(stream_key(seed, tensor), idx)


# ----------------------------------------------------------------------------
# weights, codes and frames
# ----------------------------------------------------------------------------

def make_weights(w: Workload, with_bias: bool = False, bias_scale: float = 0.1) -> dict:
    """All per-stage tensors of workload w as float32 numpy arrays."""
    Q, K, d, D = w.Q, w.K, w.d, w.D
    w_in = (_gauss_block(w.seed, T_W_IN, 0, Q * d * D) / math.sqrt(D)).reshape(Q, d, D)
    cb = _gauss_block(w.seed, T_CODEBOOK, 0, Q * K * d).reshape(Q, K, d)
    scale = np.array([w.cb_decay ** q for q in range(Q)], dtype=np.float64)
    cb = cb * scale[:, None, None]
    w_out = (_gauss_block(w.seed, T_W_OUT, 0, Q * D * d) / math.sqrt(d)).reshape(Q, D, d)
    out = {
        "w_in": w_in.astype(np.float32),
        "codebook": cb.astype(np.float32),
        "w_out": w_out.astype(np.float32),
        "b_in": None,
        "b_out": None,
    }
    if with_bias:
        out["b_in"] = (bias_scale * _gauss_block(w.seed, T_B_IN, 0, Q * d)).reshape(Q, d).astype(np.float32)
        out["b_out"] = (bias_scale * _gauss_block(w.seed, T_B_OUT, 0, Q * D)).reshape(Q, D).astype(np.float32)
    if w.fc_in:   # fc: weight [D][D_in] ~ N(0, 1/D_in), bias N(0, 0.1^2)
        out["fc_w"] = (_gauss_block(w.seed, T_FC_W, 0, D * w.fc_in) / math.sqrt(w.fc_in)).reshape(D, w.fc_in) \
            .astype(np.float32)
        out["fc_b"] = (0.1 * _gauss_block(w.seed, T_FC_B, 0, D)).astype(np.float32)
    if w.fc_out:  # fc2: weight [D_out][D] ~ N(0, 1/D), bias N(0, 0.1^2)
        out["fc2_w"] = (_gauss_block(w.seed, T_FC2_W, 0, w.fc_out * D) / math.sqrt(D)).reshape(w.fc_out, D) \
            .astype(np.float32)
        out["fc2_b"] = (0.1 * _gauss_block(w.seed, T_FC2_B, 0, w.fc_out)).astype(np.float32)
    return out


def make_codes(w: Workload, rows: Optional[np.ndarray] = None) -> np.ndarray:
    """Uniform codes [len(rows)][Q] int32 (planted or decode-only workloads)."""
    rows = np.arange(w.N, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    idx = (rows[:, None] * w.Q + np.arange(w.Q, dtype=np.int64)[None, :]).reshape(-1)
    return codes_np(stream_key(w.seed, T_CODES), idx.astype(np.uint64), w.K).reshape(len(rows), w.Q)


def make_x(w: Workload, weights: dict, rows: Optional[np.ndarray] = None,
           chunk: int = 8192) -> np.ndarray:
    """Frames x [len(rows)][D_in] float32 on the CPU (D_in = D without fc).

    gauss:   x ~ N(0, 1)
    planted: x = sum_q w_out[q] @ codebook[q][c_q] + sigma * g   (float64, rounded once)
    """
    if w.kind == "decode":
        raise ValueError("decode-only workload has no frames")
    if w.kind == "planted" and w.fc_in:
        raise ValueError("planted frames live in the quantizer's space: no fc")
    rows = np.arange(w.N, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    D = w.D_in
    out = np.empty((len(rows), D), dtype=np.float32)
    key = stream_key(w.seed, T_X)
    if w.kind == "planted":
        cb64 = weights["codebook"].astype(np.float64)
        wo64 = weights["w_out"].astype(np.float64)
        bo64 = None if weights.get("b_out") is None else weights["b_out"].astype(np.float64)
    for s in range(0, len(rows), chunk):
        r = rows[s:s + chunk]
        idx = (r[:, None] * D + np.arange(D, dtype=np.int64)[None, :]).reshape(-1).astype(np.uint64)
        g = gaussian_np(key, idx).reshape(len(r), D)
        if w.kind == "gauss":
            out[s:s + chunk] = g.astype(np.float32)
            continue
        c = make_codes(w, r)
        acc = np.zeros((len(r), D), dtype=np.float64)
        for q in range(w.Q):
            acc += cb64[q][c[:, q]] @ wo64[q].T
            if bo64 is not None:
                acc += bo64[q][None, :]
        acc += w.sigma * g
        out[s:s + chunk] = acc.astype(np.float32)
    return out


# ----------------------------------------------------------------------------
# torch backend: the same definitions, evaluated on any torch device
# ----------------------------------------------------------------------------

def _s64(v: int) -> int:
    v &= MASK64
    return v - (1 << 64) if v >= (1 << 63) else v


def _lsr(z, s: int):
    # logical right shift of int64 two's-complement words
    import torch
    return torch.bitwise_and(torch.bitwise_right_shift(z, s), (1 << (64 - s)) - 1)


def _mix_torch(z):
    z = z ^ _lsr(z, 30)
    z = z * _s64(MIX1)
    z = z ^ _lsr(z, 27)
    z = z * _s64(MIX2)
    z = z ^ _lsr(z, 31)
    return z


def words_torch(key: int, idx):
    import torch
    z = (idx.to(torch.int64) + 1) * _s64(GAMMA) + _s64(key)
    return _mix_torch(z)


def gaussian_torch(key: int, idx):
    import torch
    idx = idx.to(torch.int64)
    w1 = words_torch(key, idx * 2)
    w2 = words_torch(key, idx * 2 + 1)
    u1 = (_lsr(w1, 11) + 1).to(torch.float64) * (2.0 ** -53)
    u2 = (_lsr(w2, 11) + 1).to(torch.float64) * (2.0 ** -53)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos(2.0 * math.pi * u2)


def codes_torch(key: int, idx, K: int):
    import torch
    w = words_torch(key, idx)
    return ((_lsr(w, 32) * K) >> 32).to(torch.int32)


def make_codes_torch(w: Workload, device, rows=None):
    import torch
    if rows is None:
        rows = torch.arange(w.N, dtype=torch.int64, device=device)
    idx = (rows[:, None] * w.Q + torch.arange(w.Q, dtype=torch.int64, device=device)[None, :]).reshape(-1)
    return codes_torch(stream_key(w.seed, T_CODES), idx, w.K).reshape(-1, w.Q)


def make_x_torch(w: Workload, weights_dev: dict, device, chunk: int = 16384):
    """Frames x [N][D] float32 generated on `device` with the same definitions as make_x.

    weights_dev holds the float32 weights as torch tensors on `device`.  The
    planted sum is formed in float64 (a library matmul) and rounded once.
    """
    import torch
    if w.kind == "decode":
        raise ValueError("decode-only workload has no frames")
    if w.kind == "planted" and w.fc_in:
        raise ValueError("planted frames live in the quantizer's space: no fc")
    D = w.D_in
    out = torch.empty((w.N, D), dtype=torch.float32, device=device)
    key = stream_key(w.seed, T_X)
    ar = torch.arange(D, dtype=torch.int64, device=device)
    if w.kind == "planted":
        cb64 = weights_dev["codebook"].to(torch.float64)
        wo64 = weights_dev["w_out"].to(torch.float64)
        bo = weights_dev.get("b_out")
        bo64 = None if bo is None else bo.to(torch.float64)
    for s in range(0, w.N, chunk):
        n = min(chunk, w.N - s)
        r = torch.arange(s, s + n, dtype=torch.int64, device=device)
        g = gaussian_torch(key, (r[:, None] * D + ar[None, :]).reshape(-1)).reshape(n, D)
        if w.kind == "gauss":
            out[s:s + n] = g.to(torch.float32)
            continue
        c = make_codes_torch(w, device, r).to(torch.int64)
        acc = torch.zeros((n, D), dtype=torch.float64, device=device)
        for q in range(w.Q):
            acc += cb64[q][c[:, q]] @ wo64[q].T
            if bo64 is not None:
                acc += bo64[q][None, :]
        acc += w.sigma * g
        out[s:s + n] = acc.to(torch.float32)
    return out


def weights_to_torch(weights: dict, device) -> dict:
    import torch
    return {k: (None if v is None else torch.from_numpy(np.ascontiguousarray(v)).to(device))
            for k, v in weights.items()}
