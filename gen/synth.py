"""Seeded synthetic inputs shaped like the NAtS-L layer workloads.

Workload recipe (Neural Attention Search Linear, technical summary, "Kernmechanismen"
items 1-4; the layer's inputs are per-head Q, K, V, a per-token log-decay g and a
per-token write strength beta, the score-layer weights and the merge-gate weights):

* Q, K, V ~ N(0, 1), drawn in float32; every key vector is scaled to unit L2 norm
  (Gated DeltaNet expects normalised keys; the layer itself does not normalise).
* g = -0.1 * softplus(z_a) (so a_t = exp(g_t) lies in (0, 1)); beta = sigmoid(z_b);
  z_a, z_b ~ N(0, 1); both float32 and never rounded further.
* merge gate W_g ~ N(0, 0.02^2) per head, b_g = 0.
* Q, K, V are rounded (round-to-nearest-even) to bfloat16 for the bf16 workloads;
  the rounded values are the canonical inputs for every consumer.

Chunk selection is made by the score layer from these inputs.  To keep every
argmax margin far from a tie (so a float32 and a float64 evaluation can never
disagree), the softmax-selected chunks are *planted*: a random unit direction
u_h is added, scaled by alpha, to every query of a planted chunk, and the score
weights get a matching difference along u_h:

    W_s[h, 1] = w1,   W_s[h, 0] = w1 + gamma * [u_h; 0] + n,   b_s[h] = (-gamma*alpha/2, 0)

with w1, n ~ N(0, 0.02^2).  The score layer then prefers softmax exactly on the
planted chunks, with margins of order gamma*alpha/2 minus noise of order
gamma/sqrt(chunk).  Which chunks end up selected is decided by the layer, not
stored here; the planted mask is only the construction's intent and serves as
an independent check of the scorer.

The "all" and "none" patterns leave Q unplanted and force the argmax with a
bias of +-1e3; the "scored" pattern (tiny workload) draws W_s ~ N(0, 0.02^2)
shared by all heads with zero bias and no planting.
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

CHUNK = 64

# Planting constants (see module docstring).
PLANT_ALPHA = 2.0
PLANT_GAMMA = 1.0
SCORE_SIGMA = 0.02
GATE_SIGMA = 0.02
FORCE_BIAS = 1.0e3


@dataclasses.dataclass
class NatsInputs:
    """One workload.  Arrays are float32 holding the canonical (rounded) values."""

    B: int
    H: int
    L: int
    d: int
    chunk: int
    dtype: str  # "bf16" or "f32": storage type of Q, K, V and of the output
    q: np.ndarray  # [B, H, L, d]
    k: np.ndarray
    v: np.ndarray
    g: np.ndarray  # [B, H, L] log-decay
    beta: np.ndarray  # [B, H, L]
    w_s: np.ndarray  # [H, 2, 2d]
    b_s: np.ndarray  # [H, 2]
    w_g: np.ndarray  # [H, d]
    b_g: np.ndarray  # [H]
    planted: Optional[np.ndarray]  # [B, H, N] bool: intended softmax chunks, or None
    name: str = ""

    @property
    def n_chunks(self) -> int:
        return (self.L + self.chunk - 1) // self.chunk

    def device_arrays(self):
        """Q, K, V in their storage encoding: uint16 bf16 bit patterns or float32."""
        if self.dtype == "bf16":
            return bf16_bits(self.q), bf16_bits(self.k), bf16_bits(self.v)
        return self.q, self.k, self.v


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even), kept as float32.

    Works in place on a contiguous float32 array (a copy is made otherwise)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32)
    lsb = b >> np.uint32(16)
    lsb &= np.uint32(1)
    lsb += np.uint32(0x7FFF)
    b += lsb
    b &= np.uint32(0xFFFF0000)
    return x


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of float32 values that are exactly bf16-representable."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    halves = x.view(np.uint16)  # little-endian: [low, high] per element
    if np.any(halves[..., 0::2]):
        raise ValueError("values are not bf16-representable; round them first")
    return np.ascontiguousarray(halves[..., 1::2])


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(stream)])


def _normal(rng, shape, scale=1.0):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    return x


def _unit_rows(x: np.ndarray) -> np.ndarray:
    """Scale every vector along the last axis to unit L2 norm (in place)."""
    n = np.sqrt(np.einsum("...i,...i->...", x, x, dtype=np.float64))
    inv = (1.0 / np.maximum(n, 1e-30)).astype(np.float32)
    x *= inv[..., None]
    return x


def _softplus(z: np.ndarray) -> np.ndarray:
    z64 = z.astype(np.float64)
    return np.where(z64 > 20, z64, np.log1p(np.exp(np.minimum(z64, 20)))).astype(np.float32)


def _sigmoid(z: np.ndarray) -> np.ndarray:
    return (1.0 / (1.0 + np.exp(-z.astype(np.float64)))).astype(np.float32)


def _pattern_mask(rng, B, H, N, pattern, frac, bursts) -> np.ndarray:
    """Boolean [B, H, N] mask of softmax chunks for a planted pattern."""
    m = np.zeros((B, H, N), dtype=bool)
    if pattern == "random":
        n_sel = int(round(frac * N))
        for b in range(B):
            for h in range(H):
                idx = rng.choice(N, size=n_sel, replace=False)
                m[b, h, idx] = True
    elif pattern == "alternating":
        m[:, :, 0::2] = True
    elif pattern == "first":
        m[:, :, 0] = True
    elif pattern == "last":
        m[:, :, N - 1] = True
    elif pattern == "bursts":
        n_bursts, burst_len, n_singles = bursts
        for b in range(B):
            for h in range(H):
                m[b, h] = _bursts_one(rng, N, n_bursts, burst_len, n_singles)
    else:
        raise ValueError(f"unknown pattern {pattern!r}")
    return m


def _bursts_one(rng, N, n_bursts, burst_len, n_singles) -> np.ndarray:
    """Contiguous bursts plus isolated single chunks, none touching another."""
    for _ in range(10000):
        starts = np.sort(rng.integers(0, N - burst_len + 1, size=n_bursts))
        if np.all(np.diff(starts) > burst_len):  # at least one free chunk between bursts
            break
    else:  # pragma: no cover - impossible for the sizes used here
        raise RuntimeError("could not place bursts")
    m = np.zeros(N, dtype=bool)
    for s in starts:
        m[s : s + burst_len] = True
    placed = 0
    while placed < n_singles:
        c = int(rng.integers(0, N))
        lo, hi = max(c - 1, 0), min(c + 2, N)
        if m[lo:hi].any():
            continue
        m[c] = True
        placed += 1
    return m


def make_inputs(
    B: int,
    H: int,
    L: int,
    d: int,
    dtype: str = "bf16",
    seed: int = 0,
    pattern="random",
    frac: float = 0.5,
    bursts=(4, 24, 32),
    chunk: int = CHUNK,
    name: str = "",
) -> NatsInputs:
    """Build one seeded workload.

    pattern: "random" (exactly round(frac*N) planted chunks per (b, h)),
    "alternating", "first", "last", "bursts" (bursts=(n_bursts, burst_len,
    n_singles)), "all" / "none" (bias-forced), "scored" (plain N(0, 0.02^2)
    score weights, zero bias, nothing planted), or an explicit boolean
    [B, H, N] array of planted chunks.
    """
    if dtype not in ("bf16", "f32"):
        raise ValueError(dtype)
    N = (L + chunk - 1) // chunk
    shape = (B, H, L, d)
    q = _normal(_rng(seed, 0), shape)
    k = _unit_rows(_normal(_rng(seed, 1), shape))
    v = _normal(_rng(seed, 2), shape)
    g = -0.1 * _softplus(_normal(_rng(seed, 3), (B, H, L)))
    beta = _sigmoid(_normal(_rng(seed, 4), (B, H, L)))
    rs = _rng(seed, 5)
    w1 = _normal(rs, (H, 2 * d), SCORE_SIGMA)
    noise = _normal(rs, (H, 2 * d), SCORE_SIGMA)
    u = _unit_rows(_normal(_rng(seed, 6), (H, d)))
    w_g = _normal(_rng(seed, 7), (H, d), GATE_SIGMA)
    b_g = np.zeros((H,), np.float32)
    prng = _rng(seed, 8)

    w_s = np.zeros((H, 2, 2 * d), np.float32)
    b_s = np.zeros((H, 2), np.float32)
    planted = None
    if isinstance(pattern, str) and pattern in ("all", "none"):
        w_s[:, 0] = noise
        w_s[:, 1] = w1
        b_s[:, 0] = FORCE_BIAS if pattern == "all" else -FORCE_BIAS
        planted = np.full((B, H, N), pattern == "all")
    elif isinstance(pattern, str) and pattern == "scored":
        w = _normal(rs, (2, 2 * d), SCORE_SIGMA)
        w_s[:] = w[None]
    else:
        if isinstance(pattern, np.ndarray):
            planted = np.asarray(pattern, dtype=bool).reshape(B, H, N)
        else:
            planted = _pattern_mask(prng, B, H, N, pattern, frac, bursts)
        tok = np.repeat(planted, chunk, axis=2)[:, :, :L]  # [B, H, L]
        shift = np.float32(PLANT_ALPHA) * u  # [H, d]
        for b in range(B):
            for h in range(H):
                q[b, h, tok[b, h]] += shift[h]
        w_s[:, 1] = w1
        w_s[:, 0] = w1 + noise
        w_s[:, 0, :d] += np.float32(PLANT_GAMMA) * u
        b_s[:, 0] = -np.float32(PLANT_GAMMA * PLANT_ALPHA / 2)

    if dtype == "bf16":
        q, k, v = round_to_bf16(q), round_to_bf16(k), round_to_bf16(v)
    return NatsInputs(
        B=B, H=H, L=L, d=d, chunk=chunk, dtype=dtype,
        q=np.ascontiguousarray(q, np.float32), k=np.ascontiguousarray(k, np.float32),
        v=np.ascontiguousarray(v, np.float32), g=g.astype(np.float32), beta=beta,
        w_s=w_s, b_s=b_s, w_g=w_g, b_g=b_g, planted=planted, name=name,
    )


# The five workloads.  Shapes follow the layer sizes of the 340M / 1.3B-scale
# hybrid models and the evaluated context lengths (up to 65,536 tokens).
CONFIGS = {
    "tiny": dict(B=1, H=2, L=256, d=64, dtype="f32", seed=0, pattern="scored"),
    "small": dict(B=2, H=8, L=2048, d=128, dtype="bf16", seed=1, pattern="random", frac=0.5),
    "l8192": dict(B=4, H=16, L=8192, d=128, dtype="bf16", seed=2, pattern="random", frac=0.25),
    "sweep0": dict(B=1, H=16, L=32768, d=128, dtype="bf16", seed=3, pattern="none"),
    "sweep12": dict(B=1, H=16, L=32768, d=128, dtype="bf16", seed=3, pattern="random", frac=0.125),
    "sweep50": dict(B=1, H=16, L=32768, d=128, dtype="bf16", seed=3, pattern="random", frac=0.5),
    "sweep100": dict(B=1, H=16, L=32768, d=128, dtype="bf16", seed=3, pattern="all"),
    "long": dict(B=1, H=32, L=65536, d=128, dtype="bf16", seed=4, pattern="bursts", bursts=(4, 24, 32)),
    # the 128k context at which the pages quote prefill and decode latency
    "l128k": dict(B=1, H=4, L=131072, d=128, dtype="bf16", seed=6, pattern="random", frac=0.25),
    # the same shape with every chunk softmax: full causal attention through the same kernels
    "l128k_full": dict(B=1, H=4, L=131072, d=128, dtype="bf16", seed=6, pattern="all"),
}


def config_inputs(name: str) -> NatsInputs:
    """The named workload (see CONFIGS)."""
    cfg = dict(CONFIGS[name])
    return make_inputs(name=name, **cfg)


@dataclasses.dataclass
class NatsXInputs:
    """Hidden states and projection weights of the layer with its projections
    (bf16-representable float32 where the layer takes bf16)."""

    name: str
    B: int
    H: int
    L: int
    d: int
    hidden: int
    x: np.ndarray  # [B, L, hidden]
    w_qkv: np.ndarray  # [hidden, 3 H d]
    w_ab: np.ndarray  # [hidden, 2 H]
    b_a: np.ndarray  # [H]
    a_scale: np.ndarray  # [H]
    b_b: np.ndarray  # [H]
    w_s: np.ndarray  # [H, 2, 2d]
    b_s: np.ndarray  # [H, 2]
    w_g: np.ndarray  # [H, d]
    b_g: np.ndarray  # [H]
    w_o: np.ndarray  # [H d, hidden]


def make_x_inputs(B: int, H: int, L: int, d: int, hidden: int, seed: int = 0, name: str = "",
                  score_scale: float = 0.5) -> NatsXInputs:
    """x ~ N(0, 1); projection weights ~ N(0, 1 / fan_in) so that q, k', v,
    a, b come out ~ N(0, 1); a_scale 0.1 (log-decays like the layer's own
    workloads); score weights ~ N(0, score_scale^2), gate weights
    ~ N(0, 0.02^2).  bf16 tensors are rounded in place (RNE)."""
    rng = _rng(seed, 101)
    x = round_to_bf16(_normal(rng, (B, L, hidden)))
    w_qkv = round_to_bf16(_normal(rng, (hidden, 3 * H * d), 1.0 / np.sqrt(hidden)))
    w_ab = round_to_bf16(_normal(rng, (hidden, 2 * H), 1.0 / np.sqrt(hidden)))
    w_s = _normal(rng, (H, 2, 2 * d), score_scale)
    w_g = _normal(rng, (H, d), 0.02)
    w_o = round_to_bf16(_normal(rng, (H * d, hidden), 1.0 / np.sqrt(H * d)))
    return NatsXInputs(
        name=name, B=B, H=H, L=L, d=d, hidden=hidden, x=x, w_qkv=w_qkv, w_ab=w_ab,
        b_a=np.zeros(H, np.float32), a_scale=np.full(H, 0.1, np.float32), b_b=np.zeros(H, np.float32),
        w_s=w_s, b_s=np.zeros((H, 2), np.float32), w_g=w_g, b_g=np.zeros(H, np.float32), w_o=w_o)


X_CONFIGS = {
    "x_tiny": dict(B=1, H=2, L=256, d=64, hidden=128, seed=11),
    "x_small": dict(B=2, H=4, L=1024, d=128, hidden=512, seed=12),
    # the 1.3B-scale projections (hidden = H d = 2048, the bench's GEMM
    # shapes but for the number of tokens)
    "x_mid": dict(B=1, H=16, L=512, d=128, hidden=2048, seed=14),
    # ragged tiles of the projection GEMMs: 192 tokens (1.5 row tiles), 3 heads
    # of 64 (a column tile across two thirds, 6 gate columns), hidden 200
    # (a partial K block and a partial output tile)
    "x_ragged": dict(B=1, H=3, L=192, d=64, hidden=200, seed=15),
    # the 1.3B-scale layer of the main workload (hidden = H d = 2048)
    "x_l8192": dict(B=4, H=16, L=8192, d=128, hidden=2048, seed=13),
}


def x_config_inputs(name: str) -> NatsXInputs:
    cfg = dict(X_CONFIGS[name])
    return make_x_inputs(name=name, **cfg)


# ------------------------------------------------------------------ NHA ----
# Inputs of the Native Hybrid Attention layer (the "next" workload on the same
# attention kernels): per-head q, k, v and a per-token, per-slot forget gate
# of the slot memory, given as its logarithm.  Recipe:
#   q, k, v ~ N(0, 1) float32 (keys not normalised: the softmax over slots and
#   window sees logits of order one);
#   log_alpha = log(sigmoid(z)) / 8 with z ~ N(0, 1), float32 (the gate damping
#   of Gated Slot Attention, temperature 8: alpha in (0, 1), mostly 0.9-0.99);
#   q, k, v rounded to bf16 for the bf16 workloads (canonical inputs).


@dataclasses.dataclass
class NhaInputs:
    B: int
    H: int
    L: int
    d: int
    m: int  # slots
    window: int
    dtype: str
    q: np.ndarray  # [B, H, L, d]
    k: np.ndarray
    v: np.ndarray
    log_alpha: np.ndarray  # [B, H, L, m]
    name: str = ""


def make_nha_inputs(B: int, H: int, L: int, d: int = 128, m: int = 64, window: int = 512, dtype: str = "bf16",
                    seed: int = 0, name: str = "") -> NhaInputs:
    rng = _rng(seed, 201)
    q = _normal(rng, (B, H, L, d))
    k = _normal(rng, (B, H, L, d))
    v = _normal(rng, (B, H, L, d))
    z = _normal(rng, (B, H, L, m))
    log_alpha = (np.log(_sigmoid(z).astype(np.float64)) / 8.0).astype(np.float32)
    if dtype == "bf16":
        q, k, v = round_to_bf16(q), round_to_bf16(k), round_to_bf16(v)
    return NhaInputs(B=B, H=H, L=L, d=d, m=m, window=window, dtype=dtype, q=q, k=k, v=v, log_alpha=log_alpha,
                     name=name)


NHA_CONFIGS = {
    # parity cases: every window regime, ragged chunk counts
    "nha_tiny": dict(B=1, H=2, L=512, d=128, m=64, window=128, seed=21),
    "nha_w0": dict(B=1, H=2, L=384, d=128, m=64, window=0, seed=22),
    "nha_full": dict(B=1, H=2, L=448, d=128, m=64, window=1 << 20, seed=23),
    "nha_w256": dict(B=2, H=2, L=704, d=128, m=64, window=256, seed=24),
    "nha_mid": dict(B=1, H=4, L=2048, d=128, m=64, window=512, seed=25),
    # the measured workload: the 1.3B-scale layer's shape with a 512-token window
    "nha_l8192": dict(B=4, H=16, L=8192, d=128, m=64, window=512, seed=26),
}


def nha_config_inputs(name: str) -> NhaInputs:
    return make_nha_inputs(name=name, **NHA_CONFIGS[name])
