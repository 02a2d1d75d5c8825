"""Planted-structure attention inputs, generated from a seed, bit-exactly.

The workloads follow the planted-structure recipe that accompanies the Skip
Softmax pages ("Accelerating Long-Context Inference with Skip Softmax in NVIDIA
TensorRT-LLM"): Q, K, V are i.i.d. N(0, 1), and a unit vector u per KV head is
planted so that selected (query, key) pairs get a logit bump
a*b/sqrt(D) = 8 on top of the noise:

* sink keys: the first `sink` (64) keys;
* random blocks: a fixed fraction of the 64-key blocks, chosen per (b, kv-head)
  without replacement;
* recent window: decode has one query at the end of the cache, so the last
  `window` keys carry the bump.  Prefill has a window that moves with the
  query; no per-key weight b_j can express that, so keys are cut into
  `window`-long segments, segment t gets its own direction v_t orthogonal to u,
  and a query in segment t carries v_t + v_{t-1}.  Every query then sees the
  bump on the W..2W keys that precede it (plus its own segment prefix).

Values
------
Each element draws three 64-bit splitmix64 outputs (Steele, Lea & Flood,
"Fast splittable pseudorandom number generators", OOPSLA 2014) from a counter
``key(seed, tensor) + 3*e + j`` (e = linear element index, j = 0, 1, 2).
The twelve 16-bit fields of the three draws are summed (Irwin-Hall, 12 terms);
``(sum - 6*65535) * 2**-16`` is an approximate N(0, 1) sample that is exact in
fp32.  Planted terms are fp32 tables (fp64 values rounded once) added in a fixed
order with fp32 round-to-nearest additions, and the result is rounded to bf16
with round-to-nearest-even.  Every step is integer or a single IEEE fp32
operation, so the CUDA twin in ``planted_dev.cu`` produces identical bits.

Layouts: Q is [B][Hq][Sq][D] (decode: [B][Hq][D]), K and V are
[B][Hkv][Skv][D]; all bf16, D innermost.  Query head h reads kv head h // G.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional, Tuple

import numpy as np

_U64 = np.uint64
_GOLDEN = _U64(0x9E3779B97F4A7C15)
_MIX1 = _U64(0xBF58476D1CE4E5B9)
_MIX2 = _U64(0x94D049BB133111EB)
TENSOR_ID = {"q": 1, "k": 2, "v": 3}
IRWIN_HALL_MEAN = 6 * 65535  # 12 terms of mean 65535/2


@dataclass(frozen=True)
class Workload:
    """Shape and planted structure of one synthetic attention problem."""

    name: str
    kind: str  # "prefill" or "decode"
    B: int
    Hq: int
    Hkv: int
    Sq: int  # decode: 1
    Skv: int
    D: int
    causal: bool
    window: int
    rand_frac: float
    sink: int = 64
    rblock: int = 64
    bump: float = 8.0
    seed: int = 0
    # run parameters carried with the workload (not used by the generator)
    tile_q: int = 0
    tile_k: int = 0
    lambdas: Tuple[float, ...] = field(default=(0.0,))

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five configurations the Skip Softmax measurements are quoted on, as
# synthetic workloads (Llama-3.3-70B-shaped attention for all but the first).
WORKLOADS = {
    "prefill_1k_d64": Workload(
        "prefill_1k_d64", "prefill", B=1, Hq=1, Hkv=1, Sq=1024, Skv=1024, D=64,
        causal=True, window=128, rand_frac=0.05, tile_q=64, tile_k=64,
        lambdas=(0.0, 1e-4, 1e-2)),
    "decode_32k_gqa8": Workload(
        "decode_32k_gqa8", "decode", B=16, Hq=64, Hkv=8, Sq=1, Skv=32768, D=128,
        causal=False, window=1024, rand_frac=0.05, tile_q=1, tile_k=64,
        lambdas=(0.0, 1e-4, 1e-3, 1e-2)),
    "prefill_32k_gqa8": Workload(
        "prefill_32k_gqa8", "prefill", B=1, Hq=64, Hkv=8, Sq=32768, Skv=32768,
        D=128, causal=True, window=2048, rand_frac=0.05, tile_q=128, tile_k=128,
        lambdas=(0.0, 1e-4, 1e-3, 1e-2)),
    "prefill_128k_gqa8": Workload(
        "prefill_128k_gqa8", "prefill", B=1, Hq=64, Hkv=8, Sq=131072, Skv=131072,
        D=128, causal=True, window=4096, rand_frac=0.03, tile_q=128, tile_k=128,
        lambdas=(0.0, 1e-4, 1e-3, 1e-2)),
    "decode_128k_gqa8": Workload(
        "decode_128k_gqa8", "decode", B=8, Hq=64, Hkv=8, Sq=1, Skv=131072, D=128,
        causal=False, window=4096, rand_frac=0.03, tile_q=1, tile_k=64,
        lambdas=(0.0, 1e-4, 1e-3, 1e-2)),
}


# --------------------------------------------------------------------------
# integer noise
# --------------------------------------------------------------------------
def splitmix64(x: np.ndarray) -> np.ndarray:
    """splitmix64 finaliser applied to a uint64 array (wrapping arithmetic)."""
    with np.errstate(over="ignore"):
        z = (x + _GOLDEN).astype(_U64)
        z = (z ^ (z >> _U64(30))) * _MIX1
        z = (z ^ (z >> _U64(27))) * _MIX2
        return z ^ (z >> _U64(31))


def stream_key(seed: int, tensor: str) -> int:
    """64-bit stream key of one tensor of one seed."""
    x = np.array([(seed & 0xFFFFFFFFFFFFFFFF) ^ (TENSOR_ID[tensor] << 56)], dtype=_U64)
    return int(splitmix64(x)[0])


def normal_bits(seed: int, tensor: str, start: int, count: int) -> np.ndarray:
    """fp32 Irwin-Hall normals for linear elements [start, start + count)."""
    key = _U64(stream_key(seed, tensor))
    out = np.empty(count, dtype=np.float32)
    chunk = 1 << 21
    mask16 = _U64(0xFFFF)
    for c0 in range(0, count, chunk):
        n = min(chunk, count - c0)
        e = np.arange(start + c0, start + c0 + n, dtype=_U64)
        acc = np.zeros(n, dtype=np.int64)
        with np.errstate(over="ignore"):
            base = key + _U64(3) * e
            for j in range(3):
                h = splitmix64(base + _U64(j))
                for s in (0, 16, 32, 48):
                    acc += ((h >> _U64(s)) & mask16).astype(np.int64)
        out[c0:c0 + n] = (acc - IRWIN_HALL_MEAN).astype(np.float32) * np.float32(2.0 ** -16)
    return out


# --------------------------------------------------------------------------
# bf16 helpers (bit level)
# --------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 with round-to-nearest-even; returns uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (b + _U64(0x7FFF) + ((b >> _U64(16)) & _U64(1))) >> _U64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bits to fp64, exactly."""
    return bf16_bits_to_f32(bits).astype(np.float64)


def e4m3_round(x: np.ndarray) -> np.ndarray:
    """Round to the nearest OCP FP8 E4M3 value (ties to even), as fp64.

    E4M3: 4 exponent bits with bias 7, 3 mantissa bits, no infinities; normal values
    from 2^-6 to 448, subnormals in steps of 2^-9.  Magnitudes above 448 saturate
    to 448 (the inputs generated here stay far below it).  Used only to prepare
    FP8 test inputs; every step is exact in fp64.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, ex = np.frexp(a)                     # a = m * 2^ex, m in [0.5, 1)
    e = np.maximum(ex.astype(np.float64) - 1.0, -6.0)  # subnormals share the 2^-9 spacing
    step = np.exp2(e - 3.0)
    q = np.rint(a / step) * step
    q = np.minimum(q, 448.0)
    return np.copysign(q, x)


# --------------------------------------------------------------------------
# planted tables
# --------------------------------------------------------------------------
@dataclass
class PlantTables:
    a: float
    b: float
    qu: np.ndarray  # fp32 [Hkv][D]
    ku: np.ndarray  # fp32 [Hkv][D]
    qv: np.ndarray  # fp32 [Hkv][nW][D] (prefill window directions; nW = 0 for decode)
    kv: np.ndarray  # fp32 [Hkv][nW][D]
    rblk: np.ndarray  # uint8 [B][Hkv][nrb]


def _unit(v: np.ndarray) -> np.ndarray:
    return v / np.linalg.norm(v)


def make_tables(w: Workload) -> PlantTables:
    """Directions, amplitudes and random-block flags of a workload (host, fp64)."""
    rng = np.random.default_rng([w.seed, 0x5EED])
    amp = math.sqrt(w.bump * math.sqrt(w.D))  # a = b, so a*b/sqrt(D) = bump
    u = np.stack([_unit(rng.standard_normal(w.D)) for _ in range(w.Hkv)])
    if w.kind == "prefill" and w.window > 0:
        nw = (w.Skv - 1) // w.window + 1
        v = np.empty((w.Hkv, nw, w.D))
        for h in range(w.Hkv):
            for t in range(nw):
                x = rng.standard_normal(w.D)
                x -= np.dot(x, u[h]) * u[h]
                v[h, t] = _unit(x)
    else:
        v = np.zeros((w.Hkv, 0, w.D))
    nrb = (w.Skv + w.rblock - 1) // w.rblock
    cnt = int(math.floor(w.rand_frac * nrb + 0.5))
    rblk = np.zeros((w.B, w.Hkv, nrb), dtype=np.uint8)
    for b in range(w.B):
        for h in range(w.Hkv):
            rblk[b, h, rng.permutation(nrb)[:cnt]] = 1
    f32 = np.float32
    return PlantTables(
        a=amp, b=amp,
        qu=(amp * u).astype(f32), ku=(amp * u).astype(f32),
        qv=(amp * v).astype(f32), kv=(amp * v).astype(f32), rblk=rblk)


# --------------------------------------------------------------------------
# tensors (bf16 bits), row slices or whole tensors
# --------------------------------------------------------------------------
def _prefill_window(w: Workload) -> bool:
    return w.kind == "prefill" and w.window > 0


def gen_q_rows(w: Workload, t: PlantTables, b: int, hq: int, s0: int = 0,
               s1: Optional[int] = None) -> np.ndarray:
    """Q[b, hq, s0:s1, :] as bf16 bits (decode: s0 = 0, s1 = 1)."""
    sq = 1 if w.kind == "decode" else w.Sq
    s1 = sq if s1 is None else s1
    n = s1 - s0
    hk = hq // w.G
    start = ((b * w.Hq + hq) * sq + s0) * w.D
    x = normal_bits(w.seed, "q", start, n * w.D).reshape(n, w.D)
    x = x + t.qu[hk][None, :]
    if _prefill_window(w):
        pos = np.arange(s0, s1) + (w.Skv - w.Sq)
        seg = pos // w.window
        x = x + t.qv[hk][seg]
        prev = np.maximum(seg - 1, 0)
        has_prev = (seg >= 1)[:, None]
        x = np.where(has_prev, x + t.qv[hk][prev], x)
    return f32_to_bf16_bits(x.astype(np.float32))


def key_planted(w: Workload, t: PlantTables, b: int, hk: int, j0: int, j1: int) -> np.ndarray:
    """Boolean flags: key j in [j0, j1) carries the u bump."""
    j = np.arange(j0, j1)
    f = (j < w.sink) | (t.rblk[b, hk][j // w.rblock] != 0)
    if w.kind == "decode" and w.window > 0:
        f |= j >= w.Skv - w.window
    return f


def gen_k_rows(w: Workload, t: PlantTables, b: int, hk: int, j0: int = 0,
               j1: Optional[int] = None) -> np.ndarray:
    j1 = w.Skv if j1 is None else j1
    n = j1 - j0
    start = ((b * w.Hkv + hk) * w.Skv + j0) * w.D
    x = normal_bits(w.seed, "k", start, n * w.D).reshape(n, w.D)
    f = key_planted(w, t, b, hk, j0, j1)[:, None]
    x = np.where(f, x + t.ku[hk][None, :], x)
    if _prefill_window(w):
        seg = np.arange(j0, j1) // w.window
        x = x + t.kv[hk][seg]
    return f32_to_bf16_bits(x.astype(np.float32))


def gen_v_rows(w: Workload, b: int, hk: int, j0: int = 0, j1: Optional[int] = None) -> np.ndarray:
    j1 = w.Skv if j1 is None else j1
    n = j1 - j0
    start = ((b * w.Hkv + hk) * w.Skv + j0) * w.D
    x = normal_bits(w.seed, "v", start, n * w.D).reshape(n, w.D)
    return f32_to_bf16_bits(x)


def gen_q(w: Workload, t: PlantTables) -> np.ndarray:
    if w.kind == "decode":
        out = np.empty((w.B, w.Hq, w.D), dtype=np.uint16)
        for b in range(w.B):
            for h in range(w.Hq):
                out[b, h] = gen_q_rows(w, t, b, h)[0]
        return out
    out = np.empty((w.B, w.Hq, w.Sq, w.D), dtype=np.uint16)
    for b in range(w.B):
        for h in range(w.Hq):
            out[b, h] = gen_q_rows(w, t, b, h)
    return out


def gen_k(w: Workload, t: PlantTables) -> np.ndarray:
    out = np.empty((w.B, w.Hkv, w.Skv, w.D), dtype=np.uint16)
    for b in range(w.B):
        for h in range(w.Hkv):
            out[b, h] = gen_k_rows(w, t, b, h)
    return out


def gen_v(w: Workload, t: Optional[PlantTables] = None) -> np.ndarray:
    out = np.empty((w.B, w.Hkv, w.Skv, w.D), dtype=np.uint16)
    for b in range(w.B):
        for h in range(w.Hkv):
            out[b, h] = gen_v_rows(w, b, h)
    return out


def gen_all(w: Workload):
    """(tables, q_bits, k_bits, v_bits) for a workload small enough for the host."""
    t = make_tables(w)
    return t, gen_q(w, t), gen_k(w, t), gen_v(w, t)
