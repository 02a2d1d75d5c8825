"""Plain fp64 implementation of Skip Softmax attention (prefill and decode).

TEST INFRASTRUCTURE ONLY: the CUDA library never imports this module.

What it computes, and where the pages say so
--------------------------------------------
* "Accelerating Long-Context Inference with Skip Softmax in NVIDIA TensorRT-LLM"
  (video recap), sections "Quick Overview", "Detailed Analysis" and "Skip
  Softmax Mechanism": attention is processed block by block; the local maximum
  of a block's attention scores is compared with the maximum seen before it
  (printed "MI - 1", read here as m_{i-1}, the running maximum over the blocks
  already processed), and when the block falls below the threshold tau its whole
  attention computation is skipped.  "Impact on Accuracy vs. Speed": tau trades
  speed for accuracy.
* "NVIDIA Introduces Skip Softmax for Enhanced LLM Inference Efficiency",
  section "Understanding Skip Softmax": blocks whose contribution is negligible
  are detected early from the softmax's own properties and skipped, with no
  retraining.
* The exact rule used here (the plainest reading the pages support): for a
  (query tile, key tile) pair, with m~_r the tile's row maximum of the scaled
  logits and m_r the running row maximum before the tile, the tile is skipped
  iff lambda > 0 and, for every valid row r of the query tile,
  exp(m~_r - m_r) < lambda, i.e. m~_r - m_r < ln(lambda).  A skipped tile
  contributes nothing (no exponentials, no P.V); a kept tile takes the exact
  online-softmax update (the FlashAttention recurrence named in "Approximating
  Softmax in Pretrained LLMs", Abstract).

Readings where the pages are silent
-----------------------------------
* key tiles are visited in ascending order; the running max starts at -inf, so
  the first visited tile is never skipped (gap = +inf);
* a row with no visible key in the tile has gap -inf (it votes "skip");
* padding rows beyond Sq do not vote;
* causal masking is bottom-right aligned: query i sits at position Skv-Sq+i;
* softmax scale 1/sqrt(D) unless given;
* decode: the rows of one vote are the G query heads that share a kv head; the
  cache is cut into contiguous splits of whole key tiles (ceil(nblk/splits)
  tiles each, empty trailing splits dropped); every split starts its own
  running max at -inf and the split results are merged by an exact
  log-sum-exp combine.

Caller-supplied block mask (optional, prefill and decode)
--------------------------------------------------------
"NVIDIA Introduces Skip Softmax ...", "Benefits and Implementation": Skip Softmax
can be combined with other sparse-attention methods (a block selector in
prefill).  Reading used here: a block selector hands the kernel a mask over the
(query tile, key tile) pairs of prefill, or over the 64-key tiles of each
(batch, kv head) in decode; tiles outside it are not visited at all (no
logits, no running max, no vote), and the skip rule runs over the selected
tiles in ascending order, the first selected tile being always kept (in decode:
the first of each split).  A decode split with no selected tile contributes
nothing to the combine; a row (prefill) or group (decode) that ends with no
visible selected key gets output 0 and log-sum-exp -inf.

Rowmax-PoT weights (optional, prefill)
--------------------------------------
"Approximating Softmax in Pretrained LLMs: Model Sensitivity and Kernel
Acceleration", AI Summary and Abstract: exponentials are replaced by powers of
two, a coarse logarithmic weight representation anchored at each row maximum.
Reading used here (the pages give no formula): for a kept tile, with m'_r the
row maximum after the tile (the same exact running maximum the skip rule uses),
key c gets the weight 2^n, n = round((s_rc - m'_r) * log2 e) (ties to even),
and 0 when that exponent is below -126.5 (the smallest normal fp32 power of
two is 2^-126).  Earlier tiles are rescaled exactly by exp(m_r - m'_r) when
the maximum grows, as in the exact recurrence, so each key's weight is anchored
at the running maximum of the tile it belongs to.  The pages' "Rowmax-H15"
hardware specialisation is not described and is not modelled.  Because the
rounding of n decides a discrete value, keys whose exponent lies within
POT_AMBIGUOUS_BAND of a rounding boundary are reported: a kernel computing the
logits in fp32 may round them the other way.

FP8 P.V (optional, prefill)
---------------------------
"Approximating Softmax in Pretrained LLMs ...", AI Summary: FP8/BF16 mixed-precision
tensor cores.  With e4m3 Q, K and V the second product also runs in e4m3, so the
softmax weights themselves are quantised.  Reading used here (the pages give no
formula): on a kept tile, with m'_r the exact running row maximum after the tile,
each weight p_rc = exp(s_rc - m'_r) <= 1 enters P.V as e4m3(2^8 * p_rc) * 2^-8 --
scaled by 2^8 so that the largest weight, 1, maps to 256 (inside e4m3's 448) and every
p >= 2^-14 keeps e4m3's three mantissa bits -- rounded to nearest, ties to even.  The
row sum l takes the unquantised p (it is the softmax's denominator), and the earlier
tiles are rescaled exactly by exp(m - m') when the maximum grows, as in the exact
recurrence.  The skip vote is unchanged.  Keys whose 2^8 * p lies within a relative
FP8_AMBIGUOUS_BAND of an e4m3 rounding midpoint are reported: fp32 arithmetic may
round them to the neighbouring e4m3 value.  e4m3 rounding (OCP E4M3: 4 exponent bits of
bias 7, 3 mantissa bits, subnormal step 2^-9, largest finite 448) is written out below
from that definition.

Everything is fp64; bf16 inputs convert to fp64 exactly.  There is no blocking,
fusion or reordering beyond the tile loop that defines the method.
"""

from __future__ import annotations

import math
from dataclasses import dataclass
from typing import List, Optional, Tuple

import numpy as np

NEG_INF = -np.inf
LOG2E = 1.0 / math.log(2.0)
# half-width (in log2 units) of the band around a rounding boundary of the
# Rowmax-PoT exponent inside which an fp32 computation may round differently
POT_AMBIGUOUS_BAND = 1e-4
# relative half-width of the band around an e4m3 rounding midpoint inside which the
# fp32 weights of the FP8 P.V product may round differently
FP8_AMBIGUOUS_BAND = 2e-4
# the FP8 P.V weights are quantised as e4m3(2^FP8_P_SHIFT * p) * 2^-FP8_P_SHIFT
FP8_P_SHIFT = 8
E4M3_MAX = 448.0


# ---------------------------------------------------------------------------
# the steps of one (query tile, key tile) visit
# ---------------------------------------------------------------------------
def _tile_logits(qrows: np.ndarray, ktile: np.ndarray, scale: float, qpos: np.ndarray,
                 kidx: np.ndarray, causal: bool) -> np.ndarray:
    """Scaled logits s_rc = (q_r . k_c) * scale, -inf where key c is not visible."""
    s = (qrows @ ktile.T) * scale
    if causal:
        s = np.where(kidx[None, :] > qpos[:, None], NEG_INF, s)
    return s


def _row_gap(m_loc: np.ndarray, m_run: np.ndarray) -> np.ndarray:
    """Gap d_r = m~_r - m_r, with -inf for an empty row and +inf before any key."""
    with np.errstate(invalid="ignore"):
        d = m_loc - m_run
    d = np.where(m_run == NEG_INF, np.inf, d)
    d = np.where(m_loc == NEG_INF, NEG_INF, d)
    return d


def _vote(d: np.ndarray, lam: float) -> Tuple[bool, float]:
    """Skip iff lambda > 0 and every row has d_r < ln(lambda).

    Returns (skip, margin) where margin = |max_r d_r - ln(lambda)| in nats is
    how far the decision is from flipping (+inf when it cannot flip).
    """
    if lam <= 0.0:
        return False, math.inf
    thr = math.log(lam)
    dmax = float(np.max(d))
    skip = bool(np.all(d < thr))
    margin = math.inf if math.isinf(dmax) else abs(dmax - thr)
    return skip, margin


def _online_update(m: np.ndarray, l: np.ndarray, o: np.ndarray, s: np.ndarray,
                   vtile: np.ndarray):
    """Exact online-softmax update of (running max, row sum, output) by one tile."""
    m_new = np.maximum(m, np.max(s, axis=1))
    with np.errstate(invalid="ignore"):
        alpha = np.where(m == NEG_INF, 0.0, np.exp(m - m_new))
        p = np.where(s == NEG_INF, 0.0, np.exp(s - m_new[:, None]))
    l_new = alpha * l + p.sum(axis=1)
    o_new = alpha[:, None] * o + p @ vtile
    return m_new, l_new, o_new


def _pot_weights(s: np.ndarray, m_new: np.ndarray):
    """Rowmax-PoT weights of one tile: (w, ambiguous) with w_rc = 2^round((s - m')*log2 e),
    0 below 2^-126.5, and ambiguous_rc true where the exponent is within
    POT_AMBIGUOUS_BAND of a rounding boundary."""
    with np.errstate(invalid="ignore"):
        x = (s - m_new[:, None]) * LOG2E              # <= 0; -inf for masked keys
    x = np.maximum(x, -127.0)
    n = np.rint(x)                                    # ties to even
    w = np.where(n < -126.0, 0.0, np.exp2(n))
    amb = (np.abs(x - (np.floor(x) + 0.5)) < POT_AMBIGUOUS_BAND) & (x > -127.0)
    return w, amb


def _online_update_pot(m: np.ndarray, l: np.ndarray, o: np.ndarray, a: np.ndarray,
                       s: np.ndarray, vtile: np.ndarray):
    """The online update with Rowmax-PoT weights; `a` is the running weight of
    ambiguous keys, in the units of l."""
    m_new = np.maximum(m, np.max(s, axis=1))
    with np.errstate(invalid="ignore"):
        alpha = np.where(m == NEG_INF, 0.0, np.exp(m - m_new))
    w, amb = _pot_weights(s, m_new)
    l_new = alpha * l + w.sum(axis=1)
    o_new = alpha[:, None] * o + w @ vtile
    a_new = alpha * a + (w * amb).sum(axis=1)
    return m_new, l_new, o_new, a_new


def e4m3_step(y: np.ndarray) -> np.ndarray:
    """Spacing of the e4m3 values around |y| (y finite): 2^(e-3) in the binade
    [2^e, 2^(e+1)) for e >= -6, and the subnormal step 2^-9 below 2^-6."""
    a = np.abs(y)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))     # a = f * 2^ex, f in [0.5, 1)
    e = ex - 1
    return np.where(a >= 2.0 ** -6, np.exp2(e - 3.0), 2.0 ** -9)


def e4m3_round(y: np.ndarray) -> np.ndarray:
    """Round to the nearest OCP E4M3 value, ties to even, saturating at +-448."""
    y = np.asarray(y, dtype=np.float64)
    q = e4m3_step(y)
    r = np.rint(y / q) * q          # y / q is exact (a power-of-two scale); rint ties to even
    return np.clip(r, -E4M3_MAX, E4M3_MAX)


def _fp8_pv_weights(p: np.ndarray):
    """(w, ambiguous): w = e4m3(2^8 p) 2^-8, ambiguous where 2^8 p is within a relative
    FP8_AMBIGUOUS_BAND of an e4m3 rounding midpoint (p > 0)."""
    y = p * 2.0 ** FP8_P_SHIFT
    w = e4m3_round(y) * 2.0 ** -FP8_P_SHIFT
    q = e4m3_step(y)
    frac = y / q - np.floor(y / q)
    amb = (np.abs(frac - 0.5) * q < FP8_AMBIGUOUS_BAND * y) & (p > 0)
    return w, amb


def _online_update_fp8_pv(m: np.ndarray, l: np.ndarray, o: np.ndarray, a: np.ndarray,
                          s: np.ndarray, vtile: np.ndarray):
    """The online update with e4m3-quantised weights in P.V (l keeps the exact weights);
    `a` is the running weight, in the units of l, of keys with an ambiguous rounding."""
    m_new = np.maximum(m, np.max(s, axis=1))
    with np.errstate(invalid="ignore"):
        alpha = np.where(m == NEG_INF, 0.0, np.exp(m - m_new))
        p = np.where(s == NEG_INF, 0.0, np.exp(s - m_new[:, None]))
    w, amb = _fp8_pv_weights(p)
    l_new = alpha * l + p.sum(axis=1)
    o_new = alpha[:, None] * o + w @ vtile
    a_new = alpha * a + (p * amb).sum(axis=1)
    return m_new, l_new, o_new, a_new


def _finish(m: np.ndarray, l: np.ndarray, o: np.ndarray):
    return o / l[:, None], m + np.log(l)


# ---------------------------------------------------------------------------
# prefill
# ---------------------------------------------------------------------------
@dataclass
class PrefillResult:
    o: np.ndarray       # [B][Hq][Sq][D]
    lse: np.ndarray     # [B][Hq][Sq] natural log
    mask: np.ndarray    # int8 [B][Hq][nqt][nkt]: -1 not visited, 0 kept, 1 skipped
    margin: np.ndarray  # fp64, same shape; +inf where the decision cannot flip
    # Rowmax-PoT only: per row, the fraction of the weight sum carried by keys whose
    # exponent rounding is ambiguous in fp32 (None for exact exponentials)
    pot_ambiguous: Optional[np.ndarray] = None

    @property
    def skip_counts(self) -> np.ndarray:
        """Skipped tiles per query head, summed over batch and query tiles."""
        return (self.mask == 1).sum(axis=(0, 2, 3))

    @property
    def visited_counts(self) -> np.ndarray:
        return (self.mask >= 0).sum(axis=(0, 2, 3))


def last_visible_key(r1: int, Sq: int, Skv: int, causal: bool) -> int:
    """Last key index any row < r1 of the query tile can see."""
    return min(Skv - 1, r1 - 1 + (Skv - Sq)) if causal else Skv - 1


def prefill_qtile(qh: np.ndarray, kh: np.ndarray, vh: np.ndarray, t: int, *, tile_q: int,
                  tile_k: int, causal: bool, lam: float, scale: float, pot: bool = False,
                  block_mask_row: Optional[np.ndarray] = None, fp8_pv: bool = False):
    """One query tile of one head: returns (o_rows, lse_rows, mask[nkt], margin[nkt],
    ambiguous_fraction_rows or None).

    qh is the head's full query matrix [Sq][D]; kh, vh its kv head [Skv][D].  With
    pot=True kept tiles take Rowmax-PoT weights instead of exact exponentials; with
    fp8_pv=True their weights enter P.V quantised to e4m3 (the FP8 P.V reading above) and
    the fifth result is the ambiguous fraction of that rounding.
    block_mask_row, if given, is a boolean [nkt] of the key tiles this query tile visits.
    """
    Sq, Skv = qh.shape[0], kh.shape[0]
    nkt = (Skv + tile_k - 1) // tile_k
    r0, r1 = t * tile_q, min((t + 1) * tile_q, Sq)
    qrows = qh[r0:r1]
    qpos = np.arange(r0, r1) + (Skv - Sq)
    n = r1 - r0
    m = np.full(n, NEG_INF)
    l = np.zeros(n)
    o = np.zeros((n, qh.shape[1]))
    a = np.zeros(n)
    mask = np.full(nkt, -1, dtype=np.int8)
    margin = np.full(nkt, np.inf)
    last_tile = last_visible_key(r1, Sq, Skv, causal) // tile_k
    for j in range(last_tile + 1):
        if block_mask_row is not None and not block_mask_row[j]:
            continue                       # not selected: not visited (mask stays -1)
        c0, c1 = j * tile_k, min((j + 1) * tile_k, Skv)
        s = _tile_logits(qrows, kh[c0:c1], scale, qpos, np.arange(c0, c1), causal)
        d = _row_gap(np.max(s, axis=1), m)
        skip, mg = _vote(d, lam)
        mask[j] = 1 if skip else 0
        margin[j] = mg
        if skip:
            continue
        if pot:
            m, l, o, a = _online_update_pot(m, l, o, a, s, vh[c0:c1])
        elif fp8_pv:
            m, l, o, a = _online_update_fp8_pv(m, l, o, a, s, vh[c0:c1])
        else:
            m, l, o = _online_update(m, l, o, s, vh[c0:c1])
    seen = l > 0.0                         # rows with at least one visited visible key
    lsafe = np.where(seen, l, 1.0)
    amb = np.where(seen, a / lsafe, 0.0) if (pot or fp8_pv) else None
    o, lse = _finish(m, lsafe, o)
    o = np.where(seen[:, None], o, 0.0)
    lse = np.where(seen, lse, NEG_INF)
    return o, lse, mask, margin, amb


def prefill(q: np.ndarray, k: np.ndarray, v: np.ndarray, *, causal: bool, lam: float,
            tile_q: int, tile_k: int, scale: Optional[float] = None,
            pot: bool = False, block_mask: Optional[np.ndarray] = None,
            fp8_pv: bool = False) -> PrefillResult:
    """Skip Softmax prefill over q [B][Hq][Sq][D], k/v [B][Hkv][Skv][D] (fp64); pot=True
    uses Rowmax-PoT weights on kept tiles, fp8_pv=True e4m3-quantised weights in P.V
    (pot_ambiguous then holds that rounding's ambiguous fraction); block_mask, if given,
    is a boolean
    [B][Hq][nqt][nkt] of the (query tile, key tile) pairs to visit."""
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    if Hq % Hkv or (causal and Sq > Skv):
        raise ValueError("invalid shapes")
    if pot and fp8_pv:
        raise ValueError("pot and fp8_pv are separate readings")
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    nqt = (Sq + tile_q - 1) // tile_q
    nkt = (Skv + tile_k - 1) // tile_k
    o = np.zeros((B, Hq, Sq, D))
    lse = np.zeros((B, Hq, Sq))
    mask = np.full((B, Hq, nqt, nkt), -1, dtype=np.int8)
    margin = np.full((B, Hq, nqt, nkt), np.inf)
    amb = np.zeros((B, Hq, Sq)) if (pot or fp8_pv) else None
    for b in range(B):
        for h in range(Hq):
            kh, vh = k[b, h // G], v[b, h // G]
            for t in range(nqt):
                r0, r1 = t * tile_q, min((t + 1) * tile_q, Sq)
                ot, lt, mt, gt, at = prefill_qtile(
                    q[b, h], kh, vh, t, tile_q=tile_q, tile_k=tile_k, causal=causal, lam=lam,
                    scale=scale, pot=pot, fp8_pv=fp8_pv,
                    block_mask_row=None if block_mask is None else block_mask[b, h, t])
                o[b, h, r0:r1], lse[b, h, r0:r1] = ot, lt
                mask[b, h, t], margin[b, h, t] = mt, gt
                if pot or fp8_pv:
                    amb[b, h, r0:r1] = at
    return PrefillResult(o, lse, mask, margin, amb)


# ---------------------------------------------------------------------------
# decode (split-KV, one query token per sequence)
# ---------------------------------------------------------------------------
@dataclass
class DecodeResult:
    o: np.ndarray       # [B][Hq][D]
    lse: np.ndarray     # [B][Hq]
    mask: np.ndarray    # int8 [B][Hkv][nblk]: 0 kept, 1 skipped, -1 not selected
    margin: np.ndarray  # [B][Hkv][nblk]
    num_splits: int     # splits actually used (after dropping empty ones)

    @property
    def skip_counts(self) -> np.ndarray:
        """Skipped key tiles per query head: a group's count is given to each of its heads."""
        B, Hkv, _ = self.mask.shape
        G = self.o.shape[1] // Hkv
        return np.repeat((self.mask == 1).sum(axis=(0, 2)), G)


def decode_split_geometry(Skv: int, tile_k: int, num_splits: int) -> Tuple[int, int, int]:
    """(key tiles, tiles per split, non-empty splits) of a split-KV decode."""
    nblk = (Skv + tile_k - 1) // tile_k
    per = (nblk + num_splits - 1) // num_splits
    return nblk, per, (nblk + per - 1) // per


def decode_group(qg: np.ndarray, kh: np.ndarray, vh: np.ndarray, *, lam: float,
                 num_splits: int, tile_k: int = 64, scale: Optional[float] = None,
                 block_mask: Optional[np.ndarray] = None):
    """One GQA group: qg [G][D] against kv head kh, vh [Skv][D].

    block_mask, if given, is a boolean [nblk] of the key tiles to visit.
    Returns (o [G][D], lse [G], mask [nblk], margin [nblk], per-split (o, lse) list).
    """
    G, D = qg.shape
    Skv = kh.shape[0]
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    nblk, per, nsplit = decode_split_geometry(Skv, tile_k, num_splits)
    mask = np.zeros(nblk, dtype=np.int8)
    margin = np.full(nblk, np.inf)
    parts: List[Tuple[np.ndarray, np.ndarray]] = []
    for sp in range(nsplit):
        m = np.full(G, NEG_INF)
        l = np.zeros(G)
        o = np.zeros((G, D))
        for j in range(sp * per, min((sp + 1) * per, nblk)):
            if block_mask is not None and not block_mask[j]:
                mask[j] = -1
                continue
            c0, c1 = j * tile_k, min((j + 1) * tile_k, Skv)
            s = _tile_logits(qg, kh[c0:c1], scale, np.zeros(G), np.arange(c0, c1), False)
            d = _row_gap(np.max(s, axis=1), m)
            skip, mg = _vote(d, lam)
            mask[j] = 1 if skip else 0
            margin[j] = mg
            if skip:
                continue
            m, l, o = _online_update(m, l, o, s, vh[c0:c1])
        if np.all(l == 0.0):       # no selected tile in this split
            parts.append((np.zeros((G, D)), np.full(G, NEG_INF)))
        else:
            parts.append(_finish(m, l, o))
    # exact log-sum-exp combine of the split results (empty splits weigh 0)
    lses = np.stack([p[1] for p in parts])          # [nsplit][G]
    top = lses.max(axis=0)
    if np.all(top == NEG_INF):
        return np.zeros((G, D)), np.full(G, NEG_INF), mask, margin, parts
    wts = np.exp(lses - top[None, :])
    o = sum(wts[i][:, None] * parts[i][0] for i in range(nsplit)) / wts.sum(axis=0)[:, None]
    lse = top + np.log(wts.sum(axis=0))
    return o, lse, mask, margin, parts


def decode(q: np.ndarray, k: np.ndarray, v: np.ndarray, *, lam: float, num_splits: int,
           tile_k: int = 64, scale: Optional[float] = None,
           block_mask: Optional[np.ndarray] = None) -> DecodeResult:
    """Skip Softmax decode: q [B][Hq][D], k/v [B][Hkv][Skv][D] (fp64); block_mask, if given,
    is a boolean [B][Hkv][nblk] of the key tiles each group visits."""
    B, Hq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    nblk, _, nsplit = decode_split_geometry(Skv, tile_k, num_splits)
    o = np.zeros((B, Hq, D))
    lse = np.zeros((B, Hq))
    mask = np.zeros((B, Hkv, nblk), dtype=np.int8)
    margin = np.zeros((B, Hkv, nblk))
    for b in range(B):
        for hk in range(Hkv):
            og, lg, mg, gg, _ = decode_group(q[b, hk * G:(hk + 1) * G], k[b, hk], v[b, hk],
                                             lam=lam, num_splits=num_splits, tile_k=tile_k,
                                             scale=scale,
                                             block_mask=None if block_mask is None
                                             else block_mask[b, hk])
            o[b, hk * G:(hk + 1) * G], lse[b, hk * G:(hk + 1) * G] = og, lg
            mask[b, hk], margin[b, hk] = mg, gg
    return DecodeResult(o, lse, mask, margin, nsplit)


# ---------------------------------------------------------------------------
# dense attention and the skipped probability mass (diagnostics)
# ---------------------------------------------------------------------------
def dense_attention(qh: np.ndarray, kh: np.ndarray, vh: np.ndarray, *, causal: bool,
                    scale: Optional[float] = None, key_keep: Optional[np.ndarray] = None):
    """Plain softmax(q k^T * scale + mask) v for one head; returns (o, lse, p).

    key_keep, if given, is a boolean [Sq][Skv] matrix of keys allowed per row.
    """
    Sq, D = qh.shape
    Skv = kh.shape[0]
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    s = (qh @ kh.T) * scale
    allowed = np.ones((Sq, Skv), dtype=bool)
    if causal:
        allowed &= np.arange(Skv)[None, :] <= (np.arange(Sq) + (Skv - Sq))[:, None]
    if key_keep is not None:
        allowed &= key_keep
    s = np.where(allowed, s, NEG_INF)
    mx = s.max(axis=1, keepdims=True)
    e = np.where(allowed, np.exp(s - mx), 0.0)
    z = e.sum(axis=1, keepdims=True)
    p = e / z
    return p @ vh, (mx + np.log(z))[:, 0], p


def skipped_mass(p_dense: np.ndarray, skipped_keys: np.ndarray) -> np.ndarray:
    """epsilon_r: dense softmax probability that row r puts on skipped keys."""
    return (p_dense * skipped_keys).sum(axis=1)
