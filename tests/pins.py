"""Independent checks ("pins") of the oracle.

Each function recomputes a property of Skip Softmax attention by a route that
does not go through the oracle's tile loop, and raises AssertionError when the
oracle disagrees.  The same functions are run against deliberately broken
copies of the oracle (test_oracle_mutants.py) to show that they catch the
mistakes one would plausibly make.
"""

from __future__ import annotations

import math

import numpy as np
import torch
import torch.nn.functional as F

import oracle

NEG_INF = -np.inf


# ---------------------------------------------------------------------------
# library routine: dense (optionally key-masked) attention via torch SDPA fp64
# ---------------------------------------------------------------------------
def sdpa(qh: np.ndarray, kh: np.ndarray, vh: np.ndarray, allowed: np.ndarray, scale: float):
    """softmax(q k^T scale) v restricted to `allowed` [Sq][Skv], by torch's SDPA (fp64, CPU)."""
    q = torch.tensor(np.asarray(qh, dtype=np.float64))[None, None]
    k = torch.tensor(np.asarray(kh, dtype=np.float64))[None, None]
    v = torch.tensor(np.asarray(vh, dtype=np.float64))[None, None]
    m = torch.tensor(np.asarray(allowed, dtype=bool))[None, None]
    return F.scaled_dot_product_attention(q, k, v, attn_mask=m, scale=scale)[0, 0].numpy()


def causal_allowed(Sq: int, Skv: int, causal: bool) -> np.ndarray:
    if not causal:
        return np.ones((Sq, Skv), dtype=bool)
    return np.arange(Skv)[None, :] <= (np.arange(Sq) + (Skv - Sq))[:, None]


def rel_err(a: np.ndarray, b: np.ndarray) -> float:
    return float(np.max(np.abs(a - b)) / max(1e-300, float(np.max(np.abs(b)))))


# ---------------------------------------------------------------------------
# closed-form skip mask from prefix maxima of the full logit matrix
# ---------------------------------------------------------------------------
def prefill_mask_closed_form(qh, kh, *, causal, lam, tile_q, tile_k, scale):
    """Skip mask of one head from the full logits and prefix maxima over key tiles.

    Because a skipped tile's local max is below the running max (lambda <= 1),
    the running max before key tile j is the max of all visible logits in tiles
    < j, whatever was skipped.  So the mask follows from cumulative maxima
    without any online-softmax state.
    """
    Sq, Skv = qh.shape[0], kh.shape[0]
    s = (qh @ kh.T) * scale
    s = np.where(causal_allowed(Sq, Skv, causal), s, NEG_INF)
    nkt = (Skv + tile_k - 1) // tile_k
    nqt = (Sq + tile_q - 1) // tile_q
    pad = nkt * tile_k - Skv
    sp = np.concatenate([s, np.full((Sq, pad), NEG_INF)], axis=1)
    tmax = sp.reshape(Sq, nkt, tile_k).max(axis=2)                  # [Sq][nkt]
    before = np.concatenate([np.full((Sq, 1), NEG_INF),
                             np.maximum.accumulate(tmax, axis=1)[:, :-1]], axis=1)
    with np.errstate(invalid="ignore"):
        gap = np.where(tmax == NEG_INF, NEG_INF, np.where(before == NEG_INF, np.inf, tmax - before))
    thr = math.log(lam) if lam > 0 else NEG_INF
    mask = np.full((nqt, nkt), -1, dtype=np.int8)
    for t in range(nqt):
        r0, r1 = t * tile_q, min((t + 1) * tile_q, Sq)
        last = (min(Skv - 1, r1 - 1 + Skv - Sq) if causal else Skv - 1) // tile_k
        g = gap[r0:r1, :last + 1]
        mask[t, :last + 1] = (lam > 0) & np.all(g < thr, axis=0)
    return mask


def decode_mask_closed_form(qg, kh, *, lam, num_splits, tile_k, scale):
    """Decode skip mask of one GQA group from prefix maxima restarted per split."""
    Skv = kh.shape[0]
    s = (qg @ kh.T) * scale                                        # [G][Skv]
    nblk, per, nsplit = oracle.decode_split_geometry(Skv, tile_k, num_splits)
    pad = nblk * tile_k - Skv
    sp = np.concatenate([s, np.full((s.shape[0], pad), NEG_INF)], axis=1)
    tmax = sp.reshape(s.shape[0], nblk, tile_k).max(axis=2)          # [G][nblk]
    thr = math.log(lam) if lam > 0 else NEG_INF
    mask = np.zeros(nblk, dtype=np.int8)
    for sp_i in range(nsplit):
        a, b = sp_i * per, min((sp_i + 1) * per, nblk)
        seg = tmax[:, a:b]
        before = np.concatenate([np.full((seg.shape[0], 1), NEG_INF),
                                 np.maximum.accumulate(seg, axis=1)[:, :-1]], axis=1)
        gap = np.where(before == NEG_INF, np.inf, seg - before)
        mask[a:b] = (lam > 0) & np.all(gap < thr, axis=0)
    return mask


def kept_keys_prefill(mask_head, Sq, Skv, tile_q, tile_k, causal):
    """allowed[r][c]: key c visible to row r and its tile not skipped for r's query tile."""
    nkt = mask_head.shape[1]
    allowed = causal_allowed(Sq, Skv, causal).copy()
    tile_of_key = np.arange(Skv) // tile_k
    for t in range(mask_head.shape[0]):
        r0, r1 = t * tile_q, min((t + 1) * tile_q, Sq)
        skipped_tiles = mask_head[t] == 1
        allowed[r0:r1] &= ~skipped_tiles[tile_of_key][None, :]
    assert nkt * tile_k >= Skv
    return allowed


# ---------------------------------------------------------------------------
# pins on a prefill problem
# ---------------------------------------------------------------------------
def check_prefill(q, k, v, *, causal, lam, tile_q, tile_k, scale=None, lam_grid=None):
    """Run every prefill pin on one problem; returns the oracle result."""
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    res = oracle.prefill(q, k, v, causal=causal, lam=lam, tile_q=tile_q, tile_k=tile_k, scale=scale)
    for b in range(B):
        for h in range(Hq):
            qh, kh, vh = q[b, h], k[b, h // G], v[b, h // G]
            full = causal_allowed(Sq, Skv, causal)
            # (1) lambda = 0 reduces to dense attention (library routine)
            if lam == 0:
                ref = sdpa(qh, kh, vh, full, scale)
                assert rel_err(res.o[b, h], ref) < 1e-12, "lambda=0 differs from dense attention"
                assert not (res.mask[b, h] == 1).any()
            # (2) closed-form mask from prefix maxima
            cf = prefill_mask_closed_form(qh, kh, causal=causal, lam=lam, tile_q=tile_q,
                                          tile_k=tile_k, scale=scale)
            sure = res.margin[b, h] > 1e-9
            assert np.array_equal(cf[sure], res.mask[b, h][sure]), "mask differs from closed form"
            assert np.array_equal(cf < 0, res.mask[b, h] < 0), "visited set differs"
            # (3) output equals dense softmax over the kept keys (library routine)
            allowed = kept_keys_prefill(res.mask[b, h], Sq, Skv, tile_q, tile_k, causal)
            ref_kept = sdpa(qh, kh, vh, allowed, scale)
            assert rel_err(res.o[b, h], ref_kept) < 1e-12, "output differs from kept-key softmax"
            # (4) lse equals log-sum-exp over the kept keys
            s = np.where(allowed, (qh @ kh.T) * scale, NEG_INF)
            mx = s.max(axis=1)
            lse_ref = mx + np.log(np.exp(s - mx[:, None]).sum(axis=1))
            assert np.max(np.abs(res.lse[b, h] - lse_ref)) < 1e-10, "lse differs"
            # (5) analytic error bound against dense attention
            o_dense, _, p = oracle.dense_attention(qh, kh, vh, causal=causal, scale=scale)
            skipped = full & ~allowed
            eps = oracle.skipped_mass(p, skipped)
            vrange = vh.max(axis=0) - vh.min(axis=0)
            err = np.abs(o_dense - res.o[b, h])
            assert np.all(err <= eps[:, None] * vrange[None, :] + 1e-12), "error bound violated"
            nsk = skipped.sum(axis=1)
            assert np.all((eps < lam * nsk) | (nsk == 0)), "skipped mass above lambda * count"
    # (6) monotone skip sets in lambda
    if lam_grid is not None:
        prev = None
        for lg in sorted(lam_grid):
            r = oracle.prefill(q, k, v, causal=causal, lam=lg, tile_q=tile_q, tile_k=tile_k,
                               scale=scale)
            cur = r.mask == 1
            if prev is not None:
                assert np.all(cur | ~prev), "skip set not monotone in lambda"
            prev = cur
    return res


def check_decode(q, k, v, *, lam, num_splits, tile_k=64, scale=None):
    """Run every decode pin on one problem; returns the oracle result."""
    B, Hq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    res = oracle.decode(q, k, v, lam=lam, num_splits=num_splits, tile_k=tile_k, scale=scale)
    nblk = res.mask.shape[2]
    for b in range(B):
        for hk in range(Hkv):
            qg, kh, vh = q[b, hk * G:(hk + 1) * G], k[b, hk], v[b, hk]
            ones = np.ones((G, Skv), dtype=bool)
            if lam == 0:
                ref = sdpa(qg, kh, vh, ones, scale)
                assert rel_err(res.o[b, hk * G:(hk + 1) * G], ref) < 1e-12, "lambda=0 differs"
            cf = decode_mask_closed_form(qg, kh, lam=lam, num_splits=num_splits, tile_k=tile_k,
                                         scale=scale)
            sure = res.margin[b, hk] > 1e-9
            assert np.array_equal(cf[sure], res.mask[b, hk][sure]), "decode mask differs"
            keep_key = np.repeat(res.mask[b, hk] == 0, tile_k)[:Skv]
            allowed = np.broadcast_to(keep_key, (G, Skv))
            ref_kept = sdpa(qg, kh, vh, allowed, scale)
            assert rel_err(res.o[b, hk * G:(hk + 1) * G], ref_kept) < 1e-12, "decode output differs"
            o_dense, _, p = oracle.dense_attention(qg, kh, vh, causal=False, scale=scale)
            eps = oracle.skipped_mass(p, ~allowed)
            vrange = vh.max(axis=0) - vh.min(axis=0)
            err = np.abs(o_dense - res.o[b, hk * G:(hk + 1) * G])
            assert np.all(err <= eps[:, None] * vrange[None, :] + 1e-12), "decode bound violated"
            assert nblk * tile_k >= Skv
    return res
