"""fp64 restatement of the tiled online-softmax algorithm -- TEST INFRASTRUCTURE.

This is NOT the oracle (the oracle is the plain three-step definition in
``attn_oracle.c``).  It restates, step by step and in fp64, the algorithm the
CUDA kernels run, so that the tests can show on the CPU, before any GPU run,
that (1) the tiled online softmax with the log2-domain scale reaches the
three-step result, (2) the split-KV combine reaches it too, and (3) the parity
gate rejects the plausible mistakes one could make in that algorithm.

Algorithm (the online softmax of "The FA5090 Optimization Journey" section 2.2
and of the FlashAttention-2 kernel on "Three kernels for a chip the ecosystem
skipped" (Kernel one), with the exp2 trick of the FA5090 page section 2.6 and
the fused log2 scale of the B300 G5 page, V33 "log2exp2"):
  c = scale * log2(e); per query row keep m (running max of c*s, log2 units),
  l (running sum) and an unnormalised accumulator acc.  For each key tile:
      t     = c * (q . k_j)                      masked keys -> -inf
      m_new = max(m, max_j t)
      alpha = 2^(m - m_new)                      (1 when m does not change)
      p_j   = 2^(t_j - m_new)
      l     = alpha * l + sum_j p_j
      acc   = alpha * acc + sum_j p_j v_j
      m     = m_new
  then O = acc / l and LSE = (m + log2 l) * ln 2.
A row whose tiles are all masked keeps m = -inf; it ends with O = 0 and
LSE = -inf.

Planted mistakes (``mutation=``) exist only to show that the gate catches
them; they are never used for a parity claim.
"""
from __future__ import annotations

import math

import numpy as np

LOG2E = 1.0 / math.log(2.0)
LN2 = math.log(2.0)

MUTATIONS = (
    "no_o_rescale",        # acc not multiplied by alpha
    "no_l_rescale",        # l not multiplied by alpha
    "alpha_after_update",  # alpha computed after m is overwritten (always 1)
    "causal_off_by_one",   # key j visible iff j < i + (Skv - Sq)
    "no_normalize",        # O = acc, the final 1/l dropped
    "drop_tail_tile",      # ragged last key tile skipped
    "scale_twice",         # scale applied twice
    "transposed_pv",       # P.V with V's rows reversed inside a tile
)


def _visible(Sq: int, Skv: int, causal: bool, mutation):
    i = np.arange(Sq)[:, None]
    j = np.arange(Skv)[None, :]
    if not causal:
        return np.ones((Sq, Skv), bool)
    if mutation == "causal_off_by_one":
        return j < i + (Skv - Sq)
    return j <= i + (Skv - Sq)


def online_attention(q, k, v, scale: float, causal: bool, block_n: int = 128,
                     p_round=None, mutation: str | None = None):
    """Tile-wise online softmax over key tiles of ``block_n`` keys, fp64.

    q [B,H,Sq,D], k/v [B,H,Skv,D].  ``p_round`` (a function on fp64 arrays)
    rounds p where it enters P.V (the row sum l keeps the unrounded p) and
    rounds the output, to mimic a 16-bit pipeline.  Returns (o [B,H,Sq,D], lse [B,H,Sq])."""
    if mutation is not None and mutation not in MUTATIONS:
        raise ValueError(mutation)
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    B, H, Sq, D = q.shape
    Skv = k.shape[2]
    c = scale * LOG2E
    if mutation == "scale_twice":
        c = scale * scale * LOG2E
    vis = _visible(Sq, Skv, causal, mutation)
    o = np.zeros((B, H, Sq, D))
    lse = np.zeros((B, H, Sq))
    n_tiles = -(-Skv // block_n)
    for b in range(B):
        for h in range(H):
            Q, K, V = q[b, h], k[b, h], v[b, h]
            m = np.full(Sq, -np.inf)
            l = np.zeros(Sq)
            acc = np.zeros((Sq, D))
            for t in range(n_tiles):
                j0, j1 = t * block_n, min(Skv, (t + 1) * block_n)
                if mutation == "drop_tail_tile" and j1 - j0 < block_n:
                    continue
                s = c * (Q @ K[j0:j1].T)
                s = np.where(vis[:, j0:j1], s, -np.inf)
                m_new = np.maximum(m, s.max(axis=1))
                # rows that have seen no visible key yet keep a finite anchor
                m_use = np.where(np.isfinite(m_new), m_new, 0.0)
                if mutation == "alpha_after_update":
                    m = m_new
                alpha = np.where(np.isfinite(m), np.exp2(m - m_use), 0.0)
                p = np.exp2(s - m_use[:, None])
                # l sums the unrounded p; only the P.V operand is rounded
                l = (l if mutation == "no_l_rescale" else alpha * l) + p.sum(1)
                if p_round is not None:
                    p = p_round(p)
                Vt = V[j0:j1][::-1] if mutation == "transposed_pv" else V[j0:j1]
                acc = (acc if mutation == "no_o_rescale"
                       else alpha[:, None] * acc) + p @ Vt
                m = m_new
            ok = l > 0
            if mutation == "no_normalize":
                out = acc
            else:
                out = np.where(ok[:, None], acc / np.where(ok, l, 1.0)[:, None],
                               0.0)
            if p_round is not None:
                out = p_round(out)
            o[b, h] = out
            with np.errstate(divide="ignore"):
                lse[b, h] = np.where(ok, (m + np.log2(np.where(ok, l, 1.0))) * LN2,
                                     -np.inf)
    return o, lse


def combine_partials(o_parts, lse_parts):
    """Split-KV combine: each split s covers a disjoint slice of the keys and
    holds its own normalised output O_s and LSE_s.  Then
        LSE = log sum_s exp(LSE_s),   O = sum_s exp(LSE_s - LSE) * O_s.
    Splits with LSE_s = -inf (no visible key) carry weight 0; if every split
    is empty the row is O = 0, LSE = -inf.

    o_parts [S, ..., D], lse_parts [S, ...]."""
    o_parts = np.asarray(o_parts, np.float64)
    lse_parts = np.asarray(lse_parts, np.float64)
    mx = lse_parts.max(axis=0)
    anchor = np.where(np.isfinite(mx), mx, 0.0)
    w = np.exp(lse_parts - anchor)            # exp(-inf) = 0
    tot = w.sum(axis=0)
    ok = tot > 0
    with np.errstate(divide="ignore"):
        lse = np.where(ok, anchor + np.log(np.where(ok, tot, 1.0)), -np.inf)
    wn = np.where(ok, w / np.where(ok, tot, 1.0), 0.0)
    o = (wn[..., None] * o_parts).sum(axis=0)
    return o, lse
