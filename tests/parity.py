"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
the CPU oracle on the same seeded inputs, then apply the gate."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from oracle import gate
from attention_forward_gb300 import fa, inputs

FMT = {"bf16": oracle.FMT_BF16, "fp16": oracle.FMT_F16}


def sample_rows(B, H, Sq, per_head=8, extra=256, seed=0):
    """Flat row indices: for every (b, h) the first and last row and rows at
    tile edges (127/128/255/256 ...), plus random rows."""
    rng = np.random.default_rng(seed)
    edges = [0, Sq - 1]
    for t in range(128, Sq, 128):
        edges += [t - 1, t]
    edges = sorted(set(e for e in edges if 0 <= e < Sq))
    rows = []
    for bh in range(B * H):
        pick = list(rng.choice(edges, size=min(len(edges), per_head // 2),
                               replace=False)) + [0, Sq - 1]
        pick += list(rng.integers(0, Sq, size=per_head // 2))
        rows += [bh * Sq + int(i) for i in pick]
    rows += list(rng.integers(0, B * H * Sq, size=extra))
    return np.unique(np.array(rows, dtype=np.int64))


def run_kernel(q, k, v, causal, flags=0, num_splits=0, scale=None,
               workspace=None):
    dq, dk, dv = (t.cuda() for t in (q, k, v))
    if flags or num_splits or workspace is not None:
        o, lse = fa.fa_fwd_ex(dq, dk, dv, causal=causal, flags=flags,
                              num_splits=num_splits, scale=scale,
                              workspace=workspace)
    else:
        o, lse = fa.fa_fwd(dq, dk, dv, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    return o, lse


def check(q, k, v, o, lse, causal, dtype, rows=None, scale=None):
    """Gate the kernel's (o, lse) against the oracle on all rows or on the
    listed flat rows.  Returns the GateResult."""
    B, H, Sq, D = q.shape
    sc = float(D) ** -0.5 if scale is None else scale
    qf, kf, vf = (t.float().numpy() for t in (q, k, v))
    o_k = o.float().cpu().numpy()
    l_k = lse.cpu().numpy()
    o_ref, l_ref = oracle.attention(qf, kf, vf, sc, causal, rows=rows)
    o_fl, _ = oracle.floor_attention(qf, kf, vf, sc, causal, FMT[dtype],
                                     rows=rows)
    if rows is not None:
        o_k = o_k.reshape(-1, D)[rows]
        l_k = l_k.reshape(-1)[rows]
    return gate.check(o_k, l_k, o_ref, l_ref, o_fl, dtype)


def run_and_check(B, H, Sq, Skv, D, dtype, causal, seed, qk_mult=1.0,
                  rows="all", **kw):
    q, k, v = inputs.make_qkv(B, H, Sq, Skv, D, dtype, seed, qk_mult)
    o, lse = run_kernel(q, k, v, causal, **kw)
    r = None if isinstance(rows, str) else rows
    return check(q, k, v, o, lse, causal, dtype, rows=r)
