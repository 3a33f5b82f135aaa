"""Parity past 2^31 elements per tensor: B2 H130 S65536 D128 bf16 causal, so
that every element offset of Q, K, V and O past 2^31 (and every byte offset
past 2^32) is exercised.  Sampled rows against the fp64 oracle, on the CTA
pairs (the default here) and on single CTAs.  Gate: oracle/gate.py."""
import numpy as np
import pytest
import torch

import oracle
from oracle import gate
from attention_forward_gb300 import fa, inputs
from parity import FMT

pytestmark = pytest.mark.gpu

B, H, S, D, DT, CAUSAL, SEED = 2, 130, 65536, 128, "bf16", True, 31


@pytest.fixture(scope="module")
def big():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()
    assert B * H * S * D > 2 ** 31
    dev = torch.device("cuda")
    q, k, v = (torch.empty((B * H, S, D), dtype=inputs.DTYPES[DT], device=dev) for _ in range(3))
    chunk = 26
    for h0 in range(0, B * H, chunk):
        hs = list(range(h0, min(B * H, h0 + chunk)))
        cq, ck, cv = inputs.make_qkv(B, H, S, S, D, DT, SEED, heads=hs)
        q[hs[0]:hs[-1] + 1].copy_(cq)
        k[hs[0]:hs[-1] + 1].copy_(ck)
        v[hs[0]:hs[-1] + 1].copy_(cv)
    yield q.view(B, H, S, D), k.view(B, H, S, D), v.view(B, H, S, D)
    del q, k, v
    torch.cuda.empty_cache()


def _rows(seed):
    """Rows of 16 heads (flat indices into B*H*S): the first and last head,
    the heads on either side of the batch boundary and 12 random ones; per
    head its first and last row, three rows at 128-row tile edges and 15
    random rows."""
    rng = np.random.default_rng(seed)
    heads = {0, H - 1, H, B * H - 1}
    while len(heads) < 16:
        heads.add(int(rng.integers(0, B * H)))
    rows = []
    for bh in sorted(heads):
        rows += [bh * S, bh * S + S - 1]
        rows += [bh * S + 128 * int(t) - int(rng.integers(0, 2)) for t in rng.integers(1, S // 128, size=3)]
        rows += [bh * S + int(i) for i in rng.integers(0, S, size=15)]
    return np.unique(np.array(rows, dtype=np.int64))


def _check(o, lse, rows):
    heads = sorted(set(int(r) // S for r in rows))
    pos = {h: n for n, h in enumerate(heads)}
    local = np.array([pos[int(r) // S] * S + int(r) % S for r in rows], dtype=np.int64)
    q, k, v = inputs.make_qkv(B, H, S, S, D, DT, SEED, heads=heads)
    qf, kf, vf = (t.float().numpy()[None] for t in (q, k, v))
    sc = float(D) ** -0.5
    o_ref, l_ref = oracle.attention(qf, kf, vf, sc, CAUSAL, rows=local)
    o_fl, _ = oracle.floor_attention(qf, kf, vf, sc, CAUSAL, FMT[DT], rows=local)
    idx = torch.from_numpy(rows).to(o.device)
    o_k = o.view(-1, D).index_select(0, idx).float().cpu().numpy()
    l_k = lse.view(-1).index_select(0, idx).cpu().numpy()
    return gate.check(o_k, l_k, o_ref, l_ref, o_fl, DT)


@pytest.mark.parametrize("kernel", ["pair", "single"])
def test_tensors_past_2_31_elements_sampled_rows(big, kernel):
    q, k, v = big
    flags = fa.FA_FLAG_SINGLE_CTA if kernel == "single" else 0
    assert fa.fa_prefill_uses_pairs(B, H, S, S, D, CAUSAL, flags) == (kernel == "pair")
    o, lse = fa.fa_fwd_ex(q, k, v, causal=CAUSAL, flags=flags)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    r = _check(o, lse, _rows(7 if kernel == "pair" else 8))
    assert r.passed, str(r)
