"""The CTA-pair kernel's tail split (FA_FLAG_TAIL_SPLIT): when the 512-row
items leave the last round of pairs partly idle, each of the last items runs
as four items over a quarter of the key tiles, and the quarter that finishes
last merges the fp32 partials in the kernel.  Parity with the fp64 oracle on every row of shapes
that split (ragged rows and keys, Sq != Skv, one-tile and uneven quarters),
bitwise equality elsewhere, and the arrival counters across launches.
Gate: oracle/gate.py."""
import numpy as np
import pytest
import torch

from attention_forward_gb300 import fa, inputs
from parity import check, run_and_check, run_kernel

pytestmark = pytest.mark.gpu

PAIR = fa.FA_FLAG_PAIR
SPLIT = fa.FA_FLAG_PAIR | fa.FA_FLAG_TAIL_SPLIT
_DT = {"bf16": torch.bfloat16, "fp16": torch.float16}


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _assert(r):
    assert r.passed, str(r)


def _tail(B, H, Sq, Skv, dt="bf16", flags=SPLIT):
    return fa.fa_prefill_tail_items(B, H, Sq, Skv, 128, False, _DT[dt], flags)


def _split_heads(B, H, Sq, tail):
    """(batch*head) indices whose rows belong to split items: non-causal
    items are numbered head-major, and the split ones are the last."""
    n_q = (Sq + 511) // 512
    n_items = B * H * n_q
    return sorted({i // n_q for i in range(n_items - tail, n_items)})


CASES = [  # B, H, Sq, Skv, dtype, qk_mult
    (1, 96, 1024, 1024, "bf16", 1.0),   # 192 items: 40 split, quarters of 2 tiles
    (1, 40, 1000, 1000, "fp16", 2.0),   # ragged rows and keys: 4 items split
    (1, 80, 520, 1700, "bf16", 1.0),    # Sq != Skv, uneven quarters (3, 4, 3, 4 tiles)
    (1, 84, 1024, 512, "bf16", 1.0),    # four key tiles: one tile per quarter
    (2, 41, 600, 500, "fp16", 1.0),     # the last quarter one ragged tile
    (1, 96, 1024, 1024, "bf16", 2.0),   # sharper rows: quarters weigh unevenly
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_tail_split_all_rows(case):
    B, H, Sq, Skv, dt, mult = case
    assert _tail(B, H, Sq, Skv, dt) > 0
    _assert(run_and_check(B, H, Sq, Skv, 128, dt, False, 61, qk_mult=mult, flags=SPLIT))


def test_rows_of_unsplit_items_are_bitwise_unchanged():
    """The items before the split ones run as without the split, bit for
    bit; the split ones differ by the merge's rounding only and pass the
    gate (checked on those heads' rows)."""
    B, H, S = 4, 16, 2048
    tail = _tail(B, H, S, S)
    assert tail > 0
    q, k, v = inputs.make_qkv(B, H, S, S, 128, "bf16", 62)
    o1, l1 = run_kernel(q, k, v, False, flags=SPLIT)
    o0, l0 = run_kernel(q, k, v, False, flags=PAIR)
    heads = _split_heads(B, H, S, tail)
    keep = torch.ones(B * H, dtype=torch.bool)
    keep[heads] = False
    keep = keep.to(o1.device)
    f1, f0 = o1.reshape(B * H, S, -1), o0.reshape(B * H, S, -1)
    assert torch.equal(f1[keep], f0[keep])
    assert torch.equal(l1.reshape(B * H, S)[keep], l0.reshape(B * H, S)[keep])
    assert not torch.equal(f1[~keep], f0[~keep])  # the merge did run there
    rows = np.concatenate([np.arange(h * S, (h + 1) * S, 7) for h in heads])
    _assert(check(q, k, v, o1, l1, False, "bf16", rows=rows))


def test_tail_split_repeats_bitwise():
    """Whichever quarter arrives last, the merge reads the four partials in
    quarter order: repeated launches give the same bits."""
    q, k, v = inputs.make_qkv(1, 96, 1024, 1024, 128, "bf16", 63)
    ref = run_kernel(q, k, v, False, flags=SPLIT)
    for _ in range(4):
        o, lse = run_kernel(q, k, v, False, flags=SPLIT)
        assert torch.equal(o, ref[0]) and torch.equal(lse, ref[1])


def test_counters_carry_over_shapes_and_launches():
    """One stream, many launches with different split counts: every launch's
    arrivals are counted under its own epoch, so counts left by the previous
    launch (on the same or other items) never start a merge early."""
    shapes = [(1, 96, 1024, 1024), (1, 84, 1024, 512), (1, 80, 1024, 1024)]
    data = []
    for i, (B, H, Sq, Skv) in enumerate(shapes):
        assert _tail(B, H, Sq, Skv) > 0
        q, k, v = (t.cuda() for t in inputs.make_qkv(B, H, Sq, Skv, 128, "bf16", 64 + i))
        data.append((q, k, v, fa.fa_fwd_ex(q, k, v, flags=SPLIT)))
    torch.cuda.synchronize()
    for n in range(30):
        q, k, v, (ro, rl) = data[(n * 7) % 3]
        o, lse = fa.fa_fwd_ex(q, k, v, flags=SPLIT)
        torch.cuda.synchronize()
        assert torch.equal(o, ro) and torch.equal(lse, rl), n
    assert fa.fa_get_device_status() == fa.FA_OK


def test_after_an_aborted_launch():
    """A launch that the watchdog ends (a withheld K/V tile) leaves arrival
    counts behind; the next launch still merges every row once."""
    B, H, S = 1, 96, 1024
    assert _tail(B, H, S, S) > 0
    q, k, v = inputs.make_qkv(B, H, S, S, 128, "bf16", 65)
    dq, dk, dv = (t.cuda() for t in (q, k, v))
    ref = fa.fa_fwd_ex(dq, dk, dv, flags=SPLIT)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    fa.fa_set_watchdog_ns(20_000_000)
    try:
        fa.fa_fwd_ex(dq, dk, dv, flags=SPLIT | fa.FA_FLAG_TEST_STALL)
        assert fa.fa_get_device_status() == fa.FA_ERR_TIMEOUT
    finally:
        fa.fa_set_watchdog_ns(0)
    o, lse = fa.fa_fwd_ex(dq, dk, dv, flags=SPLIT)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    assert torch.equal(o, ref[0]) and torch.equal(lse, ref[1])


def test_selection_and_forms_agree():
    """The split needs the flag (fa_fwd never splits), pairs, a non-causal
    mask, the 128-key kernel and the merged correction form; with the
    correction warpgroup, or inside a capture, the flag is ignored and the
    call gives the unsplit bits."""
    B, H, S = 4, 16, 2048
    assert _tail(B, H, S, S) == _tail(B, H, S, S, flags=fa.FA_FLAG_TAIL_SPLIT) > 0
    assert _tail(B, H, S, S, flags=PAIR) == 0
    assert fa.fa_prefill_tail_items(B, H, S, S, 128, True, torch.bfloat16, SPLIT) == 0
    assert _tail(B, H, S, S, flags=SPLIT | fa.FA_FLAG_PAIR64) == 0
    assert _tail(B, H, S, S, flags=SPLIT | fa.FA_FLAG_SINGLE_CTA) == 0
    assert _tail(B, H, S, S, flags=SPLIT | fa.FA_FLAG_CORRECTION_WG) == 0
    q, k, v = (t.cuda() for t in inputs.make_qkv(B, H, S, S, 128, "bf16", 66))
    o0, l0 = fa.fa_fwd(q, k, v)
    o1, l1 = fa.fa_fwd_ex(q, k, v, flags=fa.FA_FLAG_TAIL_SPLIT)
    o2, l2 = fa.fa_fwd_ex(q, k, v, flags=fa.FA_FLAG_TAIL_SPLIT | fa.FA_FLAG_CORRECTION_WG)
    torch.cuda.synchronize()
    assert torch.equal(o0, o2) and torch.equal(l0, l2)
    assert not torch.equal(o0, o1)
    _assert(check(q.cpu(), k.cpu(), v.cpu(), o1, l1, False, "bf16",
                  rows=np.arange(60 * S, 64 * S, 5)))
    o, lse = torch.empty_like(o0), torch.empty_like(l0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fa.fa_fwd_ex(q, k, v, flags=fa.FA_FLAG_TAIL_SPLIT, out=o, lse=lse)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, o0) and torch.equal(lse, l0)
